// Host side of the C ABI declared in include/kgw.h: argument validation, workspace sizing,
// TMA tensor-map encoding and the two launches (plan + persistent kernel) of one call.
//
// The checks follow "Grouped GEMM + WGrad (Unified)", sections "BF16 contract", "Output modes"
// and "Scheduling, cache, and errors" (unsupported dtypes or layouts, malformed or unaligned
// pointers and devices below SM100 are rejected). Everything that needs the device-resident
// offsets is checked on the device by the plan kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kgw.h"
#include "kgw_internal.h"

namespace {

using kgw::WsLayout;

std::atomic<int64_t> g_timeout_ns{2000000000LL};
std::atomic<int64_t> g_drop_stage{-1};
std::atomic<int64_t> g_single_cta{0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

struct DevInfo {
  int sm_count = 0;
  int major = 0, minor = 0;
  bool valid = false;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

kgw_status device_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KGW_ERR_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return KGW_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev[dev].valid) {
    DevInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return KGW_ERR_CUDA;
    }
    d.valid = true;
    g_dev[dev] = d;
  }
  *out = g_dev[dev];
  return KGW_OK;
}

kgw_status get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode ? KGW_OK : KGW_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int bk_of(bool fp8) { return fp8 ? kgw::BK_FP8 : kgw::BK_BF16; }

// Rows of a work tile: problems whose hidden size is a multiple of 256 run on CTA pairs.
int32_t tile_rows(const kgw_wgrad_args* a) {
  if (a->hidden % (2 * kgw::BM) == 0 && g_single_cta.load() == 0) return 2 * kgw::BM;
  return kgw::BM;
}

// Scale rows reserved for the prepared scale words of block-scaled calls on CTA pairs: at least the
// sum over experts of ceil(n_e / 128), which tokens_sum / 128 + E bounds; NVFP4 has two 64-token
// word rows per 128-token block.
int64_t prep_rows(const kgw_wgrad_args* a, bool nv = false) {
  return (a->tokens_sum / kgw::SCALE_BLOCK + a->num_experts) * (nv ? 2 : 1);
}

// Upper bound of the FP32 partial tiles split-K can use for these shapes.
int32_t slot_cap(const kgw_wgrad_args* a, bool fp8) {
  const int64_t T = int64_t(a->hidden / tile_rows(a)) * (a->intermediate / kgw::BN);
  const int64_t kit = a->tokens_sum / bk_of(fp8);
  // an expert is split only when its k-iterations exceed the chunk (>= MIN_SPLIT_KITERS), and
  // then into fewer than 2*kiters/chunk pieces
  const int64_t bound = T * ((2 * kit) / kgw::MIN_SPLIT_KITERS);
  return static_cast<int32_t>(bound < kgw::MAX_PARTIAL_SLOTS ? bound : kgw::MAX_PARTIAL_SLOTS);
}

// count_align: the multiple every token count (and tokens_sum) must be: the pages' 256, or the
// unaligned entry point's 8 (a K-major operand: 16-byte TMA coordinates) / 1 (both MN-major).
kgw_status validate(const kgw_wgrad_args* a, bool fp8, bool fp4 = false, int64_t count_align = kgw::TOKEN_ALIGN) {
  if (!a) return KGW_ERR_INVALID_ARG;
  if (a->num_experts < 1 || a->num_experts > kgw::MAX_EXPERTS) return KGW_ERR_INVALID_ARG;
  if (a->hidden <= 0 || a->intermediate <= 0 || a->tokens_sum < 0) return KGW_ERR_INVALID_ARG;
  if (a->tokens_sum % count_align != 0) return KGW_ERR_INVALID_ARG;
  if (a->hidden % kgw::BM != 0 || a->intermediate % kgw::BN != 0) return KGW_ERR_UNSUPPORTED;
  if (a->a_major != KGW_K_MAJOR && a->a_major != KGW_MN_MAJOR) return KGW_ERR_INVALID_ARG;
  if (a->b_major != KGW_K_MAJOR && a->b_major != KGW_MN_MAJOR) return KGW_ERR_INVALID_ARG;
  if (a->input_order != KGW_TENSOR2D && a->input_order != KGW_RAGGED) return KGW_ERR_INVALID_ARG;
  if (a->out_dtype != KGW_OUT_F32 && a->out_dtype != KGW_OUT_BF16 && a->out_dtype != KGW_OUT_F16)
    return KGW_ERR_INVALID_ARG;
  if (a->accumulate != 0 && a->accumulate != 1) return KGW_ERR_INVALID_ARG;
  // FP4: both operands K-major (the token axis packed two elements per byte; the packed-FP4 MMA
  // reads K-major operands only), in either input order
  if (fp4 && (a->a_major != KGW_K_MAJOR || a->b_major != KGW_K_MAJOR)) return KGW_ERR_UNSUPPORTED;
  if (!a->offsets) return KGW_ERR_INVALID_ARG;
  if ((a->out == nullptr) == (a->out_ptrs == nullptr)) return KGW_ERR_INVALID_ARG;
  if (!aligned(a->offsets, 4)) return KGW_ERR_ALIGNMENT;
  if (a->out && !aligned(a->out, 16)) return KGW_ERR_ALIGNMENT;
  if (a->out_ptrs && !aligned(a->out_ptrs, 8)) return KGW_ERR_ALIGNMENT;
  if (a->status_dev && !aligned(a->status_dev, 4)) return KGW_ERR_ALIGNMENT;
  if (a->tokens_sum > 0) {
    if (!a->a || !a->b) return KGW_ERR_INVALID_ARG;
    if (!aligned(a->a, 16) || !aligned(a->b, 16)) return KGW_ERR_ALIGNMENT;
    const int64_t esz = fp8 ? 1 : 2;
    (void)esz;
    // TMA coordinates and per-expert extents are int32
    if (a->tokens_sum >= (int64_t(1) << 31)) return KGW_ERR_UNSUPPORTED;
  }
  // work items must fit int32: T * (E + 2*kiters/MIN_SPLIT)
  const int64_t T = int64_t(a->hidden / kgw::BM) * (a->intermediate / kgw::BN);
  const int64_t items = T * (a->num_experts + 2 * (a->tokens_sum / bk_of(fp8)) / kgw::MIN_SPLIT_KITERS + 1);
  if (items >= (int64_t(1) << 31)) return KGW_ERR_UNSUPPORTED;
  return KGW_OK;
}

// Plain (unswizzled) 2-D map of 32-bit words: the prepared scale words of FP8 on CTA pairs.
kgw_status encode_2d_words(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {box_inner, 1};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KGW_OK : KGW_ERR_CUDA;
}

kgw_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KGW_OK : KGW_ERR_CUDA;
}

// Everything one call needs: validated arguments turned into kernel parameters.
struct Prepared {
  kgw::PlanParams pp;
  kgw::MainParams mp;
  CUtensorMap tmA;  // A's descriptor (for ragged K-major A: the small-class template, unused)
  CUtensorMap tmB;  // B's descriptor (likewise)
  kgw::MapTemplates tpl;  // templates of per-expert descriptors (ragged, K-major operands)
  int grid;
};

// Token-count multiple of the unaligned entries. A TMA coordinate along an operand's innermost
// axis must start on 16 bytes, so when an operand stores tokens innermost (K-major) every
// expert's first token must sit on a 16-byte boundary: 8 BF16 tokens, 16 e4m3 tokens, 32 packed
// e2m1 tokens (FP4 operands are always K-major). With both operands MN-major any count works.
int64_t unaligned_count_multiple(const kgw_wgrad_args* a, bool fp8 = false, bool fp4 = false) {
  if (fp4) return 32;
  if (a->a_major != KGW_K_MAJOR && a->b_major != KGW_K_MAJOR) return 1;
  return fp8 ? 16 : 8;
}

kgw_status prepare(const kgw_wgrad_args* a, bool fp8, const float* sfa, const float* sfb, void* ws,
                   size_t ws_bytes, Prepared* P, bool fp4 = false, bool tail = false, bool nv = false) {
  const int64_t count_align = tail ? unaligned_count_multiple(a, fp8, fp4) : kgw::TOKEN_ALIGN;
  kgw_status st = validate(a, fp8, fp4, count_align);
  if (st != KGW_OK) return st;
  if (fp8 && !kgw::fp8_supported()) return KGW_ERR_UNSUPPORTED;
  if (fp8 && a->tokens_sum > 0) {
    if (!sfa || !sfb) return KGW_ERR_INVALID_ARG;
    if (!aligned(sfa, 16) || !aligned(sfb, 16)) return KGW_ERR_ALIGNMENT;
  }
  if (!ws || !aligned(ws, 256)) return KGW_ERR_WORKSPACE;
  const int32_t tile_m = tile_rows(a);
  const int32_t halves = tile_m / kgw::BM;
  // block-scaled calls on CTA pairs: prepared scale words of every scale row in the workspace
  const bool fp8_pair = fp8 && halves == 2;
  const int64_t sf_rows = fp8_pair ? prep_rows(a, nv) : 0;
  const WsLayout L0 = kgw::ws_layout(a->num_experts, 0, halves, sf_rows, a->hidden, a->intermediate);
  if (ws_bytes < L0.total) return KGW_ERR_WORKSPACE;
  int32_t max_slots = slot_cap(a, fp8);
  {
    const size_t room = ws_bytes - L0.total;
    const size_t fit = room / (halves * (kgw::PARTIAL_TILE_BYTES + 4 * kgw::EPI_COUNTERS));
    if (size_t(max_slots) > fit) max_slots = static_cast<int32_t>(fit);
    while (max_slots > 0 &&
           kgw::ws_layout(a->num_experts, max_slots, halves, sf_rows, a->hidden, a->intermediate).total > ws_bytes)
      --max_slots;
  }
  const WsLayout L = kgw::ws_layout(a->num_experts, max_slots, halves, sf_rows, a->hidden, a->intermediate);

  DevInfo dev;
  st = device_info(&dev);
  if (st != KGW_OK) return st;
  if (dev.major != 10 || dev.minor != 3) return KGW_ERR_DEVICE;
  if (get_encoder() != KGW_OK) return KGW_ERR_CUDA;

  // k-iteration length in tokens (K-grouped CTA pairs, aligned entries: BF16 128 tokens per stage,
  // FP4 with UE8M0 scales 512)
  const bool wide_k = (!fp8 || (fp4 && !nv)) && halves == 2 && !tail;
  const int bk = fp4 ? (wide_k ? kgw::BK_FP4_PAIR : kgw::BK_FP4)
                     : fp8 ? kgw::BK_FP8 : (wide_k ? kgw::BK_BF16_PAIR : kgw::BK_BF16);
  const uint64_t esz = fp8 ? 1 : 2;
  // token-axis box of a K-major operand in descriptor elements: one 128-byte swizzle row (packed
  // FP4 descriptors count bytes, so its 256 tokens are 128 elements; a 128-token BF16 stage loads
  // two such boxes)
  const uint32_t box_k = fp4 ? 128u : fp8 ? static_cast<uint32_t>(bk) : static_cast<uint32_t>(kgw::BK_BF16);
  std::memset(&P->tmA, 0, sizeof(P->tmA));
  std::memset(&P->tmB, 0, sizeof(P->tmB));
  std::memset(&P->tpl, 0, sizeof(P->tpl));
  const bool ragged = a->input_order == KGW_RAGGED;
  const bool a_k = a->a_major == KGW_K_MAJOR;
  const bool b_k = a->b_major == KGW_K_MAJOR;
  const uint32_t b_rows_cta = static_cast<uint32_t>(kgw::BN / halves);  // B columns one CTA loads
  if (a->tokens_sum > 0) {
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t Ts = static_cast<uint64_t>(a->tokens_sum);
    const uint64_t H = static_cast<uint64_t>(a->hidden), I = static_cast<uint64_t>(a->intermediate);
    const uint32_t atom = static_cast<uint32_t>(128 / esz);  // elements in one 128-byte swizzle row
    // Template of a per-expert [rows, n] block (row stride n elements), in the size class below or
    // at/above 128 KiB; the plan kernel sets the address, n and the stride per expert.
    auto templates = [&](const void* base, uint64_t rows, uint32_t box_rows, CUtensorMap* small,
                         CUtensorMap* large) {
      // small class: the narrowest block (16-byte rows), under 128 KiB unless rows alone reach it
      const uint64_t n_small = 16 / esz;
      uint64_t n_large = (kgw::TMAP_SIZE_CLASS_BYTES + rows * esz - 1) / (rows * esz);
      n_large = (n_large + kgw::TOKEN_ALIGN - 1) / kgw::TOKEN_ALIGN * kgw::TOKEN_ALIGN;
      if (n_large < n_small) n_large = n_small;
      kgw_status r = encode_2d(small, dt, base, n_small, rows, n_small * esz, box_k, box_rows);
      if (r == KGW_OK) r = encode_2d(large, dt, base, n_large, rows, n_large * esz, box_k, box_rows);
      return r;
    };
    if (fp4 && !ragged) {
      // packed e2m1: the tensors count bytes along the token axis (two tokens per byte)
      st = encode_2d(&P->tmA, dt, a->a, Ts / 2, H, Ts / 2, 128, kgw::BM);             // [H, tokens/2]
      if (st == KGW_OK) st = encode_2d(&P->tmB, dt, a->b, Ts / 2, I, Ts / 2, 128, b_rows_cta);  // [I, tokens/2]
      if (st != KGW_OK) return st;
    }
    // A (ragged packed FP4: per-expert [hidden, n_e/2]-byte blocks, through the templates below)
    if (fp4 && !ragged) {
    } else if (a_k && !ragged) {
      st = encode_2d(&P->tmA, dt, a->a, Ts, H, Ts * esz, box_k, kgw::BM);          // [H, tokens]
    } else if (a_k) {
      st = templates(a->a, H, kgw::BM, &P->tpl.a_small, &P->tpl.a_large);
      P->tmA = P->tpl.a_small;
    } else {
      st = encode_2d(&P->tmA, dt, a->a, H, Ts, H * esz, atom, bk);                 // [tokens, H]
    }
    if (st != KGW_OK) return st;
    // B
    if (fp4 && !ragged) {
    } else if (b_k && !ragged) {
      st = encode_2d(&P->tmB, dt, a->b, Ts, I, Ts * esz, box_k, b_rows_cta);      // [I, tokens]
    } else if (b_k) {
      st = templates(a->b, I, b_rows_cta, &P->tpl.b_small, &P->tpl.b_large);
      P->tmB = P->tpl.b_small;
    } else {
      st = encode_2d(&P->tmB, dt, a->b, I, Ts, I * esz, atom, bk);                 // [tokens, I]
    }
    if (st != KGW_OK) return st;
    if (tail) {
      // token tails: per-expert copies of the operand's own descriptor with the token extent cut
      // at end_e; an MN-major operand's small-class template has a token extent under 128 KiB
      auto tail_templates = [&](const CUtensorMap& whole, const void* base, uint64_t cols, uint64_t row_bytes,
                                bool k_major, uint32_t box_inner, uint32_t box_outer, CUtensorMap* small,
                                CUtensorMap* large) {
        *large = whole;
        if (k_major) {
          *small = whole;
          return KGW_OK;
        }
        return encode_2d(small, dt, base, cols, 1, row_bytes, box_inner, box_outer);
      };
      if (!(ragged && a_k)) {
        st = tail_templates(P->tmA, a->a, H, H * esz, a_k, atom, bk, &P->tpl.a_small, &P->tpl.a_large);
        if (st != KGW_OK) return st;
      }
      if (!(ragged && b_k)) {
        st = tail_templates(P->tmB, a->b, I, I * esz, b_k, atom, bk, &P->tpl.b_small, &P->tpl.b_large);
        if (st != KGW_OK) return st;
      }
    }
  }

  kgw::PlanParams& pp = P->pp;
  pp = kgw::PlanParams{};
  pp.E = a->num_experts;
  pp.H = a->hidden;
  pp.I = a->intermediate;
  pp.tokens_sum = a->tokens_sum;
  pp.offsets = a->offsets;
  pp.out_ptrs = a->out_ptrs;
  pp.accumulate = a->accumulate;
  pp.bk = bk;
  const int grid = halves == 2 ? (dev.sm_count & ~1) : dev.sm_count;
  pp.grid = grid / halves;  // tiles in flight at once
  pp.max_slots = max_slots;
  pp.tile_m = tile_m;
  pp.status_dev = a->status_dev;
  pp.ws = static_cast<uint8_t*>(ws);
  pp.L = L;
  pp.build_a = ragged && a_k && a->tokens_sum > 0;
  pp.build_b = ragged && b_k && a->tokens_sum > 0;
  pp.a = static_cast<const uint8_t*>(a->a);
  pp.b = static_cast<const uint8_t*>(a->b);
  pp.esz = static_cast<int32_t>(esz);
  pp.count_align = static_cast<int32_t>(count_align);
  pp.tok_per_unit = fp4 ? 2 : 1;
  if (tail && a->tokens_sum > 0) {
    pp.tail_a = (ragged && a_k) ? 0 : (a_k ? 1 : 2);   // ragged K-major blocks already end at n_e
    pp.tail_b = (ragged && b_k) ? 0 : (b_k ? 1 : 2);
    pp.row_bytes_a = static_cast<uint64_t>(a->hidden) * esz;
    pp.row_bytes_b = static_cast<uint64_t>(a->intermediate) * esz;
  }

  kgw::MainParams& mp = P->mp;
  mp = kgw::MainParams{};
  mp.E = a->num_experts;
  mp.H = a->hidden;
  mp.I = a->intermediate;
  mp.tokens_sum = a->tokens_sum;
  mp.offsets = a->offsets;
  mp.out_ptrs = a->out_ptrs;
  mp.out = a->out;
  mp.out_bf16 = a->out_dtype == KGW_OUT_BF16 || a->out_dtype == KGW_OUT_F16;
  mp.out_f16 = a->out_dtype == KGW_OUT_F16;
  mp.accumulate = a->accumulate;
  mp.ragged = ragged;
  mp.a_kmajor = a_k;
  mp.b_kmajor = b_k;
  mp.discrete = a->out_ptrs != nullptr;
  mp.fp8 = fp8;
  mp.num_m_tiles = a->hidden / tile_m;
  mp.tile_m = tile_m;
  mp.num_n_tiles = a->intermediate / kgw::BN;
  mp.sfa = sfa;
  mp.sfb = sfb;
  mp.status_dev = a->status_dev;
  mp.ws = static_cast<uint8_t*>(ws);
  mp.L = L;
  mp.timeout_ns = static_cast<uint64_t>(g_timeout_ns.load());
  mp.test_drop_stage = static_cast<int32_t>(g_drop_stage.load());
  mp.wide_k = wide_k ? 1 : 0;
  mp.tail_a = pp.tail_a;
  mp.tail_b = pp.tail_b;
  mp.sf_prep = fp8_pair;
  if (fp8_pair && a->tokens_sum > 0) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    st = encode_2d_words(&mp.tm_sfa, w + L.sf_prep_a, static_cast<uint64_t>(a->hidden), static_cast<uint64_t>(sf_rows),
                         kgw::BM);
    if (st == KGW_OK)
      st = encode_2d_words(&mp.tm_sfb, w + L.sf_prep_b, static_cast<uint64_t>(a->intermediate),
                           static_cast<uint64_t>(sf_rows), kgw::BN);
    if (st != KGW_OK) return st;
  }
  P->grid = grid;
  return KGW_OK;
}

kgw_status run(const kgw_wgrad_args* a, bool fp8, const float* sfa, const float* sfb, void* ws, size_t ws_bytes,
               void* stream, bool sf_packed = false, bool fp4 = false, bool tail = false, bool nvfp4 = false,
               const float* gscale_a = nullptr, const float* gscale_b = nullptr) {
  if ((gscale_a && !aligned(gscale_a, 4)) || (gscale_b && !aligned(gscale_b, 4))) return KGW_ERR_ALIGNMENT;
  Prepared P;
  kgw_status st = prepare(a, fp8, sfa, sfb, ws, ws_bytes, &P, fp4, tail, nvfp4);
  if (st != KGW_OK) return st;
  P.mp.sf_packed = sf_packed;
  P.mp.nvfp4 = nvfp4;
  P.mp.gscale_a = gscale_a;
  P.mp.gscale_b = gscale_b;
  // FP8 with FP32 scales: a device check of every scale decides whether the FP8 kernel uses the
  // block-scaled MMA (all powers of two) or its per-block promotion path
  const bool general = fp8 && !fp4 && !sf_packed;
  P.mp.general_dispatch = general;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kgw::launch_plan(P.pp, P.tpl, s) != cudaSuccess) return KGW_ERR_CUDA;
  // the scale kernel: the FP32 power-of-two check, and the prepared scale words of FP8 and FP4
  // pairs (with the NaN-byte check of packed words)
  if ((general || P.mp.sf_prep) && a->tokens_sum > 0 && kgw::launch_scale_check(P.mp, 4 * P.grid, s) != cudaSuccess)
    return KGW_ERR_CUDA;
  if (general && P.mp.sf_prep && a->tokens_sum > 0 && kgw::launch_promote_kernel(P.mp, P.tmA, P.tmB, P.grid, s) != cudaSuccess)
    return KGW_ERR_CUDA;
  cudaError_t e = fp4 ? kgw::launch_main_fp4(P.mp, P.tmA, P.tmB, P.grid, s)
                 : fp8 ? kgw::launch_main_fp8(P.mp, P.tmA, P.tmB, P.grid, s)
                       : kgw::launch_main_bf16(P.mp, P.tmA, P.tmB, P.grid, s);
  return e == cudaSuccess ? KGW_OK : KGW_ERR_CUDA;
}

// ---------------------------------------------------------------------------------------------
// Entry point without allocation: the scratch (schedule + split-K partials) lives in a
// file-scope device array instead of a caller-provided workspace.
// ---------------------------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB per device that loads the library
constexpr int32_t kNoAllocMaxExperts = 1024;

// Host code may not pass this name to a kernel: on the host it is only a stand-in for the
// device array. Its device address comes from cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Per device: the context the address was looked up in, and the address. A device reset (or a
// primary context torn down and created again) gives the device a new context in which the array
// lives at another address, so the address is looked up again whenever the current context differs.
void* g_noalloc_ptr[kMaxDevices] = {};
CUcontext g_noalloc_ctx[kMaxDevices] = {};
std::mutex g_noalloc_mu;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_current_once;

kgw_status current_context(CUcontext* ctx) {
  std::call_once(g_ctx_current_once, [] {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    else
      cudaGetLastError();
  });
  if (!g_ctx_current) return KGW_ERR_CUDA;
  *ctx = nullptr;
  return g_ctx_current(ctx) == CUDA_SUCCESS ? KGW_OK : KGW_ERR_CUDA;
}

// Device address of the static scratch on the current device: looked up (cudaGetSymbolAddress,
// with the device current) on the first call on each device and again after its context changed.
kgw_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KGW_ERR_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return KGW_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  void* p = g_noalloc_ptr[dev];
  if (p) {
    CUcontext ctx = nullptr;
    if (current_context(&ctx) != KGW_OK) return KGW_ERR_CUDA;
    if (ctx != g_noalloc_ctx[dev]) p = nullptr;
  }
  if (!p) {
    // the runtime binds the device's primary context here if no call has yet
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return KGW_ERR_CUDA;
    }
    CUcontext ctx = nullptr;
    if (current_context(&ctx) != KGW_OK || ctx == nullptr) return KGW_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = p;
  return KGW_OK;
}

// Rows of A (and D) and the largest tile-table size of an M-grouped call.
int64_t mg_rows(const kgw_mgrouped_args* a) {
  return a->layout == KGW_MG_MASKED ? int64_t(a->num_groups) * a->m : a->m;
}
int64_t mg_max_tiles(const kgw_mgrouped_args* a) {
  return a->layout == KGW_MG_MASKED ? int64_t(a->num_groups) * ((a->m + kgw::BM - 1) / kgw::BM) : a->m / kgw::BM;
}

kgw_status validate_mg(const kgw_mgrouped_args* a, bool fp8 = false) {
  if (!a) return KGW_ERR_INVALID_ARG;
  if (a->num_groups < 1 || a->num_groups > kgw::MAX_EXPERTS) return KGW_ERR_INVALID_ARG;
  if (a->layout != KGW_MG_OFFSETS && a->layout != KGW_MG_INDICES && a->layout != KGW_MG_MASKED)
    return KGW_ERR_INVALID_ARG;
  if (a->m < 0 || a->n <= 0 || a->k <= 0) return KGW_ERR_INVALID_ARG;
  if (a->layout != KGW_MG_MASKED && a->m % kgw::MG_ROW_ALIGN != 0) return KGW_ERR_INVALID_ARG;
  if (a->m >= (int64_t(1) << 31) || mg_rows(a) >= (int64_t(1) << 31)) return KGW_ERR_UNSUPPORTED;
  if (a->n % kgw::BN != 0 || a->k % (fp8 ? kgw::BK_FP8 : kgw::BK_BF16) != 0) return KGW_ERR_UNSUPPORTED;
  if (int64_t(a->num_groups) * a->n >= (int64_t(1) << 31) || int64_t(a->num_groups) * a->k >= (int64_t(1) << 31))
    return KGW_ERR_UNSUPPORTED;
  if (mg_max_tiles(a) * (a->n / kgw::BN) >= (int64_t(1) << 31)) return KGW_ERR_UNSUPPORTED;
  if (a->b_major != KGW_K_MAJOR && a->b_major != KGW_MN_MAJOR) return KGW_ERR_INVALID_ARG;
  if (a->out_dtype != KGW_OUT_F32 && a->out_dtype != KGW_OUT_BF16 && a->out_dtype != KGW_OUT_F16)
    return KGW_ERR_INVALID_ARG;
  if (a->accumulate != 0 && a->accumulate != 1) return KGW_ERR_INVALID_ARG;
  const bool has_rows = mg_rows(a) > 0;
  if (!a->b || (!a->groups && (a->layout != KGW_MG_INDICES || has_rows)) || (has_rows && (!a->a || !a->d)))
    return KGW_ERR_INVALID_ARG;
  if (!aligned(a->b, 16) || (a->groups && !aligned(a->groups, 4)) || (a->a && !aligned(a->a, 16)) ||
      (a->d && !aligned(a->d, 16)))
    return KGW_ERR_ALIGNMENT;
  if (a->status_dev && !aligned(a->status_dev, 4)) return KGW_ERR_ALIGNMENT;
  return KGW_OK;
}

kgw_status run_mg(const kgw_mgrouped_args* a, void* ws, size_t ws_bytes, void* stream, bool fp8 = false,
                  const void* sfa = nullptr, const void* sfb = nullptr, int32_t sf_format = 0) {
  kgw_status st = validate_mg(a, fp8);
  if (st != KGW_OK) return st;
  if (fp8) {
    if (sf_format != 0 && sf_format != 1) return KGW_ERR_INVALID_ARG;
    if (mg_rows(a) > 0 && (!sfa || !sfb)) return KGW_ERR_INVALID_ARG;
    if ((sfa && !aligned(sfa, 16)) || (sfb && !aligned(sfb, 16))) return KGW_ERR_ALIGNMENT;
  }
  if (!ws || !aligned(ws, 256)) return KGW_ERR_WORKSPACE;
  const WsLayout L = kgw::ws_layout_mg(mg_max_tiles(a));
  if (ws_bytes < L.total) return KGW_ERR_WORKSPACE;
  DevInfo dev;
  st = device_info(&dev);
  if (st != KGW_OK) return st;
  if (dev.major != 10 || dev.minor != 3) return KGW_ERR_DEVICE;
  if (get_encoder() != KGW_OK) return KGW_ERR_CUDA;
  CUtensorMap tmA, tmB;
  std::memset(&tmA, 0, sizeof(tmA));
  std::memset(&tmB, 0, sizeof(tmB));
  const uint64_t M = static_cast<uint64_t>(mg_rows(a)), N = static_cast<uint64_t>(a->n),
                 K = static_cast<uint64_t>(a->k), G = static_cast<uint64_t>(a->num_groups);
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t esz = fp8 ? 1 : 2;
  const uint32_t bk = fp8 ? kgw::BK_FP8 : kgw::BK_BF16;   // one 128-byte swizzle row of K
  // BF16 runs on CTA pairs (two 128-row tiles of one group per work row); FP8 on single CTAs.
  // In a pair each CTA loads 128 of the tile's 256 columns of B. BF16 pairs take 128-token stages
  // (two rows of K) when K is a multiple of 128, except in the masked layout: its decode batches
  // are HBM-bound, and the shorter stages keep more loads in flight (128-token stages: +3.7 %).
  const bool pair = !fp8 && g_single_cta.load() == 0;
  const bool wide_k = pair && a->k % (2 * kgw::BK_BF16) == 0 && a->layout != KGW_MG_MASKED;
  const uint32_t b_rows_cta = pair ? kgw::BN / 2 : kgw::BN;
  if (M > 0) {
    st = encode_2d(&tmA, dt, a->a, K, M, K * esz, bk, kgw::BM);                          // A [rows, K]
    if (st != KGW_OK) return st;
    if (a->b_major == KGW_K_MAJOR)
      st = encode_2d(&tmB, dt, a->b, K, G * N, K * esz, bk, b_rows_cta);               // B [G*N, K]
    else
      st = encode_2d(&tmB, dt, a->b, N, G * K, N * esz, static_cast<uint32_t>(128 / esz), bk * (wide_k ? 2 : 1));  // B [G*K, N]
    if (st != KGW_OK) return st;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  kgw::PlanParams pp{};
  pp.E = a->num_groups;
  pp.I = a->n;
  pp.offsets = a->groups;
  pp.grid = dev.sm_count;
  pp.status_dev = a->status_dev;
  pp.ws = static_cast<uint8_t*>(ws);
  pp.L = L;
  pp.tile_m = kgw::BM;
  pp.mg_layout = a->layout;
  pp.mg_m = a->m;
  pp.mg_pair = pair;
  const int grid = pair ? (dev.sm_count & ~1) : dev.sm_count;
  if (kgw::launch_plan_mgrouped(pp, s) != cudaSuccess) return KGW_ERR_CUDA;
  kgw::MainParams mp{};
  mp.E = a->num_groups;
  mp.H = static_cast<int32_t>(M);   // rows of A: the row stride of A's scales
  mp.I = a->n;
  mp.K = a->k;
  mp.fp8 = fp8;
  mp.sfa = static_cast<const float*>(sfa);
  mp.sfb = static_cast<const float*>(sfb);
  mp.sf_packed = sf_format == 1;
  mp.tokens_sum = static_cast<int64_t>(M);
  mp.out = a->d;
  mp.out_bf16 = a->out_dtype == KGW_OUT_BF16 || a->out_dtype == KGW_OUT_F16;
  mp.out_f16 = a->out_dtype == KGW_OUT_F16;
  mp.accumulate = a->accumulate;
  mp.a_kmajor = 1;
  mp.b_kmajor = a->b_major == KGW_K_MAJOR;
  mp.num_n_tiles = a->n / kgw::BN;
  mp.tile_m = pair ? 2 * kgw::BM : kgw::BM;
  mp.status_dev = a->status_dev;
  mp.ws = static_cast<uint8_t*>(ws);
  mp.L = L;
  mp.timeout_ns = static_cast<uint64_t>(g_timeout_ns.load());
  mp.test_drop_stage = -1;
  mp.wide_k = wide_k ? 1 : 0;
  return kgw::launch_main_mgrouped(mp, tmA, tmB, grid, s) == cudaSuccess ? KGW_OK : KGW_ERR_CUDA;
}

}  // namespace

extern "C" {

kgw_status kgw_workspace_size(const kgw_wgrad_args* args, int32_t is_fp8, size_t* bytes) {
  if (!bytes) return KGW_ERR_INVALID_ARG;
  kgw_status st = validate(args, is_fp8 != 0, false, 1);  // sizing only: the call checks its own count rule
  if (st != KGW_OK) return st;
  // is_fp8 sizes the FP8, FP4 and NVFP4 entries alike: the largest need (NVFP4 on CTA pairs, with
  // two prepared word rows per 128-token block) covers all three
  const int32_t halves = tile_rows(args) / kgw::BM;
  const int64_t sf_rows = (is_fp8 != 0 && halves == 2) ? prep_rows(args, true) : 0;
  *bytes = kgw::ws_layout(args->num_experts, slot_cap(args, is_fp8 != 0), halves, sf_rows, args->hidden,
                          args->intermediate).total;
  return KGW_OK;
}

kgw_status kgw_wgrad_bf16(const kgw_wgrad_args* args, void* workspace, size_t workspace_bytes, void* stream) {
  return run(args, false, nullptr, nullptr, workspace, workspace_bytes, stream);
}

kgw_status kgw_wgrad_fp8_blockscaled(const kgw_wgrad_args* args, const float* sfa, const float* sfb,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return run(args, true, sfa, sfb, workspace, workspace_bytes, stream);
}

kgw_status kgw_wgrad_fp8_ue8m0(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return run(args, true, reinterpret_cast<const float*>(sfa_packed), reinterpret_cast<const float*>(sfb_packed),
             workspace, workspace_bytes, stream, true);
}

kgw_status kgw_wgrad_bf16_unaligned(const kgw_wgrad_args* args, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  return run(args, false, nullptr, nullptr, workspace, workspace_bytes, stream, false, false, true);
}

kgw_status kgw_wgrad_fp4_ue8m0(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return run(args, true, reinterpret_cast<const float*>(sfa_packed), reinterpret_cast<const float*>(sfb_packed),
             workspace, workspace_bytes, stream, true, true);
}

kgw_status kgw_wgrad_nvfp4(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                           const float* global_scale_a, const float* global_scale_b, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return run(args, true, reinterpret_cast<const float*>(sfa_packed), reinterpret_cast<const float*>(sfb_packed),
             workspace, workspace_bytes, stream, true, true, false, true, global_scale_a, global_scale_b);
}

kgw_status kgw_wgrad_fp8_unaligned(const kgw_wgrad_args* args, const void* sfa, const void* sfb, int32_t sf_format,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (sf_format != 0 && sf_format != 1) return KGW_ERR_INVALID_ARG;
  return run(args, true, static_cast<const float*>(sfa), static_cast<const float*>(sfb), workspace, workspace_bytes,
             stream, sf_format == 1, false, true);
}

kgw_status kgw_wgrad_fp4_unaligned(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  return run(args, true, reinterpret_cast<const float*>(sfa_packed), reinterpret_cast<const float*>(sfb_packed),
             workspace, workspace_bytes, stream, true, true, true);
}

kgw_status kgw_wgrad_bf16_noalloc(const kgw_wgrad_args* args, void* stream) {
  kgw_status st = validate(args, false);
  if (st != KGW_OK) return st;
  if (args->num_experts > kNoAllocMaxExperts) return KGW_ERR_SCRATCH_LIMIT;
  DevInfo dev;
  st = device_info(&dev);
  if (st != KGW_OK) return st;
  if (dev.major != 10 || dev.minor != 3) return KGW_ERR_DEVICE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != KGW_OK) return st;
  return run(args, false, nullptr, nullptr, scratch, kNoAllocScratchBytes, stream);
}

int32_t kgw_debug_check_ragged_maps(const kgw_wgrad_args* args, int32_t is_fp8, const int32_t* host_offsets,
                                    void* workspace, size_t workspace_bytes, void* host_dump) {
  if (!args || !host_offsets || args->input_order != KGW_RAGGED || args->tokens_sum <= 0) return -KGW_ERR_INVALID_ARG;
  Prepared P;
  kgw_status st = prepare(args, is_fp8 != 0, reinterpret_cast<const float*>(args->a),
                          reinterpret_cast<const float*>(args->a), workspace, workspace_bytes, &P);
  if (st != KGW_OK) return -static_cast<int32_t>(st);
  if (kgw::launch_plan(P.pp, P.tpl, nullptr) != cudaSuccess) return -KGW_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return -KGW_ERR_CUDA;
  const int32_t E = args->num_experts;
  const size_t bytes = size_t(E) * 128;
  uint8_t* dev_maps = static_cast<uint8_t*>(std::malloc(2 * bytes));
  if (!dev_maps) return -KGW_ERR_INVALID_ARG;
  if (cudaMemcpy(dev_maps, static_cast<uint8_t*>(workspace) + P.pp.L.tmaps, bytes, cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(dev_maps + bytes, static_cast<uint8_t*>(workspace) + P.pp.L.tmaps_b, bytes,
                 cudaMemcpyDeviceToHost) != cudaSuccess) {
    std::free(dev_maps);
    return -KGW_ERR_CUDA;
  }
  const bool fp8 = is_fp8 != 0;
  const uint64_t esz = fp8 ? 1 : 2;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t b_rows_cta = static_cast<uint32_t>(kgw::BN / (P.pp.tile_m / kgw::BM));
  int32_t mismatches = 0;
  for (int32_t op = 0; op < 2; ++op) {
    if (op == 0 ? !P.pp.build_a : !P.pp.build_b) continue;
    const uint64_t rows = op == 0 ? static_cast<uint64_t>(args->hidden) : static_cast<uint64_t>(args->intermediate);
    const uint8_t* base0 = static_cast<const uint8_t*>(op == 0 ? args->a : args->b);
    for (int32_t e = 0; e < E; ++e) {
      const int64_t begin = e ? host_offsets[e - 1] : 0;
      const int64_t n = host_offsets[e] - begin;
      if (n <= 0) continue;
      CUtensorMap ref;
      std::memset(&ref, 0, sizeof(ref));
      if (encode_2d(&ref, dt, base0 + begin * rows * esz, static_cast<uint64_t>(n), rows, n * esz, bk_of(fp8),
                    op == 0 ? kgw::BM : b_rows_cta) != KGW_OK) {
        std::free(dev_maps);
        return -KGW_ERR_CUDA;
      }
      const uint8_t* got = dev_maps + size_t(op) * bytes + size_t(e) * 128;
      if (std::memcmp(&ref, got, 128) != 0) ++mismatches;
      if (host_dump) {
        uint8_t* d = static_cast<uint8_t*>(host_dump) + (size_t(e) * 2 + op) * 256;
        std::memcpy(d, got, 128);
        std::memcpy(d + 128, &ref, 128);
      }
    }
  }
  std::free(dev_maps);
  return mismatches;
}

int32_t kgw_debug_check_tail_maps_kind(const kgw_wgrad_args* args, int32_t kind, const int32_t* host_offsets,
                                       void* workspace, size_t workspace_bytes, void* host_dump) {
  if (!args || !host_offsets || args->tokens_sum <= 0 || kind < 0 || kind > 2) return -KGW_ERR_INVALID_ARG;
  const bool fp8 = kind >= 1, fp4 = kind == 2;
  Prepared P;
  // the scale pointers are only checked for presence here (the plan kernel does not read them)
  const float* dummy = reinterpret_cast<const float*>(args->a);
  kgw_status st = prepare(args, fp8, dummy, dummy, workspace, workspace_bytes, &P, fp4, true);
  if (st != KGW_OK) return -static_cast<int32_t>(st);
  if (kgw::launch_plan(P.pp, P.tpl, nullptr) != cudaSuccess) return -KGW_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return -KGW_ERR_CUDA;
  const int32_t E = args->num_experts;
  const size_t bytes = size_t(E) * 128;
  uint8_t* dev_maps = static_cast<uint8_t*>(std::malloc(2 * bytes));
  if (!dev_maps) return -KGW_ERR_INVALID_ARG;
  if (cudaMemcpy(dev_maps, static_cast<uint8_t*>(workspace) + P.pp.L.tmaps, bytes, cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(dev_maps + bytes, static_cast<uint8_t*>(workspace) + P.pp.L.tmaps_b, bytes,
                 cudaMemcpyDeviceToHost) != cudaSuccess) {
    std::free(dev_maps);
    return -KGW_ERR_CUDA;
  }
  const uint64_t esz = fp8 ? 1 : 2;
  const uint64_t tpu = fp4 ? 2 : 1;                       // tokens per element of the token axis
  const uint64_t Ts = static_cast<uint64_t>(args->tokens_sum);
  const uint64_t H = static_cast<uint64_t>(args->hidden), I = static_cast<uint64_t>(args->intermediate);
  const uint32_t b_rows_cta = static_cast<uint32_t>(kgw::BN / (P.pp.tile_m / kgw::BM));
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t box_k = fp4 ? 128u : static_cast<uint32_t>(bk_of(fp8));   // token-axis box (elements)
  const uint32_t atom = static_cast<uint32_t>(128 / esz);
  int32_t mismatches = 0;
  for (int32_t op = 0; op < 2; ++op) {
    const int mode = op == 0 ? P.pp.tail_a : P.pp.tail_b;
    const bool block = op == 0 ? P.pp.build_a : P.pp.build_b;   // ragged K-major: per-expert blocks
    if (!mode && !block) continue;
    const uint64_t rows = op == 0 ? H : I;
    const uint8_t* base = static_cast<const uint8_t*>(op == 0 ? args->a : args->b);
    const uint32_t box_rows = op == 0 ? kgw::BM : b_rows_cta;
    for (int32_t e = 0; e < E; ++e) {
      const int64_t begin = e ? host_offsets[e - 1] : 0;
      const int64_t end = host_offsets[e];
      if (end <= begin) continue;
      const uint64_t n = static_cast<uint64_t>(end - begin);
      CUtensorMap ref;
      std::memset(&ref, 0, sizeof(ref));
      kgw_status r = block ? encode_2d(&ref, dt, base + begin * rows * esz / tpu, n / tpu, rows, n * esz / tpu, box_k,
                                       box_rows)
                     : mode == 1 ? encode_2d(&ref, dt, base, static_cast<uint64_t>(end) / tpu, rows, Ts / tpu * esz,
                                             box_k, box_rows)
                                 : encode_2d(&ref, dt, base, rows, static_cast<uint64_t>(end), rows * esz, atom,
                                             static_cast<uint32_t>(P.pp.bk));   // MN-major: k-iteration rows
      if (r != KGW_OK) {
        std::free(dev_maps);
        return -KGW_ERR_CUDA;
      }
      const uint8_t* got = dev_maps + size_t(op) * bytes + size_t(e) * 128;
      if (std::memcmp(&ref, got, 128) != 0) ++mismatches;
      if (host_dump) {
        uint8_t* d = static_cast<uint8_t*>(host_dump) + (size_t(e) * 2 + op) * 256;
        std::memcpy(d, got, 128);
        std::memcpy(d + 128, &ref, 128);
      }
    }
  }
  std::free(dev_maps);
  return mismatches;
}

int32_t kgw_debug_check_tail_maps(const kgw_wgrad_args* args, const int32_t* host_offsets, void* workspace,
                                  size_t workspace_bytes, void* host_dump) {
  return kgw_debug_check_tail_maps_kind(args, 0, host_offsets, workspace, workspace_bytes, host_dump);
}

kgw_status kgw_mgrouped_workspace_size(const kgw_mgrouped_args* args, size_t* bytes) {
  if (!bytes) return KGW_ERR_INVALID_ARG;
  kgw_status st = validate_mg(args);
  if (st != KGW_OK) return st;
  *bytes = kgw::ws_layout_mg(mg_max_tiles(args)).total;
  return KGW_OK;
}

kgw_status kgw_mgrouped_bf16(const kgw_mgrouped_args* args, void* workspace, size_t workspace_bytes, void* stream) {
  return run_mg(args, workspace, workspace_bytes, stream);
}

kgw_status kgw_mgrouped_fp8(const kgw_mgrouped_args* args, const void* sfa, const void* sfb, int32_t sf_format,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return run_mg(args, workspace, workspace_bytes, stream, true, sfa, sfb, sf_format);
}

const char* kgw_status_string(int32_t status) {
  switch (status) {
    case KGW_OK: return "KGW_OK";
    case KGW_ERR_INVALID_ARG: return "KGW_ERR_INVALID_ARG";
    case KGW_ERR_UNSUPPORTED: return "KGW_ERR_UNSUPPORTED";
    case KGW_ERR_ALIGNMENT: return "KGW_ERR_ALIGNMENT";
    case KGW_ERR_DEVICE: return "KGW_ERR_DEVICE";
    case KGW_ERR_CUDA: return "KGW_ERR_CUDA";
    case KGW_ERR_OFFSETS: return "KGW_ERR_OFFSETS";
    case KGW_ERR_TIMEOUT: return "KGW_ERR_TIMEOUT";
    case KGW_ERR_WORKSPACE: return "KGW_ERR_WORKSPACE";
    case KGW_ERR_OUT_PTRS: return "KGW_ERR_OUT_PTRS";
    case KGW_ERR_SCRATCH_LIMIT: return "KGW_ERR_SCRATCH_LIMIT";
    case KGW_ERR_SCALES: return "KGW_ERR_SCALES";
    default: return "KGW_ERR_UNKNOWN";
  }
}

int32_t kgw_version(void) { return 100; }

int64_t kgw_debug_set(int32_t key, int64_t value) {
  switch (key) {
    case 1: return g_timeout_ns.exchange(value > 0 ? value : 1);
    case 2: return g_drop_stage.exchange(value);
    case 3: return g_single_cta.exchange(value);
    default: return -1;
  }
}

}  // extern "C"
