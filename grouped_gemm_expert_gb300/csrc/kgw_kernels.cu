// Kernels of the K-grouped weight-gradient GEMM for sm_103a.
//
//   plan_kernel  (1 CTA)      validates the device-resident offsets, decides split-K, orders
//                             experts longest-first and writes the per-call schedule into the
//                             workspace ("Grouped GEMM + WGrad (Unified)", sections "BF16 contract"
//                             and "Scheduling, cache, and errors": dynamic persistent scheduling).
//   wgrad_kernel (1 CTA / SM, or a CTA pair per 256-row tile) persistent, warp-specialised: a
//                             scheduler warp claims work items from an atomic counter one item
//                             ahead and publishes them decoded in a shared-memory ring; warp 0
//                             streams K-slices of A and B with TMA into a multi-stage shared-memory
//                             ring; warp 1 issues tcgen05.mma into one of two FP32 TMEM
//                             accumulators; warps 2..5 drain TMEM and write the output (overwrite /
//                             accumulate, FP32 / BF16, dense / per-expert pointers), reducing
//                             split-K partial tiles in a fixed order. The block-scaled variant adds
//                             a scale-factor converter warp and uses eight epilogue warps.
//
// A work item is (expert, m-tile, n-tile, K chunk). For expert e the contraction runs over tokens
// [begin_e, end_e) ("Grouped GEMM + WGrad (Unified)", section "Operation").
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <type_traits>

#include "kgw_internal.h"
#include "kgw_ptx.cuh"

namespace kgw {

// =============================================================================================
// Plan kernel
// =============================================================================================

__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* s_warp, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int64_t base = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[nwarps - 1];
  __syncthreads();
  return base + x - v;
}

// Per-thread contiguous chunk of [0, n): thread t owns [t*c, min(n, (t+1)*c)).
struct Chunk {
  int lo, hi;
};
__device__ __forceinline__ Chunk my_chunk(int n) {
  const int c = (n + blockDim.x - 1) / blockDim.x;
  int lo = threadIdx.x * c;
  int hi = lo + c;
  if (lo > n) lo = n;
  if (hi > n) hi = n;
  return {lo, hi};
}

__global__ void __launch_bounds__(PLAN_THREADS)
    plan_kernel(const __grid_constant__ PlanParams p, const __grid_constant__ MapTemplates tm) {
  __shared__ int32_t s_kit[MAX_EXPERTS];    // k-iterations per expert
  __shared__ int32_t s_key[MAX_EXPERTS];    // k-iterations per item (ordering key)
  __shared__ int64_t s_warp[32];
  __shared__ int32_t s_err;

  const int E = p.E;
  const int tid = threadIdx.x;
  const int T = (p.H / p.tile_m) * (p.I / BN);
  const int halves = p.tile_m / BM;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  int32_t* order = reinterpret_cast<int32_t*>(p.ws + p.L.order);
  int32_t* item_prefix = reinterpret_cast<int32_t*>(p.ws + p.L.item_prefix);
  int32_t* splits = reinterpret_cast<int32_t*>(p.ws + p.L.splits);
  int32_t* slot_base = reinterpret_cast<int32_t*>(p.ws + p.L.slot_base);
  int32_t* counter_base = reinterpret_cast<int32_t*>(p.ws + p.L.counter_base);
  int32_t* counters = reinterpret_cast<int32_t*>(p.ws + p.L.counters);

  pdl_launch_dependents();  // the main kernel may launch now; it waits for this grid to finish
  if (tid == 0) s_err = 0;
  __syncthreads();

  // 1. counts and validation (section "BF16 contract": non-decreasing cumulative sum, every
  //    count a multiple of 256, final offset == tokens_sum; "Output modes": one non-null,
  //    16-byte-aligned address per expert).
  for (int e = tid; e < E; e += blockDim.x) {
    const int64_t prev = e ? static_cast<int64_t>(p.offsets[e - 1]) : 0;
    const int64_t cur = p.offsets[e];
    const int64_t n = cur - prev;
    int err = 0;
    if (n < 0 || (n % p.count_align) != 0) err = KGW_ERR_OFFSETS;
    if (e == E - 1 && cur != p.tokens_sum) err = KGW_ERR_OFFSETS;
    if (!err && p.out_ptrs) {
      const uint64_t ptr = static_cast<uint64_t>(p.out_ptrs[e]);
      if (ptr == 0 || (ptr & 15u)) err = KGW_ERR_OUT_PTRS;
    }
    if (err) atomicMax(&s_err, err == KGW_ERR_OFFSETS ? 2 : 1);
    s_kit[e] = n > 0 ? static_cast<int32_t>((n + p.bk - 1) / p.bk) : 0;  // a partial last stage counts
  }
  __syncthreads();
  if (s_err) {
    if (tid == 0) {
      const int code = s_err == 2 ? KGW_ERR_OFFSETS : KGW_ERR_OUT_PTRS;
      hdr->error = code;
      hdr->total_items = 0;
      hdr->item_counter = 0;
      hdr->slots_used = 0;
      hdr->counters_used = 0;
      hdr->general_scales = 0;
      hdr->scale_rows = 0;
      if (p.status_dev) *p.status_dev = code;
    }
    return;
  }

  // 1b. ragged input order: one TMA descriptor per non-empty expert for each K-major operand,
  //     copied from a host-encoded template of the same size class and pointed at the expert's
  //     block ([rows, n_e] row-major at element begin_e*rows; row stride n_e elements).
  if (p.build_a || p.build_b) {
    for (int e = tid; e < E; e += blockDim.x) {
      const int64_t prev = e ? static_cast<int64_t>(p.offsets[e - 1]) : 0;
      const int64_t n = static_cast<int64_t>(p.offsets[e]) - prev;
      if (n <= 0) continue;
#pragma unroll
      for (int op = 0; op < 2; ++op) {
        if (op == 0 ? !p.build_a : !p.build_b) continue;
        const int64_t rows = op == 0 ? p.H : p.I;
        // block extent along the token axis in descriptor elements (packed FP4: bytes, two tokens each)
        const int64_t tpu = p.tok_per_unit > 1 ? p.tok_per_unit : 1;
        const int64_t nu = n / tpu;
        uint4* dst = reinterpret_cast<uint4*>(p.ws + (op == 0 ? p.L.tmaps : p.L.tmaps_b) + size_t(e) * 128);
        const bool large = uint64_t(nu) * uint64_t(rows) * uint64_t(p.esz) >= TMAP_SIZE_CLASS_BYTES;
        const CUtensorMap* t = op == 0 ? (large ? &tm.a_large : &tm.a_small) : (large ? &tm.b_large : &tm.b_small);
        const uint4* src = reinterpret_cast<const uint4*>(t);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = src[j];
        const uint8_t* base = op == 0 ? p.a : p.b;
        tmap_set_address(dst, reinterpret_cast<uint64_t>(base + prev * rows * p.esz / tpu));
        tmap_set_dim0(dst, static_cast<uint32_t>(nu));
        tmap_set_stride1(dst, static_cast<uint64_t>(nu * p.esz));
        fence_tmap_release();
      }
    }
  }

  // 1c. token counts that are not multiples of the stage: per-expert descriptors of the whole
  //     operand whose token extent ends at end_e, so that TMA zero-fills the tail of the
  //     expert's last stage instead of reading the next expert's tokens.
  if (p.tail_a || p.tail_b) {
    for (int e = tid; e < E; e += blockDim.x) {
      const int64_t prev = e ? static_cast<int64_t>(p.offsets[e - 1]) : 0;
      const int64_t end = static_cast<int64_t>(p.offsets[e]);
      if (end <= prev) continue;
#pragma unroll
      for (int op = 0; op < 2; ++op) {
        const int mode = op == 0 ? p.tail_a : p.tail_b;
        if (!mode) continue;
        uint4* dst = reinterpret_cast<uint4*>(p.ws + (op == 0 ? p.L.tmaps : p.L.tmaps_b) + size_t(e) * 128);
        // dimension 0: the size class does not change; dimension 1: end_e x row stride decides it
        const uint64_t rb = op == 0 ? p.row_bytes_a : p.row_bytes_b;
        const bool large = mode == 1 || uint64_t(end) * rb >= TMAP_SIZE_CLASS_BYTES;
        const CUtensorMap* t = op == 0 ? (large ? &tm.a_large : &tm.a_small) : (large ? &tm.b_large : &tm.b_small);
        const uint4* src = reinterpret_cast<const uint4*>(t);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = src[j];
        if (mode == 1)  // (packed FP4: the token axis of the descriptor counts bytes, two tokens each)
          tmap_set_dim0(dst, static_cast<uint32_t>(p.tok_per_unit > 1 ? end / p.tok_per_unit : end));
        else
          tmap_set_dim1(dst, static_cast<uint32_t>(end));
        fence_tmap_release();
      }
    }
  }

  // 2. total k-iterations W = T * sum(kiters)
  int64_t mysum = 0;
  const Chunk ch = my_chunk(E);
  for (int e = ch.lo; e < ch.hi; ++e) mysum += s_kit[e];
  int64_t ksum;
  block_exclusive_scan(mysum, s_warp, &ksum);
  const int64_t W = ksum * T;

  // 2b. first scale row of every expert (block-scaled entries): each expert's tokens form
  //     ceil(n_e / 128) scale blocks starting at its first token, numbered in expert order
  {
    int32_t* scale_row = reinterpret_cast<int32_t*>(p.ws + p.L.scale_row);
    auto blocks = [&](int e) {
      const int64_t prev = e ? static_cast<int64_t>(p.offsets[e - 1]) : 0;
      return (static_cast<int64_t>(p.offsets[e]) - prev + SCALE_BLOCK - 1) / SCALE_BLOCK;
    };
    int64_t mine = 0;
    for (int e = ch.lo; e < ch.hi; ++e) mine += blocks(e);
    int64_t nblk;
    int64_t run = block_exclusive_scan(mine, s_warp, &nblk);
    for (int e = ch.lo; e < ch.hi; ++e) {
      scale_row[e] = static_cast<int32_t>(run);
      run += blocks(e);
    }
    if (tid == 0) hdr->scale_rows = static_cast<int32_t>(nblk);
  }

  // 3. split-K chunk: items no longer than W/(2*grid) k-iterations (at least MIN_SPLIT_KITERS),
  //    doubled until the partial tiles fit in the workspace.
  int64_t C = (W + 2 * int64_t(p.grid) - 1) / (2 * int64_t(p.grid));
  if (C < MIN_SPLIT_KITERS) C = MIN_SPLIT_KITERS;
  int64_t slots = 0;
  for (int iter = 0; iter < 40; ++iter) {
    int64_t mine = 0;
    for (int e = ch.lo; e < ch.hi; ++e)
      if (s_kit[e] > C) mine += int64_t(T) * ((s_kit[e] + C - 1) / C);
    block_exclusive_scan(mine, s_warp, &slots);
    if (slots <= p.max_slots) break;
    C *= 2;
  }
  if (slots > p.max_slots) {  // cannot happen once C exceeds every expert; keep it safe
    C = int64_t(1) << 40;
    slots = 0;
  }

  // 4. per-expert splits, item counts and ordering keys
  for (int e = tid; e < E; e += blockDim.x) {
    const int kit = s_kit[e];
    const int ns = kit > C ? static_cast<int>((kit + C - 1) / C) : 1;
    splits[e] = ns;
    s_key[e] = kit > 0 ? (kit + ns - 1) / ns : 0;
  }
  __syncthreads();

  // 5. order: rank the experts longest item first (ties by expert index), so that the longest
  //    items start in the first wave and the short ones fill the tail of the schedule.
  for (int e = tid; e < E; e += blockDim.x) {
    const int key = s_key[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const int kf = s_key[f];
      rank += (kf > key) || (kf == key && f < e);
    }
    order[rank] = e;
  }
  __syncthreads();
  __threadfence_block();

  // 6. item prefix over the ordered experts
  int64_t myitems = 0;
  for (int q = ch.lo; q < ch.hi; ++q) {
    const int e = order[q];
    myitems += s_kit[e] > 0 ? int64_t(T) * splits[e] : (p.accumulate ? 0 : T);
  }
  int64_t total_items;
  int64_t run = block_exclusive_scan(myitems, s_warp, &total_items);
  for (int q = ch.lo; q < ch.hi; ++q) {
    item_prefix[q] = static_cast<int32_t>(run);
    const int e = order[q];
    run += s_kit[e] > 0 ? int64_t(T) * splits[e] : (p.accumulate ? 0 : T);
  }
  if (tid == 0) item_prefix[E] = static_cast<int32_t>(total_items);

  // 7. partial-slot and counter bases for split experts (expert index order)
  int64_t myslots = 0, mycnt = 0;
  for (int e = ch.lo; e < ch.hi; ++e)
    if (splits[e] > 1) {
      myslots += int64_t(T) * splits[e];
      mycnt += T;
    }
  int64_t slots_total, cnt_total;
  int64_t sb = block_exclusive_scan(myslots, s_warp, &slots_total);
  int64_t cb = block_exclusive_scan(mycnt, s_warp, &cnt_total);
  for (int e = ch.lo; e < ch.hi; ++e) {
    if (splits[e] > 1) {
      slot_base[e] = static_cast<int32_t>(sb);
      counter_base[e] = static_cast<int32_t>(cb);
      sb += int64_t(T) * splits[e];
      cb += T;
    } else {
      slot_base[e] = -1;
      counter_base[e] = -1;
    }
  }

  // 8. split-tile arrival counters start at zero every call
  for (int64_t i = tid; i < cnt_total * EPI_COUNTERS * halves; i += blockDim.x) counters[i] = 0;

  if (tid == 0) {
    hdr->error = 0;
    hdr->total_items = static_cast<int32_t>(total_items);
    hdr->chunk_kiters = static_cast<int32_t>(C > 0x7fffffff ? 0x7fffffff : C);
    hdr->slots_used = static_cast<int32_t>(slots_total);
    hdr->counters_used = static_cast<int32_t>(cnt_total);
    hdr->item_counter = 0;
    hdr->general_scales = 0;
    if (p.status_dev) *p.status_dev = KGW_OK;
  }
}

// Schedule of the M-grouped GEMM ("05 · Grouped GEMM 与 Expert 计算", section 2.1: rows of A are
// grouped by expert, each group aligned to the 128-row tile and multiplied by its own B): validate
// the cumulative row offsets and lay out the work items group by group.
// M-grouped plan: turns the device-side group description into the tile table (one entry per
// 128-row tile: its first row in A/D, its group and its valid rows) and the item count
// (tiles x n-tiles). Contiguous layouts check that no tile spans two groups; masked checks
// 0 <= masked_m[g] <= max_m. Any violation: KGW_ERR_OFFSETS and no items.
__global__ void __launch_bounds__(PLAN_THREADS) plan_mgrouped_kernel(const __grid_constant__ PlanParams p) {
  __shared__ int64_t s_warp[32];
  __shared__ int32_t s_err;
  __shared__ int32_t s_cnt[MAX_EXPERTS];   // CTA pairs: tiles per group
  __shared__ int32_t s_fill[MAX_EXPERTS];  // CTA pairs: next half-row slot of each group
  pdl_launch_dependents();
  const int G = p.E;
  const int tid = threadIdx.x;
  const int NT = p.I / BN;
  const int32_t* grp = p.offsets;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  int2* tiles = reinterpret_cast<int2*>(p.ws + p.L.item_prefix);
  int32_t* rows_out = reinterpret_cast<int32_t*>(p.ws + p.L.order);   // int4 work rows
  if (tid == 0) s_err = 0;
  __syncthreads();
  int64_t ntiles = 0;
  if (p.mg_layout == KGW_MG_OFFSETS) {
    for (int g = tid; g < G; g += blockDim.x) {
      const int64_t prev = g ? static_cast<int64_t>(grp[g - 1]) : 0;
      const int64_t cur = grp[g];
      if (cur < prev || ((cur - prev) % BM) != 0 || (g == G - 1 && cur != p.mg_m)) atomicExch(&s_err, 1);
    }
    __syncthreads();
    ntiles = p.mg_m / BM;
    if (!s_err) {
      for (int64_t t = tid; t < ntiles; t += blockDim.x) {
        const int64_t r0 = t * BM;
        int lo = 0, hi = G - 1;  // first g with offsets[g] > r0 (exists: offsets[G-1] = m > r0)
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (static_cast<int64_t>(grp[mid]) > r0) hi = mid; else lo = mid + 1;
        }
        tiles[t] = make_int2(static_cast<int32_t>(r0), lo | (BM << 16));
      }
    }
  } else if (p.mg_layout == KGW_MG_INDICES) {
    ntiles = p.mg_m / BM;
#pragma unroll 4
    for (int64_t i = tid; i < p.mg_m; i += blockDim.x) {
      const int32_t g = grp[i];
      const int32_t head = grp[i & ~int64_t(BM - 1)];
      if (g != head || g < 0 || g >= G) atomicExch(&s_err, 1);
      if ((i & (BM - 1)) == 0) tiles[i / BM] = make_int2(static_cast<int32_t>(i), g | (BM << 16));
    }
    __syncthreads();
  } else {
    // masked: group g's valid rows masked_m[g] start at row g * max_m; ceil(masked_m / 128) tiles
    const Chunk ch = my_chunk(G);
    int64_t mine = 0;
    for (int g = ch.lo; g < ch.hi; ++g) {
      const int32_t c = grp[g];
      if (c < 0 || c > p.mg_m) {
        atomicExch(&s_err, 1);
      } else {
        mine += (c + BM - 1) / BM;
      }
    }
    int64_t run = block_exclusive_scan(mine, s_warp, &ntiles);
    if (!s_err) {
      for (int g = ch.lo; g < ch.hi; ++g) {
        const int32_t c = grp[g];
        for (int t = 0; t * BM < c; ++t, ++run) {
          const int rows = c - t * BM < BM ? c - t * BM : BM;
          tiles[run] = make_int2(static_cast<int32_t>(g * p.mg_m + int64_t(t) * BM), g | (rows << 16));
        }
      }
    }
  }
  __syncthreads();
  // work rows: one tile each, or (CTA pairs) two tiles of the same group each; a group with an odd
  // tile count gets a last row whose second half repeats the first with no valid rows (its
  // results are not stored)
  int64_t nrows = ntiles;
  if (!s_err) {
    if (!p.mg_pair) {
      for (int64_t t = tid; t < ntiles; t += blockDim.x) {
        const int2 tl = tiles[t];
        reinterpret_cast<int4*>(rows_out)[t] = make_int4(tl.x, tl.x, tl.y & 0xFFFF, static_cast<int>(tl.y >> 16));
      }
    } else {
      for (int g = tid; g < G; g += blockDim.x) s_cnt[g] = 0;
      __syncthreads();
      for (int64_t t = tid; t < ntiles; t += blockDim.x) atomicAdd(&s_cnt[tiles[t].y & 0xFFFF], 1);
      __syncthreads();
      const Chunk ch = my_chunk(G);
      int64_t mine = 0;
      for (int g = ch.lo; g < ch.hi; ++g) mine += (s_cnt[g] + 1) / 2;
      int64_t run = block_exclusive_scan(mine, s_warp, &nrows);
      for (int g = ch.lo; g < ch.hi; ++g) {
        s_fill[g] = static_cast<int32_t>(2 * run);   // half-row slots of group g start at 2 * its first row
        run += (s_cnt[g] + 1) / 2;
      }
      for (int64_t r = tid; r < nrows; r += blockDim.x) rows_out[4 * r + 3] = 0;
      __syncthreads();
      for (int64_t t = tid; t < ntiles; t += blockDim.x) {
        const int2 tl = tiles[t];
        const int g = tl.y & 0xFFFF;
        const int h = atomicAdd(&s_fill[g], 1);
        const int64_t r = h >> 1;
        const int vrows = static_cast<int>(static_cast<uint32_t>(tl.y) >> 16);
        if ((h & 1) == 0) {
          rows_out[4 * r + 0] = tl.x;
          rows_out[4 * r + 2] = g;
          atomicOr(&rows_out[4 * r + 3], vrows);
        } else {
          rows_out[4 * r + 1] = tl.x;
          atomicOr(&rows_out[4 * r + 3], vrows << 16);
        }
      }
      __syncthreads();
      for (int g = tid; g < G; g += blockDim.x)
        if (s_fill[g] & 1) {  // odd tile count: the last row's second half repeats the first, no rows valid
          const int64_t r = (s_fill[g] - 1) >> 1;
          rows_out[4 * r + 1] = rows_out[4 * r + 0];
        }
    }
  }
  __syncthreads();
  if (tid == 0) {
    const int32_t err = s_err ? KGW_ERR_OFFSETS : KGW_OK;
    hdr->error = err;
    hdr->total_items = err ? 0 : static_cast<int32_t>(nrows * NT);
    hdr->chunk_kiters = 0;
    hdr->slots_used = 0;
    hdr->counters_used = 0;
    hdr->item_counter = 0;
    if (p.status_dev) *p.status_dev = err;
  }
}

// =============================================================================================
// Main kernel
// =============================================================================================

// A decoded work item. The scheduler warp decodes each item once and publishes it in the shared-
// memory work ring (and, in a pair, in the peer CTA's ring); e < 0 ends the stream.
struct alignas(16) Item {
  int e;
  int m0, n0;
  int kbeg, kend;        // k-iterations (relative to the expert's first token)
  int split, nsplit, tile;
  int rows;              // valid rows of the tile (M-grouped masked layout: may be < 128)
  int m1, rows1;         // M-grouped CTA pair: first row and valid rows of the second CTA's half
  int srow;              // block-scaled: scale row of the expert's first 128-token block
  int64_t begin;         // expert's first token
  int64_t n_e;           // expert's token count
};
static_assert(sizeof(Item) == 64, "an item is four 16-byte words");

template <bool kMG = false>
__device__ __forceinline__ Item decode_item(const MainParams& p, int idx, int bk) {
  Item it;
  if constexpr (kMG) {
    // M-grouped: item = (128-row tile, n-tile); the tile table gives the rows and the group
    const int mt = idx / p.num_n_tiles;
    const int nt = idx - mt * p.num_n_tiles;
    const int4 wr = __ldg(reinterpret_cast<const int4*>(p.ws + p.L.order) + mt);
    it.m0 = wr.x;
    it.m1 = wr.y;
    it.e = wr.z;
    it.rows = wr.w & 0xFFFF;
    it.rows1 = static_cast<int>(static_cast<uint32_t>(wr.w) >> 16);
    it.n0 = nt * BN;
    it.split = 0;
    it.nsplit = 1;
    it.tile = idx;
    it.kbeg = 0;
    it.kend = p.K / bk;
    it.srow = 0;
    it.begin = 0;
    it.n_e = 0;
    return it;
  }
  const int32_t* order = reinterpret_cast<const int32_t*>(p.ws + p.L.order);
  const int32_t* prefix = reinterpret_cast<const int32_t*>(p.ws + p.L.item_prefix);
  const int32_t* splits = reinterpret_cast<const int32_t*>(p.ws + p.L.splits);
  int lo = 0, hi = p.E;  // largest q with prefix[q] <= idx
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(prefix + mid) <= idx) lo = mid; else hi = mid;
  }
  it.e = __ldg(order + lo);
  const int local = idx - __ldg(prefix + lo);
  it.rows = p.tile_m;
  it.m1 = 0;
  it.rows1 = 0;
  it.nsplit = __ldg(splits + it.e);
  const int T = p.num_m_tiles * p.num_n_tiles;
  it.split = local / T;
  it.tile = local - it.split * T;
  const int mt = it.tile / p.num_n_tiles;
  const int nt = it.tile - mt * p.num_n_tiles;
  it.m0 = mt * p.tile_m;
  it.n0 = nt * BN;
  it.begin = it.e ? static_cast<int64_t>(__ldg(p.offsets + it.e - 1)) : 0;
  it.n_e = static_cast<int64_t>(__ldg(p.offsets + it.e)) - it.begin;
  it.srow = __ldg(reinterpret_cast<const int32_t*>(p.ws + p.L.scale_row) + it.e);
  const int64_t kit = (it.n_e + bk - 1) / bk;  // a partial last stage counts (zero-filled tail)
  it.kbeg = static_cast<int>(it.split * kit / it.nsplit);
  it.kend = static_cast<int>((it.split + 1) * kit / it.nsplit);
  return it;
}

// K-grouped item idx, decoded by a whole warp (every lane returns the item decode_item gives).
// The item lies in the largest ordered expert position q with prefix[q] <= idx. A warp's claims only
// grow, so q is at or after the position of its previous item (lo_hint, updated here): one 32-wide
// window of the prefix sums and a ballot find it (the window slides only past 31 experts;
// prefix[E], the item total, exceeds every idx). Then the expert's index, and its split count,
// token range and first scale row in parallel: three rounds of global loads instead of a dozen
// dependent ones.
__device__ __forceinline__ Item decode_item_warp(const MainParams& p, int idx, int bk, int& lo_hint, int lane) {
  const int32_t* order = reinterpret_cast<const int32_t*>(p.ws + p.L.order);
  const int32_t* prefix = reinterpret_cast<const int32_t*>(p.ws + p.L.item_prefix);
  const int32_t* splits = reinterpret_cast<const int32_t*>(p.ws + p.L.splits);
  const int32_t* scale_row = reinterpret_cast<const int32_t*>(p.ws + p.L.scale_row);
  int lo = lo_hint;
  int base = 0;
  for (;;) {
    const int q = lo + lane;
    const int v = q <= p.E ? __ldg(prefix + q) : INT_MAX;
    const int cnt = __popc(__ballot_sync(0xffffffffu, v <= idx));  // lanes 0..cnt-1 (prefix is non-decreasing)
    if (cnt < 32) {
      base = __shfl_sync(0xffffffffu, v, cnt - 1);
      lo += cnt - 1;
      break;
    }
    lo += 31;
  }
  lo_hint = lo;
  Item it;
  it.e = __ldg(order + lo);
  int32_t w = 0;
  if (lane == 0) w = __ldg(splits + it.e);
  if (lane == 1) w = it.e ? __ldg(p.offsets + it.e - 1) : 0;
  if (lane == 2) w = __ldg(p.offsets + it.e);
  if (lane == 3) w = __ldg(scale_row + it.e);
  it.nsplit = __shfl_sync(0xffffffffu, w, 0);
  it.begin = static_cast<int64_t>(__shfl_sync(0xffffffffu, w, 1));
  it.n_e = static_cast<int64_t>(__shfl_sync(0xffffffffu, w, 2)) - it.begin;
  it.srow = __shfl_sync(0xffffffffu, w, 3);
  const int local = idx - base;
  it.rows = p.tile_m;
  it.m1 = 0;
  it.rows1 = 0;
  const int T = p.num_m_tiles * p.num_n_tiles;
  it.split = local / T;
  it.tile = local - it.split * T;
  const int mt = it.tile / p.num_n_tiles;
  const int nt = it.tile - mt * p.num_n_tiles;
  it.m0 = mt * p.tile_m;
  it.n0 = nt * BN;
  const int64_t kit = (it.n_e + bk - 1) / bk;  // a partial last stage counts (zero-filled tail)
  it.kbeg = static_cast<int>(it.split * kit / it.nsplit);
  it.kend = static_cast<int>((it.split + 1) * kit / it.nsplit);
  return it;
}

struct SmemCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t wfull[WORK_RING];
  uint64_t wempty[WORK_RING];
  uint64_t mma_done;
  uint64_t sf_full[MAX_STAGES]; // block-scaled: single CTA, the converter has written a stage's scale
                                // factors in TMEM order; pair, warp 10 has copied them to TMEM once
                                // they landed (on the even CTA)
  uint64_t sfdata[MAX_STAGES];  // block-scaled: this CTA's raw scales of a stage have landed in shared memory;
                                // CTA pair: both CTAs' prepared scale factors of a stage (even CTA)
  uint64_t cp_done;             // CTA pair: warp 10's last scale-factor copies have completed
  Item work[WORK_RING];         // decoded work items (written by the scheduler of the leader CTA)
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t items_started;        // items the producer (of the leader CTA) has started
};

// Epilogue staging: 16 KiB per CTA, split over its epilogue warps (4 x 32 rows x 32 FP32, or in the
// block-scaled kernels 8 x 32 rows x 16 FP32 / 32 16-bit values).
constexpr uint32_t EPI_STAGE_TOTAL = 16384;
constexpr uint32_t EPI_STAGE_BYTES = EPI_STAGE_TOTAL / NUM_EPI_WARPS;

size_t main_smem_bytes(bool pair, bool fp8, bool nv, bool fp4, bool wide_k) {
  if (pair && fp4 && wide_k)  // fills shared memory: no alignment slack (the kernel checks the base)
    return size_t(STAGES_PAIR_FP4_WIDE) * (2 * STAGE_A_BYTES + STAGE_B_BYTES + SF_SMEM_PAD_PAIR_FP4_WIDE) +
           EPI_STAGE_TOTAL + sizeof(SmemCtl) + 64;
  const size_t ring = pair && wide_k ? size_t(STAGES_PAIR_BF16) * (2 * STAGE_A_BYTES + STAGE_B_BYTES)
                      : pair && nv ? size_t(STAGES_PAIR_NV) * (STAGE_A_BYTES + STAGE_B_BYTES / 2 + SF_SMEM_PAD_PAIR_NV)
                      : pair ? (fp4 ? size_t(STAGES_PAIR_FP4) * (STAGE_A_BYTES + STAGE_B_BYTES / 2 + SF_SMEM_PAD_PAIR_FP4)
                                  : size_t(STAGES_PAIR) * (STAGE_A_BYTES + STAGE_B_BYTES / 2 + (fp8 ? SF_SMEM_PAD_PAIR : 0u)))
                      : nv ? size_t(STAGES_NV) * (STAGE_BYTES + SF_SMEM_PAD_NV)
                           : size_t(STAGES) * (STAGE_BYTES + (fp8 ? SF_SMEM_PAD : 0u));
  return ring + EPI_STAGE_TOTAL + 1024 /* alignment slack */ + sizeof(SmemCtl) + 64;
}

// Bit 7 of every byte of w that equals 0xFF (the UE8M0 NaN encoding), branch-free: (b & 0x7F) + 1
// reaches 0x80 exactly when the low seven bits are all ones, and no carry crosses a byte.
__device__ __forceinline__ uint32_t ff_bytes(uint32_t w) {
  return ((w & 0x7F7F7F7Fu) + 0x01010101u) & w & 0x80808080u;
}

// UE8M0 scale-factor byte of a power-of-two FP32 scale, replicated to the 4 bytes of a TMEM
// column (one byte per 32-token block of the 128-token scale block). Flags non-powers of two.
__device__ __forceinline__ uint32_t ue8m0_x4(float s, bool& bad) {
  const uint32_t b = __float_as_uint(s);
  uint32_t e = (b >> 23) & 0xFFu;
  const uint32_t m = b & 0x7FFFFFu;
  if ((b >> 31) != 0u || e == 255u) bad = true;
  if (e == 0u) {
    if (m != 0x400000u) bad = true;  // only 2^-127 is representable below the normal range
  } else if (m != 0u) {
    bad = true;
  }
  return e * 0x01010101u;
}

// Wait without the abort short-cut (used only while draining at the end).
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  int dummy = 0;
  return wait_bounded(bar, parity, &dummy, timeout_ns);
}

// ---------------------------------------------------------------------------------------------
// Epilogue helpers. A warp owns 32 rows of the tile. Values come out of TMEM one row per thread;
// they are staged through a per-warp 32 x 128-byte shared buffer (16-byte chunks XOR-swizzled by
// row, so both the row-per-thread writes and the read-back are free of bank conflicts) and
// written back four rows per instruction: 8 lanes cover 32 consecutive FP32 columns of one row.
// ---------------------------------------------------------------------------------------------

// Previous contents of 4 consecutive outputs (accumulate mode) as raw bits (FP32: 4 words;
// BF16: 2 words), loaded ahead of the arithmetic so several loads are in flight together.
__device__ __forceinline__ uint4 load_old4(const MainParams& p, const char* src) {
  if (!p.out_bf16) return *reinterpret_cast<const uint4*>(src);
  const uint2 h = *reinterpret_cast<const uint2*>(src);
  return make_uint4(h.x, h.y, 0u, 0u);
}

// Write 4 consecutive output values (FP32 accumulator values v) at dst: overwrite, or add the
// previous contents (one FP32 add, then one rounding to the output type: FP32, BF16 or FP16).
__device__ __forceinline__ void emit4(const MainParams& p, char* dst, float4 v, const uint4& o) {
  if (!p.out_bf16) {
    if (p.accumulate) {
      v.x += __uint_as_float(o.x);
      v.y += __uint_as_float(o.y);
      v.z += __uint_as_float(o.z);
      v.w += __uint_as_float(o.w);
    }
    *reinterpret_cast<float4*>(dst) = v;
  } else if (!p.out_f16) {
    if (p.accumulate) {
      v.x += bf16_lo(o.x);
      v.y += bf16_hi(o.x);
      v.z += bf16_lo(o.y);
      v.w += bf16_hi(o.y);
    }
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  } else {
    if (p.accumulate) {
      v.x += f16_lo(o.x);
      v.y += f16_hi(o.x);
      v.z += f16_lo(o.y);
      v.w += f16_hi(o.y);
    }
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_f16x2(v.x, v.y), pack_f16x2(v.z, v.w));
  }
}

// Stage this thread's 32 values (row `lane` of the warp's 32 rows) into the swizzled buffer.
__device__ __forceinline__ void stage_row(uint4* stg, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    stg[lane * 8 + (c ^ (lane & 7))] = make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
}

// Read back 4 columns of row (4j + lane/8), chunk lane%8, from the swizzled buffer.
__device__ __forceinline__ float4 unstage(const uint4* stg, int j, int lane) {
  const int r = 4 * j + (lane >> 3);
  const int c = lane & 7;
  const uint4 u = stg[r * 8 + (c ^ (r & 7))];
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

template <bool kMG = false>
__device__ __forceinline__ char* out_row_ptr(const MainParams& p, const Item& it, int row) {
  const size_t esz = p.out_bf16 ? 2 : 4;
  if constexpr (kMG) {  // D [rows, N]; rows at or past BM belong to the second half of a CTA pair
    const size_t rr = static_cast<size_t>(row >= BM ? it.m1 + (row - BM) : it.m0 + row);
    return reinterpret_cast<char*>(p.out) + (rr * p.I + it.n0) * esz;
  }
  const size_t r = static_cast<size_t>(it.m0 + row);
  if (p.discrete) {
    char* base = reinterpret_cast<char*>(static_cast<uintptr_t>(__ldg(p.out_ptrs + it.e)));
    return base + (r * p.I + it.n0) * esz;
  }
  return reinterpret_cast<char*>(p.out) + ((static_cast<size_t>(it.e) * p.H + r) * p.I + it.n0) * esz;
}

// =============================================================================================
// FP8 with general FP32 scales
// =============================================================================================

// Scale kernel of the K-grouped FP8 entries, between the plan and the FP8 kernel. It reads every
// scale of the call once (the plan's scale rows x hidden / intermediate):
//  - FP32 scales: a scale that is not a positive power of two UE8M0 can hold sets general_scales
//    (the FP8 kernel then takes its promotion path); a NaN or infinite scale is KGW_ERR_SCALES;
//  - packed UE8M0 words: a byte 0xFF (NaN) is KGW_ERR_SCALES;
//  - block-scaled calls on CTA pairs (p.sf_prep): writes the scale factors in TMEM order into the
//    workspace, so that a pair stage loads them by TMA: within each group of 128 rows (columns),
//    word 4l + c holds row 32c + l, the FP32 scale's exponent byte repeated four times or the
//    packed word (UE8M0; NVFP4: UE4M3, two 64-token word rows per 128-token block, each byte
//    checked for a set top bit or the NaN code 0x7F).
// One work unit is such a 4-word group entry: four coalesced loads (32 rows apart), one 16-byte store.
__global__ void __launch_bounds__(256) scale_check_kernel(const __grid_constant__ MainParams p) {
  pdl_launch_dependents();
  pdl_wait();
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws);
  if (hdr->error != 0) return;
  // (NVFP4: two 64-token word rows per 128-token scale block)
  const int64_t rows = int64_t(hdr->scale_rows) * (p.nvfp4 ? 2 : 1);
  const int64_t ua = rows * (p.H / 4), ub = rows * (p.I / 4);
  const uint32_t* sa = reinterpret_cast<const uint32_t*>(p.sfa);
  const uint32_t* sb = reinterpret_cast<const uint32_t*>(p.sfb);
  uint32_t* pa = reinterpret_cast<uint32_t*>(p.ws + p.L.sf_prep_a);
  uint32_t* pb = reinterpret_cast<uint32_t*>(p.ws + p.L.sf_prep_b);
  uint32_t general = 0, bad = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < ua + ub; u += stride) {
    const bool is_a = u < ua;
    const int64_t v = is_a ? u : u - ua;
    const int64_t cols = is_a ? p.H : p.I;
    const int64_t kb = v / (cols / 4);
    const int64_t rem = v - kb * (cols / 4);
    const int64_t g = rem >> 5, l = rem & 31;
    const uint32_t* src = (is_a ? sa : sb) + kb * cols + g * 128 + l;
    uint32_t w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) w[c] = __ldg(src + 32 * c);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (p.nvfp4) {   // UE4M3: no byte with its top bit set, none equal to 0x7F (NaN)
        bad |= (w[c] & 0x80808080u) | (((w[c] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u);
      } else if (p.sf_packed) {
        bad |= ff_bytes(w[c]);
      } else {
        const uint32_t e = (w[c] >> 23) & 0xFFu, m = w[c] & 0x7FFFFFu;
        bad |= e == 255u;
        general |= (e != 255u) & (((w[c] >> 31) != 0u) | (e == 0u ? m != 0x400000u : m != 0u));
        w[c] = e * 0x01010101u;     // the UE8M0 byte of a power of two, one per 32-token block
      }
    }
    if (p.sf_prep)
      *reinterpret_cast<uint4*>((is_a ? pa : pb) + kb * cols + g * 128 + 4 * l) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (__any_sync(0xffffffffu, general) && (threadIdx.x & 31) == 0) atomicOr(&hdr->general_scales, 1);
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && p.status_dev) atomicExch(p.status_dev, KGW_ERR_SCALES);
}

// Promotion path: FP8 (e4m3) K-grouped wgrad with arbitrary FP32 scales per 128-token block
// ("05 · Grouped GEMM 与 Expert 计算", section 3: x_scales float, per-block 1x128 scaling). A scale
// that is not a power of two cannot be folded into the block-scaled MMA exactly, so each block's
// unscaled partial sum P = sum over its 128 tokens of a*b runs on the tensor cores
// (tcgen05.mma kind::f8f6f4, FP32 in TMEM) and eight warps add sa[m]*sb[n]*P to FP32 running sums
// held in registers: the per-block promotion of the pages' FP8 GEMMs. Tiles are 128 x 128 (two
// per 128 x 256 plan item, so the running sums fit the registers) with P double-buffered in TMEM;
// the stage ring is the block-scaled kernel's (A 128 rows, B the 256-column box of K-major B or
// the tile's 128 columns of N-major B, and the block's 128 + 128 scales). Split-K items of the plan
// are merged: split 0 covers the expert's whole token range, the others are skipped.
// Roles: warp 0 TMA producer, warp 1 MMA + TMEM owner, warps 2..9 promotion and output, warp 11
// scheduler (warp 10 idle).
constexpr int PR_TN = 128;
constexpr int PR_STAGES = 4;
constexpr uint32_t PR_SF_BYTES = 1024;                        // 128 FP32 of A + 128 FP32 of B
constexpr uint32_t PR_STAGE_BYTES = STAGE_A_BYTES + STAGE_B_BYTES + PR_SF_BYTES;   // 49 KiB
constexpr int PR_WARPS = 8;

struct PromoteCtl {
  uint64_t full[PR_STAGES];
  uint64_t empty[PR_STAGES];
  uint64_t pfull[2];
  uint64_t pempty[2];
  uint64_t wfull[WORK_RING];
  uint64_t wempty[WORK_RING];
  uint64_t sched_go;
  uint64_t mma_done;
  Item work[WORK_RING];
  uint32_t tmem_base;
  int32_t abort_flag;
};

size_t promote_smem_bytes() { return size_t(PR_STAGES) * PR_STAGE_BYTES + EPI_STAGE_TOTAL + 1024 + sizeof(PromoteCtl) + 64; }

// Runs inside the FP8 kernel (same launch, same dynamic shared memory, which is at least
// promote_smem_bytes()) once the scale check has found a scale that is not a power of two.
template <bool kAK, bool kBK>
__device__ __forceinline__ void promote_body(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                             uint8_t* smem_raw) {
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(p.ws);
  // 128 x 128 sub-tiles of the plan's items: two column halves, and two row halves when the plan
  // laid out 256-row CTA-pair tiles
  const int subs = 2 * (p.tile_m / BM);
  const int total_items = subs * hdr->total_items;
  // K-major B descriptors of CTA-pair plans have 128-row boxes (this sub-tile's columns), those of
  // single-CTA plans 256-row boxes (both halves; the MMA reads this half's)
  const bool half_box = p.tile_m == 2 * BM;
  if (total_items == 0) return;
  constexpr int bk = BK_FP8;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_mem = base;
  uint8_t* epi_stage_mem = base + size_t(PR_STAGES) * PR_STAGE_BYTES;
  PromoteCtl* ctl = reinterpret_cast<PromoteCtl*>(epi_stage_mem + EPI_STAGE_TOTAL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* item_counter = const_cast<int32_t*>(&hdr->item_counter);
  volatile int* abort_flag = &ctl->abort_flag;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PR_STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1 + PR_WARPS);   // the MMA commit and every promotion warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->pfull[b], 1);
      mbar_init(&ctl->pempty[b], PR_WARPS);
    }
    for (int w = 0; w < WORK_RING; ++w) {
      mbar_init(&ctl->wfull[w], 1);
      mbar_init(&ctl->wempty[w], 2 + PR_WARPS);    // producer, MMA thread, promotion warps
    }
    mbar_init(&ctl->sched_go, 1);
    mbar_init(&ctl->mma_done, 1);
    ctl->abort_flag = 0;
    fence_mbarrier_init();
    if (p.tokens_sum > 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
    }
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // expert k-iterations of a split-0 item (the whole expert), 0 for the other splits
  auto kiters = [&](const Item& it) { return it.split > 0 ? 0 : static_cast<int>((it.n_e + bk - 1) / bk); };
  auto read_item = [&](int n, Item& it) {
    const int slot = n % WORK_RING;
    const bool ok = wait_bounded(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns);
    it = ctl->work[slot];
    return ok;
  };

  if (warp == 0) {
    // ======================= TMA producer =======================
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    for (int n = 0;; ++n) {
      Item it;
      const bool okw = read_item(n, it);
      if (!__all_sync(0xffffffffu, okw)) break;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->wempty[n % WORK_RING]);
        if (it.e >= 0) mbar_arrive(&ctl->sched_go);
      }
      if (it.e < 0) break;
      const int kit = kiters(it);
      const CUtensorMap* amap = &tmA;
      const CUtensorMap* bmap = &tmB;
      if ((kAK && p.ragged) || p.tail_a) {
        amap = reinterpret_cast<const CUtensorMap*>(p.ws + p.L.tmaps + size_t(it.e) * 128);
        if (lane == 0 && kit > 0) fence_tmap_acquire(amap);
      }
      if ((kBK && p.ragged) || p.tail_b) {
        bmap = reinterpret_cast<const CUtensorMap*>(p.ws + p.L.tmaps_b + size_t(it.e) * 128);
        if (lane == 0 && kit > 0) fence_tmap_acquire(bmap);
      }
      const int n0_tile = it.n0 - it.m1 * PR_TN;   // the plan item's 256-column tile
      for (int kb = 0; kb < kit; ++kb) {
        bool ok2 = true;
        if (lane == 0) {
          ok2 = wait_bounded(&ctl->empty[stage], phase ^ 1, abort_flag, p.timeout_ns);
          if (ok2)
            mbar_arrive_expect_tx(&ctl->full[stage],
                                  STAGE_A_BYTES + (kBK && !half_box ? STAGE_B_BYTES : STAGE_B_BYTES / 2) + PR_SF_BYTES);
        }
        ok2 = __shfl_sync(0xffffffffu, ok2, 0);
        if (!ok2) break;
        uint8_t* sA = stage_mem + size_t(stage) * PR_STAGE_BYTES;
        uint8_t* sB = sA + STAGE_A_BYTES;
        uint8_t* sS = sB + STAGE_B_BYTES;
        const int64_t tok = it.begin + int64_t(kb) * bk;
        if (lane == 0) {
          const int64_t kblk = int64_t(it.srow) + kb;   // the expert's block kb
          bulk_load(sS, p.sfa + kblk * p.H + it.m0, BM * 4, &ctl->full[stage]);
          bulk_load(sS + BM * 4, p.sfb + kblk * p.I + it.n0, PR_TN * 4, &ctl->full[stage]);
          const int32_t kx = p.ragged ? kb * bk : static_cast<int32_t>(tok);
          if constexpr (kAK) tma_load_2d(sA, amap, &ctl->full[stage], kx, it.m0);
          else tma_load_2d(sA, amap, &ctl->full[stage], it.m0, static_cast<int32_t>(tok));
          // K-major B: the plan tile's 256-row box (the MMA reads this half's 128 rows);
          // N-major B: this half's 128 columns (one 128-byte atom)
          if constexpr (kBK) tma_load_2d(sB, bmap, &ctl->full[stage], kx, half_box ? it.n0 : n0_tile);
          else tma_load_2d(sB, bmap, &ctl->full[stage], it.n0, static_cast<int32_t>(tok));
        }
        ++issued;
        if (++stage == PR_STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
    }
    if (lane == 0) {  // the last stages land before exit
      int s = stage;
      uint32_t ph = phase;
      for (int i = 0; i < PR_STAGES && i < issued; ++i) {
        if (--s < 0) {
          s = PR_STAGES - 1;
          ph ^= 1;
        }
        int dummy = 0;
        wait_bounded(&ctl->full[s], ph, &dummy, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t blk = 0;
      constexpr uint32_t a_mn = kAK ? 0u : 1u, b_mn = kBK ? 0u : 1u;
      const uint32_t idesc = idesc_f8f6f4(BM, PR_TN, a_mn, b_mn);
      const uint64_t a_tmpl = kAK ? sdesc_sw128(0, 16, 1024) : sdesc_sw128(0, uint32_t(bk) * 128u, 1024);
      const uint64_t b_tmpl = kBK ? sdesc_sw128(0, 16, 1024) : sdesc_sw128(0, uint32_t(bk) * 128u, 1024);
      constexpr uint32_t a_step = (kAK ? 32u : 4096u) >> 4;
      constexpr uint32_t b_step = (kBK ? 32u : 4096u) >> 4;
      auto desc = [](uint64_t tmpl, uint32_t addr, uint32_t step, int k) {
        return tmpl + static_cast<uint64_t>(((addr & 0x3FFFFu) >> 4) + k * step);
      };
      for (int n = 0;; ++n) {
        Item it;
        if (!read_item(n, it)) break;
        mbar_arrive(&ctl->wempty[n % WORK_RING]);
        if (it.e < 0) break;
        const int kit = kiters(it);
        bool ok = true;
        for (int kb = 0; kb < kit; ++kb, ++blk) {
          const uint32_t pb = blk & 1;
          if (!wait_bounded(&ctl->pempty[pb], ((blk >> 1) & 1) ^ 1, abort_flag, p.timeout_ns) ||
              !wait_bounded(&ctl->full[stage], phase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_mem + size_t(stage) * PR_STAGE_BYTES);
          const uint32_t b_addr =
              a_addr + STAGE_A_BYTES + (kBK && !half_box ? static_cast<uint32_t>(it.m1) * (STAGE_B_BYTES / 2) : 0u);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8f6f4(tmem_base + pb * PR_TN, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k), idesc,
                       k > 0 ? 1u : 0u);
          mma_commit(&ctl->empty[stage]);
          mma_commit(&ctl->pfull[pb]);
          if (++stage == PR_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      mma_commit(&ctl->mma_done);
      int dummy = 0;
      wait_bounded(&ctl->mma_done, 0, &dummy, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + PR_WARPS) {
    // ======================= promotion and output (warps 2..9) =======================
    const int q = warp & 3;                    // TMEM lane quadrant: rows 32q .. 32q+31
    const int h = (warp - EPI_WARP0) >> 2;     // columns 64h .. 64h+63 of the 128-column tile
    const int row = q * 32 + lane;
    uint4* stg = reinterpret_cast<uint4*>(epi_stage_mem + (warp - EPI_WARP0) * (EPI_STAGE_TOTAL / PR_WARPS));
    const int rsub = lane >> 2, csub = lane & 3;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t blk = 0;
    for (int n = 0;; ++n) {
      Item it;
      const bool okw = read_item(n, it);
      if (!__all_sync(0xffffffffu, okw)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->wempty[n % WORK_RING]);
      if (it.e < 0) break;
      if (it.split > 0) continue;
      const int esz = p.out_bf16 ? 2 : 4;
      char* obase = out_row_ptr<false>(p, it, q * 32) + size_t(64 * h) * esz;
      const size_t ostride = size_t(p.I) * esz;
      const int kit = kiters(it);
      if (kit == 0) {  // empty expert, overwrite mode: zeros
#pragma unroll 1
        for (int r = 0; r < 32; ++r)
          for (int off = lane * 16; off < 64 * esz; off += 32 * 16)
            *reinterpret_cast<uint4*>(obase + r * ostride + off) = make_uint4(0, 0, 0, 0);
        continue;
      }
      float R[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) R[j] = 0.f;
      bool ok = true;
      for (int kb = 0; kb < kit; ++kb, ++blk) {
        const uint32_t pb = blk & 1;
        const bool okp = wait_bounded(&ctl->pfull[pb], (blk >> 1) & 1, abort_flag, p.timeout_ns) &&
                         wait_bounded(&ctl->full[stage], phase, abort_flag, p.timeout_ns);  // scales visible
        if (!__all_sync(0xffffffffu, okp)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* sS = reinterpret_cast<const float*>(stage_mem + size_t(stage) * PR_STAGE_BYTES + STAGE_A_BYTES + STAGE_B_BYTES);
        const float sa = sS[row];
        const float4* sb = reinterpret_cast<const float4*>(sS + BM + 64 * h);
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + pb * PR_TN + 64 * h;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t P[32];
          tmem_ld_32x32b_x32(taddr + 32 * c, P);
          tmem_ld_wait();
          if (c == 1) {  // both halves of this warp's partial are in registers: hand P back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->pempty[pb]);
          }
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 b4 = sb[8 * c + j4];
            const int j = 32 * c + 4 * j4;
            R[j] = fmaf(__uint_as_float(P[4 * j4]), sa * b4.x, R[j]);
            R[j + 1] = fmaf(__uint_as_float(P[4 * j4 + 1]), sa * b4.y, R[j + 1]);
            R[j + 2] = fmaf(__uint_as_float(P[4 * j4 + 2]), sa * b4.z, R[j + 2]);
            R[j + 3] = fmaf(__uint_as_float(P[4 * j4 + 3]), sa * b4.w, R[j + 3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->empty[stage]);   // this warp is done with the stage's scales
        if (++stage == PR_STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      // output: 4 rounds of 16 columns through the per-warp staging, 4 lanes per 64-byte row segment
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          stg[lane * 4 + (i ^ sw)] = make_uint4(__float_as_uint(R[16 * c + 4 * i]), __float_as_uint(R[16 * c + 4 * i + 1]),
                                                __float_as_uint(R[16 * c + 4 * i + 2]), __float_as_uint(R[16 * c + 4 * i + 3]));
        __syncwarp();
        char* cbase = obase + size_t(c * 16 + csub * 4) * esz;
        uint4 old[4];
        if (p.accumulate) {
#pragma unroll
          for (int j = 0; j < 4; ++j) old[j] = load_old4(p, cbase + (8 * j + rsub) * ostride);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 8 * j + rsub;
          const uint4 u = stg[r * 4 + (csub ^ ((r >> 1) & 3))];
          emit4(p, cbase + r * ostride,
                make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)), old[j]);
        }
        __syncwarp();
      }
    }
  } else if (warp == SCHED_WARP_FP8) {
    // ======================= scheduler =======================
    // Claims the next sub-tile one ahead of the producer (item subs * i + s is sub-tile s of plan item i).
    if (lane == 0) {
      int cur = atomicAdd(item_counter, 1);
      for (int n = 0;; ++n) {
        const int slot = n % WORK_RING;
        Item it;
        if (cur < total_items) {
          const int sub = cur % subs;
          it = decode_item<false>(p, cur / subs, bk);
          it.m0 += (sub >> 1) * BM;     // the 128-row half of a CTA-pair item
          it.m1 = sub & 1;              // the 128-column half
          it.n0 += (sub & 1) * PR_TN;
        } else {
          it = Item{};
          it.e = -1;
        }
        if (!wait_bounded(&ctl->wempty[slot], ((n / WORK_RING) & 1) ^ 1, abort_flag, p.timeout_ns)) break;
        ctl->work[slot] = it;
        mbar_arrive(&ctl->wfull[slot]);
        if (it.e < 0) break;
        if (!wait_bounded(&ctl->sched_go, n & 1, abort_flag, p.timeout_ns)) break;
        cur = atomicAdd(item_counter, 1);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 256);
  }
  if (threadIdx.x == 0 && ctl->abort_flag && p.status_dev) atomicExch(p.status_dev, KGW_ERR_TIMEOUT);
}

// The promotion path as a kernel of its own, launched before the FP8 CTA-pair kernel of calls with
// FP32 scales: it runs the call when the scale kernel found a scale that is not a power of two and
// otherwise leaves at once (the pair kernel then runs it).
template <bool kAK, bool kBK>
__global__ void __launch_bounds__(NUM_THREADS_FP8, 1)
    promote_kernel(const __grid_constant__ MainParams p, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  pdl_launch_dependents();
  pdl_wait();
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(p.ws);
  if (hdr->error != 0 || !hdr->general_scales || hdr->total_items == 0) return;
  promote_body<kAK, kBK>(p, tmA, tmB, smem_raw);
}

template <bool kAK, bool kBK>
static cudaError_t launch_promote(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                                  cudaStream_t s) {
  auto kernel = promote_kernel<kAK, kBK>;
  const size_t smem = promote_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS_FP8, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, tmA, tmB);
}

cudaError_t launch_promote_kernel(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                                  cudaStream_t s) {
  if (p.a_kmajor && !p.b_kmajor) return launch_promote<true, false>(p, tmA, tmB, grid, s);
  if (!p.a_kmajor && !p.b_kmajor) return launch_promote<false, false>(p, tmA, tmB, grid, s);
  if (p.a_kmajor && p.b_kmajor) return launch_promote<true, true>(p, tmA, tmB, grid, s);
  return launch_promote<false, true>(p, tmA, tmB, grid, s);
}

cudaError_t launch_scale_check(const MainParams& p, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, scale_check_kernel, p);
}

// One persistent kernel, two shapes:
//  - kPair = false: one CTA owns a 128 x 256 output tile (BF16 or FP8).
//  - kPair = true : a cluster of two CTAs owns a 256 x 256 tile (BF16). Each CTA loads its own
//    128 rows of A and 128 columns of B; the even CTA issues tcgen05.mma.cta_group::2, which reads
//    both CTAs' shared memory and writes each CTA's 128 rows into its own TMEM. Per SM this moves
//    32 KiB per k-iteration into shared memory instead of 48 KiB.
// kFp8 selects the block-scaled path (scale-factor converter, one accumulator); kFp4 narrows it
// to e2m1 operands (kind::mxf4, 256 tokens per stage, K-major A and B, UE8M0 words only); kNv
// makes that NVFP4 (kind::mxf4nvf4 scale_vec::4X: UE4M3 scales per 16 tokens, 48 TMEM scale
// columns per stage, 3 stages, per-tensor global scales applied in the epilogue).
template <bool kFp8, bool kPair, bool kAK, bool kBK, bool kMG = false, bool kFp4 = false, bool kNv = false,
          bool kWideK = false>
__global__ void __launch_bounds__(kFp8 ? NUM_THREADS_FP8 : NUM_THREADS, 1)
    wgrad_kernel(const __grid_constant__ MainParams p, const __grid_constant__ CUtensorMap tmA,
                 const __grid_constant__ CUtensorMap tmB) {
  // FP8, FP4 and NVFP4 on CTA pairs: K-grouped, with the scale factors prepared in TMEM order by
  // the scale kernel and loaded by TMA with each stage (the M-grouped FP8 GEMM runs on single CTAs).
  static_assert(!(kFp8 && kPair) || !kMG, "block-scaled CTA pairs: K-grouped only");
  static_assert(!kFp4 || (kFp8 && kAK && kBK && !kMG), "FP4 operands are K-major, block-scaled");
  static_assert(!kNv || kFp4, "NVFP4 is the FP4 kernel with UE4M3 scales");
  // kWideK: stages of two 128-byte rows of K per operand row on CTA pairs: BF16 128-token stages
  // (K-major operands in two 64-token boxes), FP4 512-token stages (two 256-token boxes)
  static_assert(!kWideK || (kPair && (!kFp8 || (kFp4 && !kNv))), "two-row stages: BF16 or FP4 CTA pairs");
  constexpr int kStages = kPair ? (kNv ? STAGES_PAIR_NV
                                   : kFp4 ? (kWideK ? STAGES_PAIR_FP4_WIDE : STAGES_PAIR_FP4)
                                   : kWideK ? STAGES_PAIR_BF16 : STAGES_PAIR)
                                : (kNv ? STAGES_NV : STAGES);
  constexpr uint32_t kStageA = STAGE_A_BYTES * (kWideK ? 2 : 1);
  constexpr uint32_t kStageB = (kPair ? STAGE_B_BYTES / 2 : STAGE_B_BYTES) * (kWideK ? 2 : 1);
  constexpr uint32_t kSfPad = kNv ? (kPair ? SF_SMEM_PAD_PAIR_NV : SF_SMEM_PAD_NV)
                              : !kFp8 ? 0u
                              : kPair ? (kFp4 ? (kWideK ? SF_SMEM_PAD_PAIR_FP4_WIDE : SF_SMEM_PAD_PAIR_FP4) : SF_SMEM_PAD_PAIR)
                                      : SF_SMEM_PAD;
  constexpr uint32_t kStageBytes = kStageA + kStageB + kSfPad;
  // Block-scaled CTA pairs: the prepared scale factors of a stage land on their own barrier (sfdata
  // of the even CTA), ahead of the operands, so warp 10 copies them to TMEM while the operand tiles
  // are still arriving; `full` counts the operand bytes only.
  constexpr uint32_t kStageTx = kStageA + kStageB;
  constexpr uint32_t kExpectTx = kPair ? 2 * kStageTx : kStageTx;
  constexpr uint32_t kSfTx =
      kFp8 && kPair ? (kNv ? SF_PAIR_BYTES_NV : kFp4 ? (kWideK ? SF_PAIR_BYTES_FP4_WIDE : SF_PAIR_BYTES_FP4) : SF_PAIR_BYTES)
                    : 0u;
  constexpr int kHalves = kPair ? 2 : 1;
  constexpr int kEpiWarps = kFp8 ? NUM_EPI_WARPS_FP8 : NUM_EPI_WARPS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];  // (the 512-token FP4 ring relies on it)
  const int bk = kFp4 ? (kWideK ? BK_FP4_PAIR : BK_FP4) : (kFp8 ? BK_FP8 : (kWideK ? BK_BF16_PAIR : BK_BF16));
  pdl_wait();  // the plan of this call (and any scale check before it) is complete and visible
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(p.ws);
  if (hdr->error != 0) return;  // offsets/pointers rejected by the plan: write nothing
  if constexpr (kFp8 && !kFp4 && !kMG) {
    // FP32 scales of which some is not a power of two: the per-block promotion path runs the call

    if (p.general_dispatch && hdr->general_scales) {
      // (a kernel may not mix single-CTA and CTA-pair tcgen05 instructions: for pairs the
      // promotion kernel launched before this one has run the call)
      if constexpr (!kPair) promote_body<kAK, kBK>(p, tmA, tmB, smem_raw);
      return;
    }
  }
  const int total_items = hdr->total_items;
  if (total_items == 0) return;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if constexpr (kFp4 && kWideK) {
    // sized without alignment slack (the ring fills shared memory): the base must be aligned already
    if (base != smem_raw) {
      if (threadIdx.x == 0 && p.status_dev) atomicExch(p.status_dev, KGW_ERR_CUDA);
      return;
    }
  }
  uint8_t* stage_mem = base;
  uint8_t* epi_stage_mem = base + size_t(kStages) * kStageBytes;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(epi_stage_mem + EPI_STAGE_TOTAL);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0: leader (issues MMAs, schedules work)
  const bool leader = rank == 0;
  int32_t* item_counter = const_cast<int32_t*>(&hdr->item_counter);
  volatile int* abort_flag = &ctl->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], kEpiWarps * kHalves);
    }
    for (int w = 0; w < WORK_RING; ++w) {
      mbar_init(&ctl->wfull[w], 1);
      // consumers: the producer and the epilogue warps of each CTA, the MMA thread, and in the
      // block-scaled kernels warp 10 (of the even CTA in a pair)
      mbar_init(&ctl->wempty[w], kHalves * (1 + kEpiWarps) + 1 + (kFp8 ? 1 : 0));
    }
    ctl->items_started = 0;
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->cp_done, 1);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&ctl->sf_full[st], 1);
      mbar_init(&ctl->sfdata[st], 1);
    }
    ctl->abort_flag = 0;
    fence_mbarrier_init();
    if (p.tokens_sum > 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if constexpr (kFp8 && kPair) {
        tma_prefetch_desc(&p.tm_sfa);
        tma_prefetch_desc(&p.tm_sfb);
      }
    }
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(&ctl->tmem_base, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&ctl->tmem_base, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (kPair) {
    cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // cluster addresses of the leader's barriers that the peer signals
  const uint32_t leader_full0 = kPair ? mapa_shared(smem_u32(&ctl->full[0]), 0) : 0u;
  const uint32_t leader_wempty0 = kPair ? mapa_shared(smem_u32(&ctl->wempty[0]), 0) : 0u;
  const uint32_t leader_tempty0 = kPair ? mapa_shared(smem_u32(&ctl->tempty[0]), 0) : 0u;
  const uint32_t leader_sfdata0 = kPair ? mapa_shared(smem_u32(&ctl->sfdata[0]), 0) : 0u;

  // A consumer is done with work-ring slot `slot`.
  auto release_slot = [&](int slot) {
    if (kPair && !leader)
      mbar_arrive_remote(leader_wempty0 + slot * 8);
    else
      mbar_arrive(&ctl->wempty[slot]);
  };

  // Block-scaled kernels: a stage's scale-factor blocks (32 rows x 16 bytes each, in TMEM order in
  // shared memory) -> the stage's TMEM columns, repeated in the four lane quadrants; a pair's copies
  // take each CTA's own shared memory to its own TMEM.
  constexpr int kSfBlocks = kNv ? 12 : (kFp4 ? (kWideK ? 12 : 6) : 3);
  constexpr uint32_t kSfCols =
      kNv ? SF_STAGE_COLS_NV : (kFp4 ? (kWideK ? SF_STAGE_COLS_FP4_WIDE : SF_STAGE_COLS_FP4) : SF_STAGE_COLS);
  // (single-CTA FP8 stages keep the raw FP32 scales ahead of the converted blocks)
  constexpr uint32_t kSfSrc = kStageA + kStageB + ((kFp4 || kPair) ? 0u : SF_UE8_OFFSET);
  auto copy_scale_factors = [&](int stage) {
    const uint32_t sf = tmem_base + SF_COL0 + stage * kSfCols;
    const uint32_t src = smem_u32(stage_mem + size_t(stage) * kStageBytes) + kSfSrc;
#pragma unroll
    for (int blk = 0; blk < kSfBlocks; ++blk) {
      const uint64_t d = sdesc_noswizzle(src + blk * SF_UE8_BLOCK, 16, 128);
      if constexpr (kPair)
        tmem_cp_pair_32x128b_warpx4(sf + 4 * blk, d);
      else
        tmem_cp_32x128b_warpx4(sf + 4 * blk, d);
    }
  };
  // CTA pairs, warp 10 of the even CTA, per stage: wait for the stage's prepared scale factors (their
  // own barrier: they land before the operand tiles), copy them and commit them to sf_full, which
  // the MMA thread waits on after the operands' barrier. The copies thus run while the operand
  // tiles arrive, off the stage's critical path. (Every tcgen05 instruction holds its issuing thread
  // for tens of cycles: next to its four MMAs, its waits and its commit, the MMA thread has no room
  // for the copies within the 512 cycles those MMAs run.) The stage's columns are free again by
  // then: the producers reload a stage only after the MMAs that read it have completed. Returns
  // false (in every lane) on timeout or abort.
  auto hand_off_scale_factors = [&](int stage, uint32_t phase) -> bool {
    int good = 1;
    if (lane == 0) {
      good = wait_bounded_t<kPair>(&ctl->sfdata[stage], phase, abort_flag, p.timeout_ns) ? 1 : 0;
      if (good) {
        tc_fence_after();
        copy_scale_factors(stage);
        mma_commit_pair(&ctl->sf_full[stage], 0x1);
      }
    }
    return __shfl_sync(0xffffffffu, good, 0) != 0;
  };
  // warp 10's copies complete before TMEM is released
  auto drain_scale_copies = [&]() {
    if (lane == 0) {
      mma_commit_pair(&ctl->cp_done, 0x1);
      int dummy = 0;
      wait_bounded_t<kPair>(&ctl->cp_done, 0, &dummy, p.timeout_ns);
    }
    __syncwarp();
  };

  if (warp == 0) {
    // ======================= TMA producer =======================
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    for (int n = 0;; ++n) {
      const int slot = n % WORK_RING;
      const bool okw = wait_bounded_t<kPair>(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns);
      if (!__all_sync(0xffffffffu, okw)) break;
      const Item it = ctl->work[slot];
      __syncwarp();
      if (lane == 0) {
        release_slot(slot);
        // the scheduler may claim further items
        if (leader && it.e >= 0) *reinterpret_cast<volatile int32_t*>(&ctl->items_started) = n + 1;
      }
      if (it.e < 0) break;
      // ragged + K-major operand: the expert's own descriptor, coordinates relative to its block
      const CUtensorMap* amap = &tmA;
      const CUtensorMap* bmap = &tmB;
      if ((kAK && p.ragged) || p.tail_a) {
        amap = reinterpret_cast<const CUtensorMap*>(p.ws + p.L.tmaps + size_t(it.e) * 128);
        if (lane == 0 && it.kend > it.kbeg) fence_tmap_acquire(amap);
      }
      if ((kBK && p.ragged) || p.tail_b) {
        bmap = reinterpret_cast<const CUtensorMap*>(p.ws + p.L.tmaps_b + size_t(it.e) * 128);
        if (lane == 0 && it.kend > it.kbeg) fence_tmap_acquire(bmap);
      }
      // this CTA's A rows (M-grouped pair: the row's own tile for each CTA)
      const int a_row = kMG ? (rank ? it.m1 : it.m0) : it.m0 + static_cast<int>(rank) * BM;
      const int b_col = it.n0 + static_cast<int>(rank) * (BN / kHalves);  // this CTA's B columns
      for (int kb = it.kbeg; kb < it.kend; ++kb) {
        bool ok2 = true;
        const bool drop = (p.test_drop_stage >= 0 && blockIdx.x == 0 && issued == p.test_drop_stage);
        if (lane == 0) {
          ok2 = wait_bounded_t<kPair>(&ctl->empty[stage], phase ^ 1, abort_flag, p.timeout_ns);
          if (ok2 && !drop && leader) {
            if constexpr (kSfTx > 0) mbar_arrive_expect_tx(&ctl->sfdata[stage], 2 * kSfTx);
            mbar_arrive_expect_tx(&ctl->full[stage], kExpectTx);
          }
        }
        ok2 = __shfl_sync(0xffffffffu, ok2, 0);
        if (!ok2) break;
        uint8_t* sA = stage_mem + size_t(stage) * kStageBytes;
        uint8_t* sB = sA + kStageA;
        const int64_t tok = it.begin + int64_t(kb) * bk;
        if (!drop && lane == 0) {
          const uint32_t fb = kPair ? leader_full0 + stage * 8 : 0u;
          auto load = [&](void* dst, const CUtensorMap* map, int32_t x, int32_t y) {
            if constexpr (kPair)
              tma_load_2d_pair(dst, map, fb, x, y);
            else
              tma_load_2d(dst, map, &ctl->full[stage], x, y);
          };
          // block-scaled pairs: the scale factors complete on the even CTA's sfdata barrier
          auto load_sf = [&](void* dst, const CUtensorMap* map, int32_t x, int32_t y) {
            tma_load_2d_pair(dst, map, leader_sfdata0 + stage * 8, x, y);
          };
          // token coordinate: relative to the expert's block for per-expert descriptors (and for
          // the M-grouped GEMM, whose K axis is the fixed contraction axis)
          // (FP4: the TMA tensor counts bytes, two tokens each)
          const int32_t kx = ((kMG || p.ragged) ? kb * bk : static_cast<int32_t>(tok)) / (kFp4 ? 2 : 1);
          // M-grouped: group e's B occupies rows [e*N, e*N+N) (K-major) or [e*K, e*K+K) (N-major)
          const int32_t b_row = kMG ? it.e * p.I + b_col : b_col;
          const int32_t b_tok = kMG ? it.e * p.K + kb * bk : static_cast<int32_t>(tok);
          // scales first: they are small and land before the operand tiles, so the converter's
          // work is done by the time the MMA has its operands
          if constexpr (kFp8 && kPair && kNv) {
            // prepared UE4M3 scale factors of this 256-token stage's four 64-token words, in TMEM
            // order: for each MMA k, [A word k][B word k (all 256 columns)]; word rows are the
            // expert's 64-token groups
            const int32_t w0 = 2 * it.srow + 4 * kb;
            uint8_t* sS = sB + kStageB;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              load_sf(sS + 3 * j * SF_UE8_BLOCK, &p.tm_sfa, it.m0 + static_cast<int32_t>(rank) * BM, w0 + j);
              load_sf(sS + (3 * j + 1) * SF_UE8_BLOCK, &p.tm_sfb, it.n0, w0 + j);
            }
          } else if constexpr (kFp8 && kPair && kFp4 && kWideK) {
            // prepared scale factors of this 512-token stage's four 128-token blocks, in TMEM order:
            // [A block 0..3][B block 0..3 (all 256 columns each)]; blocks past the expert's last one
            // repeat it (the MMAs of those tokens are not issued)
            const int32_t kblk = it.srow + 4 * kb;
            const int64_t left = it.n_e - int64_t(kb) * bk;
            const int32_t nb = left >= 4 * SCALE_BLOCK ? 4 : static_cast<int32_t>((left + SCALE_BLOCK - 1) / SCALE_BLOCK);
            uint8_t* sS = sB + kStageB;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int32_t bj = kblk + (j < nb ? j : nb - 1);
              load_sf(sS + j * SF_UE8_BLOCK, &p.tm_sfa, it.m0 + static_cast<int32_t>(rank) * BM, bj);
              load_sf(sS + (4 + 2 * j) * SF_UE8_BLOCK, &p.tm_sfb, it.n0, bj);
            }
          } else if constexpr (kFp8 && kPair && kFp4) {
            // prepared scale factors of this 256-token stage's two 128-token blocks, in TMEM order:
            // [A block 0][A block 1][B block 0 (all 256 columns)][B block 1]; when the expert's last
            // stage holds a single block, block 1 repeats block 0 (its second half is zero-filled)
            const int32_t kblk = it.srow + 2 * kb;
            const int32_t kblk1 = (2 * int64_t(kb) + 1) * SCALE_BLOCK < it.n_e ? kblk + 1 : kblk;
            uint8_t* sS = sB + kStageB;
            load_sf(sS, &p.tm_sfa, it.m0 + static_cast<int32_t>(rank) * BM, kblk);
            load_sf(sS + SF_UE8_BLOCK, &p.tm_sfa, it.m0 + static_cast<int32_t>(rank) * BM, kblk1);
            load_sf(sS + 2 * SF_UE8_BLOCK, &p.tm_sfb, it.n0, kblk);
            load_sf(sS + 4 * SF_UE8_BLOCK, &p.tm_sfb, it.n0, kblk1);
          } else if constexpr (kFp8 && kPair) {
            // prepared scale factors of this 128-token block, in TMEM order: this CTA's A rows and
            // all 256 B columns, by TMA onto the leader's scale-factor barrier
            const int32_t kblk = it.srow + kb;
            uint8_t* sS = sB + kStageB;
            load_sf(sS, &p.tm_sfa, it.m0 + static_cast<int32_t>(rank) * BM, kblk);
            load_sf(sS + SF_UE8_BLOCK, &p.tm_sfb, it.n0, kblk);
          } else if constexpr (kNv) {
            // NVFP4: the four 64-token scale words of this 256-token stage (UE4M3 bytes per 16
            // tokens): [A word 0..3][B word 0..3]; word rows are the expert's 64-token groups
            const int64_t w0 = 2 * int64_t(it.srow) + 4 * int64_t(kb);
            uint8_t* sS = sB + kStageB;
            mbar_arrive_expect_tx(&ctl->sfdata[stage], SF_SMEM_BYTES_NV);
#pragma unroll
            for (int j = 0; j < 4; ++j) bulk_load(sS + j * BM * 4, p.sfa + (w0 + j) * p.H + it.m0, BM * 4, &ctl->sfdata[stage]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              bulk_load(sS + 4 * BM * 4 + j * BN * 4, p.sfb + (w0 + j) * p.I + it.n0, BN * 4, &ctl->sfdata[stage]);
          } else if constexpr (kFp4) {
            // the two 128-token scale words of this 256-token stage: [A word 0][A word 1]
            // [B word 0][B word 1], on the stage's scale barrier. Scale blocks are the expert's own
            // (rows from it.srow on); when its last stage holds a single block, word 1 repeats
            // word 0 (the stage's second half is zero-filled, and no row past the tensor is read).
            const int64_t kblk = int64_t(it.srow) + 2 * int64_t(kb);
            const int64_t kblk1 = (2 * int64_t(kb) + 1) * SCALE_BLOCK < it.n_e ? kblk + 1 : kblk;
            uint8_t* sS = sB + kStageB;
            mbar_arrive_expect_tx(&ctl->sfdata[stage], SF_SMEM_BYTES_FP4);
            bulk_load(sS, p.sfa + kblk * p.H + it.m0, BM * 4, &ctl->sfdata[stage]);
            bulk_load(sS + BM * 4, p.sfa + kblk1 * p.H + it.m0, BM * 4, &ctl->sfdata[stage]);
            bulk_load(sS + 2 * BM * 4, p.sfb + kblk * p.I + it.n0, BN * 4, &ctl->sfdata[stage]);
            bulk_load(sS + 2 * BM * 4 + BN * 4, p.sfb + kblk1 * p.I + it.n0, BN * 4, &ctl->sfdata[stage]);
          } else if constexpr (kFp8) {
            // this 128-token block's FP32 scales: the tile's 128 rows of A and 256 columns of B;
            // they complete on the stage's scale barrier. K-grouped: the expert's block kb
            // (scale rows from it.srow on); M-grouped: block kb of the fixed K axis.
            const int64_t kblk = kMG ? tok / SCALE_BLOCK : int64_t(it.srow) + kb;
            uint8_t* sS = sB + kStageB;
            // (M-grouped: A's scales are [K/128, rows], the group's weight scales [G, K/128, N])
            const int64_t bblk = kMG ? int64_t(it.e) * (p.K / SCALE_BLOCK) + kblk : kblk;
            mbar_arrive_expect_tx(&ctl->sfdata[stage], SF_SMEM_BYTES);
            bulk_load(sS, p.sfa + kblk * p.H + it.m0, BM * 4, &ctl->sfdata[stage]);
            bulk_load(sS + BM * 4, p.sfb + bblk * p.I + it.n0, BN * 4, &ctl->sfdata[stage]);
          }
          constexpr int kAtom = kFp8 ? 128 : 64;  // elements per 128-byte swizzle row
          constexpr int32_t kBoxX = kFp4 ? 128 : BK_BF16;  // a K-major box's token extent in descriptor units
          // A: K-major -> one box [128 rows x bk tokens]; MN-major -> boxes [bk tokens x 128 B of rows]
          if constexpr (kAK) {
            load(sA, amap, kx, a_row);
            if constexpr (kWideK) load(sA + BM * 128, amap, kx + kBoxX, a_row);  // second box of the stage
          } else {
#pragma unroll
            for (int j = 0; j < BM / kAtom; ++j)
              load(sA + j * bk * 128, amap, a_row + kAtom * j, static_cast<int32_t>(tok));
          }
          // B: K-major -> one box [this CTA's columns x bk tokens]; MN-major -> boxes of 128 B of columns
          if constexpr (kBK) {
            load(sB, bmap, kx, b_row);
            if constexpr (kWideK) load(sB + (BN / kHalves) * 128, bmap, kx + kBoxX, b_row);
          } else {
#pragma unroll
            for (int j = 0; j < BN / kHalves / kAtom; ++j)
              load(sB + j * bk * 128, bmap, b_col + kAtom * j, b_tok);
          }
        }
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
    }
    // Drain: the leader's last kStages stages must land before exit (the peer's copies complete
    // on the leader's barriers, which the cluster barrier at the end waits for).
    if (lane == 0 && leader) {
      int s = stage;
      uint32_t ph = phase;
      for (int i = 0; i < kStages && i < issued; ++i) {
        if (--s < 0) {
          s = kStages - 1;
          ph ^= 1;
        }
        int dummy = 0;
        wait_bounded_t<kPair>(&ctl->full[s], ph, &dummy, p.timeout_ns);
        if constexpr (kSfTx > 0) wait_bounded_t<kPair>(&ctl->sfdata[s], ph, &dummy, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (leader only) =======================
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int tcount = 0;
      constexpr uint32_t a_mn = kAK ? 0u : 1u, b_mn = kBK ? 0u : 1u;
      const uint32_t idesc = kNv ? idesc_nvf4(BM * kHalves, BN) : kFp4 ? idesc_mxf4(BM * kHalves, BN)
                             : kFp8 ? idesc_mxf8(BM * kHalves, BN, a_mn, b_mn, 0)
                                    : idesc_bf16_f32(BM * kHalves, BN, a_mn, b_mn);
      // Shared-memory operand descriptors (128-byte swizzle). K-major: 128-byte rows, 8-row groups
      // 1024 B apart, K step of 32 bytes. MN-major: 128-byte atoms of rows/columns stacked along K
      // (one atom = bk x 128 B, LBO between atoms), 8-row K groups 1024 B apart, K step of
      // 16 (BF16) / 32 (FP8) rows = 2048 / 4096 bytes.
      constexpr uint32_t kMnStep = kFp8 ? 4096u : 2048u;
      // FP32 per-128 scales repeat one byte in all 4 positions: keep byte 0 for every MMA
      const uint32_t sf_sel = p.sf_packed ? 0xFFFFFFFFu : 0u;
      const uint32_t mn_lbo = static_cast<uint32_t>(bk) * 128u;
      // descriptor = template (offsets, swizzle, version) + start address / 16 in the low 14 bits;
      // the start address advances by the K step for each of the 4 MMAs of a stage
      const uint64_t a_tmpl = kAK ? sdesc_sw128(0, 16, 1024) : sdesc_sw128(0, mn_lbo, 1024);
      const uint64_t b_tmpl = kBK ? sdesc_sw128(0, 16, 1024) : sdesc_sw128(0, mn_lbo, 1024);
      constexpr uint32_t a_step = (kAK ? 32u : kMnStep) >> 4;
      constexpr uint32_t b_step = (kBK ? 32u : kMnStep) >> 4;
      auto desc = [](uint64_t tmpl, uint32_t base, uint32_t step, int k) {
        return tmpl + static_cast<uint64_t>(((base & 0x3FFFFu) >> 4) + k * step);
      };
      for (int n = 0;; ++n) {
        const int slot = n % WORK_RING;
        if (!wait_bounded_t<kPair>(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns)) break;
        const Item it = ctl->work[slot];
        release_slot(slot);
        if (it.e < 0) break;
        if (it.kend == it.kbeg) continue;
        // BF16: two accumulators alternate; FP8: one accumulator (TMEM also holds scale factors)
        const int acc = kFp8 ? 0 : (tcount & 1);
        const uint32_t use = kFp8 ? static_cast<uint32_t>(tcount) : static_cast<uint32_t>(tcount >> 1);
        if (!wait_bounded_t<kPair>(&ctl->tempty[acc], (use & 1) ^ 1, abort_flag, p.timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = it.kbeg; kb < it.kend; ++kb) {
          if (!wait_bounded_t<kPair>(&ctl->full[stage], phase, abort_flag, p.timeout_ns)) {
            ok = false;
            break;
          }
          if constexpr (kFp8 && kPair) {
            // block-scaled pairs: warp 10 has copied the stage's scale factors to TMEM
            if (!wait_bounded_t<kPair>(&ctl->sf_full[stage], phase, abort_flag, p.timeout_ns)) {
              ok = false;
              break;
            }
          }
          if constexpr (kFp8 && !kPair) {
            // single CTA: the converter has written the stage's scale factors in TMEM order
            if (!wait_bounded(&ctl->sf_full[stage], phase, abort_flag, p.timeout_ns)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          // single CTA: the copies come first in this thread's order, so its MMAs see them
          if constexpr (kFp8 && !kPair) copy_scale_factors(stage);
          const uint32_t a_addr = smem_u32(stage_mem + size_t(stage) * kStageBytes);
          const uint32_t b_addr = a_addr + kStageA;
          if constexpr (kFp8 && kPair && !kFp4) {
            // the stage's scale factors are in TMEM columns 4i of the stage's 12 in both CTAs; MMA k
            // uses byte k of every word (the FP32 scales' byte is repeated, packed UE8M0 words hold
            // one per 32-token block)
            const uint32_t sfa = tmem_base + SF_COL0 + stage * SF_STAGE_COLS;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_mxf8_pair(d_tmem, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k),
                            idesc | idesc_sf_id(static_cast<uint32_t>(k)), sfa, sfa + SF_A_COLS,
                            (kb > it.kbeg || k > 0) ? 1u : 0u);
          } else if constexpr (kNv) {
            // the stage's 12 scale blocks are in TMEM columns 4i of its 48; MMA k (64 tokens) reads
            // A block 3k (columns 12k..12k+3) and B blocks 3k+1, 3k+2 (12k+4..12k+11), all four
            // UE4M3 bytes of each column
            const uint32_t sf = tmem_base + SF_COL0 + stage * SF_STAGE_COLS_NV;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc_in = (kb > it.kbeg || k > 0) ? 1u : 0u;
              if constexpr (kPair)
                mma_nvf4_pair(d_tmem, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k), idesc,
                              sf + 12 * k, sf + 12 * k + 4, acc_in);
              else
                mma_nvf4(d_tmem, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k), idesc, sf + 12 * k,
                         sf + 12 * k + 4, acc_in);
            }
          } else if constexpr (kFp4 && kWideK) {
            // 512-token stage: 12 scale blocks in TMEM columns 4i of its 48 (A words 0..3, then B words
            // 0..3 of 8 columns each); MMA k (64 tokens, box k/4) reads word k/2 of A (columns 4(k/2))
            // and B (16 + 8(k/2)), byte pair (k%2)*2 of it. An expert's last stage may hold 256 tokens
            // only: the MMAs of the other half are not issued (the same MMAs as with 256-token stages).
            const uint32_t sf = tmem_base + SF_COL0 + stage * SF_STAGE_COLS_FP4_WIDE;
            const int nk = int64_t(kb) * bk + bk / 2 >= it.n_e ? 4 : 8;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (k < nk) {
                const uint32_t id = idesc | idesc_sf_id(static_cast<uint32_t>(k & 1) * 2u);
                const uint32_t acc_in = (kb > it.kbeg || k > 0) ? 1u : 0u;
                mma_mxf4_pair(d_tmem, desc(a_tmpl, a_addr + (k >> 2) * (BM * 128u), a_step, k & 3),
                              desc(b_tmpl, b_addr + (k >> 2) * ((BN / kHalves) * 128u), b_step, k & 3), id,
                              sf + 4 * (k >> 1), sf + 16 + 8 * (k >> 1), acc_in);
              }
            }
          } else if constexpr (kFp4) {
            // the stage's 6 scale blocks are in TMEM columns 4i of its 24; MMA k (64 tokens) reads
            // word k/2 of A (columns 0/4) and B (8/16), byte pair (k%2)*2 of it
            const uint32_t sf = tmem_base + SF_COL0 + stage * SF_STAGE_COLS_FP4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t id = idesc | idesc_sf_id(static_cast<uint32_t>(k & 1) * 2u);
              const uint32_t acc_in = (kb > it.kbeg || k > 0) ? 1u : 0u;
              if constexpr (kPair)
                mma_mxf4_pair(d_tmem, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k), id,
                              sf + 4 * (k >> 1), sf + 8 + 8 * (k >> 1), acc_in);
              else
                mma_mxf4(d_tmem, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k), id,
                         sf + 4 * (k >> 1), sf + 8 + 8 * (k >> 1), acc_in);
            }
          } else if constexpr (kFp8) {
            const uint32_t sfa = tmem_base + SF_COL0 + stage * SF_STAGE_COLS;
            const uint32_t sfb = sfa + SF_A_COLS;
#pragma unroll
            for (int k = 0; k < 4; ++k)  // packed scales: MMA k uses byte k (its 32-token block)
              mma_mxf8(d_tmem, desc(a_tmpl, a_addr, a_step, k), desc(b_tmpl, b_addr, b_step, k),
                       idesc | (idesc_sf_id(static_cast<uint32_t>(k)) & sf_sel), sfa, sfb,
                       (kb > it.kbeg || k > 0) ? 1u : 0u);
          } else {
            // 128-token stages: a K-major operand's second 64 tokens are a box of their own
            // (A 128 rows x 128 B, B this CTA's columns x 128 B further on); MN-major atoms hold all
            // of the stage's tokens
#pragma unroll
            for (int k = 0; k < (kWideK ? 8 : 4); ++k) {
              // in a pair each CTA holds 128 rows of A and 128 columns of B
              const uint64_t adesc = kAK && kWideK ? desc(a_tmpl, a_addr + (k >> 2) * (BM * 128u), a_step, k & 3)
                                                   : desc(a_tmpl, a_addr, a_step, k);
              const uint64_t bdesc = kBK && kWideK
                                         ? desc(b_tmpl, b_addr + (k >> 2) * ((BN / kHalves) * 128u), b_step, k & 3)
                                         : desc(b_tmpl, b_addr, b_step, k);
              if constexpr (kPair)
                mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb > it.kbeg || k > 0) ? 1u : 0u);
              else
                mma_bf16(d_tmem, adesc, bdesc, idesc, (kb > it.kbeg || k > 0) ? 1u : 0u);
            }
          }
          if constexpr (kPair)
            mma_commit_pair(&ctl->empty[stage], 0x3);
          else
            mma_commit(&ctl->empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (kPair)
          mma_commit_pair(&ctl->tfull[acc], 0x3);
        else
          mma_commit(&ctl->tfull[acc]);
        ++tcount;
      }
      // All MMAs issued by this thread complete before TMEM is released.
      if constexpr (kPair)
        mma_commit_pair(&ctl->mma_done, 0x1);
      else
        mma_commit(&ctl->mma_done);
      int dummy = 0;
      wait_bounded_t<kPair>(&ctl->mma_done, 0, &dummy, p.timeout_ns);
    }
    __syncwarp();
  } else if (kFp8 && warp < EPI_WARP0 + kEpiWarps) {
    // ======================= Epilogue of the block-scaled kernels (warps 2..9) =======================
    // Eight warps: warp w reads TMEM lane quadrant w % 4 and accumulator columns 128 * ((w - 2) / 4)
    // onward. With 16-bit output and no accumulation the warp first moves its whole 32 x 128 block
    // into its holding columns of TMEM (NVFP4: into registers), packed to 16 bits, and hands the
    // accumulator back, so the MMA of the next tile does not wait for the stores.
    const int q = warp & 3;
    const int ew = warp - EPI_WARP0;
    const int col0 = (ew >> 2) * (BN / 2);
    int32_t* counters = reinterpret_cast<int32_t*>(p.ws + p.L.counters);
    const int32_t* slot_base = reinterpret_cast<const int32_t*>(p.ws + p.L.slot_base);
    const int32_t* counter_base = reinterpret_cast<const int32_t*>(p.ws + p.L.counter_base);
    float* partials = reinterpret_cast<float*>(p.ws + p.L.partials);
    uint4* stg = reinterpret_cast<uint4*>(epi_stage_mem + ew * (EPI_STAGE_TOTAL / NUM_EPI_WARPS_FP8));
    const int rsub = lane >> 2;       // row within an 8-row group of the read-back
    const int csub = lane & 3;        // 16-byte chunk within a 64-byte row segment
    // NVFP4: the product of the per-tensor global scales (1 where one is not given)
    const float gscale = kNv ? (p.gscale_a ? __ldg(p.gscale_a) : 1.0f) * (p.gscale_b ? __ldg(p.gscale_b) : 1.0f) : 1.0f;
    int tcount = 0;
    for (int n = 0;; ++n) {
      const int slot = n % WORK_RING;
      const bool okw = wait_bounded_t<kPair>(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns);
      if (!__all_sync(0xffffffffu, okw)) break;
      const Item it = ctl->work[slot];
      __syncwarp();
      if (lane == 0) release_slot(slot);
      if (it.e < 0) break;
      const int esz = p.out_bf16 ? 2 : 4;
      char* obase = out_row_ptr<kMG>(p, it, static_cast<int>(rank) * BM + q * 32) + size_t(col0) * esz;
      const size_t ostride = size_t(p.I) * esz;
      if (it.kend == it.kbeg) {
        const int rb = (BN / 2) * esz;
#pragma unroll 1
        for (int r = 0; r < 32; ++r)
          for (int off = lane * 16; off < rb; off += 32 * 16)
            *reinterpret_cast<uint4*>(obase + r * ostride + off) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const bool okt = wait_bounded_t<kPair>(&ctl->tfull[0], static_cast<uint32_t>(tcount) & 1, abort_flag, p.timeout_ns);
      if (!__all_sync(0xffffffffu, okt)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + col0;
      // (the peer's arrive is relaxed: the accumulator's TMEM loads have completed, and the
      // hand-back publishes nothing)
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair && !leader)
            mbar_arrive_remote_relaxed(leader_tempty0);
          else
            mbar_arrive(&ctl->tempty[0]);
        }
      };
      // row `lane` of the staging buffer: four 16-byte chunks, chunk c at slot c ^ ((lane >> 1) & 3)
      auto stage4 = [&](uint4 v0, uint4 v1, uint4 v2, uint4 v3) {
        const int sw = (lane >> 1) & 3;
        stg[lane * 4 + (0 ^ sw)] = v0;
        stg[lane * 4 + (1 ^ sw)] = v1;
        stg[lane * 4 + (2 ^ sw)] = v2;
        stg[lane * 4 + (3 ^ sw)] = v3;
      };
      auto unstage4 = [&](int j) {
        const int r = 8 * j + rsub;
        return stg[r * 4 + (csub ^ ((r >> 1) & 3))];
      };
      if (!kNv && !(kFp4 && kWideK) && it.nsplit == 1 && p.out_bf16 && !p.accumulate) {
        // TMEM accumulator -> packed 16-bit values in this warp's holding columns -> hand back
        const uint32_t hold = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + EPI_HOLD_COL0 + (ew >> 2) * 64;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32], pk[16];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = p.out_f16 ? pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]))
                              : pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          tmem_st_32x32b_x16(hold + c * 16, pk);
        }
        release_acc();
        tmem_st_wait();
        // 32 columns (64 bytes per row) per round: 4 lanes per row, 8 rows per store instruction
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
          tmem_ld_32x32b_x16(hold + c * 16, pk);
          tmem_ld_wait();
          stage4(make_uint4(pk[0], pk[1], pk[2], pk[3]), make_uint4(pk[4], pk[5], pk[6], pk[7]),
                 make_uint4(pk[8], pk[9], pk[10], pk[11]), make_uint4(pk[12], pk[13], pk[14], pk[15]));
          __syncwarp();
          char* cbase = obase + size_t(c * 32 + csub * 8) * 2;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (!kMG || q * 32 + 8 * j + rsub < it.rows)  // M-grouped masked layout: valid rows only
              *reinterpret_cast<uint4*>(cbase + (8 * j + rsub) * ostride) = unstage4(j);
          __syncwarp();
        }
      } else if ((kNv || (kFp4 && kWideK)) && it.nsplit == 1 && p.out_bf16 && !p.accumulate) {
        // NVFP4 and 512-token FP4 stages (their scale-factor rings leave TMEM no holding columns):
        // the warp's 32 x 128 block, times the global scales (NVFP4; else 1) and packed to 16 bits,
        // waits in registers (64 per thread) while the accumulator goes back to the MMA
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x0 = __uint_as_float(r[2 * i]) * gscale, x1 = __uint_as_float(r[2 * i + 1]) * gscale;
            pk[c * 16 + i] = p.out_f16 ? pack_f16x2(x0, x1) : pack_bf16x2(x0, x1);
          }
        }
        release_acc();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          stage4(make_uint4(pk[c * 16 + 0], pk[c * 16 + 1], pk[c * 16 + 2], pk[c * 16 + 3]),
                 make_uint4(pk[c * 16 + 4], pk[c * 16 + 5], pk[c * 16 + 6], pk[c * 16 + 7]),
                 make_uint4(pk[c * 16 + 8], pk[c * 16 + 9], pk[c * 16 + 10], pk[c * 16 + 11]),
                 make_uint4(pk[c * 16 + 12], pk[c * 16 + 13], pk[c * 16 + 14], pk[c * 16 + 15]));
          __syncwarp();
          char* cbase = obase + size_t(c * 32 + csub * 8) * 2;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (!kMG || q * 32 + 8 * j + rsub < it.rows)
              *reinterpret_cast<uint4*>(cbase + (8 * j + rsub) * ostride) = unstage4(j);
          __syncwarp();
        }
      } else if (it.nsplit == 1) {
        // FP32 output or accumulation: 16 columns per TMEM load, the accumulator is handed back
        // after the last load
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          {
            uint32_t r[16];
            tmem_ld_32x32b_x16(taddr + c * 16, r);
            tmem_ld_wait();
            if (c == 7) release_acc();
            if constexpr (kNv) {   // per-tensor global scales multiply the whole product
#pragma unroll
              for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * gscale);
            }
            stage4(make_uint4(r[0], r[1], r[2], r[3]), make_uint4(r[4], r[5], r[6], r[7]),
                   make_uint4(r[8], r[9], r[10], r[11]), make_uint4(r[12], r[13], r[14], r[15]));
          }
          __syncwarp();
          char* cbase = obase + size_t(c * 16 + csub * 4) * esz;
          auto live = [&](int j) { return !kMG || q * 32 + 8 * j + rsub < it.rows; };
          uint4 old[4];
          if (p.accumulate) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (live(j)) old[j] = load_old4(p, cbase + (8 * j + rsub) * ostride);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 u = unstage4(j);
            if (live(j))
              emit4(p, cbase + (8 * j + rsub) * ostride,
                    make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)),
                    old[j]);
          }
          __syncwarp();
        }
      } else {
        // split-K: this warp's 32 x 128 partial block to the workspace, then the last arriving
        // warp for this block sums the partials in split order
        const int sb = __ldg(slot_base + it.e) + it.tile * it.nsplit;
        auto prow = [&](int s, int rr) {
          return partials + ((size_t(sb + s) * kHalves + rank) * BM + q * 32 + rr) * BN + col0;
        };
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          {
            uint32_t r[16];
            tmem_ld_32x32b_x16(taddr + c * 16, r);
            tmem_ld_wait();
            if (c == 7) release_acc();
            stage4(make_uint4(r[0], r[1], r[2], r[3]), make_uint4(r[4], r[5], r[6], r[7]),
                   make_uint4(r[8], r[9], r[10], r[11]), make_uint4(r[12], r[13], r[14], r[15]));
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            __stcg(reinterpret_cast<uint4*>(prow(it.split, 8 * j + rsub) + c * 16 + csub * 4), unstage4(j));
          __syncwarp();
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const int cidx = ((__ldg(counter_base + it.e) + it.tile) * kHalves + static_cast<int>(rank)) * EPI_COUNTERS + ew;
          last = atomicAdd(counters + cidx, 1) == it.nsplit - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            const int col = c * 16 + csub * 4;
            char* cbase = obase + size_t(col) * esz;
            uint4 old[4];
            if (p.accumulate) {
#pragma unroll
              for (int j = 0; j < 4; ++j) old[j] = load_old4(p, cbase + (8 * j + rsub) * ostride);
            }
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s2 = 0; s2 < it.nsplit; ++s2) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 x = __ldcg(reinterpret_cast<const float4*>(prow(s2, 8 * j + rsub) + col));
                v[j].x += x.x;
                v[j].y += x.y;
                v[j].z += x.z;
                v[j].w += x.w;
              }
            }
            if constexpr (kNv) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                v[j].x *= gscale;
                v[j].y *= gscale;
                v[j].z *= gscale;
                v[j].w *= gscale;
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) emit4(p, cbase + (8 * j + rsub) * ostride, v[j], old[j]);
          }
        }
      }
      ++tcount;
    }
  } else if (!kFp8 && warp < EPI_WARP0 + kEpiWarps) {
    // ======================= Epilogue (warps 2..5) =======================
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    int32_t* counters = reinterpret_cast<int32_t*>(p.ws + p.L.counters);
    const int32_t* slot_base = reinterpret_cast<const int32_t*>(p.ws + p.L.slot_base);
    const int32_t* counter_base = reinterpret_cast<const int32_t*>(p.ws + p.L.counter_base);
    float* partials = reinterpret_cast<float*>(p.ws + p.L.partials);
    int tcount = 0;
    for (int n = 0;; ++n) {
      const int slot = n % WORK_RING;
      const bool okw = wait_bounded_t<kPair>(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns);
      if (!__all_sync(0xffffffffu, okw)) break;
      const Item it = ctl->work[slot];
      __syncwarp();
      if (lane == 0) release_slot(slot);
      if (it.e < 0) break;
      // this warp's 32 output rows start at tile row rank*128 + q*32; row r is `ostride` bytes further
      char* obase = out_row_ptr<kMG>(p, it, static_cast<int>(rank) * BM + q * 32);
      const size_t ostride = size_t(p.I) * (p.out_bf16 ? 2 : 4);
      const int esz = p.out_bf16 ? 2 : 4;
      if (it.kend == it.kbeg) {
        // empty expert, overwrite mode: the output tile is zero (4 rows x 512 bytes per instruction)
        const int rb = BN * esz;  // bytes per row segment
#pragma unroll 1
        for (int r = 0; r < 32; ++r)
          for (int off = lane * 16; off < rb; off += 32 * 16)
            *reinterpret_cast<uint4*>(obase + r * ostride + off) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int acc = kFp8 ? 0 : (tcount & 1);
      const uint32_t use = kFp8 ? static_cast<uint32_t>(tcount) : static_cast<uint32_t>(tcount >> 1);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      // This warp has read its 32 TMEM lanes: hand the accumulator back to the MMA issuer (the
      // peer's arrive is relaxed: the loads have completed, and the hand-back publishes nothing).
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair && !leader)
            mbar_arrive_remote_relaxed(leader_tempty0 + acc * 8);
          else
            mbar_arrive(&ctl->tempty[acc]);
        }
      };
      uint4* stg = reinterpret_cast<uint4*>(epi_stage_mem + (warp - EPI_WARP0) * EPI_STAGE_BYTES);
      // M-grouped masked layout: rows at or past the group's valid count are not touched
      auto live_row = [&](int r) { return !kMG || q * 32 + r < (rank ? it.rows1 : it.rows); };
      auto live = [&](int j) { return live_row(4 * j + (lane >> 3)); };
      if (it.nsplit == 1 && p.out_bf16 && !p.accumulate) {
        // 16-bit outputs (BF16 / FP16), overwrite: each thread reads row `lane` of a 64-column chunk
        // (one TMEM load), rounds it in registers and stages the packed 128-byte row, so a tile
        // takes four load / stage / store rounds and the staging carries half the bytes of FP32.
        // Stores: 8 lanes per 128-byte row segment, 4 rows per instruction.
        const bool okt = wait_bounded_t<kPair>(&ctl->tfull[acc], use & 1, abort_flag, p.timeout_ns);
        if (!__all_sync(0xffffffffu, okt)) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t pk[32];
          {
            uint32_t r[64];
            tmem_ld_32x32b_x64(taddr + c * 64, r);
            tmem_ld_wait();
            if (c == BN / 64 - 1) release_acc();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              pk[i] = p.out_f16 ? pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]))
                                : pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          }
          // row `lane` = 8 16-byte chunks, chunk i at slot i ^ (lane & 7) (the FP32 staging's swizzle)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            stg[lane * 8 + (i ^ (lane & 7))] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          __syncwarp();
          char* cbase = obase + size_t(c * 64 + (lane & 7) * 8) * 2;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + (lane >> 3);
            if (live_row(r)) *reinterpret_cast<uint4*>(cbase + r * ostride) = stg[r * 8 + ((lane & 7) ^ (r & 7))];
          }
          __syncwarp();
        }
        ++tcount;
        continue;
      }
      if (it.nsplit == 1 && p.accumulate) {
        // Accumulate: the previous output is read ahead of its use. The loads of the first D
        // 32-column chunks are issued before the accumulator is ready, so they overlap the tile's
        // MMAs; the loads of chunk c + D are issued as soon as chunk c is written. W 32-bit words
        // hold 4 previous outputs (2: BF16/FP16, 4: FP32). Same arithmetic as the other paths:
        // one FP32 add, one rounding.
        auto run = [&](auto w_tag, auto d_tag) -> bool {
          constexpr int W = decltype(w_tag)::value;
          constexpr int D = decltype(d_tag)::value;
          static_assert((BN / 32) % D == 0, "the chunks divide into groups of D");
          uint32_t old[D][8][W];
          auto issue = [&](int c, uint32_t (&o)[8][W]) {
            const char* cb = obase + size_t(c * 32 + (lane & 7) * 4) * esz;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (!live(j)) continue;
              const char* src = cb + (4 * j + (lane >> 3)) * ostride;
              if constexpr (W == 2) {
                const uint2 h = *reinterpret_cast<const uint2*>(src);
                o[j][0] = h.x;
                o[j][1] = h.y;
              } else {
                const uint4 h = *reinterpret_cast<const uint4*>(src);
                o[j][0] = h.x;
                o[j][1] = h.y;
                o[j][2] = h.z;
                o[j][3] = h.w;
              }
            }
          };
#pragma unroll
          for (int d = 0; d < D; ++d) issue(d, old[d]);
          const bool okt = wait_bounded_t<kPair>(&ctl->tfull[acc], use & 1, abort_flag, p.timeout_ns);
          if (!__all_sync(0xffffffffu, okt)) return false;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < BN / 32; c0 += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
              const int c = c0 + d;
              {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_ld_wait();
                if (c == BN / 32 - 1) release_acc();
                stage_row(stg, lane, r);
              }
              __syncwarp();
              char* cbase = obase + size_t(c * 32 + (lane & 7) * 4) * esz;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint4 o = W == 2 ? make_uint4(old[d][j][0], old[d][j][1], 0u, 0u)
                                       : make_uint4(old[d][j][0], old[d][j][1], old[d][j][W > 2 ? 2 : 0],
                                                    old[d][j][W > 2 ? 3 : 0]);
                if (live(j)) emit4(p, cbase + (4 * j + (lane >> 3)) * ostride, unstage(stg, j, lane), o);
              }
              __syncwarp();
              if (c + D < BN / 32) issue(c + D, old[d]);
            }
          }
          return true;
        };
        // two chunks in flight for 16-bit outputs, one for FP32 (and in the M-grouped kernels, whose
        // row predicates leave fewer registers), within the 255-register budget without spills
        constexpr int kDepth16 = kMG ? 1 : 2;
        const bool ok = p.out_bf16 ? run(std::integral_constant<int, 2>{}, std::integral_constant<int, kDepth16>{})
                                   : run(std::integral_constant<int, 4>{}, std::integral_constant<int, 1>{});
        if (!ok) break;
        ++tcount;
        continue;
      }
      const bool okt = wait_bounded_t<kPair>(&ctl->tfull[acc], use & 1, abort_flag, p.timeout_ns);
      if (!__all_sync(0xffffffffu, okt)) break;
      tc_fence_after();
      if (it.nsplit == 1) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          char* cbase = obase + size_t(c * 32 + (lane & 7) * 4) * esz;
          {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c * 32, r);
            tmem_ld_wait();
            if (c == BN / 32 - 1) release_acc();  // all TMEM reads of this warp are done
            stage_row(stg, lane, r);
          }
          __syncwarp();
          const uint4 none = make_uint4(0u, 0u, 0u, 0u);   // overwrite: no previous values
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (live(j)) emit4(p, cbase + (4 * j + (lane >> 3)) * ostride, unstage(stg, j, lane), none);
          __syncwarp();
        }
      } else {
        // split-K: publish this chunk's FP32 partial rows (row-major 128 x 256 per CTA half), then
        // the last arriving warp for these 32 rows sums all partials in split order. Each warp has
        // its own arrival counter per (tile, CTA half, lane quadrant): no cross-warp barrier.
        const int sb = __ldg(slot_base + it.e) + it.tile * it.nsplit;
        auto prow = [&](int s, int rr) {
          return partials + ((size_t(sb + s) * kHalves + rank) * BM + q * 32 + rr) * BN;
        };
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
          if (c == BN / 32 - 1) release_acc();
          stage_row(stg, lane, r);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rr = 4 * j + (lane >> 3);
            __stcg(reinterpret_cast<float4*>(prow(it.split, rr) + c * 32 + (lane & 7) * 4), unstage(stg, j, lane));
          }
          __syncwarp();
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const int cidx = ((__ldg(counter_base + it.e) + it.tile) * kHalves + static_cast<int>(rank)) * EPI_COUNTERS + q;
          last = atomicAdd(counters + cidx, 1) == it.nsplit - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int col = c * 32 + (lane & 7) * 4;
            char* cbase = obase + size_t(col) * esz;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              uint4 old[4];
              if (p.accumulate) {
#pragma unroll
                for (int j = 0; j < 4; ++j) old[j] = load_old4(p, cbase + (4 * (4 * h + j) + (lane >> 3)) * ostride);
              }
              float4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int s2 = 0; s2 < it.nsplit; ++s2) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float4 x = __ldcg(reinterpret_cast<const float4*>(prow(s2, 4 * (4 * h + j) + (lane >> 3)) + col));
                  v[j].x += x.x;
                  v[j].y += x.y;
                  v[j].z += x.z;
                  v[j].w += x.w;
                }
              }
#pragma unroll
              for (int j = 0; j < 4; ++j) emit4(p, cbase + (4 * (4 * h + j) + (lane >> 3)) * ostride, v[j], old[j]);
            }
          }
        }
      }
      ++tcount;
    }
  }

  if constexpr (kFp8 && !kPair) {
    if (warp == SF_WARP) {
      // ======================= FP8 / FP4 scale-factor converter (warp 10) =======================
      // Per k-iteration: the stage's FP32 scales (128 of A, 256 of B) -> UE8M0 bytes (replicated
      // over the four 32-token blocks) in the TMEM layout read by the block-scaled MMA: 32 rows x
      // 4 words per block, word c of row l holding row/column 32c + l.
      int stage = 0;
      uint32_t phase = 0;
      for (int n = 0;; ++n) {
        const int slot = n % WORK_RING;
        const bool okw = wait_bounded(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns);
        if (!__all_sync(0xffffffffu, okw)) break;
        const Item it = ctl->work[slot];
        __syncwarp();
        if (lane == 0) release_slot(slot);
        if (it.e < 0) break;
        bool ok = true;
        for (int kb = it.kbeg; kb < it.kend; ++kb) {
          // the scales have landed; this also means the copies of the previous round are done
          const bool okd = wait_bounded(&ctl->sfdata[stage], phase, abort_flag, p.timeout_ns);
          if (!__all_sync(0xffffffffu, okd)) {
            ok = false;
            break;
          }
          uint8_t* sS = stage_mem + size_t(stage) * kStageBytes + kStageA + kStageB;
          if constexpr (kNv) {
            // four 64-token UE4M3 words per row/column, rearranged in place into 12 blocks: for each
            // MMA k, A word k, then B word k for columns 0..127 and 128..255
            uint32_t* sw = reinterpret_cast<uint32_t*>(sS);
            uint32_t a[4][4], b[4][8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
              for (int j = 0; j < 4; ++j) a[k][j] = sw[k * BM + 32 * j + lane];
#pragma unroll
              for (int j = 0; j < 8; ++j) b[k][j] = sw[4 * BM + k * BN + 32 * j + lane];
            }
            __syncwarp();  // every lane has read its words before any is overwritten
            uint4* ue = reinterpret_cast<uint4*>(sS);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              ue[(3 * k) * 32 + lane] = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
              ue[(3 * k + 1) * 32 + lane] = make_uint4(b[k][0], b[k][1], b[k][2], b[k][3]);
              ue[(3 * k + 2) * 32 + lane] = make_uint4(b[k][4], b[k][5], b[k][6], b[k][7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->sf_full[stage]);
            // after the hand-off: a UE4M3 byte must not have its top bit set, and 0x7F is NaN
            uint32_t bad = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
              for (int j = 0; j < 4; ++j) bad |= (a[k][j] & 0x80808080u) | (((a[k][j] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u);
#pragma unroll
              for (int j = 0; j < 8; ++j) bad |= (b[k][j] & 0x80808080u) | (((b[k][j] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u);
            }
            if (bad && p.status_dev) atomicExch(p.status_dev, KGW_ERR_SCALES);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if constexpr (kFp4) {
            // packed UE8M0 words, two per row/column; rearranged in place into the 6 TMEM blocks
            uint32_t* sw = reinterpret_cast<uint32_t*>(sS);
            uint32_t a0[4], a1[4], b0[8], b1[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              a0[j] = sw[32 * j + lane];
              a1[j] = sw[BM + 32 * j + lane];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              b0[j] = sw[2 * BM + 32 * j + lane];
              b1[j] = sw[2 * BM + BN + 32 * j + lane];
            }
            __syncwarp();  // every lane has read its words before any is overwritten
            uint4* ue = reinterpret_cast<uint4*>(sS);
            ue[lane] = make_uint4(a0[0], a0[1], a0[2], a0[3]);
            ue[32 + lane] = make_uint4(a1[0], a1[1], a1[2], a1[3]);
            ue[64 + lane] = make_uint4(b0[0], b0[1], b0[2], b0[3]);
            ue[96 + lane] = make_uint4(b0[4], b0[5], b0[6], b0[7]);
            ue[128 + lane] = make_uint4(b1[0], b1[1], b1[2], b1[3]);
            ue[160 + lane] = make_uint4(b1[4], b1[5], b1[6], b1[7]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->sf_full[stage]);
            // the NaN byte check runs after the hand-off, off the MMA's critical path
            uint32_t ff = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) ff |= ff_bytes(a0[j]) | ff_bytes(a1[j]);
#pragma unroll
            for (int j = 0; j < 8; ++j) ff |= ff_bytes(b0[j]) | ff_bytes(b1[j]);
            if (ff && p.status_dev) atomicExch(p.status_dev, KGW_ERR_SCALES);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          const float* sa = reinterpret_cast<const float*>(sS);
          const float* sb = sa + BM;
          uint4* ue = reinterpret_cast<uint4*>(sS + SF_UE8_OFFSET);
          bool bad = false;
          uint32_t packed_ff = 0;
          if (!p.sf_packed) {
            // FP32 powers of two -> one UE8M0 byte repeated in the 4 bytes of the word
            ue[lane] = make_uint4(ue8m0_x4(sa[lane], bad), ue8m0_x4(sa[32 + lane], bad),
                                  ue8m0_x4(sa[64 + lane], bad), ue8m0_x4(sa[96 + lane], bad));
            ue[32 + lane] = make_uint4(ue8m0_x4(sb[lane], bad), ue8m0_x4(sb[32 + lane], bad),
                                       ue8m0_x4(sb[64 + lane], bad), ue8m0_x4(sb[96 + lane], bad));
            ue[64 + lane] = make_uint4(ue8m0_x4(sb[128 + lane], bad), ue8m0_x4(sb[160 + lane], bad),
                                       ue8m0_x4(sb[192 + lane], bad), ue8m0_x4(sb[224 + lane], bad));
          } else {
            // packed UE8M0 words (one byte per 32-token block) are already in the TMEM word form
            const uint32_t* wa = reinterpret_cast<const uint32_t*>(sa);
            const uint32_t* wb = reinterpret_cast<const uint32_t*>(sb);
            const uint4 x = make_uint4(wa[lane], wa[32 + lane], wa[64 + lane], wa[96 + lane]);
            const uint4 y = make_uint4(wb[lane], wb[32 + lane], wb[64 + lane], wb[96 + lane]);
            const uint4 z = make_uint4(wb[128 + lane], wb[160 + lane], wb[192 + lane], wb[224 + lane]);
            ue[lane] = x;
            ue[32 + lane] = y;
            ue[64 + lane] = z;
            // the byte 0xFF encodes NaN: checked after the hand-off below
            packed_ff = ff_bytes(x.x) | ff_bytes(x.y) | ff_bytes(x.z) | ff_bytes(x.w) | ff_bytes(y.x) | ff_bytes(y.y) |
                        ff_bytes(y.z) | ff_bytes(y.w) | ff_bytes(z.x) | ff_bytes(z.y) | ff_bytes(z.z) | ff_bytes(z.w);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->sf_full[stage]);
          if ((bad || packed_ff) && p.status_dev) atomicExch(p.status_dev, KGW_ERR_SCALES);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
    }
  }

  if constexpr (kFp8 && kPair) {
    if (warp == SF_WARP && leader) {
      // ======================= scale-factor copier of a CTA pair (warp 10, even CTA) ==============
      // the prepared scale factors arrive by TMA ahead of the operands; warp 10 only copies them to TMEM
      int stage = 0;
      uint32_t phase = 0;
      for (int n = 0;; ++n) {
        const int slot = n % WORK_RING;
        const bool okw = wait_bounded_t<kPair>(&ctl->wfull[slot], (n / WORK_RING) & 1, abort_flag, p.timeout_ns);
        if (!__all_sync(0xffffffffu, okw)) break;
        const Item it = ctl->work[slot];
        __syncwarp();
        if (lane == 0) release_slot(slot);
        if (it.e < 0) break;
        bool ok = true;
        for (int kb = it.kbeg; kb < it.kend; ++kb) {
          if (!hand_off_scale_factors(stage, phase)) {
            ok = false;
            break;
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      drain_scale_copies();
    }
  }

  if (warp == (kFp8 ? SCHED_WARP_FP8 : SCHED_WARP)) {
    // ======================= Scheduler (leader CTA) =======================
    // Claims items from the call's atomic counter up to SCHED_LOOKAHEAD items ahead of the producer
    // (the claim for item n+1 waits until the producer has started item n+1-SCHED_LOOKAHEAD, so no
    // CTA hoards more than that at the end of the queue, where the items are the shortest), decodes
    // each item once with the whole warp (decode_item_warp) and publishes it in the work ring of
    // this CTA and of its peer, while the current items' k-loops run.
    if (leader) {
      int lo_hint = 0;
      int cur = 0;
      if (lane == 0) cur = atomicAdd(item_counter, 1);
      cur = __shfl_sync(0xffffffffu, cur, 0);
      for (int n = 0;; ++n) {
        const int slot = n % WORK_RING;
        Item it;
        if (cur < total_items) {
          if constexpr (kMG)
            it = decode_item<kMG>(p, cur, bk);
          else
            it = decode_item_warp(p, cur, bk, lo_hint, lane);
        } else {
          it = Item{};
          it.e = -1;
        }
        int ok = 1;
        if (lane == 0) {
          ok = wait_bounded_t<kPair>(&ctl->wempty[slot], ((n / WORK_RING) & 1) ^ 1, abort_flag, p.timeout_ns) ? 1 : 0;
          if (ok) {
            ctl->work[slot] = it;
            if constexpr (kPair) {
              const uint32_t dst = mapa_shared(smem_u32(&ctl->work[slot]), 1);
              const uint4* w = reinterpret_cast<const uint4*>(&ctl->work[slot]);
#pragma unroll
              for (int i = 0; i < 4; ++i) st_cluster_v4(dst + 16 * i, w[i]);
              mbar_arrive_remote(mapa_shared(smem_u32(&ctl->wfull[slot]), 1));
            }
            mbar_arrive(&ctl->wfull[slot]);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0) || it.e < 0) break;
        // claim item n+1 once the producer has started item n+1-SCHED_LOOKAHEAD (bounded wait)
        int go = 1;
        if (lane == 0) {
          const uint64_t t0 = global_timer_ns();
          while (*reinterpret_cast<volatile int32_t*>(&ctl->items_started) < n + 2 - SCHED_LOOKAHEAD) {
            if (*abort_flag) {
              go = 0;
              break;
            }
            if (global_timer_ns() - t0 > p.timeout_ns) {
              *abort_flag = 1;
              go = 0;
              break;
            }
            __nanosleep(64);
          }
          if (go) cur = atomicAdd(item_counter, 1);
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) break;
        cur = __shfl_sync(0xffffffffu, cur, 0);
      }
    }
  }

  // ======================= teardown =======================
  tc_fence_before();
  if constexpr (kPair) {
    cluster_sync_all();  // no CTA leaves while its peer's MMAs may still touch its memory
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, 512);
    else
      tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0 && ctl->abort_flag && p.status_dev) atomicExch(p.status_dev, KGW_ERR_TIMEOUT);
}



// =============================================================================================
// Launchers
// =============================================================================================

cudaError_t launch_plan_mgrouped(const PlanParams& p, cudaStream_t s) {
  plan_mgrouped_kernel<<<1, PLAN_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_plan(const PlanParams& p, const MapTemplates& t, cudaStream_t s) {
  int threads = ((p.E + 31) / 32) * 32;
  threads = threads < 128 ? 128 : (threads > PLAN_THREADS ? PLAN_THREADS : threads);
  plan_kernel<<<1, threads, 0, s>>>(p, t);
  return cudaGetLastError();
}

template <bool kFp8, bool kPair, bool kAK, bool kBK, bool kMG = false, bool kFp4 = false, bool kNv = false,
          bool kWideK = false>
static cudaError_t launch_main(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                               cudaStream_t s) {
  auto kernel = wgrad_kernel<kFp8, kPair, kAK, kBK, kMG, kFp4, kNv, kWideK>;
  size_t smem = main_smem_bytes(kPair, kFp8, kNv, kFp4, kWideK);
  // the K-grouped FP8 kernel also hosts the promotion path, which lays out the same memory its own way
  if (kFp8 && !kFp4 && !kMG && promote_smem_bytes() > smem) smem = promote_smem_bytes();
  // set on every launch: the attribute is per device and the call is cheap
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kFp8 ? NUM_THREADS_FP8 : NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start launching while the plan kernel runs; griddepcontrol.wait orders the reads
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, p, tmA, tmB);
}

// One instantiation per operand storage order (K-major A / K-major B), chosen at run time.
template <bool kFp8, bool kPair, bool kWideK = false>
static cudaError_t launch_orders(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                                 cudaStream_t s) {
  if (p.a_kmajor && !p.b_kmajor) return launch_main<kFp8, kPair, true, false, false, false, false, kWideK>(p, tmA, tmB, grid, s);
  if (!p.a_kmajor && !p.b_kmajor) return launch_main<kFp8, kPair, false, false, false, false, false, kWideK>(p, tmA, tmB, grid, s);
  if (p.a_kmajor && p.b_kmajor) return launch_main<kFp8, kPair, true, true, false, false, false, kWideK>(p, tmA, tmB, grid, s);
  return launch_main<kFp8, kPair, false, true, false, false, false, kWideK>(p, tmA, tmB, grid, s);
}

cudaError_t launch_main_bf16(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                             cudaStream_t s) {
  if (p.tile_m == 2 * BM && p.wide_k) return launch_orders<false, true, true>(p, tmA, tmB, grid, s);
  if (p.tile_m == 2 * BM) return launch_orders<false, true>(p, tmA, tmB, grid, s);
  return launch_orders<false, false>(p, tmA, tmB, grid, s);
}

cudaError_t launch_main_mgrouped(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                                 cudaStream_t s) {
  if (p.fp8) {
    if (p.b_kmajor) return launch_main<true, false, true, true, true>(p, tmA, tmB, grid, s);
    return launch_main<true, false, true, false, true>(p, tmA, tmB, grid, s);
  }
  if (p.tile_m == 2 * BM && p.wide_k) {
    if (p.b_kmajor) return launch_main<false, true, true, true, true, false, false, true>(p, tmA, tmB, grid, s);
    return launch_main<false, true, true, false, true, false, false, true>(p, tmA, tmB, grid, s);
  }
  if (p.tile_m == 2 * BM) {
    if (p.b_kmajor) return launch_main<false, true, true, true, true>(p, tmA, tmB, grid, s);
    return launch_main<false, true, true, false, true>(p, tmA, tmB, grid, s);
  }
  if (p.b_kmajor) return launch_main<false, false, true, true, true>(p, tmA, tmB, grid, s);
  return launch_main<false, false, true, false, true>(p, tmA, tmB, grid, s);
}

cudaError_t launch_main_fp8(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                            cudaStream_t s) {
  if (p.tile_m == 2 * BM) return launch_orders<true, true>(p, tmA, tmB, grid, s);
  return launch_orders<true, false>(p, tmA, tmB, grid, s);
}

cudaError_t launch_main_fp4(const MainParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                            cudaStream_t s) {
  if (p.nvfp4 && p.tile_m == 2 * BM) return launch_main<true, true, true, true, false, true, true>(p, tmA, tmB, grid, s);
  if (p.nvfp4) return launch_main<true, false, true, true, false, true, true>(p, tmA, tmB, grid, s);
  if (p.tile_m == 2 * BM && p.wide_k)
    return launch_main<true, true, true, true, false, true, false, true>(p, tmA, tmB, grid, s);
  if (p.tile_m == 2 * BM) return launch_main<true, true, true, true, false, true>(p, tmA, tmB, grid, s);
  return launch_main<true, false, true, true, false, true>(p, tmA, tmB, grid, s);
}

bool fp8_supported() { return true; }

}  // namespace kgw
