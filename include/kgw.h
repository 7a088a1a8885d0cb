/*
 * kgw.h — K-grouped GEMM for Mixture-of-Experts weight gradients on sm_103a (GB300).
 *
 * Operation ("Grouped GEMM + WGrad (Unified)", section "Operation"): for expert e let
 * begin = 0 when e == 0 and begin = offsets[e-1] otherwise, and end = offsets[e]; then
 *
 *     Wgrad[e] = A[:, begin:end] @ B[begin:end, :]
 *
 * with A = dY^T of shape [hidden, tokens_sum] and B = X of shape [tokens_sum, intermediate]
 * ("05 · Grouped GEMM 与 Expert 计算", section 5.2: dW_i = dY_i^T X_i, the token axis is the
 * ragged contraction axis, M and N are fixed). With accumulate != 0 the result is added to the
 * existing output (the caller initialises it); with accumulate == 0 the output is overwritten
 * and an empty expert produces zeros.
 *
 * Conventions shared by every entry point:
 *  - Every pointer in kgw_wgrad_args except status_dev and the host-side struct itself is a
 *    DEVICE pointer on the current CUDA device. The caller owns every buffer (inputs, offsets,
 *    outputs, the per-expert pointer array, the workspace) and keeps it alive until the work
 *    enqueued on `stream` completes. The library allocates nothing per call and never
 *    synchronises the stream: offsets stay on the device and are validated there.
 *  - Host-detected errors return immediately and enqueue nothing.
 *  - Device-detected errors (malformed offsets, bad per-expert output pointers, a device wait
 *    that gave up) are written to *status_dev when status_dev is non-null; when the offsets or
 *    output pointers are malformed no output element is written.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *  - Two calls that share a workspace must be ordered on the GPU (same stream or events).
 *  - Results are bitwise deterministic run to run for the same inputs and device.
 */
#ifndef KGW_H_
#define KGW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kgw_status {
  KGW_OK = 0,
  KGW_ERR_INVALID_ARG = 1,   /* null/negative/inconsistent argument (host-detected) */
  KGW_ERR_UNSUPPORTED = 2,   /* layout, dtype or shape this build does not implement */
  KGW_ERR_ALIGNMENT = 3,     /* an operand or output base address is not 16-byte aligned */
  KGW_ERR_DEVICE = 4,        /* current device is not sm_103 (or no device) */
  KGW_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed */
  KGW_ERR_OFFSETS = 6,       /* device-detected: offsets decrease, a count % 256 != 0, or
                                offsets[E-1] != tokens_sum */
  KGW_ERR_TIMEOUT = 7,       /* device-detected: a bounded wait inside the kernel gave up */
  KGW_ERR_WORKSPACE = 8,     /* workspace null, misaligned or smaller than the minimum */
  KGW_ERR_OUT_PTRS = 9,      /* device-detected: an out_ptrs[e] is null or not 16-byte aligned */
  KGW_ERR_SCRATCH_LIMIT = 10, /* kgw_wgrad_bf16_noalloc: the call exceeds its static scratch limits */
  KGW_ERR_SCALES = 11        /* device-detected: an FP32 scale is NaN or infinite, a packed UE8M0
                                byte is 0xFF, a UE4M3 byte has its top bit set or is 0x7F, or (the
                                M-grouped FP8 entry) an FP32 scale is not a power of two; the output
                                of that call is meaningless */
} kgw_status;

/* Storage order of an operand ("Grouped GEMM + WGrad (Unified)", section "BF16 contract"). */
typedef enum kgw_major {
  KGW_K_MAJOR = 0,   /* token axis has unit stride: A stride (tokens_sum, 1)             */
  KGW_MN_MAJOR = 1   /* hidden / intermediate axis has unit stride: B stride (intermediate, 1) */
} kgw_major;

/* How the token dimension is stored (section "BF16 contract", input_order). */
typedef enum kgw_input_order {
  KGW_TENSOR2D = 0,  /* one global 2-D tensor per operand */
  KGW_RAGGED = 1     /* per-expert blocks concatenated in memory, expert e's block starting at element
                        begin_e*hidden (A) or begin_e*intermediate (B) and keeping the operand's
                        unit-stride axis: K-major A [hidden, n_e], M-major A [n_e, hidden], N-major
                        B [n_e, intermediate], K-major B [intermediate, n_e] (row-major each) */
} kgw_input_order;

/* Output element type (section "BF16 contract": BF16, FP16 or FP32 outputs); FP32 accumulation,
   one rounding to the output type (FP16 overflows to infinity beyond 65504). */
typedef enum kgw_out_dtype { KGW_OUT_F32 = 0, KGW_OUT_BF16 = 1, KGW_OUT_F16 = 2 } kgw_out_dtype;

typedef struct kgw_wgrad_args {
  int32_t num_experts;      /* E >= 1 (<= 4096)                                              */
  int32_t hidden;           /* M: multiple of 128                                            */
  int32_t intermediate;     /* N: multiple of 256                                            */
  int64_t tokens_sum;       /* total tokens; must equal offsets[E-1]; multiple of 256        */
  const void* a;            /* A: bf16 (or e4m3) [hidden, tokens_sum], see a_major/input_order */
  int32_t a_major;          /* KGW_K_MAJOR: stored [hidden, tokens_sum] (token stride 1);
                               KGW_MN_MAJOR: stored [tokens_sum, hidden] (hidden stride 1), e.g.
                               dY kept token-major; ragged: per-expert [n_e, hidden] blocks      */
  const void* b;            /* B: bf16 (or e4m3) [tokens_sum, intermediate]                 */
  int32_t b_major;          /* KGW_MN_MAJOR: stored [tokens_sum, intermediate];
                               KGW_K_MAJOR: stored [intermediate, tokens_sum] (token stride 1);
                               ragged K-major: per-expert [intermediate, n_e] blocks            */
  const int32_t* offsets;   /* int32 [E]: non-decreasing cumulative token counts             */
  int32_t input_order;      /* kgw_input_order                                               */
  void* out;                /* dense output [E, hidden, intermediate] row-major, or NULL     */
  const int64_t* out_ptrs;  /* int64 [E] device addresses of per-expert [hidden, intermediate]
                               row-major outputs (discrete mode), or NULL; exactly one of out
                               and out_ptrs is non-NULL (section "Output modes")              */
  int32_t out_dtype;        /* kgw_out_dtype                                                 */
  int32_t accumulate;       /* 0: overwrite (empty expert -> zeros); 1: out += result         */
  int32_t* status_dev;      /* optional device int32 receiving device-detected kgw_status    */
} kgw_wgrad_args;

/*
 * Workspace bytes needed by kgw_wgrad_bf16 (is_fp8 = 0) or by the block-scaled entries
 * (is_fp8 = 1: FP8, FP4 and NVFP4) for these shapes. Depends only on num_experts, hidden,
 * intermediate and tokens_sum (not on the offsets' values). Host-only; never touches the GPU.
 * The workspace holds the per-call schedule of the dynamic persistent scheduler ("Grouped GEMM +
 * WGrad (Unified)", section "Scheduling, cache, and errors"), for block-scaled calls on CTA pairs
 * (hidden % 256 == 0) the scale factors prepared in TMEM order, and the FP32 partial tiles of
 * split-K; a caller may pass less than this (down to the schedule and the prepared scale
 * factors) and the kernel then splits less. Errors as for the calls it sizes (KGW_ERR_INVALID_ARG,
 * KGW_ERR_UNSUPPORTED, KGW_ERR_ALIGNMENT); *bytes is written only on KGW_OK.
 */
kgw_status kgw_workspace_size(const kgw_wgrad_args* args, int32_t is_fp8, size_t* bytes);

/*
 * BF16 x BF16 -> FP32 accumulation -> FP32 or BF16 output
 * ("Grouped GEMM + WGrad (Unified)", sections "Operation", "BF16 contract", "Output modes").
 * a, b: bf16. There are no scale arguments: the BF16 path takes none.
 * workspace: device buffer of workspace_bytes (256-byte aligned), owned by the caller.
 * stream: cudaStream_t.
 */
kgw_status kgw_wgrad_bf16(const kgw_wgrad_args* args, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kgw_wgrad_bf16 without the 256-token contract on the counts (an extension beyond the pages'
 * "BF16 contract"): every per-expert count (and tokens_sum) must be a multiple of 8 when A or B
 * stores the token axis innermost (K-major; TMA coordinates start on 16 bytes) and may be any
 * count when both operands are MN-major. An expert's last pipeline stage is partly beyond its
 * last token: the kernel reads it through a per-expert TMA descriptor whose token extent ends at
 * end_e, so the rest of the stage is zero and the next expert's tokens are not read. Same
 * operation, layouts, outputs, workspace (kgw_workspace_size) and error reporting as
 * kgw_wgrad_bf16; a count that breaks the rule is KGW_ERR_OFFSETS on the device.
 */
kgw_status kgw_wgrad_bf16_unaligned(const kgw_wgrad_args* args, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * FP8 block-scaled variant ("05 · Grouped GEMM 与 Expert 计算", section 3: per-block 1x128
 * scaling along K, scales MN-major; "Grouped GEMM + WGrad (Unified)", section "Block-scaled
 * contract"). a, b: float8 e4m3 (the "fn" encoding) in the same logical layouts as the BF16
 * entry. sfa: float32 [tokens_sum/128, hidden], sfb: float32 [tokens_sum/128, intermediate]:
 * sfa[kb][m] scales A[m, 128*kb : 128*kb+128] and sfb[kb][n] scales B[128*kb : 128*kb+128, n]
 * (token blocks are global, also in ragged order). Any finite FP32 scale is accepted ("05 · ...",
 * section 3: x_scales float): when every scale of the call is a power of two in [2^-127, 2^127]
 * the scales are exact UE8M0 factors of the block-scaled MMA; otherwise each 128-token block's
 * unscaled partial product is formed on the tensor cores and sa*sb*partial is added to FP32 running
 * sums on the CUDA cores (the per-block promotion of the pages' FP8 GEMMs). A device-side check of
 * the scales chooses between the two, so the call stays asynchronous and capturable. A NaN or
 * infinite scale is KGW_ERR_SCALES. The product is accumulated in FP32 either way.
 */
kgw_status kgw_wgrad_fp8_blockscaled(const kgw_wgrad_args* args, const float* sfa, const float* sfb,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 variant with packed UE8M0 scales of 32-token granularity ("05 · Grouped GEMM 与 Expert 计算",
 * section 3: UE8M0 scale format, MN-major TMA-aligned scale tensors; "How to Use K-Grouped GEMM for
 * MoE Weight Backward Pass in DeepGEMM", step 2: gran_k = 32 with packed UE8M0). a, b: e4m3 as in
 * kgw_wgrad_fp8_blockscaled. sfa_packed: int32 [tokens_sum/128, hidden], sfb_packed: int32
 * [tokens_sum/128, intermediate]; byte j (least significant first) of sfa_packed[kb][m] is the
 * biased exponent e of the scale 2^(e-127) of A[m, 128*kb + 32*j : 128*kb + 32*j + 32] (likewise
 * for B and column n). The byte 0xFF (NaN) is reported as KGW_ERR_SCALES. Each 32-token block's
 * scale is applied to its products before FP32 accumulation.
 */
kgw_status kgw_wgrad_fp8_ue8m0(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP4 block-scaled variant ("How to Use K-Grouped GEMM for MoE Weight Backward Pass in DeepGEMM",
 * steps 1-2: both operands cast to FP4 with the same gran_k = 32; "Grouped GEMM + WGrad (Unified)",
 * the legacy block-scaled backend selected by a matching FP4 operand pair). a, b: e2m1 (1 sign,
 * 2 exponent bits with bias 1, 1 mantissa bit; values 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte
 * along the token axis with the earlier token in the low nibble. Both operands K-major: A stored
 * [hidden, tokens_sum/2] bytes, B stored [intermediate, tokens_sum/2] bytes (a_major = b_major =
 * KGW_K_MAJOR; MN-major is KGW_ERR_UNSUPPORTED: the packed-FP4 MMA reads K-major operands only);
 * ragged input order: expert e's blocks are [hidden, n_e/2] and [intermediate, n_e/2] bytes at
 * byte offsets begin_e*hidden/2 and begin_e*intermediate/2. Scales as in
 * kgw_wgrad_fp8_ue8m0 (packed UE8M0 words, one byte per 32 tokens). Workspace as for FP8
 * (kgw_workspace_size with is_fp8 = 1).
 */
kgw_status kgw_wgrad_fp4_ue8m0(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * NVFP4 variant: the block-scaled contract with scale blocks of 16 tokens and per-tensor global
 * scales ("Grouped GEMM + WGrad (Unified)", sections "BF16 contract" -- sf_vec_size 16 -- and
 * "Block-scaled contract": sfa/sfb plus global_scale_a / global_scale_b where the low-precision
 * format requires them). a, b: e2m1 packed as in kgw_wgrad_fp4_ue8m0 (K-major A and B, tensor2d or
 * ragged). sfa_packed: int32 [tokens_sum/64, hidden], sfb_packed: int32 [tokens_sum/64,
 * intermediate]; byte j (least significant first) of word [w][r] is the unsigned E4M3 scale
 * (UE4M3: 4 exponent bits with bias 7, 3 mantissa bits, no sign) of tokens 64w + 16j .. 64w + 16j + 15
 * of row / column r. A byte with its top bit set, or 0x7F (NaN), is KGW_ERR_SCALES on the device.
 * global_scale_a, global_scale_b: device pointers to one float each (NULL = 1), 4-byte aligned.
 *
 *     Wgrad[e][m][n] = global_scale_a * global_scale_b
 *                      * sum over tokens k of expert e of (sa[k/16][m] * a[m][k]) * (sb[k/16][n] * b[k][n])
 *
 * accumulated in FP32 (the global product multiplies the FP32 sum before the output rounding).
 * Counts: multiples of 256 (the pages' contract). Workspace: kgw_workspace_size with is_fp8 = 1.
 */
kgw_status kgw_wgrad_nvfp4(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                           const float* global_scale_a, const float* global_scale_b, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Block-scaled entries without the 256-token contract on the counts (an extension beyond the
 * pages' contract, like kgw_wgrad_bf16_unaligned). An expert's last pipeline stage may be partly
 * beyond its last token: it is read through a per-expert TMA descriptor whose token extent ends at
 * end_e, so the rest of the stage is zero and the next expert's tokens are not read.
 *
 * Scale blocks. "05 · Grouped GEMM 与 Expert 计算", section 4 (quantization padding) pads every
 * expert segment to the quantisation alignment before the FP8/FP4 cast, so every scale block lies
 * inside one expert. Here the operands are not padded but the scales keep that layout: expert e's
 * tokens are cut into 128-token blocks from its first token (the last one possibly partial), and
 * its blocks are scale rows r_e, r_e + 1, ..., r_e + ceil(n_e/128) - 1, with
 * r_e = sum over f < e of ceil(n_f / 128). sfa has sum_e ceil(n_e/128) rows of hidden entries,
 * sfb as many rows of intermediate entries. When every count is a multiple of 128 these are the
 * rows tokens/128 of the aligned entries (kgw_wgrad_fp8_blockscaled, kgw_wgrad_fp8_ue8m0,
 * kgw_wgrad_fp4_ue8m0), which follow the same rule.
 *
 * kgw_wgrad_fp8_unaligned: e4m3 operands in any storage order and input order of kgw_wgrad_bf16.
 * sf_format 0: FP32 powers of two, one per 128-token block (as kgw_wgrad_fp8_blockscaled);
 * sf_format 1: packed UE8M0 words, byte j scaling tokens 32j..32j+31 of the block (as
 * kgw_wgrad_fp8_ue8m0); any other value is KGW_ERR_INVALID_ARG. Counts (and tokens_sum) must be
 * multiples of 16 when A or B is K-major (a TMA coordinate along the innermost axis starts on 16
 * bytes), any count when both are MN-major.
 * kgw_wgrad_fp4_unaligned: e2m1 operands as in kgw_wgrad_fp4_ue8m0 (K-major A and B, either
 * input order); counts multiples of 32 (16 packed bytes).
 * A count that breaks the rule is KGW_ERR_OFFSETS on the device (nothing written). Workspace:
 * kgw_workspace_size with is_fp8 = 1. Everything else as for the aligned entries.
 */
kgw_status kgw_wgrad_fp8_unaligned(const kgw_wgrad_args* args, const void* sfa, const void* sfb, int32_t sf_format,
                                   void* workspace, size_t workspace_bytes, void* stream);
kgw_status kgw_wgrad_fp4_unaligned(const kgw_wgrad_args* args, const int32_t* sfa_packed, const int32_t* sfb_packed,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * kgw_wgrad_bf16 without a workspace argument and without any device allocation.
 *
 * The paper has no counterpart to this entry point. It exists for callers that cannot allocate
 * device memory at the point of the call: for example code running under a framework
 * whose caching allocator owns all device memory, inference runtimes that forbid allocation
 * after start-up, or a plug-in that receives only stream and tensor pointers. Such a caller
 * still passes the inputs and outputs in `args`, exactly as for kgw_wgrad_bf16.
 *
 * Scratch: the per-call schedule and the split-K partial tiles live in one static device array
 * of 2 MiB inside the library, which every GPU that loads the library keeps until the process
 * exits. It holds the schedule for up to 1024 experts plus a few FP32 partial tiles (13 to 15
 * of 128 x 256, or 6 to 7 of the 256 x 256 tiles used when hidden % 256 == 0, fewer the more
 * experts there are); calls with more than 1024 experts return KGW_ERR_SCRATCH_LIMIT and enqueue
 * nothing. An expert is split along its tokens only when all of its pieces fit: splitting needs at
 * least 2 * T partial tiles, with T = (hidden / tile rows) * (intermediate / 256) output tiles
 * per expert, so split-K is off once T exceeds 3 (256-row tiles) or 6 to 7 (128-row tiles), which
 * includes every full-size workload of this library's benchmarks; long experts then run unsplit,
 * which changes the load balance under skewed routing but not the results' error bound (the
 * summation order can differ from kgw_wgrad_bf16's).
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture. The address belongs to the device's current CUDA context: after a device reset, or
 * when the primary context is destroyed and created again, the next call sees a different
 * current context and looks the address up again (that call, too, should come before any stream
 * capture). No call allocates (no cudaMalloc/cudaFree, no allocating library routine).
 *
 * Sharing: every call on a device uses the same array and it keeps the previous call's
 * contents; the kernels re-initialise every counter they read, so nothing needs clearing by
 * the caller. Calls that overlap on the GPU (different streams without ordering, or several
 * host threads) race on the array and give wrong results: order them.
 */
kgw_status kgw_wgrad_bf16_noalloc(const kgw_wgrad_args* args, void* stream);

/*
 * M-grouped GEMM: the forward / dgrad GEMM of the same MoE layer ("05 · Grouped GEMM 与 Expert 计算",
 * sections 1, 2 and 5.1: only M varies between groups, N and K are fixed). Each group g multiplies
 * its own rows of A by its own weight B_g:
 *
 *     D[rows of g, :] (+)= A[rows of g, :] @ op(B_g)
 *
 * B is K-major [G, n, k] (forward, op(B_g) = B_g^T, the "nt" layout) or N-major [G, k, n]
 * (dgrad, op(B_g) = B_g). A and D are row-major with K resp. N contiguous. FP32 accumulation, one
 * rounding to the output type (kgw_out_dtype), overwrite or accumulate (D = D + result, one FP32
 * add before that rounding). Which rows belong to which group is given on the device, in one of
 * three layouts (section 2):
 *
 *   KGW_MG_OFFSETS    A [m, k], D [m, n]. groups = int32 [G] cumulative row counts (group g owns
 *                     rows [offsets[g-1], offsets[g]), offsets[-1] = 0): contiguous layout, every
 *                     count a multiple of 128 (a 128-row tile never spans two groups) and
 *                     offsets[G-1] == m. Counts of 0 are allowed.
 *   KGW_MG_INDICES    A [m, k], D [m, n]. groups = int32 [m] group id of every row (the pages'
 *                     m_indices): contiguous layout, every aligned 128-row block carries one id in
 *                     [0, G). Blocks need not be sorted by group.
 *   KGW_MG_MASKED     A [G, m, k], D [G, m, n] with m = max_m rows reserved per group. groups =
 *                     int32 [G] valid rows per group (masked_m, 0 <= masked_m[g] <= m): masked
 *                     layout (section 2.2). Only the first masked_m[g] rows of each group are
 *                     computed and written; the other rows of D are left untouched, and the
 *                     values in the unused rows of A do not matter.
 *
 * Device-detected violations of these rules set KGW_ERR_OFFSETS (in *status_dev when given) and
 * nothing is written. Conventions as for kgw_wgrad_bf16: device pointers, caller-owned buffers,
 * asynchronous on stream, no host synchronisation (CUDA-graph capturable), host-detected errors
 * returned before anything is enqueued. Constraints: n % 256 == 0, k % 64 == 0, 1 <= G <= 4096,
 * m % 128 == 0 for the contiguous layouts, A/B/D 16-byte aligned, fewer than 2^31 rows of A and
 * of B.
 */
typedef enum { KGW_MG_OFFSETS = 0, KGW_MG_INDICES = 1, KGW_MG_MASKED = 2 } kgw_mg_layout;

typedef struct kgw_mgrouped_args {
  int32_t num_groups;       /* G                                                              */
  int32_t layout;           /* kgw_mg_layout                                                  */
  int64_t m;                /* contiguous: rows of A and D; masked: rows reserved per group   */
  int32_t n;                /* columns of D                                                   */
  int32_t k;                /* contraction length                                             */
  const void* a;            /* bf16 A (see layout)                                            */
  const void* b;            /* bf16 [G, n, k] (KGW_K_MAJOR) or [G, k, n] (KGW_MN_MAJOR)       */
  int32_t b_major;          /* kgw_major                                                      */
  const int32_t* groups;    /* device int32: offsets [G], m_indices [m] or masked_m [G]       */
  void* d;                  /* output (see layout), dtype out_dtype                           */
  int32_t out_dtype;        /* kgw_out_dtype                                                  */
  int32_t accumulate;       /* 0: overwrite; 1: D += result                                   */
  int32_t* status_dev;      /* optional device int32 receiving device-detected kgw_status     */
} kgw_mgrouped_args;

/* Workspace bytes of kgw_mgrouped_bf16 (host-only; depends on G, m and the layout). */
kgw_status kgw_mgrouped_workspace_size(const kgw_mgrouped_args* args, size_t* bytes);

/* M-grouped BF16 GEMM (see kgw_mgrouped_args). workspace: 256-byte aligned device buffer. */
kgw_status kgw_mgrouped_bf16(const kgw_mgrouped_args* args, void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 M-grouped GEMM ("05 · Grouped GEMM 与 Expert 计算", section 2.1 names m_grouped_fp8_gemm_nt_contiguous
 * and, for the masked layout, m_grouped_fp8_gemm_nt_masked; section 3: FP8 operands with per-block
 * 1x128 scaling along K). a and b are float8 e4m3 ("fn") in the layouts of kgw_mgrouped_args.
 * sf_format 0: sfa float32 [k/128, rows of A] (rows of A = m, or G*m for the masked layout),
 * sfa[kb][r] scales A[r, 128*kb : 128*kb+128]; sfb float32 [G, k/128, n], sfb[g][kb][c] scales
 * column c of op(B_g) over the same K block; every scale a power of two. sf_format 1: the same
 * shapes as int32 words of four UE8M0 bytes, byte j scaling K 32j..32j+31 of the block (as in
 * kgw_wgrad_fp8_ue8m0). Products accumulate in FP32; k must be a multiple of 128. A bad scale is
 * reported as KGW_ERR_SCALES. Workspace: kgw_mgrouped_workspace_size.
 */
kgw_status kgw_mgrouped_fp8(const kgw_mgrouped_args* args, const void* sfa, const void* sfb, int32_t sf_format,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static storage; "KGW_ERR_UNKNOWN" for any other value). The
 * codes mirror the rejections listed in "Grouped GEMM + WGrad (Unified)", section "Scheduling,
 * cache, and errors" (unsupported dtypes or layouts, malformed offsets or pointers, devices below
 * SM100), plus the device-side bounded-wait and scale checks of this library. */
const char* kgw_status_string(int32_t status);

/* Library ABI version (major*100 + minor). */
int32_t kgw_version(void);

/*
 * Testing hooks (process-wide, host side). key 1: device wait limit in nanoseconds
 * (default 2e9); key 2: when >= 0, the TMA producer of CTA 0 skips the arrival of that
 * k-iteration so that the bounded wait path is exercised (default -1); key 3: non-zero runs every
 * call that would use 256-row CTA-pair tiles (K-grouped BF16, FP8, FP4 and NVFP4; M-grouped BF16)
 * on single-CTA 128-row tiles (default 0). Returns the previous value, or -1 for an unknown key.
 */
int64_t kgw_debug_set(int32_t key, int64_t value);

/*
 * Testing hook for the ragged input order: runs only the schedule kernel of a call (which builds
 * one TMA descriptor per non-empty expert on the device, from the expert's offset and token
 * count) for every K-major operand, then compares each descriptor byte for byte with one encoded
 * on the host for the same block (host_offsets: a host copy of args->offsets). Synchronises the
 * device. Returns the number of differing descriptors (0 = all identical) or -kgw_status on
 * error. host_dump, if non-NULL, receives E x 2 x 256 bytes: per expert and operand (A, B) the
 * device-built then the host-encoded descriptor. Allocates host memory only.
 */
int32_t kgw_debug_check_ragged_maps(const kgw_wgrad_args* args, int32_t is_fp8, const int32_t* host_offsets,
                                    void* workspace, size_t workspace_bytes, void* host_dump);

/* Testing hook: like kgw_debug_check_ragged_maps for every per-expert descriptor that
 * kgw_wgrad_bf16_unaligned builds (token extent cut at end_e for tensor2d K-major and for
 * MN-major operands; per-expert blocks for ragged K-major operands): runs the plan only and
 * returns how many differ from host encodings (negative kgw_status on error). host_dump as for
 * kgw_debug_check_ragged_maps. */
int32_t kgw_debug_check_tail_maps(const kgw_wgrad_args* args, const int32_t* host_offsets, void* workspace,
                                  size_t workspace_bytes, void* host_dump);

/* Testing hook: kgw_debug_check_tail_maps for the descriptors of kgw_wgrad_bf16_unaligned (kind 0),
 * kgw_wgrad_fp8_unaligned (kind 1) or kgw_wgrad_fp4_unaligned (kind 2; the token axis of a packed
 * FP4 descriptor counts bytes). Other kinds: -KGW_ERR_INVALID_ARG. */
int32_t kgw_debug_check_tail_maps_kind(const kgw_wgrad_args* args, int32_t kind, const int32_t* host_offsets,
                                       void* workspace, size_t workspace_bytes, void* host_dump);

#ifdef __cplusplus
}
#endif

#endif /* KGW_H_ */
