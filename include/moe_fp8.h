/*
 * moe_fp8.h -- C ABI of the block-FP8 mixture-of-experts layer forward on one GB300 (sm_103a).
 *
 * The layer (composite of three pages on the subject):
 *   routing alignment into per-expert prefix-sum endpoints
 *     (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose;
 *      TensorRT-LLM "Triton FP8-activation MoE for decode-sized batches on Hopper", description)
 *   -> per-1x128 FP8 E4M3 activation quantization
 *     (TensorRT-LLM page, description; vLLM "per-layer activation scale format + fused SiLU+quant", Details)
 *   -> FC1 (gate+up) grouped FP8 x FP8 GEMM with 128x128 weight block scales
 *   -> SwiGLU (optionally clamped) fused with the 1x128 requantization of the FC2 input
 *   -> FC2 grouped GEMM, BF16 per-pair output
 *   -> routing-weighted top-k unpermute/sum (TensorRT-LLM page, rounding-fix commit).
 *
 * Conventions (every entry point):
 *   - All tensor arguments are DEVICE pointers owned by the caller. The library allocates no
 *     memory, never synchronizes the host (except moe_last_device_status), and issues all work on
 *     the given stream, so a whole forward can be captured in a CUDA graph.
 *   - Arguments are validated on the host before anything is launched; a failed check returns a
 *     status and launches nothing.  A CUDA launch error returns MOE_ERR_CUDA.
 *   - Row-major layouts; "K-major" weights store each output row's K values contiguously.
 *   - Token count: d_num_tokens, when not NULL, is a device int32 holding the number of live tokens
 *     n (clamped to [0, M_cap]); rows t >= n of x, topk_ids and topk_weights are never read and rows
 *     t >= n of out are never written (vLLM padded-work page, SM100 section: GPU token-count
 *     metadata).  NULL means n = M_cap.
 *   - Expert ids outside [0, E) (including -1) are dropped: such pairs get no workspace row and add
 *     nothing to the output.
 *   - Workspace rows outside the live part of each expert segment are never written.
 *   - Every device-side wait is bounded; on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT in the
 *     workspace status word and exits (read it with moe_last_device_status).
 *
 * Shapes: E experts, H hidden, I intermediate per expert, k = topk, M_cap token capacity,
 * P_cap = M_cap * k pairs, R_cap workspace rows (moe_ws_plan.R_cap).
 * Supported: H % 128 == 0, I % 128 == 0, 128 <= H <= 32768, 128 <= I <= 16384, 1 <= k <= 16,
 * 1 <= E <= 1024, 0 <= M_cap, M_cap * k <= 2^20.  Pointers: 16-byte aligned; workspace 256-byte aligned.
 */
#ifndef MOE_FP8_H_
#define MOE_FP8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* NULL or misaligned pointer, bad enum, negative size */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* shape outside the supported set above */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < moe_workspace_bytes(...) */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5       /* a bounded device-side wait expired (read from the workspace) */
} moe_status;

/* Scale formats (vLLM per-layer scale page, Overview and Details; vLLM padded-work page, Purpose):
 * FP32      -- fp32 scales, amax/448 (floored at 1/(448*512)).
 * FP32_POW2 -- fp32 scales rounded up to a power of two.
 * UE8M0     -- one byte b per scale, value 2^(b-127) (power of two, rounded up).
 * Weight scales are either FP32 (FP32_POW2 stores the same way) or UE8M0 bytes. */
typedef enum { MOE_SCALE_FP32 = 0, MOE_SCALE_FP32_POW2 = 1, MOE_SCALE_UE8M0 = 2 } moe_scale_fmt;

/* SwiGLU clamp (TensorRT-LLM page, test coverage: no clamp, clamp, clamp after SiLU):
 * BEFORE_SILU: gate <- min(gate, L), up <- clamp(up, -L, L), then SiLU(gate) * up.
 * AFTER_SILU:  min(SiLU(gate), L) * clamp(up, -L, L). */
typedef enum { MOE_CLAMP_NONE = 0, MOE_CLAMP_BEFORE_SILU = 1, MOE_CLAMP_AFTER_SILU = 2 } moe_clamp_mode;

/* Quantizer / epilogue numerics.
 * DIVIDE (default; vLLM "per-layer activation scale format + fused SiLU+quant", Details):
 *   codes = RNE_satfinite(x / s), s = max(RN(amax/448), RN(1/(448*512))); SwiGLU output in fp32.
 * RECIPROCAL (TensorRT-LLM "Triton FP8-activation MoE for decode-sized batches on Hopper",
 *   rounding-fix commit: the fused op's rounding): with fp32 scales, inv = min(RN(448/amax), 448*512),
 *   codes = RNE_satfinite(RN(x * inv)), stored scale s = RN(1/inv); the SwiGLU output is rounded to
 *   BF16 before its quantization.  Power-of-two scale formats quantize the same way in both modes. */
typedef enum { MOE_NUMERICS_DIVIDE = 0, MOE_NUMERICS_RECIPROCAL = 1 } moe_numerics;

/* Byte offsets of the workspace sub-buffers (all 256-byte aligned) and derived sizes.
 * Layout of each sub-buffer:
 *   status       int32        device status word (0 = ok, else a moe_status)
 *   num_tiles    int32        number of live 128-row tiles
 *   seg_start    int32[E+1]   expert segment starts (multiples of 128); seg_start[E] = rows used
 *   live_end     int32[E]     seg_start[e] + count of expert e
 *   sorted_pair  int32[R_cap] pair index p = t*k + j of each live row (padding rows not written)
 *   pair_row     int32[P_cap] workspace row of each pair p < n*k, -1 when dropped
 *   tile_expert  int32[T_cap] expert of row tile i (rows [128 i, 128 i + 128)), i < num_tiles
 *   num_chunks   int32        number of live 32-row chunks (small-batch schedule)
 *   chunk_row0   int32[C_cap] first row of each live 32-row chunk (chunks never cross a segment)
 *   align_hist   int32[align_ctas][E] per-CTA expert counts of the multi-CTA alignment
 *   a1_q         uint8[R_cap][H]       FC1 input, E4M3 codes
 *   a1_s         [H/128][R_cap]        FC1 input scales, column-major (fp32, or uint8 for UE8M0)
 *   a2_q         uint8[R_cap][I]       FC2 input, E4M3 codes
 *   a2_s         [I/128][R_cap]        FC2 input scales, column-major (fp32 or uint8)
 *   y            bf16[R_cap][H]        FC2 output per pair row (routing weights not applied)
 *   g1           bf16[R_cap][2I]       FC1 outputs (gate | up) of the 128-row-tile schedule with
 *                                      fp32 activation scales, where SwiGLU + requantization run as
 *                                      their own kernel; 0 when the plan has none
 *   splitk       fp32 partial sums and int32 tile counters of the split-K FC1 schedule */
typedef struct {
  size_t status, num_tiles, seg_start, live_end, sorted_pair, pair_row, tile_expert;
  size_t num_chunks, chunk_row0, align_hist;
  size_t a1_q, a1_s, a2_q, a2_s, y, g1, splitk_partial, splitk_count;
  size_t total_bytes;
  int32_t R_cap;   /* workspace rows: roundup(P_cap + min(E, P_cap) * 127, 128) */
  int32_t T_cap;   /* R_cap / 128 */
  int32_t C_cap;   /* R_cap / 32 */
  int32_t P_cap;   /* M_cap * k */
  int32_t fc1_ksplit;  /* K-split factor the forward uses for FC1 (1 = none) */
  int32_t small_batch; /* 1: the GEMMs run the small-batch schedule (32-row chunks, tokens on the
                          MMA's N side); chosen when P_cap <= 16 * E */
  int32_t align_ctas;  /* CTAs of the alignment (1 up to 4096 pairs, then one per 1024 pairs, <= 152) */
} moe_ws_plan;

/* Workspace plan for a layer shape; returns MOE_OK or a validation status. */
moe_status moe_workspace_plan(int M_cap, int E, int H, int I, int topk, moe_scale_fmt act_fmt,
                              moe_ws_plan* plan);

/* Bytes of workspace moe_fp8_block_forward needs (0 if the shape is unsupported). */
size_t moe_workspace_bytes(int M_cap, int E, int H, int I, int topk, moe_scale_fmt act_fmt);

/* Routing alignment (vLLM padded-work page, Purpose: "the shared permutation helper produces expert
 * endpoints"; TensorRT-LLM page: single-program moe_align).
 * Stable counting sort of the valid pairs p = t*k + j (t < n) by expert; expert e's segment starts at
 * seg_start[e] (exclusive prefix sum of counts rounded up to 128) and its live rows end at
 * live_end[e]; inside a segment pairs keep ascending p.  Writes, for p < n*k, pair_row[p] (row or -1)
 * and, for live rows, sorted_pair[row] = p; tile_expert[i] for every 128-row tile i < num_tiles;
 * chunk_row0[c] for every live 32-row chunk c < num_chunks.
 * expert_offset: the call holds experts [expert_offset, expert_offset + E) of a larger set (an
 * expert-parallel slice; 0 for a whole layer): ids are rebased by the offset, the others dropped.
 * Also resets the workspace status word.  Runs as one CTA up to 4096 pairs of capacity; above that
 * as a per-CTA counting kernel followed by a placement kernel (same result, bit for bit).
 * topk_ids: int32 [M_cap, topk]; all outputs are sub-buffers of the workspace of the same plan. */
moe_status moe_align(const int32_t* topk_ids, const int32_t* d_num_tokens, int M_cap, int topk, int E,
                     int expert_offset, int H, int I, moe_scale_fmt act_fmt, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream);

/* Per-1x128 activation quantization scattered to the aligned workspace (vLLM per-layer scale page,
 * Details: scale = max(amax/448, 1/(448*512)), codes = RNE_satfinite(x/scale) with IEEE division;
 * power-of-two formats round the scale up).  For each live token t < n and 128-group g of H, the
 * codes go to a1_q[row][g*128 ...] and the scale to a1_s[g][row] for every row = pair_row[t*k+j] >= 0.
 * x: bf16 [M_cap, H].  Requires moe_align on the same workspace first (same stream). */
moe_status moe_quant_act(const void* x_bf16, const int32_t* d_num_tokens, int M_cap, int E, int H,
                         int I, int topk, moe_scale_fmt act_fmt, moe_numerics numerics,
                         void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Problem statement of one layer call. */
typedef struct {
  const void* x;               /* bf16 [M_cap, H] */
  const int32_t* topk_ids;     /* int32 [M_cap, topk] */
  const float* topk_weights;   /* fp32 [M_cap, topk] */
  const int32_t* d_num_tokens; /* device int32 n, or NULL for n = M_cap */
  const void* w13;             /* E4M3 [E, 2I, H]: rows [0, I) gate, [I, 2I) up, K-major */
  const void* s13;             /* [E, 2I/128, H/128] fp32, or uint8 UE8M0 */
  const void* w2;              /* E4M3 [E, H, I], K-major */
  const void* s2;              /* [E, H/128, I/128] fp32, or uint8 UE8M0 */
  void* out;                   /* bf16 [M_cap, H]; rows t >= n untouched */
  int M_cap, E, H, I, topk;
  moe_scale_fmt weight_scale_fmt; /* FP32 (or FP32_POW2, same storage) or UE8M0 */
  moe_scale_fmt act_scale_fmt;    /* FP32, FP32_POW2 or UE8M0 */
  moe_clamp_mode clamp_mode;
  float clamp_limit;              /* L >= 0 when clamp_mode != NONE */
  moe_numerics numerics;          /* quantizer / epilogue numerics (DIVIDE by default) */
  /* Expert-parallel slice (TensorRT-LLM page, review of expert-parallel masking: drop ids outside
   * [0, E) instead of computing them with zero weight): the weights hold experts
   * [expert_offset, expert_offset + E) of a larger set; other ids are dropped.  0 for a whole layer. */
  int expert_offset;
  /* 0: out is BF16.  1: out is fp32 [M_cap, H], the unrounded top-k sum, so that expert-parallel
   * ranks can add their partial outputs and round to BF16 once. */
  int out_fp32;
} moe_fwd_args;

/* FC1 grouped GEMM over live 128-row tiles with the SwiGLU + 1x128 requantization epilogue
 * (vLLM padded-work page, Purpose: the prefix-sum scheduler visits only live tiles and the fused
 * activation quantization consumes the same endpoints; TensorRT-LLM page, human review: the scale
 * product a_scale*b_scale is formed before it multiplies the partial sum).
 * For each live row r of expert e and output column c:
 *   acc = sum over 128-wide K blocks kb of  p_kb * (a1_s[kb][r] * s13[e][c/128][kb])
 * with p_kb the FP8 dot of the block in fp32; g1 = bf16(acc); h = SwiGLU(gate, up) in fp32 with the
 * clamp; then a2_q / a2_s = 1x128 quantization of h.  Reads a1_q/a1_s, writes a2_q/a2_s.
 * Uses args->w13, s13, M_cap, E, H, I, topk, formats, clamp. */
moe_status moe_fc1_swiglu_quant(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream);

/* FC2 grouped GEMM over live tiles: y[r][c] = bf16(sum_kb p_kb * (a2_s[kb][r] * s2[e][c/128][kb])).
 * Routing weights are not applied here (TensorRT-LLM page, rounding-fix commit). */
moe_status moe_fc2(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                   moe_stream_t stream);
/*   For routed layers on the 128-row tiles with UE8M0 weight and activation scales, FC2 also checks,
 *   per row tile, that moe_fc1_swiglu_quant has run since the last moe_align (FC1 counts its
 *   finished items per tile; inside moe_fp8_block_forward those counts let FC2 start on finished
 *   tiles before the FC1 grid ends).  Called without that FC1, its bounded wait runs out after 1 s
 *   and the status word reads MOE_ERR_DEVICE_TIMEOUT. */

/* Top-k weighted unpermute/sum: out[t] = bf16( sum_j fp32(w[t,j] * y[pair_row[t*k+j]]) ), j ascending,
 * fp32 multiply and add rounded separately, dropped pairs skipped; rows t < n only. */
moe_status moe_topk_reduce(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream);

/* The whole layer: moe_align -> moe_quant_act -> moe_fc1_swiglu_quant -> moe_fc2 -> moe_topk_reduce,
 * all on `stream`, no host synchronization. */
moe_status moe_fp8_block_forward(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream);

/* Size of the library-owned scratch array used by moe_fp8_block_forward_static (32 MiB). */
#define MOE_STATIC_SCRATCH_BYTES (32u << 20)

/* The whole layer without a caller workspace and without any allocation.  The pages have no
 * counterpart: this is for callers that cannot allocate device memory when they run the layer (a
 * runtime that owns a fixed memory arena, a latency-critical loop that must not risk the device
 * synchronisation cudaMalloc/cudaFree can cause, plugin code that only receives input and output
 * pointers).  Same arguments and results as moe_fp8_block_forward; the workspace is a fixed
 * MOE_STATIC_SCRATCH_BYTES array inside the library, present on every GPU that loads the library
 * until the process exits.
 *  - Layers whose moe_workspace_bytes(...) exceeds MOE_STATIC_SCRATCH_BYTES are rejected with
 *    MOE_ERR_WORKSPACE_TOO_SMALL before anything is launched (e.g. single-token decode fits; the
 *    32-token, 288-expert decode layer does not).
 *  - The first call in a context looks up the array's device address (cudaGetSymbolAddress) with
 *    that device current, and caches it with the context's id; make that first call before any
 *    stream capture.  After a device reset (a new context) the next call looks the address up again.
 *  - All calls on a device share the array and it keeps the last call's contents; the state that
 *    must start at zero is reset on the GPU by every call.  Calls that overlap on the GPU (other
 *    streams or host threads) race on the array: serialise them.
 *  - The device status word of these calls is not readable through moe_last_device_status, so a
 *    device-side wait that runs out (MOE_ERR_DEVICE_TIMEOUT on the other entry points) is not
 *    reported by this path: the call has already returned MOE_OK and `out` holds wrong values.
 *    Callers that need that report use moe_fp8_block_forward with a workspace. */
moe_status moe_fp8_block_forward_static(const moe_fwd_args* args, moe_stream_t stream);

/* Batched-expert layout (vLLM per-layer scale page, Details, batched experts: per-expert rows with
 * masked counts, no host-side count reads).  x and out are [E, max_m, H] BF16; expert e's live rows
 * are r < counts[e] (device int32 [E], clamped to [0, max_m]); rows r >= counts[e] of out are never
 * written.  The layer runs per expert without routing: out[e, r] = FC2(SwiGLU-requant(FC1(
 * quant(x[e, r])))) in BF16 -- the dispatch and the weighted combine happen outside (e.g. in an
 * expert-parallel exchange).  max_m must be a multiple of 128; E * max_m <= 2^20. */
typedef struct {
  const void* x;               /* bf16 [E, max_m, H] */
  const int32_t* d_counts;     /* device int32 [E] */
  const void* w13;             /* E4M3 [E, 2I, H] */
  const void* s13;             /* [E, 2I/128, H/128] fp32 or UE8M0 */
  const void* w2;              /* E4M3 [E, H, I] */
  const void* s2;              /* [E, H/128, I/128] */
  void* out;                   /* bf16 [E, max_m, H] */
  int E, max_m, H, I;
  moe_scale_fmt weight_scale_fmt, act_scale_fmt;
  moe_clamp_mode clamp_mode;
  float clamp_limit;
  moe_numerics numerics;
} moe_batched_args;

/* Workspace bytes of moe_fp8_batched_forward (0 if the shape is unsupported). */
size_t moe_batched_workspace_bytes(int E, int max_m, int H, int I, moe_scale_fmt act_fmt);

/* The batched-expert layer on `stream`; same numerics and status conventions as the routed forward. */
moe_status moe_fp8_batched_forward(const moe_batched_args* args, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream);

/* Reads the workspace status word (synchronizes `stream` first).  MOE_OK or MOE_ERR_DEVICE_TIMEOUT. */
moe_status moe_last_device_status(const void* workspace, moe_stream_t stream);

/* Diagnostic of the bounded device-side waits.  Launches one CTA on `stream` that waits, with the
 * helper every TMA/MMA pipeline of the library uses, for an mbarrier phase that nothing completes,
 * and gives up after `limit_us` microseconds (1 to 1000000).  The expiry is recorded as in the layer
 * kernels: the workspace status word (its first int32) becomes MOE_ERR_DEVICE_TIMEOUT unless it
 * already holds an error, and moe_last_device_status returns it.  The kernel then returns normally
 * and the context stays usable; the next layer call's alignment resets the word.  Nothing else in
 * the workspace is touched.  MOE_ERR_INVALID_ARG for a null or not 256-byte-aligned workspace or a
 * limit out of range; MOE_ERR_CUDA if the launch fails. */
moe_status moe_selftest_wait_timeout(void* workspace, int limit_us, moe_stream_t stream);

/* Human-readable name of a status. */
const char* moe_status_str(moe_status status);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP8_H_ */
