// Host side of the C ABI: argument validation, the workspace plan, TMA tensor maps and the launch
// sequence of one layer forward.  Nothing here allocates device memory or synchronizes the host
// (except moe_last_device_status, which exists to read the device status word).
#include <string.h>

#include <algorithm>
#include <mutex>

#include "moe_internal.h"

namespace moe {

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Small-batch schedule (tokens on the MMA's N side, 32-row chunks) when the average expert holds at
// most 16 rows; otherwise 128-row tiles.
static bool use_small_batch(int E, long long P_cap) { return P_cap > 0 && P_cap <= 16LL * E; }

// FC1 K-split of the small-batch schedule.  Splitting K costs a fix-up round trip per item, so it
// only pays when the occupied experts give too few work items to keep the SMs streaming: split until
// the estimated items (at most min(E, P_cap) experts x I/128 column blocks) reach half of a 152-SM
// part, keeping at least two K blocks per split and the fp32 partials under 256 MB.
static int choose_fc1_ksplit(int E, int H, int I, long long P_cap, bool small) {
  if (!small) return 1;
  const long long items = std::min<long long>(E, P_cap) * (I / kGroup);
  const int kb = H / kGroup;
  int ks = 1;
  while (ks < kMaxKSplit && items * ks < 76 && kb % (ks * 2) == 0 && kb / (ks * 2) >= 2 &&
         (long long)(ks * 2) * P_cap * 2 * I * 4 <= (256LL << 20))
    ks *= 2;
  return ks;
}

static moe_status check_shape(int M_cap, int E, int H, int I, int topk, int act_fmt) {
  if (M_cap < 0 || E <= 0 || H <= 0 || I <= 0 || topk <= 0) return MOE_ERR_INVALID_ARG;
  if (act_fmt < MOE_SCALE_FP32 || act_fmt > MOE_SCALE_UE8M0) return MOE_ERR_INVALID_ARG;
  if (H % kGroup || I % kGroup || H > 32768 || I > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (topk > kMaxTopk || E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)M_cap * topk > kMaxPairs) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

moe_status make_plan(int M_cap, int E, int H, int I, int topk, int act_fmt, Plan* plan) {
  const moe_status st = check_shape(M_cap, E, H, I, topk, act_fmt);
  if (st != MOE_OK) return st;
  memset(plan, 0, sizeof(*plan));
  moe_ws_plan& w = plan->ws;
  const long long P_cap = (long long)M_cap * topk;
  const long long pad_rows = P_cap + (long long)std::min<long long>(E, P_cap) * (kAlign - 1);
  const long long R_cap = (pad_rows + kAlign - 1) / kAlign * kAlign;
  w.P_cap = (int32_t)P_cap;
  w.R_cap = (int32_t)R_cap;
  w.T_cap = (int32_t)(R_cap / kAlign);
  w.C_cap = (int32_t)(R_cap / 32);
  w.small_batch = use_small_batch(E, P_cap) ? 1 : 0;
  w.fc1_ksplit = choose_fc1_ksplit(E, H, I, P_cap, w.small_batch != 0);
  const size_t sc = act_fmt == MOE_SCALE_UE8M0 ? 1 : 4;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  w.status = take(4);
  w.num_tiles = take(4);
  w.seg_start = take((size_t)(E + 1) * 4);
  w.live_end = take((size_t)E * 4);
  w.sorted_pair = take((size_t)R_cap * 4);
  w.pair_row = take((size_t)P_cap * 4);
  w.tile_expert = take((size_t)w.T_cap * 4);
  w.num_chunks = take(4);
  w.chunk_row0 = take((size_t)w.C_cap * 4);
  w.align_ctas = P_cap > 4096 ? (int32_t)std::min<long long>(152, (P_cap + 1023) / 1024) : 1;
  w.align_hist = take(w.align_ctas > 1 ? (size_t)w.align_ctas * E * 4 : 0);
  w.a1_q = take((size_t)R_cap * H);
  w.a1_s = take((size_t)(H / kGroup) * R_cap * sc);
  w.a2_q = take((size_t)R_cap * I);
  w.a2_s = take((size_t)(I / kGroup) * R_cap * sc);
  w.y = take((size_t)R_cap * H * 2);
  // the tile schedule with fp32 activation scales runs SwiGLU + requantization as its own kernel
  // on the BF16 FC1 outputs (UE8M0 layers keep it in the block-scaled GEMM's overlapped epilogue)
  w.g1 = (!w.small_batch && act_fmt != MOE_SCALE_UE8M0) ? take((size_t)R_cap * 2 * I * 2) : 0;
  w.splitk_partial = take(w.fc1_ksplit > 1 ? (size_t)w.fc1_ksplit * P_cap * 2 * I * 4 : 0);
  // int32 counters: per (chunk, column block) split arrivals of the split-K FC1, or per row tile the
  // FC1 items done, which the block-scaled FC2 waits on instead of the whole FC1 grid (tile schedule
  // with UE8M0 activation scales)
  w.splitk_count = take(w.fc1_ksplit > 1 ? (size_t)w.C_cap * (I / kGroup) * 4
                        : (!w.small_batch && act_fmt == MOE_SCALE_UE8M0) ? (size_t)w.T_cap * 4 : 0);
  w.total_bytes = off;
  plan->M_cap = M_cap;
  plan->E = E;
  plan->H = H;
  plan->I = I;
  plan->topk = topk;
  plan->act_fmt = act_fmt;
  return MOE_OK;
}

// ------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Byte matrix [outer][inner] seen as 3-D (x = 128 bytes of a K block, y = row, z = K block), boxes of
// box_outer rows x kPK K blocks: each row of a box is one kPK*128-byte contiguous run.
static bool make_map_u8_3d_pk(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                              uint32_t box_outer, uint32_t pk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kBK, outer, inner / kBK};
  const cuuint64_t strides[2] = {inner, (cuuint64_t)kBK};
  const cuuint32_t box[3] = {(cuuint32_t)kBK, box_outer, pk};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 matrix [rows][cols] stored through 8-row x 64-column boxes with the 128-byte swizzle.
// The same BF16 matrix as 3-D (column, row inside a 32-row block, 32-row block): boxes of 64
// columns x 8 rows x 4 blocks store four 8-row groups 32 rows apart (one warp's rows of a tile).
static bool make_map_bf16_store3(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cols, 32, rows / 32};
  const cuuint64_t strides[2] = {cols * 2, cols * 2 * 32};
  const cuuint32_t box[3] = {64, 8, 4};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool make_map_bf16_store(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 8};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation rows [R][K] bytes of the tile kernel as a 5-D view: x = 128 bytes of a K block,
// i = row inside an 8-row group, k = K block, a = 32-row block, b = 8-row group inside it.  One box
// {128, 8, pk, 4, 4} at (0, 0, kb, m0/32, 0) brings the 128-row tile for pk K blocks in a single copy
// and lays 8-row group 4a + b at shared-memory group 4b + a (each group pk x 1 KB).
static bool make_map_act_tile(CUtensorMap* m, const void* base, uint64_t K, uint64_t R, uint32_t pk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[5] = {(cuuint64_t)kBK, 8, K / kBK, R / 32, 4};
  const cuuint64_t strides[4] = {K, (cuuint64_t)kBK, 32 * K, 8 * K};
  const cuuint32_t box[5] = {(cuuint32_t)kBK, 8, pk, 4, 4};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight rows [rows][K] as 4-D (x, row, K block, half with a stride of `half_rows` rows): one box
// {128, 128, pk, 2} brings two 128-row blocks for pk K blocks, laid out [half][K block][row]
// (FC1: 128 gate rows and the matching up rows, half_rows = I; FC2: 256 consecutive rows).
static bool make_map_w13_tile(CUtensorMap* m, const void* base, uint64_t H, uint64_t rows,
                              uint64_t I, uint32_t pk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kBK, rows, H / kBK, 2};
  const cuuint64_t strides[3] = {H, (cuuint64_t)kBK, I * H};
  const cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)kGroup, pk, 2};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token rows of the small-batch kernel [R][K] bytes as 4-D (x, row inside an 8-row group, K block,
// 8-row group): one box {128, 8, pk, 4} at (0, 0, kb, row0/8) brings a 32-row chunk for pk K blocks,
// laid out [group][K block][8 rows][128 bytes].
static bool make_map_tok_chunk(CUtensorMap* m, const void* base, uint64_t K, uint64_t R, uint32_t pk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kBK, 8, K / kBK, R / 8};
  const cuuint64_t strides[3] = {K, (cuuint64_t)kBK, 8 * K};
  const cuuint32_t box[4] = {(cuuint32_t)kBK, 8, pk, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation scales [K/128][R] (fp32 or UE8M0 bytes) as 2-D, boxes of 128 rows x pk K blocks.
static bool make_map_act_scales(CUtensorMap* m, const void* base, bool bytes, uint64_t R,
                                uint64_t KB, uint32_t pk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {R, KB};
  const cuuint64_t strides[1] = {R * (bytes ? 1 : 4)};
  const cuuint32_t box[2] = {(cuuint32_t)kBM, pk};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Flat array of n elements (fp32 or bytes), boxes of box_bytes (16 or 32): used to fetch the block
// scales of a pipeline stage (and their aligned neighbours).
static bool make_map_1d(CUtensorMap* m, const void* base, bool bytes, uint64_t n,
                        uint32_t box_bytes = 16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[1] = {n};
  const cuuint64_t strides[1] = {0};
  const cuuint32_t box[1] = {bytes ? box_bytes : box_bytes / 4};
  const cuuint32_t estr[1] = {1};
  return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// ------------------------------------------------------------ validation
static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static moe_status check_ws(const Plan& pl, const void* ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < pl.ws.total_bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

static moe_status check_args(const moe_fwd_args* a, const void* ws, size_t ws_bytes, Plan* pl,
                             bool need_x, bool need_w13, bool need_w2, bool need_reduce) {
  if (a == nullptr) return MOE_ERR_INVALID_ARG;
  if (a->weight_scale_fmt < MOE_SCALE_FP32 || a->weight_scale_fmt > MOE_SCALE_UE8M0)
    return MOE_ERR_INVALID_ARG;
  if (a->clamp_mode < MOE_CLAMP_NONE || a->clamp_mode > MOE_CLAMP_AFTER_SILU)
    return MOE_ERR_INVALID_ARG;
  if (a->clamp_mode != MOE_CLAMP_NONE && !(a->clamp_limit >= 0.0f && a->clamp_limit < 3.4e38f))
    return MOE_ERR_INVALID_ARG;
  if (a->numerics < MOE_NUMERICS_DIVIDE || a->numerics > MOE_NUMERICS_RECIPROCAL)
    return MOE_ERR_INVALID_ARG;
  moe_status st = make_plan(a->M_cap, a->E, a->H, a->I, a->topk, a->act_scale_fmt, pl);
  if (st != MOE_OK) return st;
  st = check_ws(*pl, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (a->d_num_tokens != nullptr && !aligned(a->d_num_tokens, 4)) return MOE_ERR_INVALID_ARG;
  if (need_x) {
    if (a->x == nullptr || !aligned(a->x, 16)) return MOE_ERR_INVALID_ARG;
    if (a->topk_ids == nullptr || !aligned(a->topk_ids, 4)) return MOE_ERR_INVALID_ARG;
  }
  if (need_w13) {
    if (a->w13 == nullptr || !aligned(a->w13, 16)) return MOE_ERR_INVALID_ARG;
    if (a->s13 == nullptr || !aligned(a->s13, 16)) return MOE_ERR_INVALID_ARG;
  }
  if (need_w2) {
    if (a->w2 == nullptr || !aligned(a->w2, 16)) return MOE_ERR_INVALID_ARG;
    if (a->s2 == nullptr || !aligned(a->s2, 16)) return MOE_ERR_INVALID_ARG;
  }
  if (need_reduce) {
    if (a->topk_weights == nullptr || !aligned(a->topk_weights, 4)) return MOE_ERR_INVALID_ARG;
    if (a->out == nullptr || !aligned(a->out, 16)) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

template <typename T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ------------------------------------------------------------- steps
static moe_status run_align(const int32_t* ids, const int32_t* d_n, int expert_offset, const Plan& pl,
                            void* ws, cudaStream_t s) {
  AlignParams p;
  p.topk_ids = ids;
  p.d_num_tokens = d_n;
  p.M_cap = pl.M_cap;
  p.topk = pl.topk;
  p.E = pl.E;
  p.expert_offset = expert_offset;
  p.seg_start = at<int32_t>(ws, pl.ws.seg_start);
  p.live_end = at<int32_t>(ws, pl.ws.live_end);
  p.sorted_pair = at<int32_t>(ws, pl.ws.sorted_pair);
  p.pair_row = at<int32_t>(ws, pl.ws.pair_row);
  p.tile_expert = at<int32_t>(ws, pl.ws.tile_expert);
  p.num_tiles = at<int32_t>(ws, pl.ws.num_tiles);
  p.status = at<int32_t>(ws, pl.ws.status);
  p.splitk_count = at<int32_t>(ws, pl.ws.splitk_count);
  p.splitk_count_len = pl.ws.fc1_ksplit > 1 ? pl.ws.C_cap * (pl.I / kGroup)
                       : (!pl.ws.small_batch && pl.act_fmt == MOE_SCALE_UE8M0) ? pl.ws.T_cap : 0;
  p.chunk_row0 = at<int32_t>(ws, pl.ws.chunk_row0);
  p.num_chunks = at<int32_t>(ws, pl.ws.num_chunks);
  p.cta_hist = at<int32_t>(ws, pl.ws.align_hist);
  p.num_ctas = pl.ws.align_ctas;
  return launch_align(p, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static moe_status run_quant(const void* x, const int32_t* d_n, const Plan& pl, int numerics,
                            void* ws, cudaStream_t s) {
  if (pl.M_cap == 0) return MOE_OK;
  QuantParams p;
  p.x = static_cast<const uint16_t*>(x);
  p.d_num_tokens = d_n;
  p.pair_row = at<int32_t>(ws, pl.ws.pair_row);
  p.M_cap = pl.M_cap;
  p.H = pl.H;
  p.topk = pl.topk;
  p.R_cap = pl.ws.R_cap;
  p.fmt = pl.act_fmt;
  p.numerics = numerics;
  p.a_q = at<uint8_t>(ws, pl.ws.a1_q);
  p.a_s = at<void>(ws, pl.ws.a1_s);
  return launch_quant(p, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static void fill_gemm_common(GemmParams& p, const Plan& pl, void* ws) {
  memset(&p, 0, sizeof(p));
  p.tile_expert = at<int32_t>(ws, pl.ws.tile_expert);
  p.num_tiles = at<int32_t>(ws, pl.ws.num_tiles);
  p.live_end = at<int32_t>(ws, pl.ws.live_end);
  p.R_cap = pl.ws.R_cap;
  p.status = at<int32_t>(ws, pl.ws.status);
  p.act_fmt = pl.act_fmt;
  p.a_scale_ue8m0 = pl.act_fmt == MOE_SCALE_UE8M0;
  p.P_cap = pl.ws.P_cap;
  p.sorted_pair = at<int32_t>(ws, pl.ws.sorted_pair);
  p.chunk_row0 = at<int32_t>(ws, pl.ws.chunk_row0);
  p.num_chunks = at<int32_t>(ws, pl.ws.num_chunks);
}

static moe_status run_fc1(const moe_fwd_args* a, const Plan& pl, void* ws, cudaStream_t s,
                          const int32_t* tile_row0 = nullptr) {
  if (pl.ws.R_cap == 0) return MOE_OK;
  CUtensorMap tmA, tmB, tmAS, tmS;
  const bool w_ue = a->weight_scale_fmt == MOE_SCALE_UE8M0;
  const bool small = pl.ws.small_batch != 0;
  const uint64_t n_ws = (uint64_t)pl.E * (2 * pl.I / kGroup) * (pl.H / kGroup);
  const bool bs = w_ue && pl.act_fmt == MOE_SCALE_UE8M0;   // scales applied inside the MMA
  const uint32_t pk = bs ? TileCfg<true, true>::PK : TileCfg<true>::PK;
  const bool maps_ok =
      small ? make_map_tok_chunk(&tmA, at<void>(ws, pl.ws.a1_q), pl.H, pl.ws.R_cap, kSmallPK) &&
                  make_map_w13_tile(&tmB, a->w13, pl.H, (uint64_t)pl.E * 2 * pl.I, pl.I, kSmallPK) &&
                  make_map_1d(&tmS, a->s13, w_ue, n_ws)
            : make_map_act_tile(&tmA, at<void>(ws, pl.ws.a1_q), pl.H, pl.ws.R_cap, pk) &&
                  make_map_w13_tile(&tmB, a->w13, pl.H, (uint64_t)pl.E * 2 * pl.I, pl.I, pk) &&
                  make_map_act_scales(&tmAS, at<void>(ws, pl.ws.a1_s), pl.act_fmt == MOE_SCALE_UE8M0,
                                      pl.ws.R_cap, pl.H / kGroup, pk) &&
                  make_map_1d(&tmS, a->s13, w_ue, n_ws, 32);
  if (!maps_ok) return MOE_ERR_CUDA;
  GemmParams p;
  fill_gemm_common(p, pl, ws);
  p.tile_row0 = tile_row0;
  p.a_scale = at<void>(ws, pl.ws.a1_s);
  p.b_scale = a->s13;
  p.b_scale_ue8m0 = a->weight_scale_fmt == MOE_SCALE_UE8M0;
  p.K = pl.H;
  p.n_blocks = pl.I / kGroup;
  p.b_rows_per_expert = 2 * pl.I;
  p.out_cols = pl.I;
  p.ksplit = pl.ws.fc1_ksplit;
  p.a2_q = at<uint8_t>(ws, pl.ws.a2_q);
  p.a2_s = at<void>(ws, pl.ws.a2_s);
  p.clamp_mode = a->clamp_mode;
  p.clamp_limit = a->clamp_limit;
  p.numerics = a->numerics;
  p.splitk_partial = at<float>(ws, pl.ws.splitk_partial);
  p.splitk_count = at<int32_t>(ws, pl.ws.splitk_count);
  if (!small && p.ksplit != 1) return MOE_ERR_UNSUPPORTED_SHAPE;   // the tile kernels do not split K
  // routed block-scaled layers: FC1 counts its finished items per row tile for FC2 (the alignment
  // reset the counters); the batched layout keeps the grid-wide dependency
  if (!small && bs && tile_row0 == nullptr) p.tile_ready = at<int32_t>(ws, pl.ws.splitk_count);
  const long items = (long)(small ? pl.ws.C_cap : pl.ws.T_cap) * p.n_blocks * p.ksplit;
  const int grid = (int)std::max(1L, std::min<long>(sm_count(), items));
  // tile schedule with fp32 activation scales: BF16 FC1 outputs, then SwiGLU + requant kernel
  const bool split_epilogue = !small && !bs && pl.ws.g1 != 0;
  if (split_epilogue) p.g1 = at<uint16_t>(ws, pl.ws.g1);
  cudaError_t err = small ? launch_fc1_small(tmA, tmB, tmS, p, grid, s)
                    : bs  ? launch_fc1_bs(tmA, tmB, tmAS, tmS, p, grid, s)
                          : launch_fc1(tmA, tmB, tmAS, tmS, p, grid, s);
  if (err == cudaSuccess && split_epilogue) {
    SwigluQuantParams q;
    q.g1 = p.g1;
    q.R_cap = pl.ws.R_cap;
    q.I = pl.I;
    q.num_tiles = p.num_tiles;
    q.tile_expert = p.tile_expert;
    q.live_end = p.live_end;
    q.all_tiles = tile_row0 != nullptr ? 1 : 0;
    q.clamp_mode = a->clamp_mode;
    q.clamp_limit = a->clamp_limit;
    q.numerics = a->numerics;
    q.fmt = pl.act_fmt;
    q.a2_q = p.a2_q;
    q.a2_s = p.a2_s;
    err = launch_swiglu_quant(q, s);
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// after_fc1: the kernel launched just before this one on the stream is this layer's FC1 (the
// whole-layer forward), so the block-scaled FC2 may rely on the per-tile FC1 counters alone and skip
// the wait for the previous grid; otherwise (the standalone FC2 step) it waits for the previous
// grid and checks the counters as well.
static moe_status run_fc2(const moe_fwd_args* a, const Plan& pl, void* ws, cudaStream_t s,
                          const int32_t* tile_row0 = nullptr, void* y_target = nullptr,
                          bool after_fc1 = false) {
  if (pl.ws.R_cap == 0) return MOE_OK;
  CUtensorMap tmA, tmB, tmAS, tmS;
  const bool w_ue = a->weight_scale_fmt == MOE_SCALE_UE8M0;
  const bool small = pl.ws.small_batch != 0;
  const uint64_t n_ws = (uint64_t)pl.E * (pl.H / kGroup) * (pl.I / kGroup);
  constexpr uint32_t pk = TileCfg<false>::PK;
  const bool maps_ok =
      small ? make_map_tok_chunk(&tmA, at<void>(ws, pl.ws.a2_q), pl.I, pl.ws.R_cap, kSmallPK) &&
                  make_map_w13_tile(&tmB, a->w2, pl.I, (uint64_t)pl.E * pl.H, kGroup, kSmallPK) &&
                  make_map_1d(&tmS, a->s2, w_ue, n_ws)
            : make_map_act_tile(&tmA, at<void>(ws, pl.ws.a2_q), pl.I, pl.ws.R_cap, pk) &&
                  make_map_u8_3d_pk(&tmB, a->w2, pl.I, (uint64_t)pl.E * pl.H, kBN, pk) &&
                  make_map_act_scales(&tmAS, at<void>(ws, pl.ws.a2_s), pl.act_fmt == MOE_SCALE_UE8M0,
                                      pl.ws.R_cap, pl.I / kGroup, pk) &&
                  make_map_1d(&tmS, a->s2, w_ue, n_ws, 32);
  if (!maps_ok) return MOE_ERR_CUDA;
  GemmParams p;
  fill_gemm_common(p, pl, ws);
  p.tile_row0 = tile_row0;
  p.a_scale = at<void>(ws, pl.ws.a2_s);
  p.b_scale = a->s2;
  p.b_scale_ue8m0 = a->weight_scale_fmt == MOE_SCALE_UE8M0;
  p.K = pl.I;
  p.n_blocks = (pl.H + kBN - 1) / kBN;
  p.b_rows_per_expert = pl.H;
  p.out_cols = pl.H;
  p.ksplit = 1;
  void* y = y_target != nullptr ? y_target : at<void>(ws, pl.ws.y);
  p.y = static_cast<uint16_t*>(y);
  const long items = (long)(small ? pl.ws.C_cap : pl.ws.T_cap) * p.n_blocks;
  const int grid = (int)std::max(1L, std::min<long>(sm_count(), items));
  CUtensorMap tmY, tmY3;
  if (!small && (!make_map_bf16_store(&tmY, y, pl.H, pl.ws.R_cap) ||
                 !make_map_bf16_store3(&tmY3, y, pl.H, pl.ws.R_cap)))
    return MOE_ERR_CUDA;
  const bool bs = w_ue && pl.act_fmt == MOE_SCALE_UE8M0;   // scales applied inside the MMA
  if (!small && bs && tile_row0 == nullptr) {
    p.tile_ready = at<int32_t>(ws, pl.ws.splitk_count);   // FC1 items done per row tile
    p.fc1_items_per_tile = pl.I / kGroup;
    p.wait_prev_grid = after_fc1 ? 0 : 1;
  }
  const cudaError_t err = small ? launch_fc2_small(tmA, tmB, tmS, p, grid, s)
                          : bs  ? launch_fc2_bs(tmA, tmB, tmAS, tmS, tmY, tmY3, p, grid, s)
                                : launch_fc2(tmA, tmB, tmAS, tmS, tmY, tmY3, p, grid, s);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static moe_status run_reduce(const moe_fwd_args* a, const Plan& pl, void* ws, cudaStream_t s) {
  if (pl.M_cap == 0) return MOE_OK;
  ReduceParams p;
  p.y = at<uint16_t>(ws, pl.ws.y);
  p.pair_row = at<int32_t>(ws, pl.ws.pair_row);
  p.topk_weights = a->topk_weights;
  p.d_num_tokens = a->d_num_tokens;
  p.M_cap = pl.M_cap;
  p.H = pl.H;
  p.topk = pl.topk;
  p.out = a->out;
  p.out_fp32 = a->out_fp32 ? 1 : 0;
  return launch_reduce(p, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ------------------------------------------------- batched-expert layout
// Expert e's rows are [e * max_m, e * max_m + counts[e]) of x [E, max_m, H] and of out; the
// workspace holds the metadata and the FP8 intermediates of the same row space.
static moe_status make_batched_plan(int E, int max_m, int H, int I, int act_fmt, Plan* plan,
                                    size_t* tile_row0_off) {
  if (E <= 0 || max_m <= 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (act_fmt < MOE_SCALE_FP32 || act_fmt > MOE_SCALE_UE8M0) return MOE_ERR_INVALID_ARG;
  if (max_m % kAlign || H % kGroup || I % kGroup || H > 32768 || I > 16384 || E > kMaxExperts)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)E * max_m > kMaxPairs) return MOE_ERR_UNSUPPORTED_SHAPE;
  memset(plan, 0, sizeof(*plan));
  moe_ws_plan& w = plan->ws;
  const long long R = (long long)E * max_m;
  w.R_cap = (int32_t)R;
  w.P_cap = (int32_t)R;
  w.T_cap = (int32_t)(R / kAlign);
  w.C_cap = (int32_t)(R / 32);
  w.small_batch = max_m <= 256 ? 1 : 0;
  w.fc1_ksplit = 1;
  w.align_ctas = 1;
  const size_t sc = act_fmt == MOE_SCALE_UE8M0 ? 1 : 4;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  w.status = take(4);
  w.num_tiles = take(4);
  w.seg_start = take((size_t)(E + 1) * 4);
  w.live_end = take((size_t)E * 4);
  w.tile_expert = take((size_t)w.T_cap * 4);
  *tile_row0_off = take((size_t)w.T_cap * 4);
  w.num_chunks = take(4);
  w.chunk_row0 = take((size_t)w.C_cap * 4);
  w.a1_q = take((size_t)R * H);
  w.a1_s = take((size_t)(H / kGroup) * R * sc);
  w.a2_q = take((size_t)R * I);
  w.a2_s = take((size_t)(I / kGroup) * R * sc);
  w.g1 = (!w.small_batch && act_fmt != MOE_SCALE_UE8M0) ? take((size_t)R * 2 * I * 2) : 0;
  w.total_bytes = off;
  plan->M_cap = max_m;
  plan->E = E;
  plan->H = H;
  plan->I = I;
  plan->topk = 1;
  plan->act_fmt = act_fmt;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_plan(int M_cap, int E, int H, int I, int topk, moe_scale_fmt act_fmt,
                              moe_ws_plan* plan) {
  if (plan == nullptr) return MOE_ERR_INVALID_ARG;
  Plan pl;
  const moe_status st = make_plan(M_cap, E, H, I, topk, act_fmt, &pl);
  if (st == MOE_OK) *plan = pl.ws;
  return st;
}

size_t moe_workspace_bytes(int M_cap, int E, int H, int I, int topk, moe_scale_fmt act_fmt) {
  Plan pl;
  return make_plan(M_cap, E, H, I, topk, act_fmt, &pl) == MOE_OK ? pl.ws.total_bytes : 0;
}

moe_status moe_align(const int32_t* topk_ids, const int32_t* d_num_tokens, int M_cap, int topk, int E,
                     int expert_offset, int H, int I, moe_scale_fmt act_fmt, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream) {
  Plan pl;
  moe_status st = make_plan(M_cap, E, H, I, topk, act_fmt, &pl);
  if (st != MOE_OK) return st;
  st = check_ws(pl, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (M_cap > 0 && (topk_ids == nullptr || !aligned(topk_ids, 4))) return MOE_ERR_INVALID_ARG;
  if (d_num_tokens != nullptr && !aligned(d_num_tokens, 4)) return MOE_ERR_INVALID_ARG;
  return run_align(topk_ids, d_num_tokens, expert_offset, pl, workspace, (cudaStream_t)stream);
}

moe_status moe_quant_act(const void* x_bf16, const int32_t* d_num_tokens, int M_cap, int E, int H,
                         int I, int topk, moe_scale_fmt act_fmt, moe_numerics numerics,
                         void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  Plan pl;
  moe_status st = make_plan(M_cap, E, H, I, topk, act_fmt, &pl);
  if (st != MOE_OK) return st;
  st = check_ws(pl, workspace, workspace_bytes);
  if (st != MOE_OK) return st;
  if (M_cap > 0 && (x_bf16 == nullptr || !aligned(x_bf16, 16))) return MOE_ERR_INVALID_ARG;
  if (d_num_tokens != nullptr && !aligned(d_num_tokens, 4)) return MOE_ERR_INVALID_ARG;
  if (numerics < MOE_NUMERICS_DIVIDE || numerics > MOE_NUMERICS_RECIPROCAL) return MOE_ERR_INVALID_ARG;
  return run_quant(x_bf16, d_num_tokens, pl, numerics, workspace, (cudaStream_t)stream);
}

moe_status moe_fc1_swiglu_quant(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream) {
  Plan pl;
  const moe_status st = check_args(args, workspace, workspace_bytes, &pl, false, true, false, false);
  if (st != MOE_OK) return st;
  return run_fc1(args, pl, workspace, (cudaStream_t)stream);
}

moe_status moe_fc2(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                   moe_stream_t stream) {
  Plan pl;
  const moe_status st = check_args(args, workspace, workspace_bytes, &pl, false, false, true, false);
  if (st != MOE_OK) return st;
  return run_fc2(args, pl, workspace, (cudaStream_t)stream);
}

moe_status moe_topk_reduce(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream) {
  Plan pl;
  const moe_status st = check_args(args, workspace, workspace_bytes, &pl, false, false, false, true);
  if (st != MOE_OK) return st;
  return run_reduce(args, pl, workspace, (cudaStream_t)stream);
}

moe_status moe_fp8_block_forward(const moe_fwd_args* args, void* workspace, size_t workspace_bytes,
                                 moe_stream_t stream) {
  Plan pl;
  moe_status st = check_args(args, workspace, workspace_bytes, &pl, true, true, true, true);
  if (st != MOE_OK) return st;
  if (pl.M_cap == 0) return MOE_OK;
  const cudaStream_t s = (cudaStream_t)stream;
  if ((st = run_align(args->topk_ids, args->d_num_tokens, args->expert_offset, pl, workspace, s)) !=
      MOE_OK)
    return st;
  if ((st = run_quant(args->x, args->d_num_tokens, pl, args->numerics, workspace, s)) != MOE_OK)
    return st;
  if ((st = run_fc1(args, pl, workspace, s)) != MOE_OK) return st;
  if ((st = run_fc2(args, pl, workspace, s, nullptr, nullptr, /*after_fc1=*/true)) != MOE_OK)
    return st;
  return run_reduce(args, pl, workspace, s);
}

size_t moe_batched_workspace_bytes(int E, int max_m, int H, int I, moe_scale_fmt act_fmt) {
  Plan pl;
  size_t tr;
  return make_batched_plan(E, max_m, H, I, act_fmt, &pl, &tr) == MOE_OK ? pl.ws.total_bytes : 0;
}

moe_status moe_fp8_batched_forward(const moe_batched_args* b, void* workspace,
                                   size_t workspace_bytes, moe_stream_t stream) {
  if (b == nullptr) return MOE_ERR_INVALID_ARG;
  Plan pl;
  size_t tile_row0_off = 0;
  moe_status st = make_batched_plan(b->E, b->max_m, b->H, b->I, b->act_scale_fmt, &pl, &tile_row0_off);
  if (st != MOE_OK) return st;
  if ((st = check_ws(pl, workspace, workspace_bytes)) != MOE_OK) return st;
  if (b->weight_scale_fmt < MOE_SCALE_FP32 || b->weight_scale_fmt > MOE_SCALE_UE8M0 ||
      b->clamp_mode < MOE_CLAMP_NONE || b->clamp_mode > MOE_CLAMP_AFTER_SILU ||
      b->numerics < MOE_NUMERICS_DIVIDE || b->numerics > MOE_NUMERICS_RECIPROCAL)
    return MOE_ERR_INVALID_ARG;
  if (b->clamp_mode != MOE_CLAMP_NONE && !(b->clamp_limit >= 0.0f && b->clamp_limit < 3.4e38f))
    return MOE_ERR_INVALID_ARG;
  if (b->x == nullptr || !aligned(b->x, 16) || b->out == nullptr || !aligned(b->out, 16) ||
      b->d_counts == nullptr || !aligned(b->d_counts, 4) || b->w13 == nullptr ||
      !aligned(b->w13, 16) || b->w2 == nullptr || !aligned(b->w2, 16) || b->s13 == nullptr ||
      !aligned(b->s13, 16) || b->s2 == nullptr || !aligned(b->s2, 16))
    return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = (cudaStream_t)stream;
  int32_t* tile_row0 = at<int32_t>(workspace, tile_row0_off);
  BatchPrepParams bp;
  bp.counts = b->d_counts;
  bp.E = b->E;
  bp.max_m = b->max_m;
  bp.seg_start = at<int32_t>(workspace, pl.ws.seg_start);
  bp.live_end = at<int32_t>(workspace, pl.ws.live_end);
  bp.tile_expert = at<int32_t>(workspace, pl.ws.tile_expert);
  bp.tile_row0 = tile_row0;
  bp.num_tiles = at<int32_t>(workspace, pl.ws.num_tiles);
  bp.chunk_row0 = at<int32_t>(workspace, pl.ws.chunk_row0);
  bp.num_chunks = at<int32_t>(workspace, pl.ws.num_chunks);
  bp.status = at<int32_t>(workspace, pl.ws.status);
  if (launch_batch_prep(bp, s) != cudaSuccess) return MOE_ERR_CUDA;
  QuantRowsParams qp;
  qp.x = static_cast<const uint16_t*>(b->x);
  qp.counts = b->d_counts;
  qp.E = b->E;
  qp.max_m = b->max_m;
  qp.H = b->H;
  qp.R_cap = pl.ws.R_cap;
  qp.fmt = b->act_scale_fmt;
  qp.numerics = b->numerics;
  qp.a_q = at<uint8_t>(workspace, pl.ws.a1_q);
  qp.a_s = at<void>(workspace, pl.ws.a1_s);
  if (launch_quant_rows(qp, s) != cudaSuccess) return MOE_ERR_CUDA;
  moe_fwd_args a;
  memset(&a, 0, sizeof(a));
  a.w13 = b->w13;
  a.s13 = b->s13;
  a.w2 = b->w2;
  a.s2 = b->s2;
  a.E = b->E;
  a.H = b->H;
  a.I = b->I;
  a.weight_scale_fmt = b->weight_scale_fmt;
  a.act_scale_fmt = b->act_scale_fmt;
  a.clamp_mode = b->clamp_mode;
  a.clamp_limit = b->clamp_limit;
  a.numerics = b->numerics;
  const int32_t* tiles = pl.ws.small_batch ? nullptr : tile_row0;
  if ((st = run_fc1(&a, pl, workspace, s, tiles)) != MOE_OK) return st;
  return run_fc2(&a, pl, workspace, s, tiles, b->out);
}

moe_status moe_last_device_status(const void* workspace, moe_stream_t stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return (v == 0) ? MOE_OK : (moe_status)v;
}

const char* moe_status_str(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* moe_version(void) { return "block_fp8_mixture_gb300 0.1 (sm_103a)"; }

}  // extern "C"
