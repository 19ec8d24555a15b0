// Internal declarations shared by the library's translation units: constants, the kernel
// parameter blocks and the launchers each .cu file provides.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_fp8.h"

namespace moe {

constexpr int kAlign = 128;               // expert segment alignment = GEMM row-tile height
constexpr int kGroup = 128;               // 1x128 activation group = 128x128 weight block
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopk = 16;
constexpr int kMaxPairs = 1 << 20;
constexpr int kMaxKSplit = 8;                      // largest FC1 K-split of the small-batch schedule
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s bound on any device-side wait
constexpr float kScaleFloor = 1.0f / 229376.0f;    // 1/(448*512), rounded to fp32

// ---------------------------------------------------------------- GEMM tiling
// 128-row-tile kernel: one CTA tile = 128 workspace rows (the MMA's M) x 256 weight rows (two
// N = 128 MMAs; FC1: 128 gate rows and the matching 128 up rows) x kPK 128-wide K blocks per
// pipeline stage.  Operands arrive through 3-D tensor maps (x = 128 bytes of K, y = rows, z = K
// block), so every row of a stage is fetched as one kPK*128-byte contiguous run.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;
constexpr int kABoxRows = 8;                          // activation rows per TMA box (one swizzle atom)
constexpr int kGemmThreads = 320;                     // small kernel: TMA, MMA, 8 epilogue warps
constexpr int kSmallPK = 2;                           // small kernel: K blocks per operand stage
constexpr int kEpiWarp0 = 2;
// 128-row-tile kernel: warpgroup 0 = TMA warp, MMA warp, two idle warps (40 registers each after
// setmaxnreg); warpgroups 1-2 = the 8 promotion/epilogue warps (232 registers each: 128
// accumulators, 64 loaded partial sums and the loop state without spills).
constexpr int kTileThreads = 384;
constexpr int kTileEpiWarp0 = 4;
constexpr int kTileRegsLow = 40;
constexpr int kTileRegsHigh = 232;
static_assert(128 * kTileRegsLow + 256 * kTileRegsHigh <= kTileThreads * 168,
              "register split must fit the launch allocation");
static_assert(32 * (kTileRegsLow + 2 * kTileRegsHigh) <= 16384, "register split per sub-partition");
constexpr int kEpiThreads = 256;
constexpr int kTmemCols = 512;                        // two 256-column accumulators
// Per-stage scale slot: [k*512, +512) the 128 activation scales of the stage's K block k (fp32 or
// UE8M0 bytes); [1024 + k*256, +16) and [1024 + k*256 + 128, +16) the 16-byte aligned chunks
// holding the two weight block scales of K block k.
// tile-kernel scale slot: [K block][128 activation scales] at 0, the two 32-byte weight-scale
// boxes (which cover the stage's K blocks) at kSlotW and kSlotW + 128
constexpr int kSlotW = 1024;
constexpr int kSlotBytes = kSlotW + 256;

// Pipeline shape of the 128-row-tile kernels: one K block per stage, so each K block's gate and up
// (or low and high) weight rows sit together and one N = 256 MMA covers them.  FC1 (long K, small
// output) streams through four stages.  FC2 (short K, a 64 KB BF16 output tile per item) uses three
// stages and a 64 KB staging area from which asynchronous TMA stores write the output tile while
// the next item proceeds (the block-scaled FC2: four stages and 2 KB of staging per warp).  Two K
// blocks per stage, tried for the promotion kernel's FC1, made its promotion warps spill registers.
template <bool kFC1, bool kBS = false>
struct TileCfg {
  static constexpr int PK = 1;
  // FC2 of the block-scaled kernel stores its output one 8-row group at a time through 2 KB per warp,
  // which leaves room for a fourth operand stage
  static constexpr bool YByGroup = !kFC1 && kBS;
  static constexpr int Stages = kFC1 ? 4 : (YByGroup ? 4 : 3);
  static constexpr int ABytes = kBM * kBK * PK;
  static constexpr int BHalf = kGroup * kBK * PK;     // 128 weight rows
  static constexpr int StageBytes = ABytes + 2 * BHalf;
  static constexpr int SlotBytes = kSlotBytes;
  static_assert(PK * kBM * 4 <= kSlotW, "activation scales of a stage fit the slot");
  // scale slots form their own ring, deeper than the operand ring: an operand stage is released
  // as soon as the MMAs have read it, while the promotion warps still read the stage's scales
  static constexpr int ScaleSlots = Stages + 2;
  // 32 rows x 128 BF16 columns per warp, or 8 rows with YByGroup
  static constexpr int YWarpBytes = kFC1 ? 0 : (YByGroup ? 2048 : 8192);
  static constexpr int Smem = Stages * StageBytes + ScaleSlots * SlotBytes + 8 * YWarpBytes +
                              1024 /*align*/ + 1024 /*bars*/ + 2 * kBM * 4 /*row amax*/;
};
static_assert(TileCfg<true>::Smem <= 232448 && TileCfg<false>::Smem <= 232448 &&
                  TileCfg<true, true>::Smem <= 232448 && TileCfg<false, true>::Smem <= 232448,
              "shared memory");

struct Plan {
  moe_ws_plan ws;
  int M_cap, E, H, I, topk;
  int act_fmt;
};

moe_status make_plan(int M_cap, int E, int H, int I, int topk, int act_fmt, Plan* plan);

// ------------------------------------------------------------ kernel params
struct AlignParams {
  const int32_t* topk_ids;
  const int32_t* d_num_tokens;
  int M_cap, topk, E;
  int expert_offset;
  int32_t* seg_start;
  int32_t* live_end;
  int32_t* sorted_pair;
  int32_t* pair_row;
  int32_t* tile_expert;
  int32_t* num_tiles;
  int32_t* status;
  int32_t* splitk_count;
  int splitk_count_len;
  int32_t* chunk_row0;
  int32_t* num_chunks;
  // large batches: num_ctas CTAs each align a contiguous range of pairs; per-CTA expert counts
  int32_t* cta_hist;        // [num_ctas][E]
  int num_ctas;
};

// Batched-expert layout: expert e's rows are [e * max_m, e * max_m + counts[e]).
struct BatchPrepParams {
  const int32_t* counts;
  int E, max_m;
  int32_t* seg_start;
  int32_t* live_end;
  int32_t* tile_expert;
  int32_t* tile_row0;
  int32_t* num_tiles;
  int32_t* chunk_row0;
  int32_t* num_chunks;
  int32_t* status;
};

struct QuantRowsParams {
  const uint16_t* x;
  const int32_t* counts;
  int E, max_m, H, R_cap;
  int fmt;
  int numerics;
  uint8_t* a_q;
  void* a_s;
};

struct QuantParams {
  const uint16_t* x;
  const int32_t* d_num_tokens;
  const int32_t* pair_row;
  int M_cap, H, topk, R_cap;
  int fmt;
  int numerics;
  uint8_t* a_q;
  void* a_s;
};

struct GemmParams {
  const int32_t* tile_expert;
  const int32_t* num_tiles;
  const int32_t* live_end;
  const void* a_scale;      // column-major [K/128][R_cap]
  int a_scale_ue8m0;
  const void* b_scale;      // [E][Nrows/128][K/128]
  int b_scale_ue8m0;
  int K;                    // reduction length (H for FC1, I for FC2)
  int R_cap;
  int n_blocks;             // output column blocks per tile (I/128 for FC1, ceil(H/256) for FC2)
  int b_rows_per_expert;    // 2I for FC1, H for FC2
  int out_cols;             // I for FC1 (a2_q row length), H for FC2 (y row length)
  int ksplit;               // FC1 K-split factor
  // FC1 epilogue
  uint8_t* a2_q;
  void* a2_s;
  int act_fmt;
  int clamp_mode;
  float clamp_limit;
  int numerics;
  float* splitk_partial;    // [ksplit][P_cap][2I] fp32
  int32_t* splitk_count;    // [T_cap * n_blocks]
  const int32_t* sorted_pair;
  int P_cap;
  // small-batch schedule: live 32-row chunks
  const int32_t* chunk_row0;
  const int32_t* num_chunks;
  // batched-expert layout: first row of each live 128-row tile (nullptr: tile i starts at 128 i)
  const int32_t* tile_row0;
  // FC2 epilogue
  uint16_t* y;
  int32_t* status;
  // tile schedule, fp32 activation scales: FC1 writes BF16 (gate | up) rows here instead of
  // running SwiGLU + requantization in its epilogue (nullptr: fused epilogue)
  uint16_t* g1;
  // block-scaled tile schedule of a routed layer: FC1 adds one per finished item of row tile t to
  // tile_ready[t]; FC2 starts a tile once fc1_items_per_tile items are in.  Inside the whole-layer
  // forward (FC1 launched just before FC2) that replaces FC2's wait for the FC1 grid (nullptr: FC2
  // waits for the previous kernel only)
  int32_t* tile_ready;
  int fc1_items_per_tile;
  int wait_prev_grid;       // with tile_ready: also wait for the previous grid (standalone FC2)
};

// SwiGLU + 1x128 requantization of the BF16 FC1 outputs of live workspace rows.
struct SwigluQuantParams {
  const uint16_t* g1;       // [R_cap][2I]
  int R_cap, I;
  const int32_t* num_tiles;
  const int32_t* tile_expert;
  const int32_t* live_end;
  int all_tiles;            // 1: tile_expert holds every tile (batched layout), 0: tiles < num_tiles
  int clamp_mode;
  float clamp_limit;
  int numerics;
  int fmt;
  uint8_t* a2_q;
  void* a2_s;
};

struct ReduceParams {
  const uint16_t* y;
  const int32_t* pair_row;
  const float* topk_weights;
  const int32_t* d_num_tokens;
  int M_cap, H, topk;
  void* out;                // bf16, or fp32 when out_fp32
  int out_fp32;
};

// Launch with programmatic stream serialization: the kernel may start while the previous kernel of
// the stream finishes; it orders itself with grid_dep_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_align(const AlignParams& p, cudaStream_t s);
cudaError_t launch_batch_prep(const BatchPrepParams& p, cudaStream_t s);
cudaError_t launch_quant_rows(const QuantRowsParams& p, cudaStream_t s);
cudaError_t launch_quant(const QuantParams& p, cudaStream_t s);
// tile kernel maps: tmA activation rows (5-D), tmB weight rows, tmAS activation scales (2-D),
// tmS weight block scales (1-D, 32-byte boxes), tmY / tmY3 the BF16 output (FC2; 8-row boxes and
// boxes of four 8-row groups 32 rows apart)
cudaError_t launch_fc1(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                       const CUtensorMap& tmS, const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_fc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                       const CUtensorMap& tmS, const CUtensorMap& tmY, const CUtensorMap& tmY3,
                       const GemmParams& p, int grid, cudaStream_t s);
// the same tile GEMMs for UE8M0 activation and weight scales, on the block-scaled MMA
cudaError_t launch_fc1_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                          const CUtensorMap& tmS, const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_fc2_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                          const CUtensorMap& tmS, const CUtensorMap& tmY, const CUtensorMap& tmY3,
                          const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_fc1_small(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmS,
                             const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_fc2_small(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmS,
                             const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t s);
cudaError_t launch_swiglu_quant(const SwigluQuantParams& p, cudaStream_t s);

}  // namespace moe
