// Persistent grouped FP8 x FP8 GEMM over live 128-row tiles for FP32 block scales (per-128-K
// promotion through registers), with the FC1 (SwiGLU + 1x128 requant, or BF16 (gate | up) rows for
// the separate SwiGLU kernel) and FC2 (BF16 store) epilogues.
//
// (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose: both grouped GEMMs visit only
// the live (expert, row-tile) work named by the prefix-sum endpoints, and the fused activation
// quantization consumes the same endpoints; SM90 section: whole padded tiles are skipped, padding
// inside a partially filled tile remains.  TensorRT-LLM "Triton FP8-activation MoE for
// decode-sized batches on Hopper", human review: per 128-wide K block the partial sum is scaled by
// the product a_scale*b_scale formed first.)
//
// Work item = (live row tile, output column block).  One CTA per SM walks items blockIdx.x,
// blockIdx.x + gridDim.x, ...; inside the CTA:
//   warp 0 (one lane)  TMA producer.  Each stage of the operand ring receives the tile's 128
//                      activation rows (one 5-D box that also permutes the 8-row groups, below)
//                      and its 256 weight rows (one box, 128-byte swizzle) for one 128-wide K
//                      block; a separate, deeper ring of scale slots receives the stage's
//                      activation scales (one 2-D box) and two 32-byte boxes of weight block
//                      scales.  Five copies per stage.  The MMA releases an operand stage on
//                      completion, the promotion warps release the scale slot once they have
//                      read it.  Rows of a tile past the expert's live end are loaded too (they
//                      stay inside the workspace) and their results are discarded.
//   warp 1 (one lane)  MMA issuer: per K block 4 tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32)
//                      into one of two 256-column fp32 accumulators in tensor memory.
//   warps 4..11        promotion + epilogue (232 registers after setmaxnreg).  A thread owns one
//                      row and 128 of the 256 columns; per K block it reads its partial sums from
//                      tensor memory (two loads in flight per wait) and accumulates
//                      acc = fma(partial, a_scale*b_scale, acc) in registers, then releases the
//                      accumulator so the MMA of a later K block overlaps the promotion.
// Row placement: 8-row group j = 4a + b of the tile (rows 32a + 8b ..) lands in shared-memory group
// 4b + a, i.e. tensor-memory lanes 32b + 8a .. +7, so even a tile with 8..32 live rows keeps all
// four lane quarters (all eight promotion warps) busy.
// FC1 columns: 128 gate rows of W13 and the matching 128 up rows, so a thread owns 64 (gate, up)
// pairs of one row.  When the workspace has an FC1 output region the thread stores its BF16 gate
// and up values and SwiGLU + requantization run as their own kernel (the fused epilogue cannot
// overlap the mainloop); otherwise it applies SwiGLU and the 1x128 requantization, which need only
// the row amax of the two threads sharing the row.  FC2 columns: 256 consecutive hidden columns,
// BF16 out.
#include "moe_tile.cuh"

namespace moe {

// M = 128, N = 256: one MMA per K step when the two weight halves are contiguous (one K block per
// stage); about 520 cycles per 128x256x128 K block against about 770 for two N = 128 MMAs
constexpr uint32_t kIdesc256 = make_idesc_e4m3(kBM, 2 * kGroup);

// acc[0..63] += partial[t0 .. t0+31, t1 .. t1+31] * sab: both tensor-memory loads in flight before
// the one wait, so a K block costs two load round trips instead of four.
__device__ __forceinline__ void promote64(uint32_t t0, uint32_t t1, float sab, float* acc) {
  uint32_t r0[32], r1[32];
  tmem_ld32(t0, r0);
  tmem_ld32(t1, r1);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = fmaf(__uint_as_float(r0[i]), sab, acc[i]);
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[32 + i] = fmaf(__uint_as_float(r1[i]), sab, acc[32 + i]);
}

template <bool kFC1>
__global__ void __launch_bounds__(kTileThreads, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmAS, const __grid_constant__ CUtensorMap tmS,
                   const __grid_constant__ CUtensorMap tmY,
                   const __grid_constant__ CUtensorMap tmY3, const GemmParams p) {
  using TC = TileCfg<kFC1>;
  constexpr int kPK = TC::PK;
  constexpr int kStages = TC::Stages;
  constexpr int kStageBytes = TC::StageBytes;
  constexpr int kABytes = TC::ABytes;
  constexpr int kBHalfBytes = TC::BHalf;
  constexpr int kScaleSlotBytes = TC::SlotBytes;
  constexpr int kSlots = TC::ScaleSlots;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  uint8_t* ystage = smem + kStages * kStageBytes;              // FC2 output staging, 1024-aligned
  uint8_t* slots = ystage + 8 * TC::YWarpBytes;                 // scale slots, 128-byte aligned
  uint8_t* ctrl = slots + kSlots * kScaleSlotBytes;
  const uint32_t slot0 = smem_addr(slots);
  const uint32_t bar0 = smem_addr(ctrl);
  // barriers: full[kStages], empty[kStages], sfull[kSlots], sempty[kSlots], tfull[2], tempty[2],
  // drain
  constexpr int kBarT = 2 * kStages + 2 * kSlots;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + kSlots + i); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (kBarT + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (kBarT + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (kBarT + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (kBarT + 5));
  static_assert(8 * (kBarT + 5) + 16 <= 1024, "barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* mma_consumed = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* red = reinterpret_cast<float*>(ctrl + 1024);   // [2][kBM] row amax of each half

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kEpiWarps = kEpiThreads / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);            // the MMAs have read the operands
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(sfull_bar(i), 1);
      mbar_init(sempty_bar(i), kEpiWarps);   // every promotion warp has read the scales
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *mma_consumed = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmAS);
    prefetch_tensormap(&tmS);
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_wait();                 // the previous kernel's outputs are complete from here on
  grid_dep_launch_dependents();

  const int num_tiles = *p.num_tiles;
  const int total = num_tiles * p.n_blocks * p.ksplit;
  const int KB = p.K / kBK;
  const int kb_per_split = KB / p.ksplit;
  const int a_ue = p.a_scale_ue8m0, b_ue = p.b_scale_ue8m0;
  const int a_kb_bytes = a_ue ? kBM : kBM * 4;   // activation scales of one K block in a slot
  const int w_mask = b_ue ? 15 : 3;              // scale elements per 16 bytes, minus one
  int* status = p.status;

  const int nst_item = (kb_per_split + kPK - 1) / kPK;   // pipeline stages per work item
  int prod_issued = 0;
  if (warp < kTileEpiWarp0) {
  // registers move from warpgroup 0 (TMA / MMA issue) to the promotion warpgroups
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTileRegsLow));
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int sc = 0;
    bool ok = true;
    const uint64_t pol_once = policy_evict_first();
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Item w = decode_item(p, item);
      const bool shared = expert_weights_shared(p, w, num_tiles);
      // FC1: 128 gate rows and the matching 128 up rows (the map's outer dimension steps I rows);
      // FC2: 256 consecutive hidden rows (past the expert's last block they are never used)
      const int brow0 = kFC1 ? w.e * p.b_rows_per_expert + w.nb * kGroup
                             : w.e * p.b_rows_per_expert + w.nb * kBN;
      int sr0, sr1;
      bool has_sr1;
      scale_rows<kFC1>(p, w, sr0, sr1, has_sr1);
      for (int st = 0; st < nst_item; ++st) {
        const int kbs = w.ks * kb_per_split + st * kPK;       // first K block of the stage
        const int s = sc % kStages;
        const uint32_t ph = (sc / kStages) & 1;
        const int sl = sc % kSlots;
        if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, status) ||
            !mbar_wait(sempty_bar(sl), ((sc / kSlots) & 1) ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        // every box is delivered whole (kPK K blocks; past the end of a dimension as zeros)
        mbar_arrive_expect_tx(full_bar(s), kABytes + 2 * kBHalfBytes);
        mbar_arrive_expect_tx(sfull_bar(sl), kPK * a_kb_bytes + (has_sr1 ? 64 : 32));
        const uint32_t sA = sbase + s * kStageBytes;
        const uint32_t sB = sA + kABytes;
        const uint32_t sS = slot0 + sl * kScaleSlotBytes;
        tma_load_5d(sA, &tmA, 0, 0, kbs, w.m0 / 32, 0, full_bar(s));
        if (kFC1 && shared)
          tma_load_4d(sB, &tmB, 0, brow0, kbs, 0, full_bar(s));
        else if (kFC1)
          tma_load_4d_hint(sB, &tmB, 0, brow0, kbs, 0, full_bar(s), pol_once);
        else if (shared)
          tma_load_3d(sB, &tmB, 0, brow0, kbs, full_bar(s));
        else
          tma_load_3d_hint(sB, &tmB, 0, brow0, kbs, full_bar(s), pol_once);
        tma_load_2d(sS, &tmAS, w.m0, kbs, sfull_bar(sl));
        // a 32-byte box from the 16-byte boundary at or below the stage's first block scale
        // holds the scales of all kPK K blocks
        const int i0 = sr0 * KB + kbs;
        tma_load_1d(sS + kSlotW, &tmS, i0 & ~w_mask, sfull_bar(sl));
        if (has_sr1) {
          const int i1 = sr1 * KB + kbs;
          tma_load_1d(sS + kSlotW + 128, &tmS, i1 & ~w_mask, sfull_bar(sl));
        }
        ++sc;
      }
    }
    prod_issued = sc;
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA
    int sc = 0, c = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Item w = decode_item(p, item);
      const int kb_end = (w.ks + 1) * kb_per_split;
      for (int st = 0; ok && st < nst_item; ++st) {
        const int kbs = w.ks * kb_per_split + st * kPK;
        const int nv = min(kPK, kb_end - kbs);
        const int s = sc % kStages;
        if (!mbar_wait(full_bar(s), (sc / kStages) & 1, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t sA = sbase + s * kStageBytes;
        const uint32_t sB = sA + kABytes;
        for (int k = 0; k < nv; ++k) {
          const int b = c & 1;
          if (!mbar_wait(tempty_bar(b), ((c >> 1) & 1) ^ 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d = tmem_base + b * kBN;
          const uint64_t adesc = make_sdesc_sw128(sA + k * (kABoxRows * kBK), kABoxRows * kBK * kPK);
          static_assert(kPK == 1, "one K block per stage: the two weight halves are contiguous");
          // both 128-row weight halves (gate and up, or low and high) are contiguous: one N = 256
          // MMA per K step
          const uint64_t b_desc = make_sdesc_sw128(sB + k * (kGroup * kBK));
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8(d, adesc + 2 * kk, b_desc + 2 * kk, kIdesc256, kk > 0 ? 1u : 0u);
          mma_commit(tfull_bar(b));
          ++c;
        }
        if (!ok) break;
        mma_commit(empty_bar(s));
        ++sc;
        *mma_consumed = sc;
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTileRegsHigh));
    // ---------------------------------------------------- promotion + epilogue
    const int ew = warp - kTileEpiWarp0;
    const int wg = ew >> 2;                        // which half of the 256 columns
    const int q = warp & 3;                        // TMEM lane quarter this warp may access
    const int row = 32 * (lane >> 3) + 8 * q + (lane & 7);   // tile row held in lane 32q + lane
    int c = 0, sc = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Item w = decode_item(p, item);
      const bool qlive = 8 * q < w.live;
      const bool rlive = row < w.live;
      int sr0, sr1;
      bool has_sr1;
      scale_rows<kFC1>(p, w, sr0, sr1, has_sr1);
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      const int kb_end = (w.ks + 1) * kb_per_split;
      for (int st = 0; ok && st < nst_item; ++st) {
        const int kbs = w.ks * kb_per_split + st * kPK;
        const int nv = min(kPK, kb_end - kbs);
        const int sl = sc % kSlots;
        const uint8_t* slot = slots + sl * kScaleSlotBytes;
        for (int k = 0; k < nv; ++k) {
          const int b = c & 1;
          // the scales need only their slot: read them before waiting for the partial sums, and
          // give the slot back to the producer once the stage's last K block has read them
          if (k == 0 && !mbar_wait(sfull_bar(sl), (sc / kSlots) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          // loads only: their values are first used after the wait below
          float sa = 0.0f, sw0 = 0.0f, sw1 = 0.0f;
          if (qlive) {
            const int i0 = sr0 * KB + kbs, i1 = sr1 * KB + kbs;
            sa = smem_scale_at(slot + k * a_kb_bytes, row, a_ue);
            sw0 = smem_scale_at(slot + kSlotW, (i0 & w_mask) + k, b_ue);
            if (has_sr1) sw1 = smem_scale_at(slot + kSlotW + 128, (i1 & w_mask) + k, b_ue);
          }
          if (k == nv - 1) {
            __syncwarp();
            if (lane == 0) mbar_arrive(sempty_bar(sl));   // this warp has read the stage's scales
          }
          if (!mbar_wait(tfull_bar(b), (c >> 1) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (qlive) {
            const float sab0 = __fmul_rn(sa, sw0), sab1 = __fmul_rn(sa, sw1);
            const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16) + b * kBN;
            if (kFC1) {
              promote64(t0 + wg * 64, t0 + wg * 64 + 32, sab0, acc);
              promote64(t0 + kGroup + wg * 64, t0 + kGroup + wg * 64 + 32, sab1, acc + 64);
            } else {
              const float sab = wg == 0 ? sab0 : sab1;
              promote64(t0 + wg * 128, t0 + wg * 128 + 32, sab, acc);
              promote64(t0 + wg * 128 + 64, t0 + wg * 128 + 96, sab, acc + 64);
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(b));
          ++c;
        }
        if (!ok) break;
        ++sc;
      }
      if (!ok) break;

      if (kFC1) {
        if (p.g1 != nullptr)
          fc1_item_store_g1(p, w, acc, row, wg, rlive);
        else
          fc1_item_epilogue(p, w, acc, row, wg, rlive, red);
      } else {
        fc2_item_epilogue(p, w, acc, row, wg, q, lane, qlive, rlive, ystage + ew * TC::YWarpBytes,
                          &tmY, &tmY3);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  if (!kFC1 && warp >= kTileEpiWarp0 && lane == 0) bulk_wait_group0();   // output stores complete
  __syncthreads();
  if (warp == 1 && lane == 0) {
    // every MMA this CTA issued has completed (and its barrier arrivals have landed)
    mma_commit(drain_bar);
    drain_wait(drain_bar, 0, status);
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    // stages issued but never consumed are still in flight: wait for them before leaving
    for (int st = *mma_consumed; st < prod_issued; ++st)
      drain_wait(full_bar(st % kStages), (st / kStages) & 1, status);
    // scale copies: the latest use of each slot (earlier uses completed before it was reissued)
    for (int st = max(0, prod_issued - kSlots); st < prod_issued; ++st)
      drain_wait(sfull_bar(st % kSlots), (st / kSlots) & 1, status);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kFC1>
static cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                               const CUtensorMap& tmS, const CUtensorMap& tmY, const CUtensorMap& tmY3,
                               const GemmParams& p, int grid, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(k_grouped_gemm<kFC1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TileCfg<kFC1>::Smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_grouped_gemm<kFC1>, dim3(grid), dim3(kTileThreads), TileCfg<kFC1>::Smem, s, tmA,
                    tmB, tmAS, tmS, tmY, tmY3, p);
}

cudaError_t launch_fc1(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                       const CUtensorMap& tmS, const GemmParams& p, int grid, cudaStream_t s) {
  return launch_gemm<true>(tmA, tmB, tmAS, tmS, tmA, tmA, p, grid, s);   // FC1 stores no BF16 tile
}

cudaError_t launch_fc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                       const CUtensorMap& tmS, const CUtensorMap& tmY, const CUtensorMap& tmY3,
                       const GemmParams& p, int grid, cudaStream_t s) {
  return launch_gemm<false>(tmA, tmB, tmAS, tmS, tmY, tmY3, p, grid, s);
}

}  // namespace moe
