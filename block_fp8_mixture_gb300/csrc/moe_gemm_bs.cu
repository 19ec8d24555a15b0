// Grouped FP8 x FP8 GEMM for layers whose activation and weight block scales are both UE8M0
// (powers of two), on the block-scaled tensor-core MMA: the scales are applied inside the MMA, so
// the whole K sum of a tile accumulates in tensor memory and no per-K-block promotion is needed.
//
// (vLLM "per-layer activation scale format + fused SiLU+quant", Details: the UE8M0 scale format
// and the block-FP8 layout of the experts; pinned arithmetic: with power-of-two scales a*s_a*s_w
// is exact, so the product of the dequantized operands equals the scaled dot of the codes up to
// the fp32 rounding of the accumulation.)
//
// Work items, tile placement, TMA producer and epilogues are those of the promotion kernel
// (moe_gemm.cu).  Per CTA:
//   warp 0 (one lane)  TMA producer: operand stages and scale slots.
//   warp 1 (one lane)  MMA issuer: per K block 4 block-scaled MMAs (M=128, N=256 over the gate and
//                      up rows, or the low and high output halves, K=32) into one 256-column fp32
//                      accumulator.
//   warps 4..7         scale-factor writers: per K block each thread writes its tile row's
//                      activation scale and the two weight block scales (each byte repeated in
//                      the four bytes of four consecutive 32-bit columns) into a 16-column
//                      tensor-memory slot of an 8-slot ring.
//   warps 8..15        epilogue: after the last K block they copy the accumulator to registers,
//                      release it (the next item's MMAs start) and run the FC1 / FC2 epilogue.
// Tile rows past the expert's live end carry whatever scale bytes the workspace holds; their
// results are discarded like their codes.
#include "moe_tile.cuh"

namespace moe {

constexpr int kBsThreads = 512;
constexpr int kBsSfWarp0 = 4;
constexpr int kBsEpiWarp0 = 8;
constexpr int kBsEpiWarps = 8;
constexpr int kBsRegsLow = 40;                 // warpgroups 0 and 1 after setmaxnreg
constexpr int kBsRegsHigh = 216;               // the two epilogue warpgroups
static_assert(2 * 128 * kBsRegsLow + 256 * kBsRegsHigh <= kBsThreads * 128,
              "register split must fit the launch allocation (128 registers a thread)");
constexpr int kBsSfSlots = 8;
constexpr uint32_t kBsSfCol0 = 256;            // scale-factor slots after the accumulator
constexpr uint32_t kBsSfSlotCols = 16;         // [0,4) activation, [4,8) weight 0, [8,12) weight 1
static_assert(kBsSfCol0 + kBsSfSlots * kBsSfSlotCols <= kTmemCols, "tensor memory columns");
constexpr uint32_t kBsIdesc = make_idesc_mx_e4m3(kBM, kGroup);
// One M = 128, N = 256 MMA runs a 128x256x128 K block in about 520 cycles; two N = 128 MMAs take
// about 770 (measured on this part with resident operands).
constexpr uint32_t kBsIdesc256 = make_idesc_mx_e4m3(kBM, 2 * kGroup);

__device__ __forceinline__ uint32_t rep4(uint32_t byte) { return byte * 0x01010101u; }

template <bool kFC1>
__global__ void __launch_bounds__(kBsThreads, 1)
    k_grouped_gemm_bs(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmAS, const __grid_constant__ CUtensorMap tmS,
                      const __grid_constant__ CUtensorMap tmY,
                      const __grid_constant__ CUtensorMap tmY3, const GemmParams p) {
  using TC = TileCfg<kFC1, true>;
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
  // barriers: full/empty[kStages], sfull/sempty[kSlots], sff/sfe[kBsSfSlots], tfull, tempty, drain
  constexpr int kBarF = 2 * kStages + 2 * kSlots;
  constexpr int kBarT = kBarF + 2 * kBsSfSlots;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (2 * kStages + kSlots + i); };
  auto sff_bar = [&](int j) { return bar0 + 8u * (kBarF + j); };
  auto sfe_bar = [&](int j) { return bar0 + 8u * (kBarF + kBsSfSlots + j); };
  const uint32_t tfull_bar = bar0 + 8u * kBarT;
  const uint32_t tempty_bar = bar0 + 8u * (kBarT + 1);
  const uint32_t drain_bar = bar0 + 8u * (kBarT + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (kBarT + 3));
  static_assert(8 * (kBarT + 3) + 16 <= 1024, "barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* mma_consumed = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* red = reinterpret_cast<float*>(ctrl + 1024);   // [2][kBM] row amax of each half

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);            // the MMAs have read the operands
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(sfull_bar(i), 1);
      mbar_init(sempty_bar(i), 4);           // the four scale-factor writers have read them
    }
    for (int j = 0; j < kBsSfSlots; ++j) {
      mbar_init(sff_bar(j), 4);              // the four writers have stored the slot
      mbar_init(sfe_bar(j), 1);              // the MMAs reading the slot have completed
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, kBsEpiWarps);
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
  // Inside the whole-layer forward, FC2 with per-tile FC1 counters does not wait for the FC1 grid:
  // its producer waits per row tile below.  The routing metadata it reads was complete before FC1's
  // CTAs passed their own dependency wait, which precedes this launch (FC1 is the kernel launched
  // just before).  The standalone FC2 step waits for the previous grid as well.
  if (kFC1 || p.tile_ready == nullptr || p.wait_prev_grid) grid_dep_wait();
  grid_dep_launch_dependents();

  const int num_tiles = *p.num_tiles;
  const int total = num_tiles * p.n_blocks * p.ksplit;
  const int KB = p.K / kBK;
  const int kb_per_split = KB / p.ksplit;
  int* status = p.status;
  const int nst_item = (kb_per_split + kPK - 1) / kPK;   // pipeline stages per work item
  int prod_issued = 0;

  if (warp < kBsEpiWarp0) {
    // warpgroups 0 (TMA, MMA) and 1 (scale-factor writers) give registers to the epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBsRegsLow));
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      int sc = 0;
      bool ok = true;
      int ready_tile = -1;
      const uint64_t pol_once = policy_evict_first();
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const Item w = decode_item(p, item);
        if (!kFC1 && p.tile_ready != nullptr && w.tile != ready_tile) {
          // every FC1 item of this row tile has written its FC2 input rows and scales
          if (!wait_counter_at_least(p.tile_ready + w.tile, p.fc1_items_per_tile, abort_flag,
                                     status)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
          ready_tile = w.tile;
        }
        const bool shared = expert_weights_shared(p, w, num_tiles);
        const int brow0 = kFC1 ? w.e * p.b_rows_per_expert + w.nb * kGroup
                               : w.e * p.b_rows_per_expert + w.nb * kBN;
        int sr0, sr1;
        bool has_sr1;
        scale_rows<kFC1>(p, w, sr0, sr1, has_sr1);
        for (int st = 0; st < nst_item; ++st) {
          const int kbs = w.ks * kb_per_split + st * kPK;
          const int s = sc % kStages;
          const int sl = sc % kSlots;
          if (!mbar_wait(empty_bar(s), ((sc / kStages) & 1) ^ 1, abort_flag, status) ||
              !mbar_wait(sempty_bar(sl), ((sc / kSlots) & 1) ^ 1, abort_flag, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), kABytes + 2 * kBHalfBytes);
          mbar_arrive_expect_tx(sfull_bar(sl), kPK * kBM + (has_sr1 ? 64 : 32));
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
          const int i0 = sr0 * KB + kbs;
          tma_load_1d(sS + kSlotW, &tmS, i0 - i0 % 16, sfull_bar(sl));
          if (has_sr1) {
            const int i1 = sr1 * KB + kbs;
            tma_load_1d(sS + kSlotW + 128, &tmS, i1 - i1 % 16, sfull_bar(sl));
          }
          ++sc;
        }
      }
      prod_issued = sc;
    } else if (warp == 1 && lane == 0) {
      // --------------------------------------------------------------- MMA
      int sc = 0, c = 0, n_items = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x, ++n_items) {
        const Item w = decode_item(p, item);
        const bool second = kFC1 || (w.nb * kBN + kGroup) < p.out_cols;
        const int kb_end = (w.ks + 1) * kb_per_split;
        int kb_item = 0;
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
          for (int k = 0; k < nv; ++k, ++kb_item) {
            const int j = c % kBsSfSlots;
            // the accumulator is free once the previous item's epilogue has copied it out
            if (!mbar_wait(sff_bar(j), (c / kBsSfSlots) & 1, abort_flag, status) ||
                (kb_item == 0 && !mbar_wait(tempty_bar, (n_items & 1) ^ 1, abort_flag, status))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t sf = tmem_base + kBsSfCol0 + j * kBsSfSlotCols;
            const uint64_t adesc = make_sdesc_sw128(sA + k * (kABoxRows * kBK), kABoxRows * kBK * kPK);
            const uint64_t b0_desc = make_sdesc_sw128(sB + k * (kGroup * kBK));
            const uint64_t b1_desc = make_sdesc_sw128(sB + kBHalfBytes + k * (kGroup * kBK));
#pragma unroll
            for (int kk = 0; kk < kBK / 32; ++kk) {
              const uint32_t accum = (kb_item > 0 || kk > 0) ? 1u : 0u;
              if constexpr (kPK == 1) {
                // the two 128-row weight halves are contiguous: one N = 256 MMA per K step (the
                // scale factors of rows 128..255 are read from the slot's next column group)
                mma_f8_bs(tmem_base, adesc + 2 * kk, b0_desc + 2 * kk, kBsIdesc256, sf, sf + 4, accum);
              } else {
                mma_f8_bs(tmem_base, adesc + 2 * kk, b0_desc + 2 * kk, kBsIdesc, sf, sf + 4, accum);
                if (second)
                  mma_f8_bs(tmem_base + kGroup, adesc + 2 * kk, b1_desc + 2 * kk, kBsIdesc, sf, sf + 8,
                            accum);
              }
            }
            mma_commit(sfe_bar(j));
            ++c;
          }
          if (!ok) break;
          mma_commit(empty_bar(s));
          ++sc;
          *mma_consumed = sc;
        }
        if (ok) mma_commit(tfull_bar);
      }
    } else if (warp >= kBsSfWarp0) {
      // ------------------------------------------------- scale-factor writers
      const int q = warp & 3;
      const int row = 32 * (lane >> 3) + 8 * q + (lane & 7);   // tile row of lane 32q + lane
      const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
      int sc = 0, c = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
        const Item w = decode_item(p, item);
        int sr0, sr1;
        bool has_sr1;
        scale_rows<kFC1>(p, w, sr0, sr1, has_sr1);
        const int kb_end = (w.ks + 1) * kb_per_split;
        for (int st = 0; ok && st < nst_item; ++st) {
          const int kbs = w.ks * kb_per_split + st * kPK;
          const int nv = min(kPK, kb_end - kbs);
          const int sl = sc % kSlots;
          const uint8_t* slot = slots + sl * kScaleSlotBytes;
          if (!mbar_wait(sfull_bar(sl), (sc / kSlots) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          const int i0 = sr0 * KB + kbs, i1 = sr1 * KB + kbs;
          for (int k = 0; k < nv; ++k) {
            const int j = c % kBsSfSlots;
            if (!mbar_wait(sfe_bar(j), ((c / kBsSfSlots) & 1) ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t a = rep4(slot[k * kBM + row]);
            const uint32_t b0 = rep4(slot[kSlotW + i0 % 16 + k]);
            const uint32_t b1 = has_sr1 ? rep4(slot[kSlotW + 128 + i1 % 16 + k]) : rep4(127u);
            const uint32_t t = lane_base + kBsSfCol0 + j * kBsSfSlotCols;
            tmem_st4(t, a, a, a, a);
            tmem_st4(t + 4, b0, b0, b0, b0);
            tmem_st4(t + 8, b1, b1, b1, b1);
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(sff_bar(j));
            ++c;
          }
          if (!ok) break;
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty_bar(sl));
          ++sc;
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBsRegsHigh));
    // ------------------------------------------------------------- epilogue
    const int ew = warp - kBsEpiWarp0;
    const int wg = ew >> 2;                        // which half of the 256 columns
    const int q = warp & 3;                        // TMEM lane quarter this warp may access
    const int row = 32 * (lane >> 3) + 8 * q + (lane & 7);   // tile row held in lane 32q + lane
    int n_items = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x, ++n_items) {
      const Item w = decode_item(p, item);
      const bool qlive = 8 * q < w.live;
      const bool rlive = row < w.live;
      if (!mbar_wait(tfull_bar, n_items & 1, abort_flag, status)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float acc[128];
      if (qlive) {
        const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16);
        uint32_t r[4][32];
        if (kFC1) {
          tmem_ld32(t0 + wg * 64, r[0]);
          tmem_ld32(t0 + wg * 64 + 32, r[1]);
          tmem_ld32(t0 + kGroup + wg * 64, r[2]);
          tmem_ld32(t0 + kGroup + wg * 64 + 32, r[3]);
        } else {
          tmem_ld32(t0 + wg * 128, r[0]);
          tmem_ld32(t0 + wg * 128 + 32, r[1]);
          tmem_ld32(t0 + wg * 128 + 64, r[2]);
          tmem_ld32(t0 + wg * 128 + 96, r[3]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[32 * i + j] = __uint_as_float(r[i][j]);
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar);     // the next item's MMAs may overwrite it
      if (kFC1) {
        fc1_item_epilogue(p, w, acc, row, wg, rlive, red);
        if (p.tile_ready != nullptr) {
          // the item's FC2 input rows are written: count it for its row tile (release at GPU scope
          // after all 256 epilogue threads' stores)
          named_barrier_sync(1, kTileEpiThreadsBar);
          if (ew == 0 && lane == 0) {
            __threadfence();
            atomicAdd(p.tile_ready + w.tile, 1);
          }
        }
      } else {
        if (TC::YByGroup)
          fc2_item_epilogue_by_group(p, w, acc, row, wg, q, lane, qlive, rlive,
                                     ystage + ew * TC::YWarpBytes, &tmY);
        else
          fc2_item_epilogue(p, w, acc, row, wg, q, lane, qlive, rlive, ystage + ew * TC::YWarpBytes,
                            &tmY, &tmY3);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  if (!kFC1 && warp >= kBsEpiWarp0 && lane == 0) bulk_wait_group0();   // output stores complete
  __syncthreads();
  if (warp == 1 && lane == 0) {
    // every MMA this CTA issued has completed (and its barrier arrivals have landed)
    mma_commit(drain_bar);
    drain_wait(drain_bar, 0, status);
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    // copies issued but never consumed are still in flight: wait for them before leaving
    for (int st = *mma_consumed; st < prod_issued; ++st)
      drain_wait(full_bar(st % kStages), (st / kStages) & 1, status);
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
static cudaError_t launch_gemm_bs(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const CUtensorMap& tmAS, const CUtensorMap& tmS,
                                  const CUtensorMap& tmY, const CUtensorMap& tmY3,
                                  const GemmParams& p, int grid, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(k_grouped_gemm_bs<kFC1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TileCfg<kFC1, true>::Smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_grouped_gemm_bs<kFC1>, dim3(grid), dim3(kBsThreads), TileCfg<kFC1, true>::Smem, s,
                    tmA, tmB, tmAS, tmS, tmY, tmY3, p);
}

cudaError_t launch_fc1_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                          const CUtensorMap& tmS, const GemmParams& p, int grid, cudaStream_t s) {
  return launch_gemm_bs<true>(tmA, tmB, tmAS, tmS, tmA, tmA, p, grid, s);
}

cudaError_t launch_fc2_bs(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                          const CUtensorMap& tmS, const CUtensorMap& tmY, const CUtensorMap& tmY3,
                          const GemmParams& p, int grid, cudaStream_t s) {
  return launch_gemm_bs<false>(tmA, tmB, tmAS, tmS, tmY, tmY3, p, grid, s);
}

}  // namespace moe
