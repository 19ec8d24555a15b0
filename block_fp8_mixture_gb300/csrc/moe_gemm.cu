// Persistent grouped FP8 x FP8 GEMM over live row tiles, with the FC1 (SwiGLU + 1x128 requant)
// and FC2 (BF16 store) epilogues.
//
// (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose: both grouped GEMMs visit only
// the live (expert, row-tile) work named by the prefix-sum endpoints, and the fused activation
// quantization consumes the same endpoints; SM90 section: whole padded tiles are skipped, padding
// inside a partially filled tile remains.  TensorRT-LLM "Triton FP8-activation MoE for
// decode-sized batches on Hopper", human review: per 128-wide K block the partial sum is scaled by
// the product a_scale*b_scale formed first.)
//
// Work item = (live row tile, output column block, K split).  One CTA per SM walks items
// blockIdx.x, blockIdx.x + gridDim.x, ...; inside the CTA:
//   warp 0 (one lane)  TMA producer.  Each stage of the operand ring receives the tile's 128
//                      activation rows (one 5-D box that also permutes the 8-row groups, below)
//                      and its 256 weight rows (one box, 128-byte swizzle) for one or two 128-wide
//                      K blocks; a separate, deeper ring of scale slots receives the stage's
//                      activation scales (one 2-D box) and two 32-byte boxes of weight block
//                      scales.  Five copies per stage.  The MMA releases an operand stage on
//                      completion, the promotion warps release the scale slot once they have
//                      read it.  Rows of a tile past the expert's live end are loaded too (they
//                      stay inside the workspace) and their results are discarded.
//   warp 1 (one lane)  MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (M=128, N=256, K=32) per K block
//                      into one of two 256-column fp32 accumulators in tensor memory.
//   warps 2..9         promotion + epilogue.  A thread owns one row and 128 of the 256 columns;
//                      per K block it reads its partial sums from tensor memory and accumulates
//                      acc = fma(partial, a_scale*b_scale, acc) in registers, then releases the
//                      accumulator so the MMA of a later K block overlaps the promotion.
// Row placement: 8-row group j = 4a + b of the tile (rows 32a + 8b ..) lands in shared-memory group
// 4b + a, i.e. tensor-memory lanes 32b + 8a .. +7, so even a tile with 8..32 live rows keeps all
// four lane quarters (all eight promotion warps) busy.
// FC1 columns: 128 gate rows of W13 and the matching 128 up rows, so a thread owns 64 (gate, up)
// pairs of one row; the SwiGLU and the 1x128 requantization need only the row amax of the two
// threads sharing the row.  FC2 columns: 256 consecutive hidden columns, BF16 out.
// Small batches split K across CTAs (FC1 only): each split writes its fp32 partial rows, the last
// split to arrive (atomic counter per item) sums the splits in fixed order and runs the epilogue.
#include "moe_device.cuh"

namespace moe {

constexpr uint32_t kIdesc = make_idesc_e4m3(kBM, kGroup);   // M = 128, N = 128 per MMA

struct Item {
  int tile, nb, ks, e, m0, live;
};

__device__ __forceinline__ Item decode_item(const GemmParams& p, int item) {
  Item it;
  const int per_tile = p.n_blocks * p.ksplit;
  it.tile = item / per_tile;
  const int rem = item - it.tile * per_tile;
  it.nb = rem / p.ksplit;
  it.ks = rem - it.nb * p.ksplit;
  // tiles are contiguous from row 0 (routed layer) or listed (batched-expert layout)
  it.m0 = p.tile_row0 != nullptr ? p.tile_row0[it.tile] : it.tile * kBM;
  it.e = p.tile_expert[it.m0 / kBM];
  it.live = min(kBM, p.live_end[it.e] - it.m0);
  return it;
}

// Weight block-scale rows of an item (indices into the [E][row blocks][K/128] scale array).
// FC1: the gate block nb and the up block I/128 + nb.  FC2: hidden blocks 2nb and 2nb + 1.
template <bool kFC1>
__device__ __forceinline__ void scale_rows(const GemmParams& p, const Item& w, int& r0, int& r1,
                                           bool& has_r1) {
  const int ncb = p.b_rows_per_expert / kGroup;
  if (kFC1) {
    r0 = w.e * ncb + w.nb;
    r1 = w.e * ncb + p.out_cols / kGroup + w.nb;
    has_r1 = true;
  } else {
    r0 = w.e * ncb + 2 * w.nb;
    r1 = r0 + 1;
    has_r1 = 2 * w.nb + 1 < ncb;
  }
}

// SiLU(g) * u with the optional clamp, fp32, IEEE division, no fused multiply-add.
__device__ __forceinline__ float swiglu(float g, float u, int mode, float lim) {
  if (mode == MOE_CLAMP_BEFORE_SILU) {
    g = fminf(g, lim);
    u = fminf(fmaxf(u, -lim), lim);
  }
  const float sig = __frcp_rn(__fadd_rn(1.0f, expf(-g)));   // correctly rounded 1/(1+e^-g)
  float silu = __fmul_rn(g, sig);
  if (mode == MOE_CLAMP_AFTER_SILU) {
    silu = fminf(silu, lim);
    u = fminf(fmaxf(u, -lim), lim);
  }
  return __fmul_rn(silu, u);
}

// Bounded wait used while tearing down: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ void promote32(uint32_t taddr, float sab, float* acc) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = fmaf(__uint_as_float(r[i]), sab, acc[i]);
}

template <bool kFC1>
__global__ void __launch_bounds__(kTileThreads, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmAS, const __grid_constant__ CUtensorMap tmS,
                   const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
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
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);
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
    *last_flag = 0;
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
  const int w_per16 = b_ue ? 16 : 4;             // scale elements per 16 bytes
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
    const uint64_t pol_w = policy_evict_first();
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Item w = decode_item(p, item);
      // FC1: 128 gate rows and the matching 128 up rows (the map's outer dimension steps I rows);
      // FC2: 256 consecutive hidden rows (past the expert's last block they are never used)
      const int brow0 = kFC1 ? w.e * p.b_rows_per_expert + w.nb * kGroup
                             : w.e * p.b_rows_per_expert + w.nb * kBN;
      int sr0, sr1;
      bool has_sr1;
      scale_rows<kFC1>(p, w, sr0, sr1, has_sr1);
      const int kb_end = (w.ks + 1) * kb_per_split;
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
        if (kFC1)
          tma_load_4d_hint(sB, &tmB, 0, brow0, kbs, 0, full_bar(s), pol_w);
        else
          tma_load_3d_hint(sB, &tmB, 0, brow0, kbs, full_bar(s), pol_w);
        tma_load_2d(sS, &tmAS, w.m0, kbs, sfull_bar(sl));
        // a 32-byte box from the 16-byte boundary at or below the stage's first block scale
        // holds the scales of all kPK K blocks
        const int i0 = sr0 * KB + kbs;
        tma_load_1d(sS + kSlotW, &tmS, i0 - i0 % w_per16, sfull_bar(sl));
        if (has_sr1) {
          const int i1 = sr1 * KB + kbs;
          tma_load_1d(sS + kSlotW + 128, &tmS, i1 - i1 % w_per16, sfull_bar(sl));
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
      const bool second = kFC1 || (w.nb * kBN + kGroup) < p.out_cols;
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
          const uint64_t g_desc = make_sdesc_sw128(sB + k * (kGroup * kBK));
          const uint64_t u_desc = make_sdesc_sw128(sB + kBHalfBytes + k * (kGroup * kBK));
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk) {
            mma_f8(d, adesc + 2 * kk, g_desc + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
            if (second) mma_f8(d + kGroup, adesc + 2 * kk, u_desc + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
          }
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
          if (!mbar_wait(tfull_bar(b), (c >> 1) & 1, abort_flag, status) ||
              (k == 0 && !mbar_wait(sfull_bar(sl), (sc / kSlots) & 1, abort_flag, status))) {
            ok = false;
            break;
          }
          float sab0 = 0.0f, sab1 = 0.0f;
          if (qlive) {
            const float sa = smem_scale_at(slot + k * a_kb_bytes, row, a_ue);
            const int i0 = sr0 * KB + kbs, i1 = sr1 * KB + kbs;
            const float sw0 = smem_scale_at(slot + kSlotW, i0 % w_per16 + k, b_ue);
            const float sw1 = has_sr1 ? smem_scale_at(slot + kSlotW + 128, i1 % w_per16 + k, b_ue)
                                      : 0.0f;
            sab0 = __fmul_rn(sa, sw0);
            sab1 = __fmul_rn(sa, sw1);
          }
          tc_fence_after_sync();
          if (qlive) {
            const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16) + b * kBN;
            if (kFC1) {
              promote32(t0 + wg * 64, sab0, acc);
              promote32(t0 + wg * 64 + 32, sab0, acc + 32);
              promote32(t0 + kGroup + wg * 64, sab1, acc + 64);
              promote32(t0 + kGroup + wg * 64 + 32, sab1, acc + 96);
            } else {
              const float sab = wg == 0 ? sab0 : sab1;
              promote32(t0 + wg * 128, sab, acc);
              promote32(t0 + wg * 128 + 32, sab, acc + 32);
              promote32(t0 + wg * 128 + 64, sab, acc + 64);
              promote32(t0 + wg * 128 + 96, sab, acc + 96);
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(b));
          ++c;
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(sempty_bar(sl));   // this warp has read the stage's scales
        ++sc;
      }
      if (!ok) break;

      if (kFC1) {
        const int I = p.out_cols;
        if (p.ksplit > 1) {
          // split-K fix-up: publish this split's partial rows, the last split sums all of them
          const int pair = rlive ? p.sorted_pair[w.m0 + row] : 0;
          if (rlive) {
            float* dst = p.splitk_partial + ((size_t)w.ks * p.P_cap + pair) * (2 * I);
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
              *reinterpret_cast<float4*>(dst + w.nb * kGroup + wg * 64 + i) =
                  make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
              *reinterpret_cast<float4*>(dst + I + w.nb * kGroup + wg * 64 + i) =
                  make_float4(acc[64 + i], acc[65 + i], acc[66 + i], acc[67 + i]);
            }
          }
          __threadfence();
          named_barrier_sync(1, kEpiThreads);
          if (ew == 0 && lane == 0) {
            const int prev = atomicAdd(&p.splitk_count[w.tile * p.n_blocks + w.nb], 1);
            *last_flag = (prev == p.ksplit - 1);
          }
          named_barrier_sync(1, kEpiThreads);
          const bool last = *last_flag != 0;
          named_barrier_sync(1, kEpiThreads);
          if (!last) continue;
          __threadfence();
          if (ew == 0 && lane == 0) p.splitk_count[w.tile * p.n_blocks + w.nb] = 0;
          if (rlive) {
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            for (int s = 0; s < p.ksplit; ++s) {
              const float* src = p.splitk_partial + ((size_t)s * p.P_cap + pair) * (2 * I);
#pragma unroll
              for (int i = 0; i < 64; i += 4) {
                const float4 g = __ldcg(reinterpret_cast<const float4*>(src + w.nb * kGroup + wg * 64 + i));
                const float4 u = __ldcg(reinterpret_cast<const float4*>(src + I + w.nb * kGroup + wg * 64 + i));
                acc[i] = __fadd_rn(acc[i], g.x);
                acc[i + 1] = __fadd_rn(acc[i + 1], g.y);
                acc[i + 2] = __fadd_rn(acc[i + 2], g.z);
                acc[i + 3] = __fadd_rn(acc[i + 3], g.w);
                acc[64 + i] = __fadd_rn(acc[64 + i], u.x);
                acc[65 + i] = __fadd_rn(acc[65 + i], u.y);
                acc[66 + i] = __fadd_rn(acc[66 + i], u.z);
                acc[67 + i] = __fadd_rn(acc[67 + i], u.w);
              }
            }
          }
        }
        // SwiGLU on the BF16-rounded FC1 outputs, then 1x128 requantization over the row's 128
        // (gate, up) columns held by this thread (64) and its partner in the other half (64).
        float amax = 0.0f;
        if (rlive) {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            float h = swiglu(bf16_round(acc[i]), bf16_round(acc[64 + i]), p.clamp_mode,
                             p.clamp_limit);
            if (p.numerics == MOE_NUMERICS_RECIPROCAL) h = bf16_round(h);
            acc[i] = h;
            amax = fmaxf(amax, fabsf(h));
          }
        }
        red[wg * kBM + row] = amax;
        named_barrier_sync(1, kEpiThreads);
        amax = fmaxf(red[row], red[kBM + row]);
        named_barrier_sync(1, kEpiThreads);
        if (rlive) {
          float inv;
          const float s = group_scale_numerics(amax, p.act_fmt, p.numerics, &inv);
          uint8_t* dst = p.a2_q + (size_t)(w.m0 + row) * I + w.nb * kGroup + wg * 64;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t wd[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float* h = acc + v * 16 + j * 4;
              wd[j] = cvt_e4m3x2(quant_div(h[0], s, inv), quant_div(h[1], s, inv)) |
                      (cvt_e4m3x2(quant_div(h[2], s, inv), quant_div(h[3], s, inv)) << 16);
            }
            *reinterpret_cast<uint4*>(dst + v * 16) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          }
          if (wg == 0)
            store_scale(p.a2_s, (size_t)w.nb * p.R_cap + w.m0 + row, s, p.act_fmt == MOE_SCALE_UE8M0);
        }
      } else {
        // BF16 tile out through TMA stores: this warp's rows come in four 8-row groups
        // (rows 32*g + 8*q .. +7).  The warp writes its 32 x 128 block into its own 8 KB staging
        // buffer as 128-byte-swizzled 8 x 64 boxes and lane 0 issues the box stores without waiting
        // for them; the buffer is reused one item later, after the stores have read it.  Groups
        // that are only partly live (the end of an expert's rows) are written row by row instead.
        const int col0 = w.nb * kBN + wg * kGroup;
        if (qlive && col0 < p.out_cols) {
          uint8_t* buf = ystage + ew * TC::YWarpBytes;
          const uint32_t buf_s = smem_addr(buf);
          const int t = lane & 7;
          const int g_mine = lane >> 3;
          const int grow_mine = 32 * g_mine + 8 * q;
          if (lane == 0) bulk_wait_group_read0();     // the previous item's stores have read it
          __syncwarp();
          if (grow_mine + 8 <= w.live) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              uint32_t wd[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                wd[j] = f32_to_bf16_bits(acc[c * 8 + 2 * j]) |
                        (f32_to_bf16_bits(acc[c * 8 + 2 * j + 1]) << 16);
              const int box = c >> 3, cc = c & 7;
              *reinterpret_cast<uint4*>(buf + g_mine * 2048 + box * 1024 + t * 128 + ((cc ^ t) << 4)) =
                  make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
          } else if (rlive) {
            uint16_t* dst = p.y + (size_t)(w.m0 + row) * p.out_cols + col0;
#pragma unroll
            for (int v = 0; v < 16; ++v) {
              uint32_t wd[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                wd[j] = f32_to_bf16_bits(acc[v * 8 + 2 * j]) |
                        (f32_to_bf16_bits(acc[v * 8 + 2 * j + 1]) << 16);
              *reinterpret_cast<uint4*>(dst + v * 8) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const int grow = 32 * g + 8 * q;
              if (grow + 8 <= w.live) {
                tma_store_2d(&tmY, col0, w.m0 + grow, buf_s + g * 2048);
                tma_store_2d(&tmY, col0 + 64, w.m0 + grow, buf_s + g * 2048 + 1024);
              }
            }
            bulk_commit_group();
          }
        }
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
                               const CUtensorMap& tmS, const CUtensorMap& tmY, const GemmParams& p,
                               int grid, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(k_grouped_gemm<kFC1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TileCfg<kFC1>::Smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_grouped_gemm<kFC1>, dim3(grid), dim3(kTileThreads), TileCfg<kFC1>::Smem, s, tmA,
                    tmB, tmAS, tmS, tmY, p);
}

cudaError_t launch_fc1(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                       const CUtensorMap& tmS, const GemmParams& p, int grid, cudaStream_t s) {
  return launch_gemm<true>(tmA, tmB, tmAS, tmS, tmA, p, grid, s);   // FC1 stores no BF16 tile
}

cudaError_t launch_fc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmAS,
                       const CUtensorMap& tmS, const CUtensorMap& tmY, const GemmParams& p, int grid,
                       cudaStream_t s) {
  return launch_gemm<false>(tmA, tmB, tmAS, tmS, tmY, p, grid, s);
}

}  // namespace moe
