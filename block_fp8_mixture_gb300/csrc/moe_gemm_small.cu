// Small-batch grouped FP8 x FP8 GEMM: weight rows on the MMA's M side, up to 32 tokens on N.
//
// (TensorRT-LLM "Triton FP8-activation MoE for decode-sized batches on Hopper", description: at
// decode sizes the grid should cover only the expert blocks the batch occupies and stream the FP8
// weights at the bandwidth bound; vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose:
// only live (expert, rows) work is visited.)
//
// At decode sizes an expert holds a handful of rows, so a 128-row tile wastes the tensor-memory
// lanes and makes the per-128-K promotion read 128 x 256 partial sums for a few live rows.  Here the
// work item is a live 32-row chunk of one expert (from the alignment kernel's chunk list) x one
// output block x one K split:
//   warp 0 (one lane)  TMA producer.  Each stage of a 3-stage ring holds two 128-wide K blocks:
//                      one copy brings 2 x 128 weight rows (FC1: gate block and the matching up
//                      block; FC2: two 128-column blocks of H) as 256-byte runs per row, one copy
//                      the chunk's 32 token rows.  A separate ring of per-K-block slots receives
//                      the chunk's 32 activation scales and the two weight block scales.
//   warp 1 (one lane)  MMA issuer: per K block 2 x 4 tcgen05.mma kind::f8f6f4 with M = 128 weight
//                      rows, N = 32 tokens, K = 32, into one of four 64-column accumulators.
//   warps 2..9         promotion + epilogue.  Warp (q, half) owns weight rows 32q..32q+31 (its TMEM
//                      lane quarter) and tokens 16*half..16*half+15: per K block two 16-column
//                      tensor-memory loads and acc += partial * (a_scale[token] * w_scale).
// The epilogue is spread over all 256 threads: FC1 thread j applies SwiGLU to its (gate j, up j)
// for each live token, the 1x128 amax of a token is a shuffle + shared-memory reduction over the
// 128 lanes, and each warp writes 32 consecutive FP8 codes per token.  FC2 threads write BF16 y.
// K splits (FC1): each split publishes fp32 partials per pair; the last split to arrive sums them
// in split order and runs the epilogue.
#include "moe_device.cuh"

namespace moe {

constexpr int kSN = 32;                       // tokens per chunk (MMA N)
constexpr int kSPK = kSmallPK;                // K blocks per operand stage
constexpr int kSStages = 3;
constexpr int kSWHalf = kGroup * kBK * kSPK;  // 128 weight rows x kSPK K blocks
constexpr int kSWBytes = 2 * kSWHalf;         // [half][K block][128 rows][128 bytes]
constexpr int kSXBytes = kSN * kBK * kSPK;    // [8-row group][K block][8 rows][128 bytes]
constexpr int kSStageBytes = kSWBytes + kSXBytes;
constexpr int kSSlotBytes = 384;              // [0,128) act scales, [128,144) w0, [256,272) w1
constexpr int kSSlotW0 = 128;
constexpr int kSSlotW1 = 256;
constexpr int kSTmemBufs = 4;
constexpr int kSBufCols = 2 * kSN;            // gate/up (or block 0/1) x 32 tokens
constexpr int kSTmemCols = kSTmemBufs * kSBufCols;
constexpr int kSThreads = 320;
// scale slots (one per K block) have their own ring: an operand stage is released when its MMAs
// complete, the scales when all promotion warps have read them (they trail the MMA by up to
// kSTmemBufs K blocks)
constexpr int kSSlots = kSStages * kSPK + kSTmemBufs;
constexpr int kSSmemBytes = kSStages * kSStageBytes + kSSlots * kSSlotBytes + 1024 /*align*/ +
                            1024 /*bars*/ + 2 * 4 * kSN * 4 /*token amax exchange*/;
static_assert(kSSmemBytes <= 232448, "shared memory");
constexpr uint32_t kSIdesc = make_idesc_e4m3(kGroup, kSN);

struct Chunk {
  int chunk, nb, ks, e, row0, live;
};

__device__ __forceinline__ Chunk decode_chunk(const GemmParams& p, int item) {
  Chunk c;
  const int per = p.n_blocks * p.ksplit;
  c.chunk = item / per;
  const int rem = item - c.chunk * per;
  c.nb = rem / p.ksplit;
  c.ks = rem - c.nb * p.ksplit;
  c.row0 = p.chunk_row0[c.chunk];
  c.e = p.tile_expert[c.row0 / kAlign];
  c.live = min(kSN, p.live_end[c.e] - c.row0);
  return c;
}

__device__ __forceinline__ void s_drain_wait(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

// One trip of a rolled per-token loop over a register array: a[0..n-1] <- a[1..n-1], a[0] for
// n = 4 or 16 (n trips restore the order; entries past n are untouched).
__device__ __forceinline__ void rotate_tokens(float* a, int n) {
  if (n == 4) {
    const float t = a[0];
    a[0] = a[1];
    a[1] = a[2];
    a[2] = a[3];
    a[3] = t;
  } else {
    const float t = a[0];
#pragma unroll
    for (int i = 0; i < 15; ++i) a[i] = a[i + 1];
    a[15] = t;
  }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <bool kFC1>
__global__ void __launch_bounds__(kSThreads, 1)
    k_small_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmS, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  uint8_t* slots = smem + kSStages * kSStageBytes;
  uint8_t* ctrl = slots + kSSlots * kSSlotBytes;
  const uint32_t slot0 = smem_addr(slots);
  const uint32_t bar0 = smem_addr(ctrl);
  // barriers: full/empty[kSStages], sfull/sempty[kSSlots], tfull/tempty[kSTmemBufs], drain
  constexpr int kBarT = 2 * kSStages + 2 * kSSlots;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kSStages + s); };
  auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * kSStages + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (2 * kSStages + kSSlots + i); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (kBarT + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (kBarT + kSTmemBufs + b); };
  const uint32_t drain_bar = bar0 + 8u * (kBarT + 2 * kSTmemBufs);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (kBarT + 2 * kSTmemBufs + 1));
  static_assert(8 * (kBarT + 2 * kSTmemBufs + 1) + 16 <= 1024, "barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* mma_consumed = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 3);
  float* red = reinterpret_cast<float*>(ctrl + 1024);   // [2 halves][4 quarters][16 tokens]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kEpiWarps = 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < kSSlots; ++i) {
      mbar_init(sfull_bar(i), 1);
      mbar_init(sempty_bar(i), kEpiWarps);
    }
    for (int b = 0; b < kSTmemBufs; ++b) {
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
    prefetch_tensormap(&tmS);
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kSTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // The routing metadata (chunk list, tile experts, live ends) is written by the alignment, which
  // completed before the kernel launched ahead of this one finished its own dependency wait (the
  // activation quantization before FC1, FC1 before FC2).  So the first work item is decoded while
  // that kernel still runs; only the activation codes and scales the copies read need the wait.
  const int total = *p.num_chunks * p.n_blocks * p.ksplit;
  Chunk first = {};
  if ((int)blockIdx.x < total) first = decode_chunk(p, blockIdx.x);
  grid_dep_wait();                 // the previous kernel's outputs are complete from here on
  grid_dep_launch_dependents();

  const int KB = p.K / kBK;
  const int kb_per_split = KB / p.ksplit;
  const int a_ue = p.a_scale_ue8m0, b_ue = p.b_scale_ue8m0;
  const int a_scale_bytes = a_ue ? kSN : kSN * 4;
  const int w_mask = b_ue ? 15 : 3;   // scale elements per 16 bytes, minus one
  const int ncb = p.b_rows_per_expert / kGroup;
  int* status = p.status;

  int prod_issued = 0, prod_scales = 0;
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int sc = 0, it = 0;
    bool ok = true;
    const uint64_t pol_w = policy_evict_first();
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Chunk w = item == (int)blockIdx.x ? first : decode_chunk(p, item);
      int brow0, sr0, sr1;
      bool second;
      if (kFC1) {
        brow0 = w.e * p.b_rows_per_expert + w.nb * kGroup;   // gate rows; up rows I further
        sr0 = w.e * ncb + w.nb;
        sr1 = w.e * ncb + p.out_cols / kGroup + w.nb;
        second = true;
      } else {
        brow0 = w.e * p.b_rows_per_expert + w.nb * 2 * kGroup;
        sr0 = w.e * ncb + 2 * w.nb;
        sr1 = sr0 + 1;
        second = 2 * w.nb + 1 < ncb;
      }
      const uint32_t sbytes = a_scale_bytes + (second ? 32 : 16);
      const int kb0 = w.ks * kb_per_split;
      for (int kbs = kb0; ok && kbs < kb0 + kb_per_split; kbs += kSPK) {
        const int nv = min(kSPK, kb0 + kb_per_split - kbs);
        const int s = sc % kSStages;
        if (!mbar_wait(empty_bar(s), ((sc / kSStages) & 1) ^ 1, abort_flag, status)) {
          ok = false;
          break;
        }
        // whole boxes always arrive (kSPK K blocks, 32 token rows, both weight halves; rows past
        // the end of the weights read as zero)
        mbar_arrive_expect_tx(full_bar(s), kSStageBytes);
        const uint32_t sW = sbase + s * kSStageBytes;
        tma_load_4d_hint(sW, &tmB, 0, brow0, kbs, 0, full_bar(s), pol_w);
        tma_load_4d(sW + kSWBytes, &tmA, 0, 0, kbs, w.row0 / 8, full_bar(s));
        ++sc;
        for (int k = 0; k < nv; ++k) {
          const int kb = kbs + k;
          const int sl = it % kSSlots;
          if (!mbar_wait(sempty_bar(sl), ((it / kSSlots) & 1) ^ 1, abort_flag, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(sfull_bar(sl), sbytes);
          const uint32_t sS = slot0 + sl * kSSlotBytes;
          bulk_copy_g2s(sS, static_cast<const uint8_t*>(p.a_scale) +
                                ((size_t)kb * p.R_cap + w.row0) * (a_ue ? 1 : 4),
                        a_scale_bytes, sfull_bar(sl));
          const int i0 = sr0 * KB + kb;
          tma_load_1d(sS + kSSlotW0, &tmS, i0 & ~w_mask, sfull_bar(sl));
          if (second) {
            const int i1 = sr1 * KB + kb;
            tma_load_1d(sS + kSSlotW1, &tmS, i1 & ~w_mask, sfull_bar(sl));
          }
          ++it;
        }
      }
    }
    prod_issued = sc;
    prod_scales = it;
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA
    int sc = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const int kb0 = (item == (int)blockIdx.x ? first : decode_chunk(p, item)).ks * kb_per_split;
      for (int kbs = kb0; ok && kbs < kb0 + kb_per_split; kbs += kSPK) {
        const int nv = min(kSPK, kb0 + kb_per_split - kbs);
        const int s = sc % kSStages;
        if (!mbar_wait(full_bar(s), (sc / kSStages) & 1, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t sW = sbase + s * kSStageBytes;
        for (int k = 0; k < nv; ++k) {
          const int b = it % kSTmemBufs;
          if (!mbar_wait(tempty_bar(b), ((it / kSTmemBufs) & 1) ^ 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // token operand: 8-row groups 2 KB apart, K block k at +1 KB
          const uint64_t xdesc = make_sdesc_sw128(sW + kSWBytes + k * (kABoxRows * kBK),
                                                  kABoxRows * kBK * kSPK);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d = tmem_base + b * kSBufCols + h * kSN;
            const uint64_t wdesc = make_sdesc_sw128(sW + h * kSWHalf + k * (kGroup * kBK));
#pragma unroll
            for (int kk = 0; kk < kBK / 32; ++kk)
              mma_f8(d, wdesc + 2 * kk, xdesc + 2 * kk, kSIdesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(tfull_bar(b));
          ++it;
        }
        if (!ok) break;
        mma_commit(empty_bar(s));
        ++sc;
        *mma_consumed = sc;
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------- promotion + epilogue
    const int ew = warp - kEpiWarp0;
    const int half = ew >> 2;            // tokens 16*half .. 16*half + 15
    const int q = warp & 3;              // weight rows 32q .. 32q + 31 (TMEM lane quarter)
    const int j = q * 32 + lane;         // weight row (output column) inside the 128 block
    const uint32_t hb = (uint32_t)(half * 16);
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < total; item += gridDim.x) {
      const Chunk w = item == (int)blockIdx.x ? first : decode_chunk(p, item);
      const int ntok = max(0, min(16, w.live - half * 16));   // live tokens of this half
      int sr0, sr1;
      bool has1;
      if (kFC1) {
        sr0 = w.e * ncb + w.nb;
        sr1 = w.e * ncb + p.out_cols / kGroup + w.nb;
        has1 = true;
      } else {
        sr0 = w.e * ncb + 2 * w.nb;
        sr1 = sr0 + 1;
        has1 = 2 * w.nb + 1 < ncb;
      }
      float acc0[16], acc1[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) acc0[c] = acc1[c] = 0.0f;
      const int kb0 = w.ks * kb_per_split;
      for (int kb = kb0; kb < kb0 + kb_per_split; ++kb) {
        const int sl = it % kSSlots;
        const int b = it % kSTmemBufs;
        if (!mbar_wait(tfull_bar(b), (it / kSTmemBufs) & 1, abort_flag, status) ||
            !mbar_wait(sfull_bar(sl), (it / kSSlots) & 1, abort_flag, status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (ntok > 0) {
          const uint8_t* slot = slots + sl * kSSlotBytes;
          const int i0 = sr0 * KB + kb, i1 = sr1 * KB + kb;
          const float sw0 = smem_scale_at(slot + kSSlotW0, (i0 & w_mask), b_ue);
          const float sw1 = has1 ? smem_scale_at(slot + kSSlotW1, (i1 & w_mask), b_ue) : 0.0f;
          uint32_t r0[16], r1[16];
          const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16) + b * kSBufCols + hb;
          tmem_ld16(t0, r0);
          tmem_ld16(t0 + kSN, r1);
          float sa[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) sa[c] = smem_scale_at(slot, half * 16 + c, a_ue);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            acc0[c] = fmaf(__uint_as_float(r0[c]), __fmul_rn(sa[c], sw0), acc0[c]);
            acc1[c] = fmaf(__uint_as_float(r1[c]), __fmul_rn(sa[c], sw1), acc1[c]);
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(sempty_bar(sl));
          mbar_arrive(tempty_bar(b));
        }
        ++it;
      }
      if (!ok) break;

      if (kFC1) {
        // The epilogue runs once per item, so its code is usually cold in the instruction cache
        // (and, after other work has passed through L2, in L2 too).  Each per-token loop stays
        // rolled and works on entry 0 of register arrays that rotate by one token per trip:
        // short code, values in registers.  `trips` (4 when this half holds at most four tokens,
        // else 16) trips of rotate_tokens restore the order.
        const int I = p.out_cols;
        const int trips = ntok <= 4 ? 4 : 16;
        if (p.ksplit > 1) {
          // split-K fix-up over pairs: partial[ks][pair][2I], the last split sums in split order
#pragma unroll 1
          for (int c = 0; c < trips; ++c) {
            if (c < ntok) {
              const int pair = p.sorted_pair[w.row0 + half * 16 + c];
              float* dst = p.splitk_partial + ((size_t)w.ks * p.P_cap + pair) * (2 * I);
              dst[w.nb * kGroup + j] = acc0[0];
              dst[I + w.nb * kGroup + j] = acc1[0];
            }
            rotate_tokens(acc0, trips);
            rotate_tokens(acc1, trips);
          }
          __threadfence();
          named_barrier_sync(1, 256);
          if (ew == 0 && lane == 0) {
            const int prev = atomicAdd(&p.splitk_count[w.chunk * p.n_blocks + w.nb], 1);
            *last_flag = (prev == p.ksplit - 1);
          }
          named_barrier_sync(1, 256);
          const bool last = *last_flag != 0;
          named_barrier_sync(1, 256);
          if (!last) continue;
          __threadfence();
          if (ew == 0 && lane == 0) p.splitk_count[w.chunk * p.n_blocks + w.nb] = 0;
#pragma unroll 1
          for (int c = 0; c < trips; ++c) {
            if (c < ntok) {
              const int pair = p.sorted_pair[w.row0 + half * 16 + c];
              // every split's load first (one round trip), then the sum in split order
              float ga[kMaxKSplit], ua[kMaxKSplit];
#pragma unroll
              for (int s = 0; s < kMaxKSplit; ++s) {
                if (s < p.ksplit) {
                  const float* src = p.splitk_partial + ((size_t)s * p.P_cap + pair) * (2 * I);
                  ga[s] = __ldcg(src + w.nb * kGroup + j);
                  ua[s] = __ldcg(src + I + w.nb * kGroup + j);
                }
              }
              float g = 0.0f, u = 0.0f;
#pragma unroll
              for (int s = 0; s < kMaxKSplit; ++s) {
                if (s < p.ksplit) {
                  g = __fadd_rn(g, ga[s]);
                  u = __fadd_rn(u, ua[s]);
                }
              }
              acc0[0] = g;
              acc1[0] = u;
            }
            rotate_tokens(acc0, trips);
            rotate_tokens(acc1, trips);
          }
        }
        // SwiGLU per (j, token), then the token's 1x128 amax over the 128 lanes j
        float* r = red + half * (4 * 16);
#pragma unroll 1
        for (int c = 0; c < trips; ++c) {
          if (c < ntok) {
            float h = swiglu(bf16_round(acc0[0]), bf16_round(acc1[0]), p.clamp_mode,
                               p.clamp_limit);
            if (p.numerics == MOE_NUMERICS_RECIPROCAL) h = bf16_round(h);
            acc0[0] = h;
            float m = fabsf(h);
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
            if (lane == 0) r[q * 16 + c] = m;
          }
          rotate_tokens(acc0, trips);
          rotate_tokens(acc1, trips);
        }
        named_barrier_sync(2 + half, 128);
#pragma unroll 1
        for (int c = 0; c < trips; ++c) {
          if (c < ntok) {
            const float amax = fmaxf(fmaxf(r[c], r[16 + c]), fmaxf(r[32 + c], r[48 + c]));
            float inv;
            const float s = group_scale_numerics(amax, p.act_fmt, p.numerics, &inv);
            const int row = w.row0 + half * 16 + c;
            p.a2_q[(size_t)row * I + w.nb * kGroup + j] =
                (uint8_t)(cvt_e4m3x2(quant_div(acc0[0], s, inv), 0.0f) & 0xFF);
            if (j == 0)
              store_scale(p.a2_s, (size_t)w.nb * p.R_cap + row, s, p.act_fmt == MOE_SCALE_UE8M0);
          }
          rotate_tokens(acc0, trips);
        }
        named_barrier_sync(2 + half, 128);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c < ntok) {
            uint16_t* yrow = p.y + (size_t)(w.row0 + half * 16 + c) * p.out_cols + w.nb * 2 * kGroup;
            yrow[j] = (uint16_t)f32_to_bf16_bits(acc0[c]);
            if (has1) yrow[kGroup + j] = (uint16_t)f32_to_bf16_bits(acc1[c]);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == 1 && lane == 0) {
    mma_commit(drain_bar);
    s_drain_wait(drain_bar, 0, status);
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    for (int st = *mma_consumed; st < prod_issued; ++st)
      s_drain_wait(full_bar(st % kSStages), (st / kSStages) & 1, status);
    // scale copies: the latest use of each slot (earlier uses completed before it was reissued)
    for (int it = max(0, prod_scales - kSSlots); it < prod_scales; ++it)
      s_drain_wait(sfull_bar(it % kSSlots), (it / kSSlots) & 1, status);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kSTmemCols);
  }
}

template <bool kFC1>
static cudaError_t launch_small(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmS,
                                const GemmParams& p, int grid, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(k_small_gemm<kFC1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSSmemBytes);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_small_gemm<kFC1>, dim3(grid), dim3(kSThreads), kSSmemBytes, s, tmA, tmB, tmS,
                    p);
}

cudaError_t launch_fc1_small(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmS,
                             const GemmParams& p, int grid, cudaStream_t s) {
  return launch_small<true>(tmA, tmB, tmS, p, grid, s);
}

cudaError_t launch_fc2_small(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmS,
                             const GemmParams& p, int grid, cudaStream_t s) {
  return launch_small<false>(tmA, tmB, tmS, p, grid, s);
}

}  // namespace moe
