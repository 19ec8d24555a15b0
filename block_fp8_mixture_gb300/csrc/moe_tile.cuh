// Work items and epilogues shared by the two 128-row-tile grouped GEMMs (per-K-block promotion
// for FP32 block scales, block-scaled MMA for UE8M0 block scales).
//
// (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose: both grouped GEMMs visit only the
// live (expert, row-tile) work named by the prefix-sum endpoints.  vLLM "per-layer activation scale
// format + fused SiLU+quant", Details: the FC1 epilogue applies SwiGLU to the FP32 FC1 outputs and
// requantizes them 1x128 in the same pass.)
#pragma once

#include "moe_device.cuh"

namespace moe {

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

// Whether another row tile of the item's expert reads the same weight blocks.  Its weight copies
// then keep normal L2 priority, so the other tiles find them there; a lone tile streams them
// once, with evict-first, so that they do not push its activation rows out of L2.
__device__ __forceinline__ bool expert_weights_shared(const GemmParams& p, const Item& w,
                                                      int num_tiles) {
  auto expert_of = [&](int t) {
    const int m0 = p.tile_row0 != nullptr ? p.tile_row0[t] : t * kBM;
    return p.tile_expert[m0 / kBM];
  };
  return (w.tile > 0 && expert_of(w.tile - 1) == w.e) ||
         (w.tile + 1 < num_tiles && expert_of(w.tile + 1) == w.e);
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

// Epilogue threads: 8 warps, two per tensor-memory lane quarter q = warp % 4; warp half wg owns
// columns [64 wg, 64 wg + 64) of the gate and of the up block (FC1) or [128 wg, 128 wg + 128) of
// the 256 output columns (FC2).  A thread holds row `row` of the tile; named barrier 1 spans the
// 256 threads.
constexpr int kTileEpiThreadsBar = 256;

// FC1: acc[0..63] gate sums, acc[64..127] up sums of the thread's row (the tile kernels do not
// split K).  SwiGLU on the BF16-rounded sums and 1x128 requantization of the row's 128 outputs,
// written to the FC2 input codes and scales.
__device__ __forceinline__ void fc1_item_epilogue(const GemmParams& p, const Item& w, float* acc,
                                                  int row, int wg, bool rlive, float* red) {
  const int I = p.out_cols;
  // SwiGLU on the BF16-rounded FC1 outputs, then 1x128 requantization over the row's 128
  // (gate, up) columns held by this thread (64) and its partner in the other half (64).
  float amax = 0.0f;
  if (rlive) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      float h = swiglu(bf16_round(acc[i]), bf16_round(acc[64 + i]), p.clamp_mode, p.clamp_limit);
      if (p.numerics == MOE_NUMERICS_RECIPROCAL) h = bf16_round(h);
      acc[i] = h;
      amax = fmaxf(amax, fabsf(h));
    }
  }
  red[wg * kBM + row] = amax;
  named_barrier_sync(1, kTileEpiThreadsBar);
  amax = fmaxf(red[row], red[kBM + row]);
  named_barrier_sync(1, kTileEpiThreadsBar);
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
}

// FC1 of the tile schedule with fp32 activation scales: the row's 64 gate and 64 up sums, rounded
// to BF16, go to the FC1 output rows (gate | up); SwiGLU and the requantization run in their own
// kernel.  Only live rows are written.
__device__ __forceinline__ void fc1_item_store_g1(const GemmParams& p, const Item& w,
                                                  const float* acc, int row, int wg, bool rlive) {
  if (!rlive) return;
  const int I = p.out_cols;
  uint16_t* g = p.g1 + (size_t)(w.m0 + row) * (2 * I) + w.nb * kGroup + wg * 64;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint16_t* dst = g + half * I;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float* v = acc + half * 64 + c * 8;
      *reinterpret_cast<uint4*>(dst + c * 8) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
  }
}

// FC2: acc[0..127] = the thread's 128 output sums.  BF16 tile out through TMA stores: this warp's
// rows come in four 8-row groups (rows 32*g + 8*q .. +7).  The warp writes its 32 x 128 block into
// its own 8 KB staging buffer `buf` (1024-byte aligned) as 128-byte-swizzled 8 x 64 boxes laid out
// [64-column half][group][row], and lane 0 issues the stores without waiting for them; the buffer
// is reused one item later, after the stores have read it.  When all four groups are live, one
// 3-D store (tmY3: 64 columns x 8 rows x 4 groups 32 rows apart) writes each half; otherwise each
// fully live group is stored on its own (tmY: 64 x 8) and partly live groups are written row by
// row from registers.
__device__ __forceinline__ void fc2_item_epilogue(const GemmParams& p, const Item& w,
                                                  const float* acc, int row, int wg, int q,
                                                  int lane, bool qlive, bool rlive, uint8_t* buf,
                                                  const CUtensorMap* tmY, const CUtensorMap* tmY3) {
  const int col0 = w.nb * kBN + wg * kGroup;
  if (!qlive || col0 >= p.out_cols) return;
  const uint32_t buf_s = smem_addr(buf);
  const int t = lane & 7;
  const int g_mine = lane >> 3;
  const int grow_mine = 32 * g_mine + 8 * q;
  if (lane == 0) bulk_wait_group_read0();     // the previous item's stores have read it
  __syncwarp();
  if (grow_mine + 8 <= w.live) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float* v = acc + c * 8;
      const int half = c >> 3, cc = c & 7;
      *reinterpret_cast<uint4*>(buf + half * 4096 + g_mine * 1024 + t * 128 + ((cc ^ t) << 4)) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
  } else if (rlive) {
    uint16_t* dst = p.y + (size_t)(w.m0 + row) * p.out_cols + col0;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float* v = acc + c * 8;
      *reinterpret_cast<uint4*>(dst + c * 8) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (96 + 8 * q + 8 <= w.live) {
      tma_store_3d(tmY3, col0, 8 * q, w.m0 / 32, buf_s);
      tma_store_3d(tmY3, col0 + 64, 8 * q, w.m0 / 32, buf_s + 4096);
    } else {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int grow = 32 * g + 8 * q;
        if (grow + 8 <= w.live) {
          tma_store_2d(tmY, col0, w.m0 + grow, buf_s + g * 1024);
          tma_store_2d(tmY, col0 + 64, w.m0 + grow, buf_s + 4096 + g * 1024);
        }
      }
    }
    bulk_commit_group();
  }
}

// FC2 with a 2 KB staging buffer per warp: the same BF16 stores as fc2_item_epilogue, one 8-row group
// at a time.  For each fully live group of this warp (rows 32*g + 8*q .. +7, in increasing g), the
// group's eight lanes write their rows into `buf` as two 128-byte-swizzled 8 x 64 boxes and lane 0
// issues two 2-D stores; the buffer is reused for the next group once the stores have read it.
// Rows of a partly live group are written from registers.  The small buffer leaves shared memory for
// a fourth operand stage.
__device__ __forceinline__ void fc2_item_epilogue_by_group(const GemmParams& p, const Item& w,
                                                           const float* acc, int row, int wg, int q,
                                                           int lane, bool qlive, bool rlive,
                                                           uint8_t* buf, const CUtensorMap* tmY) {
  const int col0 = w.nb * kBN + wg * kGroup;
  if (!qlive || col0 >= p.out_cols) return;
  const uint32_t buf_s = smem_addr(buf);
  const int t = lane & 7;
  const int g_mine = lane >> 3;
  if (32 * g_mine + 8 * q + 8 > w.live && rlive) {
    uint16_t* dst = p.y + (size_t)(w.m0 + row) * p.out_cols + col0;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float* v = acc + c * 8;
      *reinterpret_cast<uint4*>(dst + c * 8) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
  }
#pragma unroll 1
  for (int g = 0; g < 4; ++g) {
    const int grow = 32 * g + 8 * q;
    if (grow + 8 > w.live) break;            // later groups of this warp are not fully live either
    if (lane == 0) bulk_wait_group_read0();  // the previous stores have read the buffer
    __syncwarp();
    if (g_mine == g) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float* v = acc + c * 8;
        const int half = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(buf + half * 1024 + t * 128 + ((cc ^ t) << 4)) =
            make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                       pack_bf16x2(v[6], v[7]));
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmY, col0, w.m0 + grow, buf_s);
      tma_store_2d(tmY, col0 + 64, w.m0 + grow, buf_s + 1024);
      bulk_commit_group();
    }
  }
}

}  // namespace moe
