// Per-1x128 activation quantization scattered into the aligned workspace, and the top-k weighted
// unpermute/sum.  Both are HBM-bound streaming kernels: 16-byte vector loads and stores, one
// half-warp per 128-element group, and grids that only do work for live tokens.
#include "moe_device.cuh"

namespace moe {

// ------------------------------------------------------------ quantization
// (vLLM "per-layer activation scale format + fused SiLU+quant", Details: scale =
// max(amax/448, 1/(448*512)) then x/scale; TensorRT-LLM "Triton FP8-activation MoE for
// decode-sized batches on Hopper", rounding-fix commit: correctly rounded division.)
// One half-warp quantizes one 1x128 group: each lane holds 8 BF16 values (one 16-byte load),
// the group amax is reduced with shuffles inside the half-warp, and the 8 codes (8 bytes) plus the
// scale are written to every live workspace row of the token.
constexpr int kQuantThreads = 256;
constexpr int kGroupsPerBlock = kQuantThreads / 16;

__global__ void __launch_bounds__(kQuantThreads) k_quant_act(QuantParams p) {
  const int groups_per_row = p.H / kGroup;
  const int half = (threadIdx.x >> 4) & 1;
  const int l16 = threadIdx.x & 15;
  const uint32_t hmask = 0xFFFFu << (16 * half);
  const long gid = (long)blockIdx.x * kGroupsPerBlock + (threadIdx.x >> 4);
  const long t = gid / groups_per_row;
  const int g = (int)(gid % groups_per_row);
  grid_dep_wait();
  grid_dep_launch_dependents();
  int n = p.M_cap;
  if (p.d_num_tokens != nullptr) n = min(max(*p.d_num_tokens, 0), p.M_cap);
  if (t >= n) return;   // the whole half-warp leaves together

  const uint4 raw = *reinterpret_cast<const uint4*>(p.x + t * p.H + g * kGroup + l16 * 8);
  float v[8];
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, d));
  float inv;
  const float s = group_scale_numerics(amax, p.fmt, p.numerics, &inv);
  uint32_t q0 = cvt_e4m3x2(quant_div(v[0], s, inv), quant_div(v[1], s, inv)) |
                (cvt_e4m3x2(quant_div(v[2], s, inv), quant_div(v[3], s, inv)) << 16);
  uint32_t q1 = cvt_e4m3x2(quant_div(v[4], s, inv), quant_div(v[5], s, inv)) |
                (cvt_e4m3x2(quant_div(v[6], s, inv), quant_div(v[7], s, inv)) << 16);
  const int is_ue8m0 = p.fmt == MOE_SCALE_UE8M0;
  for (int j = 0; j < p.topk; ++j) {
    const int row = p.pair_row[t * p.topk + j];
    if (row < 0) continue;
    *reinterpret_cast<uint2*>(p.a_q + (size_t)row * p.H + g * kGroup + l16 * 8) = make_uint2(q0, q1);
    if (l16 == 0) store_scale(p.a_s, (size_t)g * p.R_cap + row, s, is_ue8m0);
  }
}

cudaError_t launch_quant(const QuantParams& p, cudaStream_t s) {
  const long groups = (long)p.M_cap * (p.H / kGroup);
  const long blocks = (groups + kGroupsPerBlock - 1) / kGroupsPerBlock;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(k_quant_act, dim3((unsigned)blocks), dim3(kQuantThreads), 0, s, p);
}

// ----------------------------------------------------------------- reduce
// (TensorRT-LLM page, rounding-fix commit: the routing weights scale the BF16 expert outputs in
// fp32 in the top-k sum, not the FC2 accumulators.)
// out[t, c] = bf16( sum_j RN(RN(w[t,j] * y[row_j, c]) ) ) over pairs j with a row, j ascending
// (the fp32 sum itself when out_fp32: an expert-parallel rank's partial output).
// Each thread produces 8 consecutive columns (16-byte loads of y and a 16-byte store).  The token's
// pair rows and routing weights are read first, then the y loads go out four at a time, so a
// token costs two or three dependent memory round trips instead of one per pair; the sum itself
// still runs over j in ascending order.
constexpr int kReduceThreads = 128;
constexpr int kReduceBatch = 4;

__device__ __forceinline__ void reduce_add8(float* acc, const uint4& raw, float w) {
  const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, bf16_bits_to_f32(u[i] & 0xFFFFu)));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, bf16_bits_to_f32(u[i] >> 16)));
  }
}

__global__ void __launch_bounds__(kReduceThreads) k_topk_reduce(ReduceParams p) {
  const long t = blockIdx.x;
  grid_dep_wait();
  grid_dep_launch_dependents();
  int n = p.M_cap;
  if (p.d_num_tokens != nullptr) n = min(max(*p.d_num_tokens, 0), p.M_cap);
  if (t >= n) return;
  const int c0 = (blockIdx.y * kReduceThreads + threadIdx.x) * 8;
  if (c0 >= p.H) return;
  const int topk = p.topk;
  int rows[kMaxTopk];
  float wts[kMaxTopk];
#pragma unroll
  for (int j = 0; j < kMaxTopk; ++j) {
    rows[j] = j < topk ? p.pair_row[t * topk + j] : -1;
    wts[j] = j < topk ? p.topk_weights[t * topk + j] : 0.0f;
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int j0 = 0; j0 < kMaxTopk; j0 += kReduceBatch) {
    if (j0 >= topk) break;
    uint4 raw[kReduceBatch];
#pragma unroll
    for (int u = 0; u < kReduceBatch; ++u)
      if (rows[j0 + u] >= 0)
        raw[u] = __ldg(reinterpret_cast<const uint4*>(p.y + (size_t)rows[j0 + u] * p.H + c0));
#pragma unroll
    for (int u = 0; u < kReduceBatch; ++u)
      if (rows[j0 + u] >= 0) reduce_add8(acc, raw[u], wts[j0 + u]);
  }
  if (p.out_fp32) {
    float* o = static_cast<float*>(p.out) + t * p.H + c0;
    *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(o + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    return;
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = f32_to_bf16_bits(acc[2 * i]) | (f32_to_bf16_bits(acc[2 * i + 1]) << 16);
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + t * p.H + c0) =
      make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t s) {
  if (p.M_cap == 0) return cudaSuccess;
  dim3 grid(p.M_cap, (p.H / 8 + kReduceThreads - 1) / kReduceThreads);
  return launch_pdl(k_topk_reduce, grid, dim3(kReduceThreads), 0, s, p);
}

}  // namespace moe

namespace moe {

// Batched-expert layout: quantize rows r < counts[e] of x [E, max_m, H] in place of the scatter
// (workspace row = e * max_m + r; same arithmetic as k_quant_act).
__global__ void __launch_bounds__(kQuantThreads) k_quant_rows(QuantRowsParams p) {
  const int groups_per_row = p.H / kGroup;
  const int half = (threadIdx.x >> 4) & 1;
  const int l16 = threadIdx.x & 15;
  const uint32_t hmask = 0xFFFFu << (16 * half);
  const long gid = (long)blockIdx.x * kGroupsPerBlock + (threadIdx.x >> 4);
  const long row = gid / groups_per_row;
  const int g = (int)(gid % groups_per_row);
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (row >= (long)p.E * p.max_m) return;
  const int e = (int)(row / p.max_m);
  const int r = (int)(row - (long)e * p.max_m);
  if (r >= min(max(p.counts[e], 0), p.max_m)) return;   // the whole half-warp leaves together

  const uint4 raw = *reinterpret_cast<const uint4*>(p.x + row * p.H + g * kGroup + l16 * 8);
  float v[8];
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, d));
  float inv;
  const float s = group_scale_numerics(amax, p.fmt, p.numerics, &inv);
  const uint32_t q0 = cvt_e4m3x2(quant_div(v[0], s, inv), quant_div(v[1], s, inv)) |
                      (cvt_e4m3x2(quant_div(v[2], s, inv), quant_div(v[3], s, inv)) << 16);
  const uint32_t q1 = cvt_e4m3x2(quant_div(v[4], s, inv), quant_div(v[5], s, inv)) |
                      (cvt_e4m3x2(quant_div(v[6], s, inv), quant_div(v[7], s, inv)) << 16);
  *reinterpret_cast<uint2*>(p.a_q + (size_t)row * p.H + g * kGroup + l16 * 8) = make_uint2(q0, q1);
  if (l16 == 0) store_scale(p.a_s, (size_t)g * p.R_cap + row, s, p.fmt == MOE_SCALE_UE8M0);
}

cudaError_t launch_quant_rows(const QuantRowsParams& p, cudaStream_t s) {
  const long groups = (long)p.E * p.max_m * (p.H / kGroup);
  const long blocks = (groups + kGroupsPerBlock - 1) / kGroupsPerBlock;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(k_quant_rows, dim3((unsigned)blocks), dim3(kQuantThreads), 0, s, p);
}

}  // namespace moe

namespace moe {

// SwiGLU + 1x128 requantization as its own kernel (vLLM "per-layer activation scale format + fused
// SiLU+quant", Details: the fused silu_and_mul_per_block_quant kernel reads the FP32/BF16 gate and
// up halves and writes FP8 codes with 1x128 scales).  The tile schedule with fp32 activation scales
// uses it on the BF16 FC1 outputs; the arithmetic is that of the fused FC1 epilogue.  One half-warp
// per (row, 128-column group): 16-byte loads of 8 gate and 8 up values per lane, shuffle amax.
__global__ void __launch_bounds__(kQuantThreads) k_swiglu_quant(SwigluQuantParams p) {
  const int groups = p.I / kGroup;
  const int half = (threadIdx.x >> 4) & 1;
  const int l16 = threadIdx.x & 15;
  const uint32_t hmask = 0xFFFFu << (16 * half);
  const long gid = (long)blockIdx.x * kGroupsPerBlock + (threadIdx.x >> 4);
  const long row = gid / groups;
  const int g = (int)(gid % groups);
  grid_dep_wait();
  grid_dep_launch_dependents();
  if (row >= p.R_cap) return;                 // the whole half-warp leaves together
  const int t = (int)(row / kBM);
  if (!p.all_tiles && t >= *p.num_tiles) return;
  if (row >= p.live_end[p.tile_expert[t]]) return;

  const uint16_t* src = p.g1 + row * (2 * p.I) + g * kGroup + l16 * 8;
  const uint4 gr = *reinterpret_cast<const uint4*>(src);
  const uint4 ur = *reinterpret_cast<const uint4*>(src + p.I);
  const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
  const uint32_t uw[4] = {ur.x, ur.y, ur.z, ur.w};
  float h[8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t gb = (i & 1) ? gw[i >> 1] >> 16 : gw[i >> 1] & 0xFFFFu;
    const uint32_t ub = (i & 1) ? uw[i >> 1] >> 16 : uw[i >> 1] & 0xFFFFu;
    float v = swiglu(bf16_bits_to_f32(gb), bf16_bits_to_f32(ub), p.clamp_mode, p.clamp_limit);
    if (p.numerics == MOE_NUMERICS_RECIPROCAL) v = bf16_round(v);
    h[i] = v;
    amax = fmaxf(amax, fabsf(v));
  }
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, d));
  float inv;
  const float s = group_scale_numerics(amax, p.fmt, p.numerics, &inv);
  const uint32_t q0 = cvt_e4m3x2(quant_div(h[0], s, inv), quant_div(h[1], s, inv)) |
                      (cvt_e4m3x2(quant_div(h[2], s, inv), quant_div(h[3], s, inv)) << 16);
  const uint32_t q1 = cvt_e4m3x2(quant_div(h[4], s, inv), quant_div(h[5], s, inv)) |
                      (cvt_e4m3x2(quant_div(h[6], s, inv), quant_div(h[7], s, inv)) << 16);
  *reinterpret_cast<uint2*>(p.a2_q + (size_t)row * p.I + g * kGroup + l16 * 8) = make_uint2(q0, q1);
  if (l16 == 0) store_scale(p.a2_s, (size_t)g * p.R_cap + row, s, p.fmt == MOE_SCALE_UE8M0);
}

cudaError_t launch_swiglu_quant(const SwigluQuantParams& p, cudaStream_t s) {
  const long groups = (long)p.R_cap * (p.I / kGroup);
  const long blocks = (groups + kGroupsPerBlock - 1) / kGroupsPerBlock;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(k_swiglu_quant, dim3((unsigned)blocks), dim3(kQuantThreads), 0, s, p);
}

}  // namespace moe
