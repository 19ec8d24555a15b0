// Routing alignment into per-expert prefix-sum endpoints.
//
// (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose: the permutation helper produces
// the expert endpoints both grouped GEMMs and the fused activation quantization consume;
// TensorRT-LLM "Triton FP8-activation MoE for decode-sized batches on Hopper", description: one
// program aligns the routed pairs.)
//
// A stable counting sort of the valid pairs p = t*k + j (t < n) by expert (ids rebased by the
// expert-parallel offset; ids outside [0, E) are dropped).  The pairs are cut into
// G contiguous ranges, one per CTA (G = 1 for small batches).  Inside a CTA the 32 warps each own a
// contiguous sub-range:
//   pass 1  each warp counts its sub-range per expert (warp-private histogram row, no atomics:
//           __match_any_sync groups equal ids, the group leader adds the group size);
//   counts  per expert, exclusive prefix over the warps (each warp's base inside the CTA's share)
//           and, for G > 1, over the CTAs' counts written by k_align_count (the CTA's base inside
//           the expert);
//   scan    CTA-wide exclusive scans of the 128-padded counts (segment starts) and of the 32-row
//           chunk counts (small-batch work list); every CTA computes them, CTA 0 writes them;
//   pass 2  each warp walks its sub-range again in order and places every pair at
//           seg_start[e] + CTA base + warp base + rank among the earlier equal ids of its 32 pairs.
// Ascending pair order inside a segment follows because CTAs and warps own ascending ranges and
// chunks of 32 pairs are visited in order.
#include "moe_device.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kChunkRows = 32;

// Exclusive scan of one int per thread over the 1024-thread CTA; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += t;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, w, d);
      if (lane >= d) w += t;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[kAlignWarps - 1];
  __syncthreads();
  return excl;
}

__device__ __forceinline__ int live_pairs(const AlignParams& p) {
  int n = p.M_cap;
  if (p.d_num_tokens != nullptr) n = min(max(*p.d_num_tokens, 0), p.M_cap);
  return n * p.topk;
}

__device__ __forceinline__ void reset_shared_state(const AlignParams& p) {
  if (threadIdx.x == 0) *p.status = 0;
  for (int i = threadIdx.x; i < p.splitk_count_len; i += kAlignThreads) p.splitk_count[i] = 0;
}

// Large batches, step 1: expert counts of each CTA's range of pairs.
__global__ void __launch_bounds__(kAlignThreads, 1) k_align_count(AlignParams p) {
  extern __shared__ int32_t hist[];   // [E]
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int E = p.E;
  const int num_pairs = live_pairs(p);
  if (blockIdx.x == 0) reset_shared_state(p);
  for (int e = threadIdx.x; e < E; e += kAlignThreads) hist[e] = 0;
  __syncthreads();
  const int per = (num_pairs + gridDim.x - 1) / gridDim.x;
  const int begin = min((int)blockIdx.x * per, num_pairs);
  const int end = min(begin + per, num_pairs);
  for (int i = begin + threadIdx.x; i < end; i += kAlignThreads) {
    const int id = p.topk_ids[i] - p.expert_offset;
    if (id >= 0 && id < E) atomicAdd(&hist[id], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kAlignThreads) p.cta_hist[blockIdx.x * E + e] = hist[e];
}

// The placement (and, for one CTA, the whole alignment).
__global__ void __launch_bounds__(kAlignThreads, 1) k_align(AlignParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E;
  int32_t* hist = sm;                              // [32][E]
  int32_t* seg = sm + kAlignWarps * E;             // [E + 1]
  int32_t* base = seg + E + 1;                     // [E]: this CTA's first rank inside each expert
  __shared__ int32_t warp_sums[kAlignWarps];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lanes_below = (1u << lane) - 1u;

  grid_dep_wait();
  grid_dep_launch_dependents();
  const int num_pairs = live_pairs(p);
  const int G = p.num_ctas;
  if (G == 1) reset_shared_state(p);
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) hist[i] = 0;
  __syncthreads();

  const int per_cta = (num_pairs + G - 1) / G;
  const int cbegin = min((int)blockIdx.x * per_cta, num_pairs);
  const int cend = min(cbegin + per_cta, num_pairs);
  const int chunk = (cend - cbegin + kAlignWarps - 1) / kAlignWarps;
  const int begin = min(cbegin + warp * chunk, cend);
  const int end = min(begin + chunk, cend);

  // pass 1: per-warp histogram
  for (int b0 = begin; b0 < end; b0 += 32) {
    const int pi = b0 + lane;
    int e = -1;
    if (pi < end) {
      const int id = p.topk_ids[pi] - p.expert_offset;
      if (id >= 0 && id < E) e = id;
    }
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const bool leader = (same & lanes_below) == 0;
    if (leader && e >= 0) hist[warp * E + e] += __popc(same);
    __syncwarp();
  }
  __syncthreads();

  // per-expert prefix over warps; expert totals and this CTA's base
  int padded = 0, count = 0;
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    int before = 0, total = run;
    if (G > 1) {
      total = 0;
      for (int g = 0; g < G; ++g) {
        const int c = p.cta_hist[g * E + e];
        if (g < (int)blockIdx.x) before += c;
        total += c;
      }
    }
    base[e] = before;
    count = total;
    padded = (total + kAlign - 1) / kAlign * kAlign;
  }
  // exclusive scans over experts (E <= 1024 = one expert per thread)
  int seg_total = 0;
  const int excl = block_exclusive_scan(padded, warp_sums, &seg_total);
  int chunk_total = 0;
  const int chunk_base = block_exclusive_scan((count + kChunkRows - 1) / kChunkRows, warp_sums,
                                              &chunk_total);
  if (tid < E) seg[tid] = excl;
  if (tid == 0) seg[E] = seg_total;
  if (blockIdx.x == 0) {
    if (tid < E) {
      p.seg_start[tid] = excl;
      p.live_end[tid] = excl + count;
      for (int c = 0; c * kChunkRows < count; ++c)
        p.chunk_row0[chunk_base + c] = excl + c * kChunkRows;
    }
    if (tid == 0) {
      p.seg_start[E] = seg_total;
      *p.num_tiles = seg_total / kAlign;
      *p.num_chunks = chunk_total;
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    // tile -> expert map
    for (int e = tid; e < E; e += kAlignThreads)
      for (int t = seg[e] / kAlign; t < seg[e + 1] / kAlign; ++t) p.tile_expert[t] = e;
  }

  // pass 2: stable placement
  for (int b0 = begin; b0 < end; b0 += 32) {
    const int pi = b0 + lane;
    int e = -1;
    if (pi < end) {
      const int id = p.topk_ids[pi] - p.expert_offset;
      if (id >= 0 && id < E) e = id;
    }
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(same & lanes_below);
    if (pi < end) {
      if (e >= 0) {
        const int row = seg[e] + base[e] + hist[warp * E + e] + rank;
        p.pair_row[pi] = row;
        p.sorted_pair[row] = pi;
      } else {
        p.pair_row[pi] = -1;
      }
    }
    __syncwarp();
    if (rank == 0 && e >= 0) hist[warp * E + e] += __popc(same);
    __syncwarp();
  }
}

cudaError_t launch_align(const AlignParams& p, cudaStream_t s) {
  if (p.num_ctas > 1) {
    const size_t csmem = (size_t)p.E * sizeof(int32_t);
    const cudaError_t e0 =
        launch_pdl(k_align_count, dim3(p.num_ctas), dim3(kAlignThreads), csmem, s, p);
    if (e0 != cudaSuccess) return e0;
  }
  const size_t smem = (size_t)(kAlignWarps * p.E + 2 * p.E + 1) * sizeof(int32_t);
  cudaError_t err = cudaFuncSetAttribute(k_align, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_align, dim3(p.num_ctas), dim3(kAlignThreads), smem, s, p);
}

}  // namespace moe

namespace moe {

// Batched-expert layout (vLLM "per-layer activation scale format + fused SiLU+quant", Details:
// batched experts with masked per-expert counts): expert e's rows already sit at
// [e * max_m, e * max_m + counts[e]) (max_m a multiple of 128), so no sort is needed -- only the
// live ends and the compact lists of live 128-row tiles and 32-row chunks the GEMMs walk.
__global__ void __launch_bounds__(kAlignThreads, 1) k_batch_prep(BatchPrepParams p) {
  __shared__ int32_t warp_sums[kAlignWarps];
  grid_dep_wait();
  grid_dep_launch_dependents();
  const int tid = threadIdx.x;
  if (tid == 0) *p.status = 0;
  int count = 0;
  if (tid < p.E) count = min(max(p.counts[tid], 0), p.max_m);
  int tiles_total = 0, chunks_total = 0;
  const int tile_base = block_exclusive_scan((count + kAlign - 1) / kAlign, warp_sums, &tiles_total);
  const int chunk_base =
      block_exclusive_scan((count + kChunkRows - 1) / kChunkRows, warp_sums, &chunks_total);
  if (tid < p.E) {
    const int r0 = tid * p.max_m;
    p.seg_start[tid] = r0;
    p.live_end[tid] = r0 + count;
    for (int t = 0; t * kAlign < count; ++t) p.tile_row0[tile_base + t] = r0 + t * kAlign;
    for (int c = 0; c * kChunkRows < count; ++c) p.chunk_row0[chunk_base + c] = r0 + c * kChunkRows;
    for (int t = 0; t < p.max_m / kAlign; ++t) p.tile_expert[r0 / kAlign + t] = tid;
  }
  if (tid == 0) {
    p.seg_start[p.E] = p.E * p.max_m;
    *p.num_tiles = tiles_total;
    *p.num_chunks = chunks_total;
  }
}

cudaError_t launch_batch_prep(const BatchPrepParams& p, cudaStream_t s) {
  return launch_pdl(k_batch_prep, dim3(1), dim3(kAlignThreads), 0, s, p);
}

}  // namespace moe
