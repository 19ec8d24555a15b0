// Routing alignment into per-expert prefix-sum endpoints, one CTA.
//
// (vLLM "Skip padded work in block-FP8 DeepGemmExperts", Purpose: the permutation helper produces
// the expert endpoints both grouped GEMMs and the fused activation quantization consume;
// TensorRT-LLM "Triton FP8-activation MoE for decode-sized batches on Hopper", description: one
// program aligns the routed pairs.)
//
// A stable counting sort of the valid pairs p = t*k + j (t < n) by expert.  The 32 warps of the CTA
// each own a contiguous range of pairs:
//   pass 1  each warp counts its range per expert (warp-private histogram row, no atomics:
//           __match_any_sync groups equal ids, the group leader adds the group size);
//   scan    per expert, exclusive prefix over the warps' counts (gives each warp its base inside
//           the expert) and a CTA-wide exclusive scan of the 128-padded counts (segment starts);
//   pass 2  each warp walks its range again in order and places every pair at
//           seg_start[e] + warp base + rank among the earlier equal ids of its 32-pair chunk.
// Ascending pair order inside a segment follows because warps own ascending ranges and chunks are
// visited in order.
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

__global__ void __launch_bounds__(kAlignThreads, 1) k_align(AlignParams p) {
  extern __shared__ int32_t sm[];
  const int E = p.E;
  int32_t* hist = sm;                              // [32][E]
  int32_t* seg = sm + kAlignWarps * E;             // [E + 1]
  __shared__ int32_t warp_sums[kAlignWarps];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lanes_below = (1u << lane) - 1u;

  grid_dep_wait();
  grid_dep_launch_dependents();
  int n = p.M_cap;
  if (p.d_num_tokens != nullptr) n = min(max(*p.d_num_tokens, 0), p.M_cap);
  const int num_pairs = n * p.topk;

  if (tid == 0) *p.status = 0;
  for (int i = tid; i < p.splitk_count_len; i += kAlignThreads) p.splitk_count[i] = 0;
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) hist[i] = 0;
  __syncthreads();

  const int chunk = (num_pairs + kAlignWarps - 1) / kAlignWarps;
  const int begin = min(warp * chunk, num_pairs);
  const int end = min(begin + chunk, num_pairs);

  // pass 1: per-warp histogram
  for (int base = begin; base < end; base += 32) {
    const int pi = base + lane;
    int e = -1;
    if (pi < end) {
      const int id = p.topk_ids[pi];
      if (id >= 0 && id < E) e = id;
    }
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const bool leader = (same & lanes_below) == 0;
    if (leader && e >= 0) hist[warp * E + e] += __popc(same);
    __syncwarp();
  }
  __syncthreads();

  // per-expert prefix over warps; padded count of expert e kept for the scan
  int padded = 0;
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    seg[e] = run;                                  // count, replaced by the start below
    padded = (run + kAlign - 1) / kAlign * kAlign;
  }
  // exclusive scan of padded counts (E <= 1024 = one expert per thread)
  int total = 0;
  const int excl = block_exclusive_scan(padded, warp_sums, &total);
  const int count = tid < E ? seg[tid] : 0;
  // live 32-row chunks of each expert (the small-batch schedule's work list)
  int chunk_total = 0;
  const int chunk_base = block_exclusive_scan((count + kChunkRows - 1) / kChunkRows, warp_sums,
                                              &chunk_total);
  if (tid < E) {
    seg[tid] = excl;
    p.seg_start[tid] = excl;
    p.live_end[tid] = excl + count;
    for (int c = 0; c * kChunkRows < count; ++c) p.chunk_row0[chunk_base + c] = excl + c * kChunkRows;
  }
  if (tid == 0) {
    seg[E] = total;
    p.seg_start[E] = total;
    *p.num_tiles = total / kAlign;
    *p.num_chunks = chunk_total;
  }
  __syncthreads();

  // tile -> expert map
  for (int e = tid; e < E; e += kAlignThreads) {
    for (int t = seg[e] / kAlign; t < seg[e + 1] / kAlign; ++t) p.tile_expert[t] = e;
  }

  // pass 2: stable placement
  for (int base = begin; base < end; base += 32) {
    const int pi = base + lane;
    int e = -1;
    if (pi < end) {
      const int id = p.topk_ids[pi];
      if (id >= 0 && id < E) e = id;
    }
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(same & lanes_below);
    if (pi < end) {
      if (e >= 0) {
        const int row = seg[e] + hist[warp * E + e] + rank;
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
  const size_t smem = (size_t)(kAlignWarps * p.E + p.E + 1) * sizeof(int32_t);
  cudaError_t err = cudaFuncSetAttribute(k_align, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_align, dim3(1), dim3(kAlignThreads), smem, s, p);
}

}  // namespace moe
