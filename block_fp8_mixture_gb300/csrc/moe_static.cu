// Whole-layer forward that allocates nothing and needs no caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the layer: code that runs
// while another component owns the device memory budget (a serving runtime with a fixed arena), code
// that must not trigger the implicit device synchronisation a cudaMalloc/cudaFree can cause in a
// latency-critical loop, or plugin code handed only input and output pointers.  For small layers
// (the workspace must fit in MOE_STATIC_SCRATCH_BYTES) this entry point uses a scratch array that is
// part of the library image instead of a caller-owned workspace.
//
// The scratch is one file-scope __device__ array: every GPU that loads the library holds it until
// the process exits, and every call on that GPU shares it, keeping the previous call's contents.
// The only scratch state that has to start at a known value (the status word and the split-K arrival
// counters) is reset on the GPU by the alignment kernel at the start of every call.  Calls that
// overlap on the GPU (different streams, or other host threads) use the same array and race.
#include <mutex>

#include "moe_internal.h"

namespace {

static_assert(MOE_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) uint8_t g_moe_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevicesCached = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevicesCached] = {};

// Device address of the scratch array on the current device.  A host-side reference to the array is
// only a stand-in, not a device address, so the address comes from cudaGetSymbolAddress, looked up
// once per device (with that device current) and cached.
moe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (dev >= 0 && dev < kMaxDevicesCached && g_scratch_addr[dev] != nullptr) {
    *out = g_scratch_addr[dev];
    return MOE_OK;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_moe_static_scratch) != cudaSuccess || ptr == nullptr)
    return MOE_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevicesCached) g_scratch_addr[dev] = ptr;
  *out = ptr;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_fp8_block_forward_static(const moe_fwd_args* args, moe_stream_t stream) {
  if (args == nullptr) return MOE_ERR_INVALID_ARG;
  moe_ws_plan plan;
  const moe_status st = moe_workspace_plan(args->M_cap, args->E, args->H, args->I, args->topk,
                                           args->act_scale_fmt, &plan);
  if (st != MOE_OK) return st;
  if (plan.total_bytes > (size_t)MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const moe_status sa = scratch_address(&scratch);
  if (sa != MOE_OK) return sa;
  return moe_fp8_block_forward(args, scratch, (size_t)MOE_STATIC_SCRATCH_BYTES, stream);
}
