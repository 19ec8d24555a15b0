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
//
// The array's device address is looked up in the first call made in each context (a device reset
// creates a new context, and the next call looks the address up again).  Make that first call before
// any stream capture.  A device-side wait that runs out records MOE_ERR_DEVICE_TIMEOUT in the
// array's status word, which no entry point reads back: such a timeout is not reported to the
// caller of this path.
#include <cuda.h>

#include <mutex>

#include "moe_internal.h"

namespace {

static_assert(MOE_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) uint8_t g_moe_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevicesCached = 64;

// Driver calls that name the current context (resolved once through the runtime's entry-point query,
// so the library needs no link-time dependency on the driver library).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(ptr);
  });
  return fns;
}

// Process-unique id of the context current on this thread for device `dev` (the device's primary
// context under the runtime API).  The id changes when that context is destroyed and created again
// (cudaDeviceReset, or the primary context released and retained anew), unlike the device ordinal.
moe_status current_context_id(int dev, unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return MOE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  if (ctx == nullptr) {
    // no context current on this thread yet: make the device's primary context current
    if (cudaSetDevice(dev) != cudaSuccess || f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return MOE_ERR_CUDA;
  }
  return f.get_id(ctx, id) == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

struct ScratchEntry {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
std::mutex g_scratch_mutex;
ScratchEntry g_scratch[kMaxDevicesCached];

// Device address of the scratch array in the current context.  A host-side reference to the array is
// only a stand-in, not a device address, so the address comes from cudaGetSymbolAddress, looked up
// with the device current and cached per device together with the id of the context it belongs to.
// The module, and with it the array, is loaded again in a new context (after a device reset), where
// the array can sit at another address: a context id that differs from the cached one triggers a new
// lookup, so a stale address is never used.
moe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned long long ctx_id = 0;
  const moe_status cs = current_context_id(dev, &ctx_id);
  if (cs != MOE_OK) return cs;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const bool cached = dev >= 0 && dev < kMaxDevicesCached;
  if (cached && g_scratch[dev].ptr != nullptr && g_scratch[dev].ctx_id == ctx_id) {
    *out = g_scratch[dev].ptr;
    return MOE_OK;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_moe_static_scratch) != cudaSuccess || ptr == nullptr)
    return MOE_ERR_CUDA;
  if (cached) {
    g_scratch[dev].ctx_id = ctx_id;
    g_scratch[dev].ptr = ptr;
  }
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
