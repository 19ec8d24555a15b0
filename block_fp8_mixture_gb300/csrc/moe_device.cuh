// Device-side building blocks for the sm_103a kernels: mbarriers with bounded waits, TMA tile
// loads, tcgen05 (MMA into tensor memory, loads out of it), and the numeric helpers of the layer
// (E4M3 conversion, BF16 rounding, 1x128 scales).  Written from the PTX ISA's descriptions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

// ------------------------------------------------------------------ basics
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------- programmatic dependent launch
// Wait until the preceding kernels of the stream have completed and their writes are visible.  Every
// kernel calls this before it reads or writes global memory another kernel of the layer touches.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel of the stream begin launching (it still waits in grid_dep_wait for this
// kernel to complete before touching shared data).
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase of `bar` with the given parity to complete.  Gives up when the CTA's
// abort flag is raised by another role or after limit_ns (kWaitLimitNs in the layer kernels); on
// expiry it raises the abort flag and records MOE_ERR_DEVICE_TIMEOUT in the global status word.
// Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, int* status,
                                                uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicCAS(status, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  return mbar_wait_limit(bar, parity, abort_flag, status, kWaitLimitNs);
}

// Bounded wait until the int32 at `counter` reaches `target` (acquire at GPU scope), for counters
// other CTAs release; on expiry it raises the CTA abort flag and records MOE_ERR_DEVICE_TIMEOUT.
__device__ __forceinline__ bool wait_counter_at_least(const int32_t* counter, int target,
                                                      volatile int* abort_flag, int* status) {
  auto load = [&] {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(64);
    if (load() >= target) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(status, 0, (int)MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Order this thread's acquire of data written by other CTAs through the generic proxy before its
// later async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------------- TMA
// 2-D tiled bulk tensor load into shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Same with an L2 eviction-priority hint (createpolicy.fractional).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 1-D tiled bulk tensor load (a box of a flat array; elements past the end read as zero).
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* map, int x,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2}], [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(bar)
      : "memory");
}

// 3-D tiled bulk tensor load (used with x = 128 bytes of K, y = rows, z = 128-byte K chunks).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 int c2, int c3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

// 2-D tiled bulk tensor store from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}

// 3-D tiled bulk tensor store from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until the bulk stores issued by this thread have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until the bulk stores issued by this thread are complete.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
// Tensor memory is allocated by one whole warp; the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, FP8 E4M3 x E4M3 -> fp32, issued by one thread.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// D[tmem] (+)= (A * 2^sfa)[smem] * (B * 2^sfb)[smem]^T: kind::mxf8f6f4 with UE8M0 scale factors
// in tensor memory, one per 32-element K block of every row of A (sfa: lane = row) and of every
// row of B (sfb: lane = row), issued by one thread.
__device__ __forceinline__ void mma_f8_bs(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;"
      "\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A and B E4M3, both K-major, UE8M0
// scale factors taken from byte 0 of their tensor-memory words, shape M x N (D is fp32).
__host__ __device__ constexpr uint32_t make_idesc_mx_e4m3(int M, int N) {
  return (0u << 4)                            // B scale factor: byte 0
         | (0u << 7) | (0u << 10)             // A, B format: E4M3
         | (0u << 15) | (0u << 16)            // A, B K-major
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | (1u << 23)                         // scale factor type: UE8M0
         | ((uint32_t)(M >> 4) << 24)         // M / 16
         | (0u << 29);                        // A scale factor: byte 0
}

// Four consecutive 32-bit tensor-memory columns of this warp's 32 lanes from registers.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2,
                                         uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v0), "r"(v1), "r"(v2), "r"(v3)
               : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor of kind::f8f6f4: D fp32, A and B E4M3, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int M, int N) {
  return (1u << 4)                            // D format: fp32
         | (0u << 7) | (0u << 10)             // A, B format: E4M3
         | (0u << 15) | (0u << 16)            // A, B K-major
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// Shared-memory matrix descriptor of a K-major operand stored in 128-byte swizzled rows: 8-row
// groups of 1024 bytes (stride byte offset), start address in 16-byte units.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t sbo = 1024) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused for this layout)
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;  // stride byte offset between 8-row groups
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}

// 32 lanes x 32 columns of 32-bit tensor memory -> 32 registers per thread (lane = thread's lane
// within its warp's quarter of TMEM lanes).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------ numerics
// Two fp32 -> two E4M3 codes (round to nearest even, saturating); lo goes to the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// fp32 -> nearest BF16 bit pattern (ties to even).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

// Two fp32 values -> nearest BF16 (ties to even), packed: lo in bits 0..15, hi in bits 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_round(float v) {
  return bf16_bits_to_f32(f32_to_bf16_bits(v));
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

// 1x128 group scale: max(RN(amax/448), RN(1/(448*512))); POW2/UE8M0 round up to a power of two.
__device__ __forceinline__ float group_scale(float amax, int fmt) {
  float s = fmaxf(__fdiv_rn(amax, 448.0f), kScaleFloor);
  if (fmt != MOE_SCALE_FP32) {
    uint32_t b = __float_as_uint(s);
    if (b & 0x7FFFFFu) b = (b & 0xFF800000u) + 0x00800000u;
    s = __uint_as_float(b);
  }
  return s;
}

// 1x128 quantization of one value set: scale and per-element multiplier-or-divisor handling for the
// two numerics.  Returns the scale to store; with RECIPROCAL numerics and fp32 scales *inv holds the
// multiplier RN(448/amax) (capped at 448*512), otherwise *inv = 0 and callers divide by the scale.
__device__ __forceinline__ float group_scale_numerics(float amax, int fmt, int numerics, float* inv) {
  if (numerics == MOE_NUMERICS_RECIPROCAL && fmt == MOE_SCALE_FP32) {
    const float m = fminf(__fdiv_rn(448.0f, amax), 448.0f * 512.0f);
    *inv = m;
    return __frcp_rn(m);
  }
  *inv = 0.0f;
  return group_scale(amax, fmt);
}

// RN(v / s), or RN(v * inv) when inv != 0.
__device__ __forceinline__ float quant_div(float v, float s, float inv) {
  return inv != 0.0f ? __fmul_rn(v, inv) : __fdiv_rn(v, s);
}

// Scale value from a stored scale (fp32 word, or a UE8M0 byte 2^(b-127)).
__device__ __forceinline__ float load_scale(const void* base, size_t idx, int is_ue8m0) {
  if (is_ue8m0) {
    uint32_t b = static_cast<const uint8_t*>(base)[idx];
    return __uint_as_float(b << 23);
  }
  return static_cast<const float*>(base)[idx];
}

// Scale value held in shared memory (fp32 word or UE8M0 byte) at element idx.
__device__ __forceinline__ float smem_scale_at(const uint8_t* base, int idx, int is_ue8m0) {
  if (is_ue8m0) return __uint_as_float((uint32_t)base[idx] << 23);
  return reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ void store_scale(void* base, size_t idx, float s, int is_ue8m0) {
  if (is_ue8m0)
    static_cast<uint8_t*>(base)[idx] = static_cast<uint8_t>(__float_as_uint(s) >> 23);
  else
    static_cast<float*>(base)[idx] = s;
}

}  // namespace moe
