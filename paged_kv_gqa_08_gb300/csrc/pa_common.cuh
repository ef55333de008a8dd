// Device helpers shared by the libpagedattn kernels (sm_103a only).
//
// Everything here is hand-written inline PTX or plain CUDA C++:
//   * mbarrier init / arrive / expect-tx / bounded parity waits,
//   * 1-D bulk async copies global -> shared (TMA engine, no multicast),
//   * packed fp32x2 arithmetic (one instruction for two lanes' worth of FMA),
//   * bf16 <-> fp32 conversions by bit manipulation (exact widening,
//     round-to-nearest-even narrowing via the CUDA intrinsic).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"

#define PA_DEVINL __device__ __forceinline__

namespace pa {

// ----------------------------------------------------------------------------
// error flags (the word lives in api.cu; kernels get its address)
// ----------------------------------------------------------------------------
PA_DEVINL void raise_flag(unsigned int* err, unsigned int f) {
  if (err) atomicOr(err, f);
}

// ----------------------------------------------------------------------------
// shared-memory addresses, timers
// ----------------------------------------------------------------------------
PA_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

PA_DEVINL uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
PA_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

PA_DEVINL void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

PA_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

PA_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

PA_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Upper bound on any wait for an async copy or a peer warp in this library.
// Every wait is bounded: after this long the waiter raises PA_DEVERR_TIMEOUT,
// sets the CTA's abort flag and returns false, so a kernel can never hang.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Wait for phase `parity` of `bar`.  Returns false on timeout (after
// `limit_ns`) or when another thread of the CTA has already aborted
// (`*abort` != 0).
PA_DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                 unsigned int* err, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort = 1;
        raise_flag(err, PA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, size a multiple of 16.
// ----------------------------------------------------------------------------
PA_DEVINL void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (streamed data: evict first).
PA_DEVINL uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

PA_DEVINL void bulk_g2s_hint(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ----------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel of the stream still runs;
// pdl_wait() returns once that kernel has completed and its writes are visible
// (at once when the launch had no such dependency).  pdl_trigger() lets the
// next kernel of the stream start launching.
// ----------------------------------------------------------------------------
PA_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
PA_DEVINL void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------------------
// CTA barrier entered by whole warps.  bar.sync (what __syncthreads emits)
// must be executed by all threads of a warp together; a warp whose lanes took
// different paths (one lane issuing MMAs or copies while the others skip
// ahead) reconverges first.
// ----------------------------------------------------------------------------
PA_DEVINL void cta_sync() {
  __syncwarp();
  __syncthreads();
}

// ----------------------------------------------------------------------------
// named barriers (subset of warps)
// ----------------------------------------------------------------------------
PA_DEVINL void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------------------
// packed fp32x2 arithmetic
// ----------------------------------------------------------------------------
PA_DEVINL float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

PA_DEVINL float2 fadd2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

PA_DEVINL float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

// ----------------------------------------------------------------------------
// bf16 <-> fp32
// ----------------------------------------------------------------------------
// Two packed bf16 (low half = element 0) -> two floats, exact.
PA_DEVINL float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

PA_DEVINL float bf16_bits_to_float(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

PA_DEVINL uint16_t float_to_bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

PA_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  // one cvt.rn.bf16x2.f32: hi goes to the upper half
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Round a float to the storage dtype's value set (identity for fp32).
template <typename T>
PA_DEVINL float round_to(float x);
template <>
PA_DEVINL float round_to<float>(float x) { return x; }
template <>
PA_DEVINL float round_to<__nv_bfloat16>(float x) { return bf16_bits_to_float(float_to_bf16_bits(x)); }

// 16-byte vector loads / stores.
PA_DEVINL uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
PA_DEVINL uint4 ldg16_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
PA_DEVINL void stg16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

}  // namespace pa
