// Inline-PTX helpers for sm_103a: mbarriers, TMA tensor loads, warp-level
// matrix loads / MMA, and fast exp2/log2.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ----------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tensor-core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase's completion (no suspend: for a thread that
// must react at once, at the cost of issue slots while it polls).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns; on expiry OR kErrWaitTimeout into *err and return false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// Bounded wait that also gives up as soon as any CTA has reported an expired
// wait, so one failure cannot make every later CTA wait out its own timeout.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* err,
                                              uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 255u) == 0 && (*reinterpret_cast<volatile uint32_t*>(err) & kErrWaitTimeout) != 0u) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// The same bounded wait by polling, for threads that must react to a
// completed phase without a wake-up delay (the tensor-core issuers): only one
// thread of a warp should poll.
__device__ __forceinline__ bool poll_or_abort(uint64_t* bar, uint32_t parity, uint32_t* err,
                                              uint64_t limit_ns = kWaitTimeoutNs) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_test_wait(bar, parity)) {
    if ((++spins & 255u) == 0) {
      if ((*reinterpret_cast<volatile uint32_t*>(err) & kErrWaitTimeout) != 0u) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(err, kErrWaitTimeout);
        return false;
      }
    }
  }
  return true;
}

// One 32-byte global store (dst 32-byte aligned): a whole sector per lane.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// ---- TMA ---------------------------------------------------------------------

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- warp-level matrix ops -----------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held one row-pair per thread (warp-collective).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ---- scalar helpers ------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three floats in one instruction (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// launch now / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t bits) {
  return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}

// fp8 scale as a packed fp32x2 operand of dequant_e4m3x2 (built once per call).
__device__ __forceinline__ uint64_t dequant_scale2(float s) {
  const uint64_t b = __float_as_uint(s);
  return (b << 32) | b;
}

// Two e4m3 codes -> bf16x2 of bf16_rn(float(code) * scale): the product is
// one fp32 rounding, then one rounding to bf16, the dequantisation the
// prefix-prefill page writes.  HALF selects the codes in the low (0) or high
// (1) 16 bits of w, the low byte of each pair being the first element.  The
// codes convert exactly to f16, f16 -> f32 goes through the mixed-precision
// fma (x * 1 + -0, exact, signed zeros kept), both products in one packed
// fp32x2 multiply; written out in PTX so that no extra shift or mask is
// spent selecting the half (measured: 4.9 instead of 5.3 instructions a pair,
// bitwise equal on all 65,536 code pairs at seven scales).
#define PA_DEQUANT_E4M3X2_ASM(SRC)                                              \
  "{\n\t.reg .b16 c0, c1, x, y, one;\n\t.reg .b32 h2;\n\t.reg .f32 f0, f1, z;\n\t" \
  ".reg .b64 d;\n\t"                                                            \
  "mov.b16 one, 0x3C00;\n\t"                                                    \
  "mov.f32 z, 0f80000000;\n\t"                                                  \
  "mov.b32 {c0, c1}, %1;\n\t"                                                   \
  "cvt.rn.f16x2.e4m3x2 h2, " SRC ";\n\t"                                        \
  "mov.b32 {x, y}, h2;\n\t"                                                     \
  "fma.rn.f32.f16 f0, x, one, z;\n\t"                                           \
  "fma.rn.f32.f16 f1, y, one, z;\n\t"                                           \
  "mov.b64 d, {f0, f1};\n\t"                                                    \
  "mul.rn.f32x2 d, d, %2;\n\t"                                                  \
  "mov.b64 {f0, f1}, d;\n\t"                                                    \
  "cvt.rn.bf16x2.f32 %0, f1, f0;\n\t}"

template <int HALF>
__device__ __forceinline__ uint32_t dequant_e4m3x2(uint32_t w, uint64_t scale2) {
  static_assert(HALF == 0 || HALF == 1, "low or high 16 bits");
  uint32_t r;
  if constexpr (HALF == 0) {
    asm(PA_DEQUANT_E4M3X2_ASM("c0") : "=r"(r) : "r"(w), "l"(scale2));
  } else {
    asm(PA_DEQUANT_E4M3X2_ASM("c1") : "=r"(r) : "r"(w), "l"(scale2));
  }
  return r;
}
#undef PA_DEQUANT_E4M3X2_ASM

}  // namespace pa
