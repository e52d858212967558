// tfx_common.cuh -- device helpers shared by the library's kernels: mbarrier and bulk-copy
// wrappers with bounded waits, E2M1/E4M3 conversions through the sm_100-family cvt
// instructions, and the mixed-precision fma used by the accumulation chains.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tfx_moe.h"

namespace tfx {

constexpr int kWarp = 32;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of the given parity to complete; gives up after timeout_ns and
// returns false (the caller reports TFX_ST_TIMEOUT and stops).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
#pragma unroll 1
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > timeout_ns) return false;
  }
}

// One-dimensional bulk copy global -> shared, completing `bytes` on the barrier.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Named barrier over the first `threads` threads of the block (id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------------ conversions
// Eight E2M1 codes (one 32-bit word, code i in bits 4i..4i+3) -> four f16x2 registers;
// register q holds codes 2q (low half) and 2q+1 (high half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                                 uint32_t& h3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// Two E4M3 codes (low 16 bits; lower byte -> low half) -> f16x2. Exact: every E4M3 value
// is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(h) : "r"(two));
  return h;
}

// fp32 value -> E4M3 code, nearest even, saturating at +-448 (NaN -> NaN code).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint32_t r;
  asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}"
      : "=r"(r)
      : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// c + a.lo * b.lo then + a.hi * b.hi, each step one fma with a single rounding to fp32
// (the products of two f16 values are exact in fp32 anyway).
__device__ __forceinline__ float fma2_f16(uint32_t a, uint32_t b, float c) {
  asm("{\n .reg .f16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.f16 %0, al, bl, %0;\n fma.rn.f32.f16 %0, ah, bh, %0;\n}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// E8M0 scale code -> fp32 2^(s-127); 0 -> 2^-127 (subnormal); 0xFF -> NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  uint32_t b = s << 23;
  b = (s == 0u) ? 0x00400000u : b;
  b = (s == 255u) ? 0x7FC00000u : b;
  return __uint_as_float(b);
}

// 2^(127-s) for an E8M0 code s in [0, 254] (the reciprocal of the scale, exact).
__device__ __forceinline__ float e8m0_recip_f32(uint32_t s) {
  return (s >= 254u) ? __uint_as_float(0x00400000u >> (s - 254u)) : __uint_as_float((254u - s) << 23);
}

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace tfx
