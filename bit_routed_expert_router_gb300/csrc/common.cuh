// Device-side helpers shared by the libmoe kernels (sm_103a).
//
// Inline PTX for the pieces the kernels are built from: mbarriers, 1-D bulk
// (TMA engine) copies global -> shared, the register-sourced bf16 tensor-core
// MMA used by the int4 GEMVs, and bounded spin-waits that report a timeout
// through a device error word instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

// Roughly 2 s at GB300 clocks: far beyond any legitimate wait in these kernels.
constexpr long long kSpinLimitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbarrier_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Test (and, while the phase is open, suspend the thread for up to about
// 20 us) for completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and flags the error word)
// if the phase did not complete within kSpinLimitCycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kSpinLimitCycles) {
      atomicOr(err, ERR_WAIT_TIMEOUT);
      return false;
    }
  }
  return true;
}

// 1-D bulk copy global -> shared through the TMA engine, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators, A/B from registers.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Eight packed nibbles -> four bf16x2 registers holding (128 + q).
// The word's nibble i sits at bits [4i, 4i+4); register r receives nibbles r
// and r+4 (low and high half).  0x4300 is bf16 128.0, whose unit in the last
// place is 1, so OR-ing a nibble into the mantissa gives exactly 128 + q.
__device__ __forceinline__ void nibbles_to_bf16x2(uint32_t w, uint32_t (&a)[4]) {
  a[0] = (w & 0x000F000Fu) | 0x43004300u;
  a[1] = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
  a[2] = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
  a[3] = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
}

// One m16n8k16 fp16 MMA, D = A * B + C (C = D, or zero with kZero), whose A
// fragment is the eight packed nibbles of word w: register r takes nibbles r
// (low half) and r + 4 (high half) where they sit, under the fp16 exponent of
// 1024 (unit in the last place 1), with four logic ops and one shift.
// Registers 0 and 2 (fragment rows g) hold 1024 + q; registers 1 and 3 (rows
// g + 8) keep their nibbles four bits up and hold 1024 + 16 q, which the
// epilogue undoes per row.  (bf16 has too few mantissa bits for the second
// form, which is why the activations of these MMAs are fp16.)  Unpack and
// MMA are one asm block: with the unpack in C++ the compiler moved every
// unpacked word into the MMA's operand registers (about 16 extra
// instructions per 64-wide group, by ncu instruction counts).  Not volatile,
// so the compiler may interleave the MMAs of several groups.
template <bool kZero>
__device__ __forceinline__ void mma_nib(float (&c)[4], uint32_t w, uint32_t b0, uint32_t b1) {
  const uint32_t lo = 0x000F000Fu, hi = 0x00F000F0u, e = 0x64006400u;
  if (kZero) {
    asm("{\n\t.reg .b32 a0, a1, a2, a3, w8;\n\t.reg .f32 z;\n\t"
        "mov.f32 z, 0f00000000;\n\t"
        "shr.b32 w8, %4, 8;\n\t"
        "lop3.b32 a0, %4, %7, %9, 0xEA;\n\t"
        "lop3.b32 a1, %4, %8, %9, 0xEA;\n\t"
        "lop3.b32 a2, w8, %7, %9, 0xEA;\n\t"
        "lop3.b32 a3, w8, %8, %9, 0xEA;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3}, {%5,%6}, {z,z,z,z};\n\t}"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(w), "r"(b0), "r"(b1), "r"(lo), "r"(hi), "r"(e));
  } else {
    asm("{\n\t.reg .b32 a0, a1, a2, a3, w8;\n\t"
        "shr.b32 w8, %4, 8;\n\t"
        "lop3.b32 a0, %4, %7, %9, 0xEA;\n\t"
        "lop3.b32 a1, %4, %8, %9, 0xEA;\n\t"
        "lop3.b32 a2, w8, %7, %9, 0xEA;\n\t"
        "lop3.b32 a3, w8, %8, %9, 0xEA;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3}, {%5,%6}, {%0,%1,%2,%3};\n\t}"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(w), "r"(b0), "r"(b1), "r"(lo), "r"(hi), "r"(e));
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float half_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<uint16_t>(v >> 16)));
}

// Programmatic dependent launch controls (no-ops when launched without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Exact sum of products rounded onto the 2^-40 grid, without 64-bit float ->
// integer conversions (which issue at a small fraction of the fp32 rate).
// A product v = x * w * 2^40 (|v| < 2^51, at most 24 significant bits) is cut
// as RNE(v) = q2 * 2^44 + q1 * 2^22 + q0: adding and subtracting 1.5 * 2^67
// rounds v to a multiple of 2^44 (the binade of that constant has that unit),
// the remainder is exact and is cut the same way at 2^22, and the last
// remainder (|r| <= 2^21) is rounded to an integer, ties to even, by adding
// 1.5 * 2^23.  Each q is the difference of the sum's bit pattern and the
// constant's, so the three partial sums are plain int32 additions of bit
// patterns, corrected by the number of terms at the end.  At most 512 terms
// may go into one accumulator before fix40_value.
struct Fix40 {
  uint32_t b2 = 0, b1 = 0, b0 = 0;   // sums of bit patterns (mod 2^32)
  uint32_t n = 0;                    // terms
};

__device__ __forceinline__ void fix40_add(Fix40& A, float v) {
  const float M2 = 221360928884514619392.0f;   // 1.5 * 2^67
  const float M1 = 52776558133248.0f;          // 1.5 * 2^45
  const float M0 = 12582912.0f;                // 1.5 * 2^23
  const float s2 = __fadd_rn(v, M2);
  const float r2 = __fsub_rn(v, __fsub_rn(s2, M2));
  const float s1 = __fadd_rn(r2, M1);
  const float r1 = __fsub_rn(r2, __fsub_rn(s1, M1));
  const float s0 = __fadd_rn(r1, M0);
  A.b2 += __float_as_uint(s2);
  A.b1 += __float_as_uint(s1);
  A.b0 += __float_as_uint(s0);
  A.n += 1u;
}

__device__ __forceinline__ long long fix40_value(const Fix40& A) {
  const int q2 = static_cast<int>(A.b2 - A.n * 0x61400000u);   // bit pattern of 1.5 * 2^67
  const int q1 = static_cast<int>(A.b1 - A.n * 0x56400000u);   // 1.5 * 2^45
  const int q0 = static_cast<int>(A.b0 - A.n * 0x4B400000u);   // 1.5 * 2^23
  return (static_cast<long long>(q2) << 44) + (static_cast<long long>(q1) << 22) + q0;
}

__device__ __forceinline__ int64_t shfl_xor_i64(int64_t v, int m) {
  int lo = static_cast<int>(v & 0xFFFFFFFFLL);
  int hi = static_cast<int>(v >> 32);
  lo = __shfl_xor_sync(0xFFFFFFFFu, lo, m);
  hi = __shfl_xor_sync(0xFFFFFFFFu, hi, m);
  return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

}  // namespace moe
