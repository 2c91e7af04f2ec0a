// attn_common.cuh -- device helpers shared by the tensor-core attention
// kernels (attn_tc.cu: prefill and long key lists; attn_decode.cu: decode):
// the 128-byte swizzle, the softmax warps' voting barrier, exp2, asynchronous
// copies, and the exact FP8 -> bf16 expansion of the mixed cache rows.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_ptx.cuh"

namespace csa {
namespace attn {

using namespace tc;

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk16) {
  return row * 128u + (((chunk16 ^ row) & 7u) << 4);
}

// Barrier of the four softmax warps (named barrier 1, 128 threads) that
// returns how many of them voted: every softmax warp executes the same
// sequence of these, and exits only on a count read from one of them, so no
// warp can be left waiting at a barrier the others never reach.
__device__ __forceinline__ uint32_t group_vote(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %1, 0;\n bar.red.popc.u32 %0, 1, 128, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r;
}

// 2^x by the hardware approximation (a few ulp; P is rounded to bf16 next).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// cp.async of 16 bytes, of which the first `src_bytes` (0 or 16) are read
// and the rest zero-filled.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// An arrive on `bar` once this thread's cp.async copies so far have landed;
// it is one of the arrivals the barrier's count expects.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(void* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// 16 E4M3 codes times 2^e -> 16 bf16, exact, without the conversion pipe.
// A code's 7 magnitude bits placed at bits 20..26 of an fp32 read as
// 2^(E-127) (1 + m/8) for exponent field E >= 1 and as m 2^-129 for E = 0:
// the E4M3 value times 2^-120 in both cases.  One fp32 multiply by
// 2^(120 + e) (two when 2^(120 + e) is not a finite fp32) gives the value
// times the group scale 2^e exactly -- it has at most 4 significant bits --
// so the top half of the fp32 is the bf16.
__device__ __forceinline__ uint32_t e4m3_bits(uint32_t x, int byte) {
  // fp32 bit pattern holding the magnitude bits of code `byte` of x at bits
  // 20..26 and its sign at bit 31
  switch (byte) {
    case 0: return ((x << 20) & 0x07F00000u) | ((x << 24) & 0x80000000u);
    case 1: return ((x << 12) & 0x07F00000u) | ((x << 16) & 0x80000000u);
    case 2: return ((x << 4) & 0x07F00000u) | ((x << 8) & 0x80000000u);
    default: return ((x >> 4) & 0x07F00000u) | (x & 0x80000000u);
  }
}

__device__ __forceinline__ void dequant16(const uint4 c, float sc, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t r[8];
  if (sc <= 128.0f) {                       // 2^(120 + e) is a finite fp32: one multiply
    const float s120 = __fmul_rn(sc, 0x1p120f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float f0 = __fmul_rn(__uint_as_float(e4m3_bits(w[i], 0)), s120);
      const float f1 = __fmul_rn(__uint_as_float(e4m3_bits(w[i], 1)), s120);
      const float f2 = __fmul_rn(__uint_as_float(e4m3_bits(w[i], 2)), s120);
      const float f3 = __fmul_rn(__uint_as_float(e4m3_bits(w[i], 3)), s120);
      r[2 * i] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
      r[2 * i + 1] = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) f[j] = __fmul_rn(__fmul_rn(__uint_as_float(e4m3_bits(w[i], j)), 0x1p120f), sc);
      r[2 * i] = __byte_perm(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632);
      r[2 * i + 1] = __byte_perm(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632);
    }
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

}  // namespace attn
}  // namespace csa
