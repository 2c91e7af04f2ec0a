// csa_common.cuh -- device-side number formats and helpers of libcsa_b300.
//
// Formats (see include/csa_b300.h): OCP FP8 E4M3 with power-of-two group
// scales and bf16 RoPE channels in 592-byte rows; OCP MX E2M1 elements with
// UE8M0 block scales of 32 for the lightning-indexer keys.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa_b300.h"

namespace csa {

constexpr int kMixD = 512;      // channels of a mixed row
constexpr int kMixDn = 448;     // FP8 channels
constexpr int kMixR = 64;       // bf16 RoPE channels
constexpr int kMixRow = 592;    // bytes per mixed row
constexpr int kMixScaleOff = 576;
constexpr int kMixRopeOff = 448;

// status block at the head of every workspace
struct Status {
  unsigned int flags;
  unsigned int first_bad;   // first offending key code seen (diagnostic)
  unsigned int pad[2];
};

__device__ __forceinline__ void flag_device_check(void* ws, unsigned int what) {
  if (ws) {
    Status* st = reinterpret_cast<Status*>(ws);
    unsigned int old = atomicOr(&st->flags, CSA_FLAG_DEVICE_CHECK);
    if (!(old & CSA_FLAG_DEVICE_CHECK)) st->first_bad = what;
  }
}

__device__ __forceinline__ void flag_timeout(void* ws) {
  if (ws) atomicOr(&reinterpret_cast<Status*>(ws)->flags, CSA_FLAG_TIMEOUT);
}

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the kernel before it on the stream finishes
// (launch_pdl in launch.h).  It first lets its own dependents launch, then
// waits until the grids it depends on have completed and their writes are
// visible -- before it reads or writes any global memory -- so the order of
// results is the stream order; only the launch latency overlaps.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// The same in two halves, for kernels that first set up what touches no
// memory another kernel of the library writes (shared memory, barriers,
// TMEM, reads of the caller's inputs and constant tables): pdl_trigger at
// the top, pdl_wait before the first access to data a preceding kernel of
// the library may write (or that one may still read, before writing it).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 2^n as fp32 for n in [-126, 127]
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((n + 127) << 23); }

// The library's fp32 exponential used for compression weights:
// Cody & Waite reduction x = n ln2 + r with ln 2 split into a 16-bit head and
// a tail, then the degree-7 Taylor polynomial of exp(r) (Horner, fma), then
// an exact scaling by 2^n.  Constants: log2(e) and 1/k! rounded to fp32;
// ln 2 truncated to 16 fractional bits and the remainder rounded to fp32.
// One rounding per operation, so the result is reproducible bit for bit.
__device__ __forceinline__ float sexp(float x) {
  if (!(x >= -87.0f)) return 0.0f;
  if (x > 88.0f) x = 88.0f;
  const float t = __fmul_rn(x, 0x1.715476p+0f);
  const float nf = rintf(t);
  float r = __fmaf_rn(-nf, 0x1.62e4p-1f, x);
  r = __fmaf_rn(-nf, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0x1p-1f);
  p = __fmaf_rn(p, r, 0x1p+0f);
  p = __fmaf_rn(p, r, 0x1p+0f);
  return __fmul_rn(p, pow2i((int)nf));
}

// E4M3, nearest-even, saturating to +-448 (hardware conversion).
__device__ __forceinline__ uint8_t e4m3_encode(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// E4M3 code -> exact value as fp32 (NaN codes are never stored).
__device__ __forceinline__ float e4m3_decode(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// smallest integer e with amax / 2^e <= 448, clamped to >= -126; 0 for amax == 0
__device__ __forceinline__ int fp8_group_exp(float amax) {
  if (amax == 0.0f) return 0;
  int E;
  const float f = frexpf(amax, &E);
  const int e = (f > 0.875f) ? E - 8 : E - 9;
  return e < -126 ? -126 : e;
}

// E2M1 magnitude code of |y| (nearest, ties to the even code, saturating at 6)
__device__ __forceinline__ uint32_t e2m1_mag(float y) {
  const float a = fabsf(y);
  return a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
       : a <= 2.5f ? 4u : a < 3.5f ? 5u : a <= 5.0f ? 6u : 7u;
}

__device__ __forceinline__ uint32_t e2m1_encode(float y) {
  return e2m1_mag(y) | (signbit(y) ? 8u : 0u);
}

// UE8M0 block exponent of MXFP4: floor(log2 amax) - 2, clamped to >= -127; 0 for amax == 0
__device__ __forceinline__ int mx_block_exp(float amax) {
  if (amax == 0.0f) return 0;
  int E;
  frexpf(amax, &E);
  const int sx = E - 3;
  return sx < -127 ? -127 : sx;
}

// x * 2^k exactly when the result is a normal number (k in [-252, 252])
__device__ __forceinline__ float scale_pow2(float x, int k) {
  const int k1 = k / 2, k2 = k - k1;
  return __fmul_rn(__fmul_rn(x, pow2i(k1)), pow2i(k2));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

}  // namespace csa
