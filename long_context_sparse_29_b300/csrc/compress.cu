// compress.cu -- block compression of KV / indexer keys with fused RoPE and
// storage packing (mixed FP8/BF16 rows, MXFP4 keys, or fp32), and the
// standalone mixed-row packer.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）": every m
// tokens' KV entries merge into one compressed entry by a weighted sum;
// section "HCA（重度压缩注意力）": the same at a larger ratio m'; section
// "关键技术细节": RoPE on the last 64 dims, RoPE dims stored in BF16 and the
// rest in FP8, FP4 lightning indexer.
//
// Layout of the work: one warp per compressed entry.  Lane l owns channel
// pairs p = l + 32 r (r < C/64), so each token row is read as 32 coalesced
// 4-byte (bf16x2) or 8-byte (float2) loads per r; the m tokens of a block are
// streamed once from HBM.  The compression weights of the block are computed
// by the warp (softmax of m logits with the library exponential) and kept in
// shared memory.  The fp32 operation order per channel is fixed (fma over the
// tokens in order, then the channel scale, then the rotation), so the stored
// bytes are reproducible bit for bit.
#include "csa_common.cuh"
#include "launch.h"

namespace csa {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxPairs = 8;     // C <= 512

// Pack one 512-channel post-RoPE row held as 8 pairs per lane into 592 bytes.
__device__ __forceinline__ void pack_mixed_row(const float2 (&v)[kMaxPairs], int lane,
                                               uint8_t* row) {
  // groups of the 448 FP8 channels by pair slot r: {0,1}, {2,3}, {4,5}, {6}
  float amax[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) amax[g] = 0.0f;
#pragma unroll
  for (int r = 0; r < 7; ++r) {
    const int g = r >> 1;
    amax[g] = fmaxf(amax[g], fmaxf(fabsf(v[r].x), fabsf(v[r].y)));
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax[g] = fmaxf(amax[g], __shfl_xor_sync(0xffffffffu, amax[g], o));
  }
  int e[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) e[g] = fp8_group_exp(amax[g]);
#pragma unroll
  for (int r = 0; r < 7; ++r) {
    const int g = r >> 1;
    const float inv = pow2i(-e[g]);
    const int p = lane + 32 * r;
    const uint16_t c0 = e4m3_encode(__fmul_rn(v[r].x, inv));
    const uint16_t c1 = e4m3_encode(__fmul_rn(v[r].y, inv));
    *reinterpret_cast<uint16_t*>(row + 2 * p) = (uint16_t)(c0 | (c1 << 8));
  }
  {
    const uint32_t b0 = f32_to_bf16_bits(v[7].x), b1 = f32_to_bf16_bits(v[7].y);
    *reinterpret_cast<uint32_t*>(row + kMixRopeOff + 4 * lane) = b0 | (b1 << 16);
  }
  if (lane < 4) {
    float sc = pow2i(e[0]);
#pragma unroll
    for (int g = 1; g < 4; ++g)
      if (lane == g) sc = pow2i(e[g]);
    *reinterpret_cast<float*>(row + kMixScaleOff + 4 * lane) = sc;
  }
}

template <int FMT, bool BF16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
compress_kernel(const void* __restrict__ x, const float* __restrict__ z,
                const float* __restrict__ s, const float* __restrict__ rcos,
                const float* __restrict__ rsin, int64_t pos0, int B, int64_t T, int C, int R,
                int m, int64_t N, void* __restrict__ out, uint8_t* __restrict__ out_scales) {
  __shared__ float alpha_s[kWarpsPerBlock][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ent = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
  if (ent >= (int64_t)B * N) return;
  const int64_t b = ent / N, j = ent % N;
  const int64_t tok0 = b * T + j * m;   // first token row of the block

  // ---- weights of the block: a = softmax(z) with the library exponential ----
  float mu = -INFINITY;
  for (int i = lane; i < m; i += 32) mu = fmaxf(mu, z[tok0 + i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
  for (int i = lane; i < m; i += 32) alpha_s[warp][i] = sexp(__fsub_rn(z[tok0 + i], mu));
  __syncwarp();
  float S = 0.0f;
  if (lane == 0) {
    S = alpha_s[warp][0];
    for (int i = 1; i < m; ++i) S = __fadd_rn(S, alpha_s[warp][i]);
  }
  S = __shfl_sync(0xffffffffu, S, 0);
  __syncwarp();
  for (int i = lane; i < m; i += 32) alpha_s[warp][i] = __fdiv_rn(alpha_s[warp][i], S);
  __syncwarp();

  // ---- weighted sum over the block's tokens, channel pairs per lane ----
  const int npairs = C >> 1;
  float2 v[kMaxPairs];
#pragma unroll
  for (int r = 0; r < kMaxPairs; ++r) v[r] = make_float2(0.0f, 0.0f);
  for (int i = 0; i < m; ++i) {
    const float a = alpha_s[warp][i];
    const int64_t row = (tok0 + i) * C;
#pragma unroll
    for (int r = 0; r < kMaxPairs; ++r) {
      const int p = lane + 32 * r;
      if (p < npairs) {
        float x0, x1;
        if (BF16) {
          const uint32_t w = reinterpret_cast<const uint32_t*>(x)[(row >> 1) + p];
          x0 = __uint_as_float(w << 16);
          x1 = __uint_as_float(w & 0xffff0000u);
        } else {
          const float2 w = reinterpret_cast<const float2*>(x)[(row >> 1) + p];
          x0 = w.x;
          x1 = w.y;
        }
        v[r].x = __fmaf_rn(a, x0, v[r].x);
        v[r].y = __fmaf_rn(a, x1, v[r].y);
      }
    }
  }
  const int half = R >> 1;
  const int64_t P = pos0 + j * m + m - 1;   // RoPE position: the block's last token
#pragma unroll
  for (int r = 0; r < kMaxPairs; ++r) {
    const int p = lane + 32 * r;
    if (p < npairs) {
      if (s) {
        v[r].x = __fmul_rn(v[r].x, s[2 * p]);
        v[r].y = __fmul_rn(v[r].y, s[2 * p + 1]);
      }
      const int i = p - (C - R) / 2;
      if (i >= 0) {
        const float cs = rcos[P * half + i], sn = rsin[P * half + i];
        const float x0 = v[r].x, x1 = v[r].y;
        v[r].x = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
        v[r].y = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
      }
    }
  }

  // ---- store ----
  if (FMT == CSA_FMT_F32) {
    float2* o = reinterpret_cast<float2*>(out) + ent * npairs;
#pragma unroll
    for (int r = 0; r < kMaxPairs; ++r) {
      const int p = lane + 32 * r;
      if (p < npairs) o[p] = v[r];
    }
  } else if (FMT == CSA_FMT_MIXED592) {
    pack_mixed_row(v, lane, reinterpret_cast<uint8_t*>(out) + ent * kMixRow);
  } else {  // MXFP4, C in {32, 64}: block of lane's pair = p / 16 = lane / 16
    float amax = (lane < npairs) ? fmaxf(fabsf(v[0].x), fabsf(v[0].y)) : 0.0f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int sx = mx_block_exp(amax);
    if (lane < npairs) {
      const float inv = pow2i(-sx);
      const uint32_t c0 = e2m1_encode(__fmul_rn(v[0].x, inv));
      const uint32_t c1 = e2m1_encode(__fmul_rn(v[0].y, inv));
      reinterpret_cast<uint8_t*>(out)[ent * npairs + lane] = (uint8_t)(c0 | (c1 << 4));
      if ((lane & 15) == 0) out_scales[ent * (C / 32) + (lane >> 4)] = (uint8_t)(sx + 127);
    }
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
pack_mixed_kernel(const float* __restrict__ v, int64_t n, uint8_t* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
  if (row >= n) return;
  float2 x[kMaxPairs];
  const float2* src = reinterpret_cast<const float2*>(v + row * kMixD);
#pragma unroll
  for (int r = 0; r < kMaxPairs; ++r) x[r] = src[lane + 32 * r];
  pack_mixed_row(x, lane, out + row * kMixRow);
}

cudaError_t launch_compress(const void* x, bool x_bf16, const float* z, const float* s,
                            const float* rcos, const float* rsin, int64_t pos0, int B, int64_t T,
                            int C, int R, int m, int fmt, void* out, uint8_t* out_scales,
                            cudaStream_t st) {
  const int64_t N = T / m;
  const int64_t ents = (int64_t)B * N;
  if (ents == 0) return cudaSuccess;
  const dim3 grid((unsigned)((ents + kWarpsPerBlock - 1) / kWarpsPerBlock)), block(kWarpsPerBlock * 32);
#define CSA_CK(F, BF)                                                                         \
  compress_kernel<F, BF><<<grid, block, 0, st>>>(x, z, s, rcos, rsin, pos0, B, T, C, R, m, N, \
                                                 out, out_scales)
  if (fmt == CSA_FMT_F32) {
    if (x_bf16) CSA_CK(CSA_FMT_F32, true); else CSA_CK(CSA_FMT_F32, false);
  } else if (fmt == CSA_FMT_MIXED592) {
    if (x_bf16) CSA_CK(CSA_FMT_MIXED592, true); else CSA_CK(CSA_FMT_MIXED592, false);
  } else {
    if (x_bf16) CSA_CK(CSA_FMT_MXFP4, true); else CSA_CK(CSA_FMT_MXFP4, false);
  }
#undef CSA_CK
  return cudaGetLastError();
}

cudaError_t launch_pack_mixed(const float* v, int64_t n, uint8_t* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  pack_mixed_kernel<<<(unsigned)((n + kWarpsPerBlock - 1) / kWarpsPerBlock), kWarpsPerBlock * 32, 0,
                      st>>>(v, n, out);
  return cudaGetLastError();
}

}  // namespace csa
