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

// The compression weights of one block, by one warp: alpha[i] = softmax(z)[i]
// for i < m with the library exponential (max, exponentials, their sum in
// token order, one division each).  alpha is m floats of shared memory.
__device__ __forceinline__ void entry_weights(const float* __restrict__ z, int m, float* alpha, int lane) {
  float mu = -INFINITY;
  for (int i = lane; i < m; i += 32) mu = fmaxf(mu, z[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
  for (int i = lane; i < m; i += 32) alpha[i] = sexp(__fsub_rn(z[i], mu));
  __syncwarp();
  float S = 0.0f;
  if (lane == 0) {
    S = alpha[0];
    for (int i = 1; i < m; ++i) S = __fadd_rn(S, alpha[i]);
  }
  S = __shfl_sync(0xffffffffu, S, 0);
  __syncwarp();
  for (int i = lane; i < m; i += 32) alpha[i] = __fdiv_rn(alpha[i], S);
  __syncwarp();
}

// Channels 2p, 2p+1 of x (m rows, row stride C elements) under the weights:
// fma over the tokens in order, the only order the stored bytes allow.
template <bool BF16>
__device__ __forceinline__ float2 load_pair(const void* __restrict__ x, int64_t row, int p) {
  if (BF16) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(x)[(row >> 1) + p];
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  return reinterpret_cast<const float2*>(x)[(row >> 1) + p];
}

// The weighted sum, the channel scale s (or NULL), RoPE of the last R
// channels at position P and the store in format FMT at out / out_scales, by
// one warp whose lane holds pairs p = lane + 32 r in v.
template <int FMT>
__device__ __forceinline__ void entry_finish(float2 (&v)[kMaxPairs], const float* __restrict__ s,
                                             const float* __restrict__ rcos, const float* __restrict__ rsin,
                                             int64_t P, int C, int R, void* __restrict__ out,
                                             uint8_t* __restrict__ out_scales, int lane) {
  const int npairs = C >> 1, half = R >> 1;
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
  if (FMT == CSA_FMT_F32) {
    float2* o = reinterpret_cast<float2*>(out);
#pragma unroll
    for (int r = 0; r < kMaxPairs; ++r) {
      const int p = lane + 32 * r;
      if (p < npairs) o[p] = v[r];
    }
  } else if (FMT == CSA_FMT_MIXED592) {
    pack_mixed_row(v, lane, reinterpret_cast<uint8_t*>(out));
  } else if (FMT == CSA_FMT_FP8B32) {   // FP8 keys, C in {32, 64}: block of lane's pair = lane / 16
    float amax = (lane < npairs) ? fmaxf(fabsf(v[0].x), fabsf(v[0].y)) : 0.0f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = fp8_group_exp(amax);
    if (lane < npairs) {
      const float inv = pow2i(-e);
      const uint32_t c0 = e4m3_encode(__fmul_rn(v[0].x, inv));
      const uint32_t c1 = e4m3_encode(__fmul_rn(v[0].y, inv));
      reinterpret_cast<uint16_t*>(out)[lane] = (uint16_t)(c0 | (c1 << 8));
      if ((lane & 15) == 0) out_scales[lane >> 4] = (uint8_t)(e + 127);
    }
  } else {  // MXFP4, C in {32, 64}: block of lane's pair = p / 16 = lane / 16
    float amax = (lane < npairs) ? fmaxf(fabsf(v[0].x), fabsf(v[0].y)) : 0.0f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int sx = mx_block_exp(amax);
    if (lane < npairs) {
      const float inv = pow2i(-sx);
      const uint32_t c0 = e2m1_encode(__fmul_rn(v[0].x, inv));
      const uint32_t c1 = e2m1_encode(__fmul_rn(v[0].y, inv));
      reinterpret_cast<uint8_t*>(out)[lane] = (uint8_t)(c0 | (c1 << 4));
      if ((lane & 15) == 0) out_scales[lane >> 4] = (uint8_t)(sx + 127);
    }
  }
}

// One compressed entry by one warp: the m token rows at x (row stride C
// elements), their logits z[0..m), the channel scale s (or NULL), RoPE of the
// last R channels at position P, stored in format FMT at out (entry 0 of out)
// and out_scales.  alpha is m floats of warp-private shared memory.
template <int FMT, bool BF16>
__device__ __forceinline__ void compress_entry(const void* __restrict__ x, const float* __restrict__ z,
                                               const float* __restrict__ s, const float* __restrict__ rcos,
                                               const float* __restrict__ rsin, int64_t P, int C, int R, int m,
                                               void* __restrict__ out, uint8_t* __restrict__ out_scales,
                                               float* alpha, int lane) {
  entry_weights(z, m, alpha, lane);
  const int npairs = C >> 1;
  float2 v[kMaxPairs];
#pragma unroll
  for (int r = 0; r < kMaxPairs; ++r) v[r] = make_float2(0.0f, 0.0f);
  for (int i = 0; i < m; ++i) {
    const float a = alpha[i];
#pragma unroll
    for (int r = 0; r < kMaxPairs; ++r) {
      const int p = lane + 32 * r;
      if (p < npairs) {
        const float2 w = load_pair<BF16>(x, (int64_t)i * C, p);
        v[r].x = __fmaf_rn(a, w.x, v[r].x);
        v[r].y = __fmaf_rn(a, w.y, v[r].y);
      }
    }
  }
  entry_finish<FMT>(v, s, rcos, rsin, P, C, R, out, out_scales, lane);
}

// The same with one logit per token and channel: z holds the m blocks' rows
// with stride C (z[i C + c]); channel c's weights are the softmax of its own m
// logits, by the sequence of entry_weights written per channel (max, the
// exponentials, their sum in token order, one division each), then the same
// fma over the tokens.  The exponentials are evaluated twice (sum, weights):
// the same fp32 values both times.
template <int FMT, bool BF16>
__device__ __forceinline__ void compress_entry_channel_logits(const void* __restrict__ x,
                                                              const float* __restrict__ z,
                                                              const float* __restrict__ s,
                                                              const float* __restrict__ rcos,
                                                              const float* __restrict__ rsin, int64_t P, int C,
                                                              int R, int m, void* __restrict__ out,
                                                              uint8_t* __restrict__ out_scales, int lane) {
  const int npairs = C >> 1;
  float2 v[kMaxPairs];
#pragma unroll
  for (int r = 0; r < kMaxPairs; ++r) {
    v[r] = make_float2(0.0f, 0.0f);
    const int p = lane + 32 * r;
    if (p < npairs) {
      const float2* z2 = reinterpret_cast<const float2*>(z);
      float2 mu = make_float2(-INFINITY, -INFINITY);
      for (int i = 0; i < m; ++i) {
        const float2 w = z2[((int64_t)i * C >> 1) + p];
        mu.x = fmaxf(mu.x, w.x);
        mu.y = fmaxf(mu.y, w.y);
      }
      float2 S = make_float2(0.0f, 0.0f);
      for (int i = 0; i < m; ++i) {
        const float2 w = z2[((int64_t)i * C >> 1) + p];
        const float ex = sexp(__fsub_rn(w.x, mu.x)), ey = sexp(__fsub_rn(w.y, mu.y));
        S.x = i == 0 ? ex : __fadd_rn(S.x, ex);
        S.y = i == 0 ? ey : __fadd_rn(S.y, ey);
      }
      for (int i = 0; i < m; ++i) {
        const float2 w = z2[((int64_t)i * C >> 1) + p];
        const float ax = __fdiv_rn(sexp(__fsub_rn(w.x, mu.x)), S.x);
        const float ay = __fdiv_rn(sexp(__fsub_rn(w.y, mu.y)), S.y);
        const float2 xv = load_pair<BF16>(x, (int64_t)i * C, p);
        v[r].x = __fmaf_rn(ax, xv.x, v[r].x);
        v[r].y = __fmaf_rn(ay, xv.y, v[r].y);
      }
    }
  }
  entry_finish<FMT>(v, s, rcos, rsin, P, C, R, out, out_scales, lane);
}

template <int FMT, bool BF16, bool ZC>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
compress_kernel(const void* __restrict__ x, const float* __restrict__ z,
                const float* __restrict__ s, const float* __restrict__ rcos,
                const float* __restrict__ rsin, int64_t pos0, int B, int64_t T, int C, int R,
                int m, int64_t N, void* __restrict__ out, uint8_t* __restrict__ out_scales) {
  pdl_begin();
  __shared__ float alpha_s[kWarpsPerBlock][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ent = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
  if (ent >= (int64_t)B * N) return;
  const int64_t b = ent / N, j = ent % N;
  const int64_t tok0 = b * T + j * m;   // first token row of the block
  const int64_t P = pos0 + j * m + m - 1;   // RoPE position: the block's last token
  const size_t esz = BF16 ? 2 : 4;
  void* o = FMT == CSA_FMT_F32 ? (void*)(reinterpret_cast<float*>(out) + ent * C)
            : FMT == CSA_FMT_MIXED592 ? (void*)(reinterpret_cast<uint8_t*>(out) + ent * kMixRow)
            : FMT == CSA_FMT_FP8B32   ? (void*)(reinterpret_cast<uint8_t*>(out) + ent * C)
                                      : (void*)(reinterpret_cast<uint8_t*>(out) + ent * (C / 2));
  constexpr bool kScales = FMT == CSA_FMT_MXFP4 || FMT == CSA_FMT_FP8B32;
  if (ZC)
    compress_entry_channel_logits<FMT, BF16>(reinterpret_cast<const uint8_t*>(x) + tok0 * C * esz, z + tok0 * C, s,
                                             rcos, rsin, P, C, R, m, o, kScales ? out_scales + ent * (C / 32) : nullptr,
                                             lane);
  else
    compress_entry<FMT, BF16>(reinterpret_cast<const uint8_t*>(x) + tok0 * C * esz, z + tok0, s, rcos, rsin, P, C,
                              R, m, o, kScales ? out_scales + ent * (C / 32) : nullptr, alpha_s[warp], lane);
}

// Decode-time cache maintenance: the new token at position t (t_pos[b])
// enters the ring of the sequence's last m raw tokens (slot t mod m), is
// packed into the window cache at row t - swa_pos0[b] (when that row is past
// the buffer, the last W - 1 rows first move to the front and swa_pos0[b]
// becomes t - W + 1), and when t closes a block ((t + 1) mod m == 0) the
// block is compressed into entry (t + 1) / m - 1 of the cache and, with its
// own ring, of the indexer keys.  The work of a sequence is split over
// kAppendParts CTAs with disjoint outputs, so their latency chains run side
// by side: part 0 the ring slot and the window row; parts 1-4 one 128-channel
// quarter of the closing entry each (FP8 groups 0, 1, 2, and group 3 with the
// bf16 RoPE channels); part 5 the closing indexer key.  The parts read the
// new token from kv / kI and the block's older tokens from the ring slots
// 0 .. m - 2 (part 0 writes only slot t mod m = m - 1 then), and every
// channel is summed over the m tokens in token order and packed by the same
// operations as compress_entry / pack_mixed_row: the same bytes.
constexpr int kAppendParts = 6;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
decode_append_kernel(const __nv_bfloat16* __restrict__ kv, const float* __restrict__ z,
                     const __nv_bfloat16* __restrict__ kI, const float* __restrict__ zI,
                     const float* __restrict__ s, const float* __restrict__ sI,
                     const float* __restrict__ rcos, const float* __restrict__ rsin, int64_t rope_rows,
                     const int64_t* __restrict__ t_pos, int C, int R, int CI, int m,
                     __nv_bfloat16* __restrict__ kv_tail, float* __restrict__ z_tail,
                     __nv_bfloat16* __restrict__ kI_tail, float* __restrict__ zI_tail,
                     uint8_t* __restrict__ cache, int64_t nmax, uint8_t* __restrict__ kI_codes,
                     uint8_t* __restrict__ kI_scales, uint8_t* __restrict__ swa, int64_t Ts, int W,
                     int64_t* __restrict__ swa_pos0) {
  pdl_begin();
  __shared__ float alpha_s[128];             // the block's weights
  __shared__ float z_s[128];                 // the block's logits
  __shared__ float rope_s[2][32];            // cos, sin of position t (R = 64)
  __shared__ float2 acc_s[64];               // this part's pair sums
  __shared__ float amax_s[2];
  extern __shared__ __align__(16) uint8_t ring_s[];   // closing block: m rows of this part's channels (bf16)
  const int b = blockIdx.x, part = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t = t_pos[b];
  if (t < 0 || t >= rope_rows) return;   // no RoPE row for it: nothing is stored
  const bool closes = (t + 1) % m == 0 && (t + 1) / m - 1 < nmax;
  if (part == 0) {
    // ---- the raw token into its ring slot; the window row ----
    const int64_t old0 = W > 0 ? swa_pos0[b] : 0;
    const int slot = (int)(t % m);
    for (int i = tid; i < (R >> 1); i += blockDim.x) {
      rope_s[0][i] = rcos[t * (R >> 1) + i];
      rope_s[1][i] = rsin[t * (R >> 1) + i];
    }
    for (int c = tid; c < C / 8; c += blockDim.x)
      reinterpret_cast<uint4*>(kv_tail + ((int64_t)b * m + slot) * C)[c] = reinterpret_cast<const uint4*>(kv + (int64_t)b * C)[c];
    if (kI)
      for (int c = tid; c < CI / 8; c += blockDim.x)
        reinterpret_cast<uint4*>(kI_tail + ((int64_t)b * m + slot) * CI)[c] =
            reinterpret_cast<const uint4*>(kI + (int64_t)b * CI)[c];
    if (tid == 0) {
      z_tail[(int64_t)b * m + slot] = z[b];
      if (kI) zI_tail[(int64_t)b * m + slot] = zI[b];
    }
    if (W > 0) {
      const bool slide = t - old0 >= Ts;
      __syncthreads();   // every thread has read swa_pos0[b]; the RoPE row is in
      if (slide) {
        // rows of tokens t - W + 1 .. t - 1 move to rows 0 .. W - 2; source rows
        // are >= Ts - W + 1 >= W + 1 (Ts >= 2 W): no overlap.  Rows past the
        // buffer (appends out of order) are not read.
        const int64_t keep0 = t - W + 1, src0 = keep0 - old0;
        const int per = kMixRow / 16;
        const uint4* srcp = reinterpret_cast<const uint4*>(swa + (int64_t)b * Ts * kMixRow);
        uint4* dst = reinterpret_cast<uint4*>(swa + (int64_t)b * Ts * kMixRow);
        for (int i = tid; i < (W - 1) * per; i += blockDim.x) {
          const int64_t sr = src0 + i / per;
          if (sr >= 0 && sr < Ts) dst[i] = srcp[sr * per + i % per];
        }
        __syncthreads();
        if (tid == 0) swa_pos0[b] = keep0;
      }
      const int64_t row = slide ? (int64_t)W - 1 : t - old0;
      if (warp == 0 && row >= 0 && row < Ts) {   // the token itself: m = 1, no channel scale, RoPE at t
        const float zz = 0.0f;
        compress_entry<CSA_FMT_MIXED592, true>(kv + (int64_t)b * C, &zz, nullptr, rope_s[0], rope_s[1], 0, C, R, 1,
                                               swa + ((int64_t)b * Ts + row) * kMixRow, nullptr, alpha_s, lane);
      }
    }
    return;
  }
  const bool key = part == kAppendParts - 1;
  if (!closes || (key && !kI)) return;
  // ---- a closing block: this part's channels [c0, c0 + nc) of the m rows ----
  const int64_t j = (t + 1) / m - 1;
  const int cc = key ? CI : C;                       // row width of the source
  const int c0 = key ? 0 : 128 * (part - 1), nc = key ? CI : 128;
  const __nv_bfloat16* x_new = key ? kI + (int64_t)b * CI : kv + (int64_t)b * C;
  const __nv_bfloat16* x_ring = key ? kI_tail + (int64_t)b * m * CI : kv_tail + (int64_t)b * m * C;
  {
    const int per = nc * 2 / 16;   // 16-byte pieces of a row's part
    for (int q = tid; q < m * per; q += blockDim.x) {
      const int i = q / per, c = q - i * per;
      const uint8_t* src = reinterpret_cast<const uint8_t*>(i == m - 1 ? x_new : x_ring + (int64_t)i * cc) + c0 * 2 +
                           c * 16;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(
                       ring_s + ((size_t)i * per + c) * 16)),
                   "l"(src)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  if (!key)
    for (int i = tid; i < (R >> 1); i += blockDim.x) {
      rope_s[0][i] = rcos[t * (R >> 1) + i];
      rope_s[1][i] = rsin[t * (R >> 1) + i];
    }
  if (warp == 0) {   // the logits: slots 0 .. m-2 from the ring, slot m-1 this token's; then the weights
    const float* zt = key ? zI_tail : z_tail;
    const float zn = key ? zI[b] : z[b];
    for (int i = lane; i < m; i += 32) z_s[i] = i == m - 1 ? zn : zt[(int64_t)b * m + i];
    __syncwarp();
    entry_weights(z_s, m, alpha_s, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  __syncthreads();
  // the pair sums, in token order (the fma sequence of compress_entry)
  const float* sc = key ? sI : s;
  if (tid < nc / 2) {
    const int pp = tid;   // pair (c0 / 2 + pp) of the row
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll 8
    for (int i = 0; i < m; ++i) {
      const float2 w2 = load_pair<true>(ring_s, (int64_t)i * nc, pp);
      acc.x = __fmaf_rn(alpha_s[i], w2.x, acc.x);
      acc.y = __fmaf_rn(alpha_s[i], w2.y, acc.y);
    }
    const int c = c0 + 2 * pp;   // channel of acc.x
    if (sc) {
      acc.x = __fmul_rn(acc.x, sc[c]);
      acc.y = __fmul_rn(acc.y, sc[c + 1]);
    }
    if (!key && c >= C - R) {   // RoPE at the block's last token t
      const int i = (c - (C - R)) >> 1;
      const float cs = rope_s[0][i], sn = rope_s[1][i];
      const float x0 = acc.x, x1 = acc.y;
      acc.x = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
      acc.y = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
    }
    acc_s[pp] = acc;
  }
  __syncthreads();
  if (key) {   // the MXFP4 key, by one warp: lane holds pair lane (C <= 64)
    if (warp == 0) {
      float2 v[kMaxPairs];
#pragma unroll
      for (int r = 0; r < kMaxPairs; ++r) v[r] = make_float2(0.0f, 0.0f);
      if (lane < nc / 2) v[0] = acc_s[lane];
      entry_finish<CSA_FMT_MXFP4>(v, nullptr, rope_s[0], rope_s[1], 0, CI, 0,
                                  kI_codes + ((int64_t)b * nmax + j) * (CI / 2),
                                  kI_scales + ((int64_t)b * nmax + j) * (CI / 32), lane);
    }
    return;
  }
  // the mixed row's part: FP8 codes of this quarter's group (quarter 4: channels
  // 384..447 only), its scale, and (quarter 4) the bf16 RoPE channels
  uint8_t* row = cache + ((int64_t)b * nmax + j) * kMixRow;
  const int g = part - 1;
  const int nfp8 = g < 3 ? 64 : 32;   // pairs of FP8 channels in this part
  if (warp < 2) {
    const int pp = tid;   // pairs 0 .. 63 over warps 0 and 1
    float a = 0.0f;
    if (pp < nfp8) {
      const float2 v = acc_s[pp];
      a = fmaxf(fabsf(v.x), fabsf(v.y));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) amax_s[warp] = a;
  }
  __syncthreads();
  const int e = fp8_group_exp(fmaxf(amax_s[0], amax_s[1]));
  if (tid < nfp8) {
    const float inv = pow2i(-e);
    const float2 v = acc_s[tid];
    const uint16_t c0v = e4m3_encode(__fmul_rn(v.x, inv));
    const uint16_t c1v = e4m3_encode(__fmul_rn(v.y, inv));
    *reinterpret_cast<uint16_t*>(row + c0 + 2 * tid) = (uint16_t)(c0v | (c1v << 8));
  } else if (g == 3 && tid < 64) {   // RoPE pairs: bf16
    const float2 v = acc_s[tid];
    const uint32_t b0 = f32_to_bf16_bits(v.x), b1 = f32_to_bf16_bits(v.y);
    *reinterpret_cast<uint32_t*>(row + kMixRopeOff + 4 * (tid - 32)) = b0 | (b1 << 16);
  }
  if (tid == 0) *reinterpret_cast<float*>(row + kMixScaleOff + 4 * g) = pow2i(e);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
pack_mixed_kernel(const float* __restrict__ v, int64_t n, uint8_t* __restrict__ out) {
  pdl_begin();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
  if (row >= n) return;
  float2 x[kMaxPairs];
  const float2* src = reinterpret_cast<const float2*>(v + row * kMixD);
#pragma unroll
  for (int r = 0; r < kMaxPairs; ++r) x[r] = src[lane + 32 * r];
  pack_mixed_row(x, lane, out + row * kMixRow);
}

cudaError_t launch_compress(const void* x, bool x_bf16, const float* z, bool z_per_channel, const float* s,
                            const float* rcos, const float* rsin, int64_t pos0, int B, int64_t T,
                            int C, int R, int m, int fmt, void* out, uint8_t* out_scales,
                            cudaStream_t st) {
  const int64_t N = T / m;
  const int64_t ents = (int64_t)B * N;
  if (ents == 0) return cudaSuccess;
  const dim3 grid((unsigned)((ents + kWarpsPerBlock - 1) / kWarpsPerBlock)), block(kWarpsPerBlock * 32);
#define CSA_CK(F, BF)                                                                                 \
  do {                                                                                                \
    if (z_per_channel)                                                                                \
      launch_pdl(compress_kernel<F, BF, true>, dim3(grid), dim3(block), 0, st, x, z, s, rcos, rsin, pos0, B, T, C, R, m, N, out, \
                                                           out_scales);                               \
    else                                                                                              \
      launch_pdl(compress_kernel<F, BF, false>, dim3(grid), dim3(block), 0, st, x, z, s, rcos, rsin, pos0, B, T, C, R, m, N, out, \
                                                            out_scales);                              \
  } while (0)
  if (fmt == CSA_FMT_F32) {
    if (x_bf16) CSA_CK(CSA_FMT_F32, true); else CSA_CK(CSA_FMT_F32, false);
  } else if (fmt == CSA_FMT_MIXED592) {
    if (x_bf16) CSA_CK(CSA_FMT_MIXED592, true); else CSA_CK(CSA_FMT_MIXED592, false);
  } else if (fmt == CSA_FMT_FP8B32) {
    if (x_bf16) CSA_CK(CSA_FMT_FP8B32, true); else CSA_CK(CSA_FMT_FP8B32, false);
  } else {
    if (x_bf16) CSA_CK(CSA_FMT_MXFP4, true); else CSA_CK(CSA_FMT_MXFP4, false);
  }
#undef CSA_CK
  return cudaGetLastError();
}

cudaError_t launch_decode_append(const void* kv, const float* z, const void* kI, const float* zI, const float* s,
                                 const float* sI, const float* rcos, const float* rsin, int64_t rope_rows,
                                 const int64_t* t_pos, int B,
                                 int C, int R, int CI, int m, void* kv_tail, float* z_tail, void* kI_tail,
                                 float* zI_tail, uint8_t* cache, int64_t nmax, uint8_t* kI_codes,
                                 uint8_t* kI_scales, uint8_t* swa, int64_t Ts, int W, int64_t* swa_pos0,
                                 cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const size_t ring = (size_t)m * 128 * 2;   // staged rows of a closing block: one part's channels
  launch_pdl(decode_append_kernel, dim3((unsigned)B, kAppendParts), dim3(kWarpsPerBlock * 32), ring, st, 
      reinterpret_cast<const __nv_bfloat16*>(kv), z, reinterpret_cast<const __nv_bfloat16*>(kI), zI, s, sI, rcos,
      rsin, rope_rows, t_pos, C, R, CI, m, reinterpret_cast<__nv_bfloat16*>(kv_tail), z_tail,
      reinterpret_cast<__nv_bfloat16*>(kI_tail), zI_tail, cache, nmax, kI_codes, kI_scales, swa, Ts, W, swa_pos0);
  return cudaGetLastError();
}

cudaError_t launch_pack_mixed(const float* v, int64_t n, uint8_t* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  launch_pdl(pack_mixed_kernel, dim3((unsigned)((n + kWarpsPerBlock - 1) / kWarpsPerBlock)), dim3(kWarpsPerBlock * 32), 0, st, v, n, out);
  return cudaGetLastError();
}

}  // namespace csa
