// indexer.cu -- lightning-indexer scores and top-k selection.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）": a light
// lightning indexer picks the top-k compressed entries for each query token;
// section "关键技术细节": the indexer's attention runs in FP4.
// "DeepSeek-V4 — MoE nyelvmodellek milliós kontextussal", CSA list item
// "Lightning Indexer" (k = 1024 in V4-Pro).
//
// score(t, j) = sum_h w_{t,h} relu(q_{t,h} . k_j) with the head sum as an fma
// chain from +0 in ascending h.  In the FP4 path q and k are MXFP4 (E2M1
// elements, power-of-two scales per 32-block): every E2M1 value times 2 is a
// small integer, so each 32-block dot is an exact integer (dp4a on int8) and
// the head dot is the exact sum of the two scaled block dots rounded once
// (both terms are exact fp32 values, so one IEEE add gives the nearest fp32
// of the exact sum).  The fp32 path runs the fma chain over the head dim.
//
// Selection: per query, radix select on order-preserving 32-bit keys of the
// scores (4 passes of 8 bits) finds the k-th largest value; every larger key
// is taken and ties at the threshold are taken in ascending index order; the
// chosen (score, index) pairs are then bitonic-sorted by score descending,
// index ascending.
#include "csa_common.cuh"
#include "launch.h"

namespace csa {

constexpr int kScoreThreads = 256;   // entries per CTA
constexpr int kScoreQT = 16;         // queries per CTA
constexpr int kMaxHI = 32;

__device__ __forceinline__ int64_t visible_entries(int64_t t, int m, int64_t N) {
  int64_t nv = (t + 1) / m;
  nv = nv < 0 ? 0 : nv;
  return nv < N ? nv : N;
}

// E2M1 code -> 2 * value as a signed int8 (exact)
__device__ __forceinline__ int e2m1_x2(uint32_t c) {
  const int mag = (c & 7) < 4 ? (int)(c & 7) : (c & 7) == 4 ? 4 : (c & 7) == 5 ? 6 : (c & 7) == 6 ? 8 : 12;
  return (c & 8) ? -mag : mag;
}

// d = P0 * 2^e0 + P1 * 2^e1, one rounding (the block dots are exact integers)
__device__ __forceinline__ float combine_blocks(int P0, int e0, int P1, int e1) {
  return __fadd_rn(scale_pow2((float)P0, e0), scale_pow2((float)P1, e1));
}

// The MXFP4 queries of a tile of nq rows (q0 ..) of sequence b into shared
// memory: per (query, head) 64 doubled E2M1 values as int8 (four per word),
// the two block exponents, and the head weights.  One (query, head, block)
// of 32 elements per thread and step.
__device__ __forceinline__ void quantise_query_tile(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                                                    int b, int64_t Tq, int64_t q0, int nq, int HI,
                                                    int32_t (*qv_s)[kMaxHI][16], int8_t (*qe_s)[kMaxHI][2],
                                                    float (*w_s)[kMaxHI]) {
  for (int u = threadIdx.x; u < nq * HI * 2; u += blockDim.x) {
    const int q = u / (HI * 2), h = (u / 2) % HI, blk = u & 1;
    const __nv_bfloat16* src = qI + (((b * Tq + q0 + q) * HI + h) * 64 + 32 * blk);
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = __bfloat162float(src[i]);
      amax = fmaxf(amax, fabsf(v[i]));
    }
    const int sx = mx_block_exp(amax);
    const float inv = pow2i(-sx);
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int val = e2m1_x2(e2m1_encode(__fmul_rn(v[4 * wd + e], inv)));
        word |= ((uint32_t)(val & 0xff)) << (8 * e);
      }
      qv_s[q][h][8 * blk + wd] = (int32_t)word;
    }
    qe_s[q][h][blk] = (int8_t)sx;
  }
  for (int u = threadIdx.x; u < nq * HI; u += blockDim.x) w_s[u / HI][u % HI] = w[(b * Tq + q0) * HI + u];
}

// ---------------------------------------------------------------------------
// FP4 scores: grid (entry chunks, query tiles, B); one thread per entry.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScoreThreads)
scores_fp4_kernel(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                  const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks,
                  const int64_t* __restrict__ q_pos, int64_t Tq, int HI, int64_t N, int m,
                  float* __restrict__ scores) {
  pdl_begin();
  // int8 (2 * E2M1) query values, 64 per head; block exponents; weights
  __shared__ __align__(16) int32_t qv_s[kScoreQT][kMaxHI][16];
  __shared__ int8_t qe_s[kScoreQT][kMaxHI][2];
  __shared__ float w_s[kScoreQT][kMaxHI];
  __shared__ int64_t nv_s[kScoreQT];
  const int b = blockIdx.z;
  const int64_t q0 = (int64_t)blockIdx.y * kScoreQT;
  const int nq = (int)(Tq - q0 < kScoreQT ? Tq - q0 : kScoreQT);
  const int64_t j0 = (int64_t)blockIdx.x * kScoreThreads;
  const int tid = threadIdx.x;

  if (tid < kScoreQT) nv_s[tid] = tid < nq ? visible_entries(q_pos[b * Tq + q0 + tid], m, N) : 0;
  __syncthreads();
  int64_t nv_max = 0;
  for (int q = 0; q < nq; ++q) nv_max = nv_max > nv_s[q] ? nv_max : nv_s[q];
  if (j0 >= nv_max) return;   // no query of the tile sees this chunk

  quantise_query_tile(qI, w, b, Tq, q0, nq, HI, qv_s, qe_s, w_s);
  __syncthreads();

  const int64_t j = j0 + tid;
  if (j >= nv_max) return;
  // the key: 64 E2M1 codes -> 16 words of 4 int8, and its two block exponents
  int32_t kv[16];
  const uint4* kc4 = reinterpret_cast<const uint4*>(kc + (b * N + j) * 32);
  const uint4 c_lo = kc4[0], c_hi = kc4[1];
  const uint32_t cw[8] = {c_lo.x, c_lo.y, c_lo.z, c_lo.w, c_hi.x, c_hi.y, c_hi.z, c_hi.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo |= ((uint32_t)(e2m1_x2((cw[i] >> (4 * e)) & 15) & 0xff)) << (8 * e);
      hi |= ((uint32_t)(e2m1_x2((cw[i] >> (16 + 4 * e)) & 15) & 0xff)) << (8 * e);
    }
    kv[2 * i] = (int32_t)lo;
    kv[2 * i + 1] = (int32_t)hi;
  }
  const int ke0 = (int)ks[(b * N + j) * 2] - 127, ke1 = (int)ks[(b * N + j) * 2 + 1] - 127;

  for (int q = 0; q < nq; ++q) {
    if (j >= nv_s[q]) continue;
    float s = 0.0f;
    for (int h = 0; h < HI; ++h) {
      const int4* qv4 = reinterpret_cast<const int4*>(qv_s[q][h]);
      int P0 = 0, P1 = 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int4 a = qv4[i];
        P0 = __dp4a(kv[4 * i + 0], a.x, P0);
        P0 = __dp4a(kv[4 * i + 1], a.y, P0);
        P0 = __dp4a(kv[4 * i + 2], a.z, P0);
        P0 = __dp4a(kv[4 * i + 3], a.w, P0);
      }
#pragma unroll
      for (int i = 2; i < 4; ++i) {
        const int4 a = qv4[i];
        P1 = __dp4a(kv[4 * i + 0], a.x, P1);
        P1 = __dp4a(kv[4 * i + 1], a.y, P1);
        P1 = __dp4a(kv[4 * i + 2], a.z, P1);
        P1 = __dp4a(kv[4 * i + 3], a.w, P1);
      }
      const float d = combine_blocks(P0, qe_s[q][h][0] + ke0 - 2, P1, qe_s[q][h][1] + ke1 - 2);
      const float r = d > 0.0f ? d : 0.0f;
      s = __fmaf_rn(w_s[q][h], r, s);
    }
    scores[(b * Tq + q0 + q) * N + j] = s;
  }
}

// ---------------------------------------------------------------------------
// FP4-query x FP8-key scores (keys: E4M3 codes with a power-of-two scale per
// 32 channels).  xmsumi.com DeepSeek-V4 article, section "算力与内存效率":
// an FP4 x FP8 product runs at the FP8 rate; zcldvi.com article: FP4 -> FP8
// dequantisation is lossless.
//
// Exact integer form: twice an E2M1 value is an integer in [-12, 12] and 512
// times an E4M3 value an integer below 2^18, so a 32-element block dot is an
// integer P with |P| <= 32 * 12 * 229376 < 2^27, worth P 2^(e_q + e_k - 10).
// The head's dot is the exact sum of its two blocks rounded once to fp32:
// both are put on one integer scale in 64 bits (when their exponents are more
// than 35 apart the smaller is folded in as a sticky bit, round to odd), then
// converted with one rounding.
// ---------------------------------------------------------------------------

// 512 x the value of an E4M3 code, as a signed integer (exact; NaN codes
// are never stored)
__device__ __forceinline__ int e4m3_x512(uint32_t c) {
  const int E = (int)((c >> 3) & 15u), M = (int)(c & 7u);
  const int mag = E == 0 ? M : (8 + M) << (E - 1);
  return (c & 0x80u) ? -mag : mag;
}

// RN(S 2^es) as fp32 with one rounding, subnormal results included.
__device__ __forceinline__ float ll_scaled_rn(long long S, int es) {
  if (S == 0) return 0.0f;
  const unsigned long long a = S < 0 ? 0ull - (unsigned long long)S : (unsigned long long)S;
  const int E = es + (63 - __clzll((long long)a));   // the value lies in [2^E, 2^(E+1))
  if (E >= -126) return scale_pow2(__ll2float_rn(S), es);   // rounded integer, scaled exactly
  // subnormal: nearest multiple of 2^-149, ties to even
  const int t = es + 149;
  long long q;
  if (t >= 0) {
    q = S << t;   // below 2^23 here
  } else if (-t >= 64) {
    q = 0;        // below half of 2^-149
  } else {
    const int sh = -t;
    q = S >> sh;
    const unsigned long long r = (unsigned long long)(S - (q << sh));
    const unsigned long long half = 1ull << (sh - 1);
    if (r > half || (r == half && (q & 1))) q += 1;
  }
  if (q == 0) return S < 0 ? -0.0f : 0.0f;
  return __fmul_rn(__fmul_rn((float)q, 0x1p-23f), 0x1p-126f);
}

// RN(P0 2^e0 + P1 2^e1) for integer block dots |P| < 2^27, one rounding.
__device__ __forceinline__ float fp8k_combine(int P0, int e0, int P1, int e1) {
  int Ph = P0, eh = e0, Pl = P1, el = e1;
  if (P0 == 0 || (P1 != 0 && e1 > e0)) {
    Ph = P1;
    eh = e1;
    Pl = P0;
    el = e0;
  }
  if (Ph == 0) return 0.0f;
  if (Pl == 0) return ll_scaled_rn(Ph, eh);
  const int d = eh - el;
  if (d <= 35) return ll_scaled_rn(((long long)Ph << d) + Pl, el);   // |sum| < 2^62: exact
  // Pl lies below bit 0 of Ph 2^35 (Ph != 0 has at least 36 bits there, so
  // the rounding position is bit 12 or higher): floor it onto that grid and
  // keep whether anything was dropped in bit 0 (round to odd) -- the odd
  // integer and the exact value round alike
  const int sh = d - 35;
  long long u;
  bool rem;
  if (sh >= 40) {
    u = Pl < 0 ? -1 : 0;
    rem = true;
  } else {
    u = (long long)Pl >> sh;
    rem = ((long long)Pl - (u << sh)) != 0;
  }
  long long S = ((long long)Ph << 35) + u;
  if (rem) S |= 1;
  return ll_scaled_rn(S, eh - 35);
}

__global__ void __launch_bounds__(kScoreThreads)
scores_fp8k_kernel(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                   const uint8_t* __restrict__ kc8, const uint8_t* __restrict__ ks8,
                   const int64_t* __restrict__ q_pos, int64_t Tq, int HI, int64_t N, int m,
                   float* __restrict__ scores) {
  pdl_begin();
  __shared__ __align__(16) int32_t qv_s[kScoreQT][kMaxHI][16];
  __shared__ int8_t qe_s[kScoreQT][kMaxHI][2];
  __shared__ float w_s[kScoreQT][kMaxHI];
  __shared__ int64_t nv_s[kScoreQT];
  const int b = blockIdx.z;
  const int64_t q0 = (int64_t)blockIdx.y * kScoreQT;
  const int nq = (int)(Tq - q0 < kScoreQT ? Tq - q0 : kScoreQT);
  const int64_t j0 = (int64_t)blockIdx.x * kScoreThreads;
  const int tid = threadIdx.x;
  if (tid < kScoreQT) nv_s[tid] = tid < nq ? visible_entries(q_pos[b * Tq + q0 + tid], m, N) : 0;
  __syncthreads();
  int64_t nv_max = 0;
  for (int q = 0; q < nq; ++q) nv_max = nv_max > nv_s[q] ? nv_max : nv_s[q];
  if (j0 >= nv_max) return;   // no query of the tile sees this chunk
  quantise_query_tile(qI, w, b, Tq, q0, nq, HI, qv_s, qe_s, w_s);
  __syncthreads();
  const int64_t j = j0 + tid;
  if (j >= nv_max) return;
  // the key: 64 E4M3 codes as integers (512 x value) and its two block exponents
  int kv[64];
  const uint4* src = reinterpret_cast<const uint4*>(kc8 + (b * N + j) * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 c = src[i];
    const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 16; ++e) kv[16 * i + e] = e4m3_x512((wd[e >> 2] >> (8 * (e & 3))) & 0xffu);
  }
  const int ke0 = (int)ks8[(b * N + j) * 2] - 127, ke1 = (int)ks8[(b * N + j) * 2 + 1] - 127;
  for (int q = 0; q < nq; ++q) {
    if (j >= nv_s[q]) continue;
    float s = 0.0f;
    for (int h = 0; h < HI; ++h) {
      const int4* qv4 = reinterpret_cast<const int4*>(qv_s[q][h]);
      int P[2] = {0, 0};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int4 a = qv4[i];
        const int aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qv = (aw[e >> 2] << (24 - 8 * (e & 3))) >> 24;   // signed byte e & 3
          P[i >> 1] += qv * kv[16 * i + e];
        }
      }
      const float d = fp8k_combine(P[0], qe_s[q][h][0] + ke0 - 10, P[1], qe_s[q][h][1] + ke1 - 10);
      s = __fmaf_rn(w_s[q][h], d > 0.0f ? d : 0.0f, s);
    }
    scores[(b * Tq + q0 + q) * N + j] = s;
  }
}

// ---------------------------------------------------------------------------
// FP4 scores for few query rows against long entry lists (decode): grid
// (entry chunks, rows), the chunk length chosen by the host so that the grid
// fills the resident CTA slots of the GPU about once; the row's query is
// quantised by all threads of the CTA (four elements each) while the first
// entries are in flight; each thread scores kDecKPT entries per round, their
// loads issued together.  Codes become doubled values by a byte-permute
// table; the even and odd elements of each 8-element group are dotted
// separately (an integer sum: same result).  The two block dots of a head
// meet as one integer when their scales are within 2^17 of each other, so the
// head's dot is one conversion (the single rounding) and one exact scaling.
// ---------------------------------------------------------------------------
constexpr int kDecKPT = 4;
constexpr int kDecRound = kScoreThreads * kDecKPT;   // entries per CTA round

// four E2M1 codes (one per byte, low nibble) -> their doubled values as int8x4
__device__ __forceinline__ uint32_t e2m1x2_int8x4(uint32_t b4) {
  const uint32_t mg = b4 & 0x07070707u;
  const uint32_t sel = (mg & 0x7u) | ((mg >> 4) & 0x70u) | ((mg >> 8) & 0x700u) | ((mg >> 12) & 0x7000u);
  const uint32_t mag = __byte_perm(0x03020100u, 0x0C080604u, sel);   // 0,1,2,3,4,6,8,12
  const uint32_t neg = ((b4 >> 3) & 0x01010101u) * 0xFFu;          // 0xFF in negative bytes
  return __vsub4(mag ^ neg, neg);
}

// RN(P0 2^e0 + P1 2^e1) for integer block dots |P| < 2^13: one integer when
// |e1 - e0| <= 17 (|sum| < 2^31) and the result stays normal, else the
// two-product form.  Both give the correctly rounded sum.
__device__ __forceinline__ float combine_blocks_fast(int P0, int e0, int P1, int dl) {
  const bool up = dl >= 0;
  const int sh = min(up ? dl : -dl, 17);
  const int S = up ? P0 + P1 * (1 << sh) : P1 + P0 * (1 << sh);
  const int base = up ? e0 : e0 + dl;
  if ((up ? dl : -dl) <= 17 && base >= -126 && base <= 96) return __fmul_rn((float)S, pow2i(base));
  return combine_blocks(P0, e0, P1, e0 + dl);
}

__global__ void __launch_bounds__(kScoreThreads, 3)
scores_fp4_decode_kernel(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                         const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks,
                         const int64_t* __restrict__ q_pos, int64_t Tq, int HI, int64_t N, int m,
                         int64_t chunk, float* __restrict__ scores) {
  pdl_begin();
  // doubled query values: head h, block b, group i (8 elements): word [h][b][0][i] even
  // elements, [h][b][1][i] odd elements of the group
  __shared__ __align__(16) int32_t qv_s[kMaxHI][2][2][4];
  // per head: {qe0 - 2, qe1 - qe0, w bits, 0}
  __shared__ __align__(16) int4 hx_s[kMaxHI];
  __shared__ int qe_s[kMaxHI][2];
  const int64_t row = blockIdx.y;
  const int64_t b = row / Tq;
  const int tid = threadIdx.x;
  const int64_t nv = visible_entries(q_pos[row], m, N);
  const int64_t c0 = (int64_t)blockIdx.x * chunk;
  if (c0 >= nv) return;
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  // the first round's entries, in flight during the query quantisation
  uint4 cw[kDecKPT][2];
  uint32_t se[kDecKPT];
#pragma unroll
  for (int i = 0; i < kDecKPT; ++i) {
    const int64_t j = c0 + tid + kScoreThreads * i;
    const int64_t jj = j < c1 ? j : c0;
    cw[i][0] = __ldg(reinterpret_cast<const uint4*>(kc + (b * N + jj) * 32));
    cw[i][1] = __ldg(reinterpret_cast<const uint4*>(kc + (b * N + jj) * 32) + 1);
    se[i] = __ldg(reinterpret_cast<const uint16_t*>(ks + (b * N + jj) * 2));
  }
  // quantise the query: thread t takes elements 4u .. 4u+3 (u = t mod 8) of blocks t / 8 + 32 r
  for (int blkid = tid >> 3; blkid < 2 * kMaxHI; blkid += kScoreThreads / 8) {
    const int u = tid & 7;
    const int h = blkid >> 1, blk = blkid & 1;
    const bool act = h < HI;
    float v[4];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = act ? __bfloat162float(qI[(row * HI + h) * 64 + 32 * blk + 4 * u + i]) : 0.0f;
      amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int sx = mx_block_exp(amax);
    const float inv = pow2i(-sx);
    if (act) {
      // element 4u + i is byte 2 (u & 1) + i / 2 of word [h][blk][i & 1][u / 2]
      int8_t* qb = reinterpret_cast<int8_t*>(&qv_s[h][blk][0][0]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qb[((i & 1) * 4 + (u >> 1)) * 4 + 2 * (u & 1) + (i >> 1)] =
            (int8_t)(e2m1_x2(e2m1_encode(__fmul_rn(v[i], inv))) & 0xff);
      if (u == 0) qe_s[h][blk] = sx;
    }
  }
  __syncthreads();
  if (tid < HI) hx_s[tid] = make_int4(qe_s[tid][0] - 2, qe_s[tid][1] - qe_s[tid][0], __float_as_int(w[row * HI + tid]), 0);
  __syncthreads();
  for (int64_t base = c0; base < c1; base += kDecRound) {
#pragma unroll
    for (int i = 0; i < kDecKPT; ++i) {
      const int64_t j = base + tid + kScoreThreads * i;
      if (base > c0) {   // this round's entries (the first round's were loaded above)
        const int64_t jj = j < c1 ? j : c0;
        cw[i][0] = __ldg(reinterpret_cast<const uint4*>(kc + (b * N + jj) * 32));
        cw[i][1] = __ldg(reinterpret_cast<const uint4*>(kc + (b * N + jj) * 32) + 1);
        se[i] = __ldg(reinterpret_cast<const uint16_t*>(ks + (b * N + jj) * 2));
      }
    }
#pragma unroll
    for (int i = 0; i < kDecKPT; ++i) {
      const int64_t j = base + tid + kScoreThreads * i;
      // entry words: block b = codes 32 b .. 32 b + 31 = words 4 b .. 4 b + 3 (8 codes each)
      const uint32_t wd[8] = {cw[i][0].x, cw[i][0].y, cw[i][0].z, cw[i][0].w,
                              cw[i][1].x, cw[i][1].y, cw[i][1].z, cw[i][1].w};
      int32_t kev[8], kod[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        kev[g] = (int32_t)e2m1x2_int8x4(wd[g] & 0x0F0F0F0Fu);
        kod[g] = (int32_t)e2m1x2_int8x4((wd[g] >> 4) & 0x0F0F0F0Fu);
      }
      const int ke0 = (int)(se[i] & 0xff) - 127, dk = (int)(se[i] >> 8) - 127 - ke0;
      float sc = 0.0f;
      for (int h = 0; h < HI; ++h) {
        const int4* q4 = reinterpret_cast<const int4*>(&qv_s[h][0][0][0]);
        const int4 q0e = q4[0], q0o = q4[1], q1e = q4[2], q1o = q4[3];
        const int4 hx = hx_s[h];
        int P0 = 0, P1 = 0;
        P0 = __dp4a(kev[0], q0e.x, P0); P0 = __dp4a(kod[0], q0o.x, P0);
        P0 = __dp4a(kev[1], q0e.y, P0); P0 = __dp4a(kod[1], q0o.y, P0);
        P0 = __dp4a(kev[2], q0e.z, P0); P0 = __dp4a(kod[2], q0o.z, P0);
        P0 = __dp4a(kev[3], q0e.w, P0); P0 = __dp4a(kod[3], q0o.w, P0);
        P1 = __dp4a(kev[4], q1e.x, P1); P1 = __dp4a(kod[4], q1o.x, P1);
        P1 = __dp4a(kev[5], q1e.y, P1); P1 = __dp4a(kod[5], q1o.y, P1);
        P1 = __dp4a(kev[6], q1e.z, P1); P1 = __dp4a(kod[6], q1o.z, P1);
        P1 = __dp4a(kev[7], q1e.w, P1); P1 = __dp4a(kod[7], q1o.w, P1);
        const float d = combine_blocks_fast(P0, hx.x + ke0, P1, hx.y + dk);
        sc = __fmaf_rn(__int_as_float(hx.z), d > 0.0f ? d : 0.0f, sc);
      }
      if (j < c1) scores[row * N + j] = sc;
    }
  }
}

// entries per decode-scoring CTA: a multiple of kScoreThreads, so that the
// grid (chunks x rows) is about one CTA per resident slot (at least 2 rounds)
int64_t decode_chunk(int64_t N, int64_t rows) {
  static PerDevice slots_dev;
  const int slots = slots_dev.get([] {
    return device_sms() * resident_ctas(reinterpret_cast<const void*>(scores_fp4_decode_kernel), kScoreThreads, 0);
  });
  int64_t per_row = slots / rows;
  if (per_row < 1) per_row = 1;
  int64_t c = (N + per_row - 1) / per_row;
  c = (c + kScoreThreads - 1) / kScoreThreads * kScoreThreads;
  return c < 2 * kDecRound ? 2 * kDecRound : c;
}

// ---------------------------------------------------------------------------
// fp32 scores (dI <= 64): fma chain over the head dim.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScoreThreads)
scores_f32_kernel(const float* __restrict__ qI, const float* __restrict__ w,
                  const float* __restrict__ kI, const int64_t* __restrict__ q_pos, int64_t Tq,
                  int HI, int dI, int64_t N, int m, float* __restrict__ scores) {
  pdl_begin();
  __shared__ float q_s[kScoreQT][512];   // HI * dI <= 512
  __shared__ float w_s[kScoreQT][kMaxHI];
  __shared__ int64_t nv_s[kScoreQT];
  const int b = blockIdx.z;
  const int64_t q0 = (int64_t)blockIdx.y * kScoreQT;
  const int nq = (int)(Tq - q0 < kScoreQT ? Tq - q0 : kScoreQT);
  const int64_t j0 = (int64_t)blockIdx.x * kScoreThreads;
  const int tid = threadIdx.x;
  if (tid < kScoreQT) nv_s[tid] = tid < nq ? visible_entries(q_pos[b * Tq + q0 + tid], m, N) : 0;
  for (int u = tid; u < nq * HI * dI; u += kScoreThreads)
    q_s[u / (HI * dI)][u % (HI * dI)] = qI[(b * Tq + q0) * HI * dI + u];
  for (int u = tid; u < nq * HI; u += kScoreThreads) w_s[u / HI][u % HI] = w[(b * Tq + q0) * HI + u];
  __syncthreads();
  const int64_t j = j0 + tid;
  float kv[64];
  const float* kr = kI + (b * N + (j < N - 1 ? j : N - 1)) * dI;
#pragma unroll
  for (int i = 0; i < 64; ++i) kv[i] = i < dI ? kr[i] : 0.0f;
  for (int q = 0; q < nq; ++q) {
    if (j >= nv_s[q]) continue;
    float s = 0.0f;
    for (int h = 0; h < HI; ++h) {
      float d = 0.0f;
#pragma unroll
      for (int i = 0; i < 64; ++i)
        if (i < dI) d = __fmaf_rn(q_s[q][h * dI + i], kv[i], d);
      const float r = d > 0.0f ? d : 0.0f;
      s = __fmaf_rn(w_s[q][h], r, s);
    }
    scores[(b * Tq + q0 + q) * N + j] = s;
  }
}

// ---------------------------------------------------------------------------
// top-k.  A row's candidates are visited in index order; the k-th largest
// order key is found by radix select (4 passes of 8 bits over shared-memory
// histograms); the chosen keys -- every key above that threshold and the first
// `remaining` keys equal to it, in index order -- are compacted in index order
// (per-warp segments: count, prefix, write); then sorted by (score desc, index
// asc) as 64-bit composite keys: warps sort runs of 32 with shuffles, runs are
// merged pairwise by binary search.  Rows longer than kTkChunk go in two
// stages: every chunk of C candidates (C ~ sqrt(N k), at least kTkChunk, so
// both stages get similar work) keeps its own top-k (the global
// top-k lies in their union: the order is total), then one CTA per row
// selects among the chunk winners.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;       // CTA of the two-stage kernels (few long rows)
constexpr int kTopkRowThreads = 128;     // CTA of the one-row kernel (many rows of at most kTkChunk)
constexpr int kTkChunk = 8192;
constexpr size_t kTkStageMax = 200 * 1024;   // dynamic shared memory for staged candidates

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;   // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_key_value(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

__device__ __forceinline__ unsigned long long composite(uint32_t key, uint32_t idx) {
  return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - idx);
}

template <int NT>
struct TkShared {
  unsigned int hist[256];
  unsigned int cnt_gt[NT / 32], cnt_eq[NT / 32];
  unsigned int prefix, remaining, equal;
};

// Candidate streams: get(i, key, idx) for i in [0, n), false when slot i holds
// no candidate.  Order keys of real scores are never 0.
struct DenseRow {   // scores[base + i], index base + i, for i < n
  const float* s;
  int64_t base;
  __device__ __forceinline__ bool get(int64_t i, uint32_t& key, uint32_t& idx) const {
    key = order_key(s[base + i]);
    idx = (uint32_t)(base + i);
    return true;
  }
};
struct CandList {   // composite keys, 0 = empty slot
  const unsigned long long* c;
  __device__ __forceinline__ bool get(int64_t i, uint32_t& key, uint32_t& idx) const {
    const unsigned long long v = c[i];
    key = (uint32_t)(v >> 32);
    idx = 0xffffffffu - (uint32_t)(v & 0xffffffffull);
    return key != 0u;
  }
};

struct SmemDense {   // staged scores: s[i] (shared memory), index base + i
  const float* s;
  int64_t base;
  __device__ __forceinline__ bool get(int64_t i, uint32_t& key, uint32_t& idx) const {
    key = order_key(s[i]);
    idx = (uint32_t)(base + i);
    return true;
  }
};

// Copies n elements of E bytes (4 or 8) from global src to shared dst, every
// copy in flight at once (asynchronous copies), then waits and syncs the CTA.
template <int NT, int E>
__device__ __forceinline__ void stage_to_smem(void* dst, const void* src, int64_t n) {
  const uint32_t d0 = (uint32_t)__cvta_generic_to_shared(dst);
  for (int64_t i = threadIdx.x; i < n; i += NT) {
    const char* g = reinterpret_cast<const char*>(src) + i * E;
    if (E == 8)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d0 + (uint32_t)(i * E)), "l"(g) : "memory");
    else
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d0 + (uint32_t)(i * E)), "l"(g) : "memory");
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  __syncthreads();
}

// The kk-th largest key of the stream (kk >= 1 and at most the number of
// candidates): returns its value; sh.remaining = how many keys equal to it
// are taken, sh.equal = how many there are.  Keys known to share their top
// 8 (32 - first_shift) bits `top` start the search at first_shift.
template <int NT, class Src>
__device__ uint32_t radix_threshold(const Src& src, int64_t n, int kk, TkShared<NT>& sh, int first_shift = 24,
                                   uint32_t top = 0) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sh.prefix = top;
    sh.remaining = (unsigned)kk;
  }
  uint32_t mask = first_shift == 24 ? 0u : ~0u << (first_shift + 8);
  for (int shift = first_shift; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sh.prefix;
    for (int64_t i = tid; i < n; i += NT) {
      uint32_t u, id;
      if (src.get(i, u, id) && (u & mask) == prefix) atomicAdd(&sh.hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane L holds bins 255-8L .. 248-8L (descending); find the digit where
      // the count of larger keys first reaches `remaining`
      const unsigned int rem = sh.remaining;
      unsigned int c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = sh.hist[255 - 8 * lane - i];
        tot += c[i];
      }
      unsigned int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned int excl = incl - tot;
      const bool here = excl < rem && incl >= rem;
      const unsigned int who = __ballot_sync(0xffffffffu, here);
      if (lane == __ffs(who) - 1) {
        unsigned int acc = excl, eqc = 0;
        int d = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + c[i] >= rem) {
            d = 255 - 8 * lane - i;
            eqc = c[i];
            break;
          }
          acc += c[i];
        }
        sh.remaining = rem - acc;
        sh.equal = eqc;
        sh.prefix = prefix | ((uint32_t)d << shift);
      }
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  return sh.prefix;
}

// Writes the chosen candidates (key > thr, and the first need_eq keys == thr in
// stream order) to dst[0..) in stream order as composite keys.  Warp w scans
// slots [w seg, (w + 1) seg).
template <int NT, class Src>
__device__ void ordered_collect(const Src& src, int64_t n, uint32_t thr, unsigned int need_eq,
                                unsigned long long* dst, TkShared<NT>& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t seg = ((n + (NT / 32) - 1) / (NT / 32) + 31) & ~int64_t(31);
  const int64_t lo = warp * seg, hi = lo + seg < n ? lo + seg : n;
  unsigned int ngt = 0, neq = 0;
  for (int64_t b = lo; b < hi; b += 32) {
    const int64_t i = b + lane;
    uint32_t u = 0, id = 0;
    const bool ok = i < hi && src.get(i, u, id);
    ngt += __popc(__ballot_sync(0xffffffffu, ok && u > thr));
    neq += __popc(__ballot_sync(0xffffffffu, ok && u == thr));
  }
  if (lane == 0) {
    sh.cnt_gt[warp] = ngt;
    sh.cnt_eq[warp] = neq;
  }
  __syncthreads();
  unsigned int eq_before = 0, out = 0;
  for (int w2 = 0; w2 < warp; ++w2) {
    const unsigned int e = sh.cnt_eq[w2];
    const unsigned int te = eq_before >= need_eq ? 0u : (need_eq - eq_before < e ? need_eq - eq_before : e);
    out += sh.cnt_gt[w2] + te;
    eq_before += e;
  }
  unsigned int eq_seen = eq_before;   // equal keys before this warp's current chunk
  const unsigned int lt = (1u << lane) - 1u;
  for (int64_t b = lo; b < hi; b += 32) {
    const int64_t i = b + lane;
    uint32_t u = 0, id = 0;
    const bool ok = i < hi && src.get(i, u, id);
    const bool gt = ok && u > thr, eq = ok && u == thr;
    const unsigned int beq = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_seen + __popc(beq & lt) < need_eq);
    const unsigned int bt = __ballot_sync(0xffffffffu, take);
    if (take) dst[out + __popc(bt & lt)] = composite(u, id);
    out += __popc(bt);
    eq_seen += __popc(beq);
  }
  __syncthreads();
}

// Sorts buf[0..P) descending (P a power of two >= 32, slots past `count` are
// padded with distinct keys below every real one); buf has 2 P slots.
// Returns the buffer that holds the result.
template <int NT>
__device__ unsigned long long* merge_sort_desc(unsigned long long* buf, int count, int P) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long* b0 = buf;
  unsigned long long* b1 = buf + P;
  for (int i = tid; i < P; i += NT)
    if (i >= count) b0[i] = (unsigned long long)(P - i);
  __syncthreads();
  for (int r = warp; r < P / 32; r += (NT / 32)) {
    unsigned long long v = b0[r * 32 + lane];
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, stride);
        const bool desc = size == 32 || (lane & size) == 0, lower = (lane & stride) == 0;
        v = (desc == lower) ? (v > o ? v : o) : (v < o ? v : o);
      }
    }
    b0[r * 32 + lane] = v;
  }
  __syncthreads();
  for (int L = 32; L < P; L <<= 1) {
    for (int i = tid; i < P; i += NT) {
      const unsigned long long x = b0[i];
      const int r = i / L, pos = i - r * L;
      const unsigned long long* part = b0 + (r ^ 1) * L;
      int c = 0;   // keys of the partner run larger than x (a prefix: runs are descending)
      for (int st = L; st > 0; st >>= 1)
        if (c + st <= L && part[c + st - 1] > x) c += st;
      b1[(r & ~1) * L + pos + c] = x;
    }
    __syncthreads();
    unsigned long long* t = b0;
    b0 = b1;
    b1 = t;
  }
  return b0;
}

template <int NT>
__device__ __forceinline__ void emit_topk(const unsigned long long* sorted, int kk, int k, int64_t row,
                                          int32_t* idx_out, float* score_out) {
  for (int r = threadIdx.x; r < k; r += NT) {
    int32_t j = -1;
    float sc = -INFINITY;
    if (r < kk) {
      const unsigned long long key = sorted[r];
      j = (int32_t)(0xffffffffu - (uint32_t)(key & 0xffffffffull));
      sc = order_key_value((uint32_t)(key >> 32));
    }
    idx_out[row * k + r] = j;
    if (score_out) score_out[row * k + r] = sc;
  }
}

// One CTA per query row over its visible scores (rows of any length).
__global__ void __launch_bounds__(kTopkRowThreads)
topk_kernel(const float* __restrict__ scores, const int64_t* __restrict__ q_pos, int64_t N, int m, int k, int P,
            int32_t* __restrict__ idx_out, float* __restrict__ score_out) {
  pdl_begin();
  constexpr int NT = kTopkRowThreads;
  extern __shared__ unsigned long long keys_s[];   // 2 P composite keys
  __shared__ TkShared<NT> sh;
  const int64_t row = blockIdx.x;
  const int64_t nv = visible_entries(q_pos[row], m, N);
  const int kk = (int)((int64_t)k < nv ? (int64_t)k : nv);
  const DenseRow src{scores + row * N, 0};
  if (kk > 0) {
    // every visible key taken: no selection (real order keys are never 0)
    const uint32_t thr = kk == nv ? 0u : radix_threshold<NT>(src, nv, kk, sh);
    ordered_collect<NT>(src, nv, thr, kk == nv ? 0u : sh.remaining, keys_s, sh);
  }
  const unsigned long long* sorted = merge_sort_desc<NT>(keys_s, kk, P);
  emit_topk<NT>(sorted, kk, k, row, idx_out, score_out);
}

// Stage 1 of long rows: grid (rows, chunks); chunk c keeps the top-k of its
// visible candidates [c C, (c + 1) C) in index order, at cand[(row chunks + c) k].
// With stage set, the chunk's scores are first copied to shared memory (C
// floats of dynamic shared memory) and every pass reads them there.
__global__ void __launch_bounds__(kTopkThreads)
topk_stage1_kernel(const float* __restrict__ scores, const int64_t* __restrict__ q_pos, int64_t N, int m, int k,
                   int chunks, int64_t C, bool stage, unsigned long long* __restrict__ cand) {
  pdl_begin();
  constexpr int NT = kTopkThreads;
  extern __shared__ __align__(16) float chunk_s[];
  __shared__ TkShared<NT> sh;
  const int64_t row = blockIdx.x;
  const int c = blockIdx.y;
  const int64_t nv = visible_entries(q_pos[row], m, N);
  const int64_t c0 = (int64_t)c * C;
  const int64_t n = nv - c0 < 0 ? 0 : (nv - c0 < C ? nv - c0 : C);
  const int kk = (int)((int64_t)k < n ? (int64_t)k : n);
  unsigned long long* dst = cand + ((int64_t)row * chunks + c) * k;
  if (kk > 0) {
    if (stage) {
      stage_to_smem<NT, 4>(chunk_s, scores + row * N + c0, n);
      const SmemDense src{chunk_s, c0};
      const uint32_t thr = kk == n ? 0u : radix_threshold<NT>(src, n, kk, sh);
      ordered_collect<NT>(src, n, thr, kk == n ? 0u : sh.remaining, dst, sh);
    } else {
      const DenseRow src{scores + row * N, c0};
      const uint32_t thr = kk == n ? 0u : radix_threshold<NT>(src, n, kk, sh);
      ordered_collect<NT>(src, n, thr, kk == n ? 0u : sh.remaining, dst, sh);
    }
  }
  for (int i = kk + threadIdx.x; i < k; i += NT) dst[i] = 0ull;   // empty slots
}

// Stage 2: one CTA per row selects among its chunks' winners (in index order).
__global__ void __launch_bounds__(kTopkThreads)
topk_stage2_kernel(const int64_t* __restrict__ q_pos, int64_t N, int m, int k, int chunks, int P, bool stage,
                   const unsigned long long* __restrict__ cand, int32_t* __restrict__ idx_out,
                   float* __restrict__ score_out) {
  pdl_begin();
  constexpr int NT = kTopkThreads;
  // 2 P composite keys, then (stage) the row's chunks x k candidates
  extern __shared__ __align__(16) unsigned long long keys_s[];
  __shared__ TkShared<NT> sh;
  const int64_t row = blockIdx.x;
  const int64_t nv = visible_entries(q_pos[row], m, N);
  const int kk = (int)((int64_t)k < nv ? (int64_t)k : nv);
  const int64_t n = (int64_t)chunks * k;
  if (stage) stage_to_smem<NT, 8>(keys_s + 2 * P, cand + (int64_t)row * n, n);
  const CandList src{stage ? keys_s + 2 * P : cand + (int64_t)row * n};
  if (kk > 0) {
    // kk == nv: every chunk kept all its visible candidates, all are taken
    const uint32_t thr = kk == nv ? 0u : radix_threshold<NT>(src, n, kk, sh);
    ordered_collect<NT>(src, n, thr, kk == nv ? 0u : sh.remaining, keys_s, sh);
  }
  const unsigned long long* sorted = merge_sort_desc<NT>(keys_s, kk, P);
  emit_topk<NT>(sorted, kk, k, row, idx_out, score_out);
}

// ---------------------------------------------------------------------------
// Top-k of few long rows from a score histogram (decode).  The tensor-core
// decode scorer counts every visible score of a row into kHistBins bins by
// the top kHistBits bits of its order key.  From that histogram every CTA
// of the row finds the bin b* that holds the k-th largest key: every score
// in a bin above b* is among the top k ("sure": fewer than k of them) and
// the rest of the top k are the best of bin b* ("ties").  Chunk CTAs append
// the row's sure and tie candidates, as 64-bit composite keys, to workspace
// lists (warp-aggregated); the last chunk CTA of the row to finish selects
// the needed ties exactly (radix threshold on the order key, equal keys by
// ascending index), sorts the k winners (score descending, index ascending)
// and writes them.  When bin b* holds more than kTieCap candidates the last
// CTA selects over the row's whole score array instead (same result).
// ---------------------------------------------------------------------------
constexpr int kHistBits = 11;
constexpr int kHistBins = 1 << kHistBits;
constexpr int kTieCap = 8192;
constexpr int kSelThreads = 1024;
constexpr int kSelChunk = 8192;       // scores scanned per chunk CTA (8 per thread)

// Candidate stream over staged composite keys whose order key equals `thr`:
// their low words (the complement of the index) as the key, so the largest
// of them are the lowest indices.
struct EqualKeyList {
  const unsigned long long* c;
  uint32_t thr;
  __device__ __forceinline__ bool get(int64_t i, uint32_t& key, uint32_t& idx) const {
    const unsigned long long v = c[i];
    key = (uint32_t)(v & 0xffffffffull);
    idx = 0xffffffffu - key;
    return (uint32_t)(v >> 32) == thr;
  }
};

constexpr int kSelPerThread = kSelChunk / kSelThreads;

// The need-th largest order key among composite keys c[0..n) that all share
// their top kHistBits bits `top` (the bin b*): two passes of 11 and 10 bits,
// histograms of up to 2048 bins (the ties differ only below the bin, so
// 8-bit digits would crowd few bins).  sh.remaining = how many keys equal to
// it are taken, sh.equal = how many there are.
template <int NT>
__device__ uint32_t tie_threshold(const unsigned long long* c, int n, int need, uint32_t top, unsigned int* hist,
                                  unsigned int* warp_sum, TkShared<NT>& sh) {
  static_assert(kHistBits == 11 && NT >= 1024, "two passes of 11 and 10 bits, two bins per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = top << 21, mask = 0xffe00000u;
  unsigned int rem = (unsigned)need;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0, nb = pass == 0 ? 2048 : 1024;
    for (int i = tid; i < nb; i += NT) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      const uint32_t key = (uint32_t)(c[i] >> 32);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
    }
    __syncthreads();
    // thread t owns bins nb-1-2t and nb-2-2t (descending)
    unsigned int h0 = 0, h1 = 0;
    if (2 * tid < nb) {
      h0 = hist[nb - 1 - 2 * tid];
      h1 = hist[nb - 2 - 2 * tid];
    }
    const unsigned int own = h0 + h1;
    unsigned int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    unsigned int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += warp_sum[w2];
    const unsigned int excl = before + incl - own;
    if (2 * tid < nb) {
      if (excl < rem && excl + h0 >= rem) {
        sh.prefix = prefix | ((uint32_t)(nb - 1 - 2 * tid) << shift);
        sh.remaining = rem - excl;
        sh.equal = h0;
      } else if (excl + h0 < rem && excl + own >= rem) {
        sh.prefix = prefix | ((uint32_t)(nb - 2 - 2 * tid) << shift);
        sh.remaining = rem - excl - h0;
        sh.equal = h1;
      }
    }
    __syncthreads();
    prefix = sh.prefix;
    rem = sh.remaining;
    mask |= (uint32_t)(nb - 1) << shift;
  }
  return prefix;
}

__global__ void __launch_bounds__(kSelThreads)
topk_hist_select_kernel(const float* __restrict__ scores, const unsigned int* __restrict__ hist,
                        const int64_t* __restrict__ q_pos, int64_t N, int m, int k, int nchunk, int P,
                        unsigned long long* __restrict__ cand, int* __restrict__ ctr, int32_t* __restrict__ idx_out,
                        float* __restrict__ score_out) {
  pdl_begin();
  constexpr int NT = kSelThreads;
  // chunk phase: this CTA's sure keys [P] and ties [kTieCap]; final phase:
  // 2 P sort keys, then the row's staged ties
  extern __shared__ __align__(16) unsigned long long dyn_s[];
  __shared__ unsigned int warp_sum[NT / 32];
  __shared__ unsigned int hist2_s[2048];
  __shared__ int bstar_s, last_s, base_s, base_t;
  __shared__ unsigned int nls_s, nlt_s, take_s;
  __shared__ TkShared<NT> sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;
  const int c = blockIdx.x;
  const int64_t nv = visible_entries(q_pos[row], m, N);
  const int kk = (int)((int64_t)k < nv ? (int64_t)k : nv);
  unsigned long long* sure = cand + row * (int64_t)(P + kTieCap);
  unsigned long long* tie = sure + P;
  int* rc = ctr + row * 4;   // [0] sure appended, [1] ties appended, [2] chunk CTAs done
  // this chunk's scores, loaded while the histogram is read
  const int64_t j0 = (int64_t)c * kSelChunk, j1 = j0 + kSelChunk < nv ? j0 + kSelChunk : nv;
  float sv[kSelPerThread];
#pragma unroll
  for (int r = 0; r < kSelPerThread; ++r) {
    const int64_t j = j0 + r * NT + tid;
    sv[r] = j < j1 ? scores[row * N + j] : 0.0f;
  }

  // ---- b*: the largest bin whose suffix count (bins >= it) reaches kk ----
  {
    const unsigned int* hr = hist + row * (int64_t)kHistBins;
    // thread t owns bins kHistBins-1-2t and kHistBins-2-2t (descending order)
    const unsigned int h0 = hr[kHistBins - 1 - 2 * tid], h1 = hr[kHistBins - 2 - 2 * tid];
    const unsigned int own = h0 + h1;
    unsigned int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    if (tid == 0) {
      bstar_s = -1;
      nls_s = 0;
      nlt_s = 0;
    }
    __syncthreads();
    unsigned int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += warp_sum[w2];
    const unsigned int excl = before + incl - own;   // keys in bins above this thread's two
    if (kk > 0 && kk < nv) {
      if (excl < (unsigned)kk && excl + h0 >= (unsigned)kk) {
        bstar_s = kHistBins - 1 - 2 * tid;
      } else if (excl + h0 < (unsigned)kk && excl + own >= (unsigned)kk) {
        bstar_s = kHistBins - 2 - 2 * tid;
      }
    }
    __syncthreads();
  }
  const int bstar = bstar_s;   // -1: every visible key is taken
  // ---- this chunk's candidates: into shared lists, then one reservation per list ----
  unsigned long long* sure_l = dyn_s;
  unsigned long long* tie_l = dyn_s + P;
#pragma unroll
  for (int r = 0; r < kSelPerThread; ++r) {
    const int64_t j = j0 + r * NT + tid;
    if (j < j1) {
      const uint32_t key = order_key(sv[r]);
      const int bin = (int)(key >> (32 - kHistBits));
      if (bin > bstar) {
        const unsigned int pos = atomicAdd(&nls_s, 1u);
        if (pos < (unsigned)P) sure_l[pos] = composite(key, (uint32_t)j);
      } else if (bin == bstar) {
        const unsigned int pos = atomicAdd(&nlt_s, 1u);
        if (pos < (unsigned)kTieCap) tie_l[pos] = composite(key, (uint32_t)j);
      }
    }
  }
  __syncthreads();
  const int nls = min((int)nls_s, P), nlt_all = (int)nlt_s, nlt = min(nlt_all, kTieCap);
  if (tid == 0) {
    base_s = nls ? atomicAdd(rc + 0, nls) : 0;
    base_t = nlt_all ? atomicAdd(rc + 1, nlt_all) : 0;
  }
  __syncthreads();
  for (int i = tid; i < nls; i += NT)
    if (base_s + i < P) sure[base_s + i] = sure_l[i];
  for (int i = tid; i < nlt; i += NT)
    if (base_t + i < kTieCap) tie[base_t + i] = tie_l[i];
  __threadfence();
  __syncthreads();
  if (tid == 0) last_s = atomicAdd(rc + 2, 1) == nchunk - 1;
  __syncthreads();
  if (!last_s) return;
  // ================= the row's last chunk CTA: select and sort =================
  __threadfence();
  const int nsure = min(*reinterpret_cast<volatile int*>(rc + 0), P);
  const int ntie = *reinterpret_cast<volatile int*>(rc + 1);
  unsigned long long* keys_s = dyn_s;          // 2 P
  unsigned long long* tie_s = dyn_s + 2 * P;   // kTieCap
  if (kk > 0) {
    if (bstar >= 0 && ntie > kTieCap) {
      // bin b* too full for the tie list: select over the whole row
      const DenseRow src{scores + row * N, 0};
      const uint32_t thr = radix_threshold<NT>(src, nv, kk, sh);
      ordered_collect<NT>(src, nv, thr, sh.remaining, keys_s, sh);
    } else {
      // the row's sure and tie keys into shared memory, every load in flight together
      {
        unsigned long long t[kTieCap / NT];
#pragma unroll
        for (int r = 0; r < kTieCap / NT; ++r) {
          const int i = tid + r * NT;
          t[r] = i < ntie ? __ldcg(tie + i) : 0ull;
        }
        for (int i = tid; i < nsure; i += NT) keys_s[i] = __ldcg(sure + i);
#pragma unroll
        for (int r = 0; r < kTieCap / NT; ++r) {
          const int i = tid + r * NT;
          if (i < ntie) tie_s[i] = t[r];
        }
      }
      const int need = kk - nsure;   // ties to take (0 when every key is taken)
      if (need > 0) {
        if (tid == 0) take_s = nsure;
        __syncthreads();
        const uint32_t thr = tie_threshold<NT>(tie_s, ntie, need, (uint32_t)bstar, hist2_s, warp_sum, sh);
        // keys equal to thr to take, lowest indices first; when all of them
        // are taken no index threshold is needed
        const unsigned int rem = sh.remaining, neq = sh.equal;
        uint32_t ithr = 0;
        if (rem < neq) {
          __syncthreads();
          ithr = radix_threshold<NT>(EqualKeyList{tie_s, thr}, ntie, (int)rem, sh);
        }
        // the chosen ties appended after the sure keys, one reservation per warp
        for (int i0 = 0; i0 < ntie; i0 += NT) {
          const int i = i0 + tid;
          unsigned long long v = 0;
          bool take = false;
          if (i < ntie) {
            v = tie_s[i];
            const uint32_t key = (uint32_t)(v >> 32), low = (uint32_t)(v & 0xffffffffull);
            take = key > thr || (key == thr && low >= ithr);
          }
          const unsigned int bt = __ballot_sync(0xffffffffu, take);
          unsigned int base = 0;
          if (lane == 0 && bt) base = atomicAdd(&take_s, (unsigned)__popc(bt));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (take) keys_s[base + __popc(bt & ((1u << lane) - 1u))] = v;
        }
      }
      __syncthreads();
    }
  }
  emit_topk<NT>(merge_sort_desc<NT>(keys_s, kk, P), kk, k, row, idx_out, score_out);
  if (tid == 0) {   // the workspace counters for the next call
    rc[0] = 0;
    rc[1] = 0;
    rc[2] = 0;
  }
}

int topk_pad(int k) {
  int p = 32;
  while (p < k) p <<= 1;
  return p;
}

// candidates per stage-1 chunk: a power of two near sqrt(N k), at least kTkChunk
int64_t topk_chunk_size(int64_t N, int k) {
  int64_t c = kTkChunk;
  while (c * c < N * (int64_t)k && c < N) c <<= 1;
  return c;
}
int topk_chunks(int64_t N, int k) {
  if (N <= kTkChunk) return 0;
  const int64_t c = topk_chunk_size(N, k);
  return (int)((N + c - 1) / c);
}

// scratch of the histogram path: [rows][kHistBins] counts, [rows][4] counters,
// [rows][P + kTieCap] candidate keys
size_t topk_hist_bytes(int64_t rows, int k) {
  const size_t P = (size_t)topk_pad(k);
  return ((size_t)rows * kHistBins * 4 + (size_t)rows * 16 + 255) / 256 * 256 + (size_t)rows * (P + kTieCap) * 8;
}

size_t topk_cand_bytes(int B, int64_t Tq, int64_t N, int k) {
  const int ch = topk_chunks(N, k);
  const size_t two = ch ? (size_t)B * (size_t)Tq * (size_t)ch * (size_t)k * 8 : 0;
  const size_t hh = topk_hist_bytes((int64_t)B * Tq, k);
  return ch ? (two > hh ? two : hh) : 0;
}

bool topk_two_stage(int B, int64_t Tq, int64_t N) {
  return N > kTkChunk && (int64_t)B * Tq < 4 * 148;
}

cudaError_t launch_indexer_topk(const void* qI, int key_fmt, const float* w, const void* kI,
                                const uint8_t* kI_scales, const int64_t* q_pos, int B, int64_t Tq,
                                int HI, int dI, int64_t N, int m, int k, int32_t* idx_out,
                                float* score_out, float* scores_ws, void* tc_ws, void* cand_ws, void* flags_ws,
                                bool tensor_cores, cudaStream_t st) {
  if ((int64_t)B * Tq == 0) return cudaSuccess;
  const bool fp4 = key_fmt == CSA_FMT_MXFP4;
  unsigned int* hist = nullptr;   // set when the scorer also counts the scores into bins
  if (N > 0) {
    cudaError_t e;
    if (key_fmt == CSA_FMT_FP8B32) {
      const dim3 grid((unsigned)((N + kScoreThreads - 1) / kScoreThreads),
                      (unsigned)((Tq + kScoreQT - 1) / kScoreQT), (unsigned)B);
      launch_pdl(scores_fp8k_kernel, dim3(grid), dim3(kScoreThreads), 0, st, reinterpret_cast<const __nv_bfloat16*>(qI), w,
                                                         reinterpret_cast<const uint8_t*>(kI), kI_scales, q_pos, Tq,
                                                         HI, N, m, scores_ws);
      e = cudaGetLastError();
    } else if (fp4 && tc_ws && indexer_tc_applies(B, Tq, HI, dI, N)) {
      e = launch_indexer_scores_tc(qI, w, reinterpret_cast<const uint8_t*>(kI), kI_scales, q_pos, B, Tq, HI, N,
                                   m, scores_ws, tc_ws, flags_ws, st);
    } else if (fp4 && tensor_cores && decode_tc_applies(Tq, HI, dI, N)) {
      // with the two-stage scratch given: the scores' histogram for the top-k
      if (cand_ws && topk_two_stage(B, Tq, N)) {
        hist = reinterpret_cast<unsigned int*>(cand_ws);
        e = cudaMemsetAsync(cand_ws, 0, (size_t)B * Tq * (kHistBins * 4 + 16), st);
        if (e != cudaSuccess) return e;
      }
      e = launch_scores_fp4_decode_tc(qI, w, reinterpret_cast<const uint8_t*>(kI), kI_scales, q_pos, B, Tq, HI, N,
                                      m, scores_ws, hist, flags_ws, st);
    } else if (fp4 && dI == 64 && Tq <= 4 && HI <= kMaxHI && N >= 8 * kDecRound) {
      const int64_t chunk = decode_chunk(N, (int64_t)B * Tq);
      const dim3 grid((unsigned)((N + chunk - 1) / chunk), (unsigned)(B * Tq));
      launch_pdl(scores_fp4_decode_kernel, dim3(grid), dim3(kScoreThreads), 0, st, reinterpret_cast<const __nv_bfloat16*>(qI), w,
                                                               reinterpret_cast<const uint8_t*>(kI), kI_scales,
                                                               q_pos, Tq, HI, N, m, chunk, scores_ws);
      e = cudaGetLastError();
    } else {
      const dim3 grid((unsigned)((N + kScoreThreads - 1) / kScoreThreads),
                      (unsigned)((Tq + kScoreQT - 1) / kScoreQT), (unsigned)B);
      if (fp4)
        launch_pdl(scores_fp4_kernel, dim3(grid), dim3(kScoreThreads), 0, st, 
            reinterpret_cast<const __nv_bfloat16*>(qI), w, reinterpret_cast<const uint8_t*>(kI),
            kI_scales, q_pos, Tq, HI, N, m, scores_ws);
      else
        launch_pdl(scores_f32_kernel, dim3(grid), dim3(kScoreThreads), 0, st, reinterpret_cast<const float*>(qI), w,
                                                          reinterpret_cast<const float*>(kI), q_pos,
                                                          Tq, HI, dI, N, m, scores_ws);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  const int P = topk_pad(k);
  const size_t smem = sizeof(unsigned long long) * 2 * (size_t)P;
  static PerDevice attr_row, attr_s1, attr_s2;
  smem_limit_once(attr_row, reinterpret_cast<const void*>(topk_kernel), 64 * 1024);
  smem_limit_once(attr_s1, reinterpret_cast<const void*>(topk_stage1_kernel), (int)kTkStageMax);
  smem_limit_once(attr_s2, reinterpret_cast<const void*>(topk_stage2_kernel), (int)kTkStageMax);
  const int64_t rows = (int64_t)B * Tq;
  if (hist) {
    static PerDevice attr_h;
    const size_t hsmem = sizeof(unsigned long long) * (2 * (size_t)P + kTieCap);
    // the largest request (k = 4096), set once per device
    smem_limit_once(attr_h, reinterpret_cast<const void*>(topk_hist_select_kernel),
                    (int)(sizeof(unsigned long long) * (2 * 4096 + kTieCap)));
    const size_t hoff = ((size_t)rows * kHistBins * 4 + (size_t)rows * 16 + 255) / 256 * 256;
    int* ctr = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(cand_ws) + (size_t)rows * kHistBins * 4);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(cand_ws) + hoff);
    const int nchunk = (int)((N + kSelChunk - 1) / kSelChunk);
    launch_pdl(topk_hist_select_kernel, dim3((unsigned)nchunk, (unsigned)rows), dim3(kSelThreads), hsmem, st,
               (const float*)scores_ws, (const unsigned int*)hist, q_pos, N, m, k, nchunk, P, cand, ctr, idx_out,
               score_out);
  } else if (cand_ws && topk_two_stage(B, Tq, N)) {
    const int ch = topk_chunks(N, k);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(cand_ws);
    // stage a chunk's scores / a row's candidates in shared memory when they fit
    const int64_t C = topk_chunk_size(N, k);
    const bool st1 = (size_t)C * 4 <= kTkStageMax, st2 = smem + (size_t)ch * k * 8 <= kTkStageMax;
    launch_pdl(topk_stage1_kernel, dim3(dim3((unsigned)rows, (unsigned)ch)), dim3(kTopkThreads), st1 ? (size_t)C * 4 : 0, st, 
        scores_ws, q_pos, N, m, k, ch, C, st1, cand);
    launch_pdl(topk_stage2_kernel, dim3((unsigned)rows), dim3(kTopkThreads), st2 ? smem + (size_t)ch * k * 8 : smem, st, 
        q_pos, N, m, k, ch, P, st2, cand, idx_out, score_out);
  } else {
    launch_pdl(topk_kernel, dim3((unsigned)rows), dim3(kTopkRowThreads), smem, st, scores_ws, q_pos, N, m, k, P, idx_out, score_out);
  }
  return cudaGetLastError();
}

}  // namespace csa
