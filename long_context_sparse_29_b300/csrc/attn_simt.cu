// attn_simt.cu -- CUDA-core attention over compressed entries + window.
//
// Serves the fp32 cache format (fp32 q, keys and output, accumulation in
// fp32) and is also a straightforward second kernel for the mixed FP8/BF16
// cache.  One CTA per query; heads in sequence; keys in tiles of one key per
// thread with an online softmax.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）":
// multi-query attention over the selected compressed entries only, plus a
// sliding-window branch; section "HCA（重度压缩注意力）": dense attention
// over all compressed entries; section "关键技术细节": RoPE on the last 64
// dims of q and KV, inverse rotation of the output.
#include "csa_common.cuh"
#include "launch.h"

namespace csa {

constexpr int kSimtThreads = 256;
constexpr int kSkip = -0x7fffffff - 1;

// dequantised channel c of a key row
template <bool MIXED>
__device__ __forceinline__ float key_at(const uint8_t* row, int c) {
  if (MIXED) {
    if (c < kMixDn) {
      const float sc = reinterpret_cast<const float*>(row + kMixScaleOff)[c >> 7];
      return e4m3_decode(row[c]) * sc;
    }
    return bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(row + kMixRopeOff)[c - kMixDn]);
  }
  return reinterpret_cast<const float*>(row)[c];
}

__device__ __forceinline__ float block_reduce_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kSimtThreads / 32; ++i) r = fmaxf(r, red[i]);
  return r;
}

__device__ __forceinline__ float block_reduce_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.0f;
  for (int i = 0; i < kSimtThreads / 32; ++i) r += red[i];
  return r;
}

template <bool MIXED, bool BF16>
__global__ void __launch_bounds__(kSimtThreads)
attn_simt_kernel(const void* __restrict__ q, const int64_t* __restrict__ q_pos, int64_t Tq, int H,
                 int D, int R, const uint8_t* __restrict__ cache, int64_t N, int m,
                 const int32_t* __restrict__ idx, int k, const uint8_t* __restrict__ swa,
                 const int64_t* __restrict__ swa_pos0, int64_t Ts, int W, float scale,
                 const float* __restrict__ rcos, const float* __restrict__ rsin,
                 int64_t rope_rows, void* __restrict__ out, float* __restrict__ lse, void* ws,
                 int max_keys) {
  pdl_begin();
  extern __shared__ float sm[];
  float* qr = sm;                       // [D]
  float* pt = qr + D;                   // [kSimtThreads] probabilities of the tile
  float* ot = pt + kSimtThreads;        // [D] output staging
  float* red = ot + D;                  // [32]
  int* keys = reinterpret_cast<int*>(red + 32);   // [max_keys] key codes

  const int64_t row_q = blockIdx.x;     // b * Tq + i
  const int64_t b = row_q / Tq;
  const int64_t t = q_pos[row_q];
  const int tid = threadIdx.x;
  const size_t rowb = MIXED ? kMixRow : (size_t)D * 4;
  if (t < 0 || t >= rope_rows) {   // no RoPE row for this position: skip the query
    if (tid == 0) flag_device_check(ws, 0x40000000u);
    for (int64_t c = tid; c < (int64_t)H * D; c += kSimtThreads) {
      if (BF16) reinterpret_cast<__nv_bfloat16*>(out)[row_q * H * D + c] = __float2bfloat16_rn(0.0f);
      else reinterpret_cast<float*>(out)[row_q * H * D + c] = 0.0f;
    }
    if (lse)
      for (int h = tid; h < H; h += kSimtThreads) lse[row_q * H + h] = -INFINITY;
    return;
  }
  // ---- key list (deterministic order): entry j -> j; window row r -> -(r + 1);
  //      a key that must be skipped -> kSkip ----
  int ne;
  if (idx) {
    for (int r = tid; r < k; r += kSimtThreads) {
      int32_t j = idx[row_q * k + r];
      if (j >= 0 && ((int64_t)j >= N || (int64_t)(j + 1) * m - 1 > t)) {
        flag_device_check(ws, (unsigned)j);
        j = -1;
      }
      keys[r] = j >= 0 ? j : kSkip;
    }
    ne = k;
  } else {
    int64_t nv = (t + 1) / m;
    nv = nv < N ? nv : N;
    for (int64_t j = tid; j < nv; j += kSimtThreads) keys[j] = (int)j;
    ne = (int)nv;
  }
  for (int i = tid; i < W; i += kSimtThreads) {
    const int64_t u = t - W + 1 + i;
    int code = kSkip;
    if (u >= 0) {
      const int64_t r = u - swa_pos0[b];
      if (r < 0 || r >= Ts) flag_device_check(ws, 0x80000000u | (unsigned)i);
      else code = -(int)(r + 1);
    }
    keys[ne + i] = code;
  }
  __syncthreads();
  const int nk = ne + W;
  const int half = R >> 1;
  const float* cs = rcos + t * half;
  const float* sn = rsin + t * half;

  for (int h = 0; h < H; ++h) {
    // rotated query (fp32, one rounding per operation)
    const int64_t qoff = (row_q * H + h) * D;
    for (int c = tid; c < D; c += kSimtThreads)
      qr[c] = BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[qoff + c])
                   : reinterpret_cast<const float*>(q)[qoff + c];
    __syncthreads();
    for (int i = tid; i < half; i += kSimtThreads) {
      const float x0 = qr[D - R + 2 * i], x1 = qr[D - R + 2 * i + 1];
      qr[D - R + 2 * i] = __fsub_rn(__fmul_rn(x0, cs[i]), __fmul_rn(x1, sn[i]));
      qr[D - R + 2 * i + 1] = __fadd_rn(__fmul_rn(x0, sn[i]), __fmul_rn(x1, cs[i]));
    }
    __syncthreads();
    float mrun = -INFINITY, lrun = 0.0f;
    float o0 = 0.0f, o1 = 0.0f;           // channels tid and tid + 256
    for (int base = 0; base < nk; base += kSimtThreads) {
      const int i = base + tid;
      float lg = -INFINITY;
      if (i < nk && keys[i] != kSkip) {
        const int code = keys[i];
        const uint8_t* kr = code >= 0 ? cache + ((size_t)b * N + code) * rowb
                                      : swa + ((size_t)b * Ts + (-code - 1)) * rowb;
        float d = 0.0f;
        for (int c = 0; c < D; ++c) d = fmaf(qr[c], key_at<MIXED>(kr, c), d);
        lg = d * scale;
      }
      const float tmax = block_reduce_max(lg, red);
      const float mnew = fmaxf(mrun, tmax);
      const float p = (lg != -INFINITY) ? __expf(lg - mnew) : 0.0f;
      pt[tid] = p;
      const float tsum = block_reduce_sum(p, red);
      const float alpha = (mnew == -INFINITY) ? 1.0f : __expf(mrun - mnew);
      lrun = lrun * alpha + tsum;
      o0 *= alpha;
      o1 *= alpha;
      mrun = mnew;
      __syncthreads();
      const int cnt = min(kSimtThreads, nk - base);
      for (int ii = 0; ii < cnt; ++ii) {
        const int code = keys[base + ii];
        if (code == kSkip) continue;
        const uint8_t* kr = code >= 0 ? cache + ((size_t)b * N + code) * rowb
                                      : swa + ((size_t)b * Ts + (-code - 1)) * rowb;
        const float pi = pt[ii];
        if (tid < D) o0 = fmaf(pi, key_at<MIXED>(kr, tid), o0);
        if (tid + kSimtThreads < D) o1 = fmaf(pi, key_at<MIXED>(kr, tid + kSimtThreads), o1);
      }
      __syncthreads();
    }
    const float inv = lrun > 0.0f ? 1.0f / lrun : 0.0f;
    if (tid < D) ot[tid] = o0 * inv;
    if (tid + kSimtThreads < D) ot[tid + kSimtThreads] = o1 * inv;
    __syncthreads();
    for (int i = tid; i < half; i += kSimtThreads) {   // inverse rotation
      const float x0 = ot[D - R + 2 * i], x1 = ot[D - R + 2 * i + 1];
      ot[D - R + 2 * i] = x0 * cs[i] + x1 * sn[i];
      ot[D - R + 2 * i + 1] = -x0 * sn[i] + x1 * cs[i];
    }
    __syncthreads();
    for (int c = tid; c < D; c += kSimtThreads) {
      if (BF16) reinterpret_cast<__nv_bfloat16*>(out)[qoff + c] = __float2bfloat16_rn(ot[c]);
      else reinterpret_cast<float*>(out)[qoff + c] = ot[c];
    }
    if (lse && tid == 0) lse[row_q * H + h] = lrun > 0.0f ? mrun + logf(lrun) : -INFINITY;
    __syncthreads();
  }
}

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.Tq;
  if (rows == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (2 * (size_t)a.D + kSimtThreads + 32) + sizeof(int) * (size_t)a.max_keys;
  const bool mixed = a.cache_fmt == CSA_FMT_MIXED592;
  const bool bf16 = a.q_bf16;
#define CSA_AS(MX, BF)                                                                          \
  do {                                                                                          \
    cudaFuncSetAttribute(attn_simt_kernel<MX, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                         (int)smem);                                                            \
    launch_pdl(attn_simt_kernel<MX, BF>, dim3((unsigned)rows), dim3(kSimtThreads), smem, st,                        \
        a.q, a.q_pos, a.Tq, a.H, a.D, a.R, reinterpret_cast<const uint8_t*>(a.cache), a.N, a.m, \
        a.idx, a.k, reinterpret_cast<const uint8_t*>(a.swa), a.swa_pos0, a.Ts, a.W, a.scale,    \
        a.rcos, a.rsin, a.rope_rows, a.out, a.lse, a.ws, a.max_keys);                                        \
  } while (0)
  if (mixed) {
    if (bf16) CSA_AS(true, true); else CSA_AS(true, false);
  } else {
    if (bf16) CSA_AS(false, true); else CSA_AS(false, false);
  }
#undef CSA_AS
  return cudaGetLastError();
}

}  // namespace csa
