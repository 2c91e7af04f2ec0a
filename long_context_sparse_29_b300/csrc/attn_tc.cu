// attn_tc.cu -- tensor-core (tcgen05 / TMEM) attention of every query over
// its compressed entries and its sliding window, mixed FP8/BF16 cache.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）": MQA over
// the selected compressed entries plus a sliding-window branch; section
// "HCA（重度压缩注意力）": dense attention over all compressed entries;
// section "关键技术细节": RoPE on the last 64 dims with inverse rotation of
// the output, RoPE dims BF16 and the rest FP8 in the KV cache.
//
// One CTA per query token, all 64 heads (they share the KV: MQA).  Keys run
// in tiles of 128:
//   producer warps 4-7  gather the tile's 592-byte rows from HBM/L2,
//                       dequantise FP8 x 2^e (exact in bf16) and write a
//                       128 x 512 bf16 tile, 128-byte swizzled, into smem;
//   MMA warp 8          S = Q K^T   (M = 64 heads, N = 128 keys, K = 512)
//                       into TMEM, then O^T += V^T P^T (M = 128 dims x 4,
//                       N = 64 heads, K = 128 keys) into TMEM -- the value
//                       of a key is the key itself, so the same smem tile is
//                       read K-major for QK^T and MN-major for PV;
//   softmax warps 0-3   read S from TMEM, online softmax in the exp2 domain
//                       with a lazy rescale of O^T (only when a running max
//                       grows by more than 2^8), write bf16 P to smem, and in
//                       the end normalise O, rotate its RoPE dims back and
//                       store bf16.
// Waits are bounded; on expiry the CTA records a timeout and returns.
#include "csa_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace csa {

using namespace tc;

namespace {

constexpr int kH = 64;
constexpr int kD = 512;
constexpr int kTile = 128;
constexpr int kThreads = 9 * 32;
constexpr int kMmaWarp = 8;

constexpr uint32_t kQOff = 0;                     // 8 x [64 x 128 B]
constexpr uint32_t kKVOff = 65536;                // 8 x [128 x 128 B]
constexpr uint32_t kPOff = kKVOff + 131072;       // 2 x [64 x 128 B]
constexpr uint32_t kMiscOff = kPOff + 16384;      // 1 KB of barriers and per-head state
constexpr uint32_t kListOff = kMiscOff + 1024;    // int32 key list
constexpr uint32_t kSmemLimit = 232448;
constexpr int kMaxList = (int)((kSmemLimit - 1024 - kListOff) / 4);

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;      // O^T: 4 blocks of 64 columns (heads), lanes = dims
constexpr uint32_t kTmemS = 256;    // S: 2 buffers of 128 columns (keys)

constexpr uint32_t kWaitLimit = 1u << 20;
constexpr float kLazy = 8.0f;       // log2 growth of a running max that forces a rescale

// rows of a 64-row (M = 64) accumulator: warp quadrant q, lanes 0-15 hold rows 16 q + lane
__device__ __forceinline__ bool s_row_valid(int lane) { return lane < 16; }
__device__ __forceinline__ int s_row(int q, int lane) { return 16 * q + lane; }

struct Misc {
  uint64_t bar_full, bar_s, bar_p, bar_o;
  uint32_t tmem;
  int abort;
  int any_rescale[2];
  int nkeys;
  float alpha[kH];
  float l_fin[kH];
};

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk16) {
  return row * 128u + (((chunk16 ^ row) & 7u) << 4);
}

// 16 E4M3 codes (one uint4) times 2^e -> 16 bf16 (two uint4), exact
__device__ __forceinline__ void dequant16(const uint4 c, float sc, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((w[i] >> (16 * h)) & 0xffffu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
      const float2 f = __half22float2(__half2(hr));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      r[2 * i + h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

template <bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __nv_bfloat16* __restrict__ q, const int64_t* __restrict__ q_pos, int64_t Tq,
               const uint8_t* __restrict__ cache, int64_t N, int m, const int32_t* __restrict__ idx,
               int k, const uint8_t* __restrict__ swa, const int64_t* __restrict__ swa_pos0,
               int64_t Ts, int W, float scale_log2, const float* __restrict__ rcos,
               const float* __restrict__ rsin, int64_t rope_rows, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse, void* ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kQOff;
  uint8_t* sKV = sm + kKVOff;
  uint8_t* sP = sm + kPOff;
  Misc* ms = reinterpret_cast<Misc*>(sm + kMiscOff);
  int32_t* list = reinterpret_cast<int32_t*>(sm + kListOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row_q = blockIdx.x;
  const int64_t b = row_q / Tq;
  const int64_t t = q_pos[row_q];
  const bool t_ok = t >= 0 && t < rope_rows;

  // ---------------- set-up: key list, window range, Q with RoPE ----------------
  if (tid == 0) {
    ms->abort = 0;
    ms->any_rescale[0] = 0;
    ms->any_rescale[1] = 0;
    if (!t_ok) flag_device_check(ws, 0x40000000u);
    mbar_init(&ms->bar_full, 4);
    mbar_init(&ms->bar_s, 1);
    mbar_init(&ms->bar_p, 4);
    mbar_init(&ms->bar_o, 1);
    mbar_fence_init();
  }
  int ne = 0;                       // entries in the key list (sparse) or visible (dense)
  if (!DENSE) {
    if (warp == 0 && t_ok) {        // ordered compaction of the valid selected entries
      int cnt = 0;
      for (int base = 0; base < k; base += 32) {
        const int r = base + lane;
        int32_t j = r < k ? idx[row_q * k + r] : -1;
        if (j >= 0 && ((int64_t)j >= N || (int64_t)(j + 1) * m - 1 > t)) {
          flag_device_check(ws, (unsigned)j);
          j = -1;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, j >= 0);
        const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
        if (j >= 0 && pos < kMaxList) list[pos] = j;
        cnt += __popc(bal);
      }
      if (lane == 0) ms->nkeys = cnt < kMaxList ? cnt : kMaxList;
    }
  } else if (tid == 0) {
    int64_t nv = t_ok ? (t + 1) / m : 0;
    ms->nkeys = (int)(nv < N ? nv : N);
  }
  // window tokens u in [max(0, t-W+1), t] held by the window cache
  int64_t u_lo = t - W + 1 < 0 ? 0 : t - W + 1;
  const int64_t p0 = W > 0 ? swa_pos0[b] : 0;
  int64_t w_lo = u_lo < p0 ? p0 : u_lo;
  int64_t w_hi = t < p0 + Ts - 1 ? t : p0 + Ts - 1;
  int nwin = (t_ok && W > 0 && w_hi >= w_lo) ? (int)(w_hi - w_lo + 1) : 0;
  if (tid == 0 && t_ok && W > 0 && (w_lo > u_lo || w_hi < t)) flag_device_check(ws, 0x80000000u);
  if (t_ok) {
    // Q: 64 heads x 512 dims bf16 -> smem (8 chunks of 64 dims, SW128); RoPE on chunk 7
    const uint4* qg = reinterpret_cast<const uint4*>(q + row_q * (int64_t)(kH * kD));
    const float* cs = rcos + t * 32;
    const float* sn = rsin + t * 32;
    for (int v = tid; v < kH * kD / 8; v += kThreads) {
      const int h = v >> 6, c16 = v & 63;       // 16-byte vector c16 of head h (8 dims)
      uint4 x = qg[v];
      if (c16 >= 56) {                          // dims 448..511: rotate 4 pairs
        uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int i = (c16 - 56) * 4 + p;     // pair index within the RoPE slice
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[p]));
          const float y0 = __fsub_rn(__fmul_rn(f.x, cs[i]), __fmul_rn(f.y, sn[i]));
          const float y1 = __fadd_rn(__fmul_rn(f.x, sn[i]), __fmul_rn(f.y, cs[i]));
          const __nv_bfloat162 r = __floats2bfloat162_rn(y0, y1);
          wd[p] = *reinterpret_cast<const uint32_t*>(&r);
        }
        x = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
      const int chunk = c16 >> 3, sub = c16 & 7;
      *reinterpret_cast<uint4*>(sQ + chunk * 8192 + sw128(h, sub)) = x;
    }
  }
  if (warp == kMmaWarp) tmem_alloc(&ms->tmem, kTmemCols);
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;
  ne = ms->nkeys;
  const int nkeys = ne + nwin;
  const int ntiles = (nkeys + kTile - 1) / kTile;

  if (warp >= 4 && warp < 8) {
    // ============================ producers ============================
    const int pw = warp - 4;
    for (int i = 0; i < ntiles; ++i) {
      if (i > 0 && !mbar_wait(&ms->bar_o, (i - 1) & 1, kWaitLimit)) {
        ms->abort = 1;
        flag_timeout(ws);
        break;
      }
      if (ms->abort) break;
      for (int r = pw; r < kTile; r += 4) {
        const int key = i * kTile + r;
        const uint8_t* row = nullptr;
        if (key < ne) {
          const int64_t j = DENSE ? (int64_t)key : (int64_t)list[key];
          row = cache + ((size_t)b * N + j) * kMixRow;
        } else if (key < nkeys) {
          row = swa + ((size_t)b * Ts + (w_lo - p0 + (key - ne))) * kMixRow;
        }
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
        if (lane < 28) {
          if (row) {
            const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);
            const float sc = __ldg(reinterpret_cast<const float*>(row + kMixScaleOff) + (lane >> 3));
            dequant16(c, sc, o0, o1);
          }
          const int chunk = lane >> 2, sub = 2 * (lane & 3);
          uint8_t* dst = sKV + chunk * 16384;
          *reinterpret_cast<uint4*>(dst + sw128(r, sub)) = o0;
          *reinterpret_cast<uint4*>(dst + sw128(r, sub + 1)) = o1;
        } else {
          const int l4 = lane - 28;
          if (row) {
            o0 = __ldg(reinterpret_cast<const uint4*>(row + kMixRopeOff) + 2 * l4);
            o1 = __ldg(reinterpret_cast<const uint4*>(row + kMixRopeOff) + 2 * l4 + 1);
          }
          uint8_t* dst = sKV + 7 * 16384;
          *reinterpret_cast<uint4*>(dst + sw128(r, 2 * l4)) = o0;
          *reinterpret_cast<uint4*>(dst + sw128(r, 2 * l4 + 1)) = o1;
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->bar_full);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issue ============================
    if (lane == 0) {
      const uint32_t aQ = smem_u32(sQ), aKV = smem_u32(sKV), aP = smem_u32(sP);
      constexpr uint32_t idQK = idesc_bf16(64, kTile, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(128, kH, 1, 0);
      for (int i = 0; i < ntiles; ++i) {
        if (!mbar_wait(&ms->bar_full, i & 1, kWaitLimit)) {
          ms->abort = 1;
          flag_timeout(ws);
          break;
        }
        fence_after_sync();
        const uint32_t dS = tmem + kTmemS + 128u * (i & 1);
#pragma unroll 4
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk & 3) * 32u;
          mma_bf16(dS, sdesc_sw128(aQ + (kk >> 2) * 8192 + off, 16, 1024),
                   sdesc_sw128(aKV + (kk >> 2) * 16384 + off, 16, 1024), idQK, kk > 0);
        }
        mma_commit(&ms->bar_s);
        if (!mbar_wait(&ms->bar_p, i & 1, kWaitLimit)) {
          ms->abort = 1;
          flag_timeout(ws);
          break;
        }
        fence_after_sync();
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            const uint64_t a = sdesc_sw128(aKV + (2 * mt) * 16384 + ks * 2048, 16384, 1024);
            const uint64_t bb = sdesc_sw128(aP + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
            mma_bf16(tmem + kTmemO + 64u * mt, a, bb, idPV, (i > 0 || ks > 0) ? 1u : 0u);
          }
        }
        mma_commit(&ms->bar_o);
      }
    }
    __syncwarp();
  } else {
    // ============================ softmax ============================
    const int qd = warp;                 // TMEM lane quadrant
    const bool hv = s_row_valid(lane);
    const int h = s_row(qd, lane);
    float m_run = -INFINITY, l_run = 0.0f;
    for (int i = 0; i < ntiles; ++i) {
      if (!mbar_wait(&ms->bar_s, i & 1, kWaitLimit)) {
        ms->abort = 1;
        flag_timeout(ws);
        break;
      }
      fence_after_sync();
      const int nvalid = min(kTile, nkeys - i * kTile);
      const uint32_t sbase = tmem + ((uint32_t)(32 * qd) << 16) + kTmemS + 128u * (i & 1);
      // pass 1: tile max
      float tmax = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kTile; c += 32) {
        uint32_t v[32];
        tmem_ld32(sbase + c, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < nvalid) tmax = fmaxf(tmax, __uint_as_float(v[j]) * scale_log2);
      }
      const bool need = hv && tmax > m_run + kLazy;
      const float m_new = need ? tmax : m_run;
      const float alpha = need ? exp2f(m_run - m_new) : 1.0f;   // exp2(-inf) = 0 on the first tile
      if (i > 0) {
        // rescale O^T when any head's running max jumped
        if (__any_sync(0xffffffffu, need) && lane == 0) atomicOr(&ms->any_rescale[i & 1], 1);
        if (hv) ms->alpha[h] = alpha;
        named_bar_sync(1, 128);
        if (tid == 0) ms->any_rescale[(i + 1) & 1] = 0;
        if (ms->any_rescale[i & 1]) {
          float al[kH];
#pragma unroll
          for (int hh = 0; hh < kH; ++hh) al[hh] = ms->alpha[hh];
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t v[32];
              const uint32_t oa = tmem + ((uint32_t)(32 * qd) << 16) + kTmemO + 64u * mt + 32u * half;
              tmem_ld32(oa, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * al[32 * half + j]);
              tmem_st32(oa, v);
            }
          }
          tmem_wait_st();
        }
        named_bar_sync(1, 128);
      }
      m_run = m_new;
      // pass 2: probabilities -> bf16 P rows (head h, 128 keys), row sums
      float psum = 0.0f;
#pragma unroll 1
      for (int c = 0; c < kTile; c += 32) {
        uint32_t v[32];
        tmem_ld32(sbase + c, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = (c + j < nvalid) ? exp2f(__uint_as_float(v[j]) * scale_log2 - m_run) : 0.0f;
          const float p1 = (c + j + 1 < nvalid) ? exp2f(__uint_as_float(v[j + 1]) * scale_log2 - m_run) : 0.0f;
          psum += p0 + p1;
          const __nv_bfloat162 bp = __floats2bfloat162_rn(p0, p1);
          pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&bp);
        }
        if (hv) {
          uint8_t* dst = sP + (c >> 6) * 8192;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t sub = ((c & 63) >> 3) + s;
            *reinterpret_cast<uint4*>(dst + sw128(h, sub)) =
                make_uint4(pk[4 * s], pk[4 * s + 1], pk[4 * s + 2], pk[4 * s + 3]);
          }
        }
      }
      l_run = l_run * alpha + psum;
      fence_proxy_async();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->bar_p);
    }
    // ============================ epilogue ============================
    if (hv) ms->l_fin[h] = l_run;
    if (hv && lse) lse[row_q * kH + h] = l_run > 0.0f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    bool ok = ntiles > 0;
    if (ok && !mbar_wait(&ms->bar_o, (ntiles - 1) & 1, kWaitLimit)) {
      ms->abort = 1;
      flag_timeout(ws);
      ok = false;
    }
    named_bar_sync(1, 128);
    fence_after_sync();
    float inv[kH];
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) inv[hh] = (ok && ms->l_fin[hh] > 0.0f) ? 1.0f / ms->l_fin[hh] : 0.0f;
    const float* cs = rcos + (t_ok ? t : 0) * 32;
    const float* sn = rsin + (t_ok ? t : 0) * 32;
    __nv_bfloat16* og = out + row_q * (int64_t)(kH * kD);
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      const int d = 128 * mt + 32 * qd + lane;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
        if (ok) {
          tmem_ld32(tmem + ((uint32_t)(32 * qd) << 16) + kTmemO + 64u * mt + 32u * half, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float o = __uint_as_float(v[j]) * inv[32 * half + j];
          if (d >= kMixDn) {          // inverse rotation of the RoPE dims (pairs in adjacent lanes)
            const float other = __shfl_xor_sync(0xffffffffu, o, 1);
            const int pi = (d - kMixDn) >> 1;
            o = (d & 1) ? (-other * sn[pi] + o * cs[pi]) : (o * cs[pi] + other * sn[pi]);
          }
          og[(32 * half + j) * kD + d] = __float2bfloat16_rn(o);
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t attn_tc_workspace(int, int64_t, int, int, int64_t) { return 0; }

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.Tq;
  if (rows == 0) return cudaSuccess;
  if (a.H != kH || a.D != kD || a.R != 64) return launch_attn_simt(a, st);
  if (a.idx && a.k > kMaxList) return launch_attn_simt(a, st);
  const size_t smem = kSmemLimit;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  if (a.idx) {
    cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attn_tc_kernel<false><<<(unsigned)rows, kThreads, smem, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(a.q), a.q_pos, a.Tq,
        reinterpret_cast<const uint8_t*>(a.cache), a.N, a.m, a.idx, a.k,
        reinterpret_cast<const uint8_t*>(a.swa), a.swa_pos0, a.Ts, a.W, scale_log2, a.rcos, a.rsin,
        a.rope_rows, reinterpret_cast<__nv_bfloat16*>(a.out), a.lse, a.ws);
  } else {
    cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attn_tc_kernel<true><<<(unsigned)rows, kThreads, smem, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(a.q), a.q_pos, a.Tq,
        reinterpret_cast<const uint8_t*>(a.cache), a.N, a.m, nullptr, 0,
        reinterpret_cast<const uint8_t*>(a.swa), a.swa_pos0, a.Ts, a.W, scale_log2, a.rcos, a.rsin,
        a.rope_rows, reinterpret_cast<__nv_bfloat16*>(a.out), a.lse, a.ws);
  }
  return cudaGetLastError();
}

}  // namespace csa
