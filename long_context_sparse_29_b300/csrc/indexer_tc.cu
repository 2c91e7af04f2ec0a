// indexer_tc.cu -- lightning-indexer scores on the FP8 tensor cores.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）": a lightning
// indexer scores every visible compressed entry for each query token, and
// section "关键技术细节": its attention runs in FP4.
//
// score(t, j) = sum_h w_{t,h} relu(d_{t,h,j}), the head sum an fma chain from
// +0 in ascending h, and d = P0 2^(e_q0 + e_k0 - 2) + P1 2^(e_q1 + e_k1 - 2)
// rounded once, where P_b is the dot of the two 32-element MXFP4 blocks b
// with every E2M1 value doubled (an integer in [-12, 12]).  These are the
// same numbers as the dp4a kernel in indexer.cu computes.
//
// Here P_b comes from tcgen05.mma kind::f8f6f4: the doubled E2M1 values are
// small integers, exact in E4M3, and every partial sum of 32 products of
// them is an integer below 2^13, exact in the fp32 accumulator whatever the
// order of the additions -- so P_b is the exact integer, and the scores are
// bit-identical to the integer path.
//
// Work: one CTA per (128 query rows, 256 entries) of a sequence, entries past
// the last visible one skipped.  Warp 8 loads the quantised queries (all
// heads, 128 KiB) once and a ring of entry tiles (64 entries) with TMA;
// warp 9 issues, per tile and head, the two block MMAs (M = 128 rows, N = 64
// entries, K = 32) into one of four TMEM buffers; warps 0-7 (row quadrant
// w % 4, entry half w / 4) combine the blocks, apply relu and the head
// weights in ascending head order and store the scores.
#include <cuda.h>

#include "csa_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace csa {

using namespace tc;

namespace {

constexpr int kIxRows = 128;       // query rows per CTA (MMA M)
constexpr int kIxKeys = 64;        // entries per tile (MMA N)
constexpr int kIxChunk = 256;      // entries per CTA
constexpr int kIxStages = 4;       // entry-tile ring
constexpr int kIxBufs = 4;         // TMEM head buffers, 128 columns each (block 0 | block 1)
constexpr int kIxMaxHeads = 16;
constexpr int kIxThreads = 10 * 32;
constexpr int kIxProducer = 8, kIxMma = 9;

constexpr uint32_t kIxQChunk = kIxRows * 128;                 // two heads x 64 dims, 128 rows
constexpr uint32_t kIxKTile = kIxKeys * 128;                  // 64 entries x 128 B (64 data + 64 zero)
constexpr uint32_t kIxKOff = (kIxMaxHeads / 2) * kIxQChunk;   // 128 KiB of queries
constexpr uint32_t kIxMiscOff = kIxKOff + kIxStages * kIxKTile;
constexpr uint32_t kIxSmem = kIxMiscOff + 1024 + 1024;        // + slack for 1 KiB alignment

constexpr uint32_t kIxWait = 1u << 20;
constexpr uint32_t kIxNapWait = 1u << 22;     // polls with ~64 ns naps between them (~0.3 s)

struct IxMisc {
  uint64_t q_full, k_full[kIxStages], k_empty[kIxStages], t_full[kIxBufs], t_empty[kIxBufs], drain;
  uint32_t tmem;
  int nv_max;
};

// 2 x E2M1 value of a code, as the E4M3 byte that holds it exactly
// (magnitudes 0, 1, 2, 3, 4, 6, 8, 12; bit 3 of the code is the sign)
__device__ __forceinline__ uint32_t e2m1x2_e4m3(uint32_t code) {
  const uint32_t mag = 0x54504C4844403800ull >> (8 * (code & 7)) & 0xffu;   // (lookup in a 64-bit word)
  return mag | ((code & 8u) << 4);
}

// kind::f8f6f4 instruction descriptor: E4M3 A and B (format 0), fp32 D,
// both K-major; N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3_elect(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, 0, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc));
}

__device__ __forceinline__ int64_t visible(int64_t t, int m, int64_t N) {
  int64_t nv = (t + 1) / m;
  nv = nv < 0 ? 0 : nv;
  return nv < N ? nv : N;
}

}  // namespace

// Query quantisation: one thread per (row, head, 32-block); MXFP4 with the
// block exponent floor(log2 amax) - 2, each value stored as the E4M3 byte of
// twice its E2M1 value.  qx: [rows, HI * 64] bytes; qe: [rows, HI, 2].
__global__ void __launch_bounds__(256)
ix_quant_q_kernel(const __nv_bfloat16* __restrict__ qI, int64_t rows, int HI, uint8_t* __restrict__ qx,
                  int8_t* __restrict__ qe) {
  pdl_begin();
  const int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (u >= rows * HI * 2) return;
  const int64_t rh = u >> 1;        // row * HI + h
  const int blk = (int)(u & 1);
  const uint4* src = reinterpret_cast<const uint4*>(qI + rh * 64 + 32 * blk);
  float v[32];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 x = __ldg(src + i);
    const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * i + 2 * e] = __uint_as_float(wd[e] << 16);
      v[8 * i + 2 * e + 1] = __uint_as_float(wd[e] & 0xffff0000u);
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int sx = mx_block_exp(amax);
  const float inv = pow2i(-sx);
  uint32_t wq[8];
#pragma unroll
  for (int wd = 0; wd < 8; ++wd) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) word |= e2m1x2_e4m3(e2m1_encode(__fmul_rn(v[4 * wd + e], inv))) << (8 * e);
    wq[wd] = word;
  }
  uint4* dst = reinterpret_cast<uint4*>(qx + rh * 64 + 32 * blk);
  dst[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
  dst[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
  qe[u] = (int8_t)sx;
}

// Entry expansion: 64 E2M1 codes (byte c/2, low nibble first) -> 64 E4M3
// bytes of the doubled values, then 64 zero bytes (128-byte rows for the
// swizzled TMA layout).  One thread per (entry, 16-byte output unit).
__global__ void __launch_bounds__(256)
ix_expand_k_kernel(const uint8_t* __restrict__ kc, int64_t n, uint8_t* __restrict__ kx) {
  pdl_begin();
  const int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (u >= n * 8) return;
  const int64_t key = u >> 3;
  const int part = (int)(u & 7);
  uint4 out = make_uint4(0, 0, 0, 0);
  if (part < 4) {   // codes 16 part .. 16 part + 15 from bytes 8 part .. 8 part + 7
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(kc + key * 32) + part);
    const uint32_t cw[2] = {c.x, c.y};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t src = cw[i >> 1] >> (16 * (i & 1));   // codes 4i .. 4i + 3 of this unit
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) word |= e2m1x2_e4m3((src >> (4 * e)) & 15u) << (8 * e);
      o[i] = word;
    }
    out = make_uint4(o[0], o[1], o[2], o[3]);
  }
  reinterpret_cast<uint4*>(kx + key * 128)[part] = out;
}

struct IxParams {
  const int8_t* qe;         // [B * Tq, HI, 2]
  const float* w;           // [B * Tq, HI]
  const uint8_t* ks;        // [B * N, 2] E8M0 entry block scales
  const int64_t* q_pos;
  int64_t Tq, N;
  int HI, m;
  float* scores;            // [B * Tq, N]
  void* ws;                 // status flags
};

__global__ void __launch_bounds__(kIxThreads, 1)
ix_scores_tc_kernel(const IxParams p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  IxMisc* ms = reinterpret_cast<IxMisc*>(sm + kIxMiscOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  const int64_t t0 = (int64_t)blockIdx.y * kIxRows;
  const int64_t c0 = (int64_t)blockIdx.x * kIxChunk;

  if (tid == 0) ms->nv_max = 0;
  __syncthreads();
  if (tid < kIxRows && t0 + tid < p.Tq) {
    const int nv = (int)visible(p.q_pos[b * p.Tq + t0 + tid], p.m, p.N);
    atomicMax(&ms->nv_max, nv);
  }
  __syncthreads();
  const int64_t nv_max = ms->nv_max;
  if (c0 >= nv_max) return;   // no row of the tile sees this chunk (uniform exit)
  const int nt = (int)(((nv_max - c0 < kIxChunk ? nv_max - c0 : kIxChunk) + kIxKeys - 1) / kIxKeys);

  if (tid == 0) {
    mbar_init(&ms->q_full, 1);
    for (int i = 0; i < kIxStages; ++i) {
      mbar_init(&ms->k_full[i], 1);
      mbar_init(&ms->k_empty[i], 1);
    }
    for (int i = 0; i < kIxBufs; ++i) {
      mbar_init(&ms->t_full[i], 1);
      mbar_init(&ms->t_empty[i], 8);
    }
    mbar_init(&ms->drain, 1);
    mbar_fence_init();
  }
  if (warp == kIxMma) tmem_alloc(&ms->tmem, 512);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;
  const uint32_t aQ = smem_u32(sm), aK = smem_u32(sm + kIxKOff);
  const int nchunks = p.HI / 2;

  if (warp == kIxProducer) {
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(&ms->q_full, (uint32_t)nchunks * kIxQChunk);
      for (int c = 0; c < nchunks; ++c)
        tma_load_2d(aQ + c * kIxQChunk, &tm_q, 128 * c, (int)(b * p.Tq + t0), &ms->q_full);
      for (int kt = 0; kt < nt && ok; ++kt) {
        const int s = kt % kIxStages;
        if (kt >= kIxStages && !mbar_wait(&ms->k_empty[s], ((kt / kIxStages) - 1) & 1, kIxWait)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&ms->k_full[s], kIxKTile);
        tma_load_2d(aK + s * kIxKTile, &tm_k, 0, (int)(b * p.N + c0 + (int64_t)kIxKeys * kt), &ms->k_full[s]);
      }
      if (!ok) flag_timeout(p.ws);
      // copies still in flight land before the CTA exits
      mbar_wait(&ms->q_full, 0, kIxWait);
      if (nt > 0) mbar_wait(&ms->k_full[(nt - 1) % kIxStages], ((nt - 1) / kIxStages) & 1, kIxWait);
    }
    __syncwarp();
  } else if (warp == kIxMma) {
    constexpr uint32_t id = idesc_e4m3(kIxRows, kIxKeys);
    bool ok = mbar_wait(&ms->q_full, 0, kIxWait);
    fence_after_sync();
    uint32_t u = 0;   // head steps issued
    for (int kt = 0; kt < nt && ok; ++kt) {
      const int s = kt % kIxStages;
      if (!mbar_wait(&ms->k_full[s], (kt / kIxStages) & 1, kIxWait)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint64_t kd = sdesc_sw128(aK + s * kIxKTile, 16, 1024);
      for (int h = 0; h < p.HI; ++h, ++u) {
        const uint32_t hb = u % kIxBufs;
        if (u >= kIxBufs && !mbar_wait(&ms->t_empty[hb], ((u / kIxBufs) - 1) & 1, kIxWait)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint64_t qd = sdesc_sw128(aQ + (h >> 1) * kIxQChunk, 16, 1024);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
          mma_e4m3_elect(tmem + 128u * hb + 64u * blk, qd + (uint64_t)((64 * (h & 1) + 32 * blk) >> 4),
                         kd + (uint64_t)((32 * blk) >> 4), id);
        mma_commit_elect(&ms->t_full[hb]);
        __syncwarp();
      }
      if (!ok) break;
      mma_commit_elect(&ms->k_empty[s]);
      __syncwarp();
    }
    if (!ok && lane == 0) flag_timeout(p.ws);
    mma_commit_elect(&ms->drain);
    __syncwarp();
    mbar_wait(&ms->drain, 0, kIxWait);
  } else {
    // ============ epilogue: warp w = rows 32 (w % 4) + lane, entries 32 (w / 4) + j of a tile ============
    const int qd = warp & 3, kh = warp >> 2;
    const int64_t t = t0 + 32 * qd + lane;
    const bool row_ok = t < p.Tq;
    const int64_t row = b * p.Tq + (row_ok ? t : 0);
    const float* wrow = p.w + row * p.HI;            // head weights of the row
    const int8_t* qerow = p.qe + row * p.HI * 2;      // its block exponents (read per head, L1-resident)
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    bool ok = true;
    uint32_t u = 0;
    for (int kt = 0; kt < nt && ok; ++kt) {
      const int64_t j0 = c0 + (int64_t)kIxKeys * kt + 32 * kh;
      // the 32 entries' raw E8M0 block exponents (e_k + 127): ek0w / ek1w hold
      // those of blocks 0 / 1, entry j at byte j % 4 of word j / 4
      uint32_t ek0w[8], ek1w[8];
      {
        const uint8_t* src = p.ks + (b * p.N + j0) * 2;
        uint32_t raw[16];
        if (j0 + 32 <= p.N && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 x = __ldg(reinterpret_cast<const uint4*>(src) + i);
            raw[4 * i] = x.x;
            raw[4 * i + 1] = x.y;
            raw[4 * i + 2] = x.z;
            raw[4 * i + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint32_t word = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int64_t jj = 2 * i + e / 2;   // entry of byte 4 i + e
              word |= (j0 + jj < p.N ? (uint32_t)__ldg(src + 4 * i + e) : 127u) << (8 * e);
            }
            raw[i] = word;
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ek0w[i] = __byte_perm(raw[2 * i], raw[2 * i + 1], 0x6420);
          ek1w[i] = __byte_perm(raw[2 * i], raw[2 * i + 1], 0x7531);
        }
      }
      uint32_t lo0 = 255, hi0 = 0, lo1 = 255, hi1 = 0;   // exponent ranges of the tile's entries
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t x0 = (ek0w[j >> 2] >> (8 * (j & 3))) & 0xffu, x1 = (ek1w[j >> 2] >> (8 * (j & 3))) & 0xffu;
        lo0 = min(lo0, x0);
        hi0 = max(hi0, x0);
        lo1 = min(lo1, x1);
        hi1 = max(hi1, x1);
      }
      float sc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[j] = 0.0f;
      for (int h = 0; h < p.HI; ++h, ++u) {
        const uint32_t hb = u % kIxBufs;
        if (!mbar_wait(&ms->t_full[hb], (u / kIxBufs) & 1, kIxWait)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const int eq0 = __ldg(qerow + 2 * h), eq1 = __ldg(qerow + 2 * h + 1);
        const float wh = __ldg(wrow + h);
        // block b of entry j is scaled by 2^(e_qb + x_bj - 129), x = raw exponent
        // byte; when every such power lies in [2^-100, 2^100] one multiply by
        // it is exact, as is the two-step scale_pow2 otherwise
        const bool fast = eq0 + (int)lo0 >= 29 && eq0 + (int)hi0 <= 229 && eq1 + (int)lo1 >= 29 && eq1 + (int)hi1 <= 229;
        const int c0 = (eq0 - 2) << 23, c1 = (eq1 - 2) << 23;   // + (x << 23): fp32 bits of the power
#pragma unroll
        for (int half = 0; half < 2; ++half) {   // 16 entries at a time (registers)
          uint32_t P0[16], P1[16];
          tmem_ld32x16(tmem + lane_base + 128u * hb + 32u * kh + 16u * half, P0);
          tmem_ld32x16(tmem + lane_base + 128u * hb + 64u + 32u * kh + 16u * half, P1);
          tmem_wait_ld();
          if (half == 1) {   // the buffer is read: release it to the MMA warp
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms->t_empty[hb]);
          }
          if (fast) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = 16 * half + i;
              const int x0 = (int)((ek0w[j >> 2] >> (8 * (j & 3))) & 0xffu);
              const int x1 = (int)((ek1w[j >> 2] >> (8 * (j & 3))) & 0xffu);
              // both products are exact here, so one fma rounds their sum once, as the add did;
              // relu by fmaxf: a -0 can only add a zero product to a sum that starts at +0
              const float d = __fmaf_rn(__uint_as_float(P0[i]), __int_as_float(x0 * (1 << 23) + c0),
                                        __fmul_rn(__uint_as_float(P1[i]), __int_as_float(x1 * (1 << 23) + c1)));
              sc[j] = __fmaf_rn(wh, fmaxf(d, 0.0f), sc[j]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = 16 * half + i;
              const int x0 = (int)((ek0w[j >> 2] >> (8 * (j & 3))) & 0xffu);
              const int x1 = (int)((ek1w[j >> 2] >> (8 * (j & 3))) & 0xffu);
              const float d = __fadd_rn(scale_pow2(__uint_as_float(P0[i]), eq0 + x0 - 129),
                                        scale_pow2(__uint_as_float(P1[i]), eq1 + x1 - 129));
              sc[j] = __fmaf_rn(wh, d > 0.0f ? d : 0.0f, sc[j]);
            }
          }
        }
      }
      if (!ok) break;
      if (row_ok) {
        float* dst = p.scores + row * p.N + j0;
        if (j0 + 32 <= p.N && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0)) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(sc[j], sc[j + 1], sc[j + 2], sc[j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j0 + j < p.N) dst[j] = sc[j];
        }
      }
    }
    if (!ok && lane == 0) flag_timeout(p.ws);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kIxMma) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Decode scoring on the tensor cores: few query rows, long entry lists.
//
// The same numbers as above with the roles of the operands swapped: 128
// entries of one sequence form the MMA's M side (A, one row per entry), the
// row's quantised query the N side (B, one row per head, 16 rows), and
// kind::f8f6f4 takes the E2M1 codes as they are stored: a 16-element run of
// K is 8 bytes of packed codes followed by 8 bytes of padding in shared
// memory, so an entry's 32 code bytes become its operand row by four 8-byte
// asynchronous copies straight from global memory.  Products of E2M1 values
// are multiples of 1/4 and a block dot is below 2^11 in magnitude: exact in
// the fp32 accumulator.  Block b of all heads lands in TMEM columns
// 16 b .. 16 b + 15 of the tile's buffer.
//
// One CTA of 4 warps streams a chunk of entries through kDtSlots operand
// tile slots (two tiles share each 16 KiB stage: one in the first 64 bytes of
// every 128-byte row, one in the second): every thread copies its entry of
// tile u + kDtAhead while warp 0 issues the two block MMAs of tile u into one
// of four TMEM buffers and all threads combine tile u - kDtLag (thread =
// entry): loads, MMAs and the epilogue of different tiles overlap.  The
// chunk's scale bytes are staged once.  All
// waits have iteration limits; a thread whose wait expires records the
// timeout and stops, and the CTA waits (bounded) for its copies and MMAs
// before freeing TMEM.
// ---------------------------------------------------------------------------
namespace {

constexpr int kDtThreads = 128;             // entries per tile (MMA M) = threads
constexpr int kDtHeads = 16;                // MMA N
constexpr int kDtStages = 4;                // operand ring: 16 KiB stages of two tiles each
constexpr int kDtSlots = 2 * kDtStages;     // tile slots: tile u in slot u % kDtSlots
constexpr int kDtAhead = 5;                 // tiles whose copies are in flight ahead of the MMAs
constexpr int kDtTbufs = 4;                 // TMEM buffers of 32 columns
constexpr int kDtLag = 2;                   // tiles between a tile's MMAs and its epilogue
constexpr uint32_t kDtBOff = 0;             // query operand, 16 rows x 128 B
constexpr uint32_t kDtAOff = 2048;          // entry operand ring: kDtStages x [128 rows x 128 B]
constexpr int kDtMaxChunk = 4096;           // entries per CTA at most (their scale bytes are staged)
constexpr uint32_t kDtSOff = kDtAOff + kDtStages * 128 * 128;   // the chunk's scale bytes: kDtMaxChunk x 2 B
constexpr uint32_t kDtHOff = kDtSOff + kDtMaxChunk * 2;      // score histogram of the chunk: 2048 bins
constexpr int kDtHistBits = 11;
constexpr uint32_t kDtMiscOff = kDtHOff + (1u << kDtHistBits) * 4;
constexpr uint32_t kDtSmem = kDtMiscOff + 512 + 1024;   // + alignment slack

struct DtMisc {
  uint64_t full[kDtSlots], empty[kDtSlots], tfull[kDtTbufs], tempty[kDtTbufs];
  uint32_t tmem;
  int qlo0, qhi0, qlo1, qhi1;   // range of the query's block exponents over the heads
  int4 hx[kDtHeads];            // per head: {eq0 << 23, eq1 << 23, w bits, 0}
};
static_assert(sizeof(DtMisc) <= 512, "DtMisc overflows its smem slot");

// kind::f8f6f4 with E2M1 A and B (format 5), fp32 D, both K-major
__host__ __device__ constexpr uint32_t idesc_e2m1(int M, int N) {
  return (1u << 4) | (5u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f8f6f4_elect(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, 0, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc));
}

// byte offset of logical 16-byte chunk c of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// arrive on `bar` once this thread's copies so far have landed (counted arrival)
__device__ __forceinline__ void cp_async_arrive(void* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kDtThreads, 3)
scores_fp4_decode_tc_kernel(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                            const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks,
                            const int64_t* __restrict__ q_pos, int64_t Tq, int HI, int64_t N, int m,
                            int64_t chunk, float* __restrict__ scores, unsigned int* __restrict__ hist, void* ws) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DtMisc* ms = reinterpret_cast<DtMisc*>(sm + kDtMiscOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row = blockIdx.y;
  const int64_t b = row / Tq;
  const int64_t nv = visible(q_pos[row], m, N);
  const int64_t c0 = (int64_t)blockIdx.x * chunk;
  if (c0 >= nv) return;   // uniform
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  const int ntiles = (int)((c1 - c0 + kDtThreads - 1) / kDtThreads);

  // ---- set-up: zeroed operands (the padding bytes stay zero), barriers, TMEM ----
  for (int i = tid; i < (int)(kDtSOff / 16); i += kDtThreads) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  unsigned int* hist_s = reinterpret_cast<unsigned int*>(sm + kDtHOff);
  if (hist)
    for (int i = tid; i < (1 << kDtHistBits); i += kDtThreads) hist_s[i] = 0u;
  if (tid == 0) {
    for (int s = 0; s < kDtSlots; ++s) {
      mbar_init(&ms->full[s], kDtThreads);   // every thread's copies of the slot's tile
      mbar_init(&ms->empty[s], 1);           // the slot's MMAs completed
    }
    for (int i = 0; i < kDtTbufs; ++i) {
      mbar_init(&ms->tfull[i], 1);
      mbar_init(&ms->tempty[i], 4);          // one arrival per warp once it has read the buffer
    }
    mbar_fence_init();
    ms->qlo0 = ms->qlo1 = 1 << 30;
    ms->qhi0 = ms->qhi1 = -(1 << 30);
  }
  if (warp == 0) tmem_alloc(&ms->tmem, kDtTbufs * 32);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;

  // this thread's entry of tile u into slot u % kDtSlots -- stage slot / 2,
  // 16-byte units 4 (slot & 1) .. + 3 of its 128-byte operand row (the two
  // tiles of a stage share its rows): its 32 code bytes as four 8-byte
  // copies into the padded layout; then its counted arrival on the slot
  auto load_tile = [&](int u) {
    const int s = u % kDtSlots;
    int64_t j = c0 + (int64_t)u * kDtThreads + tid;
    j = j < c1 ? j : c0;   // past the chunk: any valid entry (its score is not stored)
    const uint8_t* src = kc + (b * N + j) * 32;
    const uint32_t a = smem_u32(sm + kDtAOff + (s >> 1) * 16384);
#pragma unroll
    for (int i = 0; i < 4; ++i) cp_async8(a + sw128_off(tid, 4 * (s & 1) + i), src + 8 * i);
    cp_async_arrive(&ms->full[s]);
  };
  bool ok = true;
  for (int u = 0; u < kDtAhead && u < ntiles; ++u) load_tile(u);
  // the chunk's scale bytes (two per entry), staged once: every load of the
  // thread in flight before the first store
  {
    uint16_t* sc_s = reinterpret_cast<uint16_t*>(sm + kDtSOff);
    const uint16_t* ks16 = reinterpret_cast<const uint16_t*>(ks) + b * N + c0;
    const int n = (int)(c1 - c0);
    uint16_t v[kDtMaxChunk / kDtThreads];
#pragma unroll
    for (int r = 0; r < kDtMaxChunk / kDtThreads; ++r) {
      const int i = tid + r * kDtThreads;
      v[r] = i < n ? __ldg(ks16 + i) : (uint16_t)0;
    }
#pragma unroll
    for (int r = 0; r < kDtMaxChunk / kDtThreads; ++r) {
      const int i = tid + r * kDtThreads;
      if (i < n) sc_s[i] = v[r];
    }
  }

  // ---- the query: MXFP4 codes into the B operand, block exponents ----
  // thread t: elements 4u .. 4u + 3 (u = t mod 8) of blocks t / 8 + 16 r
  for (int blkid = tid >> 3; blkid < 2 * kDtHeads; blkid += kDtThreads / 8) {
    const int u = tid & 7, h = blkid >> 1, blk = blkid & 1;
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
      uint32_t cd = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) cd |= e2m1_encode(__fmul_rn(v[i], inv)) << (4 * i);
      // element 32 blk + 4 u + i: run 2 blk + u / 4 of the head's row, data bytes 2 (u mod 4) .. + 1
      *reinterpret_cast<uint16_t*>(sm + kDtBOff + sw128_off(h, 2 * blk + (u >> 2)) + 2 * (u & 3)) = (uint16_t)cd;
      if (u == 0) {
        if (blk == 0) {
          atomicMin(&ms->qlo0, sx);
          atomicMax(&ms->qhi0, sx);
          ms->hx[h].x = sx << 23;
          ms->hx[h].z = __float_as_int(w[row * HI + h]);
        } else {
          atomicMin(&ms->qlo1, sx);
          atomicMax(&ms->qhi1, sx);
          ms->hx[h].y = sx << 23;
        }
      }
    }
  }
  fence_proxy_async();   // the query operand, written through the generic proxy
  fence_before_sync();
  __syncthreads();
  const int qlo0 = ms->qlo0, qhi0 = ms->qhi0, qlo1 = ms->qlo1, qhi1 = ms->qhi1;
  const uint32_t aA = smem_u32(sm + kDtAOff), aB = smem_u32(sm + kDtBOff);
  constexpr uint32_t id = idesc_e2m1(kDtThreads, kDtHeads);
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  int issued = 0;   // tiles whose MMAs warp 0 has issued

  // the epilogue of tile u: lane = entry, 16 heads x 2 blocks from TMEM
  auto combine = [&](int u) {
    const int tb = u % kDtTbufs;
    if (ok && !mbar_wait(&ms->tfull[tb], (uint32_t)(u / kDtTbufs) & 1, kIxWait)) ok = false;
    fence_after_sync();
    uint32_t P[32];
    tmem_ld32(tmem + lane_base + 32u * tb, P);
    tmem_wait_ld();
    fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->tempty[tb]);
    const int64_t jj = (int64_t)u * kDtThreads + tid;
    const uint32_t sc = jj < c1 - c0 ? reinterpret_cast<const uint16_t*>(sm + kDtSOff)[jj] : 0x7f7fu;
    const int x0 = (int)(sc & 0xffu), x1 = (int)(sc >> 8);
    const int X0 = x0 << 23, X1 = x1 << 23;
    // block b of head h is scaled by 2^(eq_bh + x_b - 127): one exact multiply
    // when every such power of the entry lies in [2^-100, 2^100]
    const bool fast = qlo0 + x0 >= 27 && qhi0 + x0 <= 227 && qlo1 + x1 >= 27 && qhi1 + x1 <= 227;
    float s = 0.0f;
    if (fast) {
#pragma unroll
      for (int h = 0; h < kDtHeads; ++h) {
        if (h < HI) {
          const int4 hx = ms->hx[h];
          const float d = __fmaf_rn(__uint_as_float(P[h]), __int_as_float(hx.x + X0),
                                    __fmul_rn(__uint_as_float(P[16 + h]), __int_as_float(hx.y + X1)));
          s = __fmaf_rn(__int_as_float(hx.z), fmaxf(d, 0.0f), s);
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < kDtHeads; ++h) {
        if (h < HI) {
          const int4 hx = ms->hx[h];
          const float d = __fadd_rn(scale_pow2(__uint_as_float(P[h]), (hx.x >> 23) + x0 - 127),
                                    scale_pow2(__uint_as_float(P[16 + h]), (hx.y >> 23) + x1 - 127));
          s = __fmaf_rn(__int_as_float(hx.z), d > 0.0f ? d : 0.0f, s);
        }
      }
    }
    const int64_t j = c0 + (int64_t)u * kDtThreads + tid;
    if (ok && j < c1) {
      scores[row * N + j] = s;
      if (hist) {   // the bin of its order key (top bits; -0 ranks as +0)
        uint32_t key = __float_as_uint(s);
        if (key == 0x80000000u) key = 0u;
        key = (key & 0x80000000u) ? ~key : (key | 0x80000000u);
        atomicAdd(hist_s + (key >> (32 - kDtHistBits)), 1u);
      }
    }
  };

  for (int u = 0; u < ntiles && ok; ++u) {
    // the copies of tile u + kDtAhead, once the MMAs of its slot's last tile are done
    const int ul = u + kDtAhead;
    if (ul < ntiles) {
      if (ul >= kDtSlots && !mbar_wait(&ms->empty[ul % kDtSlots], (uint32_t)(ul / kDtSlots - 1) & 1, kIxWait))
        ok = false;
      if (ok) load_tile(ul);
    }
    // warp 0: the two block MMAs of tile u into TMEM buffer u % kDtTbufs
    if (warp == 0 && ok) {
      const int s = u % kDtSlots, tb = u % kDtTbufs;
      bool got = mbar_wait(&ms->full[s], (uint32_t)(u / kDtSlots) & 1, kIxWait);
      if (got && u >= kDtTbufs) got = mbar_wait(&ms->tempty[tb], (uint32_t)(u / kDtTbufs - 1) & 1, kIxWait);
      if (got) {
        fence_after_sync();
        fence_proxy_async();   // the operand rows came through the generic proxy (cp.async)
        // the slot's tile starts 64 bytes into the rows for odd slots (K offset within the swizzle atom)
        const uint64_t ad = sdesc_sw128(aA + (s >> 1) * 16384, 16, 1024) + (uint64_t)(4 * (s & 1)),
                       bd = sdesc_sw128(aB, 16, 1024);
        const uint32_t d = tmem + 32u * tb;
        mma_f8f6f4_elect(d, ad, bd, id);
        mma_f8f6f4_elect(d + 16u, ad + 2, bd + 2, id);
        mma_commit_elect(&ms->tfull[tb]);
        mma_commit_elect(&ms->empty[s]);
        ++issued;
      } else {
        ok = false;
      }
      __syncwarp();
    }
    // the epilogue runs kDtLag tiles behind the MMAs (kDtLag < kDtTbufs)
    if (u >= kDtLag) combine(u - kDtLag);
  }
  for (int u = max(0, ntiles - kDtLag); u < ntiles && ok; ++u) combine(u);
  if (!ok) {
    if (lane == 0) flag_timeout(ws);
  }
  // this chunk's histogram into the row's
  if (hist) {
    __syncthreads();
    for (int i = tid; i < (1 << kDtHistBits); i += kDtThreads) {
      const unsigned int v = hist_s[i];
      if (v) atomicAdd(hist + row * (int64_t)(1 << kDtHistBits) + i, v);
    }
  }
  // copies and MMAs of this CTA land before its TMEM and shared memory go
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (warp == 0 && issued > 0) {
    const int u = issued - 1;
    mbar_wait(&ms->tfull[u % kDtTbufs], (uint32_t)(u / kDtTbufs) & 1, kIxWait);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kDtTbufs * 32);
  }
}

// ---------------------------------------------------------------------------
// The same decode scoring with the operand tiles brought in by TMA: the key
// codes viewed as rows of two entries (128 E2M1 values, 64 bytes), loaded
// with the tensor-map element type that writes every 16 packed values as 8
// bytes followed by an 8-byte gap -- the padded operand form above; the gaps
// are not written, and a box's transaction count is its global bytes -- so one
// box of 128 rows is 256 entries: entry 2r in bytes 0..63 of row r, entry
// 2r + 1 in bytes 64..127.  Four MMAs per tile (two entry parities x two
// blocks) into 64 TMEM columns; thread r of the epilogue combines entries 2r
// and 2r + 1 (two independent head chains).  Needs an even N (a row of the
// view never straddles two sequences).
// ---------------------------------------------------------------------------
namespace {

constexpr int kDmEntries = 256;             // entries per tile
constexpr int kDmEpiWarps = 8;              // epilogue: warp w reads TMEM lanes 32 (w % 4) .., entry parity w / 4
constexpr int kDmMmaWarp = 8;               // MMA issue
constexpr int kDmTmaWarp = 9;               // TMA boxes and L2 prefetches
constexpr int kDmThreads = 320;
constexpr int kDmEpi = 32 * kDmEpiWarps;    // epilogue threads
constexpr int kDmStages = 4;                // 16 KiB TMA boxes
constexpr int kDmTbufs = 4;                 // TMEM buffers of 64 columns
constexpr int kDmMaxChunk = 4096;           // entries per CTA at most (their scale bytes are staged)
constexpr uint32_t kDmBOff = 0;             // query operand, 16 rows x 128 B
constexpr uint32_t kDmAOff = 2048;          // kDmStages x [128 rows x 128 B]
constexpr uint32_t kDmSOff = kDmAOff + kDmStages * 16384;
constexpr uint32_t kDmHOff = kDmSOff + kDmMaxChunk * 2;
constexpr uint32_t kDmMiscOff = kDmHOff + (1u << kDtHistBits) * 4;
constexpr uint32_t kDmSmem = kDmMiscOff + 512 + 1024;

struct DmMisc {
  uint64_t full[kDmStages], empty[kDmStages], tfull[kDmTbufs], tempty[kDmTbufs], qready;
  uint32_t tmem;
  int qlo0, qhi0, qlo1, qhi1;
  int4 hx[kDtHeads];
};
static_assert(sizeof(DmMisc) <= 512, "DmMisc overflows its smem slot");

// the epilogue threads only
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDmEpi) : "memory"); }

}  // namespace

__global__ void __launch_bounds__(kDmThreads, 2)
scores_fp4_decode_tma_kernel(const __nv_bfloat16* __restrict__ qI, const float* __restrict__ w,
                             const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ks,
                             const int64_t* __restrict__ q_pos, int64_t Tq,
                             int HI, int64_t N, int m, int64_t chunk, float* __restrict__ scores,
                             unsigned int* __restrict__ hist, void* ws, const __grid_constant__ CUtensorMap tm_k) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DmMisc* ms = reinterpret_cast<DmMisc*>(sm + kDmMiscOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row = blockIdx.y;
  const int64_t b = row / Tq;
  const int64_t nv = visible(q_pos[row], m, N);
  const int64_t c0 = (int64_t)blockIdx.x * chunk;
  if (c0 >= nv) return;   // uniform
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  const int ntiles = (int)((c1 - c0 + kDmEntries - 1) / kDmEntries);
  const int64_t vrow0 = (b * N + c0) / 2;   // first row of the two-entry view
  const int n = (int)(c1 - c0);

  // threads 0..127: this thread's query values (a caller input), loaded
  // before the wait on the preceding kernel, in flight during the set-up
  uint16_t v[kDmMaxChunk / kDmEpi];
  float qv[2][4];
  if (warp < kDmEpiWarps) {
    if (tid < 128) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int blkid = (tid >> 3) + 16 * it, u = tid & 7, h = blkid >> 1, blk = blkid & 1;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          qv[it][i] = h < HI ? __bfloat162float(qI[(row * HI + h) * 64 + 32 * blk + 4 * u + i]) : 0.0f;
      }
    }
  }

  // the query operand and the key stages zeroed: TMA leaves the gaps of the padded form untouched
  for (int i = tid; i < (int)(kDmSOff / 16); i += kDmThreads) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  unsigned int* hist_s = reinterpret_cast<unsigned int*>(sm + kDmHOff);
  if (hist)
    for (int i = tid; i < (1 << kDtHistBits); i += kDmThreads) hist_s[i] = 0u;
  if (tid == 0) {
    for (int s = 0; s < kDmStages; ++s) {
      mbar_init(&ms->full[s], 1);
      mbar_init(&ms->empty[s], 1);
    }
    for (int i = 0; i < kDmTbufs; ++i) {
      mbar_init(&ms->tfull[i], 1);
      mbar_init(&ms->tempty[i], kDmEpiWarps);
    }
    mbar_init(&ms->qready, 128);
    mbar_fence_init();
    ms->qlo0 = ms->qlo1 = 1 << 30;
    ms->qhi0 = ms->qhi1 = -(1 << 30);
  }
  if (warp == 0) tmem_alloc(&ms->tmem, kDmTbufs * 64);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;
  bool ok = true;
  // the keys (codes and scales) may come from the preceding kernel
  pdl_wait();
  if (warp < kDmEpiWarps) {
    const uint16_t* ks16 = reinterpret_cast<const uint16_t*>(ks) + b * N + c0;
#pragma unroll
    for (int r = 0; r < kDmMaxChunk / kDmEpi; ++r) {
      const int i = tid + r * kDmEpi;
      v[r] = i < n ? __ldg(ks16 + i) : (uint16_t)0;
    }
  }

  if (warp == kDmTmaWarp) {
    // ---- TMA: tile u = one box of 128 view rows into stage u % kDmStages, once
    // the MMAs of the stage's previous tile are done; codes prefetched into L2
    // a stage set ahead (no shared memory held meanwhile) ----
    const uint32_t aA = smem_u32(sm + kDmAOff);
    auto prefetch_tile = [&](int u) {
      const int64_t e0 = (int64_t)u * kDmEntries;
      const int64_t ne = n - e0 < kDmEntries ? n - e0 : kDmEntries;
      prefetch_l2(kc + (b * N + c0 + e0) * 32, (uint32_t)ne * 32);
    };
    if (lane == 0) {
      for (int u = kDmStages; u < 2 * kDmStages && u < ntiles; ++u) prefetch_tile(u);
      int u = 0;
      for (; u < ntiles; ++u) {
        const int s = u % kDmStages;
        if (u >= kDmStages && !mbar_wait_backoff(&ms->empty[s], (uint32_t)(u / kDmStages - 1) & 1, kIxNapWait, 64)) break;
        mbar_arrive_expect_tx(&ms->full[s], 8192);   // the box's global bytes: the gaps are neither written nor counted
        tma_load_2d(aA + s * 16384, &tm_k, 0, (int)(vrow0 + (int64_t)u * (kDmEntries / 2)), &ms->full[s]);
        if (u >= kDmStages && u + kDmStages < ntiles) prefetch_tile(u + kDmStages);
      }
      if (u < ntiles) {
        ok = false;
        flag_timeout(ws);
      }
      // boxes issued land before shared memory goes (those the MMA warp consumed are done)
      for (int v2 = max(0, u - kDmStages); v2 < u; ++v2)
        mbar_wait(&ms->full[v2 % kDmStages], (uint32_t)(v2 / kDmStages) & 1, kIxWait);
    }
    __syncwarp();
  } else if (warp == kDmMmaWarp) {
    // ---- MMA issue: four per tile (two entry parities x two blocks) into TMEM buffer u % kDmTbufs ----
    const uint32_t aA = smem_u32(sm + kDmAOff), aB = smem_u32(sm + kDmBOff);
    constexpr uint32_t id = idesc_e2m1(kDtThreads, kDtHeads);
    int issued = 0;
    bool got = __all_sync(0xffffffffu, mbar_wait(&ms->qready, 0, kIxWait));
    for (int u = 0; u < ntiles && got; ++u) {
      const int s = u % kDmStages, tb = u % kDmTbufs;
      got = mbar_wait_backoff(&ms->full[s], (uint32_t)(u / kDmStages) & 1, kIxNapWait, 64);
      if (got && u >= kDmTbufs) got = mbar_wait_backoff(&ms->tempty[tb], (uint32_t)(u / kDmTbufs - 1) & 1, kIxNapWait, 64);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      fence_after_sync();
      const uint64_t ad = sdesc_sw128(aA + s * 16384, 16, 1024), bd = sdesc_sw128(aB, 16, 1024);
      const uint32_t d = tmem + 64u * tb;
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        mma_f8f6f4_elect(d + 32u * par, ad + (uint64_t)(4 * par), bd, id);
        mma_f8f6f4_elect(d + 32u * par + 16u, ad + (uint64_t)(4 * par + 2), bd + 2, id);
      }
      mma_commit_elect(&ms->tfull[tb]);
      mma_commit_elect(&ms->empty[s]);
      ++issued;
      __syncwarp();
    }
    if (!got) {
      ok = false;
      if (lane == 0) flag_timeout(ws);
    }
    // the MMAs issued complete before TMEM and shared memory go
    if (issued > 0) mbar_wait(&ms->tfull[(issued - 1) % kDmTbufs], (uint32_t)((issued - 1) / kDmTbufs) & 1, kIxWait);
  } else {
    // ---- threads 0..127: the query's MXFP4 codes into the B operand, block exponents ----
    uint16_t* sc_s = reinterpret_cast<uint16_t*>(sm + kDmSOff);
    if (tid < 128) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int blkid = (tid >> 3) + 16 * it, u = tid & 7, h = blkid >> 1, blk = blkid & 1;
        const bool act = h < HI;
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(qv[it][i]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int sx = mx_block_exp(amax);
        const float inv = pow2i(-sx);
        if (act) {
          uint32_t cd = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) cd |= e2m1_encode(__fmul_rn(qv[it][i], inv)) << (4 * i);
          *reinterpret_cast<uint16_t*>(sm + kDmBOff + sw128_off(h, 2 * blk + (u >> 2)) + 2 * (u & 3)) = (uint16_t)cd;
          if (u == 0) {
            if (blk == 0) {
              atomicMin(&ms->qlo0, sx);
              atomicMax(&ms->qhi0, sx);
              ms->hx[h].x = sx << 23;
              ms->hx[h].z = __float_as_int(w[row * HI + h]);
            } else {
              atomicMin(&ms->qlo1, sx);
              atomicMax(&ms->qhi1, sx);
              ms->hx[h].y = sx << 23;
            }
          }
        }
      }
      fence_proxy_async();
      mbar_arrive(&ms->qready);
    }
#pragma unroll
    for (int r = 0; r < kDmMaxChunk / kDmEpi; ++r) {
      const int i = tid + r * kDmEpi;
      if (i < n) sc_s[i] = v[r];
    }
    epi_sync();
    const int qlo0 = ms->qlo0, qhi0 = ms->qhi0, qlo1 = ms->qlo1, qhi1 = ms->qhi1;
    const int q4 = warp & 3, par = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int r = 32 * q4 + lane;   // view row of this thread: entry 2r + par
    // the heads' block exponents and weights, in registers for every tile
    int hx0[kDtHeads], hx1[kDtHeads];
    float hw[kDtHeads];
#pragma unroll
    for (int h = 0; h < kDtHeads; ++h) {
      const int4 hx = h < HI ? ms->hx[h] : make_int4(0, 0, 0, 0);   // past HI: exponent 0, weight +0
      hx0[h] = hx.x;
      hx1[h] = hx.y;
      hw[h] = __int_as_float(hx.z);
    }

    auto to_key_bin = [&](float sv) -> uint32_t {
      uint32_t key = __float_as_uint(sv);
      if (key == 0x80000000u) key = 0u;
      key = (key & 0x80000000u) ? ~key : (key | 0x80000000u);
      return key >> (32 - kDtHistBits);
    };
    // ---- the epilogue of every tile: this thread's entry from its 32 block dots ----
    for (int u = 0; u < ntiles && ok; ++u) {
      const int tb = u % kDmTbufs;
      ok = __all_sync(0xffffffffu, mbar_wait(&ms->tfull[tb], (uint32_t)(u / kDmTbufs) & 1, kIxWait));
      if (!ok) break;
      fence_after_sync();
      uint32_t P[32];
      tmem_ld32(tmem + lane_base + 64u * tb + 32u * par, P);
      tmem_wait_ld();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->tempty[tb]);
      const int64_t jl = (int64_t)u * kDmEntries + 2 * r + par;   // chunk-relative index of the entry
      const bool valid = jl < n;
      const uint32_t sc = valid ? (uint32_t)reinterpret_cast<const uint16_t*>(sm + kDmSOff)[jl] : 0x7f7fu;
      const int x0 = (int)(sc & 0xffu), x1 = (int)((sc >> 8) & 0xffu);
      float sv = 0.0f;
      if (qlo0 + x0 >= 27 && qhi0 + x0 <= 227 && qlo1 + x1 >= 27 && qhi1 + x1 <= 227) {
        const int X0 = x0 << 23, X1 = x1 << 23;
        // heads past HI: zero query codes (block dots 0) and weight 0, so
        // their terms add +0 to the non-negative sum -- no per-head branch
#pragma unroll
        for (int h = 0; h < kDtHeads; ++h) {
          const float d = __fmaf_rn(__uint_as_float(P[h]), __int_as_float(hx0[h] + X0),
                                    __fmul_rn(__uint_as_float(P[16 + h]), __int_as_float(hx1[h] + X1)));
          sv = __fmaf_rn(hw[h], fmaxf(d, 0.0f), sv);
        }
      } else {
#pragma unroll
        for (int h = 0; h < kDtHeads; ++h) {
          const float d = __fadd_rn(scale_pow2(__uint_as_float(P[h]), (hx0[h] >> 23) + x0 - 127),
                                    scale_pow2(__uint_as_float(P[16 + h]), (hx1[h] >> 23) + x1 - 127));
          sv = __fmaf_rn(hw[h], d > 0.0f ? d : 0.0f, sv);
        }
      }
      if (valid) {
        scores[row * N + c0 + jl] = sv;
        if (hist) atomicAdd(hist_s + to_key_bin(sv), 1u);
      }
    }
    if (!ok && lane == 0) flag_timeout(ws);
  }
  __syncthreads();
  if (hist) {
    for (int i = tid; i < (1 << kDtHistBits); i += kDmThreads) {
      const unsigned int hv = hist_s[i];
      if (hv) atomicAdd(hist + row * (int64_t)(1 << kDtHistBits) + i, hv);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem, kDmTbufs * 64);
  }
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn ix_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// byte rows of `width` bytes, boxes of 128 bytes x box_rows, 128-byte swizzle
bool ix_byte_map(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = ix_encode_fn();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool indexer_tc_applies(int B, int64_t Tq, int HI, int dI, int64_t N) {
  return Tq >= 64 && dI == 64 && HI >= 2 && HI <= kIxMaxHeads && HI % 2 == 0 && N > 0 &&
         (int64_t)B * Tq < INT32_MAX && (int64_t)B * N < INT32_MAX;
}

size_t indexer_tc_workspace(int B, int64_t Tq, int HI, int64_t N) {
  const size_t rows = (size_t)B * (size_t)Tq;
  return al256(rows * (size_t)HI * 64) + al256(rows * (size_t)HI * 2) + al256((size_t)B * (size_t)N * 128);
}

cudaError_t launch_indexer_scores_tc(const void* qI, const float* w, const uint8_t* kc, const uint8_t* ks,
                                     const int64_t* q_pos, int B, int64_t Tq, int HI, int64_t N, int m,
                                     float* scores, void* tc_ws, void* flags_ws, cudaStream_t st) {
  const int64_t rows = (int64_t)B * Tq;
  uint8_t* base = reinterpret_cast<uint8_t*>(tc_ws);
  uint8_t* qx = base;
  int8_t* qe = reinterpret_cast<int8_t*>(base + al256((size_t)rows * HI * 64));
  uint8_t* kx = base + al256((size_t)rows * HI * 64) + al256((size_t)rows * HI * 2);
  const int64_t nq = rows * HI * 2, nk = (int64_t)B * N * 8;
  launch_pdl(ix_quant_q_kernel, dim3((unsigned)((nq + 255) / 256)), dim3(256), 0, st, reinterpret_cast<const __nv_bfloat16*>(qI), rows,
                                                                 HI, qx, qe);
  launch_pdl(ix_expand_k_kernel, dim3((unsigned)((nk + 255) / 256)), dim3(256), 0, st, kc, (int64_t)B * N, kx);
  CUtensorMap tm_q, tm_k;
  if (!ix_byte_map(&tm_q, qx, (uint64_t)HI * 64, (uint64_t)rows, kIxRows)) return cudaErrorInvalidValue;
  if (!ix_byte_map(&tm_k, kx, 128, (uint64_t)B * N, kIxKeys)) return cudaErrorInvalidValue;
  IxParams p;
  p.qe = qe;
  p.w = w;
  p.ks = ks;
  p.q_pos = q_pos;
  p.Tq = Tq;
  p.N = N;
  p.HI = HI;
  p.m = m;
  p.scores = scores;
  p.ws = flags_ws;
  static PerDevice attr;
  smem_limit_once(attr, reinterpret_cast<const void*>(ix_scores_tc_kernel), (int)kIxSmem);
  const dim3 grid((unsigned)((N + kIxChunk - 1) / kIxChunk), (unsigned)((Tq + kIxRows - 1) / kIxRows), (unsigned)B);
  launch_pdl(ix_scores_tc_kernel, dim3(grid), dim3(kIxThreads), kIxSmem, st, p, tm_q, tm_k);
  return cudaGetLastError();
}

// Failure-detection self-test: one thread waits on an mbarrier whose phase
// nothing completes, with the same bounded wait every kernel here uses, and
// records the expiry in the workspace's status flags.
__global__ void wait_selftest_kernel(void* ws, uint32_t polls) {
  pdl_begin();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, polls)) flag_timeout(ws);
}

cudaError_t launch_wait_selftest(void* ws, uint32_t polls, cudaStream_t st) {
  launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, st, ws, polls);
  return cudaGetLastError();
}

bool decode_tc_applies(int64_t Tq, int HI, int dI, int64_t N) {
  return Tq <= 4 && dI == 64 && HI >= 1 && HI <= kDtHeads && N >= 8 * kDtThreads * 8;
}

cudaError_t launch_scores_fp4_decode_tc(const void* qI, const float* w, const uint8_t* kc, const uint8_t* ks,
                                        const int64_t* q_pos, int B, int64_t Tq, int HI, int64_t N, int m,
                                        float* scores, unsigned int* hist, void* flags_ws, cudaStream_t st) {
  static PerDevice attr, slots_dev;
  smem_limit_once(attr, reinterpret_cast<const void*>(scores_fp4_decode_tc_kernel), (int)kDtSmem);
  const int slots = slots_dev.get([] {
    int per = resident_ctas(reinterpret_cast<const void*>(scores_fp4_decode_tc_kernel), kDtThreads, kDtSmem);
    per = per > 4 ? 4 : per;   // 128 TMEM columns each: at most 4 per SM
    return device_sms() * per;
  });
  const int64_t rows = (int64_t)B * Tq;
  // chunks of whole tiles, about one CTA per resident slot, at least 2 tiles
  // and at most kDtMaxChunk entries each
  int64_t per_row = slots / rows;
  if (per_row < 1) per_row = 1;
  int64_t chunk = (N + per_row - 1) / per_row;
  chunk = (chunk + kDtThreads - 1) / kDtThreads * kDtThreads;
  if (chunk < 2 * kDtThreads) chunk = 2 * kDtThreads;
  if (chunk > kDtMaxChunk) chunk = kDtMaxChunk;
  // even N: the TMA-fed kernel (the two-entry view of the codes never
  // straddles two sequences); otherwise the copy-fed one
  CUtensorMap tm;
  if ((N & 1) == 0 && (reinterpret_cast<uintptr_t>(kc) & 31) == 0 && ix_encode_fn()) {
    const cuuint64_t dims[2] = {128, (cuuint64_t)((int64_t)B * N / 2)};
    const cuuint64_t strides[1] = {64};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    if (ix_encode_fn()(&tm, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(kc), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      static PerDevice attr_m, slots_m;
      smem_limit_once(attr_m, reinterpret_cast<const void*>(scores_fp4_decode_tma_kernel), (int)kDmSmem);
      const int sl = slots_m.get([] {
        int per = resident_ctas(reinterpret_cast<const void*>(scores_fp4_decode_tma_kernel), kDmThreads, kDmSmem);
        per = per > 2 ? 2 : per;   // 256 TMEM columns each: at most 2 per SM
        return device_sms() * per;
      });
      int64_t pr = sl / rows;
      if (pr < 1) pr = 1;
      int64_t ch = (N + pr - 1) / pr;
      ch = (ch + kDmEntries - 1) / kDmEntries * kDmEntries;
      if (ch < 2 * kDmEntries) ch = 2 * kDmEntries;
      if (ch > kDmMaxChunk) ch = kDmMaxChunk;
      const dim3 g2((unsigned)((N + ch - 1) / ch), (unsigned)rows);
      launch_pdl(scores_fp4_decode_tma_kernel, g2, dim3(kDmThreads), kDmSmem, st,
                 reinterpret_cast<const __nv_bfloat16*>(qI), w, kc, ks, q_pos, Tq, HI, N, m, ch, scores, hist, flags_ws,
                 tm);
      return cudaGetLastError();
    }
  }
  const dim3 grid((unsigned)((N + chunk - 1) / chunk), (unsigned)rows);
  launch_pdl(scores_fp4_decode_tc_kernel, dim3(grid), dim3(kDtThreads), kDtSmem, st, reinterpret_cast<const __nv_bfloat16*>(qI), w, kc,
                                                                 ks, q_pos, Tq, HI, N, m, chunk, scores, hist, flags_ws);
  return cudaGetLastError();
}

}  // namespace csa
