// attn_decode.cu -- attention of few query rows (decode) over their
// compressed entries and sliding window, mixed FP8/BF16 cache, in one launch.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）": MQA over
// the selected compressed entries plus a sliding-window branch; section
// "HCA（重度压缩注意力）": dense attention over all compressed entries;
// section "关键技术细节": RoPE on the last 64 dims with inverse rotation of
// the output, RoPE dims BF16 and the rest FP8 in the KV cache.
//
// The same arithmetic as attn_tc.cu (QK^T and PV on the tensor cores with
// bf16 operands, fp32 accumulation in TMEM, online softmax in the exp2
// domain with a lazy rescale), organised for a handful of rows: a row's
// keys are split over several CTAs (one work item = one row and one split of
// its 64-key tiles).  The keys of a tile reach shared memory one of two ways:
//  * gathered: decode_gather_kernel first writes every row's keys -- its
//    valid selected entries in idx order (invalid ones set the device-check
//    flag), or every visible entry, then its window tokens -- as contiguous
//    bf16 rows (exact expansion of the 592-byte rows), with many CTAs per
//    row, and each tile is one set of TMA boxes from them;
//  * expanded (items of few tiles): four producer warps load the tile's
//    592-byte rows into registers before its slot is free and write their
//    exact bf16 expansion into the slot, with a mask of the valid keys (an
//    invalid selected index is a masked slot).
// The query is loaded by TMA and its RoPE dims rotated to its position in
// shared memory by the softmax warps.  Each item normalises its partial
// output (bf16) and keeps its softmax statistics; the items of a row merge
// -- through one thread-block cluster's shared memory (many rows) or through
// global memory after a bounded per-row counter (few rows, many splits) --
// each item one slice of the row's dims over all splits in split order, with
// the RoPE dims rotated back.
// Every wait is bounded; on expiry the CTA records the timeout flag in the
// workspace, waits (bounded) for its own copies and MMAs and frees TMEM.
#include <cuda.h>

#include <cstring>

#include "attn_common.cuh"
#include "csa_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace csa {

using namespace tc;

namespace {

using namespace attn;

constexpr int kH = 64;
constexpr int kD = 512;
constexpr int kTile = 64;
constexpr int kThreads = 10 * 32;
constexpr int kMmaWarp = 8;       // query load, QK^T issue, TMEM owner
constexpr int kPvWarp = 9;        // PV issue

constexpr uint32_t kQOff = 0;                     // 8 chunks x [64 heads x 128 B]
constexpr uint32_t kKVOff = 65536;                // 2 slots x 8 chunks x [64 keys x 128 B]
constexpr uint32_t kPOff = kKVOff + 131072;       // 2 buffers x [64 heads x 64 keys bf16]
constexpr uint32_t kMiscOff = kPOff + 16384;      // barriers and per-head state
constexpr uint32_t kSmemBytes = 232448;           // 227 KiB
constexpr int kMaxK = 4096;                       // selected entries per row at most

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;       // O^T: 4 blocks of 64 columns (heads); lanes = dims
constexpr uint32_t kTmemS = 256;     // S: 2 buffers of 64 columns (keys); M = 64 layout

constexpr uint32_t kWaitLimit = 1u << 20;     // suspending polls of one mbarrier wait
constexpr int kMaxSplits = 16;                // splits of a row = CTAs of one cluster (cluster merge)
constexpr int kClusterMergeMax = 8;           // rows needing more splits than this merge through global memory
constexpr uint32_t kGridWaitLimit = 1u << 22; // polls of the row counter (64 ns naps; global merge)
constexpr float kLazy = 8.0f;

struct Misc {
  uint64_t kv_full[2], kv_empty[2], s_full[2], p_full[2];
  uint64_t q_full, q_ready, o_full, drain[2], recv, merge_in;
  int go;                           // the row counter reached every split (global merge)
  uint32_t kmask[2][2];             // per KV slot: which of its 64 keys are valid (bits)
  uint32_t tmem;
  int abort;
  alignas(16) float alpha[2][kH];   // per-head rescale factors of a tile, double-buffered
};
static_assert(sizeof(Misc) <= 2048, "Misc overflows its smem slot");
static_assert(offsetof(Misc, alpha) % 16 == 0, "vector reads of Misc");

__device__ __forceinline__ bool vabort(const Misc* ms) {
  return *reinterpret_cast<const volatile int*>(&ms->abort) != 0;
}


struct DParams {
  const __nv_bfloat16* q;   // [rows, 64, 512]
  const int64_t* q_pos;
  int64_t Tq;
  const uint8_t* cache;     // [B, N, 592]
  int64_t N;
  int m;
  const int32_t* idx;       // [rows, k] or NULL (dense: every visible entry)
  int k;
  const uint8_t* swa;       // [B, Ts, 592]
  const int64_t* swa_pos0;
  int64_t Ts;
  int W;
  float scale_log2;
  const float* rcos;
  const float* rsin;
  int64_t rope_rows;
  __nv_bfloat16* out;       // [rows, 64, 512]
  float* lse;               // [rows, 64] or NULL
  void* ws;                 // status flags
  int nsplit;               // items per row (the cluster size when they merge through shared memory)
  int expand;               // the producers expand the cache rows themselves (no gathered rows)
  __nv_bfloat16* part_o;    // global merge: [items, 512 dims, 64 heads] normalised partial outputs
  float* part_ml;           // global merge: [items, 64, 2] running max (log2 units), sum
  int* arrive;              // global merge: [rows] items that finished their partial (zero at launch)
  __nv_bfloat16* xg;        // [rows, kp, 512] every row's keys in bf16, in order, zero past them
  int64_t kp;               // key slots per row of xg (a multiple of the tile)
  int* ecount;              // [rows] valid selected entries of each row (sparse)
};

// ---------------------------------------------------------------------------
// Per row, ahead of the attention: the row's keys -- its valid selected
// entries in idx order (or every visible entry), then its window tokens --
// expanded exactly from the 592-byte rows to bf16 rows of xg, 64 per CTA
// (grid: the row's key tiles x rows), with zeros past the row's keys in its
// last tile.  A sparse row's CTAs each find the valid entries of their tile
// from idx (a block-wide count of the valid ones before each position);
// invalid indices set the device-check flag (tile 0's CTA) and are skipped.
// ---------------------------------------------------------------------------
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
decode_gather_kernel(const DParams p) {
  pdl_begin();
  __shared__ int32_t src_s[kTile];            // this tile's selected entries
  __shared__ unsigned int wcnt_s[kGatherThreads / 32];
  __shared__ int ne_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const int64_t row = blockIdx.y;
  const int64_t b = row / p.Tq;
  const int64_t t = p.q_pos[row];
  const bool t_ok = t >= 0 && t < p.rope_rows;
  const bool dense = p.idx == nullptr;
  int ne = 0;
  if (t_ok && dense) {
    const int64_t nv = (t + 1) / p.m;
    ne = (int)(nv < p.N ? nv : p.N);
  } else if (t_ok) {
    // thread tid owns idx entries [16 tid, 16 tid + 16): valid ones counted,
    // their ranks found by a block-wide exclusive scan of the counts
    constexpr int kPer = 16;   // k <= 4096 = 256 x 16
    const int32_t* ir = p.idx + row * (int64_t)p.k;
    int32_t js[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = kPer * tid + r;
      js[r] = i < p.k ? __ldg(ir + i) : -1;
    }
    uint32_t okbits = 0;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int32_t j = js[r];
      const bool ok = j >= 0 && (int64_t)j < p.N && (int64_t)(j + 1) * p.m - 1 <= t;
      if (tile == 0 && j >= 0 && !ok) flag_device_check(p.ws, (unsigned)j);
      okbits |= ok ? 1u << r : 0u;
    }
    const unsigned int own = __popc(okbits);
    unsigned int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wcnt_s[warp] = incl;
    __syncthreads();
    unsigned int before = 0, total = 0;
    for (int w2 = 0; w2 < kGatherThreads / 32; ++w2) {
      if (w2 < warp) before += wcnt_s[w2];
      total += wcnt_s[w2];
    }
    unsigned int pos = before + incl - own;
    const int lo = tile * kTile;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      if ((okbits >> r) & 1u) {
        if ((int)pos >= lo && (int)pos < lo + kTile) src_s[pos - lo] = js[r];
        ++pos;
      }
    }
    ne = (int)total;
    if (tile == 0 && tid == 0) p.ecount[row] = ne;
  }
  if (dense && tile == 0 && tid == 0) p.ecount[row] = ne;
  if (tid == 0) ne_s = ne;
  __syncthreads();
  ne = ne_s;
  const int64_t u_lo = t - p.W + 1 < 0 ? 0 : t - p.W + 1;
  const int64_t p0 = p.W > 0 ? p.swa_pos0[b] : 0;
  const int64_t w_lo = u_lo < p0 ? p0 : u_lo;
  const int64_t w_hi = t < p0 + p.Ts - 1 ? t : p0 + p.Ts - 1;
  const int nwin = (t_ok && p.W > 0 && w_hi >= w_lo) ? (int)(w_hi - w_lo + 1) : 0;
  const int nkeys = ne + nwin;
  if (tile * kTile >= nkeys) return;   // past the row's keys (uniform)
  // warp w: slots 8 w .. 8 w + 7 of the tile; all eight rows' loads in flight together
  uint4 c[8];
  float sc[8];
  uint4 rp[8][2];
  bool have[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int key = tile * kTile + 8 * warp + i;
    const uint8_t* rowp = nullptr;
    if (key < ne) rowp = p.cache + (b * p.N + (dense ? (int64_t)key : (int64_t)src_s[key - tile * kTile])) * kMixRow;
    else if (key < nkeys) rowp = p.swa + (b * p.Ts + (w_lo - p0 + (key - ne))) * kMixRow;
    have[i] = rowp != nullptr;
    c[i] = make_uint4(0, 0, 0, 0);
    sc[i] = 0.0f;
    rp[i][0] = rp[i][1] = make_uint4(0, 0, 0, 0);
    if (rowp) {
      if (lane < 28) {
        c[i] = __ldg(reinterpret_cast<const uint4*>(rowp) + lane);
        sc[i] = __ldg(reinterpret_cast<const float*>(rowp + kMixScaleOff) + (lane >> 3));
      } else {
        rp[i][0] = __ldg(reinterpret_cast<const uint4*>(rowp + kMixRopeOff) + 2 * (lane - 28));
        rp[i][1] = __ldg(reinterpret_cast<const uint4*>(rowp + kMixRopeOff) + 2 * (lane - 28) + 1);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int key = tile * kTile + 8 * warp + i;
    uint4* dst = reinterpret_cast<uint4*>(p.xg + (row * p.kp + key) * kD);
    if (lane < 28) {
      uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
      if (have[i]) dequant16(c[i], sc[i], o0, o1);
      dst[2 * lane] = o0;
      dst[2 * lane + 1] = o1;
    } else {
      dst[56 + 2 * (lane - 28)] = rp[i][0];
      dst[56 + 2 * (lane - 28) + 1] = rp[i][1];
    }
  }
}

// The merge of one dim slice [d0, d0 + nd) of a row over its ns splits:
// rows[(c stride + dl) 128 bytes] holds split c's partial row of dim d0 + dl
// (64 heads bf16; 16-byte chunk g at g ^ (d mod 8) when `swz`, else at g).
// Thread: a pair of dims (d, d + 1) of eight heads, weighted sum in split
// order, times 1 / L, RoPE dims rotated back, stored to out_row [64][512].
__device__ __forceinline__ void merge_slice(const uint8_t* rows, uint32_t stride, bool swz, int ns, int d0, int nd,
                                            const float* wgt, const float* Linv, const float* cs, const float* sn,
                                            __nv_bfloat16* out_row) {
  for (int u = threadIdx.x; u < (nd >> 1) * 8; u += kThreads) {
    const int hg = u & 7, dl = 2 * (u >> 3), d = d0 + dl;
    const uint32_t k0 = (((uint32_t)hg) ^ (swz ? ((uint32_t)d & 7u) : 0u)) << 4;
    const uint32_t k1 = (((uint32_t)hg) ^ (swz ? ((uint32_t)(d + 1) & 7u) : 0u)) << 4;
    float o0[8], o1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o0[j] = o1[j] = 0.0f;
#pragma unroll 4
    for (int c = 0; c < ns; ++c) {
      const uint8_t* rr = rows + ((uint32_t)c * stride + (uint32_t)dl) * 128u;
      const uint4 x0 = *reinterpret_cast<const uint4*>(rr + k0);
      const uint4 x1 = *reinterpret_cast<const uint4*>(rr + 128 + k1);
      const float4 wa = *reinterpret_cast<const float4*>(wgt + c * kH + 8 * hg);
      const float4 wb = *reinterpret_cast<const float4*>(wgt + c * kH + 8 * hg + 4);
      const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      const uint32_t a0[4] = {x0.x, x0.y, x0.z, x0.w}, a1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a0[j]));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a1[j]));
        o0[2 * j] = __fmaf_rn(w[2 * j], f0.x, o0[2 * j]);
        o0[2 * j + 1] = __fmaf_rn(w[2 * j + 1], f0.y, o0[2 * j + 1]);
        o1[2 * j] = __fmaf_rn(w[2 * j], f1.x, o1[2 * j]);
        o1[2 * j + 1] = __fmaf_rn(w[2 * j + 1], f1.y, o1[2 * j + 1]);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int h = 8 * hg + j;
      float y0 = o0[j] * Linv[h], y1 = o1[j] * Linv[h];
      if (d >= kMixDn) {
        const int pi = (d - kMixDn) >> 1;
        const float z0 = y0 * cs[pi] + y1 * sn[pi];
        const float z1 = -y0 * sn[pi] + y1 * cs[pi];
        y0 = z0;
        y1 = z1;
      }
      *reinterpret_cast<__nv_bfloat162*>(out_row + h * (int64_t)kD + d) = __floats2bfloat162_rn(y0, y1);
    }
  }
}

// kCluster: the items of a row are one thread-block cluster and merge through
// each other's shared memory; otherwise they write their partials to global
// memory, meet at a per-row counter (cooperative launch) and merge from there.
// kExpand: the producers expand the cache rows themselves (a mask marks the
// valid keys of each tile); otherwise they load rows gathered ahead.
template <bool kCluster, bool kExpand>
__global__ void __launch_bounds__(kThreads, 1)
attn_decode_kernel(const DParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_xg, const __grid_constant__ CUtensorMap tm_po) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kQOff;
  uint8_t* sKV = sm + kKVOff;
  uint8_t* sP = sm + kPOff;
  Misc* ms = reinterpret_cast<Misc*>(sm + kMiscOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t item = blockIdx.x;
  const int64_t row = item / p.nsplit;
  const int split = (int)(item - row * p.nsplit);
  const int64_t b = row / p.Tq;
  const int64_t t = p.q_pos[row];
  const bool t_ok = t >= 0 && t < p.rope_rows;
  const bool dense = p.idx == nullptr;
  // the RoPE row of t for the merge's inverse rotation, loaded now (threads 64..95)
  float rope_c = 0.0f, rope_s = 0.0f;
  if (tid >= 64 && tid < 96) {
    rope_c = p.rcos[(t_ok ? t : 0) * 32 + tid - 64];
    rope_s = p.rsin[(t_ok ? t : 0) * 32 + tid - 64];
  }

  if (tid == 0) {
    ms->abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->kv_full[i], kExpand ? 4 : 1);   // expanding: one arrival per producer warp; else the TMA boxes
      mbar_init(&ms->kv_empty[i], 1);
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->p_full[i], 4);
    }
    mbar_init(&ms->q_full, 1);
    mbar_init(&ms->q_ready, 4);
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->drain[0], 1);
    mbar_init(&ms->drain[1], 1);
    mbar_init(&ms->recv, 1);          // the row's partial slices and statistics pushed by its items
    mbar_init(&ms->merge_in, 1);
    ms->go = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ms->tmem, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;

  // ---- the query: 8 TMA boxes (a caller input: issued before the wait) ----
  if (warp == kMmaWarp) {
    if (lane == 0) mbar_arrive_expect_tx(&ms->q_full, kH * kD * 2);
    __syncwarp();
    if (lane < 8) tma_load_2d(smem_u32(sQ) + lane * 8192, &tm_q, 64 * lane, (int)(row * kH), &ms->q_full);
    __syncwarp();
  }
  // the gathered rows, their counts and the row counters come from the
  // preceding launches
  pdl_wait();
  // ---- this item's keys: entries first, then the window tokens ----
  // key slots: the visible entries (dense) or the row's valid selected
  // entries (gathered) or all k selected positions (expanded here: an
  // invalid index is a masked slot), then the window tokens
  int ne = 0;
  if (t_ok) {
    if (dense) {
      const int64_t nv = (t + 1) / p.m;
      ne = (int)(nv < p.N ? nv : p.N);
    } else {
      ne = kExpand ? p.k : p.ecount[row];
    }
  }
  const int64_t u_lo = t - p.W + 1 < 0 ? 0 : t - p.W + 1;
  const int64_t p0 = p.W > 0 ? p.swa_pos0[b] : 0;
  const int64_t w_lo = u_lo < p0 ? p0 : u_lo;
  const int64_t w_hi = t < p0 + p.Ts - 1 ? t : p0 + p.Ts - 1;
  const int nwin = (t_ok && p.W > 0 && w_hi >= w_lo) ? (int)(w_hi - w_lo + 1) : 0;
  if (tid == 0 && split == 0) {
    if (!t_ok) flag_device_check(p.ws, 0x40000000u);
    if (t_ok && p.W > 0 && nwin < t - u_lo + 1) flag_device_check(p.ws, 0x80000000u);
  }
  const int nkeys = ne + nwin;
  const int ntiles = (nkeys + kTile - 1) / kTile;
  const int per = (ntiles + p.nsplit - 1) / p.nsplit;
  const int tlo = min(ntiles, split * per);
  const int thi = min(ntiles, tlo + per);
  const int key_hi = min(nkeys, thi * kTile);
  bool fail = false;

  if (warp >= 4 && warp < 8) {
    if constexpr (kExpand) {
      // ================================ producers ================================
      // Warp pw expands rows 16 pw .. 16 pw + 15 of each 64-key tile from the
      // 592-byte cache rows straight into the tile's shared-memory slot (bf16,
      // 128-byte swizzle, 8 column boxes of 64 dims): lane l takes the FP8 16-byte
      // chunks l + 32 m (m < 14) of the warp's 16 x 28 and the bf16 RoPE chunks
      // l + 32 m (m < 4) of its 16 x 8.  All of a tile's loads are issued into
      // registers before the slot is free (they fly while earlier tiles compute).
      const int pw = warp - 4;
      uint32_t g = 0;
      bool ok = true;
      for (int tl = tlo; tl < thi && ok && !vabort(ms); ++tl, ++g) {
        const int buf = g & 1;
        // this warp's 16 rows: lane i < 16 resolves key slot 64 tl + 16 pw + i
        const uint8_t* myrow = nullptr;
        bool myok = false;
        if (lane < 16) {
          const int key = tl * kTile + 16 * pw + lane;
          if (key < ne) {
            int64_t j = key;
            bool v = true;
            if (!dense) {
              j = __ldg(p.idx + row * (int64_t)p.k + key);
              v = j >= 0 && j < p.N && (j + 1) * p.m - 1 <= t;
              if (!v && j >= 0) flag_device_check(p.ws, (unsigned)j);
            }
            if (v) myrow = p.cache + (b * p.N + j) * kMixRow;
          } else if (key < nkeys) {
            myrow = p.swa + (b * p.Ts + (w_lo - p0 + (key - ne))) * kMixRow;
          }
          myok = myrow != nullptr;
        }
        const uint32_t vbits = __ballot_sync(0xffffffffu, myok) & 0xffffu;
        uint4 c[14];
        float sc[14];
        uint4 rp[4];
#pragma unroll
        for (int m = 0; m < 14; ++m) {
          const int f = lane + 32 * m, rr = f / 28, ch = f - 28 * rr;
          const uint64_t rw = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(myrow), rr);
          const uint8_t* r = reinterpret_cast<const uint8_t*>(rw);
          c[m] = make_uint4(0, 0, 0, 0);
          sc[m] = 0.0f;
          if (r) {
            c[m] = __ldg(reinterpret_cast<const uint4*>(r) + ch);
            sc[m] = __ldg(reinterpret_cast<const float*>(r + kMixScaleOff) + (ch >> 3));
          }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int f = lane + 32 * m, rr = f >> 3, ch = f & 7;
          const uint64_t rw = __shfl_sync(0xffffffffu, reinterpret_cast<uint64_t>(myrow), rr);
          const uint8_t* r = reinterpret_cast<const uint8_t*>(rw);
          rp[m] = r ? __ldg(reinterpret_cast<const uint4*>(r + kMixRopeOff) + ch) : make_uint4(0, 0, 0, 0);
        }
        if (g >= 2 && !mbar_wait(&ms->kv_empty[buf], ((g >> 1) - 1) & 1, kWaitLimit)) {
          ok = false;
          break;
        }
        uint8_t* kv = sKV + buf * 65536;
#pragma unroll
        for (int m = 0; m < 14; ++m) {
          const int f = lane + 32 * m, rr = f / 28, ch = f - 28 * rr;
          const uint32_t r = (uint32_t)(16 * pw + rr);
          uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
          if ((vbits >> rr) & 1u) dequant16(c[m], sc[m], o0, o1);
          uint8_t* box = kv + (ch >> 2) * 8192;
          *reinterpret_cast<uint4*>(box + sw128(r, 2u * (ch & 3))) = o0;
          *reinterpret_cast<uint4*>(box + sw128(r, 2u * (ch & 3) + 1)) = o1;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int f = lane + 32 * m, rr = f >> 3, ch = f & 7;
          *reinterpret_cast<uint4*>(kv + 7 * 8192 + sw128((uint32_t)(16 * pw + rr), (uint32_t)ch)) = rp[m];
        }
        if (lane == 0) reinterpret_cast<uint16_t*>(&ms->kmask[buf][0])[pw] = (uint16_t)vbits;
        fence_proxy_async();   // the rows were written through the generic proxy; the MMAs read them
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms->kv_full[buf]);
      }
      if (!ok) {
        ms->abort = 1;
        if (lane == 0) flag_timeout(p.ws);
        fail = true;
      }
    } else {
      // ================================ producers ================================
      // the row's keys are contiguous bf16 rows of xg: 8 TMA boxes of 64 rows x
      // 64 columns per tile, from producer warp 0 (the tile's other warps idle)
      const int pw = warp - 4;
      uint32_t g = 0;
      bool ok = true;
      if (pw == 0) {
        for (int tl = tlo; tl < thi && ok && !vabort(ms); ++tl, ++g) {
          const int buf = g & 1;
          if (g >= 2 && !mbar_wait(&ms->kv_empty[buf], ((g >> 1) - 1) & 1, kWaitLimit)) {
            ok = false;
            break;
          }
          const uint32_t tb = smem_u32(sKV + buf * 65536);
          if (lane == 0) mbar_arrive_expect_tx(&ms->kv_full[buf], kTile * kD * 2);
          __syncwarp();
          if (lane < 8)
            tma_load_2d(tb + lane * 8192, &tm_xg, 64 * lane, (int)(row * p.kp + (int64_t)tl * kTile), &ms->kv_full[buf]);
          __syncwarp();
        }
        if (!ok) {
          ms->abort = 1;
          if (lane == 0) flag_timeout(p.ws);
          fail = true;
        }
        // the copies of this warp land before the CTA can exit
        if (g > 0) mbar_wait(&ms->kv_full[(g - 1) & 1], ((g - 1) >> 1) & 1, kWaitLimit);
      }
    }
  } else if (warp == kMmaWarp) {
    // ============================== QK^T issue ==============================
    const uint32_t aQ = smem_u32(sQ), aKV = smem_u32(sKV);
    constexpr uint32_t idQK = idesc_bf16(64, kTile, 0, 0);
    bool ok = mbar_wait(&ms->q_full, 0, kWaitLimit) && mbar_wait(&ms->q_ready, 0, kWaitLimit);
    uint32_t g = 0;
    for (int tl = tlo; tl < thi && ok && !vabort(ms); ++tl, ++g) {
      // S buffer g & 1 is free once the softmax of tile g - 2 has made its P
      if (g >= 2 && !mbar_wait(&ms->p_full[g & 1], ((g >> 1) - 1) & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      if (!mbar_wait(&ms->kv_full[g & 1], (g >> 1) & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint32_t dS = tmem + kTmemS + 64u * (g & 1);
      const uint64_t qd0 = sdesc_sw128(aQ, 16, 1024);
      const uint64_t kd0 = sdesc_sw128(aKV + (g & 1) * 65536, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
        mma_bf16_elect(dS, qd0 + off, kd0 + off, idQK, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&ms->s_full[g & 1]);
      __syncwarp();
    }
    if (!ok) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
      fail = true;
      mbar_wait(&ms->q_full, 0, kWaitLimit);   // the query copy in flight
    }
    mma_commit_elect(&ms->drain[0]);
    __syncwarp();
    mbar_wait(&ms->drain[0], 0, kWaitLimit);
  } else if (warp == kPvWarp) {
    // ================================ PV issue ================================
    const uint32_t aKV = smem_u32(sKV), aP = smem_u32(sP);
    constexpr uint32_t idPV = idesc_bf16(128, kH, 1, 0);
    uint32_t g = 0;
    bool ok = true;
    for (int tl = tlo; tl < thi && ok && !vabort(ms); ++tl, ++g) {
      if (!mbar_wait(&ms->p_full[g & 1], (g >> 1) & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint64_t vd0 = sdesc_sw128(aKV + (g & 1) * 65536, 8192, 1024);
      const uint64_t pd0 = sdesc_sw128(aP + (g & 1) * 8192, 16, 1024);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          mma_bf16_elect(tmem + kTmemO + 64u * mt, vd0 + (uint64_t)((2 * mt * 8192 + ks * 2048) >> 4),
                         pd0 + (uint64_t)((ks * 32) >> 4), idPV, (tl > tlo || ks > 0) ? 1u : 0u);
      }
      mma_commit_elect(&ms->kv_empty[g & 1]);
      if (tl == thi - 1) mma_commit_elect(&ms->o_full);
      __syncwarp();
    }
    if (!ok) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
      fail = true;
    }
    mma_commit_elect(&ms->drain[1]);
    __syncwarp();
    mbar_wait(&ms->drain[1], 0, kWaitLimit);
  } else {
    // ============================ softmax / epilogue ============================
    const int qd = warp;
    const int cq = 2 * (lane & 3);
    const int ha = 16 * qd + (lane >> 2), hb = ha + 8;
    const bool leader = (lane & 3) == 0;
    const uint32_t tq_lane = (uint32_t)(32 * qd) << 16;
    // the query's RoPE dims (chunk 7) rotated to position t, in place:
    // thread tid takes head tid / 2, pairs 16 (tid & 1) .. + 15
    float csr[16], snr[16];   // cos / sin of this thread's 16 pairs, loaded while the query is in flight
    {
      const float* cs = p.rcos + (t_ok ? t : 0) * 32 + 16 * (tid & 1);
      const float* sn = p.rsin + (t_ok ? t : 0) * 32 + 16 * (tid & 1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        csr[i] = __ldg(cs + i);
        snr[i] = __ldg(sn + i);
      }
    }
    if (mbar_wait(&ms->q_full, 0, kWaitLimit)) {
      const int h = tid >> 1;
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        const int u = 4 * (tid & 1) + uu;      // 16-byte unit: pairs 4u .. 4u + 3
        uint4* a = reinterpret_cast<uint4*>(sQ + 7 * 8192 + sw128((uint32_t)h, (uint32_t)u));
        uint4 v = *a;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
          const float c = csr[4 * uu + e], s = snr[4 * uu + e];
          const float y0 = __fsub_rn(__fmul_rn(f.x, c), __fmul_rn(f.y, s));
          const float y1 = __fadd_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, c));
          const __nv_bfloat162 r2 = __floats2bfloat162_rn(y0, y1);
          w[e] = *reinterpret_cast<const uint32_t*>(&r2);
        }
        *a = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      fail = true;
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms->q_ready);
    float ma = -INFINITY, mb = -INFINITY, la = 0.0f, lb = 0.0f;
    uint32_t g = 0;
    bool stop = false;
    for (int tl = tlo; tl < thi; ++tl, ++g) {
      if (!fail && !mbar_wait(&ms->s_full[g & 1], (g >> 1) & 1, kWaitLimit)) fail = true;
      // the tile's valid keys: the expanding producers' mask (published with
      // kv_full; S being ready implies it), or those below the item's end
      uint64_t kmask;
      if constexpr (kExpand) {
        if (!fail && !mbar_wait(&ms->kv_full[g & 1], (g >> 1) & 1, kWaitLimit)) fail = true;
        fence_after_sync();
        kmask = (uint64_t)ms->kmask[g & 1][0] | ((uint64_t)ms->kmask[g & 1][1] << 32);
      } else {
        fence_after_sync();
        const int nvalid = min(kTile, key_hi - tl * kTile);
        kmask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
      }
      uint32_t v[32];
      tmem_ld16x256b_x8(tmem + tq_lane + kTmemS + 64u * (g & 1), v);
      tmem_wait_ld();
      float xa[16], xb[16];
      float ta = -INFINITY, tb = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool valid = (kmask >> (8 * j + cq + e)) & 1ull;
          xa[2 * j + e] = valid ? __uint_as_float(v[4 * j + e]) * p.scale_log2 : -INFINITY;
          xb[2 * j + e] = valid ? __uint_as_float(v[4 * j + 2 + e]) * p.scale_log2 : -INFINITY;
          ta = fmaxf(ta, xa[2 * j + e]);
          tb = fmaxf(tb, xb[2 * j + e]);
        }
      }
      ta = fmaxf(ta, __shfl_xor_sync(0xffffffffu, ta, 1));
      ta = fmaxf(ta, __shfl_xor_sync(0xffffffffu, ta, 2));
      tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, 1));
      tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, 2));
      const bool need_a = ta > ma + kLazy, need_b = tb > mb + kLazy;
      const float na = need_a ? ta : ma, nb = need_b ? tb : mb;
      const float aa = need_a ? ex2(ma - na) : 1.0f;
      const float ab = need_b ? ex2(mb - nb) : 1.0f;
      if (tl > tlo) {
        if (leader) {
          ms->alpha[g & 1][ha] = aa;
          ms->alpha[g & 1][hb] = ab;
        }
        // one vote per warp that must rescale, 32 per warp that failed
        const bool wfail = __any_sync(0xffffffffu, fail || vabort(ms));
        const bool wresc = __any_sync(0xffffffffu, need_a || need_b);
        const uint32_t votes = group_vote(wfail || (lane == 0 && wresc));
        if (votes >= 32) {
          stop = true;
          break;
        }
        if (votes > 0) {
          // the previous tile's PV must be complete before O^T is touched
          const uint32_t gv = g - 1;
          if (!fail && !mbar_wait(&ms->kv_empty[gv & 1], (gv >> 1) & 1, kWaitLimit)) fail = true;
          fence_after_sync();
          if (!fail) {
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t o[32];
              const uint32_t oa = tmem + tq_lane + kTmemO + 32u * c;
              tmem_ld32(oa, o);
              tmem_wait_ld();
              const float* al = ms->alpha[g & 1] + 32 * (c & 1);
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * al[j]);
              tmem_st32(oa, o);
            }
            tmem_wait_st();
          }
        }
      }
      ma = na;
      mb = nb;
      // P buffer g & 1 was last read by PV of tile g - 2
      if (g >= 2 && !fail && !mbar_wait(&ms->kv_empty[g & 1], ((g >> 1) - 1) & 1, kWaitLimit)) fail = true;
      float sa = 0.0f, sb2 = 0.0f;
      uint8_t* dst = sP + (g & 1) * 8192;
      // a head whose keys so far are all masked keeps m = -inf: its P is 0
      // (only with expanded rows: a gathered item's first tile has a key)
      const float mea = (kExpand && ma == -INFINITY) ? 0.0f : ma, meb = (kExpand && mb == -INFINITY) ? 0.0f : mb;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float pa0 = ex2(xa[2 * j] - mea), pa1 = ex2(xa[2 * j + 1] - mea);
        const float pb0 = ex2(xb[2 * j] - meb), pb1 = ex2(xb[2 * j + 1] - meb);
        sa += pa0 + pa1;
        sb2 += pb0 + pb1;
        const __nv_bfloat162 qa = __floats2bfloat162_rn(pa0, pa1);
        const __nv_bfloat162 qb = __floats2bfloat162_rn(pb0, pb1);
        *reinterpret_cast<uint32_t*>(dst + sw128(ha, j) + 2 * cq) = *reinterpret_cast<const uint32_t*>(&qa);
        *reinterpret_cast<uint32_t*>(dst + sw128(hb, j) + 2 * cq) = *reinterpret_cast<const uint32_t*>(&qb);
      }
      la = la * aa + sa;
      lb = lb * ab + sb2;
      fence_proxy_async();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->p_full[g & 1]);
    }
    // ---- this item's partial state: statistics and the normalised output ----
    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    const bool any_keys = thi > tlo;
    if (any_keys && !stop && !fail && !mbar_wait(&ms->o_full, 0, kWaitLimit)) fail = true;
    fence_after_sync();
    // this item's statistics per head, (m, l), in P buffer 1 (free now): the
    // row's other items read them there
    float2* ml_own = kCluster ? reinterpret_cast<float2*>(sP + 8192)
                              : reinterpret_cast<float2*>(p.part_ml + item * (kH * 2));
    if (leader) {
      ml_own[ha] = make_float2(any_keys ? ma : -INFINITY, any_keys ? la : 0.0f);
      ml_own[hb] = make_float2(any_keys ? mb : -INFINITY, any_keys ? lb : 0.0f);
    }
    // 1 / l per head through shared memory (P buffer 0)
    float* inv_s = reinterpret_cast<float*>(sP);
    group_vote(false);   // every softmax warp is past its last P
    if (leader) {
      inv_s[ha] = la > 0.0f ? 1.0f / la : 0.0f;
      inv_s[hb] = lb > 0.0f ? 1.0f / lb : 0.0f;
    }
    group_vote(false);
    const bool bad = group_vote(__any_sync(0xffffffffu, fail || stop || vabort(ms))) != 0;
    // O^T lanes are dims: thread (qd, lane) holds dim 128 mt + 32 qd + lane of
    // every head; the normalised partial stays in the query's shared memory
    // (free once o_full has passed) as [dim][head] bf16 rows of 128 bytes,
    // 16-byte chunk c of row d at chunk c ^ (d mod 8), where the row's other
    // items read it
#pragma unroll 1
    for (int mt = 0; mt < 4 && !bad; ++mt) {   // (a failed item leaves sQ alone: MMAs may still read it)
      // both head halves of dim block mt: two TMEM loads in flight per wait
      uint32_t o[2][32];
      if (any_keys) {
        tmem_ld32(tmem + tq_lane + kTmemO + 64u * mt, o[0]);
        tmem_ld32(tmem + tq_lane + kTmemO + 64u * mt + 32u, o[1]);
        tmem_wait_ld();
      }
      const int d = 128 * mt + 32 * qd + lane;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int h0 = 32 * hh + 2 * j;
          const float f0 = any_keys ? __uint_as_float(o[hh][2 * j]) * inv_s[h0] : 0.0f;
          const float f1 = any_keys ? __uint_as_float(o[hh][2 * j + 1]) * inv_s[h0 + 1] : 0.0f;
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(f0, f1);
          pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(sQ + (uint32_t)d * 128u + ((((uint32_t)(4 * hh + j)) ^ ((uint32_t)d & 7u)) << 4)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      }
    }
    if (bad) fail = true;
    if constexpr (!kCluster) {
      // the staged partial to global memory: four TMA boxes of 128 dims
      fence_proxy_async();
      group_vote(false);   // the whole partial is staged
      if (tid == 0 && !bad) {
        for (int mt = 0; mt < 4; ++mt) tma_store_2d(&tm_po, smem_u32(sQ) + mt * 16384, 0, (int)(item * kD + 128 * mt));
        bulk_commit_wait_all();
        // visible to the row's other items (read there by bulk copies: the
        // async proxy) before the arrival on the row counter
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __threadfence();
    }
  }
  if (fail) {
    ms->abort = 1;
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (kCluster) {
  // ---- the row's items meet: every partial of the row is staged, every
  // item's KV slots are free and its barriers initialised (cluster barrier) ----
  cluster_sync_all();
  // ---- each item pushes to item c the rows of item c's dim slice and its
  // statistics; then merges its own slice over the splits ----
  // dims of a slice: [d0, d1), even bounds (RoPE pairs stay together)
  const int ns = p.nsplit;
  const int dp = ((kD + ns - 1) / ns + 1) & ~1;
  const int d0 = min(kD, split * dp), d1 = min(kD, d0 + dp);
  const int nd = d1 - d0;
  // receive area in the KV slots: [ns][dp] partial rows of 128 bytes, then
  // [ns][64] (m, l); scratch after it
  uint8_t* rcv = sKV;
  float2* mls = reinterpret_cast<float2*>(sKV + 73728);
  float* Ms = reinterpret_cast<float*>(sKV + 73728 + kMaxSplits * kH * 8);   // [64]
  float* Linv = Ms + kH;                                                      // [64]
  float* wgt = Linv + kH;                                                     // [ns][64]
  float* cs = wgt + kMaxSplits * kH;   // the RoPE row of t: 32 cos, 32 sin
  float* sn = cs + 32;
  static_assert((kMaxSplits * ((kD + kMaxSplits - 1) / kMaxSplits + 2)) * 128 <= 73728, "receive rows");
  static_assert(73728 + kMaxSplits * kH * 8 + (2 * kH + kMaxSplits * kH + 64) * 4 <= 131072, "merge scratch");
  if (tid == 0) mbar_arrive_expect_tx(&ms->recv, (uint32_t)ns * ((uint32_t)nd * 128u + kH * 8u));
  if (tid >= 32 && tid < 32 + ns) {   // thread 32 + c pushes to item c
    const int c = tid - 32;
    const int c0 = min(kD, c * dp), c1 = min(kD, c0 + dp);
    const uint32_t bar = map_cluster(&ms->recv, (uint32_t)c);
    if (c1 > c0)
      bulk_push_cluster(map_cluster(rcv + (uint32_t)split * dp * 128u, (uint32_t)c), smem_u32(sQ) + (uint32_t)c0 * 128u,
                        (uint32_t)(c1 - c0) * 128u, bar);
    bulk_push_cluster(map_cluster(mls + split * kH, (uint32_t)c), smem_u32(sP + 8192), kH * 8u, bar);
  }
  if (tid >= 64 && tid < 96) {
    cs[tid - 64] = rope_c;
    sn[tid - 64] = rope_s;
  }
  if (!mbar_wait(&ms->recv, 0, kWaitLimit) && tid == 0) flag_timeout(p.ws);
  // per head: M, the maximum over the splits, then every weight 2^(m_s - M) l_s,
  // then 1 / L, L their sum in split order
  if (tid < kH) {
    float M = -INFINITY;
    for (int c = 0; c < ns; ++c) M = fmaxf(M, mls[c * kH + tid].x);
    Ms[tid] = M;
  }
  __syncthreads();
  for (int i = tid; i < ns * kH; i += kThreads) {
    const float2 v = mls[i];
    wgt[i] = v.x == -INFINITY ? 0.0f : exp2f(v.x - Ms[i & (kH - 1)]) * v.y;
  }
  __syncthreads();
  if (tid < kH) {
    float L = 0.0f;
    for (int c = 0; c < ns; ++c) L += wgt[c * kH + tid];
    Linv[tid] = L > 0.0f ? 1.0f / L : 0.0f;
    if (split == 0 && p.lse) p.lse[row * kH + tid] = L > 0.0f ? (Ms[tid] + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  merge_slice(rcv, (uint32_t)dp, true, ns, d0, nd, wgt, Linv, cs, sn, p.out + row * (int64_t)(kH * kD));
  // every item of the row has read this one's shared memory before it exits
  cluster_sync_all();
  } else {
  // ---- the row's items meet: every partial of the row is written ----
  if (tid == 0) {
    atomicAdd(p.arrive + row, 1);
    bool ok = false;
    for (uint32_t it = 0; it < kGridWaitLimit; ++it) {
      if (*reinterpret_cast<volatile int*>(p.arrive + row) >= p.nsplit) {
        ok = true;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    if (!ok) flag_timeout(p.ws);
    ms->go = ok ? 1 : 0;
  }
  __syncthreads();
  if (!ms->go) return;
  // ---- merge this item's slice of the row's dims over the splits ----
  // dims of this slice: [d0, d1), even bounds (RoPE pairs stay together)
  const int ns = p.nsplit;
  const int dp = ((kD + ns - 1) / ns + 1) & ~1;
  const int d0 = min(kD, split * dp), d1 = min(kD, d0 + dp);
  const int nd = d1 - d0;
  // shared memory is free now: the row's statistics [ns][64] (m, l) at 0,
  // this slice's partial rows [ns][nd] of 128 bytes after them (plain rows:
  // the tensor map of the partials' store undid the staging swizzle), staged
  // by bulk copies (all in flight together)
  const uint32_t ml_bytes = (uint32_t)ns * kH * 8;
  const uint32_t sl_off = (ml_bytes + 1023) & ~1023u;
  const float2* ml_s = reinterpret_cast<const float2*>(sm);
  const uint8_t* sl_s = sm + sl_off;
  if (tid == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_arrive_expect_tx(&ms->merge_in, ml_bytes + (uint32_t)ns * nd * 128u);
    bulk_copy_g2s(smem_u32(sm), p.part_ml + row * (int64_t)ns * kH * 2, ml_bytes, &ms->merge_in);
    if (nd > 0)
      for (int c = 0; c < ns; ++c)
        bulk_copy_g2s(smem_u32(sm + sl_off + (uint32_t)c * nd * 128u),
                      p.part_o + (row * (int64_t)ns + c) * (kH * kD) + (int64_t)d0 * kH, (uint32_t)nd * 128u,
                      &ms->merge_in);
  }
  if (!mbar_wait(&ms->merge_in, 0, kWaitLimit)) {
    if (tid == 0) flag_timeout(p.ws);
    return;   // (a copy still in flight lands in memory nobody reads again)
  }
  // per head: M, the maximum over the splits (five partial maxima each), every
  // weight 2^(m_s - M) l_s, then 1 / L, L their sum in split order
  float* wgt = reinterpret_cast<float*>(sm + sl_off + (((uint32_t)ns * nd * 128u + 1023) & ~1023u));
  float* red = wgt + (size_t)ns * kH;   // [5][64] partial maxima
  float* Linv = red + 5 * kH;           // [64]
  float* cs = Linv + kH;                // the RoPE row of t: 32 cos, 32 sin
  float* sn = cs + 32;
  {
    const int g = tid >> 6, h = tid & (kH - 1);   // kThreads = 5 x 64
    float M = -INFINITY;
    for (int c = g; c < ns; c += 5) M = fmaxf(M, ml_s[c * kH + h].x);
    red[g * kH + h] = M;
  }
  if (tid >= 64 && tid < 96) {
    cs[tid - 64] = rope_c;
    sn[tid - 64] = rope_s;
  }
  __syncthreads();
  for (int i = tid; i < ns * kH; i += kThreads) {
    const int h = i & (kH - 1);
    const float M = fmaxf(fmaxf(fmaxf(red[h], red[kH + h]), fmaxf(red[2 * kH + h], red[3 * kH + h])), red[4 * kH + h]);
    const float2 v = ml_s[i];
    wgt[i] = v.x == -INFINITY ? 0.0f : exp2f(v.x - M) * v.y;
  }
  __syncthreads();
  if (tid < kH) {
    float L = 0.0f;
    for (int c = 0; c < ns; ++c) L += wgt[c * kH + tid];
    Linv[tid] = L > 0.0f ? 1.0f / L : 0.0f;
    if (split == 0 && p.lse) {
      const float M = fmaxf(fmaxf(fmaxf(red[tid], red[kH + tid]), fmaxf(red[2 * kH + tid], red[3 * kH + tid])),
                            red[4 * kH + tid]);
      p.lse[row * kH + tid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
  }
  __syncthreads();
  merge_slice(sl_s, (uint32_t)nd, false, ns, d0, nd, wgt, Linv, cs, sn, p.out + row * (int64_t)(kH * kD));
  }
}

// cuTensorMapEncodeTiled, fetched from the driver once
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (!f) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(ptr);
      fn.store(f);
    }
  }
  return f;
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace {

// How many clusters of `s` attention CTAs (one per SM: 227 KiB of shared
// memory each) the device can hold at once, asked once per device and size
// (clusters stay inside a GPC, so this depends on how its SMs are grouped).
int decode_clusters_resident(int s) {
  static PerDevice attrs;
  static PerDevice count[kMaxSplits + 1];
  attrs.get([] {
    const void* ks[4] = {reinterpret_cast<const void*>(attn_decode_kernel<true, false>),
                         reinterpret_cast<const void*>(attn_decode_kernel<true, true>),
                         reinterpret_cast<const void*>(attn_decode_kernel<false, false>),
                         reinterpret_cast<const void*>(attn_decode_kernel<false, true>)};
    for (int i = 0; i < 4; ++i) {
      cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
      if (i < 2) cudaFuncSetAttribute(ks[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    cudaGetLastError();
    return 1;
  });
  // stored plus one (a stored zero would be asked again)
  return count[s].get([s] {
           cudaLaunchConfig_t cfg = {};
           cfg.gridDim = dim3((unsigned)s);
           cfg.blockDim = dim3(kThreads);
           cfg.dynamicSmemBytes = kSmemBytes;
           cudaLaunchAttribute at[1];
           at[0].id = cudaLaunchAttributeClusterDimension;
           at[0].val.clusterDim.x = (unsigned)s;
           at[0].val.clusterDim.y = 1;
           at[0].val.clusterDim.z = 1;
           cfg.attrs = at;
           cfg.numAttrs = 1;
           int n = 0;
           if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(attn_decode_kernel<true, false>), &cfg) !=
               cudaSuccess) {
             cudaGetLastError();
             n = 0;
           }
           return n + 1;
         }) -
         1;
}

}  // namespace

// Items per row: as many as fill the SMs once, at most one per key tile.
// When that is at most kClusterMergeMax the items of a row form a cluster
// (then the largest size whose clusters, one per row, the device holds all
// at once: a size that leaves rows for a second wave costs more than fewer
// splits); more, they merge through global memory.
static int64_t decode_fill_splits(int64_t rows, int64_t max_keys) {
  const int sms = device_sms() > 0 ? device_sms() : 148;
  const int64_t tiles = (max_keys + kTile - 1) / kTile;
  int64_t s = sms / (rows > 0 ? rows : 1);
  if (s > tiles) s = tiles;
  return s < 1 ? 1 : s;
}
static bool decode_cluster_merge(int64_t rows, int64_t max_keys) {
  return decode_fill_splits(rows, max_keys) <= kClusterMergeMax;
}
int attn_decode_splits(int64_t rows, int64_t max_keys) {
  int64_t s = decode_fill_splits(rows, max_keys);
  if (s <= kClusterMergeMax)
    while (s > 1 && decode_clusters_resident((int)s) < rows) --s;
  return (int)s;
}

bool attn_decode_applies(int H, int D, int R, int64_t rows, int k, bool sparse) {
  const int sms = device_sms() > 0 ? device_sms() : 148;
  return H == kH && D == kD && R == 64 && rows > 0 && rows < sms && (!sparse || k <= kMaxK);
}

int64_t attn_decode_kp(int64_t max_keys) { return (max_keys + kTile - 1) / kTile * kTile; }

// Items of at most kExpandTiles key tiles expand the cache rows themselves
// (each tile's row loads are one exposed round trip, cheaper than a gather
// launch); longer items read rows gathered ahead of them (their loads ride
// TMA boxes of gathered rows, two tiles deep).
constexpr int kExpandTiles = 4;
static bool decode_expand(int64_t rows, int64_t max_keys) {
  const int64_t tiles = (max_keys + kTile - 1) / kTile;
  const int64_t s = attn_decode_splits(rows, max_keys);
  return (tiles + s - 1) / s <= kExpandTiles;
}
size_t attn_decode_workspace(int64_t rows, int64_t max_keys) {
  size_t bytes = decode_expand(rows, max_keys)
                     ? 0
                     : al256((size_t)rows * 4) + al256((size_t)rows * attn_decode_kp(max_keys) * kD * 2);
  if (!decode_cluster_merge(rows, max_keys)) {
    const int64_t items = rows * attn_decode_splits(rows, max_keys);
    bytes += al256((size_t)items * kH * kD * 2) + al256((size_t)items * kH * 2 * 4) + al256((size_t)rows * 4);
  }
  return bytes;
}

cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.Tq;
  DParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.q_pos = a.q_pos;
  p.Tq = a.Tq;
  p.cache = reinterpret_cast<const uint8_t*>(a.cache);
  p.N = a.N;
  p.m = a.m;
  p.idx = a.idx;
  p.k = a.idx ? a.k : 0;
  p.swa = reinterpret_cast<const uint8_t*>(a.swa);
  p.swa_pos0 = a.swa_pos0;
  p.Ts = a.W > 0 ? a.Ts : 0;
  p.W = a.W;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.rcos = a.rcos;
  p.rsin = a.rsin;
  p.rope_rows = a.rope_rows;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.ws = a.ws;
  p.nsplit = attn_decode_splits(rows, a.max_keys);
  const int64_t items = rows * p.nsplit;
  const bool cl = decode_cluster_merge(rows, a.max_keys);
  p.expand = decode_expand(rows, a.max_keys) ? 1 : 0;
  uint8_t* base = reinterpret_cast<uint8_t*>(a.ws) + kWsHeader;
  p.ecount = nullptr;
  p.xg = nullptr;
  p.kp = attn_decode_kp(a.max_keys);
  if (!p.expand) {
    p.ecount = reinterpret_cast<int*>(base);
    base += al256((size_t)rows * 4);
    p.xg = reinterpret_cast<__nv_bfloat16*>(base);
    base += al256((size_t)rows * p.kp * kD * 2);
  }
  p.part_o = nullptr;
  p.part_ml = nullptr;
  p.arrive = nullptr;
  if (!cl) {
    p.part_o = reinterpret_cast<__nv_bfloat16*>(base);
    base += al256((size_t)items * kH * kD * 2);
    p.part_ml = reinterpret_cast<float*>(base);
    base += al256((size_t)items * kH * 2 * 4);
    p.arrive = reinterpret_cast<int*>(base);
  }
  CUtensorMap tm_q, tm_xg, tm_po;
  memset(&tm_po, 0, sizeof(tm_po));
  memset(&tm_xg, 0, sizeof(tm_xg));
  {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)(rows * kH)};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64u, 64u};
    const cuuint32_t estr[2] = {1u, 1u};
    if (fn(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (!cl) {
      const cuuint64_t pdims[2] = {(cuuint64_t)kH, (cuuint64_t)(items * kD)};
      const cuuint64_t pstrides[1] = {(cuuint64_t)kH * 2};
      const cuuint32_t pbox[2] = {(cuuint32_t)kH, 128u};
      if (fn(&tm_po, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.part_o, pdims, pstrides, pbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    if (!p.expand) {
      const cuuint64_t gdims[2] = {(cuuint64_t)kD, (cuuint64_t)(rows * p.kp)};
      if (fn(&tm_xg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.xg, gdims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  cudaError_t e = cudaSuccess;
  if (!cl) {
    e = cudaMemsetAsync(p.arrive, 0, (size_t)rows * 4, st);
    if (e != cudaSuccess) return e;
  }
  if (!p.expand) {
    e = launch_pdl(decode_gather_kernel, dim3((unsigned)(p.kp / kTile), (unsigned)rows), dim3(kGatherThreads), 0, st,
                   p);
    if (e != cudaSuccess) return e;
  }
  decode_clusters_resident(1);   // the kernels' shared-memory and cluster-size attributes, set once per device
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  if (cl) {
    // one cluster per row: its items meet at cluster barriers and merge
    // through each other's shared memory
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = (unsigned)p.nsplit;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return p.expand ? cudaLaunchKernelEx(&cfg, attn_decode_kernel<true, true>, p, tm_q, tm_xg, tm_po)
                    : cudaLaunchKernelEx(&cfg, attn_decode_kernel<true, false>, p, tm_q, tm_xg, tm_po);
  }
  // every item resident at once (an item waits on its row's counter)
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return p.expand ? cudaLaunchKernelEx(&cfg, attn_decode_kernel<false, true>, p, tm_q, tm_xg, tm_po)
                  : cudaLaunchKernelEx(&cfg, attn_decode_kernel<false, false>, p, tm_q, tm_xg, tm_po);
}

}  // namespace csa
