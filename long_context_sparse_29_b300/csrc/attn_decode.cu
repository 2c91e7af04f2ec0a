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
// keys are split over many CTAs (one work item = one row and one split, at
// most one item per SM, every item resident at once: cooperative launch),
// and everything the long-row path does in separate launches happens here:
//  * the query is loaded by TMA and its RoPE dims rotated to its position
//    in shared memory by the softmax warps;
//  * the producer warps build the row's ordered list of valid selected
//    entries from idx (invalid ones set the device-check flag), prefetch the
//    item's key rows into L2, and fetch each 64-key tile's 592-byte rows
//    with bulk copies into the end of its ring slot; they then expand the
//    FP8 codes (times their group scale: exact) and the bf16 RoPE dims into
//    the slot's bf16 tile in place -- first the dims whose bf16 lines lie
//    below the raw rows, then, once every producer warp holds the rest in
//    registers, the others;
//  * each item writes its normalised partial output (bf16) and its softmax
//    statistics, the items of a row meet at a bounded grid barrier (a
//    counter per row), and each item then merges one slice of the row's
//    dims over all splits in split order, rotates the RoPE dims back and
//    stores the output.
// Every wait is bounded; on expiry the CTA records the timeout flag in the
// workspace, waits (bounded) for its own copies and MMAs and frees TMEM.
#include <cuda.h>

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
constexpr uint32_t kListOff = kMiscOff + 2048;    // int32 list of the row's valid selected entries
constexpr uint32_t kSmemBytes = 232448;           // 227 KiB
constexpr int kMaxList = (int)((kSmemBytes - 1024 - kListOff) / 4);
constexpr uint32_t kRawOff = 65536 - 64 * kMixRow;   // a tile's raw rows, at the end of its slot
static_assert(kRawOff == 27648 && kRawOff > 3 * 8192, "raw rows must lie above bf16 chunks 0-2");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;       // O^T: 4 blocks of 64 columns (heads); lanes = dims
constexpr uint32_t kTmemS = 256;     // S: 2 buffers of 64 columns (keys); M = 64 layout

constexpr uint32_t kWaitLimit = 1u << 20;     // suspending polls of one mbarrier wait
constexpr uint32_t kGridWaitLimit = 1u << 22; // polls of the row barrier (64 ns naps)
constexpr float kLazy = 8.0f;

struct Misc {
  uint64_t raw_full[2], kv_full[2], kv_empty[2], s_full[2], p_full[2];
  uint64_t q_full, q_ready, o_full, drain[2], merge_in;
  uint32_t tmem;
  int abort;
  int cnt[4];                       // valid selected entries per producer warp's share of idx
  int go;                           // the row barrier passed
  alignas(16) float alpha[2][kH];   // per-head rescale factors of a tile, double-buffered
};
static_assert(sizeof(Misc) <= 2048, "Misc overflows its smem slot");
static_assert(offsetof(Misc, alpha) % 16 == 0, "vector reads of Misc");

__device__ __forceinline__ bool vabort(const Misc* ms) {
  return *reinterpret_cast<const volatile int*>(&ms->abort) != 0;
}

// Barrier of the four producer warps (named barrier 2, 128 threads).
__device__ __forceinline__ void producer_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

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
  int nsplit;
  __nv_bfloat16* part_o;    // [items, 512 dims, 64 heads] normalised partial outputs
  float* part_ml;           // [items, 64, 2]: running max (log2 units), sum
  int* arrive;              // [rows] items that finished their partial (zero at launch)
};

__global__ void __launch_bounds__(kThreads, 1)
attn_decode_kernel(const DParams p, const __grid_constant__ CUtensorMap tm_q) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kQOff;
  uint8_t* sKV = sm + kKVOff;
  uint8_t* sP = sm + kPOff;
  Misc* ms = reinterpret_cast<Misc*>(sm + kMiscOff);
  int32_t* list = reinterpret_cast<int32_t*>(sm + kListOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t item = blockIdx.x;
  const int64_t row = item / p.nsplit;
  const int split = (int)(item - row * p.nsplit);
  const int64_t b = row / p.Tq;
  const int64_t t = p.q_pos[row];
  const bool t_ok = t >= 0 && t < p.rope_rows;
  const bool dense = p.idx == nullptr;

  if (tid == 0) {
    ms->abort = 0;
    ms->go = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->raw_full[i], 4 + 128);   // one arrive per producer warp, one counted per producer lane
      mbar_init(&ms->kv_full[i], 4);    // one arrive per producer warp once its rows are expanded
      mbar_init(&ms->kv_empty[i], 1);
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->p_full[i], 4);
    }
    mbar_init(&ms->q_full, 1);
    mbar_init(&ms->q_ready, 4);
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->drain[0], 1);
    mbar_init(&ms->drain[1], 1);
    mbar_init(&ms->merge_in, 1);
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ms->tmem, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;

  // ---- the query: 8 TMA boxes, in flight while the entry list is built ----
  if (warp == kMmaWarp) {
    if (lane == 0) mbar_arrive_expect_tx(&ms->q_full, kH * kD * 2);
    __syncwarp();
    if (lane < 8) tma_load_2d(smem_u32(sQ) + lane * 8192, &tm_q, 64 * lane, (int)(row * kH), &ms->q_full);
    __syncwarp();
  }
  // ---- sparse: the row's valid selected entries, in idx order ----
  if (!dense && warp >= 4 && warp < 8) {
    const int pw = warp - 4;
    const int seg = ((p.k + 3) / 4 + 31) / 32 * 32;
    const int lo = pw * seg, hi = min(p.k, lo + seg);
    const int32_t* ir = p.idx + row * (int64_t)p.k;
    // the warp's share of idx: at most 32 per lane (k <= 4096), all loads in flight together
    int32_t js[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const int i = lo + 32 * r + lane;
      js[r] = i < hi ? __ldg(ir + i) : -1;
    }
    uint32_t okbits = 0;
    int cnt = 0;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const int32_t j = js[r];
      const bool ok = t_ok && j >= 0 && (int64_t)j < p.N && (int64_t)(j + 1) * p.m - 1 <= t;
      if (split == 0 && t_ok && j >= 0 && !ok) flag_device_check(p.ws, (unsigned)j);
      okbits |= ok ? 1u << r : 0u;
      cnt += __popc(__ballot_sync(0xffffffffu, ok));
    }
    if (lane == 0) ms->cnt[pw] = cnt;
    producer_sync();
    int out = 0;
    for (int w2 = 0; w2 < pw; ++w2) out += ms->cnt[w2];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const bool ok = (okbits >> r) & 1u;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (ok) list[out + __popc(bal & ((1u << lane) - 1u))] = js[r];
      out += __popc(bal);
    }
  }
  __syncthreads();

  // ---- this item's keys: entries first, then the window tokens ----
  int ne = 0;
  if (t_ok) {
    if (dense) {
      const int64_t nv = (t + 1) / p.m;
      ne = (int)(nv < p.N ? nv : p.N);
    } else {
      ne = min(ms->cnt[0] + ms->cnt[1] + ms->cnt[2] + ms->cnt[3], kMaxList);
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
  // the key row of key number `key` of this row, or NULL past its keys
  auto key_row = [&](int key) -> const uint8_t* {
    if (key >= key_hi) return nullptr;
    if (key < ne) return p.cache + (b * p.N + (dense ? (int64_t)key : (int64_t)list[key])) * kMixRow;
    return p.swa + (b * p.Ts + (w_lo - p0 + (key - ne))) * kMixRow;
  };
  bool fail = false;

  if (warp >= 4 && warp < 8) {
    // ================================ producers ================================
    const int pw = warp - 4;
    // dense keys are runs of consecutive rows (the entries, then the window):
    // the item's runs into L2 now, in pieces of at most 64 rows
    if (dense && pw == 0) {
      const int e_lo = tlo * kTile, e_hi = min(ne, key_hi);
      for (int r = e_lo + 64 * lane; r < e_hi; r += 64 * 32)
        prefetch_l2(p.cache + (b * p.N + r) * kMixRow, (uint32_t)min(64, e_hi - r) * kMixRow);
      const int w_lo2 = max(ne, tlo * kTile), w_hi2 = key_hi;
      for (int r = w_lo2 + 64 * lane; r < w_hi2; r += 64 * 32)
        prefetch_l2(p.swa + (b * p.Ts + (w_lo - p0 + (r - ne))) * kMixRow, (uint32_t)min(64, w_hi2 - r) * kMixRow);
    }
    uint32_t g = 0;
    bool ok = true;
    for (int tl = tlo; tl < thi && ok && !vabort(ms); ++tl, ++g) {
      const int buf = g & 1;
      if (g >= 2 && !mbar_wait(&ms->kv_empty[buf], ((g >> 1) - 1) & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      uint8_t* slot = sKV + buf * 65536;
      uint8_t* raw = slot + kRawOff;
      // this warp's 16 rows of the tile (valid ones in vmask); dense: the
      // tile's runs of consecutive rows as at most two bulk copies (warp 0);
      // sparse: 16-byte asynchronous copies, 37 per row, spread over the lanes
      const int r0 = 16 * pw;
      const uint8_t* src = lane < 16 ? key_row(tl * kTile + r0 + lane) : nullptr;
      const unsigned vmask = __ballot_sync(0xffffffffu, src != nullptr);
      if (dense) {
        if (pw == 0 && lane == 0) {
          const int k0 = tl * kTile, k1 = min(key_hi, k0 + kTile);
          const int ce = max(k0, min(ne, k1));   // entries [k0, ce), window [ce, k1)
          mbar_arrive_expect_tx(&ms->raw_full[buf], (uint32_t)(k1 - k0) * kMixRow);
          if (ce > k0)
            bulk_copy_g2s(smem_u32(raw), p.cache + (b * p.N + k0) * kMixRow, (uint32_t)(ce - k0) * kMixRow,
                          &ms->raw_full[buf]);
          if (k1 > ce)
            bulk_copy_g2s(smem_u32(raw + (ce - k0) * kMixRow), p.swa + (b * p.Ts + (w_lo - p0 + (ce - ne))) * kMixRow,
                          (uint32_t)(k1 - ce) * kMixRow, &ms->raw_full[buf]);
        } else if (lane == 0) {
          mbar_arrive(&ms->raw_full[buf]);
        }
      } else {
        if (lane == 0) mbar_arrive(&ms->raw_full[buf]);
        const unsigned long long sp = reinterpret_cast<unsigned long long>(src);
#pragma unroll 1
        for (int it = 0; it < (16 * 37 + 31) / 32; ++it) {
          const int q = lane + 32 * it;
          const int i = q / 37, u = q - 37 * (q / 37);
          const unsigned long long rp = __shfl_sync(0xffffffffu, sp, q < 16 * 37 ? i : 0);
          if (q < 16 * 37 && rp)
            cp_async16(smem_u32(raw + (r0 + i) * kMixRow + 16 * u), reinterpret_cast<const uint8_t*>(rp) + 16 * u);
        }
      }
      cp_async_mbar_arrive_noinc(&ms->raw_full[buf]);
      __syncwarp();
      if (!mbar_wait(&ms->raw_full[buf], (g >> 1) & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      // phase 1: bf16 chunks 0-2 (dims 0..191, below the raw rows), and the
      // rest of this warp's rows into registers
#pragma unroll 4
      for (int v = 0; v < 12; ++v) {
        const int U = lane + 32 * v;                // 16 rows x 24 units of 8 dims
        const int i = U / 24, u = U - 24 * (U / 24);
        const int r = r0 + i;
        uint4 o = make_uint4(0, 0, 0, 0);
        if ((vmask >> i) & 1u) {
          const uint8_t* rr = raw + r * kMixRow;
          const uint2 c = *reinterpret_cast<const uint2*>(rr + 8 * u);
          const float sc = *reinterpret_cast<const float*>(rr + kMixScaleOff + 4 * (u >> 4));
          o = dequant8(c, sc);
        }
        *reinterpret_cast<uint4*>(slot + (u >> 3) * 8192 + sw128((uint32_t)r, (uint32_t)(u & 7))) = o;
      }
      // dims 192..447: unit 24 + lane of each row (group 1, 2 or 3 by lane)
      // (the group scales are powers of two: their exponent bytes, four per word)
      const int gsc = lane < 8 ? 1 : (lane < 24 ? 2 : 3);
      uint2 hc[16];
      uint32_t hs[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        hc[i] = make_uint2(0, 0);
        if ((vmask >> i) & 1u) {
          const uint8_t* rr = raw + (r0 + i) * kMixRow;
          hc[i] = *reinterpret_cast<const uint2*>(rr + 8 * (24 + lane));
          const uint32_t sb = *reinterpret_cast<const uint32_t*>(rr + kMixScaleOff + 4 * gsc);
          hs[i >> 2] |= ((sb >> 23) & 0xffu) << (8 * (i & 3));
        }
      }
      // RoPE dims: 16 rows x 8 units of 16 bytes, four per lane
      uint4 hr[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int U = lane + 32 * v, i = U >> 3, u = U & 7;
        hr[v] = make_uint4(0, 0, 0, 0);
        if ((vmask >> i) & 1u) hr[v] = *reinterpret_cast<const uint4*>(raw + (r0 + i) * kMixRow + kMixRopeOff + 16 * u);
      }
      producer_sync();   // every producer warp holds what it still needs of the raw rows
      // phase 2: chunks 3-6 (FP8) and 7 (RoPE) over the raw rows
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int u = 24 + lane, r = r0 + i;
        const float sc = __uint_as_float(((hs[i >> 2] >> (8 * (i & 3))) & 0xffu) << 23);
        const uint4 o = ((vmask >> i) & 1u) ? dequant8(hc[i], sc) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(slot + (u >> 3) * 8192 + sw128((uint32_t)r, (uint32_t)(u & 7))) = o;
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int U = lane + 32 * v, i = U >> 3, u = U & 7, r = r0 + i;
        *reinterpret_cast<uint4*>(slot + 7 * 8192 + sw128((uint32_t)r, (uint32_t)u)) = hr[v];
      }
      fence_proxy_async();   // generic-proxy writes, read next by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->kv_full[buf]);
    }
    if (!ok) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
      fail = true;
      // a bulk copy of this tile may still be in flight: let it land
      cp_async_wait_all();
      if (g < (uint32_t)(thi - tlo)) mbar_wait(&ms->raw_full[g & 1], (g >> 1) & 1, kWaitLimit);
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
      fence_after_sync();
      const int nvalid = min(kTile, key_hi - tl * kTile);
      uint32_t v[32];
      tmem_ld16x256b_x8(tmem + tq_lane + kTmemS + 64u * (g & 1), v);
      tmem_wait_ld();
      float xa[16], xb[16];
      float ta = -INFINITY, tb = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool valid = 8 * j + cq + e < nvalid;
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
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float pa0 = ex2(xa[2 * j] - ma), pa1 = ex2(xa[2 * j + 1] - ma);
        const float pb0 = ex2(xb[2 * j] - mb), pb1 = ex2(xb[2 * j + 1] - mb);
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
    if (leader) {
      float* ml = p.part_ml + item * (kH * 2);
      ml[2 * ha] = any_keys ? ma : -INFINITY;
      ml[2 * ha + 1] = any_keys ? la : 0.0f;
      ml[2 * hb] = any_keys ? mb : -INFINITY;
      ml[2 * hb + 1] = any_keys ? lb : 0.0f;
    }
    // 1 / l per head through shared memory (the P buffers are free now)
    float* inv_s = reinterpret_cast<float*>(sP);
    group_vote(false);   // every softmax warp is past its last P (its PV may still read P? no: o_full)
    if (leader) {
      inv_s[ha] = la > 0.0f ? 1.0f / la : 0.0f;
      inv_s[hb] = lb > 0.0f ? 1.0f / lb : 0.0f;
    }
    group_vote(false);
    const bool bad = group_vote(__any_sync(0xffffffffu, fail || stop || vabort(ms))) != 0;
    // O^T lanes are dims: thread (qd, lane) holds dim 128 mt + 32 qd + lane of
    // heads 64 mt .. ; stored as [dim][head] bf16 rows of 128 bytes
    __nv_bfloat16* po = p.part_o + item * (int64_t)(kH * kD);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      const int mt = c >> 1, hh = c & 1;
      uint32_t o[32];
      if (any_keys && !bad) {
        tmem_ld32(tmem + tq_lane + kTmemO + 64u * mt + 32u * hh, o);
        tmem_wait_ld();
      }
      const int d = 128 * mt + 32 * qd + lane;
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int h0 = 32 * hh + 2 * j;
        const float f0 = (any_keys && !bad) ? __uint_as_float(o[2 * j]) * inv_s[h0] : 0.0f;
        const float f1 = (any_keys && !bad) ? __uint_as_float(o[2 * j + 1]) * inv_s[h0 + 1] : 0.0f;
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(f0, f1);
        pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      uint4* dst = reinterpret_cast<uint4*>(po + (int64_t)d * kH + 32 * hh);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
    if (bad) fail = true;
    // the partial is visible to the row's other items (read there by bulk
    // copies: the async proxy) before the arrival below
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
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
  // this slice's partial rows [ns][nd][64 heads] bf16 after them, staged by
  // bulk copies (all in flight together)
  const uint32_t ml_bytes = (uint32_t)ns * kH * 8;
  const uint32_t sl_off = (ml_bytes + 1023) & ~1023u;
  const float2* ml_s = reinterpret_cast<const float2*>(sm);
  const __nv_bfloat16* sl_s = reinterpret_cast<const __nv_bfloat16*>(sm + sl_off);
  if (tid == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_arrive_expect_tx(&ms->merge_in, ml_bytes + (uint32_t)ns * nd * kH * 2);
    bulk_copy_g2s(smem_u32(sm), p.part_ml + row * (int64_t)ns * kH * 2, ml_bytes, &ms->merge_in);
    if (nd > 0)
      for (int s = 0; s < ns; ++s)
        bulk_copy_g2s(smem_u32(sm + sl_off + (uint32_t)s * nd * kH * 2),
                      p.part_o + (row * (int64_t)ns + s) * (kH * kD) + (int64_t)d0 * kH, (uint32_t)nd * kH * 2,
                      &ms->merge_in);
  }
  if (!mbar_wait(&ms->merge_in, 0, kWaitLimit)) {
    if (tid == 0) flag_timeout(p.ws);
    return;   // (a copy still in flight lands in memory nobody reads again)
  }
  // per head: the splits' weights 2^(m_s - M) l_s, then 1 / L
  float* wgt = reinterpret_cast<float*>(sm + sl_off + (((uint32_t)ns * nd * kH * 2 + 1023) & ~1023u));
  float* Ls = wgt + (size_t)ns * kH;
  if (tid < kH) {
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, ml_s[s * kH + tid].x);
    float L = 0.0f;
    for (int s = 0; s < ns; ++s) {
      const float2 v = ml_s[s * kH + tid];
      const float w = v.x == -INFINITY ? 0.0f : exp2f(v.x - M) * v.y;
      wgt[s * kH + tid] = w;
      L += w;
    }
    Ls[tid] = L > 0.0f ? 1.0f / L : 0.0f;
    if (split == 0 && p.lse) p.lse[row * kH + tid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  float* cs = Ls + kH;   // the RoPE row of t: 32 cos, 32 sin
  float* sn = cs + 32;
  if (tid >= 64 && tid < 96) {
    cs[tid - 64] = p.rcos[(t_ok ? t : 0) * 32 + tid - 64];
    sn[tid - 64] = p.rsin[(t_ok ? t : 0) * 32 + tid - 64];
  }
  __syncthreads();
  // thread: a pair of dims (d, d + 1) of one head, weighted sum in split order
  for (int u = tid; u < (nd >> 1) * kH; u += kThreads) {
    const int h = u % kH, dl = 2 * (u / kH), d = d0 + dl;
    float o0 = 0.0f, o1 = 0.0f;
    for (int s = 0; s < ns; ++s) {
      const float w = wgt[s * kH + h];
      const __nv_bfloat16* src = sl_s + ((size_t)s * nd + dl) * kH + h;
      o0 = __fmaf_rn(w, __bfloat162float(src[0]), o0);
      o1 = __fmaf_rn(w, __bfloat162float(src[kH]), o1);
    }
    o0 *= Ls[h];
    o1 *= Ls[h];
    if (d >= kMixDn) {
      const int pi = (d - kMixDn) >> 1;
      const float y0 = o0 * cs[pi] + o1 * sn[pi];
      const float y1 = -o0 * sn[pi] + o1 * cs[pi];
      o0 = y0;
      o1 = y1;
    }
    *reinterpret_cast<__nv_bfloat162*>(p.out + (row * kH + h) * (int64_t)kD + d) = __floats2bfloat162_rn(o0, o1);
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

// Splits per row: as many as fill the SMs once, at most one per key tile.
int attn_decode_splits(int64_t rows, int64_t max_keys) {
  const int sms = device_sms() > 0 ? device_sms() : 148;
  const int64_t tiles = (max_keys + kTile - 1) / kTile;
  int64_t s = sms / (rows > 0 ? rows : 1);
  if (s > tiles) s = tiles;
  return (int)(s < 1 ? 1 : s);
}

bool attn_decode_applies(int H, int D, int R, int64_t rows, int k, bool sparse) {
  const int sms = device_sms() > 0 ? device_sms() : 148;
  return H == kH && D == kD && R == 64 && rows > 0 && rows < sms && (!sparse || k <= kMaxList);
}

size_t attn_decode_workspace(int64_t rows, int64_t max_keys) {
  const int64_t items = rows * attn_decode_splits(rows, max_keys);
  return al256((size_t)items * kH * kD * 2) + al256((size_t)items * kH * 2 * 4) + al256((size_t)rows * 4);
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
  uint8_t* base = reinterpret_cast<uint8_t*>(a.ws) + kWsHeader;
  p.part_o = reinterpret_cast<__nv_bfloat16*>(base);
  base += al256((size_t)items * kH * kD * 2);
  p.part_ml = reinterpret_cast<float*>(base);
  base += al256((size_t)items * kH * 2 * 4);
  p.arrive = reinterpret_cast<int*>(base);
  CUtensorMap tm_q;
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
  }
  cudaError_t e = cudaMemsetAsync(p.arrive, 0, (size_t)rows * 4, st);
  if (e != cudaSuccess) return e;
  static PerDevice attr;
  smem_limit_once(attr, reinterpret_cast<const void*>(attn_decode_kernel), (int)kSmemBytes);
  // every item resident at once (the row barrier waits on its siblings)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_decode_kernel, p, tm_q);
  return e;
}

}  // namespace csa
