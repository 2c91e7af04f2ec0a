// attn_tc.cu -- tensor-core (tcgen05 / TMEM) attention of every query over
// its compressed entries and its sliding window, mixed FP8/BF16 cache.
//
// xmsumi.com DeepSeek-V4 article, section "CSA（压缩稀疏注意力）": MQA over
// the selected compressed entries plus a sliding-window branch; section
// "HCA（重度压缩注意力）": dense attention over all compressed entries;
// section "关键技术细节": RoPE on the last 64 dims with inverse rotation of
// the output, RoPE dims BF16 and the rest FP8 in the KV cache.
//
// Persistent kernel, one CTA per SM.  A work item is one query token (all
// 64 heads share the KV: MQA) or, for small batches, a contiguous range of
// its key tiles (split-K; a second kernel merges the partial softmaxes).
// Keys run in tiles of 64 through a two-deep smem ring:
//   producer warps 4-7  fetch each tile's rows: TMA gathers of bf16 rows
//                       (prefill: the rows are expanded once up front) or
//                       loads of the 592-byte mixed rows dequantised in
//                       registers (decode), into a 64 x 512 bf16 tile,
//                       128-byte swizzled; the compacted entry list of the
//                       next item is bulk-copied one item ahead;
//   MMA warp 8          an event loop over two kinds of work, whichever is
//                       ready: S = Q K^T (M = 64 heads, N = 64 keys, K = 512)
//                       into TMEM, and O^T += V^T P^T (M = 128 dims x 4,
//                       N = 64 heads, K = 64 keys) into TMEM -- V = K, so
//                       the same smem tile is read K-major for QK^T and
//                       MN-major for PV; it also loads each item's query
//                       with TMA (dims 448..511 pre-rotated by a small
//                       per-row kernel);
//   softmax warps 0-3   read S from TMEM, online softmax in the exp2 domain
//                       with a lazy rescale of O^T (only when a running max
//                       grows by more than 2^8), write bf16 P to smem; at the
//                       end of an item normalise O, rotate its RoPE dims back
//                       and store bf16 (or store the partial state).
// Every ring slot has its own full / empty mbarrier, so a waiter is never
// more than one phase behind.  Waits are bounded: on expiry the CTA records a
// timeout flag in the workspace and gives up; the four softmax warps take
// that decision together, through a reducing named barrier.
#include <cuda.h>

#include <cstdlib>

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
constexpr int kMaxSplits = 256;   // split-K partial states per row (the combine stages their statistics)
constexpr int kThreads = 10 * 32;
constexpr int kMmaWarp = 8;       // QK^T issue, query loads, TMEM owner
constexpr int kPvWarp = 9;        // PV issue

constexpr uint32_t kQOff = 0;                     // 8 chunks x [64 heads x 128 B]
constexpr uint32_t kKVOff = 65536;                // 2 buffers x 8 chunks x [64 keys x 128 B]
constexpr uint32_t kPOff = kKVOff + 131072;       // 2 buffers x [64 heads x 64 keys bf16]
constexpr uint32_t kMiscOff = kPOff + 16384;      // barriers and per-head state
constexpr uint32_t kListOff = kMiscOff + 2048;    // int32 entry lists, two buffers
constexpr uint32_t kSmemBytes = 232448;           // 227 KiB
constexpr int kMaxList = (int)((kSmemBytes - 1024 - kListOff) / 8);   // per buffer (two buffers)

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;       // O^T: 4 blocks of 64 columns (heads); lanes = dims
constexpr uint32_t kTmemS = 256;     // S: 2 buffers of 64 columns (keys); M = 64 layout

constexpr uint32_t kWaitLimit = 1u << 20;    // suspending polls of one mbarrier wait
constexpr float kLazy = 8.0f;        // log2 growth of a running max that forces a rescale

struct Misc {
  uint64_t kv_full[2], kv_empty[2], s_full[2], p_full[2];
  uint64_t q_full, q_empty, o_full, o_empty, drain[2];
  uint64_t list_full[2], list_empty[2];  // entry list handover, double-buffered
  uint32_t tmem;
  int abort;
  alignas(16) float alpha[2][kH];   // per-head rescale factors of a tile, double-buffered
  alignas(16) float lsum[2][kH];    // per-head 1 / sum of an item, double-buffered (read as float4)
};
static_assert(sizeof(Misc) <= 2048, "Misc overflows its smem slot");
static_assert(offsetof(Misc, lsum) % 16 == 0 && offsetof(Misc, alpha) % 16 == 0, "vector reads of Misc");

__device__ __forceinline__ bool vabort(const Misc* ms) {
  return *reinterpret_cast<const volatile int*>(&ms->abort) != 0;
}

// Mixed 592-byte rows -> bf16 rows of 512 (exact), one warp per row.  Used
// when every row serves many queries, so the expansion is paid once.
__global__ void __launch_bounds__(256) expand_rows_kernel(const uint8_t* __restrict__ rows, int64_t n,
                                                          __nv_bfloat16* __restrict__ out) {
  pdl_begin();
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= n) return;
  const uint8_t* row = rows + r * kMixRow;
  uint4* dst = reinterpret_cast<uint4*>(out + r * kD);
  if (lane < 28) {
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);
    const float sc = __ldg(reinterpret_cast<const float*>(row + kMixScaleOff) + (lane >> 3));
    uint4 o0, o1;
    dequant16(c, sc, o0, o1);
    dst[2 * lane] = o0;
    dst[2 * lane + 1] = o1;
  } else {
    const int l4 = lane - 28;
    dst[56 + 2 * l4] = __ldg(reinterpret_cast<const uint4*>(row + kMixRopeOff) + 2 * l4);
    dst[56 + 2 * l4 + 1] = __ldg(reinterpret_cast<const uint4*>(row + kMixRopeOff) + 2 * l4 + 1);
  }
}

struct Params {
  const __nv_bfloat16* q;
  const int64_t* q_pos;
  int64_t Tq;
  const uint8_t* cache;
  int64_t N;
  int m;
  int k;
  const uint8_t* swa;
  const int64_t* swa_pos0;
  int64_t Ts;
  int W;
  float scale_log2;
  const float* rcos;
  const float* rsin;
  int64_t rope_rows;
  __nv_bfloat16* out;
  float* lse;
  void* ws;
  int64_t items;      // rows * nsplit
  int nsplit;
  float* part_o;      // [items, 64, 512] unnormalised O (split mode)
  float* part_ml;     // [items, 64, 2] running max (log2 units) and sum
  const __nv_bfloat16* xcache;   // bf16 copy of the cache rows [B, N, 512], or NULL
  const __nv_bfloat16* xg;       // or: every row's own keys in bf16, [rows, kp, 512], zero padded
  int64_t kp;                    // key slots per row of xg (a multiple of the tile)
  int64_t xrows;                 // rows of the bf16 copy (cache rows, then window rows)
  int64_t xwin0;                 // first window row in the copy (= B * N)
  const int32_t* clist;          // [rows, kpad] valid selected entries of each row, in idx order
  const int32_t* ccount;         // [rows] their number
  int kpad;                      // row stride of clist (multiple of 4)
};

// Keys of one work item: entries first (selected, in idx order, or all
// visible ones), then the window tokens; this split owns tiles [tlo, thi).
struct Item {
  int64_t it, row, b, t;
  bool t_ok;
  int ne, nwin, nkeys;
  int64_t w_lo, p0;
  int tlo, thi;
  int key_hi;
};

// The global loads an item description needs, issued one item ahead.
struct ItemPre {
  int64_t t, p0;
  int cnt;
};

template <bool DENSE>
__device__ __forceinline__ ItemPre item_fetch(const Params& p, int64_t it) {
  ItemPre r;
  r.t = -1;
  r.p0 = 0;
  r.cnt = 0;
  if (it < p.items) {
    const int64_t row = it / p.nsplit;
    r.t = p.q_pos[row];
    if (p.W > 0) r.p0 = p.swa_pos0[row / p.Tq];
    if (!DENSE) r.cnt = p.ccount[row];
  }
  return r;
}

template <bool DENSE>
__device__ __forceinline__ Item item_make(const Params& p, int64_t it, const ItemPre& r) {
  Item I;
  I.it = it;
  I.row = it / p.nsplit;
  const int split = (int)(it - I.row * p.nsplit);
  I.b = I.row / p.Tq;
  I.t = r.t;
  I.t_ok = I.t >= 0 && I.t < p.rope_rows;
  int ne = 0;
  if (I.t_ok) {
    if (DENSE) {
      const int64_t nv = (I.t + 1) / p.m;   // entries whose block ends at or before t
      ne = (int)(nv < p.N ? nv : p.N);
    } else {
      ne = min(r.cnt, kMaxList);
    }
  }
  I.ne = ne;
  const int64_t u_lo = I.t - p.W + 1 < 0 ? 0 : I.t - p.W + 1;
  I.p0 = r.p0;
  I.w_lo = u_lo < I.p0 ? I.p0 : u_lo;
  const int64_t w_hi = I.t < I.p0 + p.Ts - 1 ? I.t : I.p0 + p.Ts - 1;
  I.nwin = (I.t_ok && p.W > 0 && w_hi >= I.w_lo) ? (int)(w_hi - I.w_lo + 1) : 0;
  I.nkeys = I.ne + I.nwin;
  const int ntiles = (I.nkeys + kTile - 1) / kTile;
  const int per = (ntiles + p.nsplit - 1) / p.nsplit;
  I.tlo = min(ntiles, split * per);
  I.thi = min(ntiles, I.tlo + per);
  I.key_hi = min(I.nkeys, I.thi * kTile);
  return I;
}

// This CTA's items in order (blockIdx.x, + gridDim.x, ...), the loads of
// the next one in flight while the current one is worked on.
template <bool DENSE>
struct Cursor {
  int64_t next;
  ItemPre pre;
  __device__ __forceinline__ explicit Cursor(const Params& p) : next(blockIdx.x) { pre = item_fetch<DENSE>(p, next); }
  __device__ __forceinline__ bool any(const Params& p, Item& I) {
    if (next >= p.items) return false;
    I = item_make<DENSE>(p, next, pre);
    next += gridDim.x;
    pre = item_fetch<DENSE>(p, next);
    return true;
  }
  __device__ __forceinline__ bool nonempty(const Params& p, Item& I) {
    while (any(p, I))
      if (I.thi > I.tlo) return true;
    return false;
  }
  // like nonempty, but keeps only the item's index and loads (few registers)
  __device__ __forceinline__ int64_t seek(const Params& p, ItemPre& out) {
    Item I;
    while (next < p.items) {
      const int64_t it = next;
      out = pre;
      if (!any(p, I)) break;
      if (I.thi > I.tlo) return it;
    }
    return p.items;
  }
};

constexpr int kIdxBatch = 16;   // selected indices loaded per lane before any is used

// Per query row, ahead of the attention: the query's RoPE dims rotated to
// its position and rounded to bf16 (qr, [rows, 64 heads, 64 dims]), and for
// sparse attention the ordered list of its valid selected entries (idx >= 0,
// < N, block complete at the query's position); invalid ones set the
// device-check flag.  One block of 8 warps per row.
__global__ void __launch_bounds__(256)
prep_rows_kernel(const __nv_bfloat16* __restrict__ q, const int64_t* __restrict__ q_pos, const float* __restrict__ rcos,
                 const float* __restrict__ rsin, int64_t rope_rows, __nv_bfloat16* __restrict__ qr,
                 const int32_t* __restrict__ idx, int k, int kpad, int64_t N, int m, int32_t* __restrict__ clist,
                 int32_t* __restrict__ ccount, void* ws) {
  pdl_begin();
  const int64_t row = blockIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = q_pos[row];
  const bool t_ok = t >= 0 && t < rope_rows;
  {
    const float c = rcos[(t_ok ? t : 0) * 32 + lane], s = rsin[(t_ok ? t : 0) * 32 + lane];
    __nv_bfloat162 x[8];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh)
      x[hh] = *reinterpret_cast<const __nv_bfloat162*>(q + (row * kH + 8 * w + hh) * kD + kMixDn + 2 * lane);
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      const float2 f = __bfloat1622float2(x[hh]);
      const float y0 = __fsub_rn(__fmul_rn(f.x, c), __fmul_rn(f.y, s));
      const float y1 = __fadd_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, c));
      *reinterpret_cast<__nv_bfloat162*>(qr + (row * kH + 8 * w + hh) * 64 + 2 * lane) = __floats2bfloat162_rn(y0, y1);
    }
  }
  if (!idx || w != 0) return;
  int cnt = 0;
  for (int base = 0; base < k; base += 32 * kIdxBatch) {
    int32_t js[kIdxBatch];
#pragma unroll
    for (int i = 0; i < kIdxBatch; ++i) {
      const int r = base + 32 * i + lane;
      js[i] = r < k ? __ldg(idx + row * k + r) : -1;
    }
#pragma unroll
    for (int i = 0; i < kIdxBatch; ++i) {
      const int32_t j = js[i];
      const bool ok = t_ok && j >= 0 && (int64_t)j < N && (int64_t)(j + 1) * m - 1 <= t;
      if (t_ok && j >= 0 && !ok) flag_device_check(ws, (unsigned)j);
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (ok) clist[row * kpad + cnt + __popc(bal & ((1u << lane) - 1u))] = j;
      cnt += __popc(bal);
    }
  }
  if (lane == 0) ccount[row] = cnt;
}

// Per-row key rows in bf16 (decode): slot (r, key) of xg holds key `key` of
// query row r -- its selected (or, dense, visible) entries in order, then its
// window tokens -- expanded exactly from the mixed rows; slots past the row's
// keys are zero.  One warp per slot.
__global__ void __launch_bounds__(256)
gather_expand_kernel(const Params p, int64_t rows, int dense, __nv_bfloat16* __restrict__ xg) {
  pdl_begin();
  const int64_t slot = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t r = slot / p.kp;
  if (r >= rows) return;
  const int64_t key = slot - r * p.kp;
  const int64_t b = r / p.Tq, t = p.q_pos[r];
  const bool t_ok = t >= 0 && t < p.rope_rows;
  int64_t ne = 0;
  if (t_ok) {
    if (dense) {
      const int64_t nv = (t + 1) / p.m;
      ne = nv < p.N ? nv : p.N;
    } else {
      ne = p.ccount[r];
    }
  }
  const int64_t u_lo = t - p.W + 1 < 0 ? 0 : t - p.W + 1;
  const int64_t p0 = p.W > 0 ? p.swa_pos0[b] : 0;
  const int64_t w_lo = u_lo < p0 ? p0 : u_lo;
  const int64_t w_hi = t < p0 + p.Ts - 1 ? t : p0 + p.Ts - 1;
  const int64_t nwin = (t_ok && p.W > 0 && w_hi >= w_lo) ? w_hi - w_lo + 1 : 0;
  const uint8_t* row = nullptr;
  if (key < ne) row = p.cache + (b * p.N + (dense ? key : (int64_t)p.clist[r * p.kpad + key])) * kMixRow;
  else if (key < ne + nwin) row = p.swa + (b * p.Ts + (w_lo - p0 + (key - ne))) * kMixRow;
  uint4* dst = reinterpret_cast<uint4*>(xg + slot * kD);
  if (!row) {
    dst[2 * lane] = make_uint4(0, 0, 0, 0);
    dst[2 * lane + 1] = make_uint4(0, 0, 0, 0);
  } else if (lane < 28) {
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);
    const float sc = __ldg(reinterpret_cast<const float*>(row + kMixScaleOff) + (lane >> 3));
    uint4 o0, o1;
    dequant16(c, sc, o0, o1);
    dst[2 * lane] = o0;
    dst[2 * lane + 1] = o1;
  } else {
    const int l4 = lane - 28;
    dst[56 + 2 * l4] = __ldg(reinterpret_cast<const uint4*>(row + kMixRopeOff) + 2 * l4);
    dst[56 + 2 * l4 + 1] = __ldg(reinterpret_cast<const uint4*>(row + kMixRopeOff) + 2 * l4 + 1);
  }
}

template <bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const Params p, const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_qr) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kQOff;
  uint8_t* sKV = sm + kKVOff;
  uint8_t* sP = sm + kPOff;
  Misc* ms = reinterpret_cast<Misc*>(sm + kMiscOff);
  int32_t* list = reinterpret_cast<int32_t*>(sm + kListOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    ms->abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->kv_full[i], 4 + 128);   // per producer warp: one arrival, + one per lane
      mbar_init(&ms->kv_empty[i], 1);
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->p_full[i], 4);
      mbar_init(&ms->list_full[i], 1);
      mbar_init(&ms->list_empty[i], 4);
    }
    mbar_init(&ms->q_full, 1);
    mbar_init(&ms->q_empty, 1);
    mbar_init(&ms->o_full, 1);
    mbar_init(&ms->o_empty, 4);
    mbar_init(&ms->drain[0], 1);
    mbar_init(&ms->drain[1], 1);
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&ms->tmem, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = ms->tmem;

  if (warp >= 4 && warp < 8) {
    // ================================ producers ================================
    const int pw = warp - 4;
    Cursor<DENSE> cur(p);
    Item I;
    bool have = cur.nonempty(p, I);
    ItemPre pj;                  // the next item (for its list): index jn, loads pj
    int64_t jn = (!DENSE && have) ? cur.seek(p, pj) : p.items;
    uint32_t g = 0, nq = 0;      // tiles and non-empty items produced so far
    uint32_t nl = 0;             // entry lists issued (warp 0)
    bool ok = true;
    // entry list of item ordinal n -> smem buffer n & 1, once every producer
    // warp is done with item n - 2 (warp 0 issues)
    auto issue_list = [&](const Item& L, uint32_t n) -> bool {
      int good = 1;
      if (lane == 0) {
        if (n >= 2 && !mbar_wait(&ms->list_empty[n & 1], ((n >> 1) - 1) & 1, kWaitLimit)) {
          good = 0;
        } else {
          const uint32_t bytes = (uint32_t)((L.ne + 3) & ~3) * 4u;
          mbar_arrive_expect_tx(&ms->list_full[n & 1], bytes);
          if (bytes)
            bulk_copy_g2s(smem_u32(list + (n & 1) * kMaxList), p.clist + L.row * p.kpad, bytes,
                          &ms->list_full[n & 1]);
        }
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (good) nl = n + 1;
      return good != 0;
    };
    if (!DENSE && have && pw == 0) ok = issue_list(I, 0);
    while (have && ok && !vabort(ms)) {
      const int32_t* lst = list + (nq & 1) * kMaxList;
      if (!DENSE) {
        if (jn < p.items && pw == 0) ok = issue_list(item_make<DENSE>(p, jn, pj), nq + 1);
        if (ok && !mbar_wait(&ms->list_full[nq & 1], (nq >> 1) & 1, kWaitLimit)) ok = false;
        if (!ok) break;
      }
      if (p.xg) {
        // the row's keys are contiguous bf16 rows: 8 TMA boxes of 64 rows x
        // 64 columns per tile from producer warp 0; the others only arrive
        for (int tl = I.tlo; tl < I.thi; ++tl, ++g) {
          const int buf = g & 1;
          if (g >= 2 && !mbar_wait(&ms->kv_empty[buf], ((g >> 1) - 1) & 1, kWaitLimit)) {
            ok = false;
            break;
          }
          const uint32_t tb = smem_u32(sKV + buf * 65536);
          if (pw == 0) {
            if (lane == 0) mbar_arrive_expect_tx(&ms->kv_full[buf], kTile * kD * 2);
            __syncwarp();
            if (lane < 8)
              tma_load_2d(tb + lane * 8192, &tm_rows, 64 * lane, (int)(I.row * p.kp + (int64_t)tl * kTile),
                          &ms->kv_full[buf]);
          } else if (lane == 0) {
            mbar_arrive(&ms->kv_full[buf]);
          }
          cp_async_mbar_arrive_noinc(&ms->kv_full[buf]);   // no copies of this lane: arrives at once
          __syncwarp();
        }
      } else if (p.xcache) {
        // bf16 rows are ready.  Producer warp pw fetches rows 16 pw .. 16 pw + 15
        // of each tile: dims 0..255 by TMA gathers (4 rows x 128 bytes per
        // instruction, lanes 0..15) and dims 256..511 by 16-byte cp.async
        // (lane l: 16-byte unit l of each row's upper half) -- the TMA unit
        // alone cannot gather rows as fast as the tensor core consumes them.
        // Both complete on kv_full: the TMA by its byte count, the cp.async
        // through a counted asynchronous arrive of every lane.
        for (int tl = I.tlo; tl < I.thi; ++tl, ++g) {
          const int buf = g & 1;
          int myrow = (int)p.xrows;          // lane i < 16: row of key 16 pw + i (xrows: none)
          if (lane < 16) {
            const int key = tl * kTile + 16 * pw + lane;
            if (key < I.key_hi) {
              if (key < I.ne) myrow = (int)((int64_t)I.b * p.N + (DENSE ? (int64_t)key : (int64_t)lst[key]));
              else myrow = (int)(p.xwin0 + (int64_t)I.b * p.Ts + (I.w_lo - I.p0 + (key - I.ne)));
            }
          }
          if (g >= 2 && !mbar_wait(&ms->kv_empty[buf], ((g >> 1) - 1) & 1, kWaitLimit)) {
            ok = false;
            break;
          }
          const uint32_t tb = smem_u32(sKV + buf * 65536);
          if (lane == 0) mbar_arrive_expect_tx(&ms->kv_full[buf], 16 * (kD / 2) * 2);
          __syncwarp();
          {
            const int rg = (lane >> 2) & 3, cb = lane & 3;
            const int y0 = __shfl_sync(0xffffffffu, myrow, 4 * rg);
            const int y1 = __shfl_sync(0xffffffffu, myrow, 4 * rg + 1);
            const int y2 = __shfl_sync(0xffffffffu, myrow, 4 * rg + 2);
            const int y3 = __shfl_sync(0xffffffffu, myrow, 4 * rg + 3);
            if (lane < 16)
              tma_gather4(tb + cb * 8192 + (uint32_t)(16 * pw + 4 * rg) * 128u, &tm_rows, 64 * cb, y0, y1, y2, y3,
                          &ms->kv_full[buf]);
          }
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const int row = __shfl_sync(0xffffffffu, myrow, rr);
            const uint32_t r = (uint32_t)(16 * pw + rr);
            const bool v = row < p.xrows;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.xcache) + (size_t)(v ? row : 0) * (kD * 2) +
                                 kD + 16 * lane;
            cp_async16_zfill(tb + (4 + (lane >> 3)) * 8192 + r * 128u + ((((uint32_t)lane & 7u) ^ (r & 7u)) << 4), src,
                             v ? 16u : 0u);
          }
          cp_async_mbar_arrive_noinc(&ms->kv_full[buf]);
          __syncwarp();
        }
      } else {
        // mixed rows, dequantised here: this warp takes rows pw + 4 rr of the
        // tile, 16 of them in flight per lane
        for (int tl = I.tlo; tl < I.thi; ++tl, ++g) {
          const int buf = g & 1;
          const int kbase = tl * kTile;
          uint4 c[16];
          float sc[16];
          const uint8_t* rowp[16];
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const int key = kbase + pw + 4 * rr;
            const uint8_t* row = nullptr;
            if (key < I.key_hi) {
              if (key < I.ne) {
                const int64_t j = DENSE ? (int64_t)key : (int64_t)lst[key];
                row = p.cache + ((size_t)I.b * p.N + j) * kMixRow;
              } else {
                row = p.swa + ((size_t)I.b * p.Ts + (I.w_lo - I.p0 + (key - I.ne))) * kMixRow;
              }
            }
            rowp[rr] = row;
            c[rr] = make_uint4(0, 0, 0, 0);
            sc[rr] = 0.0f;
            if (lane < 28 && row) {
              c[rr] = __ldg(reinterpret_cast<const uint4*>(row) + lane);
              sc[rr] = __ldg(reinterpret_cast<const float*>(row + kMixScaleOff) + (lane >> 3));
            }
          }
          if (g >= 2 && !mbar_wait(&ms->kv_empty[buf], ((g >> 1) - 1) & 1, kWaitLimit)) {
            ok = false;
            break;
          }
          uint8_t* kv = sKV + buf * 65536;
          const uint32_t aKV = smem_u32(kv);
          if (lane >= 28) {                 // bf16 RoPE columns: async copies first
            const int l4 = lane - 28;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
              const int r = pw + 4 * rr;
              if (rowp[rr]) {
                cp_async16(aKV + 7 * 8192 + sw128(r, 2 * l4), rowp[rr] + kMixRopeOff + 32 * l4);
                cp_async16(aKV + 7 * 8192 + sw128(r, 2 * l4 + 1), rowp[rr] + kMixRopeOff + 32 * l4 + 16);
              } else {
                *reinterpret_cast<uint4*>(kv + 7 * 8192 + sw128(r, 2 * l4)) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(kv + 7 * 8192 + sw128(r, 2 * l4 + 1)) = make_uint4(0, 0, 0, 0);
              }
            }
          } else {                          // FP8 columns: dequantise
            uint8_t* dst = kv + (lane >> 2) * 8192;
            const uint32_t sub = 2 * (lane & 3);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
              const int r = pw + 4 * rr;
              uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
              if (rowp[rr]) dequant16(c[rr], sc[rr], o0, o1);
              *reinterpret_cast<uint4*>(dst + sw128(r, sub)) = o0;
              *reinterpret_cast<uint4*>(dst + sw128(r, sub + 1)) = o1;
            }
          }
          cp_async_wait_all();
          fence_proxy_async();
          cp_async_mbar_arrive_noinc(&ms->kv_full[buf]);   // nothing in flight: arrives at once
          __syncwarp();
          if (lane == 0) mbar_arrive(&ms->kv_full[buf]);
        }
      }
      if (!ok) break;
      if (!DENSE) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms->list_empty[nq & 1]);
      }
      ++nq;
      if (DENSE) {
        have = cur.nonempty(p, I);
      } else {
        have = jn < p.items;
        if (have) {
          I = item_make<DENSE>(p, jn, pj);
          jn = cur.seek(p, pj);
        }
      }
    }
    if (!ok) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
    }
    // copies of this warp still in flight land before the CTA can exit
    if (p.xcache && g > 0) mbar_wait(&ms->kv_full[(g - 1) & 1], ((g - 1) >> 1) & 1, kWaitLimit);
    if (nl > 0) mbar_wait(&ms->list_full[(nl - 1) & 1], ((nl - 1) >> 1) & 1, kWaitLimit);
  } else if (warp == kMmaWarp) {
    // ============================== QK^T issue ==============================
    // S of tile g goes to TMEM buffer g & 1; it is written once the softmax
    // has released the buffer's previous tile (its P is ready) and the keys
    // are in.  The query of the next item is loaded when the last QK^T of
    // this one has completed, and pulled into L2 one item earlier.
    const uint32_t aQ = smem_u32(sQ), aKV = smem_u32(sKV);
    constexpr uint32_t idQK = idesc_bf16(64, kTile, 0, 0);
    Cursor<DENSE> cur(p);
    Item I, In;
    bool have = cur.nonempty(p, I);
    bool have_n = have && cur.nonempty(p, In);
    uint32_t g = 0, nq = 0;
    bool ok = true, q_pending = false;
    auto issue_q = [&](int64_t row) {
      if (lane == 0) mbar_arrive_expect_tx(&ms->q_full, kH * kD * 2);
      __syncwarp();
      if (lane < 7) tma_load_2d(aQ + lane * 8192, &tm_q, 64 * lane, (int)(row * kH), &ms->q_full);
      else if (lane == 7) tma_load_2d(aQ + 7 * 8192, &tm_qr, 0, (int)(row * kH), &ms->q_full);
      __syncwarp();
    };
    while (have && ok && !vabort(ms)) {
      if (nq > 0 && !mbar_wait(&ms->q_empty, (nq - 1) & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      issue_q(I.row);
      q_pending = true;
      if (have_n && lane == 0) {   // the next item's query: into L2 now
        prefetch_l2(p.q + In.row * (int64_t)(kH * kD), kH * kD * 2);
      }
      if (!mbar_wait(&ms->q_full, nq & 1, kWaitLimit)) {
        ok = false;
        break;
      }
      q_pending = false;
      for (int tl = I.tlo; tl < I.thi; ++tl, ++g) {
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
        fence_proxy_async();   // the tile's cp.async part was written through the generic proxy
        const uint32_t dS = tmem + kTmemS + 64u * (g & 1);
        const uint64_t qd0 = sdesc_sw128(aQ, 16, 1024);
        const uint64_t kd0 = sdesc_sw128(aKV + (g & 1) * 65536, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
          mma_bf16_elect(dS, qd0 + off, kd0 + off, idQK, kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(&ms->s_full[g & 1]);
        if (tl == I.thi - 1) mma_commit_elect(&ms->q_empty);
        __syncwarp();
      }
      if (!ok) break;
      ++nq;
      I = In;
      have = have_n;
      if (have) have_n = cur.nonempty(p, In);
    }
    if (!ok) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
      if (q_pending) mbar_wait(&ms->q_full, nq & 1, kWaitLimit);   // the query copy in flight
    }
    // every MMA this warp issued completes before TMEM is released
    mma_commit_elect(&ms->drain[0]);
    __syncwarp();
    mbar_wait(&ms->drain[0], 0, kWaitLimit);
  } else if (warp == kPvWarp) {
    // ================================ PV issue ================================
    // O^T += V^T P^T as soon as P of the tile is in smem; the first tile of
    // an item overwrites O^T, so it waits for the previous item's epilogue.
    // Its completion frees the tile's ring slot (kv_empty).
    const uint32_t aKV = smem_u32(sKV), aP = smem_u32(sP);
    constexpr uint32_t idPV = idesc_bf16(128, kH, 1, 0);
    Cursor<DENSE> cur(p);
    Item I;
    uint32_t g = 0, nq = 0;
    bool ok = true;
    while (ok && !vabort(ms) && cur.nonempty(p, I)) {
      for (int tl = I.tlo; tl < I.thi; ++tl, ++g) {
        const bool first = tl == I.tlo, last = tl == I.thi - 1;
        if (!mbar_wait(&ms->p_full[g & 1], (g >> 1) & 1, kWaitLimit) ||
            (first && nq > 0 && !mbar_wait(&ms->o_empty, (nq - 1) & 1, kWaitLimit))) {
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
                           pd0 + (uint64_t)((ks * 32) >> 4), idPV, (!first || ks > 0) ? 1u : 0u);
        }
        mma_commit_elect(&ms->kv_empty[g & 1]);
        if (last) mma_commit_elect(&ms->o_full);
        __syncwarp();
      }
      ++nq;
    }
    if (!ok) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
    }
    mma_commit_elect(&ms->drain[1]);
    __syncwarp();
    mbar_wait(&ms->drain[1], 0, kWaitLimit);
  } else {
    // ============================ softmax / epilogue ============================
    // S (64 heads x 64 keys) sits in lanes 0-15 of every TMEM quadrant; the
    // 16x256b load spreads those 16 rows over all 32 lanes: lane t holds rows
    // ra = t / 4 and rb = 8 + t / 4 of its quadrant, keys 8j + 2 (t % 4) and
    // 8j + 2 (t % 4) + 1, j = 0..7.  Row maxima reduce over the 4 lanes of a
    // row; row sums stay per lane until the epilogue.
    const int qd = warp;
    const int cq = 2 * (lane & 3);
    const int ha = 16 * qd + (lane >> 2), hb = ha + 8;
    const bool leader = (lane & 3) == 0;
    const bool split = p.part_o != nullptr;
    const uint32_t tq_lane = (uint32_t)(32 * qd) << 16;   // this warp's TMEM lane quadrant
    Cursor<DENSE> cur(p);
    Item I;
    uint32_t g = 0, nq = 0;
    bool fail = false, stop = false;
    while (!stop && cur.any(p, I)) {
      const int64_t it = I.it;
      if (tid == 0 && I.row * p.nsplit == it) {
        if (!I.t_ok) flag_device_check(p.ws, 0x40000000u);
        const int64_t u_lo = I.t - p.W + 1 < 0 ? 0 : I.t - p.W + 1;
        if (I.t_ok && p.W > 0 && I.nwin < I.t - u_lo + 1) flag_device_check(p.ws, 0x80000000u);
      }
      const float* cs = p.rcos + (I.t_ok ? I.t : 0) * 32;
      const float* sn = p.rsin + (I.t_ok ? I.t : 0) * 32;
      if (I.thi <= I.tlo) {           // no keys: zero output / empty partial state
        if (split) {
          for (int e = tid; e < kH * kD; e += 128) p.part_o[it * (kH * kD) + e] = 0.0f;
          if (tid < kH) {
            p.part_ml[(it * kH + tid) * 2] = -INFINITY;
            p.part_ml[(it * kH + tid) * 2 + 1] = 0.0f;
          }
        } else {
          for (int e = tid; e < kH * kD; e += 128) p.out[I.row * (kH * kD) + e] = __float2bfloat16_rn(0.0f);
          if (p.lse && tid < kH) p.lse[I.row * kH + tid] = -INFINITY;
        }
        continue;
      }
      float ma = -INFINITY, mb = -INFINITY, la = 0.0f, lb = 0.0f;
      for (int tl = I.tlo; tl < I.thi; ++tl, ++g) {
        if (!fail && !mbar_wait(&ms->s_full[g & 1], (g >> 1) & 1, kWaitLimit)) fail = true;
        fence_after_sync();
        const int nvalid = min(kTile, I.key_hi - tl * kTile);
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
        const float aa = need_a ? ex2(ma - na) : 1.0f;   // 2^-inf = 0 on the first tile
        const float ab = need_b ? ex2(mb - nb) : 1.0f;
        if (tl > I.tlo) {
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
        // P buffer g & 1 was last read by PV of tile g - 2 (another warp's
        // MMAs: S being ready does not imply it), so wait for that PV
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
      if (stop) break;
      // ---- epilogue: the item's O^T is complete after its last PV ----
      la += __shfl_xor_sync(0xffffffffu, la, 1);
      la += __shfl_xor_sync(0xffffffffu, la, 2);
      lb += __shfl_xor_sync(0xffffffffu, lb, 1);
      lb += __shfl_xor_sync(0xffffffffu, lb, 2);
      if (!fail && !mbar_wait(&ms->o_full, nq & 1, kWaitLimit)) fail = true;
      fence_after_sync();
      float* lsv = ms->lsum[nq & 1];
      if (leader) {
        lsv[ha] = la > 0.0f ? 1.0f / la : 0.0f;   // per-head 1/sum for every lane
        lsv[hb] = lb > 0.0f ? 1.0f / lb : 0.0f;
        if (split) {
          p.part_ml[(it * kH + ha) * 2] = ma;
          p.part_ml[(it * kH + ha) * 2 + 1] = la;
          p.part_ml[(it * kH + hb) * 2] = mb;
          p.part_ml[(it * kH + hb) * 2 + 1] = lb;
        } else if (p.lse) {
          p.lse[I.row * kH + ha] = la > 0.0f ? (ma + log2f(la)) * 0.69314718055994531f : -INFINITY;
          p.lse[I.row * kH + hb] = lb > 0.0f ? (mb + log2f(lb)) * 0.69314718055994531f : -INFINITY;
        }
      }
      if (group_vote(__any_sync(0xffffffffu, fail || vabort(ms))) != 0) break;
      if (split) {
        float* po = p.part_o + it * (int64_t)(kH * kD);
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + tq_lane + kTmemO + 32u * c, o);
          tmem_wait_ld();
          const int d = 128 * (c >> 1) + 32 * qd + lane;
          const int h0 = 32 * (c & 1);
#pragma unroll
          for (int j = 0; j < 32; ++j) po[(h0 + j) * kD + d] = __uint_as_float(o[j]);
        }
      } else {
        // lane pairs swap values so that each lane holds two adjacent dims of
        // one head: lane 2i takes head j, lane 2i + 1 head j + 1; a RoPE pair
        // is then rotated back within one lane and stored as one bf16x2.  The
        // phases (scale all, swap all, store all) keep the latencies overlapped.
        __nv_bfloat16* og = p.out + I.row * (int64_t)(kH * kD);
        const int odd = lane & 1;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          const int mt = c >> 1, hh = c & 1;
          uint32_t o[32];
          tmem_ld32(tmem + tq_lane + kTmemO + 64u * mt + 32u * hh, o);
          float inv[32];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(lsv + 32 * hh + j);
            inv[j] = v4.x;
            inv[j + 1] = v4.y;
            inv[j + 2] = v4.z;
            inv[j + 3] = v4.w;
          }
          const int de = 128 * mt + 32 * qd + (lane & ~1);
          const bool rope = de >= kMixDn;          // warp-uniform
          const int pi = rope ? (de - kMixDn) >> 1 : 0;
          const float cc = rope ? cs[pi] : 1.0f, ss = rope ? sn[pi] : 0.0f;
          tmem_wait_ld();
          float f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(o[j]) * inv[j];
          float r[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = __shfl_xor_sync(0xffffffffu, odd ? f[2 * j] : f[2 * j + 1], 1);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float x = odd ? r[j] : f[2 * j], y = odd ? f[2 * j + 1] : r[j];   // even / odd dim
            if (rope) {
              const float x2 = x * cc + y * ss;
              const float y2 = y * cc - x * ss;
              x = x2;
              y = y2;
            }
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(x, y);
            pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint32_t* orow = reinterpret_cast<uint32_t*>(og + (int64_t)(32 * hh + odd) * kD + de);
#pragma unroll
          for (int j = 0; j < 16; ++j) orow[(int64_t)j * kD] = pk[j];   // head 32 hh + 2 j + odd
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->o_empty);
      ++nq;
    }
    if (fail) {
      ms->abort = 1;
      if (lane == 0) flag_timeout(p.ws);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the split partial softmax states of one (query row, head) into out
// and lse: one CTA per pair, thread t owns dims 2t and 2t + 1 (a RoPE pair when
// 2t >= 448); the partial states are weighted by 2^(m_s - max m) in split order.
__global__ void __launch_bounds__(256) attn_combine_kernel(const Params p) {
  pdl_begin();
  __shared__ float m_s[kMaxSplits], l_s[kMaxSplits];
  const int64_t row = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int64_t t = p.q_pos[row];
  const bool t_ok = t >= 0 && t < p.rope_rows;
  const int d0 = 2 * tid;
  const int ns = p.nsplit;
  // the splits' running max and sum, read once by the CTA
  const float* ml = p.part_ml + (row * ns * kH + h) * 2;   // split s at + s * kH * 2
  for (int s = tid; s < ns; s += 256) {
    m_s[s] = ml[s * kH * 2];
    l_s[s] = ml[s * kH * 2 + 1];
  }
  __syncthreads();
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, m_s[s]);
  float L = 0.0f, o0 = 0.0f, o1 = 0.0f;
  if (M != -INFINITY) {
    const float* po = p.part_o + row * ns * (int64_t)(kH * kD) + h * kD + d0;
    // in split order as before; the partial rows' loads of 8 splits issued together
#pragma unroll 8
    for (int s = 0; s < ns; ++s) {
      const float mi = m_s[s];
      if (mi != -INFINITY) {
        const float w = exp2f(mi - M);
        L += w * l_s[s];
        const float2 v = *reinterpret_cast<const float2*>(po + s * (int64_t)(kH * kD));
        o0 += w * v.x;
        o1 += w * v.y;
      }
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  o0 *= inv;
  o1 *= inv;
  if (d0 >= kMixDn) {
    const float* cs = p.rcos + (t_ok ? t : 0) * 32;
    const float* sn = p.rsin + (t_ok ? t : 0) * 32;
    const int pi = (d0 - kMixDn) >> 1;
    const float y0 = o0 * cs[pi] + o1 * sn[pi];
    const float y1 = -o0 * sn[pi] + o1 * cs[pi];
    o0 = y0;
    o1 = y1;
  }
  *reinterpret_cast<__nv_bfloat162*>(p.out + row * (int64_t)(kH * kD) + h * kD + d0) = __floats2bfloat162_rn(o0, o1);
  if (tid == 0 && p.lse) p.lse[row * kH + h] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

int num_sms() {
  const int n = device_sms();
  return n > 0 ? n : 148;
}

// Split count: 1 when there are enough rows to fill the GPU, else enough
// splits to give every SM an item (at most one per 64-key tile).
int choose_splits(int64_t rows, int64_t max_keys) {
  const int sms = num_sms();
  if (rows >= sms) return 1;
  const int64_t tiles = (max_keys + kTile - 1) / kTile;
  // rows x splits at most one item per SM: a second round for a few items
  // would double the time of the call
  int64_t s = sms / rows;
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  return (int)(s < 1 ? 1 : s);
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// CSA_ATTN_DECODE=0 keeps few-row calls on the long-row path (for A/B tests)
bool attn_decode_disabled() {
  const char* e = getenv("CSA_ATTN_DECODE");
  return e && e[0] == '0';
}

// How a call runs: the split count (partial states in the workspace) and
// whether the cache and window rows are first expanded to bf16 in the
// workspace -- worth it when every row serves many queries (prefill), not
// when each is read about once (decode).
struct Plan {
  int nsplit;
  bool expand;              // shared bf16 copy of all cache and window rows (prefill)
  bool gather;              // or every row's own keys in bf16 (decode)
  int kpad;
  int64_t kp;               // key slots per row when gathered
  size_t qr_bytes, list_bytes, part_bytes, x_bytes, g_bytes;
};

Plan make_plan(int B, int64_t Tq, int64_t max_keys, int64_t N, int64_t Ts, int k) {
  Plan pl;
  const int64_t rows = (int64_t)B * Tq;
  pl.kpad = (k + 3) & ~3;
  pl.qr_bytes = al256((size_t)rows * kH * 64 * 2);
  pl.list_bytes = k > 0 ? al256((size_t)rows * pl.kpad * 4) + al256((size_t)rows * 4) : 0;
  pl.nsplit = choose_splits(rows, max_keys);
  pl.part_bytes = pl.nsplit > 1 ? al256((size_t)rows * pl.nsplit * ((size_t)kH * kD * 4 + (size_t)kH * 2 * 4)) : 0;
  const double uses = (double)rows * (double)max_keys;
  const double nrows = (double)B * (double)(N + Ts);
  pl.expand = nrows > 0 && uses >= 8.0 * nrows;
  pl.x_bytes = pl.expand ? al256((size_t)B * (size_t)(N + Ts) * kD * 2) : 0;
  pl.kp = (max_keys + kTile - 1) / kTile * kTile;
  const double gbytes = (double)rows * (double)pl.kp * kD * 2;
  pl.gather = !pl.expand && pl.kp > 0 && gbytes <= (double)(2ull << 30) && (double)rows * pl.kp < 2147483647.0;
  pl.g_bytes = pl.gather ? al256((size_t)gbytes) : 0;
  return pl;
}

// cuTensorMapEncodeTiled, fetched from the driver once
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// Tensor map over packed bf16 rows of `width` elements: boxes of 64 columns
// x box_rows rows, 128-byte swizzle, zero fill outside.
bool make_row_map(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t attn_tc_workspace(int B, int64_t Tq, int H, int D, int64_t max_keys, int64_t N, int64_t Ts, int k) {
  if (H != kH || D != kD) return 0;
  const int64_t rows = (int64_t)B * Tq;
  if (attn_decode_applies(H, D, 64, rows, k, k > 0)) return attn_decode_workspace(rows, max_keys);
  const Plan pl = make_plan(B, Tq, max_keys, N, Ts, k);
  return pl.qr_bytes + pl.list_bytes + pl.part_bytes + pl.x_bytes + pl.g_bytes;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.Tq;
  if (rows == 0) return cudaSuccess;
  if (a.H != kH || a.D != kD || a.R != 64) return launch_attn_simt(a, st);
  if (a.idx && a.k > kMaxList) return launch_attn_simt(a, st);
  // few rows: the one-launch decode kernel, when its scratch is given
  if (attn_decode_applies(a.H, a.D, a.R, rows, a.idx ? a.k : 0, a.idx != nullptr) && !attn_decode_disabled() &&
      a.ws_bytes >= kWsHeader + attn_decode_workspace(rows, a.max_keys))
    return launch_attn_decode(a, st);
  Params p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.q_pos = a.q_pos;
  p.Tq = a.Tq;
  p.cache = reinterpret_cast<const uint8_t*>(a.cache);
  p.N = a.N;
  p.m = a.m;
  p.k = a.idx ? a.k : 0;
  p.swa = reinterpret_cast<const uint8_t*>(a.swa);
  p.swa_pos0 = a.swa_pos0;
  p.Ts = a.Ts;
  p.W = a.W;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.rcos = a.rcos;
  p.rsin = a.rsin;
  p.rope_rows = a.rope_rows;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.ws = a.ws;
  p.part_o = nullptr;
  p.part_ml = nullptr;
  p.xcache = nullptr;
  Plan pl = make_plan(a.B, a.Tq, a.max_keys, a.N, a.W > 0 ? a.Ts : 0, a.idx ? a.k : 0);
  size_t avail = a.ws_bytes > csa::kWsHeader ? a.ws_bytes - csa::kWsHeader : 0;
  uint8_t* base = reinterpret_cast<uint8_t*>(a.ws) + csa::kWsHeader;
  // the rotated query dims and the entry lists are required
  if (pl.qr_bytes + pl.list_bytes > avail) return launch_attn_simt(a, st);
  __nv_bfloat16* qr = reinterpret_cast<__nv_bfloat16*>(base);
  base += pl.qr_bytes;
  avail -= pl.qr_bytes;
  p.kpad = pl.kpad;
  p.clist = nullptr;
  p.ccount = nullptr;
  if (a.idx) {
    p.clist = reinterpret_cast<int32_t*>(base);
    p.ccount = reinterpret_cast<int32_t*>(base + al256((size_t)rows * pl.kpad * 4));
    base += pl.list_bytes;
    avail -= pl.list_bytes;
  }
  launch_pdl(prep_rows_kernel, dim3((unsigned)rows), dim3(256), 0, st, p.q, a.q_pos, a.rcos, a.rsin, a.rope_rows, qr, a.idx, p.k, pl.kpad,
                                                   a.N, a.m, const_cast<int32_t*>(p.clist),
                                                   const_cast<int32_t*>(p.ccount), a.ws);
  if (pl.nsplit > 1 && pl.part_bytes > avail) {   // too little scratch: no split
    pl.nsplit = 1;
    pl.part_bytes = 0;
  }
  if (pl.expand && pl.part_bytes + pl.x_bytes > avail) pl.expand = false;
  if (pl.gather && pl.part_bytes + pl.g_bytes > avail) pl.gather = false;
  if ((int64_t)a.B * (a.N + (a.W > 0 ? a.Ts : 0)) >= INT32_MAX) pl.expand = false;   // TMA rows are int32
  p.nsplit = pl.nsplit;
  p.items = rows * p.nsplit;
  if (p.nsplit > 1) {
    p.part_o = reinterpret_cast<float*>(base);
    p.part_ml = reinterpret_cast<float*>(base + (size_t)p.items * kH * kD * 4);
    base += pl.part_bytes;
  }
  CUtensorMap tm_q, tm_qr, tm_rows;
  if (!make_row_map(&tm_q, a.q, kD, (uint64_t)rows * kH, 64)) return cudaErrorInvalidValue;
  if (!make_row_map(&tm_qr, qr, 64, (uint64_t)rows * kH, 64)) return cudaErrorInvalidValue;
  tm_rows = tm_q;
  p.xrows = 0;
  p.xwin0 = 0;
  p.xg = nullptr;
  p.kp = pl.kp;
  if (pl.gather) {
    __nv_bfloat16* xg = reinterpret_cast<__nv_bfloat16*>(base);
    const int64_t slots = rows * pl.kp;
    launch_pdl(gather_expand_kernel, dim3((unsigned)((slots + 7) / 8)), dim3(256), 0, st, p, rows, a.idx ? 0 : 1, xg);
    p.xg = xg;
    if (!make_row_map(&tm_rows, xg, kD, (uint64_t)slots, 64)) return cudaErrorInvalidValue;
  } else if (pl.expand) {
    const int64_t nc = (int64_t)a.B * a.N, nw = (a.W > 0) ? (int64_t)a.B * a.Ts : 0;
    __nv_bfloat16* xc = reinterpret_cast<__nv_bfloat16*>(base);
    if (nc > 0) launch_pdl(expand_rows_kernel, dim3((unsigned)((nc + 7) / 8)), dim3(256), 0, st, p.cache, nc, xc);
    if (nw > 0) launch_pdl(expand_rows_kernel, dim3((unsigned)((nw + 7) / 8)), dim3(256), 0, st, p.swa, nw, xc + nc * kD);
    p.xcache = xc;
    p.xrows = nc + nw;
    p.xwin0 = nc;
    if (!make_row_map(&tm_rows, xc, kD, (uint64_t)(nc + nw), 1)) return cudaErrorInvalidValue;
  }
  const int grid = (int)(p.items < num_sms() ? p.items : num_sms());
  static PerDevice attr_sparse, attr_dense;
  if (a.idx) {
    smem_limit_once(attr_sparse, reinterpret_cast<const void*>(attn_tc_kernel<false>), (int)kSmemBytes);
    launch_pdl(attn_tc_kernel<false>, dim3(grid), dim3(kThreads), kSmemBytes, st, p, tm_rows, tm_q, tm_qr);
  } else {
    smem_limit_once(attr_dense, reinterpret_cast<const void*>(attn_tc_kernel<true>), (int)kSmemBytes);
    launch_pdl(attn_tc_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes, st, p, tm_rows, tm_q, tm_qr);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.nsplit == 1) return e;
  launch_pdl(attn_combine_kernel, dim3(dim3((unsigned)rows, kH)), dim3(256), 0, st, p);
  return cudaGetLastError();
}

}  // namespace csa
