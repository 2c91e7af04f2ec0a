/*
 * csa_b300.h -- C ABI of the B300 (sm_103a) compressed-attention library
 * libcsa_b300.so: DeepSeek-V4's hybrid attention, compressed sparse
 * attention (CSA) and heavily compressed attention (HCA).
 *
 * Sources (page title, section) cited below:
 *  [XM] xmsumi.com DeepSeek-V4 article: "CSA（压缩稀疏注意力）",
 *       "HCA（重度压缩注意力）", "关键技术细节" (key technical details), and the
 *       heterogeneous KV cache paragraph under "百万Token 长上下文真实表现".
 *  [HU] "DeepSeek-V4 — MoE nyelvmodellek milliós kontextussal" (hortopato.cc
 *       wiki): the CSA list (Tömörítés, Lightning Indexer, Sliding Window
 *       figyelem) and "Heavily Compressed Attention (HCA)".
 *  [ZC] zcldvi.com DeepSeek-V4 news article: FP4 indexer, lossless FP4->FP8,
 *       the window branch in both attentions.
 *
 * Conventions shared by every call
 *  - Return value: CSA_OK or a negative csa status.  CSA_ERR_INVALID_ARG and
 *    CSA_ERR_UNSUPPORTED are returned before anything is enqueued; the text
 *    of the last error of the calling thread is in csa_last_error().
 *  - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream).  They never allocate, free or
 *    synchronise.
 *  - Every pointer marked (device) is a device pointer owned by the caller;
 *    arrays are dense, row-major, in the shapes given, and must not overlap
 *    the outputs.  Pointers marked (host) are host memory.
 *  - Scratch: calls that need it take `ws` (device, at least the size given
 *    by csa_workspace_size, 256-byte aligned) and its size `ws_bytes`.  The
 *    first 16 bytes of ws are a status block of sticky device-check flags:
 *    clear it with csa_status_reset once before first use, read it with
 *    csa_status_read.  A kernel that meets an index it must not follow (an
 *    entry >= N or not yet visible, a window row outside the window cache)
 *    skips that key and sets CSA_FLAG_DEVICE_CHECK; a bounded wait that
 *    expires sets CSA_FLAG_TIMEOUT.  Calls that overlap on the GPU must use
 *    different workspaces.
 *  - Formats: CSA_FMT_F32 rows are C fp32 channels.  CSA_FMT_MIXED592 rows
 *    (C = 512, the last 64 channels RoPE) are 592 bytes: [0,448) E4M3 codes
 *    of the 448 non-RoPE channels, each scaled by 2^-e_g of its 128-channel
 *    group g (groups of 128,128,128,64); [448,576) the 64 RoPE channels as
 *    bf16 (little endian, nearest-even); [576,592) four fp32 scales 2^e_g,
 *    e_g the smallest integer with max|v| / 2^e_g <= 448 (>= -126; 0 for an
 *    all-zero group).  [XM] key technical details: RoPE dims in BF16, the
 *    rest in FP8.  CSA_FMT_MXFP4 (indexer keys, C a multiple of 32): C/2
 *    bytes of E2M1 codes (even element in the low nibble) per row plus C/32
 *    UE8M0 scale bytes per row in a separate array; scale exponent =
 *    floor(log2 max|v|) - 2 over each block of 32 (OCP MX v1.0).
 *    CSA_FMT_FP8B32 (FP8 indexer keys, C = 32 or 64): C E4M3 codes per row
 *    (one byte each) plus C/32 scale bytes per row in a separate array,
 *    e + 127 with e the smallest integer such that max|v| / 2^e <= 448 over
 *    the block of 32 (the mixed rows' group rule: no element saturates; 0 for
 *    an all-zero block, >= -126).  [XM] "算力与内存效率": an FP4 x FP8
 *    product runs at the FP8 x FP8 rate; [ZC]: FP4 -> FP8 is lossless.
 *  - RoPE: rope_cos / rope_sin (device, fp32 [rope_rows, R/2]) hold
 *    cos/sin(p * base^(-2i/R)); pairs (2i, 2i+1) of the last R channels
 *    rotate by angle p*theta_i.  Build them with csa_rope_table.
 *    [XM] key technical details: RoPE acts on the last 64 dims of q and of
 *    the KV entries, and the attention output gets the inverse rotation.
 */
#ifndef CSA_B300_H
#define CSA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA_OK 0
#define CSA_ERR_INVALID_ARG (-1)
#define CSA_ERR_UNSUPPORTED (-2)
#define CSA_ERR_CUDA (-3)
#define CSA_ERR_DEVICE_CHECK (-4)
#define CSA_ERR_TIMEOUT (-5)

#define CSA_FLAG_DEVICE_CHECK 1u
#define CSA_FLAG_TIMEOUT 2u

#define CSA_DTYPE_F32 0
#define CSA_DTYPE_BF16 1

#define CSA_FMT_F32 0
#define CSA_FMT_MIXED592 1
#define CSA_FMT_MXFP4 2
#define CSA_FMT_FP8B32 3

#define CSA_OP_INDEXER_TOPK 1
#define CSA_OP_SPARSE_MQA 2
#define CSA_OP_HCA_DENSE 3

/* Text of the last error returned on the calling thread ("" if none). */
const char *csa_last_error(void);

/* Library version string. */
const char *csa_version(void);

/*
 * csa_rope_table (host): fill cos_out / sin_out (host, fp32 [P, R/2]) with
 * the nearest fp32 of cos / sin(p * base^(-2i/R)), evaluated in fp64.
 * [XM] key technical details (RoPE on the last 64 dims).
 * Errors: INVALID_ARG for P < 1, odd or non-positive R, NULL pointers.
 */
int csa_rope_table(int64_t P, int R, double base, float *cos_out, float *sin_out);

/*
 * csa_workspace_size: bytes of `ws` that `op` (CSA_OP_*) needs for B
 * sequences of Tq queries, N entries per sequence, top-k k (CSA), H heads of
 * dim D, the largest key count per query max_keys (attention: k + W for CSA,
 * entries + W for HCA) and Ts window-cache rows per sequence.  Never less
 * than 256 (the status block).  Returns -1 for an unknown op.  The attention
 * calls use the space for a bf16 copy of the cache rows when every row serves
 * many queries (prefill), and for few queries (decode) for the bf16 rows each
 * query's keys are gathered into when a query's keys span many tiles and for
 * the split-softmax partial states when a query's keys are split over more
 * CTAs than one thread-block cluster holds; with less workspace they fall
 * back to slower plans.
 */
int64_t csa_workspace_size(int op, int B, int64_t Tq, int64_t N, int k, int H, int D,
                           int64_t max_keys, int64_t Ts);

/* Clear the status block of ws (async on stream). */
int csa_status_reset(void *ws, void *stream);

/* Copy the status flags of ws to *flags (host) and wait for stream. */
int csa_status_read(const void *ws, void *stream, uint32_t *flags);

/*
 * csa_selftest_wait_timeout: exercise the expiry of the library's bounded
 * device waits (failure detection).  One CTA waits at most `polls` times on
 * an mbarrier phase that nothing completes, gives up and sets
 * CSA_FLAG_TIMEOUT in ws, as any kernel of the library does when one of its
 * waits expires; csa_status_read then reports CSA_ERR_TIMEOUT.  No fault and
 * no hang: the context stays usable.  Async on stream.
 * Errors: INVALID_ARG (NULL ws, polls outside [1, 2^20]); CUDA.
 */
int csa_selftest_wait_timeout(void *ws, uint32_t polls, void *stream);

/*
 * kvcache_pack_fp8_bf16: pack n post-RoPE rows of 512 fp32 channels
 * (v, device [n, 512]) into the mixed FP8/BF16 layout (out, device
 * [n, 592] bytes, CSA_FMT_MIXED592 above).  [XM] key technical details
 * (KV cache in mixed precision).  Used for the window ("state") cache and
 * standalone packing; csa_compress_kv packs its own output.
 * Errors: INVALID_ARG for n < 0 or NULL pointers with n > 0.
 */
int kvcache_pack_fp8_bf16(const float *v, int64_t n, uint8_t *out, void *stream);

/*
 * csa_compress_kv: block compression of KV (or of indexer keys) into
 * compressed entries, with RoPE and storage packing fused.
 * [XM] CSA: the KV entries of every m tokens are fused into one compressed
 * entry by a weighted sum; [HU] Tömörítés (m = 4); [XM]/[HU] HCA: m' = 128.
 *  x         (device) [B, T, C] activations, x_dtype CSA_DTYPE_BF16 or _F32
 *  z         (device) fp32 [B, T] compression logits, one per token
 *  s         (device) fp32 [C] per-channel scale, or NULL for all ones
 *  rope_cos/sin, rope_rows: RoPE tables (needed when R > 0)
 *  pos0      absolute position of x's first token; a multiple of m
 *  R         RoPE channels (the last R of C); 0 for indexer keys
 *  m         block size (1..128); N = floor(T / m) entries are written
 *  out_fmt   CSA_FMT_F32 (out fp32 [B, N, C]), CSA_FMT_MIXED592 (C = 512,
 *            R = 64; out [B, N, 592] bytes), CSA_FMT_MXFP4 (R = 0, C a
 *            multiple of 32, at most 64; out [B, N, C/2] codes and
 *            out_scales [B, N, C/32] bytes) or CSA_FMT_FP8B32 (R = 0, C =
 *            32 or 64; out [B, N, C] codes and out_scales [B, N, C/32])
 * Entry j (of this call) covers tokens [jm, jm + m); its weights are
 * a = softmax(z over the block), computed as mu = max z, e_i = sexp(z_i -
 * mu) (the library's fp32 exponential), S = e_0 + ... + e_{m-1} in order,
 * a_i = e_i / S; channel c is (sum_i fma order) a_i x_{i,c}, times s_c; the
 * last R channels then rotate at position pos0 + jm + m - 1, the block's
 * last token.  With m = 1 and s = NULL this stores the tokens themselves
 * (the sliding-window cache).
 * Errors: INVALID_ARG (NULL pointers, bad dtype/format, pos0 % m != 0,
 * RoPE rows not covering the last position); UNSUPPORTED (m > 128, format
 * and C/R combinations not listed).
 */
int csa_compress_kv(const void *x, int x_dtype, const float *z, const float *s,
                    const float *rope_cos, const float *rope_sin, int64_t rope_rows,
                    int64_t pos0, int B, int64_t T, int C, int R, int m, int out_fmt, void *out,
                    uint8_t *out_scales, void *stream);

/*
 * csa_compress_kv_channel_logits: csa_compress_kv with one logit per token
 * and channel -- the other plain reading of [XM] CSA's weighted sum of every
 * m tokens' KV entries (a learned weight per slot and channel).
 *  z         (device) fp32 [B, T, C] compression logits
 *  every other argument, the layout of out / out_scales and the errors as
 *  csa_compress_kv.
 * Channel c of entry j has its own weights a_{i,c} = softmax over the block
 * of z_{jm+i, c}, by the sequence above written per channel (mu_c = max,
 * e_i = sexp(z_{i,c} - mu_c), S_c in token order, a_i = e_i / S_c); then
 * (sum_i fma order) a_{i,c} x_{i,c}, times s_c, and the same RoPE and
 * packing.  Logits equal across channels give csa_compress_kv's bytes.
 */
int csa_compress_kv_channel_logits(const void *x, int x_dtype, const float *z, const float *s,
                                   const float *rope_cos, const float *rope_sin, int64_t rope_rows,
                                   int64_t pos0, int B, int64_t T, int C, int R, int m, int out_fmt,
                                   void *out, uint8_t *out_scales, void *stream);

/*
 * csa_decode_append: decode-time maintenance of one layer's caches -- one new
 * token per sequence.  [XM] CSA / HCA: every m tokens become one compressed
 * entry; [XM] "百万Token 长上下文真实表现" (state cache for the uncompressed
 * tail) and [HU] Sliding Window: the newest tokens stay uncompressed in a
 * window cache.  Per sequence b, with t = t_pos[b] (device) the new token's
 * position:
 *  - kv [b] (C = 512 bf16) and z [b] go to ring slot t mod m of kv_tail
 *    [B, m, C] bf16 / z_tail [B, m] fp32 (the raw tokens of the block being
 *    filled); likewise kI [b] (CI bf16) and zI [b] to kI_tail / zI_tail when
 *    kI is not NULL (indexer keys, CSA layers);
 *  - the token is packed into the window cache swa [B, Ts, 592] at row
 *    t - swa_pos0[b] exactly as csa_compress_kv with m = 1 and s = NULL
 *    stores it (RoPE at t).  When that row is Ts, the last W - 1 rows first
 *    move to rows 0 .. W - 2 and swa_pos0[b] (device, updated) becomes
 *    t - W + 1; so the window cache always holds tokens swa_pos0[b] .. t,
 *    the form csa_sparse_mqa / hca_dense_attn read.  Requires Ts >= 2 W;
 *  - when (t + 1) mod m == 0 the block [t - m + 1, t] is compressed from the
 *    ring into entry j = (t + 1) / m - 1 of cache [B, nmax, 592] (RoPE at t)
 *    and, when kI is given, of kI_codes [B, nmax, CI/2] / kI_scales
 *    [B, nmax, CI/32] (MXFP4, no RoPE), with the very operations of
 *    csa_compress_kv (s, sI: the channel scales, or NULL); entries j >= nmax
 *    are not stored.
 * Tokens of a sequence must be appended in order (t = previous t + 1; the
 * first one at t = swa_pos0[b], with the ring slots of its block filled by
 * earlier calls), so that after the call for token t the caches equal those
 * csa_compress_kv builds from tokens 0 .. t.  A sequence whose t has no RoPE
 * row (t < 0 or t >= rope_rows) is left unchanged; rows outside the window
 * buffer are never written.
 * Errors: INVALID_ARG (NULL pointers, m outside 1..128, Ts < 2 W, kv / kI /
 * kv_tail / kI_tail not 16-byte aligned); UNSUPPORTED (C != 512, R != 64, CI
 * not 32 or 64 with kI given).
 */
int csa_decode_append(const void *kv, const float *z, const void *kI, const float *zI, const float *s,
                      const float *sI, const float *rope_cos, const float *rope_sin, int64_t rope_rows,
                      const int64_t *t_pos,
                      int B, int C, int R, int CI, int m, void *kv_tail, float *z_tail, void *kI_tail,
                      float *zI_tail, uint8_t *cache, int64_t nmax, uint8_t *kI_codes, uint8_t *kI_scales,
                      uint8_t *swa, int64_t Ts, int W, int64_t *swa_pos0, void *stream);

/*
 * csa_indexer_topk: lightning-indexer scores of every visible compressed
 * entry for every query, and the top-k of them.
 * [XM] CSA: the lightning indexer picks the top-k compressed entries per
 * query token; [HU] Lightning Indexer (k = 1024); [XM] key technical details:
 * the indexer's attention runs in FP4.
 *  qI        (device) [B, Tq, HI, dI] indexer queries: CSA_DTYPE_BF16 with
 *            kI_fmt CSA_FMT_MXFP4 or CSA_FMT_FP8B32 (quantised to MXFP4
 *            per 32-block inside), or CSA_DTYPE_F32 with kI_fmt CSA_FMT_F32
 *  w         (device) fp32 [B, Tq, HI] head weights
 *  kI        (device) keys: MXFP4 codes [B, N, dI/2] with kI_scales
 *            [B, N, dI/32], FP8 codes [B, N, dI] with kI_scales [B, N,
 *            dI/32] (CSA_FMT_FP8B32: the FP4-query x FP8-key indexer), or
 *            fp32 [B, N, dI] (kI_scales NULL)
 *  q_pos     (device) int64 [B, Tq] absolute position t of each query
 *  N, m      entries per sequence and their block size
 *  k         entries to keep (1..4096)
 *  idx_out   (device) int32 [B, Tq, k]: entry indices, best first, -1 pad
 *  score_out (device) fp32 [B, Tq, k] or NULL: their scores (-inf pad)
 * score(t, j) = sum over heads h, ascending, of s = fma(w_h, relu(d_h), s)
 * from +0; d_h is the exact dot of the dequantised MXFP4 query with the
 * dequantised MXFP4 or FP8 key, rounded once to fp32, or the fma chain over
 * dI from +0 (fp32).  Candidates:
 * j < N with (j + 1) m - 1 <= t.  Order: score descending, then index
 * ascending.
 * Errors: INVALID_ARG (sizes, NULL pointers, ws smaller than the scores or
 * not 256-byte aligned); UNSUPPORTED (k outside 1..4096; FP4 or FP8 keys:
 * dI != 64 or HI > 32; fp32: dI > 64, HI > 32 or HI * dI > 512); CUDA.
 * Workspace: csa_workspace_size(CSA_OP_INDEXER_TOPK, ...) bytes give every
 * path (the tensor-core prefill scores, the two-stage top-k of few long
 * rows); the status block plus B * Tq * N fp32 scores is the least accepted,
 * and then prefill scores run on the CUDA cores and the top-k one CTA per
 * row.  Same indices and scores on every path.
 */
int csa_indexer_topk(const void *qI, int qI_dtype, const float *w, const void *kI,
                     const uint8_t *kI_scales, int kI_fmt, const int64_t *q_pos, int B,
                     int64_t Tq, int HI, int dI, int64_t N, int m, int k, int32_t *idx_out,
                     float *score_out, void *ws, size_t ws_bytes, void *stream);

/*
 * csa_sparse_mqa: multi-query attention of every query over its selected
 * compressed entries and its sliding window, in one softmax.
 * [XM] CSA: attention runs only over the selected entries, with a sliding
 * window branch for the nearest tokens; [HU] Sliding Window figyelem (128);
 * [ZC] both attentions carry the window branch; [XM] key technical details:
 * partial RoPE and inverse rotation of the output.
 *  q         (device) [B, Tq, H, D] queries before RoPE (q_dtype BF16 with
 *            cache_fmt MIXED592, D = 512, R = 64; or F32 with cache_fmt F32)
 *  q_pos     (device) int64 [B, Tq] absolute positions t
 *  cache     (device) [B, N, row] compressed entries (cache_fmt rows)
 *  idx       (device) int32 [B, Tq, k] selected entries (-1 = none)
 *  swa       (device) [B, Ts, row] window cache: token u of sequence b is
 *            row u - swa_pos0[b]; swa_pos0 (device) int64 [B]
 *  W         window: tokens t - W < u <= t, u >= 0
 *  softmax_scale  multiplies q.k
 *  out       (device) [B, Tq, H, D], same dtype as q
 *  lse       (device) fp32 [B, Tq, H] natural-log sum-exp, or NULL
 * All H heads share one KV; the value of a key is its entry (V = K).
 * Logits = scale * RoPE_t(q_h) . kappa over the union of the selected
 * entries and the window (an entry that also lies in the window is not
 * removed), one softmax, o_h = sum p kappa, then the last R channels of o_h
 * rotate by -t.  No keys: o = 0, lse = -inf.
 * Errors: INVALID_ARG, UNSUPPORTED (shapes other than listed, k + W >
 * 8192), CUDA; device check flag for indices >= N, not yet visible, or
 * window rows outside swa.
 */
int csa_sparse_mqa(const void *q, int q_dtype, const int64_t *q_pos, int B, int64_t Tq, int H,
                   int D, int R, int cache_fmt, const void *cache, int64_t N, int m,
                   const int32_t *idx, int k, const void *swa, const int64_t *swa_pos0,
                   int64_t Ts, int W, float softmax_scale, const float *rope_cos,
                   const float *rope_sin, int64_t rope_rows, void *out, float *lse, void *ws,
                   size_t ws_bytes, void *stream);

/*
 * hca_dense_attn: as csa_sparse_mqa, with every visible entry
 * (j < min(N, floor((t + 1) / m))) in place of the selected ones.
 * [XM] HCA: a larger compression ratio m' and dense attention over all
 * compressed entries, no selection; [HU] Heavily Compressed Attention
 * (m' = 128).
 * Errors: as csa_sparse_mqa (UNSUPPORTED when visible entries + W > 16384).
 */
int hca_dense_attn(const void *q, int q_dtype, const int64_t *q_pos, int B, int64_t Tq, int H,
                   int D, int R, int cache_fmt, const void *cache, int64_t N, int m,
                   const void *swa, const int64_t *swa_pos0, int64_t Ts, int W,
                   float softmax_scale, const float *rope_cos, const float *rope_sin,
                   int64_t rope_rows, void *out, float *lse, void *ws, size_t ws_bytes,
                   void *stream);

/*
 * csa_indexer_topk_noalloc: csa_indexer_topk without a caller workspace.
 * The method has no counterpart to this call; it exists for callers that
 * cannot allocate device memory.  Serving runtimes that plan every device
 * buffer before they start and refuse allocation afterwards, and plugins
 * that such a runtime hands the tensors of one call but no allocator,
 * cannot provide the score scratch that csa_indexer_topk needs; this call
 * keeps that scratch in a fixed device array owned by the library.
 * Arguments, results and errors are those of csa_indexer_topk, without
 * ws / ws_bytes.  Rules:
 *  - the array holds 16 MiB (B * Tq * N <= 4194304 scores); larger calls
 *    return CSA_ERR_UNSUPPORTED before anything is enqueued;
 *  - every GPU that loads the library holds the array until exit;
 *  - all calls share the array and it keeps the last call's contents:
 *    calls that overlap on the GPU race, so order them on one stream;
 *  - the first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture;
 *  - the scores come from the library's integer (CUDA-core) kernels, which
 *    have no device-side waits, so no wait can expire and CSA_OK covers the
 *    whole call (no status block is needed); results are bit-identical to
 *    csa_indexer_topk's.
 * It calls no cudaMalloc / cudaFree and no allocating library routine.
 */
int csa_indexer_topk_noalloc(const void *qI, int qI_dtype, const float *w, const void *kI,
                             const uint8_t *kI_scales, int kI_fmt, const int64_t *q_pos, int B,
                             int64_t Tq, int HI, int dI, int64_t N, int m, int k,
                             int32_t *idx_out, float *score_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA_B300_H */
