// abi.cu -- the extern "C" entry points of libcsa_b300 (declared in
// include/csa_b300.h): argument validation, workspace accounting and
// dispatch to the kernels.  Nothing here allocates device memory or
// synchronises, except csa_status_read, which waits for its stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "csa_common.cuh"
#include "launch.h"

namespace {

thread_local char g_err[512];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = 0;
  return CSA_OK;
}

int cuda_result(cudaError_t e, const char* where) {
  if (e != cudaSuccess) return fail(CSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
  return ok();
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// the scores; required
size_t indexer_ws(int B, int64_t Tq, int64_t N) {
  return csa::kWsHeader + align256(sizeof(float) * (size_t)B * (size_t)Tq * (size_t)N);
}
// + the chunk winners of the two-stage top-k (few long rows) and the quantised
// queries and expanded entries of the tensor-core scoring, where they apply
size_t indexer_cand_ws(int B, int64_t Tq, int64_t N, int k) {
  return csa::topk_two_stage(B, Tq, N) ? align256(csa::topk_cand_bytes(B, Tq, N, k)) : 0;
}
size_t indexer_ws_full(int B, int64_t Tq, int64_t N, int HI, int dI, int k) {
  const size_t base = indexer_ws(B, Tq, N) + indexer_cand_ws(B, Tq, N, k);
  return csa::indexer_tc_applies(B, Tq, HI, dI, N) ? base + align256(csa::indexer_tc_workspace(B, Tq, HI, N)) : base;
}

bool indexer_use_dp4a() {
  const char* e = getenv("CSA_INDEXER_IMPL");
  return e && strcmp(e, "dp4a") == 0;
}

bool attn_use_simt() {
  const char* e = getenv("CSA_ATTN_IMPL");
  return e && strcmp(e, "simt") == 0;
}

// shared validation of the two attention calls; fills a
int attn_prepare(csa::AttnArgs& a, const void* q, int q_dtype, const int64_t* q_pos, int B,
                 int64_t Tq, int H, int D, int R, int cache_fmt, const void* cache, int64_t N,
                 int m, const int32_t* idx, int k, const void* swa, const int64_t* swa_pos0,
                 int64_t Ts, int W, float scale, const float* rc, const float* rs,
                 int64_t rope_rows, void* out, float* lse, void* ws, size_t ws_bytes,
                 const char* name) {
  if (B < 0 || Tq < 0 || H < 1 || N < 0 || m < 1 || k < 0 || W < 0 || Ts < 0)
    return fail(CSA_ERR_INVALID_ARG, "%s: negative or zero size argument", name);
  if ((int64_t)B * Tq > 0 && (!q || !q_pos || !out || !rc || !rs))
    return fail(CSA_ERR_INVALID_ARG, "%s: NULL q, q_pos, out or RoPE table", name);
  if (N > 0 && !cache) return fail(CSA_ERR_INVALID_ARG, "%s: NULL cache", name);
  if (W > 0 && (!swa || !swa_pos0)) return fail(CSA_ERR_INVALID_ARG, "%s: NULL window cache", name);
  if (idx == nullptr && k > 0 && strcmp(name, "csa_sparse_mqa") == 0)
    return fail(CSA_ERR_INVALID_ARG, "%s: NULL idx", name);
  if (!ws || ws_bytes < csa::kWsHeader) return fail(CSA_ERR_INVALID_ARG, "%s: workspace missing", name);
  if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(CSA_ERR_INVALID_ARG, "%s: ws not 256-byte aligned", name);
  if (rope_rows < 1) return fail(CSA_ERR_INVALID_ARG, "%s: empty RoPE table", name);
  if (q_dtype == CSA_DTYPE_BF16) {
    if (cache_fmt != CSA_FMT_MIXED592 || D != 512 || R != 64)
      return fail(CSA_ERR_UNSUPPORTED, "%s: bf16 queries need the mixed 592-byte cache, D=512, R=64", name);
  } else if (q_dtype == CSA_DTYPE_F32) {
    if (cache_fmt != CSA_FMT_F32 || D < 2 || D > 512 || (D & 1) || R < 0 || R > D || (R & 1))
      return fail(CSA_ERR_UNSUPPORTED, "%s: fp32 queries need the fp32 cache, even D <= 512, even R <= D", name);
  } else {
    return fail(CSA_ERR_INVALID_ARG, "%s: unknown q dtype %d", name, q_dtype);
  }
  const int64_t max_keys = (idx ? (int64_t)k : N) + W;
  if (max_keys > 16384) return fail(CSA_ERR_UNSUPPORTED, "%s: more than 16384 keys per query", name);
  a.q = q;
  a.q_bf16 = q_dtype == CSA_DTYPE_BF16;
  a.q_pos = q_pos;
  a.B = B;
  a.Tq = Tq;
  a.H = H;
  a.D = D;
  a.R = R;
  a.cache_fmt = cache_fmt;
  a.cache = cache;
  a.N = N;
  a.m = m;
  a.idx = idx;
  a.k = idx ? k : 0;
  a.swa = swa;
  a.swa_pos0 = swa_pos0;
  a.Ts = Ts;
  a.W = W;
  a.scale = scale;
  a.rcos = rc;
  a.rsin = rs;
  a.rope_rows = rope_rows;
  a.out = out;
  a.lse = lse;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.max_keys = (int)max_keys;
  const size_t need = csa::kWsHeader;   // more is used when given (see csa_workspace_size)
  if (ws_bytes < need)
    return fail(CSA_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name, ws_bytes, need);
  return CSA_OK;
}

int attn_run(const csa::AttnArgs& a, void* stream, const char* name) {
  if ((int64_t)a.B * a.Tq == 0) return ok();
  const bool tc = a.cache_fmt == CSA_FMT_MIXED592 && a.q_bf16 && !attn_use_simt();
  const cudaError_t e = tc ? csa::launch_attn_tc(a, as_stream(stream))
                           : csa::launch_attn_simt(a, as_stream(stream));
  return cuda_result(e, name);
}

}  // namespace

extern "C" {

const char* csa_last_error(void) { return g_err; }

const char* csa_version(void) { return "csa_b300 1.0 sm_103a"; }

int csa_rope_table(int64_t P, int R, double base, float* cos_out, float* sin_out) {
  if (P < 1 || R < 2 || (R & 1) || !cos_out || !sin_out || !(base > 0.0))
    return fail(CSA_ERR_INVALID_ARG, "csa_rope_table: bad arguments");
  const int half = R / 2;
  for (int64_t p = 0; p < P; ++p) {
    for (int i = 0; i < half; ++i) {
      const double theta = pow(base, -2.0 * i / R);
      const double a = (double)p * theta;
      cos_out[p * half + i] = (float)cos(a);
      sin_out[p * half + i] = (float)sin(a);
    }
  }
  return ok();
}

int64_t csa_workspace_size(int op, int B, int64_t Tq, int64_t N, int k, int H, int D,
                           int64_t max_keys, int64_t Ts) {
  if (B < 0 || Tq < 0 || N < 0) return -1;
  switch (op) {
    case CSA_OP_INDEXER_TOPK:   // H, D: indexer heads and head dim (0: the minimum)
      return (int64_t)indexer_ws_full(B, Tq, N, H, D, k);
    case CSA_OP_SPARSE_MQA:
    case CSA_OP_HCA_DENSE:
      return (int64_t)(csa::kWsHeader +
                       align256(csa::attn_tc_workspace(B, Tq, H, D, max_keys, N, Ts, op == CSA_OP_SPARSE_MQA ? k : 0)));
    default:
      return -1;
  }
}

int csa_status_reset(void* ws, void* stream) {
  if (!ws) return fail(CSA_ERR_INVALID_ARG, "csa_status_reset: NULL ws");
  return cuda_result(cudaMemsetAsync(ws, 0, sizeof(csa::Status), as_stream(stream)), "csa_status_reset");
}

int csa_selftest_wait_timeout(void* ws, uint32_t polls, void* stream) {
  const char* nm = "csa_selftest_wait_timeout";
  if (!ws) return fail(CSA_ERR_INVALID_ARG, "%s: NULL ws", nm);
  if (polls < 1 || polls > (1u << 20)) return fail(CSA_ERR_INVALID_ARG, "%s: polls must be in [1, 2^20]", nm);
  return cuda_result(csa::launch_wait_selftest(ws, polls, as_stream(stream)), nm);
}

int csa_status_read(const void* ws, void* stream, uint32_t* flags) {
  if (!ws || !flags) return fail(CSA_ERR_INVALID_ARG, "csa_status_read: NULL argument");
  csa::Status st;
  cudaError_t e = cudaMemcpyAsync(&st, ws, sizeof st, cudaMemcpyDeviceToHost, as_stream(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_result(e, "csa_status_read");
  *flags = st.flags;
  if (st.flags & CSA_FLAG_TIMEOUT) return fail(CSA_ERR_TIMEOUT, "a bounded device wait expired");
  if (st.flags & CSA_FLAG_DEVICE_CHECK)
    return fail(CSA_ERR_DEVICE_CHECK, "device check: skipped an invalid key (first code 0x%08x)", st.first_bad);
  return ok();
}

int kvcache_pack_fp8_bf16(const float* v, int64_t n, uint8_t* out, void* stream) {
  if (n < 0) return fail(CSA_ERR_INVALID_ARG, "kvcache_pack_fp8_bf16: n < 0");
  if (n > 0 && (!v || !out)) return fail(CSA_ERR_INVALID_ARG, "kvcache_pack_fp8_bf16: NULL pointer");
  return cuda_result(csa::launch_pack_mixed(v, n, out, as_stream(stream)), "kvcache_pack_fp8_bf16");
}

static int compress_call(const char* nm, bool z_per_channel, const void* x, int x_dtype, const float* z,
                         const float* s, const float* rope_cos, const float* rope_sin, int64_t rope_rows,
                         int64_t pos0, int B, int64_t T, int C, int R, int m, int out_fmt, void* out,
                         uint8_t* out_scales, void* stream) {
  if (B < 0 || T < 0 || C < 2 || (C & 1) || m < 1 || pos0 < 0 || R < 0 || (R & 1) || R > C)
    return fail(CSA_ERR_INVALID_ARG, "%s: bad sizes (B=%d T=%lld C=%d R=%d m=%d pos0=%lld)", nm, B,
                (long long)T, C, R, m, (long long)pos0);
  if (x_dtype != CSA_DTYPE_F32 && x_dtype != CSA_DTYPE_BF16)
    return fail(CSA_ERR_INVALID_ARG, "%s: unknown x dtype %d", nm, x_dtype);
  if (pos0 % m) return fail(CSA_ERR_INVALID_ARG, "%s: pos0 %% m != 0", nm);
  if (m > 128) return fail(CSA_ERR_UNSUPPORTED, "%s: m > 128", nm);
  if (C > 512) return fail(CSA_ERR_UNSUPPORTED, "%s: C > 512", nm);
  const int64_t N = T / m;
  if ((int64_t)B * N == 0) return ok();
  if (!x || !z || !out) return fail(CSA_ERR_INVALID_ARG, "%s: NULL x, z or out", nm);
  if (R > 0) {
    if (!rope_cos || !rope_sin) return fail(CSA_ERR_INVALID_ARG, "%s: NULL RoPE table", nm);
    if (pos0 + N * m - 1 >= rope_rows)
      return fail(CSA_ERR_INVALID_ARG, "%s: RoPE table has %lld rows, position %lld needed", nm,
                  (long long)rope_rows, (long long)(pos0 + N * m - 1));
  }
  if (out_fmt == CSA_FMT_MIXED592) {
    if (C != 512 || R != 64) return fail(CSA_ERR_UNSUPPORTED, "%s: mixed rows need C=512, R=64", nm);
  } else if (out_fmt == CSA_FMT_MXFP4 || out_fmt == CSA_FMT_FP8B32) {
    if (R != 0 || (C != 32 && C != 64))
      return fail(CSA_ERR_UNSUPPORTED, "%s: MXFP4 / FP8 keys need R=0 and C in {32, 64}", nm);
    if (!out_scales) return fail(CSA_ERR_INVALID_ARG, "%s: NULL out_scales", nm);
  } else if (out_fmt != CSA_FMT_F32) {
    return fail(CSA_ERR_INVALID_ARG, "%s: unknown output format %d", nm, out_fmt);
  }
  return cuda_result(csa::launch_compress(x, x_dtype == CSA_DTYPE_BF16, z, z_per_channel, s, rope_cos, rope_sin,
                                          pos0, B, T, C, R, m, out_fmt, out, out_scales,
                                          as_stream(stream)),
                     nm);
}

int csa_compress_kv(const void* x, int x_dtype, const float* z, const float* s,
                    const float* rope_cos, const float* rope_sin, int64_t rope_rows, int64_t pos0,
                    int B, int64_t T, int C, int R, int m, int out_fmt, void* out,
                    uint8_t* out_scales, void* stream) {
  return compress_call("csa_compress_kv", false, x, x_dtype, z, s, rope_cos, rope_sin, rope_rows, pos0, B, T, C, R,
                       m, out_fmt, out, out_scales, stream);
}

int csa_compress_kv_channel_logits(const void* x, int x_dtype, const float* z, const float* s,
                                   const float* rope_cos, const float* rope_sin, int64_t rope_rows, int64_t pos0,
                                   int B, int64_t T, int C, int R, int m, int out_fmt, void* out,
                                   uint8_t* out_scales, void* stream) {
  return compress_call("csa_compress_kv_channel_logits", true, x, x_dtype, z, s, rope_cos, rope_sin, rope_rows,
                       pos0, B, T, C, R, m, out_fmt, out, out_scales, stream);
}

int csa_decode_append(const void* kv, const float* z, const void* kI, const float* zI, const float* s,
                      const float* sI, const float* rope_cos, const float* rope_sin, int64_t rope_rows,
                      const int64_t* t_pos,
                      int B, int C, int R, int CI, int m, void* kv_tail, float* z_tail, void* kI_tail,
                      float* zI_tail, uint8_t* cache, int64_t nmax, uint8_t* kI_codes, uint8_t* kI_scales,
                      uint8_t* swa, int64_t Ts, int W, int64_t* swa_pos0, void* stream) {
  const char* nm = "csa_decode_append";
  if (B < 0 || m < 1 || m > 128 || nmax < 0 || W < 0 || Ts < 0)
    return fail(CSA_ERR_INVALID_ARG, "%s: bad sizes", nm);
  if (C != 512 || R != 64) return fail(CSA_ERR_UNSUPPORTED, "%s: needs C = 512 and R = 64", nm);
  if (kI && CI != 32 && CI != 64) return fail(CSA_ERR_UNSUPPORTED, "%s: CI must be 32 or 64", nm);
  if (W > 0 && Ts < 2 * (int64_t)W) return fail(CSA_ERR_INVALID_ARG, "%s: Ts must be >= 2 W", nm);
  if (B == 0) return ok();
  if (!kv || !z || !t_pos || !kv_tail || !z_tail || !rope_cos || !rope_sin || (nmax > 0 && !cache) ||
      (W > 0 && (!swa || !swa_pos0)) || (kI && (!zI || !kI_tail || !zI_tail || (nmax > 0 && (!kI_codes || !kI_scales)))))
    return fail(CSA_ERR_INVALID_ARG, "%s: NULL pointer", nm);
  if (((reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(kv_tail) | reinterpret_cast<uintptr_t>(kI) |
        reinterpret_cast<uintptr_t>(kI_tail)) & 15))
    return fail(CSA_ERR_INVALID_ARG, "%s: kv, kI and their rings must be 16-byte aligned", nm);
  return cuda_result(csa::launch_decode_append(kv, z, kI, zI, s, sI, rope_cos, rope_sin, rope_rows, t_pos, B, C, R,
                                               kI ? CI : 0, m,
                                               kv_tail, z_tail, kI_tail, zI_tail, cache, nmax, kI_codes, kI_scales,
                                               swa, Ts, W, swa_pos0, as_stream(stream)),
                     nm);
}

int csa_indexer_topk(const void* qI, int qI_dtype, const float* w, const void* kI,
                     const uint8_t* kI_scales, int kI_fmt, const int64_t* q_pos, int B, int64_t Tq,
                     int HI, int dI, int64_t N, int m, int k, int32_t* idx_out, float* score_out,
                     void* ws, size_t ws_bytes, void* stream) {
  const char* nm = "csa_indexer_topk";
  if (B < 0 || Tq < 0 || N < 0 || m < 1 || HI < 1 || dI < 1)
    return fail(CSA_ERR_INVALID_ARG, "%s: bad sizes", nm);
  if (k < 1 || k > 4096) return fail(CSA_ERR_UNSUPPORTED, "%s: k must be in [1, 4096]", nm);
  const bool fp4 = qI_dtype == CSA_DTYPE_BF16 && kI_fmt == CSA_FMT_MXFP4;
  const bool fp8k = qI_dtype == CSA_DTYPE_BF16 && kI_fmt == CSA_FMT_FP8B32;
  const bool f32 = qI_dtype == CSA_DTYPE_F32 && kI_fmt == CSA_FMT_F32;
  if (!fp4 && !fp8k && !f32) return fail(CSA_ERR_UNSUPPORTED, "%s: dtype/format pair not supported", nm);
  if ((fp4 || fp8k) && (dI != 64 || HI > 32))
    return fail(CSA_ERR_UNSUPPORTED, "%s: FP4 / FP8 keys need dI=64, HI<=32", nm);
  if (f32 && (dI > 64 || HI > 32 || HI * dI > 512))
    return fail(CSA_ERR_UNSUPPORTED, "%s: fp32 path needs dI<=64, HI<=32, HI*dI<=512", nm);
  if ((int64_t)B * Tq == 0) return ok();
  if (!qI || !w || !q_pos || !idx_out || (N > 0 && !kI) || ((fp4 || fp8k) && N > 0 && !kI_scales))
    return fail(CSA_ERR_INVALID_ARG, "%s: NULL pointer", nm);
  if (!ws || ws_bytes < indexer_ws(B, Tq, N))
    return fail(CSA_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", nm, ws_bytes,
                indexer_ws(B, Tq, N));
  if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(CSA_ERR_INVALID_ARG, "%s: ws not 256-byte aligned", nm);
  float* scores = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + csa::kWsHeader);
  // the optional parts when the whole plan fits: [scores | chunk winners | tensor-core scratch]
  void* cand_ws = nullptr;
  void* tc_ws = nullptr;
  const size_t full = indexer_ws_full(B, Tq, N, HI, dI, k);
  if (ws_bytes >= full) {
    char* p = reinterpret_cast<char*>(ws) + indexer_ws(B, Tq, N);
    if (indexer_cand_ws(B, Tq, N, k)) cand_ws = p;
    p += indexer_cand_ws(B, Tq, N, k);
    if (fp4 && !indexer_use_dp4a() && csa::indexer_tc_applies(B, Tq, HI, dI, N)) tc_ws = p;
  }
  return cuda_result(csa::launch_indexer_topk(qI, kI_fmt, w, kI, kI_scales, q_pos, B, Tq, HI, dI, N,
                                              m, k, idx_out, score_out, scores, tc_ws, cand_ws, ws,
                                              !indexer_use_dp4a(), as_stream(stream)),
                     nm);
}

int csa_sparse_mqa(const void* q, int q_dtype, const int64_t* q_pos, int B, int64_t Tq, int H,
                   int D, int R, int cache_fmt, const void* cache, int64_t N, int m,
                   const int32_t* idx, int k, const void* swa, const int64_t* swa_pos0, int64_t Ts,
                   int W, float softmax_scale, const float* rope_cos, const float* rope_sin,
                   int64_t rope_rows, void* out, float* lse, void* ws, size_t ws_bytes,
                   void* stream) {
  csa::AttnArgs a;
  const int r = attn_prepare(a, q, q_dtype, q_pos, B, Tq, H, D, R, cache_fmt, cache, N, m, idx, k,
                             swa, swa_pos0, Ts, W, softmax_scale, rope_cos, rope_sin, rope_rows,
                             out, lse, ws, ws_bytes, "csa_sparse_mqa");
  if (r != CSA_OK) return r;
  if (!idx && k > 0) return fail(CSA_ERR_INVALID_ARG, "csa_sparse_mqa: NULL idx");
  return attn_run(a, stream, "csa_sparse_mqa");
}

int hca_dense_attn(const void* q, int q_dtype, const int64_t* q_pos, int B, int64_t Tq, int H,
                   int D, int R, int cache_fmt, const void* cache, int64_t N, int m,
                   const void* swa, const int64_t* swa_pos0, int64_t Ts, int W,
                   float softmax_scale, const float* rope_cos, const float* rope_sin,
                   int64_t rope_rows, void* out, float* lse, void* ws, size_t ws_bytes,
                   void* stream) {
  csa::AttnArgs a;
  const int r = attn_prepare(a, q, q_dtype, q_pos, B, Tq, H, D, R, cache_fmt, cache, N, m, nullptr,
                             0, swa, swa_pos0, Ts, W, softmax_scale, rope_cos, rope_sin, rope_rows,
                             out, lse, ws, ws_bytes, "hca_dense_attn");
  if (r != CSA_OK) return r;
  return attn_run(a, stream, "hca_dense_attn");
}

}  // extern "C"

namespace csa {

// Records an error for csa_last_error() from other translation units.
int report_error(int code, const char* msg) { return fail(code, "%s", msg); }

}  // namespace csa
