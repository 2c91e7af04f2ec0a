// launch.h -- internal launchers of libcsa_b300 (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace csa {

// A nonzero int per device, computed by f() the first time it is asked for
// with that device current, then read.  Thread-safe: threads that race on the
// first use each compute it (f must give the same value every time); a zero
// from f (a failed query) is not stored, so the next call tries again.
constexpr int kMaxDevices = 64;
class PerDevice {
 public:
  template <class F>
  int get(F f) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return f();
    int v = v_[d].load(std::memory_order_acquire);
    if (v == 0) {
      v = f();
      if (v != 0) v_[d].store(v, std::memory_order_release);
    }
    return v;
  }

 private:
  std::atomic<int> v_[kMaxDevices]{};
};

// Launches `kernel` on `st` with programmatic stream serialisation allowed:
// the kernel may be scheduled while the previous kernel on the stream is
// still running; it waits for it (pdl_begin) before touching memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device and call site (`once`).
inline void smem_limit_once(PerDevice& once, const void* kernel, int bytes) {
  once.get([&] {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess ? 1 : 0;
  });
}

// Streaming multiprocessors of the current device.
inline int device_sms() {
  static PerDevice sms;
  return sms.get([] {
    int d = 0, n = 0;
    cudaGetDevice(&d);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    return n;
  });
}

struct AttnArgs {
  const void* q;
  bool q_bf16;
  const int64_t* q_pos;
  int B;
  int64_t Tq;
  int H, D, R;
  int cache_fmt;
  const void* cache;
  int64_t N;
  int m;
  const int32_t* idx;   // NULL: dense (every visible entry)
  int k;
  const void* swa;
  const int64_t* swa_pos0;
  int64_t Ts;
  int W;
  float scale;
  const float* rcos;
  const float* rsin;
  int64_t rope_rows;
  void* out;
  float* lse;
  void* ws;             // status block at ws; scratch after kWsHeader
  size_t ws_bytes;
  int max_keys;         // upper bound of keys per query (list length)
};

constexpr size_t kWsHeader = 256;

cudaError_t launch_compress(const void* x, bool x_bf16, const float* z, bool z_per_channel, const float* s,
                            const float* rcos, const float* rsin, int64_t pos0, int B, int64_t T,
                            int C, int R, int m, int fmt, void* out, uint8_t* out_scales,
                            cudaStream_t st);
cudaError_t launch_pack_mixed(const float* v, int64_t n, uint8_t* out, cudaStream_t st);
cudaError_t launch_decode_append(const void* kv, const float* z, const void* kI, const float* zI, const float* s,
                                 const float* sI, const float* rcos, const float* rsin, int64_t rope_rows,
                                 const int64_t* t_pos, int B,
                                 int C, int R, int CI, int m, void* kv_tail, float* z_tail, void* kI_tail,
                                 float* zI_tail, uint8_t* cache, int64_t nmax, uint8_t* kI_codes,
                                 uint8_t* kI_scales, uint8_t* swa, int64_t Ts, int W, int64_t* swa_pos0,
                                 cudaStream_t st);
// key_fmt: CSA_FMT_MXFP4 or CSA_FMT_FP8B32 (bf16 queries, quantised to MXFP4
// inside) or CSA_FMT_F32 (fp32 queries)
cudaError_t launch_indexer_topk(const void* qI, int key_fmt, const float* w, const void* kI,
                                const uint8_t* kI_scales, const int64_t* q_pos, int B, int64_t Tq,
                                int HI, int dI, int64_t N, int m, int k, int32_t* idx_out,
                                float* score_out, float* scores_ws, void* tc_ws, void* cand_ws, void* flags_ws,
                                bool tensor_cores, cudaStream_t st);
// CTAs of `kernel` that fit on one SM at once: the tightest of its register,
// shared-memory (228 KiB per SM, 1 KiB reserved per CTA), thread (2048) and
// block (32) limits, from the compiled kernel's attributes
inline int resident_ctas(const void* kernel, int threads, size_t dyn_smem) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return 1;
  const int warps = (threads + 31) / 32;
  const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;   // allocated per warp in units of 256
  const int by_regs = regs_warp > 0 ? 65536 / (regs_warp * warps) : 32;
  const int by_smem = (int)((size_t)233472 / (fa.sharedSizeBytes + dyn_smem + 1024));
  const int by_threads = 2048 / (warps * 32);
  int n = by_regs < by_smem ? by_regs : by_smem;
  n = n < by_threads ? n : by_threads;
  n = n < 32 ? n : 32;
  return n < 1 ? 1 : n;
}

// a bounded device wait that expires on purpose (failure-detection self-test)
cudaError_t launch_wait_selftest(void* ws, uint32_t polls, cudaStream_t st);

// decode scoring on the tensor cores (few query rows, long entry lists)
bool decode_tc_applies(int64_t Tq, int HI, int dI, int64_t N);
cudaError_t launch_scores_fp4_decode_tc(const void* qI, const float* w, const uint8_t* kc, const uint8_t* ks,
                                        const int64_t* q_pos, int B, int64_t Tq, int HI, int64_t N, int m,
                                        float* scores, unsigned int* hist, void* flags_ws, cudaStream_t st);
// two-stage top-k for long rows when there are few of them, and its scratch
bool topk_two_stage(int B, int64_t Tq, int64_t N);
size_t topk_cand_bytes(int B, int64_t Tq, int64_t N, int k);
// FP8 tensor-core scoring (indexer_tc.cu): whether it applies, its extra
// scratch, and the launch (scores only; top-k follows in indexer.cu)
bool indexer_tc_applies(int B, int64_t Tq, int HI, int dI, int64_t N);
size_t indexer_tc_workspace(int B, int64_t Tq, int HI, int64_t N);
cudaError_t launch_indexer_scores_tc(const void* qI, const float* w, const uint8_t* kc, const uint8_t* ks,
                                     const int64_t* q_pos, int B, int64_t Tq, int HI, int64_t N, int m,
                                     float* scores, void* tc_ws, void* flags_ws, cudaStream_t st);
cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t st);
// decode attention (attn_decode.cu): few rows, every step in one launch
bool attn_decode_applies(int H, int D, int R, int64_t rows, int k, bool sparse);
size_t attn_decode_workspace(int64_t rows, int64_t max_keys);
cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t st);
size_t attn_tc_workspace(int B, int64_t Tq, int H, int D, int64_t max_keys, int64_t N, int64_t Ts, int k);

}  // namespace csa
