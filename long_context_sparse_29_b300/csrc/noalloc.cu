// noalloc.cu -- csa_indexer_topk_noalloc: the lightning-indexer top-k call
// for callers that cannot allocate device memory.
//
// Some hosts own every byte of device memory themselves: serving runtimes
// that plan all device buffers before they start answering requests and
// refuse any allocation afterwards, and plugins loaded into such a runtime
// that are handed the tensors of one call but no allocator.  They cannot
// provide the scratch workspace that csa_indexer_topk takes.  This entry
// point keeps that scratch (the per-query score rows) in a fixed array in
// device memory that belongs to the library, so the caller passes only
// inputs and outputs.
//
// Costs and rules of that choice:
//  * every GPU that loads libcsa_b300.so holds the array (kScratchBytes)
//    until the process exits;
//  * the array holds B * Tq * N fp32 scores at most; larger calls are
//    rejected with CSA_ERR_UNSUPPORTED before anything is enqueued;
//  * all calls share the one array and it keeps the last call's contents:
//    calls that overlap on the GPU (other streams, other host threads)
//    race on it, so the caller must order them;
//  * nothing in it has to start at zero: each call writes every score it
//    later reads;
//  * the scores are computed by the library's integer (CUDA-core) kernels,
//    which have no device-side waits: nothing in this call can expire, so
//    CSA_OK from it covers the whole call (the workspace call's tensor-core
//    scorers wait on mbarriers and report an expired wait in the caller's
//    workspace, which this call does not have).  The indices and scores are
//    bit-identical to csa_indexer_topk's on every path;
//  * the first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (the device must be current); make that first
//    call before any stream capture.
#include <mutex>

#include "csa_common.cuh"
#include "launch.h"

namespace csa {
int report_error(int code, const char* msg);
}

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB: 4,194,304 fp32 scores
constexpr int kMaxDevices = 64;

// In host code this name is only a host-side stand-in for the array; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_indexer_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_indexer_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return csa::report_error(CSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return csa::report_error(CSA_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_indexer_scratch);
    if (e != cudaSuccess || !p) {
      return csa::report_error(CSA_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                              : "cudaGetSymbolAddress returned NULL");
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CSA_OK;
}

}  // namespace

extern "C" int csa_indexer_topk_noalloc(const void* qI, int qI_dtype, const float* w,
                                        const void* kI, const uint8_t* kI_scales, int kI_fmt,
                                        const int64_t* q_pos, int B, int64_t Tq, int HI, int dI,
                                        int64_t N, int m, int k, int32_t* idx_out,
                                        float* score_out, void* stream) {
  if (B < 0 || Tq < 0 || N < 0 || m < 1 || HI < 1 || dI < 1)
    return csa::report_error(CSA_ERR_INVALID_ARG, "csa_indexer_topk_noalloc: bad sizes");
  if (k < 1 || k > 4096)
    return csa::report_error(CSA_ERR_UNSUPPORTED, "csa_indexer_topk_noalloc: k must be in [1, 4096]");
  const bool fp4 = qI_dtype == CSA_DTYPE_BF16 && kI_fmt == CSA_FMT_MXFP4;
  const bool fp8k = qI_dtype == CSA_DTYPE_BF16 && kI_fmt == CSA_FMT_FP8B32;
  const bool f32 = qI_dtype == CSA_DTYPE_F32 && kI_fmt == CSA_FMT_F32;
  if (!fp4 && !fp8k && !f32)
    return csa::report_error(CSA_ERR_UNSUPPORTED, "csa_indexer_topk_noalloc: dtype/format pair not supported");
  if ((fp4 || fp8k) && (dI != 64 || HI > 32))
    return csa::report_error(CSA_ERR_UNSUPPORTED, "csa_indexer_topk_noalloc: FP4 / FP8 keys need dI=64, HI<=32");
  if (f32 && (dI > 64 || HI > 32 || HI * dI > 512))
    return csa::report_error(CSA_ERR_UNSUPPORTED,
                             "csa_indexer_topk_noalloc: fp32 path needs dI<=64, HI<=32, HI*dI<=512");
  const double need = 4.0 * (double)B * (double)Tq * (double)N;
  if (need > (double)kScratchBytes)
    return csa::report_error(CSA_ERR_UNSUPPORTED,
                             "csa_indexer_topk_noalloc: B*Tq*N scores exceed the built-in 16 MiB scratch "
                             "(4194304 scores); use csa_indexer_topk with a workspace");
  if ((int64_t)B * Tq == 0) return CSA_OK;
  if (!qI || !w || !q_pos || !idx_out || (N > 0 && !kI) || ((fp4 || fp8k) && N > 0 && !kI_scales))
    return csa::report_error(CSA_ERR_INVALID_ARG, "csa_indexer_topk_noalloc: NULL pointer");
  void* scratch = nullptr;
  const int r = scratch_address(&scratch);
  if (r != CSA_OK) return r;
  const cudaError_t e = csa::launch_indexer_topk(qI, kI_fmt, w, kI, kI_scales, q_pos, B, Tq, HI, dI, N, m,
                                                 k, idx_out, score_out, reinterpret_cast<float*>(scratch),
                                                 nullptr, nullptr, nullptr, /*tensor_cores=*/false,
                                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return csa::report_error(CSA_ERR_CUDA, cudaGetErrorString(e));
  return CSA_OK;
}
