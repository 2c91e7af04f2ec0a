// attn_tc.cu -- placeholder while the tensor-core kernel is written.
#include "csa_common.cuh"
#include "launch.h"

namespace csa {

size_t attn_tc_workspace(int, int64_t, int, int, int64_t) { return 0; }

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t st) { return launch_attn_simt(a, st); }

}  // namespace csa
