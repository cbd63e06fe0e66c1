// Grouped W8A8 GEMM on the tcgen05 tensor cores (sm_103a).
#include "wq_common.cuh"

namespace wq {

bool gemm_tc_supported(const GemmArgs &) { return false; }

int launch_gemm_tc(const GemmArgs &, const Tile *, const int32_t *, int, cudaStream_t) {
  return WQ_ERR_UNSUPPORTED;
}

}  // namespace wq
