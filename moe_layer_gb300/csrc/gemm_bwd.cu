// Backward instantiations of the tensor-core GEMM.
#include "gemm_launch.cuh"

namespace moe {

cudaError_t launch_gemm_bwd(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st) {
  switch (kind) {
    case GK_DGRAD_DOWN:
      return launch_rows_two_pass<A_K_TILE, B_MN_TILE, EPI_SWIGLU_BWD>(p, grid, st);
    case GK_DGRAD_GATEUP:
      return launch_rows_two_pass<A_K_TILE, B_MN_DUAL_K, EPI_BF16>(p, grid, st);
    case GK_WGRAD:
      return launch_wgrad_two_pass<A_MN_TILE, B_MN_TILE>(p, grid, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
