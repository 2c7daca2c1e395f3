// Forward instantiations of the tensor-core GEMM.
#include "gemm_launch.cuh"

namespace moe {

cudaError_t launch_gemm_fwd(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st) {
  switch (kind) {
    case GK_ROUTER:
      return launch_gemm_inst<A_K_TILE, B_K_TILE, EPI_F32_BIAS, SCHED_ROWS>(p, grid, st);
    case GK_GATEUP:
      return launch_rows_two_pass<A_K_TILE, B_K_DUAL_N, EPI_SWIGLU_FWD>(p, grid, st);
    case GK_DOWN:
      return launch_rows_two_pass<A_K_TILE, B_K_TILE, EPI_BF16>(p, grid, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
