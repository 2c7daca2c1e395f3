// MXFP8 (block-scaled E4M3) instantiations of the tensor-core GEMM.
#include "gemm_launch.cuh"

namespace moe {

cudaError_t launch_gemm_mx(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st) {
  switch (kind) {
    case GK_MX_GATEUP:
      return launch_gemm_inst<A_K_TILE, B_K_DUAL_N, EPI_SWIGLU_FWD, SCHED_ROWS, true>(p, grid, st);
    case GK_MX_DOWN:
    case GK_MX_DGRAD_GATEUP:
      return launch_gemm_inst<A_K_TILE, B_K_TILE, EPI_BF16, SCHED_ROWS, true>(p, grid, st);
    case GK_MX_DGRAD_DOWN:
      return launch_gemm_inst<A_K_TILE, B_K_TILE, EPI_SWIGLU_BWD, SCHED_ROWS, true>(p, grid, st);
    case GK_MX_WGRAD:
      return launch_gemm_inst<A_K_TILE, B_K_TILE, EPI_BF16, SCHED_WGRAD, true>(p, grid, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
