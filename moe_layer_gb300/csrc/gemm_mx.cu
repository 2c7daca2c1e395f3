// MXFP8 (block-scaled E4M3) instantiations of the tensor-core GEMM.  The
// gate/up projection runs as a 2-SM pass over the experts with an even number
// of 128-row tiles and a 1-SM pass over the others; the other GEMMs run every
// tile on one SM.  Measured at the DSV3 shape (same box, alternating runs):
// on SM pairs gate/up took 3.49-3.50 ms against 3.50-3.55 on one SM, but the
// down projection 1.86-1.87 against 1.76-1.78 and the dgrad of gate/up
// 3.33-3.34 against 3.20-3.23.  Unlike the bf16 GEMMs, the MXFP8 ones are
// not bound by the shared-memory traffic that pairs halve (their scale
// transfers and copies cost 10-13 %, the single accumulator's hand-off about
// 2 %; a block-scaled 128x256x32 MMA issues in as many cycles as a bf16
// 128x256x16 one).
#include "gemm_launch.cuh"

namespace moe {

cudaError_t launch_gemm_mx(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st) {
  switch (kind) {
    case GK_MX_GATEUP:
      return launch_rows_two_pass<A_K_TILE, B_K_DUAL_N, EPI_SWIGLU_FWD, true>(p, grid, st);
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
