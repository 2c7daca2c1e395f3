// Launch helper for one instantiation of the tensor-core GEMM: sets the
// dynamic shared-memory limit once per device, then launches persistently
// (2-SM instantiations as clusters of two CTAs, on an even grid).
#pragma once
#include <atomic>

#include "moe_internal.h"
#include "tc_gemm.cuh"

namespace moe {

template <int AM, int BMO, int EPI, int SCH, bool MX = false>
cudaError_t launch_gemm_inst(const GemmParams& p, int grid, cudaStream_t st) {
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto kfn = tc_gemm_kernel<AM, BMO, EPI, SCH, MX>;
  constexpr int smem = gemm_smem_bytes_for<MX, EPI, SCH>();
  static_assert(smem <= 227 * 1024, "shared memory of one CTA");
  constexpr int threads = gemm_threads<MX, EPI, SCH>();
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit == 0 || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  if constexpr (sched_pair(SCH)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid < 2 ? 2 : grid & ~1));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, p);
  } else {
    kfn<<<grid, threads, smem, st>>>(p);
    return cudaGetLastError();
  }
}

// The row GEMMs other than the router projection (bf16 and MXFP8): a 2-SM pass over the
// pairs of m-tiles, then a 1-SM pass over the rest: every tile of each expert
// with an odd number of them (grouped rows), or the last m-tile of an odd
// dense row range.  Grouped problems launch both passes always (their tile
// counts live on the device; a pass without tiles exits at once).
template <int AM, int BMO, int EPI, bool MX = false>
cudaError_t launch_rows_two_pass(const GemmParams& p, int grid, cudaStream_t st) {
  const int dense_mt = p.dense_rows > 0 ? (p.dense_rows + kBM - 1) / kBM : 0;
  if (p.dense_rows == 0 || dense_mt >= 2) {
    const cudaError_t e = launch_gemm_inst<AM, BMO, EPI, SCHED_ROWS2, MX>(p, grid, st);
    if (e != cudaSuccess) return e;
  }
  if (p.dense_rows > 0 && dense_mt % 2 == 0) return cudaSuccess;
  GemmParams q = p;
  q.part = 1;
  if (p.dense_rows == 0 || dense_mt >= 2) ++extra_kernel_launches();
  return launch_gemm_inst<AM, BMO, EPI, SCHED_ROWS, MX>(q, grid, st);
}

// Weight gradients likewise: pairs of m-tiles (weight rows) on SM pairs, and
// the last m-tile on one SM when M_out / 128 is odd; or all on one SM when
// the host asks (wgrad_mode 1: short K, where a pair's two epilogues, which
// its MMAs wait for, cost more than the halved shared-memory traffic saves;
// wgrad_mode 2: the shortest K, with twice the epilogue warps).
template <int AM, int BMO>
cudaError_t launch_wgrad_two_pass(const GemmParams& p, int grid, cudaStream_t st) {
  if (p.wgrad_mode == 2) return launch_gemm_inst<AM, BMO, EPI_BF16, SCHED_WGRAD_WIDE>(p, grid, st);
  if (p.wgrad_mode == 1) return launch_gemm_inst<AM, BMO, EPI_BF16, SCHED_WGRAD>(p, grid, st);
  const int num_mt = (p.M_out + kBM - 1) / kBM;
  if (num_mt >= 2) {
    const cudaError_t e = launch_gemm_inst<AM, BMO, EPI_BF16, SCHED_WGRAD2>(p, grid, st);
    if (e != cudaSuccess) return e;
  }
  if (num_mt % 2 == 0) return cudaSuccess;
  GemmParams q = p;
  q.part = 1;
  if (num_mt >= 2) ++extra_kernel_launches();
  return launch_gemm_inst<AM, BMO, EPI_BF16, SCHED_WGRAD>(q, grid, st);
}

cudaError_t launch_gemm_fwd(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_gemm_bwd(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_gemm_mx(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);

}  // namespace moe
