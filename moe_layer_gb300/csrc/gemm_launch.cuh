// Launch helper for one instantiation of the tensor-core GEMM: sets the
// dynamic shared-memory limit once per device, then launches persistently.
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
  constexpr int threads = gemm_threads<MX, EPI, SCH>();
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit == 0 || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  kfn<<<grid, threads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_fwd(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_gemm_bwd(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);
cudaError_t launch_gemm_mx(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);

}  // namespace moe
