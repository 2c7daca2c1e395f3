// The routing of the layer in one persistent launch: router projection with
// the softmax + top-k in its epilogue, the per-expert scan of the chunk
// histograms and the stable scatter.  One CTA per SM, launched cooperatively
// so that all CTAs are resident together; the stages hand off through device
// counters (grid barriers).  This is a first slice of the single-GPU form of
// the pages' persistent megakernel (Mixture-of-Kittens blog post, sections
// "Megakernel" and "Scheduling the overlaps"): the stages run back to back in
// one launch with no host involvement between them.
//
// It computes bitwise what the separate kernels compute (routing.cu): the
// same router GEMM, the same selection order and weight arithmetic
// (routing_dev.cuh), the same scan and scatter.  The dispatch of the x rows
// stays a separate kernel: measured at the DSV3 shape, copying the 3.8 GB of
// rows inside this launch (one CTA per SM) took 0.66 ms with 16-byte register
// copies, 16 or 32 in flight per lane, and 0.87 ms with a ring of 14 KB
// cp.async.bulk row copies through shared memory, against 0.53 ms for the
// standalone permute kernel with many CTAs per SM.
//
// Failure path.  Every wait is bounded (kWaitTimeoutNs of %globaltimer).  A
// CTA whose GEMM stage aborted, or whose barrier wait ran out, records
// MOE_ERR_DEVICE_TIMEOUT, raises the launch's failure flag and returns; the
// others see the flag after their next barrier (or time out on it) and return
// too.  The host zeroes the routing arrays before the launch, so whatever
// stage was cut short, every index a later kernel reads stays in range.
#include <string.h>

#include <atomic>

#include "moe_internal.h"
#include "routing_dev.cuh"
#include "tc_gemm.cuh"

namespace moe {

namespace {

// Shared memory of the launch (the router GEMM's), reused by the scatter.
constexpr int kRouteFusedSmem = gemm_smem_bytes_for<false, EPI_ROUTE, SCHED_ROWS>();

struct RouteFusedArgs {
  ScatterArgs sc;         // scan / scatter inputs and outputs
  int32_t* chunk_counts;  // [nchunk, E], zero at launch (the epilogue adds to it)
  int32_t* chunk_base;    // [nchunk, E]
  int nchunk;
  int* status;
  int* sync;              // [4]: barrier counters and the failure flag (sync[3]), zero at launch
  int extra_arrivals;     // test hook: arrivals the first barrier waits for beyond the grid
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier on counter `c` (target arrivals), bounded.  Returns false (for
// every thread of the CTA) when the wait ran out or another CTA raised the
// failure flag; the CTA must then return.
__device__ __forceinline__ bool grid_barrier(int* c, int target, int* fail, int* status, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's writes before its arrival
    atomicAdd(c, 1);
    const unsigned long long t0 = globaltimer_ns();
    int ok = 1;
    while (ld_acquire(c) < target) {
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
        atomicCAS(status, 0, kDevTimeout);
        atomicExch(fail, 1);
        ok = 0;
        break;
      }
    }
    __threadfence();
    if (ok && ld_acquire(fail)) ok = 0;
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    route_fused_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ RouteFusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_ok;
  int* fail = a.sync + 3;
  // 1. router logits + softmax / top-k per token, chunk histograms
  if (!tc_gemm_run<A_K_TILE, B_K_TILE, EPI_ROUTE, SCHED_ROWS>(p, smem_raw)) {
    if (threadIdx.x == 0) {
      atomicExch(fail, 1);
      __threadfence();
    }
    return;
  }
  if (!grid_barrier(a.sync + 0, static_cast<int>(gridDim.x) + a.extra_arrivals, fail, a.status, &s_ok)) return;
  // 2. per-expert scan of the chunk histograms: a warp per expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x / 32;
  for (int e = blockIdx.x * nw + warp; e < a.sc.E; e += gridDim.x * nw)
    route_scan_expert(a.chunk_counts, a.nchunk, a.sc.E, e, lane, a.chunk_base, const_cast<int32_t*>(a.sc.counts));
  if (!grid_barrier(a.sync + 1, static_cast<int>(gridDim.x), fail, a.status, &s_ok)) return;
  // 3. scatter: the offsets in every CTA, the padding rows and the chunks spread over the CTAs
  int* sbuf = reinterpret_cast<int*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const ScatterSmem sm{sbuf, sbuf + (kMaxExperts + 1), sbuf + 2 * (kMaxExperts + 1), sbuf + 3 * (kMaxExperts + 1),
                       sbuf + 4 * (kMaxExperts + 1), sbuf + 5 * (kMaxExperts + 1)};
  route_scatter_prefix(a.sc, sm, blockIdx.x == 0);
  for (int e = blockIdx.x; e < a.sc.E; e += gridDim.x) route_scatter_pad(a.sc, sm, e);
  for (int c = blockIdx.x; c < a.nchunk; c += gridDim.x) route_scatter_chunk(a.sc, sm, c);
}

static_assert(kGemmThreads == kChunkWarps * 32, "the scatter stage runs on the GEMM's CTA");
static_assert(kBM == 2 * kChunkTokens, "a GEMM row tile covers two routing chunks");

}  // namespace

bool route_fused_supported(int64_t E, int64_t k) { return E <= kBN && k <= kRouteMaxK; }

cudaError_t launch_route_fused(const GemmParams& p, const ScatterArgs& sc, int32_t* chunk_counts,
                               int32_t* chunk_base, int nchunk, int* status, int* sync, int extra_arrivals, int grid,
                               cudaStream_t st) {
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  constexpr int smem = kRouteFusedSmem;
  static_assert(smem >= 1024 + kScatterSmemInts * 4, "the scatter reuses the GEMM's shared memory");
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit == 0 || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(route_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  RouteFusedArgs a;
  memset(static_cast<void*>(&a), 0, sizeof(a));
  a.sc = sc;
  a.chunk_counts = chunk_counts;
  a.chunk_base = chunk_base;
  a.nchunk = nchunk;
  a.status = status;
  a.sync = sync;
  a.extra_arrivals = extra_arrivals;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_fused_kernel, p, a);
}

}  // namespace moe
