// moe_route_topk_noalloc: the routing entry point for callers that cannot
// allocate device memory.
//
// moe_route_topk needs a caller-provided workspace for its intermediate
// arrays (per-chunk expert histograms and their prefix sums, the padded
// expert-grouped permutation).  Some callers have no way to provide one: a
// process whose device memory is handed out only by a pool fixed at start-up,
// or code that must not create new allocations while it runs (an allocation
// can block, fail, or fragment memory another component manages).  This entry
// point keeps those intermediates in one static device array that the library
// owns, so a call needs nothing beyond its inputs and outputs.
//
// The array is file-scope `__device__` memory of kNoAllocScratchBytes; every
// GPU that loads the library keeps it until the process exits.  All calls on a
// device share it: two calls whose work overlaps on the GPU (different streams,
// no ordering between them) race on it and give wrong results.  Calls ordered
// on one stream are fine.
#include <string.h>

#include <mutex>

#include "gemm_launch.cuh"
#include "moe_internal.h"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace moe {
namespace {

// Size of the static scratch.  The routing intermediates take about
// 12 T k + 8 E ceil(T / 64) + 504 E bytes plus 2 KB (noalloc_bytes), so 9 MiB
// hold up to 65536 tokens at top-8 with 256 experts (8.52 MB); larger shapes
// are rejected.
constexpr size_t kNoAllocScratchBytes = size_t(9) << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch for the current device.  Looked up
// once per device with that device current (the host-side name of the array
// is not a device address).
moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct NoAllocLayout {
  size_t status, chunk_counts, chunk_base, row_start, tile_start, perm_token_pad, route_row_pad, perm_w_pad,
      total;
};

NoAllocLayout noalloc_bytes(int64_t T, int64_t E, int64_t k) {
  const int64_t nchunk = (T + kChunkTokens - 1) / kChunkTokens;
  const int64_t Rp = T * k + E * (kRowAlign - 1);
  NoAllocLayout L;
  size_t off = 0;
  L.status = off;
  off = align256(off + 256);
  L.chunk_counts = off;
  off = align256(off + size_t(nchunk * E) * 4);
  L.chunk_base = off;
  off = align256(off + size_t(nchunk * E) * 4);
  L.row_start = off;
  off = align256(off + size_t(E + 1) * 4);
  L.tile_start = off;
  off = align256(off + size_t(E + 1) * 4);
  L.perm_token_pad = off;
  off = align256(off + size_t(Rp) * 4);
  L.route_row_pad = off;
  off = align256(off + size_t(T * k) * 4);
  L.perm_w_pad = off;
  off = align256(off + size_t(Rp) * 4);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_topk_noalloc(const moe_config* cfg, const void* x, const void* W_router,
                                             const float* router_bias, const float* logits_in,
                                             float* logits_out, int32_t* topk_idx, float* topk_w,
                                             int32_t* counts, int32_t* offsets, int32_t* perm_token,
                                             int32_t* route_row, void* stream) {
  // the configuration checks of moe_route_topk (the expert and shared-expert
  // widths do not enter the routing, but a configuration moe_route_topk
  // rejects is rejected here too)
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (cfg->T < 0 || cfg->d <= 0 || cfg->I <= 0 || cfg->E <= 0 || cfg->top_k <= 0 || cfg->n_shared < 0 ||
      (cfg->n_shared && cfg->I_shared <= 0))
    return MOE_ERR_INVALID_ARG;
  if (cfg->precision != MOE_BF16 || cfg->flags != 0) return MOE_ERR_UNSUPPORTED;
  if (cfg->E > kMaxExperts || cfg->top_k > kMaxTopK || cfg->top_k > cfg->E || cfg->n_shared > 1 ||
      cfg->d % 64 || cfg->I % 64 || (cfg->n_shared && cfg->I_shared % 64))
    return MOE_ERR_UNSUPPORTED;
  const int64_t T = cfg->T, E = cfg->E, k = cfg->top_k, d = cfg->d;
  if (T == 0) return MOE_OK;
  if (!topk_idx || !topk_w || !counts || !offsets || !perm_token || !route_row) return MOE_ERR_INVALID_ARG;
  // the logits are not kept in the static scratch: computed logits go to logits_out
  if (!logits_in && (!logits_out || !x || !W_router || !aligned16(x) || !aligned16(W_router)))
    return MOE_ERR_INVALID_ARG;
  const NoAllocLayout L = noalloc_bytes(T, E, k);
  if (L.total > kNoAllocScratchBytes || T * k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;

  void* base = nullptr;
  const moe_status st0 = scratch_for_current_device(&base);
  if (st0 != MOE_OK) return st0;
  char* b = static_cast<char*>(base);
  int* status = reinterpret_cast<int*>(b + L.status);
  int32_t* chunk_counts = reinterpret_cast<int32_t*>(b + L.chunk_counts);
  int32_t* chunk_base = reinterpret_cast<int32_t*>(b + L.chunk_base);
  int32_t* row_start = reinterpret_cast<int32_t*>(b + L.row_start);
  int32_t* tile_start = reinterpret_cast<int32_t*>(b + L.tile_start);
  int32_t* perm_token_pad = reinterpret_cast<int32_t*>(b + L.perm_token_pad);
  int32_t* route_row_pad = reinterpret_cast<int32_t*>(b + L.route_row_pad);
  float* perm_w_pad = reinterpret_cast<float*>(b + L.perm_w_pad);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // The status word is the only part that must start at zero; every other
  // array is fully written by the kernels below before it is read.
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  const float* lg = logits_in;
  if (!lg) {
    GemmParams p;
    memset(static_cast<void*>(&p), 0, sizeof(p));
    if (!make_tmap_bf16(&p.tmA, x, uint64_t(d), uint64_t(T), uint64_t(d), 64, kBM)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16(&p.tmB0, W_router, uint64_t(d), uint64_t(E), uint64_t(d), 64, kBN))
      return MOE_ERR_CUDA;
    p.dense_rows = static_cast<int>(T);
    p.N = static_cast<int>(E);
    p.K = static_cast<int>(d);
    p.out = logits_out;
    p.ldo = E;
    p.bias = router_bias;
    p.status = status;
    const int64_t tiles = ((T + kBM - 1) / kBM) * ((E + kBN - 1) / kBN);
    const int grid = static_cast<int>(tiles < device_sm_count() ? tiles : device_sm_count());
    if (launch_gemm(GK_ROUTER, p, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
    lg = logits_out;
  }
  const int Ti = static_cast<int>(T), Ei = static_cast<int>(E), ki = static_cast<int>(k);
  const int nchunk = static_cast<int>((T + kChunkTokens - 1) / kChunkTokens);
  if (launch_topk_count(lg, Ti, Ei, ki, topk_idx, topk_w, chunk_counts, status, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_chunk_scan(chunk_counts, nchunk, Ei, chunk_base, counts, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_scatter(topk_idx, topk_w, Ti, Ei, ki, kRowAlign, chunk_base, counts, offsets, row_start, tile_start,
                     nullptr, nullptr, perm_token, route_row, perm_token_pad, route_row_pad, perm_w_pad, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
