// Routing on the device, no host synchronization:
//   topk_count  softmax + top-k per token (one warp per token) and a per-chunk
//               expert histogram;
//   chunk_scan  for every expert, the exclusive prefix of its chunk counts and
//               its total count;
//   scatter     expert offsets (plain, padded to the row alignment, and in GEMM row
//               tiles), then the stable position of every route inside its
//               expert's row range.
// The scan and scatter bodies are the device functions of routing_dev.cuh,
// shared with the fused persistent routing launch (route_fused.cu).
#include "routing_dev.cuh"

namespace moe {

namespace {

// Softmax + top-k for the tokens of one chunk (kTopkWarpTokens tokens per
// warp).  Lane l holds the logits of experts l, l + 32, ... (NS slots, NS >=
// E / 32), sorts them once into selection order, and each of the k rounds
// takes the best of the 32 lanes' heads (a shuffle reduction) and moves the
// winning lane's list up by one.  A NaN logit becomes -inf with an index past
// E (route_candidate): it loses to every real logit, and selecting it (only
// NaN left) records MOE_ERR_DEVICE.
// Selection: logits descending, equal logits to the lower expert index.
// Weights: exp(l_j - l_max) / sum over the k selected (softmax over all E
// logits restricted to the selection and renormalized), the sum a butterfly
// over the warp (route_weight_sum runs the same tree in one thread).
constexpr int kTopkWarps = 16;
constexpr int kTopkWarpTokens = kChunkTokens / kTopkWarps;
static_assert(kChunkTokens % kTopkWarps == 0, "whole tokens per warp");
template <int NS>  // two blocks per SM with 8 slots; 16 need more registers than that leaves
__global__ void __launch_bounds__(kTopkWarps * 32, NS <= 8 ? 2 : 1)
    topk_count_kernel(const float* __restrict__ logits, int T, int E, int k,
                      int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                      int32_t* __restrict__ chunk_counts, int* status) {
  __shared__ int cnt[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kChunkTokens + warp * kTopkWarpTokens;
  for (int i = 0; i < kTopkWarpTokens; ++i) {
    const int t = t0 + i;
    if (t >= T) break;
    const float* lr = logits + static_cast<size_t>(t) * E;
    float v[NS];
    int ei[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int e = lane + 32 * s;
      if (e < E) {
        route_candidate(__ldg(lr + e), e, v[s], ei[s]);
      } else {
        v[s] = -INFINITY;
        ei[s] = INT_MAX;
      }
    }
    route_sort<NS>(v, ei);
    int my_e = 0;
    float my_v = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = v[0];
      int be = ei[0];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFullMask, bv, off);
        const int oe = __shfl_xor_sync(kFullMask, be, off);
        if (route_beats(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if (be >= E) {  // only reachable with NaN logits
        if (lane == 0) atomicCAS(status, 0, kDevBadValue);
        be = 0;
      } else if (ei[0] == be) {  // this lane's head was taken: move its list up
#pragma unroll
        for (int s = 0; s + 1 < NS; ++s) {
          v[s] = v[s + 1];
          ei[s] = ei[s + 1];
        }
        v[NS - 1] = -INFINITY;
        ei[NS - 1] = INT_MAX;
      }
      if (lane == j) {
        my_e = be;
        my_v = bv;
      }
    }
    const float m = __shfl_sync(kFullMask, my_v, 0);
    const float ex = lane < k ? expf(my_v - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
    if (lane < k) {
      topk_idx[static_cast<size_t>(t) * k + lane] = my_e;
      topk_w[static_cast<size_t>(t) * k + lane] = ex / sum;
      atomicAdd(&cnt[my_e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<size_t>(blockIdx.x) * E + e] = cnt[e];
}

// One warp per expert: exclusive prefix of the expert's chunk counts.
__global__ void __launch_bounds__(256)
    chunk_scan_kernel(const int32_t* __restrict__ chunk_counts, int nchunk, int E,
                      int32_t* __restrict__ chunk_base, int32_t* __restrict__ counts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  if (e >= E) return;
  route_scan_expert(chunk_counts, nchunk, E, e, lane, chunk_base, counts);
}

// One CTA per chunk of kChunkTokens tokens.
__global__ void __launch_bounds__(kChunkWarps * 32) scatter_kernel(const ScatterArgs a) {
  __shared__ int sbuf[kScatterSmemInts];
  const ScatterSmem sm{sbuf, sbuf + (kMaxExperts + 1), sbuf + 2 * (kMaxExperts + 1), sbuf + 3 * (kMaxExperts + 1),
                       sbuf + 4 * (kMaxExperts + 1), sbuf + 5 * (kMaxExperts + 1)};
  route_scatter_prefix(a, sm, blockIdx.x == 0);
  for (int e = blockIdx.x; e < a.E; e += gridDim.x) route_scatter_pad(a, sm, e);
  route_scatter_chunk(a, sm, blockIdx.x);
}

}  // namespace

cudaError_t launch_topk_count(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* topk_w, int32_t* chunk_counts, int* status, cudaStream_t st) {
  const int nchunk = (T + kChunkTokens - 1) / kChunkTokens;
  if (E <= 256)
    topk_count_kernel<8><<<nchunk, kTopkWarps * 32, 0, st>>>(logits, T, E, k, topk_idx, topk_w, chunk_counts,
                                                             status);
  else
    topk_count_kernel<16><<<nchunk, kTopkWarps * 32, 0, st>>>(logits, T, E, k, topk_idx, topk_w, chunk_counts,
                                                              status);
  return cudaGetLastError();
}

cudaError_t launch_chunk_scan(const int32_t* chunk_counts, int nchunk, int E, int32_t* chunk_base,
                              int32_t* counts, cudaStream_t st) {
  chunk_scan_kernel<<<(E + 7) / 8, 256, 0, st>>>(chunk_counts, nchunk, E, chunk_base, counts);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t* topk_idx, const float* topk_w, int T, int E, int k,
                           int row_align, const int32_t* chunk_base, const int32_t* counts, int32_t* offsets,
                           int32_t* row_start, int32_t* tile_start, int32_t* pair_start, int32_t* rem_start,
                           int32_t* perm_token, int32_t* route_row, int32_t* perm_token_pad,
                           int32_t* route_row_pad, float* perm_w_pad, cudaStream_t st) {
  const int nchunk = (T + kChunkTokens - 1) / kChunkTokens;
  const ScatterArgs a{topk_idx, topk_w, T, E, k, row_align, chunk_base, counts, offsets, row_start, tile_start,
                      pair_start, rem_start, perm_token, route_row, perm_token_pad, route_row_pad, perm_w_pad};
  scatter_kernel<<<nchunk, kChunkWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
