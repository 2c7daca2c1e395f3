// Routing on the device, no host synchronization:
//   topk_count  softmax + top-k per token (one warp per token) and a per-chunk
//               expert histogram;
//   chunk_scan  for every expert, the exclusive prefix of its chunk counts and
//               its total count;
//   scatter     expert offsets (plain, padded to the row alignment, and in GEMM row
//               tiles), then the stable position of every route inside its
//               expert's row range.
// Together they are the one-rank form of the counting schedule in the
// Mixture-of-Kittens blog post, section "Choosing the right communication
// direction / Scheduling": a counting pass, region offsets, then a pass that
// writes every route in (token, slot) order.  Only integer atomics on shared
// memory are used, so the result is exact and deterministic.
#include <float.h>
#include <limits.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Selection order: a candidate (logit v, expert e) comes before another when
// its logit is larger, or equal with a lower expert index.
__device__ __forceinline__ bool beats(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

// Sorts N candidates into selection order with Batcher's odd-even merge
// network (19 compare-exchanges for N = 8, 63 for N = 16), in registers.
template <int N>
__device__ __forceinline__ void sort_candidates(float (&v)[N], int (&e)[N]) {
#pragma unroll
  for (int p = 1; p < N; p <<= 1)
#pragma unroll
    for (int kk = p; kk >= 1; kk >>= 1)
#pragma unroll
      for (int j = kk % p; j + kk < N; j += 2 * kk)
#pragma unroll
        for (int i = 0; i < kk && i + j + kk < N; ++i)
          if ((i + j) / (2 * p) == (i + j + kk) / (2 * p) && beats(v[i + j + kk], e[i + j + kk], v[i + j], e[i + j])) {
            const float tv = v[i + j];
            v[i + j] = v[i + j + kk];
            v[i + j + kk] = tv;
            const int te = e[i + j];
            e[i + j] = e[i + j + kk];
            e[i + j + kk] = te;
          }
}

// Softmax + top-k for the tokens of one chunk (kTopkWarpTokens tokens per
// warp).  Lane l holds the logits of experts l, l + 32, ... (NS slots, NS >=
// E / 32), sorts them once into selection order, and each of the k rounds
// takes the best of the 32 lanes' heads (a shuffle reduction) and moves the
// winning lane's list up by one.  A NaN logit becomes -inf with an index past
// E: it loses to every real logit, and selecting it (only NaN left) records
// MOE_ERR_DEVICE.
// Selection: logits descending, equal logits to the lower expert index.
// Weights: exp(l_j - l_max) / sum over the k selected (softmax over all E
// logits restricted to the selection and renormalized).
constexpr int kTopkWarps = 16;
constexpr int kTopkWarpTokens = kChunkTokens / kTopkWarps;
static_assert(kChunkTokens % kTopkWarps == 0, "whole tokens per warp");
constexpr int kNanIndex = 1 << 30;  // or-ed into a NaN logit's index
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
        const float x = __ldg(lr + e);
        const bool nan = x != x;
        v[s] = nan ? -INFINITY : x;
        ei[s] = nan ? (e | kNanIndex) : e;
      } else {
        v[s] = -INFINITY;
        ei[s] = INT_MAX;
      }
    }
    sort_candidates<NS>(v, ei);
    int my_e = 0;
    float my_v = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = v[0];
      int be = ei[0];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (beats(ov, oe, bv, be)) {
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
    const float m = __shfl_sync(kFull, my_v, 0);
    const float ex = lane < k ? expf(my_v - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
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
  int carry = 0;
  for (int c0 = 0; c0 < nchunk; c0 += 32 * 8) {
    int v[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + lane * 8 + i;
      v[i] = c < nchunk ? __ldg(chunk_counts + static_cast<size_t>(c) * E + e) : 0;
      s += v[i];
    }
    int inc = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, inc, off);
      if (lane >= off) inc += o;
    }
    int run = carry + inc - s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + lane * 8 + i;
      if (c < nchunk) chunk_base[static_cast<size_t>(c) * E + e] = run;
      run += v[i];
    }
    carry += __shfl_sync(kFull, inc, 31);
  }
  if (lane == 0) counts[e] = carry;
}

__device__ __forceinline__ int pad_rows(int c, int align) { return (c + align - 1) / align * align; }
__device__ __forceinline__ int row_tiles(int c, int align) {
  return (pad_rows(c, align) + kTileRows - 1) / kTileRows;
}

// Tile pairs of an expert with `tiles` GEMM row tiles: all of them pair up when
// the count is even; an odd count runs every tile on one SM (a lone last tile
// would make that pass read the expert's weights a second time).
__device__ __forceinline__ int expert_pairs(int tiles) { return (tiles & 1) ? 0 : tiles >> 1; }

__global__ void __launch_bounds__(kChunkWarps * 32)
    scatter_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int T,
                   int E, int k, int align, const int32_t* __restrict__ chunk_base,
                   const int32_t* __restrict__ counts, int32_t* __restrict__ offsets_out,
                   int32_t* __restrict__ row_start_out, int32_t* __restrict__ tile_start_out,
                   int32_t* __restrict__ pair_start_out, int32_t* __restrict__ rem_start_out,
                   int32_t* __restrict__ perm_token,
                   int32_t* __restrict__ route_row, int32_t* __restrict__ perm_token_pad,
                   int32_t* __restrict__ route_row_pad, float* __restrict__ perm_w_pad) {
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_rs[kMaxExperts + 1];
  __shared__ int s_ts[kMaxExperts + 1];
  __shared__ int s_ps[kMaxExperts + 1];
  __shared__ int s_qs[kMaxExperts + 1];
  __shared__ int wcnt[kChunkWarps][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // 1. expert offsets: exclusive prefix of counts, of padded row counts, of
  //    GEMM row tiles, and of the tiles the grouped GEMMs run in pairs on SM
  //    pairs and alone on one SM (expert_pairs)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    int sum = 0, psum = 0, tsum = 0, qsum = 0, osum = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        const int c = __ldg(counts + e);
        const int tiles = row_tiles(c, align);
        sum += c;
        psum += pad_rows(c, align);
        tsum += tiles;
        qsum += expert_pairs(tiles);
        osum += tiles - 2 * expert_pairs(tiles);
      }
    }
    int inc = sum, pinc = psum, tinc = tsum, qinc = qsum, oinc = osum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, inc, off);
      const int po = __shfl_up_sync(kFull, pinc, off);
      const int to = __shfl_up_sync(kFull, tinc, off);
      const int qo = __shfl_up_sync(kFull, qinc, off);
      const int oo = __shfl_up_sync(kFull, oinc, off);
      if (lane >= off) {
        inc += o;
        pinc += po;
        tinc += to;
        qinc += qo;
        oinc += oo;
      }
    }
    int run = inc - sum, prun = pinc - psum, trun = tinc - tsum, qrun = qinc - qsum, orun = oinc - osum;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        s_off[e] = run;
        s_rs[e] = prun;
        s_ts[e] = trun;
        s_ps[e] = qrun;
        s_qs[e] = orun;
        const int c = __ldg(counts + e);
        const int tiles = row_tiles(c, align);
        run += c;
        prun += pad_rows(c, align);
        trun += tiles;
        qrun += expert_pairs(tiles);
        orun += tiles - 2 * expert_pairs(tiles);
      }
    }
    if (lane == 31) {
      s_off[E] = inc;
      s_rs[E] = pinc;
      s_ts[E] = tinc;
      s_ps[E] = qinc;
      s_qs[E] = oinc;
    }
  }
  for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) wcnt[i / E][i % E] = 0;
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      offsets_out[e] = s_off[e];
      row_start_out[e] = s_rs[e];
      tile_start_out[e] = s_ts[e];
      if (pair_start_out) pair_start_out[e] = s_ps[e];
      if (rem_start_out) rem_start_out[e] = s_qs[e];
    }
  }
  // padding rows of the padded layout: no token, weight 0
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int beg = s_rs[e] + __ldg(counts + e), end = s_rs[e + 1];
    for (int r = beg + threadIdx.x; r < end; r += blockDim.x) {
      perm_token_pad[r] = -1;
      perm_w_pad[r] = 0.f;
    }
  }

  // 2. per-warp expert counts of this chunk
  const int tw0 = blockIdx.x * kChunkTokens + warp * kWarpTokens;
  const int ntok = max(0, min(kWarpTokens, T - tw0));
  const int nr = ntok * k;
  const int32_t* my_idx = topk_idx + static_cast<size_t>(tw0) * k;
  for (int r = lane; r < nr; r += 32) atomicAdd(&wcnt[warp][__ldg(my_idx + r)], 1);
  __syncthreads();
  // 3. warp bases: chunk base of the expert plus the routes of earlier warps
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int base = __ldg(chunk_base + static_cast<size_t>(blockIdx.x) * E + e);
    for (int w = 0; w < kChunkWarps; ++w) {
      const int c = wcnt[w][e];
      wcnt[w][e] = base;
      base += c;
    }
  }
  __syncthreads();
  // 4. stable ranks, 32 routes at a time in (token, slot) order
  for (int r0 = 0; r0 < nr; r0 += 32) {
    const int r = r0 + lane;
    const bool valid = r < nr;
    const int e = valid ? __ldg(my_idx + r) : -1;
    const unsigned peers = __match_any_sync(kFull, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int local = 0;
    if (valid) local = wcnt[warp][e] + rank;
    __syncwarp();
    if (valid && rank == 0) wcnt[warp][e] += __popc(peers);
    __syncwarp();
    if (valid) {
      const int tl = r / k;
      const int t = tw0 + tl;
      const int j = r - tl * k;
      const size_t tj = static_cast<size_t>(t) * k + j;
      const int ru = s_off[e] + local;
      const int rp = s_rs[e] + local;
      perm_token[ru] = t;
      route_row[tj] = ru;
      perm_token_pad[rp] = t;
      route_row_pad[tj] = rp;
      perm_w_pad[rp] = __ldg(topk_w + tj);
    }
  }
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
  scatter_kernel<<<nchunk, kChunkWarps * 32, 0, st>>>(topk_idx, topk_w, T, E, k, row_align, chunk_base, counts,
                                                      offsets, row_start, tile_start, pair_start, rem_start,
                                                      perm_token,
                                                      route_row, perm_token_pad, route_row_pad,
                                                      perm_w_pad);
  return cudaGetLastError();
}

}  // namespace moe
