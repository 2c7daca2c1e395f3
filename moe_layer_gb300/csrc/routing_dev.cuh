// Device functions of the routing: softmax + top-k of one token, the per-expert
// scan of chunk histograms, and the stable scatter of one chunk's routes.  The
// standalone routing kernels (routing.cu) and the fused persistent routing
// launch (route_fused.cu) run the same functions, so both produce bitwise the
// same routing.
//
// Together they are the one-rank form of the counting schedule in the
// Mixture-of-Kittens blog post, section "Choosing the right communication
// direction / Scheduling": a counting pass, region offsets, then a pass that
// writes every route in (token, slot) order.  Only integer atomics on shared
// memory are used, so the result is exact and deterministic.
//
// Arrays another CTA of the same launch may have written (the fused launch)
// are read with __ldcg (L2, not the non-coherent read-only path).
#pragma once
#include <float.h>
#include <limits.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kNanIndex = 1 << 30;  // or-ed into a NaN logit's index

// Selection order: a candidate (logit v, expert e) comes before another when
// its logit is larger, or equal with a lower expert index.
__device__ __forceinline__ bool route_beats(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

// A logit as a selection candidate: a NaN becomes -inf with an index past E,
// so that it loses to every real logit and selecting it is detectable.
__device__ __forceinline__ void route_candidate(float x, int e, float& v, int& ei) {
  const bool nan = x != x;
  v = nan ? -INFINITY : x;
  ei = nan ? (e | kNanIndex) : e;
}

// Compare-exchange in selection order: afterwards (va, ea) comes first.
// Branch-free (selects), so a network of them keeps the values in registers.
__device__ __forceinline__ void route_ce(float& va, int& ea, float& vb, int& eb) {
  const bool sw = route_beats(vb, eb, va, ea);
  const float tv = sw ? vb : va;
  const int te = sw ? eb : ea;
  vb = sw ? va : vb;
  eb = sw ? ea : eb;
  va = tv;
  ea = te;
}

// Sorts N candidates into selection order with Batcher's odd-even merge
// network (19 compare-exchanges for N = 8, 63 for N = 16), in registers.
template <int N>
__device__ __forceinline__ void route_sort(float (&v)[N], int (&e)[N]) {
#pragma unroll
  for (int p = 1; p < N; p <<= 1)
#pragma unroll
    for (int kk = p; kk >= 1; kk >>= 1)
#pragma unroll
      for (int j = kk % p; j + kk < N; j += 2 * kk)
#pragma unroll
        for (int i = 0; i < kk && i + j + kk < N; ++i)
          if ((i + j) / (2 * p) == (i + j + kk) / (2 * p)) route_ce(v[i + j], e[i + j], v[i + j + kk], e[i + j + kk]);
}

// The KM best of a sorted list (l, KM entries) and a sorted chunk (c, C >= KM
// entries), sorted, into l: pairing l[i] with c[KM - 1 - i] and keeping the
// better of each pair leaves the KM best as a bitonic sequence, which KM/2-
// wide half-cleaners then sort (KM a power of two).
template <int KM, int C>
__device__ __forceinline__ void route_merge_top(float (&lv)[KM], int (&le)[KM], const float (&cv)[C], const int (&ce)[C]) {
  static_assert(C >= KM && (KM & (KM - 1)) == 0, "merge shape");
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    const bool take = route_beats(cv[KM - 1 - i], ce[KM - 1 - i], lv[i], le[i]);
    lv[i] = take ? cv[KM - 1 - i] : lv[i];
    le[i] = take ? ce[KM - 1 - i] : le[i];
  }
#pragma unroll
  for (int j = KM / 2; j > 0; j >>= 1)
#pragma unroll
    for (int i = 0; i < KM; ++i)
      if ((i & j) == 0) route_ce(lv[i], le[i], lv[i + j], le[i + j]);
}

// Router weights of a token from its k selected logits in slot order (held by
// lanes 0..k-1 of a warp, or by one thread as v[0..k-1]): exp(l_j - l_0)
// normalized by their sum.  The sum is taken in the order of a 32-lane xor
// butterfly (offsets 16, 8, 4, 2, 1) over lanes whose slot is >= k holding 0;
// route_weight_sum runs that tree in one thread, so the warp form and the
// single-thread form give bitwise the same weights.
template <int KM>
__device__ __forceinline__ float route_weight_sum(const float (&ex)[KM], int k) {
  float a[32];
#pragma unroll
  for (int l = 0; l < 32; ++l) a[l] = (l < KM && l < k) ? ex[l < KM ? l : 0] : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float b[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) b[l] = a[l] + a[l ^ off];
#pragma unroll
    for (int l = 0; l < 32; ++l) a[l] = b[l];
  }
  return a[0];
}

// ---------------------------------------------------------------- scan
// One warp, one expert e: exclusive prefix of the expert's chunk counts
// (chunk_base[c][e]) and its total (counts[e]).
__device__ __forceinline__ void route_scan_expert(const int32_t* chunk_counts, int nchunk, int E, int e,
                                                  int lane, int32_t* chunk_base, int32_t* counts) {
  int carry = 0;
  for (int c0 = 0; c0 < nchunk; c0 += 32 * 8) {
    int v[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + lane * 8 + i;
      v[i] = c < nchunk ? __ldcg(chunk_counts + static_cast<size_t>(c) * E + e) : 0;
      s += v[i];
    }
    int inc = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFullMask, inc, off);
      if (lane >= off) inc += o;
    }
    int run = carry + inc - s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = c0 + lane * 8 + i;
      if (c < nchunk) chunk_base[static_cast<size_t>(c) * E + e] = run;
      run += v[i];
    }
    carry += __shfl_sync(kFullMask, inc, 31);
  }
  if (lane == 0) counts[e] = carry;
}

// ---------------------------------------------------------------- scatter
__device__ __forceinline__ int route_pad_rows(int c, int align) { return (c + align - 1) / align * align; }
__device__ __forceinline__ int route_row_tiles(int c, int align) {
  return (route_pad_rows(c, align) + kTileRows - 1) / kTileRows;
}
// Tile pairs of an expert with `tiles` GEMM row tiles: all of them pair up when
// the count is even; an odd count runs every tile on one SM (a lone last tile
// would make that pass read the expert's weights a second time).
__device__ __forceinline__ int route_expert_pairs(int tiles) { return (tiles & 1) ? 0 : tiles >> 1; }

// Shared-memory arrays of the scatter (each [kMaxExperts + 1], wcnt
// [kChunkWarps][kMaxExperts]): the expert offsets of every layout and the
// per-warp route counts of the chunk being scattered.
struct ScatterSmem {
  int* off;  // unpadded row offsets
  int* rs;   // padded row offsets
  int* ts;   // GEMM row tiles
  int* ps;   // tile pairs (SM pairs)
  int* qs;   // tiles on one SM
  int* wcnt;
};
constexpr int kScatterSmemInts = 5 * (kMaxExperts + 1) + kChunkWarps * kMaxExperts;

struct ScatterArgs {
  const int32_t* topk_idx;
  const float* topk_w;
  int T, E, k, align;
  const int32_t* chunk_base;
  const int32_t* counts;
  int32_t *offsets, *row_start, *tile_start, *pair_start, *rem_start;
  int32_t *perm_token, *route_row, *perm_token_pad, *route_row_pad;
  float* perm_w_pad;
};

// 1. Expert offsets (kChunkWarps warps of the CTA): exclusive prefix of
//    counts, of padded row counts, of GEMM row tiles, and of the tiles the
//    grouped GEMMs run in pairs on SM pairs and alone on one SM.  Ends with a
//    CTA barrier.  write_global: also store them as the layout arrays.
__device__ __forceinline__ void route_scatter_prefix(const ScatterArgs& a, const ScatterSmem& sm, bool write_global) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, align = a.align;
  if (warp == 0) {
    const int per = (E + 31) / 32;
    int sum = 0, psum = 0, tsum = 0, qsum = 0, osum = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        const int c = __ldcg(a.counts + e);
        const int tiles = route_row_tiles(c, align);
        sum += c;
        psum += route_pad_rows(c, align);
        tsum += tiles;
        qsum += route_expert_pairs(tiles);
        osum += tiles - 2 * route_expert_pairs(tiles);
      }
    }
    int inc = sum, pinc = psum, tinc = tsum, qinc = qsum, oinc = osum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFullMask, inc, off);
      const int po = __shfl_up_sync(kFullMask, pinc, off);
      const int to = __shfl_up_sync(kFullMask, tinc, off);
      const int qo = __shfl_up_sync(kFullMask, qinc, off);
      const int oo = __shfl_up_sync(kFullMask, oinc, off);
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
        sm.off[e] = run;
        sm.rs[e] = prun;
        sm.ts[e] = trun;
        sm.ps[e] = qrun;
        sm.qs[e] = orun;
        const int c = __ldcg(a.counts + e);
        const int tiles = route_row_tiles(c, align);
        run += c;
        prun += route_pad_rows(c, align);
        trun += tiles;
        qrun += route_expert_pairs(tiles);
        orun += tiles - 2 * route_expert_pairs(tiles);
      }
    }
    if (lane == 31) {
      sm.off[E] = inc;
      sm.rs[E] = pinc;
      sm.ts[E] = tinc;
      sm.ps[E] = qinc;
      sm.qs[E] = oinc;
    }
  }
  __syncthreads();
  if (write_global) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      a.offsets[e] = sm.off[e];
      a.row_start[e] = sm.rs[e];
      a.tile_start[e] = sm.ts[e];
      if (a.pair_start) a.pair_start[e] = sm.ps[e];
      if (a.rem_start) a.rem_start[e] = sm.qs[e];
    }
  }
}

// Padding rows of the padded layout of expert e: no token, weight 0.
__device__ __forceinline__ void route_scatter_pad(const ScatterArgs& a, const ScatterSmem& sm, int e) {
  const int beg = sm.rs[e] + __ldcg(a.counts + e), end = sm.rs[e + 1];
  for (int r = beg + threadIdx.x; r < end; r += blockDim.x) {
    a.perm_token_pad[r] = -1;
    a.perm_w_pad[r] = 0.f;
  }
}

// 2-4. The routes of chunk `chunk` (kChunkTokens tokens, kWarpTokens per
//    warp) to their rows: per-warp expert counts, warp bases (chunk base of
//    the expert plus the routes of earlier warps), then stable ranks, 32
//    routes at a time in (token, slot) order.  Needs route_scatter_prefix's
//    offsets in sm; starts and ends with a CTA barrier.
__device__ __forceinline__ void route_scatter_chunk(const ScatterArgs& a, const ScatterSmem& sm, int chunk) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  int* wcnt = sm.wcnt + warp * kMaxExperts;
  __syncthreads();
  for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) sm.wcnt[(i / E) * kMaxExperts + i % E] = 0;
  __syncthreads();
  const int tw0 = chunk * kChunkTokens + warp * kWarpTokens;
  const int ntok = max(0, min(kWarpTokens, a.T - tw0));
  const int nr = ntok * k;
  const int32_t* my_idx = a.topk_idx + static_cast<size_t>(tw0) * k;
  for (int r = lane; r < nr; r += 32) atomicAdd(&wcnt[__ldcg(my_idx + r)], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int base = __ldcg(a.chunk_base + static_cast<size_t>(chunk) * E + e);
    for (int w = 0; w < kChunkWarps; ++w) {
      const int c = sm.wcnt[w * kMaxExperts + e];
      sm.wcnt[w * kMaxExperts + e] = base;
      base += c;
    }
  }
  __syncthreads();
  for (int r0 = 0; r0 < nr; r0 += 32) {
    const int r = r0 + lane;
    const bool valid = r < nr;
    const int e = valid ? __ldcg(my_idx + r) : -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int local = 0;
    if (valid) local = wcnt[e] + rank;
    __syncwarp();
    if (valid && rank == 0) wcnt[e] += __popc(peers);
    __syncwarp();
    if (valid) {
      const int tl = r / k;
      const int t = tw0 + tl;
      const int j = r - tl * k;
      const size_t tj = static_cast<size_t>(t) * k + j;
      const int ru = sm.off[e] + local;
      const int rp = sm.rs[e] + local;
      a.perm_token[ru] = t;
      a.route_row[tj] = ru;
      a.perm_token_pad[rp] = t;
      a.route_row_pad[tj] = rp;
      a.perm_w_pad[rp] = __ldcg(a.topk_w + tj);
    }
  }
  __syncthreads();
}

struct GemmParams;

// The fused persistent routing launch (route_fused.cu).  Supported when the
// router's logits fit one GEMM tile (E <= 256) and top_k <= 16.  p: the router
// GEMM's parameters with the EPI_ROUTE outputs set; chunk_counts and sync
// ([4] ints) must be zero at launch.  Returns the launch's error
// (cudaErrorCooperativeLaunchTooLarge when the grid cannot be resident at
// once).
bool route_fused_supported(int64_t E, int64_t k);
cudaError_t launch_route_fused(const GemmParams& p, const ScatterArgs& sc, int32_t* chunk_counts,
                               int32_t* chunk_base, int nchunk, int* status, int* sync, int extra_arrivals, int grid,
                               cudaStream_t st);

}  // namespace moe
