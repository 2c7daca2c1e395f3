// Memory-bound kernels of the layer.  Each sums in one fixed order with no
// floating-point atomics, so results are bitwise reproducible (Mixture-of-
// Kittens blog post, section "Determinism"):
//   combine        y_t = y_shared,t + sum_j o[row(t, j)]          (weighted sum;
//                  the router weight is already applied by the down GEMM)
//   router_grad    dg_tj = sum of the per-n-tile partials of <h, dh>, then the
//                  softmax backward dl_tj = g_tj (dg_tj - sum_i g_ti dg_ti)
//   router_wgrad   dW_router[e] = sum over e's rows of dl_row x_token: in chunks
//                  of rows (ascending), the chunks' sums added in order
//   unpermute      dx_t = dx_shared,t + sum_j dxp[row(t, j)] + sum_j dl_tj W_router[e_tj]
//   scatter_rows   copies each token row to its k rows of the expert-grouped
//                  row order (the "dispatch" of the pages, local to one GPU)
#include <algorithm>
#include <climits>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 a;
  a.x = pack_bf16x2(v[0], v[1]);
  a.y = pack_bf16x2(v[2], v[3]);
  a.z = pack_bf16x2(v[4], v[5]);
  a.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = a;
}

constexpr int kEwThreads = 128;

__global__ void __launch_bounds__(kEwThreads)
    combine_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ ys,
                   const int32_t* __restrict__ route_row_pad, int d, int k,
                   __nv_bfloat16* __restrict__ y) {
  __shared__ long long rows[kMaxTopK];
  const int t = blockIdx.x;
  if (threadIdx.x < k)
    rows[threadIdx.x] = static_cast<long long>(__ldg(route_row_pad + static_cast<size_t>(t) * k + threadIdx.x)) * d;
  __syncthreads();
  const int nv = d / 8;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float acc[8];
    if (ys) {
      ld8(ys + static_cast<size_t>(t) * d + 8 * v, acc);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    }
    for (int j = 0; j < k; ++j) {
      float u[8];
      ld8(o + rows[j] + 8 * v, u);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += u[i];
    }
    st8(y + static_cast<size_t>(t) * d + 8 * v, acc);
  }
}

// one warp per token, lane j owns slot j
__global__ void __launch_bounds__(256)
    router_grad_kernel(const float* __restrict__ dg_part, int nparts,
                       const int32_t* __restrict__ route_row_pad, const float* __restrict__ topk_w,
                       int T, int k, float* __restrict__ d_topk_w, float* __restrict__ dl_tk,
                       float* __restrict__ dl_row) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float dg = 0.f, g = 0.f;
  int row = 0;
  if (lane < k) {
    const size_t tj = static_cast<size_t>(t) * k + lane;
    row = __ldg(route_row_pad + tj);
    g = __ldg(topk_w + tj);
    const float* pp = dg_part + static_cast<size_t>(row) * nparts;
    for (int p = 0; p < nparts; ++p) dg += __ldg(pp + p);
  }
  float s = g * dg;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane < k) {
    const size_t tj = static_cast<size_t>(t) * k + lane;
    const float dl = g * (dg - s);
    if (d_topk_w) d_topk_w[tj] = dg;
    dl_tk[tj] = dl;
    dl_row[row] = dl;
  }
}

// dW_router[e, :] = sum over the rows routed to e of dlogit(row) * x[token(row), :]: only the
// chosen logits carry a gradient, so the product is a gather over each expert's rows.  Each
// expert's rows are cut into chunks of `chunk` rows (sized so that the chunks about fill the
// resident blocks, and no fewer than one per expert at a quarter above the average), so that an
// expert routed several times the average (skewed routing) is spread over several blocks.  router_wgrad_part_kernel sums one chunk per block (rows
// ascending): the further chunks of the experts that have them (grid z = 0, in expert order;
// dispatched first, so that they run beside the first chunks) and the first chunk of every
// expert (z = 1, block x = the expert).  The sum of an expert's only chunk goes to dW_router,
// the others to fp32 partials (slot e for the first chunk, E + j for further chunk j);
// router_wgrad_sum_kernel adds those experts' partials in chunk order and zeroes the experts
// without rows.  Each thread owns eight adjacent columns (one 16-byte load per row), four
// gathers in flight.
constexpr int kRwThreads = 128;
constexpr int kRwCols = 8 * kRwThreads;

__device__ __forceinline__ int rw_chunks(const int32_t* __restrict__ counts, int e, int chunk) {
  return (__ldg(counts + e) + chunk - 1) / chunk;
}

// s_pre[e] = number of further chunks (past the first) of the experts before e, e = 0..E
// (E <= kMaxExperts = 4 per thread).  Called by every thread of the block.
__device__ __forceinline__ void rw_extra_prefix(const int32_t* __restrict__ counts, int E, int chunk, int* s_pre,
                                                int* s_warp) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  int c[4], sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * t + j;
    c[j] = e < E ? max(0, rw_chunks(counts, e, chunk) - 1) : 0;
    sum += c[j];
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < w; ++i) base += s_warp[i];
  int ex = base + incl - sum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (4 * t + j < E) s_pre[4 * t + j] = ex;
    ex += c[j];
  }
  if (t == kRwThreads - 1) s_pre[E] = ex;  // the total: experts past E have none
  __syncthreads();
}

// grid (max(E, bound on the further chunks), ceil(d / kRwCols), 2).  Twelve blocks per SM (at
// most 42 registers a thread): one block per expert and column block, 256 x 7 of them, are all
// resident at once.
__global__ void __launch_bounds__(kRwThreads, 12)
    router_wgrad_part_kernel(const float* __restrict__ dl_row, const int32_t* __restrict__ perm_token_pad,
                             const int32_t* __restrict__ row_start, const int32_t* __restrict__ counts,
                             const __nv_bfloat16* __restrict__ x, int E, int d, int chunk,
                             float* __restrict__ part, float* __restrict__ dW) {
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ int s_warp[kRwThreads / 32];
  __shared__ int s_tok[kRwThreads];
  __shared__ float s_dl[kRwThreads];
  int e, q, slot;  // expert, its chunk, the partial slot
  if (blockIdx.z == 1) {
    e = blockIdx.x;
    if (e >= E || __ldg(counts + e) == 0) return;
    q = 0;
    slot = e;
  } else {
    rw_extra_prefix(counts, E, chunk, s_pre, s_warp);
    const int j = blockIdx.x;
    if (j >= s_pre[E]) return;
    int lo = 0, hi = E - 1;  // the expert of this chunk: the last e with s_pre[e] <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= j)
        lo = mid;
      else
        hi = mid - 1;
    }
    e = lo;
    q = 1 + j - s_pre[e];
    slot = E + j;
  }
  const int first = q * chunk;
  const int r0 = __ldg(row_start + e) + first;
  const int n = min(chunk, __ldg(counts + e) - first);
  const int c = blockIdx.y * kRwCols + threadIdx.x * 8;
  const __nv_bfloat16* xc = x + c;
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = 0.f;
  for (int base = 0; base < n; base += kRwThreads) {
    const int m = min(kRwThreads, n - base);
    __syncthreads();
    if (threadIdx.x < m) {
      s_tok[threadIdx.x] = __ldg(perm_token_pad + r0 + base + threadIdx.x);
      s_dl[threadIdx.x] = __ldg(dl_row + r0 + base + threadIdx.x);
    }
    __syncthreads();
    if (c < d) {
      int i = 0;
      for (; i + 4 <= m; i += 4) {  // four rows' loads issued before any is used
        uint4 raw[4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          raw[k4] = __ldg(reinterpret_cast<const uint4*>(xc + static_cast<size_t>(s_tok[i + k4]) * d));
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const float g = s_dl[i + k4];
          const uint32_t w[4] = {raw[k4].x, raw[k4].y, raw[k4].z, raw[k4].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            a[2 * j] += g * bf16lo(w[j]);
            a[2 * j + 1] += g * bf16hi(w[j]);
          }
        }
      }
      for (; i < m; ++i) {
        float u[8];
        ld8(xc + static_cast<size_t>(s_tok[i]) * d, u);
        const float g = s_dl[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] += g * u[j];
      }
    }
  }
  if (c < d) {
    const bool only = blockIdx.z == 1 && __ldg(counts + e) <= chunk;
    float* o = only ? dW + static_cast<size_t>(e) * d : part + static_cast<size_t>(slot) * d;
    float4* out = reinterpret_cast<float4*>(o + c);
    out[0] = make_float4(a[0], a[1], a[2], a[3]);
    out[1] = make_float4(a[4], a[5], a[6], a[7]);
  }
}

// grid (E, ceil(d / kRwCols)): dW_router[e] = the sum of e's chunk partials in chunk order for an
// expert with several chunks, zero for one without rows (router_wgrad_part_kernel wrote the
// others).
__global__ void __launch_bounds__(kRwThreads)
    router_wgrad_sum_kernel(const int32_t* __restrict__ counts, const float* __restrict__ part, int E, int d,
                            int chunk, float* __restrict__ dW) {
  __shared__ int s_pre[kMaxExperts + 1];
  __shared__ int s_warp[kRwThreads / 32];
  const int e = blockIdx.x;
  const int nch = rw_chunks(counts, e, chunk);
  if (nch == 1) return;
  const int c = blockIdx.y * kRwCols + threadIdx.x * 8;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  if (nch > 1) {
    rw_extra_prefix(counts, E, chunk, s_pre, s_warp);
    if (c >= d) return;
    const float4* p = reinterpret_cast<const float4*>(part + static_cast<size_t>(e) * d + c);
    a0 = __ldg(p);
    a1 = __ldg(p + 1);
#pragma unroll 4
    for (int j = s_pre[e]; j < s_pre[e + 1]; ++j) {
      p = reinterpret_cast<const float4*>(part + static_cast<size_t>(E + j) * d + c);
      const float4 u0 = __ldg(p), u1 = __ldg(p + 1);
      a0.x += u0.x; a0.y += u0.y; a0.z += u0.z; a0.w += u0.w;
      a1.x += u1.x; a1.y += u1.y; a1.z += u1.z; a1.w += u1.w;
    }
  }
  if (c >= d) return;
  float4* out = reinterpret_cast<float4*>(dW + static_cast<size_t>(e) * d + c);
  out[0] = a0;
  out[1] = a1;
}

__global__ void __launch_bounds__(kEwThreads)
    unpermute_kernel(const __nv_bfloat16* __restrict__ dxp, const __nv_bfloat16* __restrict__ dxs,
                     const int32_t* __restrict__ route_row_pad, const int32_t* __restrict__ topk_idx,
                     const float* __restrict__ dl_tk, const __nv_bfloat16* __restrict__ Wr, int d,
                     int k, __nv_bfloat16* __restrict__ dx) {
  __shared__ long long rows[kMaxTopK];
  __shared__ long long erows[kMaxTopK];
  __shared__ float dls[kMaxTopK];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const size_t tj = static_cast<size_t>(t) * k + threadIdx.x;
    rows[threadIdx.x] = static_cast<long long>(__ldg(route_row_pad + tj)) * d;
    erows[threadIdx.x] = static_cast<long long>(__ldg(topk_idx + tj)) * d;
    dls[threadIdx.x] = __ldg(dl_tk + tj);
  }
  __syncthreads();
  const int nv = d / 8;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    float acc[8];
    if (dxs) {
      ld8(dxs + static_cast<size_t>(t) * d + 8 * v, acc);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    }
    for (int j = 0; j < k; ++j) {
      float u[8];
      ld8(dxp + rows[j] + 8 * v, u);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += u[i];
    }
    for (int j = 0; j < k; ++j) {
      float u[8];
      ld8(Wr + erows[j] + 8 * v, u);
      const float s = dls[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += s * u[i];
    }
    st8(dx + static_cast<size_t>(t) * d + 8 * v, acc);
  }
}

// The dispatch as a scatter: block t < T reads token t's row once and writes
// it to its k rows of the padded expert-grouped layout (route_row_pad);
// block T + e writes zeros into expert e's padding rows.  Every row of the
// layout is written once, as by a gather over the rows, but each source row
// is read once instead of k times (the source, larger than L2 at full size,
// would otherwise come from DRAM k times).
constexpr int kScatterChunks = 4;  // 16-byte chunks per thread in flight
__global__ void __launch_bounds__(kEwThreads)
    scatter_rows_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ route_row_pad,
                        const int32_t* __restrict__ row_start, const int32_t* __restrict__ counts, int T, int d,
                        int k, __nv_bfloat16* __restrict__ dst) {
  __shared__ int s_rows[kMaxTopK];
  const int b = blockIdx.x;
  const int nv = d / 8;
  if (b >= T) {  // padding rows of expert b - T
    const int e = b - T;
    const int beg = __ldg(row_start + e) + __ldg(counts + e), end = __ldg(row_start + e + 1);
    for (int r = beg; r < end; ++r) {
      uint4* o = reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * d);
      for (int v = threadIdx.x; v < nv; v += blockDim.x) o[v] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  if (threadIdx.x < k) s_rows[threadIdx.x] = __ldg(route_row_pad + static_cast<size_t>(b) * k + threadIdx.x);
  __syncthreads();
  const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<size_t>(b) * d);
  for (int v0 = threadIdx.x; v0 < nv; v0 += kScatterChunks * kEwThreads) {
    uint4 a[kScatterChunks];
#pragma unroll
    for (int i = 0; i < kScatterChunks; ++i) {
      const int v = v0 + i * kEwThreads;
      if (v < nv) a[i] = __ldg(s + v);
    }
    for (int j = 0; j < k; ++j) {
      uint4* o = reinterpret_cast<uint4*>(dst + static_cast<size_t>(s_rows[j]) * d);
#pragma unroll
      for (int i = 0; i < kScatterChunks; ++i) {
        const int v = v0 + i * kEwThreads;
        if (v < nv) o[v] = a[i];
      }
    }
  }
}

}  // namespace

cudaError_t launch_scatter_rows(const __nv_bfloat16* src, const int32_t* route_row_pad, const int32_t* row_start,
                                const int32_t* counts, int T, int E, int d, int k, __nv_bfloat16* dst,
                                cudaStream_t st) {
  if (T + E <= 0) return cudaSuccess;
  scatter_rows_kernel<<<T + E, kEwThreads, 0, st>>>(src, route_row_pad, row_start, counts, T, d, k, dst);
  return cudaGetLastError();
}

cudaError_t launch_combine(const __nv_bfloat16* o, const __nv_bfloat16* ys,
                           const int32_t* route_row_pad, int T, int d, int k, __nv_bfloat16* y,
                           cudaStream_t st) {
  combine_kernel<<<T, kEwThreads, 0, st>>>(o, ys, route_row_pad, d, k, y);
  return cudaGetLastError();
}

cudaError_t launch_router_grad(const float* dg_part, int nparts, const int32_t* route_row_pad,
                               const float* topk_w, int T, int k, float* d_topk_w, float* dl_tk,
                               float* dl_row, cudaStream_t st) {
  router_grad_kernel<<<(T + 7) / 8, 256, 0, st>>>(dg_part, nparts, route_row_pad, topk_w, T, k,
                                                 d_topk_w, dl_tk, dl_row);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const float* dl_row, const int32_t* perm_token_pad,
                                const int32_t* row_start, const int32_t* counts,
                                const __nv_bfloat16* x, int E, int d, int64_t R, float* part,
                                int64_t part_floats, float* dW_router, cudaStream_t st) {
  const int ncb = (d + kRwCols - 1) / kRwCols;
  // chunk: about one chunk per resident block (12 per SM) or per expert, whichever is more, with
  // a quarter of slack so that experts near the average stay whole; 128-row steps, at least 128
  const int64_t target = std::max<int64_t>(E, int64_t(device_sm_count()) * 12 / ncb);
  const int64_t want = (R + R / 4 + target - 1) / target;
  const int64_t chunk = std::max<int64_t>(128, (want + 127) / 128 * 128);
  if (chunk > INT_MAX) return cudaErrorInvalidValue;
  // further chunks (past each expert's first): at most sum_e counts[e] / chunk = R / chunk
  const int64_t extra = (R + chunk - 1) / chunk;
  if ((E + extra) * d > part_floats || extra > INT_MAX) return cudaErrorInvalidValue;
  const unsigned gx = static_cast<unsigned>(std::max<int64_t>(E, extra));
  router_wgrad_part_kernel<<<dim3(gx, ncb, 2), kRwThreads, 0, st>>>(
      dl_row, perm_token_pad, row_start, counts, x, E, d, static_cast<int>(chunk), part, dW_router);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  ++extra_kernel_launches();
  router_wgrad_sum_kernel<<<dim3(E, ncb), kRwThreads, 0, st>>>(counts, part, E, d, static_cast<int>(chunk),
                                                                dW_router);
  return cudaGetLastError();
}

cudaError_t launch_unpermute(const __nv_bfloat16* dxp, const __nv_bfloat16* dxs,
                             const int32_t* route_row_pad, const int32_t* topk_idx,
                             const float* dl_tk, const __nv_bfloat16* W_router, int T, int d,
                             int k, __nv_bfloat16* dx, cudaStream_t st) {
  unpermute_kernel<<<T, kEwThreads, 0, st>>>(dxp, dxs, route_row_pad, topk_idx, dl_tk, W_router, d,
                                             k, dx);
  return cudaGetLastError();
}

}  // namespace moe
