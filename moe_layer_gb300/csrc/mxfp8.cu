// MXFP8 quantization kernels (E4M3 elements, one E8M0 scale per 32 elements
// along the reduction axis of the GEMM the operand feeds).  The MX rule: the
// block scale is X = 2^(floor(log2(amax)) - 8) (8 = largest E4M3 exponent),
// stored as the biased exponent (bias 127); elements are v / X rounded to the
// nearest E4M3 value with saturation at +-448; an all-zero block gets scale
// code 0.  (Mixture-of-Kittens blog post, section "MXFP8 support": weights are
// pre-quantized, activation quantization is fused into the data movement.)
//
// Scale layout ("tcgen05.cp 32x128b" order): for an operand with R rows and K
// columns, the scales of rows [128 q, 128 q + 128) and columns
// [128 g, 128 g + 128) form one 512-byte block at offset (g * R/128 + q) * 512;
// inside it the byte of row r (0..127) and 32-column block j (0..3) sits at
// 16 * (r % 32) + 4 * (r / 32) + j.  The GEMM copies one such block straight
// into tensor memory per operand tile and stage.
#include <atomic>

#include "moe_internal.h"
#include "mx_common.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

// Row-wise quantization of a [R, K] bf16 matrix (row pitch src_ld), blocks
// of 32 along the row.  One group of four threads per (row, 128-column group).
constexpr int kQThreads = 256;
__global__ void __launch_bounds__(kQThreads)
    mx_rows_kernel(const __nv_bfloat16* __restrict__ src, long long src_ld, int64_t R, int K,
                   uint8_t* __restrict__ dst, uint8_t* __restrict__ sf) {
  const int64_t ng = K / 128;
  const int64_t units = R * ng;
  for (int64_t u = (static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x) / 4; u < units;
       u += static_cast<int64_t>(gridDim.x) * kQThreads / 4) {
    const int64_t r = u / ng, g = u - r * ng;
    const int j = threadIdx.x & 3;
    const int col = static_cast<int>(g * 128 + 32 * j);
    float v[32];
    const uint4* s4 = reinterpret_cast<const uint4*>(src + r * src_ld + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = __ldg(s4 + q);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * q + 2 * i] = bf16lo(ws[i]);
        v[8 * q + 2 * i + 1] = bf16hi(ws[i]);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_scale_exp(amax);
    uint4 lo, hi;
    quant32(v, e, lo, hi);
    uint4* d4 = reinterpret_cast<uint4*>(dst + r * static_cast<int64_t>(K) + col);
    d4[0] = lo;
    d4[1] = hi;
    // the four scale codes of this (row, 128-column group) form one word
    uint32_t code = static_cast<uint32_t>(e + 127) << (8 * j);
    code |= __shfl_xor_sync(0xffffffffu, code, 1);
    code |= __shfl_xor_sync(0xffffffffu, code, 2);
    if (j == 0) *reinterpret_cast<uint32_t*>(sf + sf_word_offset(r, g, (R + 127) / 128)) = code;
  }
}

// The dispatch without the transposed copy (the forward of a call that keeps
// no state) as a scatter: each token row of src [T, K] is quantized once
// along K (blocks of 32, the arithmetic of mx_rows_kernel: one group of four
// threads per (token, 128-column group)) and written to the token's k rows of
// the padded expert-grouped layout (route_row_pad), codes and scale words
// alike; blocks past the tokens' ones write zero codes and zero scale words
// into each expert's padding rows.  The bytes are those of the gathered
// quantization below (a row's blocks do not depend on the expert), but each
// source row is read once instead of k times.  (With the transposed copy to
// write too, the gather serves both copies at once; a scatter beside a
// transposed-only gather measured slower.)
__global__ void __launch_bounds__(kQThreads)
    mx_scatter_rows_kernel(const __nv_bfloat16* __restrict__ src, long long src_ld, int T, int k,
                           const int32_t* __restrict__ route_row_pad, const int32_t* __restrict__ row_start,
                           const int32_t* __restrict__ counts, int64_t R, int K, int token_blocks,
                           uint8_t* __restrict__ rq, uint8_t* __restrict__ rq_sf) {
  const int64_t ng = K / 128;
  const int64_t rblocks = (R + 127) / 128;
  const int j = threadIdx.x & 3;
  if (static_cast<int>(blockIdx.x) >= token_blocks) {  // padding rows of expert blockIdx.x - token_blocks
    const int e = static_cast<int>(blockIdx.x) - token_blocks;
    const int64_t beg = __ldg(row_start + e) + __ldg(counts + e), end = __ldg(row_start + e + 1);
    const int64_t units = (end - beg) * ng;
    for (int64_t u = threadIdx.x / 4; u < units; u += kQThreads / 4) {
      const int64_t r = beg + u / ng, g = u % ng;
      uint4* d4 = reinterpret_cast<uint4*>(rq + r * static_cast<int64_t>(K) + g * 128 + 32 * j);
      d4[0] = make_uint4(0, 0, 0, 0);
      d4[1] = make_uint4(0, 0, 0, 0);
      if (j == 0) *reinterpret_cast<uint32_t*>(rq_sf + sf_word_offset(r, g, rblocks)) = 0u;
    }
    return;
  }
  const int64_t units = static_cast<int64_t>(T) * ng;
  for (int64_t u = (static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x) / 4; u < units;
       u += static_cast<int64_t>(token_blocks) * kQThreads / 4) {
    const int64_t t = u / ng, g = u - t * ng;
    const int col = static_cast<int>(g * 128 + 32 * j);
    float v[32];
    const uint4* s4 = reinterpret_cast<const uint4*>(src + t * src_ld + col);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = __ldg(s4 + q);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * q + 2 * i] = bf16lo(ws[i]);
        v[8 * q + 2 * i + 1] = bf16hi(ws[i]);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_scale_exp(amax);
    uint4 lo, hi;
    quant32(v, e, lo, hi);
    // the quad's four codes form one word (a quad is active or not as a whole;
    // the last pass of the loop may leave other quads of the warp out)
    const unsigned quad = 0xfu << (threadIdx.x & 28);
    uint32_t code = static_cast<uint32_t>(e + 127) << (8 * j);
    code |= __shfl_xor_sync(quad, code, 1);
    code |= __shfl_xor_sync(quad, code, 2);
    for (int s = 0; s < k; ++s) {
      const int64_t r = __ldg(route_row_pad + t * k + s);
      uint4* d4 = reinterpret_cast<uint4*>(rq + r * static_cast<int64_t>(K) + col);
      d4[0] = lo;
      d4[1] = hi;
      if (j == 0) *reinterpret_cast<uint32_t*>(rq_sf + sf_word_offset(r, g, rblocks)) = code;
    }
  }
}

// Dispatch with quantization: dst row r is src row idx[r] (a zero row for a
// negative index); rows from *total_rows on are left alone.  Writes up to two
// MXFP8 copies of the gathered [R, K] matrix:
//   rq  [R, K], blocks of 32 columns (operand of the GEMMs that reduce over K);
//   tq  [K, R], the transpose, blocks of 32 consecutive rows of the gathered
//       matrix (operand of the weight gradients, whose reduction axis is the
//       rows; groups start on 128-row boundaries, so a block never mixes
//       experts); skipped when tq is null.
// Block: one 128 x 128 tile (R and K multiples of 128), 256 threads; the bf16
// tile sits in shared memory so that both quantizations read it along their
// own axis, both without bank conflicts: the row quantization gives the eight
// threads of a quarter warp eight different rows (the 272-byte row pitch puts
// them in different banks), the transposed one reads two adjacent columns per
// 32-bit load.  Each thread's 32 output bytes of a block go out as one
// 256-bit store (a whole 32-byte sector; rq, tq 32-byte aligned).
constexpr int kDualTile = 128;
constexpr int kDualPitch = kDualTile + 8;  // bf16 elements per shared row (16-byte aligned rows)
constexpr int kDualBlocksPerSm = 3;

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Quantizes one column of 32 rows held two columns per word (hi: the upper
// bf16 of each word) with scale 2^e into 32 E4M3 bytes.
__device__ __forceinline__ void quant32_col(const uint32_t* w, bool hi, int e, uint4& q0, uint4& q1) {
  const float inv = mx_inv_scale(e);
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = (hi ? bf16hi(w[4 * i + j]) : bf16lo(w[4 * i + j])) * inv;
    o[i] = e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16);
  }
  q0 = make_uint4(o[0], o[1], o[2], o[3]);
  q1 = make_uint4(o[4], o[5], o[6], o[7]);
}

// Persistent: each block walks tiles blockIdx.x, + gridDim.x, ...; the gather
// of the next tile is in flight (cp.async, double-buffered) while the current
// one is quantized, and the source row indices of the tile after it are
// loaded meanwhile.
__global__ void __launch_bounds__(kQThreads, kDualBlocksPerSm)
    mx_permute_dual_kernel(const __nv_bfloat16* __restrict__ src, long long src_ld,
                           const int32_t* __restrict__ idx, const int32_t* __restrict__ total_rows,
                           int64_t R, int K, uint8_t* __restrict__ rq, uint8_t* __restrict__ rq_sf,
                           uint8_t* __restrict__ tq, uint8_t* __restrict__ tq_sf) {
  extern __shared__ __align__(16) uint8_t dual_smem[];
  typedef uint16_t Tile[kDualTile][kDualPitch];
  Tile* tiles = reinterpret_cast<Tile*>(dual_smem);  // two buffers
  // E8M0 words of the tile, double-buffered: [buf][0] per row (4 column
  // blocks), [buf][1] per column (4 row blocks)
  typedef uint32_t ScaleWords[2][kDualTile];
  ScaleWords* sfw = reinterpret_cast<ScaleWords*>(dual_smem + 2 * sizeof(Tile));
  const int ncol = K / kDualTile;
  const int64_t used = total_rows ? static_cast<int64_t>(__ldg(total_rows)) : R;
  const int64_t ntiles = ((used + kDualTile - 1) / kDualTile) * ncol;  // only row tiles that hold used rows
  // gather: thread -> rows (tid / 16) + 16 k, 16 bytes at column 8 (tid % 16)
  const int grow = threadIdx.x >> 4, gq = threadIdx.x & 15;
  auto load_rows = [&](int64_t tau, int32_t (&ix)[8]) {
    const int64_t r0 = (tau / ncol) * kDualTile;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ix[k] = idx ? __ldg(idx + r0 + grow + 16 * k) : static_cast<int32_t>(r0 + grow + 16 * k);
  };
  auto gather = [&](int64_t tau, const int32_t (&ix)[8], Tile& t) {
    const int c0 = static_cast<int>(tau % ncol) * kDualTile;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t srow = ix[k];
      const __nv_bfloat16* g = src + (srow >= 0 ? srow : 0) * src_ld + c0 + 8 * gq;
      cp_async16(&t[grow + 16 * k][8 * gq], g, srow >= 0 ? 16 : 0);
    }
    cp_async_commit();
  };
  int32_t ix[8];
  int buf = 0;
  if (static_cast<int64_t>(blockIdx.x) < ntiles) {
    load_rows(blockIdx.x, ix);
    gather(blockIdx.x, ix, tiles[0]);
    if (static_cast<int64_t>(blockIdx.x) + gridDim.x < ntiles) load_rows(blockIdx.x + gridDim.x, ix);
  }
  for (int64_t tau = blockIdx.x; tau < ntiles; tau += gridDim.x) {
    const int64_t next = tau + gridDim.x;
    if (next < ntiles) {
      gather(next, ix, tiles[buf ^ 1]);
      if (next + gridDim.x < ntiles) load_rows(next + gridDim.x, ix);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile `buf` is in shared memory
    const Tile& tile = tiles[buf];
    const int64_t r0 = (tau / ncol) * kDualTile;
    const int c0 = static_cast<int>(tau % ncol) * kDualTile;
    {  // along the row: thread -> (row, 64-column half), two blocks of 32
      const int r = (threadIdx.x & 7) + 8 * (threadIdx.x >> 4), half = (threadIdx.x >> 3) & 1;
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        float v[32], amax = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(&tile[r][64 * half + 32 * b + 8 * q]);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * q + 2 * k] = bf16lo(ws[k]);
            v[8 * q + 2 * k + 1] = bf16hi(ws[k]);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const int e = mx_scale_exp(amax);
        uint4 lo, hi;
        quant32(v, e, lo, hi);
        st_global_v8(rq + (r0 + r) * K + c0 + 64 * half + 32 * b, lo, hi);
        word |= static_cast<uint32_t>(e + 127) << (8 * (2 * half + b));
      }
      word |= __shfl_xor_sync(0xffffffffu, word, 8);  // the row's other half
      if (half == 0) sfw[buf][0][r] = word;
    }
    if (tq) {  // along the rows: thread -> (column pair, 32-row block)
      const int cp = threadIdx.x & 63, tb = threadIdx.x >> 6;
      uint32_t w[32];
      __nv_bfloat162 m2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        w[i] = *reinterpret_cast<const uint32_t*>(&tile[32 * tb + i][2 * cp]);
        m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[i])));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = mx_scale_exp(h ? __high2float(m2) : __low2float(m2));
        uint4 q0, q1;
        quant32_col(w, h != 0, e, q0, q1);
        st_global_v8(tq + static_cast<int64_t>(c0 + 2 * cp + h) * R + r0 + 32 * tb, q0, q1);
        reinterpret_cast<uint8_t*>(sfw[buf][1])[4 * (2 * cp + h) + tb] = static_cast<uint8_t>(e + 127);
      }
    }
    __syncthreads();  // scale words complete; tile `buf` no longer read
    // Each tile's scales are one whole 512-byte block per copy: bytes 16 t .. 16 t + 15
    // hold the words of rows (columns) t, t + 32, t + 64, t + 96.  The next
    // iteration writes the other scale buffer, and the one after that passes
    // the next iteration's second barrier first.
    if (threadIdx.x < 32) {
      const int t = threadIdx.x;
      const uint32_t* sw = sfw[buf][0];
      uint8_t* blk = rq_sf + ((c0 / 128) * ((R + 127) / 128) + r0 / 128) * 512;
      *reinterpret_cast<uint4*>(blk + 16 * t) = make_uint4(sw[t], sw[t + 32], sw[t + 64], sw[t + 96]);
    } else if (tq && threadIdx.x < 64) {
      const int t = threadIdx.x - 32;
      const uint32_t* sw = sfw[buf][1];
      uint8_t* blk = tq_sf + ((r0 / 128) * (K / 128) + c0 / 128) * 512;
      *reinterpret_cast<uint4*>(blk + 16 * t) = make_uint4(sw[t], sw[t + 32], sw[t + 64], sw[t + 96]);
    }
    buf ^= 1;
  }
}
constexpr int kDualSmemBytes = 2 * kDualTile * kDualPitch * 2 + 2 * 2 * kDualTile * 4;

// Transposing quantization: src is [rows, cols] (row pitch src_ld) and feeds
// a GEMM whose reduction axis is `rows`.  Writes dst[c, k_off + r] (row pitch
// dst_ld, K-major for the GEMM) with blocks of 32 along r.  blockIdx.z walks a
// batch of such matrices (per expert): src += z * src_bstride, dst row offset
// += z * dst_brows.  Tile: 128 rows x 64 columns per block.
__global__ void __launch_bounds__(kQThreads)
    mx_cols_kernel(const __nv_bfloat16* __restrict__ src, long long src_ld, long long src_bstride, int rows,
                   int cols, uint8_t* __restrict__ dst, long long dst_ld, long long dst_brows, int k_off,
                   uint8_t* __restrict__ sf, long long dst_rows_total) {
  __shared__ float tile[128][65];
  const int r0 = blockIdx.y * 128, c0 = blockIdx.x * 64;
  const __nv_bfloat16* s = src + static_cast<long long>(blockIdx.z) * src_bstride;
  // coalesced load: each warp reads rows, 64 columns = 128 bytes per row
  for (int i = threadIdx.x; i < 128 * 32; i += kQThreads) {
    const int r = i / 32, cp = (i % 32) * 2;
    float a = 0.f, b = 0.f;
    if (r0 + r < rows && c0 + cp < cols) {
      const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(s + static_cast<long long>(r0 + r) * src_ld + c0 + cp));
      a = bf16lo(w);
      b = bf16hi(w);
    }
    tile[r][cp] = a;
    tile[r][cp + 1] = b;
  }
  __syncthreads();
  const int c = threadIdx.x >> 2, j = threadIdx.x & 3;
  float v[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = tile[32 * j + i][c];
    amax = fmaxf(amax, fabsf(v[i]));
  }
  const int e = mx_scale_exp(amax);
  uint4 lo, hi;
  quant32(v, e, lo, hi);
  if (c0 + c < cols) {
    const long long drow = static_cast<long long>(blockIdx.z) * dst_brows + c0 + c;
    uint4* d4 = reinterpret_cast<uint4*>(dst + drow * dst_ld + k_off + r0 + 32 * j);
    d4[0] = lo;
    d4[1] = hi;
  }
  uint32_t code = static_cast<uint32_t>(e + 127) << (8 * j);
  code |= __shfl_xor_sync(0xffffffffu, code, 1);
  code |= __shfl_xor_sync(0xffffffffu, code, 2);
  if (j == 0 && c0 + c < cols) {
    const long long drow = static_cast<long long>(blockIdx.z) * dst_brows + c0 + c;
    *reinterpret_cast<uint32_t*>(sf + sf_word_offset(drow, (k_off + r0) / 128, dst_rows_total / 128)) = code;
  }
}

}  // namespace

cudaError_t launch_mx_rows(const __nv_bfloat16* src, long long src_ld, int64_t R, int K, uint8_t* dst,
                           uint8_t* sf, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  const int64_t units = R * (K / 128);
  int64_t blocks = (units * 4 + kQThreads - 1) / kQThreads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  mx_rows_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, st>>>(src, src_ld, R, K, dst, sf);
  return cudaGetLastError();
}

cudaError_t launch_mx_permute_dual(const __nv_bfloat16* src, long long src_ld, const int32_t* idx,
                                   const int32_t* total_rows, int64_t R, int K, uint8_t* rq, uint8_t* rq_sf,
                                   uint8_t* tq, uint8_t* tq_sf, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  if (K % kDualTile || R % kDualTile) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit == 0 || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(mx_permute_dual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDualSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const int64_t tiles = (R / kDualTile) * (K / kDualTile);
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * kDualBlocksPerSm;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  mx_permute_dual_kernel<<<grid, kQThreads, kDualSmemBytes, st>>>(src, src_ld, idx, total_rows, R, K, rq, rq_sf,
                                                                 tq, tq_sf);
  return cudaGetLastError();
}

cudaError_t launch_mx_dispatch(const __nv_bfloat16* src, long long src_ld, int T, int k, int E,
                               const int32_t* perm_token_pad, const int32_t* route_row_pad, const int32_t* row_start,
                               const int32_t* counts, int64_t R, int K, uint8_t* rq, uint8_t* rq_sf, uint8_t* tq,
                               uint8_t* tq_sf, cudaStream_t st) {
  if (tq) return launch_mx_permute_dual(src, src_ld, perm_token_pad, row_start + E, R, K, rq, rq_sf, tq, tq_sf, st);
  if (R <= 0) return cudaSuccess;
  if (K % kDualTile || R % kDualTile) return cudaErrorInvalidValue;
  const int64_t ng = K / 128;
  const int64_t want = (static_cast<int64_t>(T) * ng * 4 + kQThreads - 1) / kQThreads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  const int token_blocks = static_cast<int>(want < cap ? want : cap);
  if (token_blocks + E <= 0) return cudaSuccess;
  mx_scatter_rows_kernel<<<token_blocks + E, kQThreads, 0, st>>>(src, src_ld, T, k, route_row_pad, row_start, counts,
                                                                 R, K, token_blocks, rq, rq_sf);
  return cudaGetLastError();
}

cudaError_t launch_mx_cols(const __nv_bfloat16* src, long long src_ld, long long src_bstride, int rows,
                           int cols, int batch, uint8_t* dst, long long dst_ld, long long dst_brows,
                           int k_off, uint8_t* sf, long long dst_rows_total, cudaStream_t st) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
  dim3 grid((cols + 63) / 64, (rows + 127) / 128, batch);
  mx_cols_kernel<<<grid, kQThreads, 0, st>>>(src, src_ld, src_bstride, rows, cols, dst, dst_ld, dst_brows,
                                             k_off, sf, dst_rows_total);
  return cudaGetLastError();
}

}  // namespace moe
