// Internal declarations shared by the translation units of libmoe.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

struct GemmParams;

// Tokens per routing chunk (one CTA of the top-k and scatter kernels) and per
// warp inside it.
constexpr int kChunkTokens = 64;
constexpr int kChunkWarps = 8;
constexpr int kWarpTokens = kChunkTokens / kChunkWarps;
constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 32;
// Each expert's row group starts at a multiple of kRowAlign rows.  The GEMMs
// cut a group into 128-row tiles plus, when its length is an odd multiple of
// 64, one 64-row tail tile (computed with an M=64 MMA).  The MXFP8 path pads
// groups to kRowAlignMx rows: its weight-gradient GEMMs take K (token rows)
// 128 at a time and its scale blocks cover 128 rows.
constexpr int kRowAlign = 64;
constexpr int kRowAlignMx = 128;
constexpr int kTileRows = 128;

// ---- routing kernels (routing.cu)
cudaError_t launch_topk_count(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* topk_w, int32_t* chunk_counts, int* status, cudaStream_t st);
cudaError_t launch_chunk_scan(const int32_t* chunk_counts, int nchunk, int E, int32_t* chunk_base,
                              int32_t* counts, cudaStream_t st);
cudaError_t launch_scatter(const int32_t* topk_idx, const float* topk_w, int T, int E, int k,
                           int row_align, const int32_t* chunk_base, const int32_t* counts, int32_t* offsets,
                           int32_t* row_start, int32_t* tile_start, int32_t* pair_start, int32_t* rem_start,
                           int32_t* perm_token, int32_t* route_row,
                           int32_t* perm_token_pad, int32_t* route_row_pad, float* perm_w_pad,
                           cudaStream_t st);
// pair_start / rem_start (optional, [E+1]): prefixes, over the experts, of the
// tile pairs that run on SM pairs and of the tiles that run on one SM, tiles =
// an expert's 128-row GEMM tiles: an even count runs as tiles / 2 pairs, an
// odd count entirely on one SM (so that no expert's weights are read by both
// passes).

// ---- memory-bound kernels (elementwise.cu)
cudaError_t launch_combine(const __nv_bfloat16* o, const __nv_bfloat16* ys,
                           const int32_t* route_row_pad, int T, int d, int k, __nv_bfloat16* y,
                           cudaStream_t st);
cudaError_t launch_router_grad(const float* dg_part, int nparts, const int32_t* route_row_pad,
                               const float* topk_w, int T, int k, float* d_topk_w, float* dl_tk,
                               float* dl_row, cudaStream_t st);
// part: scratch of part_floats floats for the per-chunk partial sums, at least
// (ceil(R / 128) + E) * d (R = the routed rows, sum of counts).
cudaError_t launch_router_wgrad(const float* dl_row, const int32_t* perm_token_pad,
                                const int32_t* row_start, const int32_t* counts,
                                const __nv_bfloat16* x, int E, int d, int64_t R, float* part,
                                int64_t part_floats, float* dW_router, cudaStream_t st);
cudaError_t launch_scatter_rows(const __nv_bfloat16* src, const int32_t* route_row_pad, const int32_t* row_start,
                                const int32_t* counts, int T, int E, int d, int k, __nv_bfloat16* dst,
                                cudaStream_t st);
cudaError_t launch_unpermute(const __nv_bfloat16* dxp, const __nv_bfloat16* dxs,
                             const int32_t* route_row_pad, const int32_t* topk_idx,
                             const float* dl_tk, const __nv_bfloat16* W_router, int T, int d,
                             int k, __nv_bfloat16* dx, cudaStream_t st);

// ---- MXFP8 quantization (mxfp8.cu)
cudaError_t launch_mx_rows(const __nv_bfloat16* src, long long src_ld, int64_t R, int K, uint8_t* dst,
                           uint8_t* sf, cudaStream_t st);
cudaError_t launch_mx_permute_dual(const __nv_bfloat16* src, long long src_ld, const int32_t* idx,
                                   const int32_t* total_rows, int64_t R, int K, uint8_t* rq, uint8_t* rq_sf,
                                   uint8_t* tq, uint8_t* tq_sf, cudaStream_t st);
// The dispatch with MXFP8 quantization of the rows of src [T, K] into the
// padded expert-grouped layout of R rows: rq (blocks of 32 along K, zeros in
// padding rows) and, when tq is given, its transpose tq [K, R]
// (launch_mx_permute_dual); without tq, rq alone as a scatter of the token
// rows (each read once).
cudaError_t launch_mx_dispatch(const __nv_bfloat16* src, long long src_ld, int T, int k, int E,
                               const int32_t* perm_token_pad, const int32_t* route_row_pad, const int32_t* row_start,
                               const int32_t* counts, int64_t R, int K, uint8_t* rq, uint8_t* rq_sf, uint8_t* tq,
                               uint8_t* tq_sf, cudaStream_t st);
cudaError_t launch_mx_cols(const __nv_bfloat16* src, long long src_ld, long long src_bstride, int rows,
                           int cols, int batch, uint8_t* dst, long long dst_ld, long long dst_brows,
                           int k_off, uint8_t* sf, long long dst_rows_total, cudaStream_t st);
// Bytes of the scale array of an MXFP8 operand with `rows` rows and K columns.
inline size_t mx_sf_bytes(int64_t rows, int64_t K) {
  return static_cast<size_t>(((rows + 127) / 128) * (K / 128) * 512);
}
// Scale arrays are allocated with one spare 512-byte block: a 256-row B tile
// whose second half lies past the operand's last row still fetches two blocks
// (the columns it feeds are never stored).
inline size_t mx_sf_alloc(int64_t rows, int64_t K) { return mx_sf_bytes(rows, K) + 512; }

// ---- tensor-core GEMM instantiations (gemm_fwd.cu, gemm_bwd.cu)
enum GemmKind : int {
  GK_ROUTER = 0,     // x rows . W_router^T, fp32 + bias
  GK_GATEUP,         // rows . [W_gate; W_up]^T, SwiGLU epilogue
  GK_DOWN,           // rows . W_down^T, bf16 (optionally scaled by the router weight)
  GK_DGRAD_DOWN,     // dy rows . W_down (MN-major), SwiGLU backward epilogue
  GK_DGRAD_GATEUP,   // [da|db] rows . [W_gate; W_up] (MN-major, two stacks along K)
  GK_WGRAD,          // A^T . B over a group's rows (both MN-major): weight gradients
  // MXFP8 block-scaled forms (E4M3 operands):
  GK_MX_GATEUP,       // x rows . [W_gate; W_up]^T, SwiGLU epilogue quantizing h
  GK_MX_DOWN,         // h rows . W_down^T, scaled by the router weight
  GK_MX_DGRAD_DOWN,   // dy rows . W_down (as W_down^T rows), SwiGLU backward quantizing [da|db]
  GK_MX_DGRAD_GATEUP, // [da|db] rows . [W_gate; W_up] (as its transpose's rows)
  GK_MX_WGRAD,        // weight gradients from transposes quantized along the tokens
  GK_COUNT
};
cudaError_t launch_gemm(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st);
// Kernels launched beyond the first by the current launch call on this host
// thread (a launch helper that issues several adds to it; the per-kernel
// timing resets and reads it around each call).
int& extra_kernel_launches();

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace moe
