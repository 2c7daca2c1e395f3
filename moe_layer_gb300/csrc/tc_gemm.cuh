// Persistent warp-specialised GEMM on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA with the 128-byte
// swizzle).  One template serves every contraction of the MoE layer:
//
//   * the router projection (dense rows, fp32 + bias epilogue);
//   * the expert-grouped gate/up projection with the SwiGLU epilogue, over
//     token rows already permuted into expert order;
//   * the expert-grouped down projection scaled by the router weight;
//   * the backward dgrads (down with the fused SwiGLU backward and router
//     weight-gradient partials; gate/up with two weight stacks along K);
//   * the weight gradients, whose reduction axis is an expert's (ragged) row
//     range.
//
// The MoE computation these serve is the DeepSeek-V3-style layer described in
// "Mixture-of-Kittens: MoE Megakernel for NVL72s" (blog post, section
// "Overlapping computation and communication in MoE"; paper section 2.1).
//
// Two number formats:
//   bf16   kind::f16 MMAs, K = 64 per pipeline stage, operands K-major or
//          MN-major: 128x256x16 on one SM (router projection; the experts
//          with an odd number of row tiles; weight gradients of experts with
//          few rows), or 256x256x16 on a pair of SMs (SCHED_ROWS2 /
//          SCHED_WGRAD2, cta_group::2: each SM holds its 128 rows of A and
//          half of B) for the other bf16 GEMM tiles;
//   MXFP8  (MX = true; blog section "MXFP8 support") kind::mxf8f6f4 block-scaled
//          MMAs (128x256x32) on E4M3 operands, both K-major, K = 128 per stage.
//          Each stage also brings the E8M0 scales of its A and B tiles (one
//          512-byte tcgen05.cp block per 128 rows); the MMA thread copies them
//          into a ring of TMEM columns next to the accumulator before issuing
//          the stage's four MMAs.
//
// Roles per CTA (one CTA per SM, persistent over tiles; 256 threads; in the
// 2-SM modes clusters of two CTAs):
//   warp 0      TMA producer (lane 0 issues the tile loads)
//   warp 1      MMA issuer (lane 0; in a pair, the even CTA's only)
//   warp 2      TMEM allocator (512 columns)
//   warps 4..7  epilogue: TMEM -> registers -> fused math -> swizzled smem
//               staging -> TMA bulk stores (or direct stores)
// The MXFP8 SwiGLU backward and SCHED_WGRAD_WIDE run 320 threads with
// epilogue warps 2..9, two per TMEM lane quadrant (see epi_wide).
// Pipelines: smem stages (full/empty mbarriers) and accumulator buffers
// (acc_full/acc_empty): two 256-column buffers in bf16 mode so the epilogue of
// tile i overlaps the MMAs of tile i+1; one in MXFP8 mode, whose other TMEM
// columns hold the scale ring and a stash for the epilogue.  In a pair, the
// even CTA's full barriers count both CTAs' loads, its MMA commits free the
// stage and fill the accumulator in both CTAs, and both CTAs' epilogues
// release the accumulator on the even CTA's barrier.  Every wait is bounded
// (see mbar_wait): a stuck pipeline records MOE_ERR_DEVICE_TIMEOUT in the
// status word and the CTA exits cleanly.
#pragma once
#include "mx_common.cuh"
#include "ptx.cuh"
#include "routing_dev.cuh"

namespace moe {

enum AMode : int { A_K_TILE = 0, A_MN_TILE = 1 };
enum BMode : int { B_K_TILE = 0, B_K_DUAL_N = 1, B_MN_TILE = 2, B_MN_DUAL_K = 3 };
// EPI_ROUTE: the router projection with the routing's softmax + top-k fused
// into the epilogue (route_fused.cu): each epilogue thread holds one token's
// logits, E <= 256 columns of the tile.
enum EpiMode : int { EPI_F32_BIAS = 0, EPI_SWIGLU_FWD = 1, EPI_BF16 = 2, EPI_SWIGLU_BWD = 3, EPI_ROUTE = 4 };
// SCHED_ROWS2 / SCHED_WGRAD2: the same tiles in pairs of m-tiles on one
// n-tile, each pair computed by a cluster of two CTAs with cta_group::2 MMAs
// (M = 256).
// SCHED_WGRAD_WIDE: weight gradients on one SM with eight epilogue warps (see
// epi_wide), for the shortest K loops.
enum SchedMode : int { SCHED_ROWS = 0, SCHED_WGRAD = 1, SCHED_ROWS2 = 2, SCHED_WGRAD2 = 3, SCHED_WGRAD_WIDE = 4 };
__host__ __device__ constexpr bool sched_wgrad(int sch) {
  return sch == SCHED_WGRAD || sch == SCHED_WGRAD2 || sch == SCHED_WGRAD_WIDE;
}
__host__ __device__ constexpr bool sched_pair(int sch) { return sch == SCHED_ROWS2 || sch == SCHED_WGRAD2; }

constexpr int kBM = 128;  // rows per tile (TMEM lanes)
constexpr int kBN = 256;  // accumulator columns per tile
constexpr int kBK = 64;   // bf16 K per stage: one 128-byte swizzle row
constexpr int kBKmx = 128;  // MXFP8 K per stage: one 128-byte swizzle row of E4M3
constexpr int kStages = 4;  // pipeline stages with 256-column tiles
constexpr int kATileBytes = kBM * 128;  // 16 KB (128 rows of 128 bytes)
constexpr int kBTileBytes = kBN * 128;  // 32 KB
constexpr int kStageBytes = kATileBytes + kBTileBytes;
constexpr int kSfStageBytes = 512 + 1024;  // MXFP8: scales of the A tile and the B tile
constexpr int kSfTmemCol = 256;            // MXFP8: first TMEM column of the scale ring
constexpr int kSfTmemStride = 16;          // MXFP8: columns per stage (A at +0, B at +8)
constexpr int kMNChunkBytes = kBK * 128;   // one 64-wide MN chunk of an MN-major tile
constexpr int kTmemCols = 512;
constexpr int kGemmThreads = 256;  // warps 0-3 roles (TMA, MMA, TMEM allocation, idle), 4-7 epilogue
constexpr int kStageBoxBytes = 32 * 128;   // one epilogue staging box: 32 rows x 128 bytes

// Tile width (accumulator columns) per instantiation: 256 everywhere.  A
// width of 128 gives MXFP8 kernels room for two accumulators beside the scale
// ring; measured for the MXFP8 weight gradients it was slower (2.11 -> 2.96 ms
// at the DSV3 shape: twice the tiles, each with a fixed cost), so no
// instantiation uses it.
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int gemm_bn() { return kBN; }
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int acc_bufs() { return (MX && gemm_bn<MX, EPI, SCH>() == kBN) ? 1 : 2; }
// A stage holds the A tile and the B tile, or in the 2-SM mode this CTA's
// half of B.
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int stage_bytes() {
  return kATileBytes + (sched_pair(SCH) ? gemm_bn<MX, EPI, SCH>() / 2 : gemm_bn<MX, EPI, SCH>()) * 128;
}
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int sf_stage_bytes() { return MX ? 512 + gemm_bn<MX, EPI, SCH>() / 128 * 512 : 0; }

// Epilogue warps.  One per TMEM lane quadrant (warps 4-7), except where the
// epilogue would be slower than the MMAs with one: the MXFP8 SwiGLU backward
// (heavy arithmetic) and the bf16 weight gradients of experts with very few
// rows (SCHED_WGRAD_WIDE: a 128 x 256 tile to store after a K loop of a few
// MMAs).  Those get two per quadrant (warps 2-9, 320 threads; the TMEM
// allocator, warp 2, is one of them), each taking half of the columns.
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr bool epi_wide() {
  return (MX && EPI == EPI_SWIGLU_BWD) || (!MX && EPI == EPI_BF16 && SCH == SCHED_WGRAD_WIDE);
}
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int epi_warps() { return epi_wide<MX, EPI, SCH>() ? 8 : 4; }
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int first_epi_warp() { return epi_wide<MX, EPI, SCH>() ? 2 : 4; }
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int gemm_threads() {
  return 32 * (first_epi_warp<MX, EPI, SCH>() + epi_warps<MX, EPI, SCH>());
}
// Pipeline stages: four 48 KB stages, six 32 KB ones in the 2-SM mode (five
// 32 KB ones with 128-column tiles, which no instantiation uses), three 48 KB
// ones in SCHED_WGRAD_WIDE,
// whose eight epilogue warps take 64 KB of staging (with K loops of a few
// MMAs per tile, deeper rings buy nothing there; with longer ones the fourth
// stage is worth more than the wide epilogue).
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int gemm_stages() {
  if (!MX && epi_wide<MX, EPI, SCH>()) return 3;
  // MXFP8 on SM pairs: four 32 KB stages, as many as the TMEM scale ring
  // has slots (the accumulator, the ring and the epilogue stash fill TMEM)
  if (MX && sched_pair(SCH)) return kStages;
  return sched_pair(SCH) ? 6 : (gemm_bn<MX, EPI, SCH>() == kBN ? kStages : 5);
}
// MXFP8 kernels, with a single 256-column accumulator beside the scale ring,
// run the stash epilogue (with 128-column tiles and two accumulators they
// would run the bf16-mode one).
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr bool epi_mx_stash() { return MX && acc_bufs<MX, EPI, SCH>() == 1; }
// Epilogue shared memory per epilogue warp: 4 KB staging boxes that TMA
// stores to global memory while the next box is being filled (two per warp
// with two accumulators); in the stash epilogue, whose kernels keep the scale
// stages in shared memory too, one box (in 5 KB), or for the SwiGLU backward
// the 32 x 17 fp32 transpose buffer.
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int epi_slots() {
  return (!epi_mx_stash<MX, EPI, SCH>() && !(MX && epi_wide<MX, EPI, SCH>())) ? 2 : 1;
}
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int epi_warp_bytes() {
  return !epi_mx_stash<MX, EPI, SCH>() ? epi_slots<MX, EPI, SCH>() * 32 * 128
                                       : (epi_wide<MX, EPI, SCH>() ? 32 * 17 * 4 : 5 * 1024);
}
template <bool MX>
__host__ __device__ constexpr int stage_k() { return MX ? kBKmx : kBK; }
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr int gemm_smem_bytes_for() {
  return 1024 + gemm_stages<MX, EPI, SCH>() * (stage_bytes<MX, EPI, SCH>() + sf_stage_bytes<MX, EPI, SCH>()) +
         epi_warps<MX, EPI, SCH>() * epi_warp_bytes<MX, EPI, SCH>() + 256;
}

// The bf16 GEMMs other than the router projection run as two launches: a
// 2-SM pass (SCHED_ROWS2, SCHED_WGRAD2) over pairs of m-tiles, and a 1-SM
// pass over the rest (grouped rows: every tile of the experts with an odd
// number of them, so that no expert's weights are streamed by both passes;
// dense rows and weight gradients: the last m-tile of an odd count).  A 128 x 256 tile
// per SM stages 48 KB per K step and its MMAs read as much again from shared
// memory; with the B tile split between the two SMs of a pair both become
// 32 KB.  Measured at the DSV3 shape, staging only half of the gate/up weight
// tile took that kernel from 5.73 to 5.17 ms, while multicasting halves of a
// shared operand between two CTAs (fewer L2 reads, same shared-memory
// traffic) gained nothing: shared-memory traffic per SM bounds these GEMMs.
// Both passes load B in halves (128-row or two-chunk boxes), so they share
// their tensor maps.  The MXFP8 row GEMMs run the same two passes; on SM
// pairs each CTA also loads the scales of its 128 rows of A and of all of B
// (which both CTAs' MMAs read from their own TMEM) through tmSfA / tmSfB*.
template <bool MX, int EPI, int SCH>
__host__ __device__ constexpr bool b_halves() {
  // the router projection (fp32 logits, or with the fused top-k) loads its
  // 256-row B tile with one box
  return EPI != EPI_F32_BIAS && EPI != EPI_ROUTE && (!MX || !sched_wgrad(SCH));
}

struct GemmParams {
  // Operand maps: K-major operands are 2-D [rows, K] maps with 128-byte x rows
  // boxes; MN-major operands are 3-D maps (make_tmap_mn3d) whose box holds
  // every 64-column chunk of the tile (2 for A, 4 for B).
  CUtensorMap tmA;
  CUtensorMap tmB0;
  CUtensorMap tmB1;
  // Output tensor maps (boxes of 64 columns x 32 rows, 128-byte swizzle):
  //   EPI_BF16      tmO0 over `out` ([rows, N], or [G, M_out, N] for SCHED_WGRAD)
  //   EPI_SWIGLU_FWD tmO0 over the [a|b] rows, tmO1 over h
  CUtensorMap tmO0;
  CUtensorMap tmO1;
  // The same outputs with 16-row boxes, for the 64-row tail tiles of grouped
  // problems (an M=64 accumulator leaves 16 rows per epilogue warp).
  CUtensorMap tmO0h;
  CUtensorMap tmO1h;
  // MXFP8 on SM pairs: the scale arrays of A (512-byte boxes) and of B (one
  // 1024-byte box, or 512 bytes from each stack of a dual-N operand), viewed
  // as [bytes / 256, 256] (make_tmap_bytes).
  CUtensorMap tmSfA;
  CUtensorMap tmSfB0;
  CUtensorMap tmSfB1;
  // ---- schedule
  int dense_rows;          // > 0: a single group of this many rows; 0: grouped by row_start
  int num_groups;          // number of groups (experts) when grouped
  const int* row_start;    // [G+1] padded row offsets, multiples of 64 (128 in MXFP8 mode)
  const int* tile_start;   // [G+1] prefix of 128-row tiles per group (grouped SCHED_ROWS)
  const int* pair_start;   // [G+1] prefix of tile pairs per group (grouped SCHED_ROWS2)
  const int* rem_start;    // [G+1] prefix of the tiles per group left to one SM (grouped, part 1)
  int part;                // 1-SM passes: 0 every tile; 1 only the tiles that are not in
                           // pairs (grouped rows: every tile of a group with an odd tile
                           // count; dense rows and weight gradients: the last m-tile when
                           // the m-tile count is odd)
  const int* counts;       // [G] real rows per group (grouped)
  int N;                   // output columns
  int K;                   // reduction length (SCHED_ROWS)
  int M_out;               // output rows per group (SCHED_WGRAD)
  int b_group_rows;        // rows of the B tensor map per group (0: B rows are absolute)
  int a_col_off;           // SCHED_WGRAD: first column (A_MN_TILE) or row (A_K_TILE) of A's M range
  int b_split;             // B_MN_DUAL_K: K index from which B comes from tmB1
  // ---- MXFP8 operand scales (tcgen05.cp block layout, see mx_common.cuh)
  const uint8_t* sfa;      // scales of A; rows of A / 128 = sfa_rb
  long long sfa_rb;
  const uint8_t* sfb0;     // scales of B (of the first stack for B_K_DUAL_N)
  const uint8_t* sfb1;     // scales of the second stack (B_K_DUAL_N)
  long long sfb_rb;
  // ---- epilogue
  void* out;               // direct-store outputs: EPI_F32_BIAS logits; bf16 EPI_SWIGLU_BWD [da|db];
                           // MXFP8 EPI_SWIGLU_FWD the saved [a|b] rows
  long long ldo;
  void* out2;              // bf16 EPI_SWIGLU_BWD g*h
  long long ldo2;
  float* out3;
  int ldo3;
  const float* bias;
  const float* row_scale;
  const __nv_bfloat16* ab;
  int I;
  int store_ab;
  // MXFP8 quantized epilogue output (E4M3 rows + scales), required in MXFP8
  // mode: h for EPI_SWIGLU_FWD (whose a and b rows then go to `out` when
  // store_ab), [da|db] for EPI_SWIGLU_BWD.
  uint8_t* qout;
  long long qld;
  uint8_t* qsf;
  long long q_rb;
  // MXFP8 EPI_SWIGLU_BWD: the transposes [da|db]^T ([2I, rows]) and (g*h)^T
  // ([I, rows]) quantized along the token rows (blocks of 32), the K-major
  // operands of the weight gradients.  These replace the bf16 out / out2.
  uint8_t* qt;
  long long qt_ld;
  uint8_t* qt_sf;
  long long qt_rb;
  uint8_t* qt2;
  long long qt2_ld;
  uint8_t* qt2_sf;
  long long qt2_rb;
  int* status;
  // Test hook (0 normally): bytes the first pipeline stage of each CTA's first
  // tile expects beyond what its loads bring (on SM pairs: the even CTA's, whose
  // barrier counts both CTAs' loads), so that its MMA warp's bounded wait runs
  // out and both CTAs of the pair take their abort paths.
  uint32_t debug_extra_tx;
  // Weight gradients, chosen by the host from the experts' row ranges (the K
  // of these GEMMs): 0 pairs of m-tiles on SM pairs (and the last m-tile on
  // one SM), 1 every tile on one SM (short K), 2 every tile on one SM with
  // the wide epilogue (the shortest K).
  int wgrad_mode;
  // Weight gradients: nonzero when tmO0 maps an fp32 output (boxes of 32
  // columns x 32 rows) instead of a bf16 one (64 x 32).
  int wgrad_f32;
  // EPI_ROUTE: top-k ids and weights [T, route_k], per-chunk expert
  // histograms [ceil(T / kChunkTokens), N] (N = E; `out` optionally receives
  // the logits, with the bias added).
  int32_t* route_idx;
  float* route_w;
  int32_t* route_chunk;
  int route_k;
};

// The softmax + top-k fused into the router projection's epilogue keeps a
// sorted list of this many candidates per token (top_k <= kRouteMaxK).
constexpr int kRouteMaxK = 16;

template <int EPI>
__host__ __device__ constexpr int tile_out_cols() {
  return EPI == EPI_SWIGLU_FWD ? kBN / 2 : kBN;
}

struct TileInfo {
  int e;           // group (expert)
  int row0;        // first row of the tile (SCHED_ROWS) in the padded row space
  int rows_valid;  // rows of the tile that hold real data
  int m64;         // 1: 64-row tail tile of a group (M=64 MMA, 16 rows per epilogue warp)
  int m0;          // first output row (SCHED_WGRAD)
  int n0;          // first output column
  int nt;          // n-tile index
  int kb0;         // first K block
  int nkb;         // number of K blocks
};

__device__ __forceinline__ int find_group(const int* row_start, int G, int row) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(row_start + mid) <= row)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Work items per launch: tiles, or in the 2-SM mode pairs of tiles.
template <int EPI, int SCH, int BN>
__device__ __forceinline__ int gemm_num_tiles(const GemmParams& p) {
  if constexpr (!sched_wgrad(SCH)) {
    const int num_nt = (p.N + tile_out_cols<EPI>() - 1) / tile_out_cols<EPI>();
    if (p.dense_rows > 0) {
      const int mt = (p.dense_rows + kBM - 1) / kBM;
      if (SCH == SCHED_ROWS2) return (mt / 2) * num_nt;
      return (p.part ? (mt & 1) : mt) * num_nt;
    }
    const int* prefix = SCH == SCHED_ROWS2 ? p.pair_start : (p.part ? p.rem_start : p.tile_start);
    return __ldg(prefix + p.num_groups) * num_nt;
  } else {
    const int num_nt = (p.N + BN - 1) / BN;
    const int num_mt = (p.M_out + kBM - 1) / kBM;
    const int G = p.dense_rows > 0 ? 1 : p.num_groups;
    if (SCH == SCHED_WGRAD2) return G * (num_mt / 2) * num_nt;
    return G * (p.part ? (num_mt & 1) : num_mt) * num_nt;
  }
}

// Rows of m-tile mt of group e (grouped row problems).
__device__ __forceinline__ void grouped_rows(const GemmParams& p, int e, int mt, TileInfo& t) {
  t.e = e;
  t.row0 = __ldg(p.row_start + e) + mt * kBM;
  t.m64 = (__ldg(p.row_start + e + 1) - t.row0) < kBM ? 1 : 0;
  t.rows_valid = max(0, min(t.m64 ? kBM / 2 : kBM, __ldg(p.counts + e) - mt * kBM));
}

// Tile of work item tau.  Row problems: grouped ones go expert by expert,
// n-tile outer and m-tile inner, so that CTAs running at the same time share
// one weight tile while the expert's activation rows stay in L2; dense ones
// go m-tile outer, n-tile inner (the weight panel stays L2-resident while
// the rows stream once).  In the 2-SM mode item tau is a pair of m-tiles
// (2j, 2j+1) on one n-tile, of which the CTA of rank `rank` takes 2j + rank.
template <int EPI, int SCH, int BK, int BN = kBN>
__device__ __forceinline__ TileInfo gemm_tile(const GemmParams& p, int tau, uint32_t rank = 0) {
  TileInfo t;
  if constexpr (!sched_wgrad(SCH)) {
    constexpr int W = tile_out_cols<EPI>();
    const int num_nt = (p.N + W - 1) / W;
    const int r = static_cast<int>(rank);
    int mt, nt;
    if (p.dense_rows > 0) {
      const int dense_mt = (p.dense_rows + kBM - 1) / kBM;
      if (SCH == SCHED_ROWS2) {
        mt = 2 * (tau / num_nt) + r;
        nt = tau % num_nt;
      } else if (p.part) {
        mt = dense_mt - 1;
        nt = tau;
      } else {
        mt = tau / num_nt;
        nt = tau - mt * num_nt;
      }
      t.e = 0;
      t.row0 = mt * kBM;
      t.rows_valid = min(kBM, p.dense_rows - t.row0);
      t.m64 = 0;
    } else {
      const int G = p.num_groups;
      int e;
      if (SCH == SCHED_ROWS2) {
        e = find_group(p.pair_start, G, tau / num_nt);
        const int ps = __ldg(p.pair_start + e);
        const int np = __ldg(p.pair_start + e + 1) - ps;
        const int local = tau - ps * num_nt;
        nt = local / np;
        mt = 2 * (local - nt * np) + r;
      } else if (p.part) {
        // this expert's m-tiles that are not in pairs: the ones after its pairs
        e = find_group(p.rem_start, G, tau / num_nt);
        const int rs = __ldg(p.rem_start + e);
        const int nr = __ldg(p.rem_start + e + 1) - rs;
        const int local = tau - rs * num_nt;
        nt = local / nr;
        mt = 2 * (__ldg(p.pair_start + e + 1) - __ldg(p.pair_start + e)) + (local - nt * nr);
      } else {
        const int q = tau / num_nt;
        e = find_group(p.tile_start, G, q);
        const int ts = __ldg(p.tile_start + e);
        const int mt_e = __ldg(p.tile_start + e + 1) - ts;
        const int local = tau - ts * num_nt;
        nt = local / mt_e;
        mt = local - nt * mt_e;
      }
      grouped_rows(p, e, mt, t);
    }
    t.m0 = 0;
    t.nt = nt;
    t.n0 = nt * W;
    t.kb0 = 0;
    t.nkb = p.K / BK;
  } else {
    // weight gradients: group outer, m-tile, n-tile inner
    const int num_nt = (p.N + BN - 1) / BN;
    const int num_mt = (p.M_out + kBM - 1) / kBM;
    int e, mt, nt;
    if (SCH == SCHED_WGRAD2) {
      const int per_g = (num_mt / 2) * num_nt;
      e = tau / per_g;
      const int local = tau - e * per_g;
      const int j = local / num_nt;
      nt = local - j * num_nt;
      mt = 2 * j + static_cast<int>(rank);
    } else if (p.part) {
      e = tau / num_nt;
      nt = tau - e * num_nt;
      mt = num_mt - 1;
    } else {
      const int per_g = num_mt * num_nt;
      e = tau / per_g;
      const int local = tau - e * per_g;
      mt = local / num_nt;
      nt = local - mt * num_nt;
    }
    t.e = e;
    t.m0 = mt * kBM;
    t.nt = nt;
    t.n0 = nt * BN;
    t.row0 = 0;
    t.rows_valid = 0;
    t.m64 = 0;
    if (p.dense_rows > 0) {
      t.kb0 = 0;
      t.nkb = (p.dense_rows + BK - 1) / BK;
    } else {
      const int rs = __ldg(p.row_start + e);
      t.kb0 = rs / BK;
      t.nkb = (__ldg(p.row_start + e + 1) - rs) / BK;
    }
  }
  return t;
}

// The loop every role runs: items first, first + stride, ... below count;
// in the 2-SM mode over cluster indices, `rank` being the CTA's in the pair.
struct WorkRange {
  int first, stride, count;
  uint32_t rank;
};

// ------------------------------------------------------------------ producer
// Half h of a 256-column B tile (its rows n0 + 128h .. n0 + 128h + 127): one
// 128-row K-major box, the gate (h = 0) or up (h = 1) stack of a dual-N
// operand, or two 64-column chunks of an MN-major operand, into dst.  PAIR:
// completion on the pair's full barrier (shared::cluster address).
template <int BMO, bool PAIR>
__device__ __forceinline__ void load_b_half(const GemmParams& p, uint32_t dst, const TileInfo& t, int kabs,
                                            int brow, int h, uint32_t bar) {
  if constexpr (BMO == B_K_TILE || BMO == B_K_DUAL_N) {
    const void* map = (BMO == B_K_DUAL_N && h) ? &p.tmB1 : &p.tmB0;
    const int row = BMO == B_K_TILE ? brow + h * (kBN / 2) : brow;
    if constexpr (PAIR)
      tma_load_2d_pair(dst, map, kabs, row, bar);
    else
      tma_load_2d(dst, map, kabs, row, bar);
  } else {
    const bool second = BMO == B_MN_DUAL_K && kabs >= p.b_split;
    const void* map = second ? &p.tmB1 : &p.tmB0;
    const int krow = t.e * p.b_group_rows + (second ? kabs - p.b_split : kabs);
    if constexpr (PAIR)
      tma_load_3d_pair(dst, map, 0, krow, t.n0 / 64 + 2 * h, bar);
    else
      tma_load_3d(dst, map, 0, krow, t.n0 / 64 + 2 * h, bar);
  }
}

// The A tile: 128 K-major rows from arow, or (MN-major, weight gradients)
// both 64-column chunks of the M range with one 3-D box.
template <int AM, bool PAIR>
__device__ __forceinline__ void load_a(const GemmParams& p, uint32_t dst, const TileInfo& t, int kabs, int arow,
                                       uint32_t bar) {
  if constexpr (AM == A_K_TILE) {
    if constexpr (PAIR)
      tma_load_2d_pair(dst, &p.tmA, kabs, arow, bar);
    else
      tma_load_2d(dst, &p.tmA, kabs, arow, bar);
  } else {
    if constexpr (PAIR)
      tma_load_3d_pair(dst, &p.tmA, 0, kabs, (p.a_col_off + t.m0) / 64, bar);
    else
      tma_load_3d(dst, &p.tmA, 0, kabs, (p.a_col_off + t.m0) / 64, bar);
  }
}

template <int AM, int BMO, int EPI, int SCH, bool MX>
__device__ __forceinline__ void gemm_producer(const GemmParams& p, uint32_t s_tiles, uint32_t s_sf,
                                              uint32_t full0, uint32_t empty0, const WorkRange& wr,
                                              volatile int* abort_flag, int lane) {
  constexpr bool PAIR = sched_pair(SCH);
  constexpr bool HALVES = b_halves<MX, EPI, SCH>();
  constexpr int BK = stage_k<MX>();
  constexpr int BN = gemm_bn<MX, EPI, SCH>();
  constexpr int SB = stage_bytes<MX, EPI, SCH>(), SFB = sf_stage_bytes<MX, EPI, SCH>();
  constexpr uint32_t kTx = SB + SFB;
  static_assert(!HALVES || BN == kBN, "B halves: 256-column tiles");
  int s = 0;
  uint32_t ph = 0;
  // Per stage: parity of the last load issued into it, or -1.
  constexpr int ST = gemm_stages<MX, EPI, SCH>();
  int issued_parity[ST];
#pragma unroll
  for (int i = 0; i < ST; ++i) issued_parity[i] = -1;
  bool aborted = false;
  // 2-SM mode: both CTAs' loads complete on the even CTA's full barriers
  const uint32_t lead_full0 = PAIR ? mapa_shared(full0, 0) : full0;

  for (int w = wr.first; w < wr.count && !aborted; w += wr.stride) {
    const TileInfo t = gemm_tile<EPI, SCH, BK, BN>(p, w, wr.rank);
    // row coordinate of the A tile: token rows, or output rows of a weight gradient
    const int arow = sched_wgrad(SCH) ? p.a_col_off + t.m0 : t.row0;
    const int brow = t.e * p.b_group_rows + t.n0;
    for (int kb = 0; kb < t.nkb; ++kb) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        aborted = true;
        break;
      }
      const uint32_t full = full0 + 8 * s;
      const uint32_t sA = s_tiles + s * SB;
      const uint32_t sB = sA + kATileBytes;
      const int kabs = (t.kb0 + kb) * BK;
      if constexpr (PAIR || HALVES) {
        // 2-SM mode: this CTA's 128 rows (or MN columns) of A and its half of
        // B, the even CTA's barrier counting both CTAs' bytes
        if (lane == 0) {
          if (!PAIR || wr.rank == 0)
            mbar_arrive_expect_tx(full, (PAIR ? 2 * kTx : kTx) + ((w == wr.first && kb == 0) ? p.debug_extra_tx : 0u));
          const uint32_t fb = PAIR ? lead_full0 + 8 * s : full;
          load_a<AM, PAIR>(p, sA, t, kabs, arow, fb);
          if constexpr (PAIR) {
            load_b_half<BMO, true>(p, sB, t, kabs, brow, static_cast<int>(wr.rank), fb);
          } else {
            load_b_half<BMO, false>(p, sB, t, kabs, brow, 0, full);
            load_b_half<BMO, false>(p, sB + kBTileBytes / 2, t, kabs, brow, 1, full);
          }
          if constexpr (MX) {
            // scales of this CTA's A rows and of the whole B tile (both CTAs of a
            // pair hold all of B's: each CTA's MMA half reads them from its TMEM)
            const long long g = kabs / kBKmx;
            const uint32_t sfs = s_sf + s * SFB;
            const int ablk = static_cast<int>(g * p.sfa_rb + arow / 128);
            const int bblk = static_cast<int>(g * p.sfb_rb + brow / 128);
            if constexpr (PAIR) {
              tma_load_2d_pair(sfs, &p.tmSfA, 0, 2 * ablk, fb);
              if constexpr (BMO == B_K_DUAL_N) {
                tma_load_2d_pair(sfs + 512, &p.tmSfB0, 0, 2 * bblk, fb);
                tma_load_2d_pair(sfs + 1024, &p.tmSfB1, 0, 2 * bblk, fb);
              } else {
                tma_load_2d_pair(sfs + 512, &p.tmSfB0, 0, 2 * bblk, fb);
              }
            } else {
              bulk_load(sfs, p.sfa + static_cast<size_t>(ablk) * 512, 512, full);
              if constexpr (BMO == B_K_DUAL_N) {
                bulk_load(sfs + 512, p.sfb0 + static_cast<size_t>(bblk) * 512, 512, full);
                bulk_load(sfs + 1024, p.sfb1 + static_cast<size_t>(bblk) * 512, 512, full);
              } else {
                bulk_load(sfs + 512, p.sfb0 + static_cast<size_t>(bblk) * 512, BN / 128 * 512, full);
              }
            }
          }
        }
        __syncwarp();
      } else {
        if (lane == 0) mbar_arrive_expect_tx(full, kTx + ((w == wr.first && kb == 0) ? p.debug_extra_tx : 0u));
        __syncwarp();
        // ---- A operand
        if constexpr (AM == A_K_TILE) {
          if (lane == 0) tma_load_2d(sA, &p.tmA, kabs, arow, full);
        } else {  // A_MN_TILE (bf16): both 64-column chunks with one 3-D box
          if (lane == 0) tma_load_3d(sA, &p.tmA, 0, kabs, (p.a_col_off + t.m0) / 64, full);
        }
        // ---- B operand
        if constexpr (BMO == B_K_TILE) {
          if (lane == 0) tma_load_2d(sB, &p.tmB0, kabs, brow, full);
        } else if constexpr (BMO == B_K_DUAL_N) {
          if (lane == 0) {
            tma_load_2d(sB, &p.tmB0, kabs, brow, full);
            tma_load_2d(sB + kBTileBytes / 2, &p.tmB1, kabs, brow, full);
          }
        } else if constexpr (BMO == B_MN_TILE) {  // four 64-column chunks, one 3-D box
          if (lane == 0) tma_load_3d(sB, &p.tmB0, 0, t.e * p.b_group_rows + kabs, t.n0 / 64, full);
        } else {  // B_MN_DUAL_K
          if (lane == 0) {
            const bool second = kabs >= p.b_split;
            const int kk = second ? kabs - p.b_split : kabs;
            tma_load_3d(sB, second ? (const void*)&p.tmB1 : (const void*)&p.tmB0, 0,
                        t.e * p.b_group_rows + kk, t.n0 / 64, full);
          }
        }
        // ---- MXFP8 scales of this stage's A and B tiles (one 128-column group)
        if constexpr (MX) {
          if (lane == 0) {
            const long long g = kabs / kBKmx;
            const uint32_t sfs = s_sf + s * SFB;
            bulk_load(sfs, p.sfa + (g * p.sfa_rb + arow / 128) * 512, 512, full);
            const size_t boff = static_cast<size_t>((g * p.sfb_rb + brow / 128) * 512);
            if constexpr (BMO == B_K_DUAL_N) {
              bulk_load(sfs + 512, p.sfb0 + boff, 512, full);
              bulk_load(sfs + 1024, p.sfb1 + boff, 512, full);
            } else {
              bulk_load(sfs + 512, p.sfb0 + boff, BN / 128 * 512, full);
            }
          }
        }
      }
      issued_parity[s] = static_cast<int>(ph);
      if (++s == ST) {
        s = 0;
        ph ^= 1;
      }
    }
  }
  if (lane == 0 && (!PAIR || wr.rank == 0)) {
    // Loads still in flight must land before the CTA's shared memory goes
    // away (2-SM mode: the even CTA's barriers also count the odd CTA's).  In
    // a run without faults these phases have completed already; after an
    // abort (the MMA warp may never have waited for them) the wait is bounded.
#pragma unroll
    for (int i = 0; i < ST; ++i)
      if (issued_parity[i] >= 0)
        mbar_wait(full0 + 8 * i, static_cast<uint32_t>(issued_parity[i]), abort_flag, p.status,
                  false);
  }
  if constexpr (PAIR) {
    // The even CTA's MMA commits arrive on both CTAs' empty barriers: wait for
    // the last round of every stage to be released, so that none of them is
    // still in flight when the CTA exits.
    if (!aborted && lane == 0) {
      for (int i = 0; i < ST; ++i) {
        if (!mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag, p.status)) break;
        if (++s == ST) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
template <int AM, int BMO, int EPI, int SCH, bool MX>
__device__ __forceinline__ void gemm_mma(const GemmParams& p, uint32_t s_tiles, uint32_t s_sf,
                                         uint32_t full0, uint32_t empty0, uint32_t accf0,
                                         uint32_t acce0, uint32_t drain, uint32_t tmem_base,
                                         const WorkRange& wr, volatile int* abort_flag) {
  // 2-SM mode: the even CTA issues the pair's MMAs (M = 256: its 128 rows of
  // A and the odd CTA's), the odd CTA's MMA warp has nothing to do
  constexpr bool PAIR = sched_pair(SCH);
  if (PAIR && wr.rank != 0) return;
  constexpr int BK = stage_k<MX>();
  constexpr int ST = gemm_stages<MX, EPI, SCH>();
  constexpr int BN = gemm_bn<MX, EPI, SCH>();
  constexpr int SB = stage_bytes<MX, EPI, SCH>(), SFB = sf_stage_bytes<MX, EPI, SCH>();
  constexpr bool a_mn = (AM == A_MN_TILE);
  constexpr bool b_mn = (BMO == B_MN_TILE || BMO == B_MN_DUAL_K);
  constexpr uint32_t idesc128 = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN, a_mn ? 1 : 0, b_mn ? 1 : 0);
  constexpr int kMxM = PAIR ? 2 * kBM : kBM;
  constexpr uint32_t idesc64 = idesc_bf16_f32(kBM / 2, BN, a_mn ? 1 : 0, b_mn ? 1 : 0);
  int s = 0;
  uint32_t ph = 0;
  int acc = 0;
  uint32_t aph = 0;
  bool issued = false, aborted = false;
  for (int w = wr.first; w < wr.count && !aborted; w += wr.stride) {
    const TileInfo t = gemm_tile<EPI, SCH, BK, BN>(p, w, wr.rank);
    if (!mbar_wait(acce0 + 8 * acc, aph ^ 1, abort_flag, p.status)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
    // a pair always runs M = 256 (the rows past a 64-row tail are not stored)
    const uint32_t idesc = (t.m64 && !PAIR) ? idesc64 : idesc128;
    for (int kb = 0; kb < t.nkb; ++kb) {
      if (!mbar_wait(full0 + 8 * s, ph, abort_flag, p.status)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t sA = s_tiles + s * SB;
      const uint32_t sB = sA + kATileBytes;
      if constexpr (MX) {
        // scale ring slot s: reused by stage s + ST, whose data can only
        // have been loaded after these MMAs released stage s
        const uint32_t sfa_t = tmem_base + kSfTmemCol + s * kSfTmemStride;
        const uint32_t sfs = s_sf + s * SFB;
        if constexpr (PAIR) {  // each CTA's scale blocks into its own TMEM
          tc_cp_32x128b_pair(sfa_t, sfs);
          tc_cp_32x128b_pair(sfa_t + 8, sfs + 512);
          tc_cp_32x128b_pair(sfa_t + 12, sfs + 1024);
        } else {
          tc_cp_32x128b(sfa_t, sfs);
          tc_cp_32x128b(sfa_t + 8, sfs + 512);
          if constexpr (BN == 256) tc_cp_32x128b(sfa_t + 12, sfs + 1024);
        }
        // both operands K-major: K = 32 is 32 bytes along the swizzled row
        static_assert(!a_mn && !b_mn, "MXFP8 operands are K-major");
#pragma unroll
        for (int kk = 0; kk < kBKmx / 32; ++kk) {
          const uint64_t ad = smem_desc_sw128(sA + kk * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sB + kk * 32, 16, 1024);
          if constexpr (PAIR)
            tc_mma_mxf8_pair(d_tmem, ad, bd, idesc_mxf8(kMxM, BN, kk), sfa_t, sfa_t + 8, (kb > 0 || kk > 0) ? 1u : 0u);
          else
            tc_mma_mxf8(d_tmem, ad, bd, idesc_mxf8(kMxM, BN, kk), sfa_t, sfa_t + 8, (kb > 0 || kk > 0) ? 1u : 0u);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = a_mn ? smem_desc_sw128(sA + kk * 2048, kMNChunkBytes, 1024)
                                   : smem_desc_sw128(sA + kk * 32, 16, 1024);
          const uint64_t bd = b_mn ? smem_desc_sw128(sB + kk * 2048, kMNChunkBytes, 1024)
                                   : smem_desc_sw128(sB + kk * 32, 16, 1024);
          if constexpr (PAIR)
            tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          else
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
      }
      if constexpr (PAIR)
        tc_commit_pair_mc(empty0 + 8 * s, 3);  // frees the stage in both CTAs
      else
        tc_commit(empty0 + 8 * s);
      issued = true;
      if (++s == ST) {
        s = 0;
        ph ^= 1;
      }
    }
    if (aborted) break;
    if constexpr (PAIR) {
      if (t.nkb > 0) {
        tc_commit_pair_mc(accf0 + 8 * acc, 3);
      } else {
        mbar_arrive(accf0 + 8 * acc);
        mbar_arrive_remote(mapa_shared(accf0 + 8 * acc, 1));
      }
    } else if (t.nkb > 0) {
      tc_commit(accf0 + 8 * acc);
    } else {
      mbar_arrive(accf0 + 8 * acc);
    }
    if (++acc == acc_bufs<MX, EPI, SCH>()) {
      acc = 0;
      aph ^= 1;
    }
  }
  if (aborted && issued) {
    // MMAs still in flight must finish before TMEM is released.
    if constexpr (PAIR)
      tc_commit_pair(drain);
    else
      tc_commit(drain);
    mbar_wait(drain, 0, abort_flag, p.status, false);
  }
}

// ------------------------------------------------------------------ epilogue
// Each epilogue thread owns one accumulator row (TMEM lane).  Results are
// converted to bf16 and written into the warp's staging boxes in the swizzled
// layout, then one lane issues a TMA store of the 32 x 64 box; with two boxes
// per warp, filling one overlaps the store of the other.
template <int NSLOT>
struct EpiStager {
  uint32_t base;  // this warp's boxes
  int slot;
  int lane;
  __device__ __forceinline__ uint32_t begin() {
    if (lane == 0) bulk_wait_group_read<NSLOT - 1>();  // the box about to be filled is free
    __syncwarp();
    return base + static_cast<uint32_t>(slot) * kStageBoxBytes;
  }
  __device__ __forceinline__ void next() { slot = slot + 1 == NSLOT ? 0 : slot + 1; }
  __device__ __forceinline__ void store2d(const CUtensorMap* tm, uint32_t box, int c0, int c1) {
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm, c0, c1, box);
      bulk_commit_group();
    }
    next();
  }
  __device__ __forceinline__ void store3d(const CUtensorMap* tm, uint32_t box, int c0, int c1, int c2) {
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tm, c0, c1, c2, box);
      bulk_commit_group();
    }
    next();
  }
  // stage 64 values of this thread's row and store them at (c0, c1)
  __device__ __forceinline__ void row64_2d(const CUtensorMap* tm, const float* v, int c0, int c1) {
    const uint32_t box = begin();
    stage_row_sw128(box, lane, v);
    store2d(tm, box, c0, c1);
  }
};

// EPI_ROUTE, one tile of 128 tokens: this thread's token (row `grow` of the
// dense rows) reads its E logits (+ bias) from TMEM 16 columns at a time, sorts
// each 16 into selection order (logits descending, equal logits to the lower
// expert index; a NaN as -inf with an index past E) with a sorting network and
// merges them into its running list of the KM best (route_merge_top), then
// writes the top-k ids and router weights (exp(l_j - l_0) over their sum, in
// the summation order of route_weight_sum) and adds its picks to the expert
// histogram of its chunk (integer atomics into route_chunk, which starts at
// zero).  The logits also go to `out` when it is set.  `release` frees the
// accumulator as soon as the logits are read.  KM: 8 for top_k <= 8, else 16.
template <int KM, class Release>
__device__ __forceinline__ void epi_route(const GemmParams& p, uint32_t tr, bool real, int grow, Release release) {
  const int E = p.N, k = p.route_k;
  float lv[KM];
  int le[KM];
#pragma unroll
  for (int s = 0; s < KM; ++s) {
    lv[s] = -INFINITY;
    le[s] = INT_MAX;
  }
  float* lo = (real && p.out) ? reinterpret_cast<float*>(p.out) + static_cast<long long>(grow) * p.ldo : nullptr;
  for (int c0 = 0; c0 < E; c0 += 16) {
    float v[16];
    int ei[16];
    tmem_ld16(tr + c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int n = c0 + i;
      if (n < E) {
        const float x = v[i] + (p.bias ? __ldg(p.bias + n) : 0.f);
        if (lo) lo[n] = x;
        route_candidate(x, n, v[i], ei[i]);
      } else {
        v[i] = -INFINITY;
        ei[i] = INT_MAX;
      }
    }
    route_sort<16>(v, ei);
    route_merge_top<KM, 16>(lv, le, v, ei);
  }
  release();
  if (!real) return;
  float ex[KM];
  const float m = lv[0];
#pragma unroll
  for (int s = 0; s < KM; ++s) ex[s] = s < k ? expf(lv[s] - m) : 0.f;
  const float sum = route_weight_sum<KM>(ex, k);
  int32_t* hist = p.route_chunk + static_cast<size_t>(grow / kChunkTokens) * E;
  int32_t* oi = p.route_idx + static_cast<size_t>(grow) * k;
  float* ow = p.route_w + static_cast<size_t>(grow) * k;
#pragma unroll
  for (int s = 0; s < KM; ++s) {
    if (s < k) {
      int e = le[s];
      if (e >= E) {  // only reachable with NaN logits
        if (p.status) atomicCAS(p.status, 0, kDevBadValue);
        e = 0;
      }
      oi[s] = e;
      ow[s] = ex[s] / sum;
      atomicAdd(hist + e, 1);
    }
  }
}

// Epilogue with two accumulator buffers: every bf16-mode GEMM (and MXFP8 ones
// with 128-column tiles, whose output is bf16 as well; no instantiation).
template <int EPI, int SCH, bool MX>
__device__ __forceinline__ void gemm_epilogue(const GemmParams& p, uint32_t accf0, uint32_t acce0,
                                              uint32_t tmem_base, uint32_t s_warp, const WorkRange& wr,
                                              volatile int* abort_flag, int warp_e, int half, int lane) {
  constexpr bool kWide = epi_wide<MX, EPI, SCH>();
  constexpr int BN = gemm_bn<MX, EPI, SCH>();
  constexpr int BK = stage_k<MX>();
  // columns of the tile this warp stores (a half with two warps per quadrant)
  const int cbeg = kWide ? 128 * half : 0, cend = kWide ? cbeg + 128 : BN;
  int acc = 0;
  uint32_t aph = 0;
  EpiStager<epi_slots<MX, EPI, SCH>()> stg{s_warp, 0, lane};
  constexpr bool PAIR = sched_pair(SCH);
  // 2-SM mode: the accumulator is released on the even CTA's barrier
  const uint32_t acce_lead = PAIR ? mapa_shared(acce0, 0) : acce0;
  for (int w = wr.first; w < wr.count; w += wr.stride) {
    const TileInfo t = gemm_tile<EPI, SCH, BK, BN>(p, w, wr.rank);
    // Tile row held by this thread's TMEM lane: lane l of warp w is row 32w + l
    // of an M=128 accumulator; an M=64 accumulator keeps rows 16w..16w+15 in
    // lanes 0..15 of each warp (lanes 16..31 hold nothing of this tile).  A
    // pair's tile always has the M=128 layout: for a 64-row tail tile, warps
    // 2 and 3 hold rows of the next group, which they must not store.
    const bool m64l = t.m64 && !PAIR;
    const int wrows = m64l ? 16 : 32;
    const bool warp_live = !(PAIR && t.m64 && warp_e >= 2);
    const bool lane_ok = warp_live && lane < wrows;
    const int row = warp_e * wrows + lane;
    if constexpr (EPI == EPI_SWIGLU_BWD) {  // the saved a, b of this tile's rows: into L2 while the MMAs run
      if (lane_ok && row < t.rows_valid) {
        const char* ar = reinterpret_cast<const char*>(p.ab + (static_cast<long long>(t.row0) + row) * (2LL * p.I) + t.n0);
        const int lines = min(kBN, p.N - t.n0) / 64;
        for (int q = 0; q < lines; ++q) {
          prefetch_l2(ar + 128 * q);
          prefetch_l2(ar + 2LL * p.I + 128 * q);
        }
      }
    }
    const bool ok = mbar_wait(accf0 + 8 * acc, aph, abort_flag, p.status);
    if (!__all_sync(0xffffffffu, ok)) break;
    tc_fence_after();
    const uint32_t tr = tmem_base + (static_cast<uint32_t>(warp_e * 32) << 16) +
                        static_cast<uint32_t>(acc * BN);

    if constexpr (sched_wgrad(SCH)) {
      const int r0 = t.m0 + warp_e * 32;
      // 64 accumulator columns of this lane's row (zeros for an expert without rows)
      auto load64 = [&](int c0, float* v) {
        if (t.nkb > 0) {
          tmem_ld32(tr + c0, v);
          tmem_ld32(tr + c0 + 32, v + 32);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = 0.f;
        }
      };
      if (p.wgrad_f32) {  // fp32 weight gradients: two 32-column fp32 boxes per 64 columns
        for (int c0 = cbeg; c0 < cend && t.n0 + c0 < p.N; c0 += 64) {
          float v[64];
          load64(c0, v);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t box = stg.begin();
            stage_row_sw128_f32(box, lane, v + 32 * h);
            if (p.dense_rows > 0)
              stg.store2d(&p.tmO0, box, t.n0 + c0 + 32 * h, r0);
            else
              stg.store3d(&p.tmO0, box, t.n0 + c0 + 32 * h, r0, t.e);
          }
        }
      } else {
        for (int c0 = cbeg; c0 < cend && t.n0 + c0 < p.N; c0 += 64) {
          float v[64];
          load64(c0, v);
          const uint32_t box = stg.begin();
          stage_row_sw128(box, lane, v);
          if (p.dense_rows > 0)
            stg.store2d(&p.tmO0, box, t.n0 + c0, r0);
          else
            stg.store3d(&p.tmO0, box, t.n0 + c0, r0, t.e);
        }
      }
    } else {
      const bool real = lane_ok && row < t.rows_valid;
      const long long grow = static_cast<long long>(t.row0) + row;
      const int r0 = t.row0 + warp_e * wrows;
      const CUtensorMap* o0 = m64l ? &p.tmO0h : &p.tmO0;
      const CUtensorMap* o1 = m64l ? &p.tmO1h : &p.tmO1;
      if constexpr (EPI == EPI_ROUTE) {
        auto release = [&]() {  // frees the accumulator once the logits are read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce0 + 8 * acc);
        };
        if (p.route_k <= 8)
          epi_route<8>(p, tr, real, static_cast<int>(grow), release);
        else
          epi_route<kRouteMaxK>(p, tr, real, static_cast<int>(grow), release);
      } else if constexpr (EPI == EPI_F32_BIAS) {
        const bool in_mem = p.dense_rows > 0 ? real : lane_ok;
        float* o = reinterpret_cast<float*>(p.out) + grow * p.ldo;
        for (int c0 = 0; c0 < kBN && t.n0 + c0 < p.N; c0 += 16) {
          float v[16];
          tmem_ld16(tr + c0, v);
          tmem_ld_wait();
          if (in_mem) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int n = t.n0 + c0 + i;
              if (n < p.N) o[n] = v[i] + (p.bias ? __ldg(p.bias + n) : 0.f);
            }
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU_FWD) {
        for (int c0 = 0; c0 < kBN / 2 && t.n0 + c0 < p.N && warp_live; c0 += 64) {
          float a[64], b[64];
          tmem_ld32(tr + c0, a);
          tmem_ld32(tr + c0 + 32, a + 32);
          tmem_ld32(tr + kBN / 2 + c0, b);
          tmem_ld32(tr + kBN / 2 + c0 + 32, b + 32);
          tmem_ld_wait();
          if (!real) {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              a[i] = 0.f;
              b[i] = 0.f;
            }
          }
          if (p.store_ab) {
            stg.row64_2d(o0, a, t.n0 + c0, r0);
            stg.row64_2d(o0, b, p.I + t.n0 + c0, r0);
          }
#pragma unroll
          for (int i = 0; i < 64; ++i) a[i] = a[i] * sigmoidf_(a[i]) * b[i];
          stg.row64_2d(o1, a, t.n0 + c0, r0);
        }
      } else if constexpr (EPI == EPI_BF16) {
        float scale = 1.f;
        if (p.row_scale && p.dense_rows == 0 && lane_ok) scale = __ldg(p.row_scale + grow);
        if (!real) scale = 0.f;
        for (int c0 = 0; c0 < kBN && t.n0 + c0 < p.N && warp_live; c0 += 64) {
          float v[64];
          tmem_ld32(tr + c0, v);
          tmem_ld32(tr + c0 + 32, v + 32);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] *= scale;
          stg.row64_2d(o0, v, t.n0 + c0, r0);
        }
      } else {  // EPI_SWIGLU_BWD: direct row stores; a long K loop hides this epilogue
        const bool in_mem = p.dense_rows > 0 ? real : lane_ok;
        __nv_bfloat16* dadb = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * p.ldo;
        __nv_bfloat16* hg = reinterpret_cast<__nv_bfloat16*>(p.out2) + grow * p.ldo2;
        const __nv_bfloat16* abr = p.ab + grow * (2LL * p.I);
        float g = 1.f;
        if (in_mem && real && p.row_scale) g = __ldg(p.row_scale + grow);
        float dgp = 0.f;
        for (int c0 = 0; c0 < kBN && t.n0 + c0 < p.N; c0 += 16) {
          float dh[16];
          tmem_ld16(tr + c0, dh);
          tmem_ld_wait();
          if (in_mem) {
            float da[16], db[16], hv[16];
            if (real) {
              float a[16], b[16];
              load_bf16x16(abr + t.n0 + c0, a);
              load_bf16x16(abr + p.I + t.n0 + c0, b);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float sg = sigmoidf_(a[i]);
                const float silu = a[i] * sg;
                const float hh = silu * b[i];
                dgp += dh[i] * hh;
                const float dhs = g * dh[i];
                da[i] = dhs * b[i] * sg * (1.f + a[i] * (1.f - sg));
                db[i] = dhs * silu;
                hv[i] = g * hh;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                da[i] = 0.f;
                db[i] = 0.f;
                hv[i] = 0.f;
              }
            }
            store_bf16x16(dadb + t.n0 + c0, da);
            store_bf16x16(dadb + p.I + t.n0 + c0, db);
            store_bf16x16(hg + t.n0 + c0, hv);
          }
        }
        if (in_mem && p.out3) p.out3[grow * p.ldo3 + t.nt] = real ? dgp : 0.f;
      }
    }
    if constexpr (EPI != EPI_ROUTE) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && wr.rank != 0)
          mbar_arrive_remote(acce_lead + 8 * acc);
        else
          mbar_arrive(acce0 + 8 * acc);
      }
    }
    if (++acc == 2) {
      acc = 0;
      aph ^= 1;
    }
  }
  // every TMA store of this warp has finished before the CTA may exit
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

// ------------------------------------------------------------------ MXFP8 epilogue
// MXFP8 mode has one 256-column accumulator: the scale ring takes the other
// TMEM columns.  So that the next tile's MMAs need not wait for the whole
// epilogue, each warp first copies three quarters of its accumulator columns
// into spare TMEM columns (the stash), loads the last quarter, releases the
// accumulator and finishes from the stash while the tensor cores work on the
// next tile.  One epilogue warp per TMEM lane quadrant handles all 256
// columns, except in the SwiGLU backward, where two warps per quadrant split
// them (quad = warp index mod 4, half = which 128 columns).
constexpr uint32_t kStashCol = kSfTmemCol + kStages * kSfTmemStride;
constexpr int kStashCols = 192;
static_assert(kStashCol + kStashCols <= static_cast<uint32_t>(kTmemCols), "TMEM budget");

// Stores 32 floats of a row as bf16 (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  store_bf16x16(dst, *reinterpret_cast<const float(*)[16]>(v));
  store_bf16x16(dst + 16, *reinterpret_cast<const float(*)[16]>(v + 16));
}

// Quantization along the token rows of a 32-column chunk held one row per
// lane (v[i] = this lane's value in column i; the warp's 32 lanes are 32
// consecutive rows, one MX block).  The warp transposes 16 columns at a time
// through its 32 x 17 fp32 buffer; lane (c, h) takes rows 16h..16h+15 of
// column c, the two halves agree on the block maximum, and each writes 16
// codes of the transpose's row: dst + (16 pass + c) * ld + 16 h.  The E8M0
// code of chunk column j goes to sf[sf_off(j)].
template <class SfOff>
__device__ __forceinline__ void quant32_tok(const float* v, float* buf, uint8_t* dst, long long ld, uint8_t* sf,
                                            SfOff sf_off, int lane) {
  const int c = lane & 15, h = lane >> 4;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
    for (int i = 0; i < 16; ++i) buf[lane * 17 + i] = v[16 * pass + i];
    __syncwarp();
    float u[16], amax = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      u[r] = buf[(16 * h + r) * 17 + c];
      amax = fmaxf(amax, fabsf(u[r]));
    }
    __syncwarp();
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
    const int e = mx_scale_exp(amax);
    const float inv = mx_inv_scale(e);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = e4m3x2(u[4 * i] * inv, u[4 * i + 1] * inv) | (e4m3x2(u[4 * i + 2] * inv, u[4 * i + 3] * inv) << 16);
    *reinterpret_cast<uint4*>(dst + (16 * pass + c) * ld + 16 * h) = make_uint4(w[0], w[1], w[2], w[3]);
    if (h == 0) sf[sf_off(16 * pass + c)] = static_cast<uint8_t>(e + 127);
  }
}

template <int EPI, int SCH>
__device__ __forceinline__ void gemm_epilogue_mx(const GemmParams& p, uint32_t accf0, uint32_t acce0,
                                                 uint32_t tmem_base, uint32_t s_warp, float* buf, const WorkRange& wr,
                                                 volatile int* abort_flag, int quad, int half, int lane) {
  static_assert(EPI != EPI_F32_BIAS, "no fp32 epilogue in MXFP8 mode");
  uint32_t aph = 0;
  EpiStager<epi_slots<true, EPI, SCH>()> stg{s_warp, 0, lane};
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t acc = tmem_base + lane_off;
  // wide (SwiGLU backward): 96 stash columns per warp; otherwise 192
  const uint32_t stash = tmem_base + lane_off + kStashCol + half * (kStashCols / 2);
  const int row = quad * 32 + lane;  // MXFP8 groups are 128-row aligned: no 64-row tiles
  const int warp_e = quad;
  // SM pairs: each CTA's epilogue takes its own 128 rows (its m-tile of the
  // pair) and releases the accumulator on the even CTA's barrier
  constexpr bool PAIR = sched_pair(SCH);
  const uint32_t acce_lead = PAIR ? mapa_shared(acce0, 0) : acce0;
  for (int w = wr.first; w < wr.count; w += wr.stride) {
    const TileInfo t = gemm_tile<EPI, SCH, kBKmx>(p, w, wr.rank);
    if constexpr (EPI == EPI_SWIGLU_BWD) {  // the saved a, b of this warp's rows and columns: into L2 now
      const int c0 = t.n0 + 128 * half;
      if (row < t.rows_valid && c0 < p.N) {
        const char* ar = reinterpret_cast<const char*>(p.ab + (static_cast<long long>(t.row0) + row) * (2LL * p.I) + c0);
        prefetch_l2(ar);
        prefetch_l2(ar + 128);
        prefetch_l2(ar + 2LL * p.I);
        prefetch_l2(ar + 2LL * p.I + 128);
      }
    }
    const bool ok = mbar_wait(accf0, aph, abort_flag, p.status);
    if (!__all_sync(0xffffffffu, ok)) break;
    tc_fence_after();
    auto release = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && wr.rank != 0)
          mbar_arrive_remote(acce_lead);
        else
          mbar_arrive(acce0);
      }
      aph ^= 1;
    };

    if constexpr (EPI == EPI_BF16) {
      const bool have = SCH == SCHED_WGRAD ? t.nkb > 0 : true;
      float scale = 1.f;
      int r0;
      if constexpr (SCH == SCHED_WGRAD) {
        r0 = t.m0 + warp_e * 32;
      } else {
        r0 = t.row0 + warp_e * 32;
        if (p.row_scale && p.dense_rows == 0) scale = __ldg(p.row_scale + t.row0 + row);
        if (row >= t.rows_valid) scale = 0.f;
      }
      auto emit64 = [&](int c0, float* v) {
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] *= scale;
        const uint32_t box = stg.begin();
        stage_row_sw128(box, lane, v);
        if (SCH == SCHED_WGRAD && p.dense_rows == 0)
          stg.store3d(&p.tmO0, box, t.n0 + c0, r0, t.e);
        else
          stg.store2d(&p.tmO0, box, t.n0 + c0, r0);
      };
      if (have) {
        for (int c = 0; c < kStashCols && t.n0 + c < p.N; c += 96) tmem_copy96(stash + c, acc + c);
        tmem_st_wait();
      }
      float v[64];
      const bool tail = t.n0 + kStashCols < p.N;
      if (tail && have) {
        tmem_ld32(acc + kStashCols, v);
        tmem_ld32(acc + kStashCols + 32, v + 32);
        tmem_ld_wait();
      }
      release();
      if (tail) {
        if (!have) {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = 0.f;
        }
        emit64(kStashCols, v);
      }
      for (int c0 = 0; c0 < kStashCols && t.n0 + c0 < p.N; c0 += 64) {
        if (have) {
          tmem_ld32(stash + c0, v);
          tmem_ld32(stash + c0 + 32, v + 32);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = 0.f;
        }
        emit64(c0, v);
      }
    } else if constexpr (EPI == EPI_SWIGLU_FWD) {
      // accumulator: gate columns 0..127, up columns 128..255 of the tile's 128
      // h columns; stash: gate 0..95 -> +0, up 0..95 -> +96; h columns 96..127
      // are done before the release
      const bool real = row < t.rows_valid;
      const long long grow = static_cast<long long>(t.row0) + row;
      __nv_bfloat16* abw = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * p.ldo;
      uint32_t qword = 0;
      auto chunk = [&](int j, float* a, float* b) {  // h columns 32j..32j+31 of the tile
        if (!real) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = 0.f;
            b[i] = 0.f;
          }
        }
        if (p.store_ab) {
          store_bf16x32(abw + t.n0 + 32 * j, a);
          store_bf16x32(abw + p.I + t.n0 + 32 * j, b);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = a[i] * sigmoidf_(a[i]) * b[i];
        qword |= quant32_store(a, p.qout + grow * p.qld + t.n0 + 32 * j) << (8 * j);
      };
      tmem_copy96(stash, acc);
      tmem_copy96(stash + 96, acc + kBN / 2);
      tmem_st_wait();
      float a[32], b[32];
      tmem_ld32(acc + 96, a);
      tmem_ld32(acc + kBN / 2 + 96, b);
      tmem_ld_wait();
      release();
      chunk(3, a, b);
      for (int j = 0; j < 3; ++j) {
        tmem_ld32(stash + 32 * j, a);
        tmem_ld32(stash + 96 + 32 * j, b);
        tmem_ld_wait();
        chunk(j, a, b);
      }
      *reinterpret_cast<uint32_t*>(p.qsf + sf_word_offset(grow, t.n0 / 128, p.q_rb)) = qword;
    } else {  // EPI_SWIGLU_BWD
      // this warp: tile columns 128 half .. +127 (one 128-column scale group);
      // da, db quantized along the columns for the dgrad of gate/up (qout),
      // and da, db, g*h along the token rows for the weight gradients (qt, qt2)
      const int cw = 128 * half;
      const bool valid = t.n0 + cw < p.N;  // N is a multiple of 128
      const bool real = row < t.rows_valid;
      const long long grow = static_cast<long long>(t.row0) + row;
      const long long tok0 = static_cast<long long>(t.row0) + quad * 32;  // first row of the warp's block
      const __nv_bfloat16* abr = p.ab + grow * (2LL * p.I);
      const float g = (real && p.row_scale) ? __ldg(p.row_scale + grow) : 1.f;
      float dgp = 0.f;
      uint32_t wa = 0, wb = 0;  // column-quant scale words of da and db
      auto chunk = [&](int c0, const float* dh) {  // tile columns c0..c0+31
        float da[32], db[32], hv[32];
#pragma unroll
        for (int h16 = 0; h16 < 2; ++h16) {
          if (real) {
            float a[16], b[16];
            load_bf16x16(abr + t.n0 + c0 + 16 * h16, a);
            load_bf16x16(abr + p.I + t.n0 + c0 + 16 * h16, b);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float sg = sigmoidf_(a[i]);
              const float silu = a[i] * sg;
              const float hh = silu * b[i];
              const float d = dh[16 * h16 + i];
              dgp += d * hh;
              const float dhs = g * d;
              da[16 * h16 + i] = dhs * b[i] * sg * (1.f + a[i] * (1.f - sg));
              db[16 * h16 + i] = dhs * silu;
              hv[16 * h16 + i] = g * hh;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              da[16 * h16 + i] = 0.f;
              db[16 * h16 + i] = 0.f;
              hv[16 * h16 + i] = 0.f;
            }
          }
        }
        const int col = t.n0 + c0;
        const int j = (c0 / 32) & 3;
        wa |= quant32_store(da, p.qout + grow * p.qld + col) << (8 * j);
        wb |= quant32_store(db, p.qout + grow * p.qld + p.I + col) << (8 * j);
        quant32_tok(da, buf, p.qt + col * p.qt_ld + tok0, p.qt_ld, p.qt_sf,
                    [&](int jc) { return sf_byte_offset(col + jc, tok0, p.qt_rb); }, lane);
        quant32_tok(db, buf, p.qt + (p.I + col) * p.qt_ld + tok0, p.qt_ld, p.qt_sf,
                    [&](int jc) { return sf_byte_offset(p.I + col + jc, tok0, p.qt_rb); }, lane);
        quant32_tok(hv, buf, p.qt2 + col * p.qt2_ld + tok0, p.qt2_ld, p.qt2_sf,
                    [&](int jc) { return sf_byte_offset(col + jc, tok0, p.qt2_rb); }, lane);
      };
      float dh[32];
      if (valid) {
        tmem_copy96(stash, acc + cw);
        tmem_st_wait();
        tmem_ld32(acc + cw + 96, dh);
        tmem_ld_wait();
      }
      release();
      if (valid) {
        chunk(cw + 96, dh);
        for (int j = 0; j < 3; ++j) {
          tmem_ld32(stash + 32 * j, dh);
          tmem_ld_wait();
          chunk(cw + 32 * j, dh);
        }
        const int col = t.n0 + cw;
        *reinterpret_cast<uint32_t*>(p.qsf + sf_word_offset(grow, col / 128, p.q_rb)) = wa;
        *reinterpret_cast<uint32_t*>(p.qsf + sf_word_offset(grow, (p.I + col) / 128, p.q_rb)) = wb;
      }
      // router-weight gradient partials: one slot per (n-tile, column half)
      if (p.out3) p.out3[grow * p.ldo3 + 2 * t.nt + half] = (real && valid) ? dgp : 0.f;
    }
  }
  // every TMA store of this warp has finished before the CTA may exit
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

// ------------------------------------------------------------------ kernel
// The whole GEMM on one CTA (or CTA pair): barrier and TMEM set-up, the roles,
// and the teardown (TMEM freed).  Returns whether the CTA finished without an
// abort (a bounded wait that ran out).
template <int AM, int BMO, int EPI, int SCH, bool MX = false>
__device__ __forceinline__ bool tc_gemm_run(const GemmParams& p, uint8_t* smem_raw) {
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int ST = gemm_stages<MX, EPI, SCH>();
  constexpr int SB = stage_bytes<MX, EPI, SCH>();
  constexpr int kSfBytes = ST * sf_stage_bytes<MX, EPI, SCH>();
  constexpr int kStagingBytes = epi_warps<MX, EPI, SCH>() * epi_warp_bytes<MX, EPI, SCH>();
  const uint32_t s_tiles = smem_u32(smem);
  const uint32_t s_staging = s_tiles + ST * SB;
  const uint32_t s_sf = s_staging + kStagingBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ST * SB + kStagingBytes + kSfBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * ST;
  const uint32_t accf0 = empty0 + 8 * ST;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * ST + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  constexpr bool PAIR = sched_pair(SCH);
  constexpr int CG = PAIR ? 2 : 1;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf0 + 8 * i, 1);
      // 2-SM mode: the even CTA's counts both CTAs' epilogue warps
      mbar_init(acce0 + 8 * i, (PAIR ? 2 : 1) * epi_warps<MX, EPI, SCH>());
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB0);
    if (BMO == B_K_DUAL_N || BMO == B_MN_DUAL_K) tma_prefetch_desc(&p.tmB1);
    if (MX && PAIR) {
      tma_prefetch_desc(&p.tmSfA);
      tma_prefetch_desc(&p.tmSfB0);
      if (BMO == B_K_DUAL_N) tma_prefetch_desc(&p.tmSfB1);
    }
    // only the output maps this launch stores through (MXFP8 mode stores directly)
    if (!MX && (EPI == EPI_BF16 || EPI == EPI_SWIGLU_FWD)) {
      tma_prefetch_desc(&p.tmO0);
      if (!sched_wgrad(SCH)) tma_prefetch_desc(&p.tmO0h);
    }
    if (!MX && EPI == EPI_SWIGLU_FWD) {
      tma_prefetch_desc(&p.tmO1);
      tma_prefetch_desc(&p.tmO1h);
    }
  }
  if (warp == 2) {
    tmem_alloc<CG>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  // 2-SM mode: the peer's barriers are initialised before anything reaches them
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  WorkRange wr;
  if constexpr (PAIR) {
    wr.first = static_cast<int>(cluster_id_x());
    wr.stride = static_cast<int>(num_clusters_x());
    wr.count = gemm_num_tiles<EPI, SCH, gemm_bn<MX, EPI, SCH>()>(p);
    wr.rank = cluster_ctarank();
  } else {
    wr.first = blockIdx.x;
    wr.stride = gridDim.x;
    wr.count = gemm_num_tiles<EPI, SCH, gemm_bn<MX, EPI, SCH>()>(p);
    wr.rank = 0;
  }

  if (warp == 0) {
    gemm_producer<AM, BMO, EPI, SCH, MX>(p, s_tiles, s_sf, full0, empty0, wr, abort_flag, lane);
  } else if (warp == 1) {
    if (lane == 0)
      gemm_mma<AM, BMO, EPI, SCH, MX>(p, s_tiles, s_sf, full0, empty0, accf0, acce0, drain,
                                      tmem_base, wr, abort_flag);
  } else if (warp >= first_epi_warp<MX, EPI, SCH>()) {
    const int ew = warp - first_epi_warp<MX, EPI, SCH>();
    constexpr int kWarpBytes = epi_warp_bytes<MX, EPI, SCH>();
    if constexpr (epi_mx_stash<MX, EPI, SCH>())
      gemm_epilogue_mx<EPI, SCH>(p, accf0, acce0, tmem_base, s_staging + ew * kWarpBytes,
                                 reinterpret_cast<float*>(smem + ST * SB + ew * kWarpBytes),
                                 wr, abort_flag, warp & 3, ew >> 2, lane);
    else
      gemm_epilogue<EPI, SCH, MX>(p, accf0, acce0, tmem_base, s_staging + ew * kWarpBytes, wr, abort_flag,
                                  warp & 3, ew >> 2, lane);
  }
  tc_fence_before();
  __syncthreads();
  // 2-SM mode: neither CTA leaves (or frees TMEM) while the pair's MMAs or
  // signals may still reach it
  if constexpr (PAIR) cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
  }
  const bool ok = *abort_flag == 0;
  __syncthreads();
  return ok;
}

template <int AM, int BMO, int EPI, int SCH, bool MX = false>
__global__ void __launch_bounds__(gemm_threads<MX, EPI, SCH>(), 1) tc_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  tc_gemm_run<AM, BMO, EPI, SCH, MX>(p, smem_raw);
}

}  // namespace moe
