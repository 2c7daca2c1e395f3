// Host side of libmoe: argument checks, workspace carving, tensor maps and the
// launch sequence of the forward and backward passes.  Everything is enqueued
// on the caller's stream; the host never waits for the device.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "gemm_launch.cuh"
#include "moe_internal.h"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace moe {

int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64) {
    const int c = cache[dev].load();
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev < 64) cache[dev].store(n);
  return n;
}

cudaError_t launch_gemm(GemmKind kind, const GemmParams& p, int grid, cudaStream_t st) {
  if (kind == GK_ROUTER || kind == GK_GATEUP || kind == GK_DOWN) return launch_gemm_fwd(kind, p, grid, st);
  if (kind >= GK_MX_GATEUP) return launch_gemm_mx(kind, p, grid, st);
  return launch_gemm_bwd(kind, p, grid, st);
}

// ---------------------------------------------------------------- profiling
// Optional per-kernel timing (moe_profile_enable / moe_profile_report): each
// launch is bracketed by two CUDA events recorded on the launching stream.
enum ProfLabel : int {
  PL_ROUTER_GEMM, PL_TOPK, PL_CHUNK_SCAN, PL_SCATTER, PL_PERMUTE_X, PL_GATEUP_SHARED, PL_GATEUP_ROUTED,
  PL_DOWN_ROUTED, PL_DOWN_SHARED, PL_COMBINE, PL_DGRAD_DOWN_ROUTED, PL_DGRAD_DOWN_SHARED,
  PL_ROUTER_GRAD, PL_DGRAD_GATEUP_ROUTED, PL_DGRAD_GATEUP_SHARED, PL_UNPERMUTE, PL_ROUTER_WGRAD,
  PL_WGRAD_DOWN, PL_WGRAD_GATE, PL_WGRAD_UP, PL_WGRAD_SHARED_DOWN, PL_WGRAD_SHARED_GATE,
  PL_WGRAD_SHARED_UP, PL_PERMUTE_DY, PL_MX_WEIGHTS, PL_MX_QUANT_X, PL_MX_QUANT_DY, PL_ROUTE_FUSED, PL_COUNT
};
static const char* const kProfNames[PL_COUNT] = {
    "router_gemm", "topk_count", "chunk_scan", "scatter", "permute_x", "gateup_shared", "gateup_routed",
    "down_routed", "down_shared", "combine", "dgrad_down_routed", "dgrad_down_shared",
    "router_grad", "dgrad_gateup_routed", "dgrad_gateup_shared", "unpermute", "router_wgrad",
    "wgrad_down", "wgrad_gate", "wgrad_up", "wgrad_shared_down", "wgrad_shared_gate",
    "wgrad_shared_up", "permute_dy", "mx_quantize_weights", "mx_permute_quant_x", "mx_permute_quant_dy",
    "route_fused"};

struct ProfRecord {
  int label;
  int kernels;
  cudaEvent_t start, stop;
};
struct Profiler {
  std::mutex mu;
  std::atomic<bool> on{false};
  std::vector<ProfRecord> recs;
};
Profiler& profiler() {
  static Profiler p;
  return p;
}

int& extra_kernel_launches() {
  static thread_local int n = 0;
  return n;
}

template <class F>
moe_status prof_launch(int label, cudaStream_t st, F&& f) {
  Profiler& P = profiler();
  if (!P.on.load(std::memory_order_relaxed)) return f() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  cudaEvent_t a = nullptr, b = nullptr;
  if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return MOE_ERR_CUDA;
  cudaEventRecord(a, st);
  extra_kernel_launches() = 0;
  const cudaError_t e = f();
  cudaEventRecord(b, st);
  {
    std::lock_guard<std::mutex> g(P.mu);
    P.recs.push_back({label, 1 + extra_kernel_launches(), a, b});
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

constexpr size_t kAlign = 256;

struct Shape {
  int64_t T, d, I, E, k, S, Is, R, Rp, nchunk, nparts;
  int64_t ra;   // row alignment of the expert groups
  bool mx;      // MXFP8 routed experts
  bool replay;     // saved state without the routed activations; the backward recomputes them
  bool wgrad_f32;  // weight gradients written in fp32
};

// Carves 256-byte aligned sub-buffers from a base pointer (or only sizes them
// when base is null).
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <class T>
  T* take(int64_t n) {
    off = (off + kAlign - 1) / kAlign * kAlign;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += static_cast<size_t>(n) * sizeof(T);
    return p;
  }
};

struct Routing {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_start;
  int32_t* tile_start;
  int32_t* pair_start;  // prefix of the tile pairs per expert (run on SM pairs)
  int32_t* rem_start;   // prefix of the tiles per expert that run on one SM
  int32_t* perm_token;
  int32_t* route_row;
  int32_t* perm_token_pad;
  int32_t* route_row_pad;
  float* perm_w_pad;
};

void carve_routing(Carver& c, const Shape& s, Routing& r) {
  r.topk_idx = c.take<int32_t>(s.T * s.k);
  r.topk_w = c.take<float>(s.T * s.k);
  r.counts = c.take<int32_t>(s.E);
  r.offsets = c.take<int32_t>(s.E + 1);
  r.row_start = c.take<int32_t>(s.E + 1);
  r.tile_start = c.take<int32_t>(s.E + 1);
  r.pair_start = c.take<int32_t>(s.E + 1);
  r.rem_start = c.take<int32_t>(s.E + 1);
  r.perm_token = c.take<int32_t>(s.R);
  r.route_row = c.take<int32_t>(s.T * s.k);
  r.perm_token_pad = c.take<int32_t>(s.Rp);
  r.route_row_pad = c.take<int32_t>(s.T * s.k);
  r.perm_w_pad = c.take<float>(s.Rp);
}

// The forward's activations the backward needs: the x rows for the weight
// gradients of gate/up and the pre-activations a, b of the SwiGLU backward.
struct Acts {
  __nv_bfloat16* xp;   // [Rp, d] x rows in expert-grouped order (bf16 mode)
  __nv_bfloat16* ab;   // [Rp, 2I]
  __nv_bfloat16* abs;  // [T, 2Is]
  uint8_t *xt, *xt_sf;  // MXFP8: the x rows transposed, quantized along the tokens [d, Rp]
};
// The routed experts' activations (everything in Acts but abs).
void carve_routed_acts(Carver& c, const Shape& s, Acts& a) {
  const int64_t m = s.mx ? 1 : 0;
  a.xp = c.take<__nv_bfloat16>((1 - m) * s.Rp * s.d);
  a.ab = c.take<__nv_bfloat16>(s.Rp * 2 * s.I);
  a.xt = c.take<uint8_t>(m * s.Rp * s.d);
  a.xt_sf = c.take<uint8_t>(m * mx_sf_alloc(s.d, s.Rp));
}

// State moe_forward leaves for moe_backward: the routing, the shared expert's
// a and b, and the routed experts' activations unless they are replayed
// (MOE_FLAG_REPLAY; then those live in the backward workspace: the shared
// expert's are T rows against the routed T·k, not worth recomputing).
struct Saved {
  Routing rt;
  Acts act;
};
void carve_saved(void* base, const Shape& s, Saved& v, size_t* bytes) {
  Carver c(base);
  c.take<char>(kAlign);
  carve_routing(c, s, v.rt);
  v.act = Acts{};
  v.act.abs = c.take<__nv_bfloat16>(s.S ? s.T * 2 * s.Is : 0);
  if (!s.replay) carve_routed_acts(c, s, v.act);
  if (bytes) *bytes = c.off;
}

struct FwdWs {
  int* status;
  int* sync;  // [4] the fused routing launch's barrier counters and failure flag
  float* logits;
  int32_t* chunk_counts;
  int32_t* chunk_base;
  Routing rt;          // used when the caller keeps no saved state
  __nv_bfloat16* xp;   // [Rp, d], used when the caller keeps no saved state
  __nv_bfloat16* h;    // [Rp, I]
  __nv_bfloat16* hs;   // [T, Is]
  __nv_bfloat16* o;    // [Rp, d]
  __nv_bfloat16* ys;   // [T, d]
  // MXFP8: x rows and h rows as E4M3 codes + scales (h is not kept in bf16)
  uint8_t *xq, *xq_sf;  // [Rp, d]
  uint8_t *hq, *hq_sf;  // [Rp, I]
};
void carve_fwd(void* base, const Shape& s, FwdWs& w, size_t* bytes) {
  Carver c(base);
  w.status = c.take<int>(kAlign / sizeof(int));
  w.sync = c.take<int>(4);
  w.logits = c.take<float>(s.T * s.E);
  w.chunk_counts = c.take<int32_t>(s.nchunk * s.E);
  w.chunk_base = c.take<int32_t>(s.nchunk * s.E);
  carve_routing(c, s, w.rt);
  w.xp = c.take<__nv_bfloat16>(s.mx ? 0 : s.Rp * s.d);
  w.h = c.take<__nv_bfloat16>(s.mx ? 0 : s.Rp * s.I);
  w.hs = c.take<__nv_bfloat16>(s.S ? s.T * s.Is : 0);
  w.o = c.take<__nv_bfloat16>(s.Rp * s.d);
  w.ys = c.take<__nv_bfloat16>(s.S ? s.T * s.d : 0);
  const int64_t m = s.mx ? 1 : 0;
  w.xq = c.take<uint8_t>(m * s.Rp * s.d);
  w.xq_sf = c.take<uint8_t>(m * mx_sf_alloc(s.Rp, s.d));
  w.hq = c.take<uint8_t>(m * s.Rp * s.I);
  w.hq_sf = c.take<uint8_t>(m * mx_sf_alloc(s.Rp, s.I));
  if (bytes) *bytes = c.off;
}

struct BwdWs {
  int* status;
  __nv_bfloat16* dyp;    // [Rp, d] dy rows in expert-grouped order
  __nv_bfloat16* dadb;   // [Rp, 2I]
  __nv_bfloat16* hg;     // [Rp, I]
  float* dg_part;        // [Rp, nparts]
  __nv_bfloat16* dadbs;  // [T, 2Is]
  __nv_bfloat16* hs;     // [T, Is]
  float* dl_tk;          // [T, k]
  float* dl_row;         // [Rp]
  __nv_bfloat16* dxp;    // [Rp, d]
  __nv_bfloat16* dxs;    // [T, d]
  // MXFP8: E4M3 codes + scales of the GEMM operands: *q are the expert-grouped
  // rows quantized along their columns (dgrad operands); *t are transposes
  // quantized along the token rows (K-major weight-gradient operands).
  uint8_t *dyq, *dyq_sf;      // [Rp, d]
  uint8_t *dadbq, *dadbq_sf;  // [Rp, 2I]
  uint8_t *dyt, *dyt_sf;      // [d, Rp]
  uint8_t *dadbt, *dadbt_sf;  // [2I, Rp]
  uint8_t *hgt, *hgt_sf;      // [I, Rp]
  Acts act;                   // MOE_FLAG_REPLAY: the recomputed activations
};
void carve_bwd(void* base, const Shape& s, BwdWs& w, size_t* bytes) {
  Carver c(base);
  w.status = c.take<int>(kAlign / sizeof(int));
  const int64_t bf = s.mx ? 0 : 1;  // bf16 intermediates that MXFP8 mode does not keep
  w.dyp = c.take<__nv_bfloat16>(bf * s.Rp * s.d);
  w.dadb = c.take<__nv_bfloat16>(bf * s.Rp * 2 * s.I);
  w.hg = c.take<__nv_bfloat16>(bf * s.Rp * s.I);
  w.dg_part = c.take<float>(s.Rp * s.nparts);
  w.dadbs = c.take<__nv_bfloat16>(s.S ? s.T * 2 * s.Is : 0);
  w.hs = c.take<__nv_bfloat16>(s.S ? s.T * s.Is : 0);
  w.dl_tk = c.take<float>(s.T * s.k);
  w.dl_row = c.take<float>(s.Rp);
  w.dxp = c.take<__nv_bfloat16>(s.Rp * s.d);
  w.dxs = c.take<__nv_bfloat16>(s.S ? s.T * s.d : 0);
  const int64_t m = s.mx ? 1 : 0;
  w.dyq = c.take<uint8_t>(m * s.Rp * s.d);
  w.dyq_sf = c.take<uint8_t>(m * mx_sf_alloc(s.Rp, s.d));
  w.dadbq = c.take<uint8_t>(m * s.Rp * 2 * s.I);
  w.dadbq_sf = c.take<uint8_t>(m * mx_sf_alloc(s.Rp, 2 * s.I));
  w.dyt = c.take<uint8_t>(m * s.Rp * s.d);
  w.dyt_sf = c.take<uint8_t>(m * mx_sf_alloc(s.d, s.Rp));
  w.dadbt = c.take<uint8_t>(m * s.Rp * 2 * s.I);
  w.dadbt_sf = c.take<uint8_t>(m * mx_sf_alloc(2 * s.I, s.Rp));
  w.hgt = c.take<uint8_t>(m * s.Rp * s.I);
  w.hgt_sf = c.take<uint8_t>(m * mx_sf_alloc(s.I, s.Rp));
  w.act = Acts{};
  if (s.replay) carve_routed_acts(c, s, w.act);
  if (bytes) *bytes = c.off;
}

// MXFP8 copies of the routed expert weights (E4M3 codes + E8M0 scales in the
// tcgen05.cp block order), one per GEMM orientation:
//   wg/wu  [E*I, d]  W_gate, W_up quantized along d          (gate/up forward)
//   wd     [E*d, I]  W_down quantized along I                (down forward)
//   wdt    [E*I, d]  W_down^T per expert, along d            (dgrad of down)
//   wgut   [E*d, 2I] [W_gate; W_up]^T per expert, along 2I   (dgrad of gate/up)
struct MxWeights {
  uint8_t *wg, *wg_sf, *wu, *wu_sf, *wd, *wd_sf, *wdt, *wdt_sf, *wgut, *wgut_sf;
};
void carve_mx(void* base, const Shape& s, MxWeights& m, size_t* bytes) {
  Carver c(base);
  m.wg = c.take<uint8_t>(s.E * s.I * s.d);
  m.wg_sf = c.take<uint8_t>(mx_sf_alloc(s.E * s.I, s.d));
  m.wu = c.take<uint8_t>(s.E * s.I * s.d);
  m.wu_sf = c.take<uint8_t>(mx_sf_alloc(s.E * s.I, s.d));
  m.wd = c.take<uint8_t>(s.E * s.d * s.I);
  m.wd_sf = c.take<uint8_t>(mx_sf_alloc(s.E * s.d, s.I));
  m.wdt = c.take<uint8_t>(s.E * s.I * s.d);
  m.wdt_sf = c.take<uint8_t>(mx_sf_alloc(s.E * s.I, s.d));
  m.wgut = c.take<uint8_t>(s.E * s.d * 2 * s.I);
  m.wgut_sf = c.take<uint8_t>(mx_sf_alloc(s.E * s.d, 2 * s.I));
  if (bytes) *bytes = c.off;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Workspaces and the saved state: their sub-buffers take 32-byte vector accesses.
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

moe_status check_config(const moe_config* cfg, Shape& s) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (cfg->T < 0 || cfg->d <= 0 || cfg->I <= 0 || cfg->E <= 0 || cfg->top_k <= 0 ||
      cfg->n_shared < 0 || (cfg->n_shared && cfg->I_shared <= 0))
    return MOE_ERR_INVALID_ARG;
  if (cfg->precision != MOE_BF16 && cfg->precision != MOE_MXFP8) return MOE_ERR_UNSUPPORTED;
  if (cfg->precision == MOE_MXFP8 && (cfg->d % 128 || cfg->I % 128)) return MOE_ERR_UNSUPPORTED;
  if (cfg->flags & ~(MOE_FLAG_REPLAY | MOE_FLAG_WGRAD_FP32)) return MOE_ERR_UNSUPPORTED;
  if (cfg->precision == MOE_MXFP8 && (cfg->flags & MOE_FLAG_WGRAD_FP32)) return MOE_ERR_UNSUPPORTED;
  if (cfg->E > kMaxExperts || cfg->top_k > kMaxTopK || cfg->top_k > cfg->E) return MOE_ERR_UNSUPPORTED;
  if (cfg->n_shared > 1) return MOE_ERR_UNSUPPORTED;
  if (cfg->d % 64 || cfg->I % 64 || (cfg->n_shared && cfg->I_shared % 64)) return MOE_ERR_UNSUPPORTED;
  s.T = cfg->T;
  s.d = cfg->d;
  s.I = cfg->I;
  s.E = cfg->E;
  s.k = cfg->top_k;
  s.S = cfg->n_shared;
  s.Is = cfg->n_shared ? cfg->I_shared : 0;
  s.R = s.T * s.k;
  s.mx = cfg->precision == MOE_MXFP8;
  s.replay = (cfg->flags & MOE_FLAG_REPLAY) != 0;
  s.wgrad_f32 = (cfg->flags & MOE_FLAG_WGRAD_FP32) != 0;
  s.ra = s.mx ? kRowAlignMx : kRowAlign;
  s.Rp = s.R + s.E * (s.ra - 1);
  if (s.mx) s.Rp = (s.Rp + kRowAlignMx - 1) / kRowAlignMx * kRowAlignMx;  // whole scale blocks
  s.nchunk = (s.T + kChunkTokens - 1) / kChunkTokens;
  // router-weight gradient partials per row: one per n-tile of the SwiGLU
  // backward (two in MXFP8 mode, whose epilogue splits a tile's columns)
  s.nparts = (s.mx ? 2 : 1) * ((s.I + kBN - 1) / kBN);
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (s.Rp >= lim || s.T >= lim || s.d >= lim || s.I * s.E >= lim || s.d * s.E >= lim)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                        \
  do {                                       \
    const moe_status st__ = (expr);          \
    if (st__ != MOE_OK) return st__;         \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))
#define MOE_LAUNCH(label, stream, expr) MOE_TRY(prof_launch((label), (stream), [&]() { return (expr); }))

void zero_params(GemmParams& p) { memset(static_cast<void*>(&p), 0, sizeof(p)); }

// Tensor map over a row-major bf16 matrix [rows, cols] (pitch = cols).
moe_status tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  if (!make_tmap_bf16(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                      static_cast<uint64_t>(cols), box_cols, box_rows))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// E4M3 K-major operand [rows, cols] (K = cols), boxes of 128 columns x box_rows.
moe_status qmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
  if (!make_tmap_u8(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                    static_cast<uint32_t>(box_rows)))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Persistent GEMM grid: one CTA per SM, fewer when there are fewer tiles.  The
// environment variable MOE_GRID_LIMIT caps it further (used to check that
// results do not depend on the grid size).
// MN-major operand map: one box = box_chunks 64-column chunks of 64 K-rows.
moe_status mnmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_chunks) {
  if (!make_tmap_mn3d(m, base, static_cast<uint64_t>(rows), static_cast<uint64_t>(cols), 64,
                      static_cast<uint32_t>(box_chunks)))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// The bf16 GEMMs other than the router projection load B in halves: 128-row
// boxes (K-major) or two 64-column chunks (MN-major); see launch_rows_two_pass
// and launch_wgrad_two_pass.
// Output map: boxes of 64 columns x 32 rows (one epilogue warp's staging box).
moe_status omap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  return tmap(m, base, rows, cols, 64, 32);
}
// Output maps of a grouped GEMM: 32-row boxes and 16-row boxes (for the
// 64-row tail tiles).
moe_status omap2(CUtensorMap* m32, CUtensorMap* m16, const void* base, int64_t rows, int64_t cols) {
  MOE_TRY(tmap(m32, base, rows, cols, 64, 32));
  return tmap(m16, base, rows, cols, 64, 16);
}

// fp32 output maps (the weight gradients with MOE_FLAG_WGRAD_FP32): boxes of
// 32 columns x 32 rows, 128 bytes per box row as in the bf16 maps.
moe_status omap_f32(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  return make_tmap_f32(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), 32, 32) ? MOE_OK
                                                                                                  : MOE_ERR_CUDA;
}
moe_status omap3_f32(CUtensorMap* m, const void* base, int64_t G, int64_t rows, int64_t cols) {
  return make_tmap_f32_3d(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                          static_cast<uint64_t>(G), 32, 32)
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// Per-expert output [G, rows, cols]: a box never crosses into the next expert.
moe_status omap3(CUtensorMap* m, const void* base, int64_t G, int64_t rows, int64_t cols) {
  if (!make_tmap_bf16_3d(m, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                         static_cast<uint64_t>(G), 64, 32))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int grid_for(int64_t max_tiles) {
  int sms = device_sm_count();
  if (const char* lim = getenv("MOE_GRID_LIMIT")) {
    const int v = atoi(lim);
    if (v > 0 && v < sms) sms = v;
  }
  if (max_tiles < 1) max_tiles = 1;
  return static_cast<int>(max_tiles < sms ? max_tiles : sms);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The routed weight gradients reduce over each expert's rows: with fewer than
// 384 per expert on average they run on one SM per tile rather than on SM
// pairs (measured at the DSV3 shape: 16 rows, pairs 1.70 ms against 1.45 on
// one SM per gradient; 512 rows, pairs 2.97 against 3.36 ms), and with fewer
// than 128 with eight epilogue warps (64 rows: 1.45-1.53 -> 1.27-1.29 ms per
// gradient; 256 rows: 2.02-2.08 -> 2.39-2.63 ms, so not there).
int wgrad_mode(const Shape& s) { return s.R < 128 * s.E ? 2 : (s.R < 384 * s.E ? 1 : 0); }

// ---------------------------------------------------------------- routing
// The routing runs as one persistent launch (route_fused.cu: router GEMM with
// the top-k in its epilogue, scan and scatter) where it applies: logits
// computed here, E <= 256, top_k <= 16, and a workspace with its sync words.
// Otherwise, or with the environment variable MOE_ROUTING_SEPARATE set (the
// tests compare the two bitwise), the separate kernels run.  zero_routing: the
// routing arrays rt points into are one block (the saved state's or the
// workspace's), zeroed before the fused launch so that a launch cut short by a
// timeout leaves only in-range indices for the kernels after it.
bool fused_routing_enabled() {
  const char* v = getenv("MOE_ROUTING_SEPARATE");
  return !(v && v[0] && v[0] != '0');
}

moe_status run_routing(const Shape& s, const void* x, const void* W_router, const float* bias,
                       const float* logits_in, float* logits, const Routing& rt,
                       int32_t* chunk_counts, int32_t* chunk_base, int* status, cudaStream_t st,
                       int* sync = nullptr, bool zero_routing = false, bool keep_logits = true) {
  const float* lg = logits_in;
  GemmParams p;
  zero_params(p);
  if (!lg) {
    MOE_TRY(tmap(&p.tmA, x, s.T, s.d, 64, kBM));
    MOE_TRY(tmap(&p.tmB0, W_router, s.E, s.d, 64, kBN));
    p.dense_rows = static_cast<int>(s.T);
    p.N = static_cast<int>(s.E);
    p.K = static_cast<int>(s.d);
    p.out = logits;
    p.ldo = s.E;
    p.bias = bias;
    p.status = status;
    // Test hook for the device-side failure path: with MOE_DEBUG_STALL_ROUTER
    // set, the router projection's first stage waits for 16 bytes that never
    // come; its bounded waits run out (about 4 s each) and the launch records
    // MOE_ERR_DEVICE_TIMEOUT instead of hanging.
    if (const char* v = getenv("MOE_DEBUG_STALL_ROUTER"))
      if (v[0] && v[0] != '0') p.debug_extra_tx = 16;
  }
  if (!lg && sync && fused_routing_enabled() && route_fused_supported(s.E, s.k)) {
    const int nchunk = static_cast<int>(s.nchunk);
    MOE_CUDA(cudaMemsetAsync(chunk_counts, 0, static_cast<size_t>(s.nchunk * s.E) * sizeof(int32_t), st));
    MOE_CUDA(cudaMemsetAsync(sync, 0, 4 * sizeof(int), st));
    if (zero_routing) {
      const char* beg = reinterpret_cast<const char*>(rt.topk_idx);
      const char* end = reinterpret_cast<const char*>(rt.perm_w_pad + s.Rp);
      MOE_CUDA(cudaMemsetAsync(rt.topk_idx, 0, static_cast<size_t>(end - beg), st));
    }
    p.out = keep_logits ? logits : nullptr;  // the fused launch writes logits only when asked
    p.route_idx = rt.topk_idx;
    p.route_w = rt.topk_w;
    p.route_chunk = chunk_counts;
    p.route_k = static_cast<int>(s.k);
    const ScatterArgs sc{rt.topk_idx, rt.topk_w, static_cast<int>(s.T), static_cast<int>(s.E), static_cast<int>(s.k),
                         static_cast<int>(s.ra), chunk_base, rt.counts, rt.offsets, rt.row_start, rt.tile_start,
                         rt.pair_start, rt.rem_start, rt.perm_token, rt.route_row, rt.perm_token_pad,
                         rt.route_row_pad, rt.perm_w_pad};
    // Test hook: with MOE_DEBUG_STALL_COUNTER set, the first grid barrier waits
    // for one arrival more than the grid has; every CTA's bounded wait runs out
    // and the launch records MOE_ERR_DEVICE_TIMEOUT.
    int extra = 0;
    if (const char* v = getenv("MOE_DEBUG_STALL_COUNTER"))
      if (v[0] && v[0] != '0') extra = 1;
    // as many CTAs as the widest stage has work for: row tiles of the GEMM,
    // chunks of the scatter, warps of the scan (eight experts per CTA)
    const int grid = grid_for(std::max<int64_t>(std::max<int64_t>(cdiv(s.T, kBM), s.nchunk), cdiv(s.E, 8)));
    cudaError_t e = cudaSuccess;
    const moe_status ms = prof_launch(PL_ROUTE_FUSED, st, [&]() {
      e = launch_route_fused(p, sc, chunk_counts, chunk_base, nchunk, status, sync, extra, grid, st);
      return e;
    });
    if (ms == MOE_OK) return MOE_OK;
    // a grid that cannot be resident at once (another context holding SMs):
    // the separate kernels below
    if (e != cudaErrorCooperativeLaunchTooLarge) return MOE_ERR_CUDA;
    (void)cudaGetLastError();
    p.out = logits;
  }
  if (!lg) {
    MOE_LAUNCH(PL_ROUTER_GEMM, st, launch_gemm(GK_ROUTER, p, grid_for(cdiv(s.T, kBM) * cdiv(s.E, kBN)), st));
    lg = logits;
  }
  MOE_LAUNCH(PL_TOPK, st, launch_topk_count(lg, static_cast<int>(s.T), static_cast<int>(s.E), static_cast<int>(s.k),
                             rt.topk_idx, rt.topk_w, chunk_counts, status, st));
  MOE_LAUNCH(PL_CHUNK_SCAN, st, launch_chunk_scan(chunk_counts, static_cast<int>(s.nchunk), static_cast<int>(s.E),
                             chunk_base, rt.counts, st));
  MOE_LAUNCH(PL_SCATTER, st, launch_scatter(rt.topk_idx, rt.topk_w, static_cast<int>(s.T), static_cast<int>(s.E),
                          static_cast<int>(s.k), static_cast<int>(s.ra), chunk_base, rt.counts, rt.offsets, rt.row_start,
                          rt.tile_start, rt.pair_start, rt.rem_start, rt.perm_token, rt.route_row, rt.perm_token_pad,
                          rt.route_row_pad, rt.perm_w_pad, st));
  return MOE_OK;
}

moe_status check_weights(const Shape& s, const moe_weights* w, bool need_router) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (need_router && (!w->W_router || !aligned16(w->W_router))) return MOE_ERR_INVALID_ARG;
  const void* req[] = {w->W_gate, w->W_up, w->W_down};
  for (const void* p : req)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (s.S) {
    const void* sh[] = {w->Ws_gate, w->Ws_up, w->Ws_down};
    for (const void* p : sh)
      if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (s.mx && (!w->mxfp8 || (reinterpret_cast<uintptr_t>(w->mxfp8) & 255u))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Sets the MXFP8 operand scales of a GEMM: A's scales with A's row count,
// B's (one or two stacks) with B's row count.
void set_mx_scales(GemmParams& p, const uint8_t* sfa, int64_t a_rows, const uint8_t* sfb0,
                   const uint8_t* sfb1, int64_t b_rows) {
  p.sfa = sfa;
  p.sfa_rb = cdiv(a_rows, 128);
  p.sfb0 = sfb0;
  p.sfb1 = sfb1;
  p.sfb_rb = cdiv(b_rows, 128);
}
// The same scales for the row GEMMs, which run partly on SM pairs: also the
// tensor maps over the scale arrays (K = the reduction length) that the pairs
// load them through: 512-byte boxes for A and for each stack of a dual-N B,
// 1024-byte ones (two 128-row blocks) for a single B.
moe_status set_mx_row_scales(GemmParams& p, const uint8_t* sfa, int64_t a_rows, const uint8_t* sfb0,
                             const uint8_t* sfb1, int64_t b_rows, int64_t K) {
  set_mx_scales(p, sfa, a_rows, sfb0, sfb1, b_rows);
  if (!make_tmap_bytes(&p.tmSfA, sfa, mx_sf_alloc(a_rows, K), 2) ||
      !make_tmap_bytes(&p.tmSfB0, sfb0, mx_sf_alloc(b_rows, K), sfb1 ? 2 : 4) ||
      (sfb1 && !make_tmap_bytes(&p.tmSfB1, sfb1, mx_sf_alloc(b_rows, K), 2)))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Routed gate/up of the forward in MXFP8 mode (blog section "MXFP8 support"):
// on the quantized x rows xq, the SwiGLU epilogue writing h as E4M3 + scales
// (hq) and, when act is given, the a and b rows for the backward.
moe_status gateup_routed_mx(const Shape& s, const moe_weights* wts, const Routing& rt, const Acts* act,
                            const uint8_t* xq, const uint8_t* xq_sf, uint8_t* hq, uint8_t* hq_sf, int* status,
                            cudaStream_t st) {
  MxWeights m;
  carve_mx(const_cast<void*>(wts->mxfp8), s, m, nullptr);
  GemmParams p;
  zero_params(p);
  MOE_TRY(qmap(&p.tmA, xq, s.Rp, s.d, kBM));
  MOE_TRY(qmap(&p.tmB0, m.wg, s.E * s.I, s.d, kBN / 2));
  MOE_TRY(qmap(&p.tmB1, m.wu, s.E * s.I, s.d, kBN / 2));
  MOE_TRY(set_mx_row_scales(p, xq_sf, s.Rp, m.wg_sf, m.wu_sf, s.E * s.I, s.d));
  p.num_groups = static_cast<int>(s.E);
  p.row_start = rt.row_start;
  p.tile_start = rt.tile_start;
  p.pair_start = rt.pair_start;
  p.rem_start = rt.rem_start;
  p.counts = rt.counts;
  p.N = static_cast<int>(s.I);
  p.K = static_cast<int>(s.d);
  p.b_group_rows = static_cast<int>(s.I);
  if (act) {  // a and b rows kept for the backward (direct row stores)
    p.out = act->ab;
    p.ldo = 2 * s.I;
    p.store_ab = 1;
  }
  p.I = static_cast<int>(s.I);
  p.qout = hq;
  p.qld = s.I;
  p.qsf = hq_sf;
  p.q_rb = cdiv(s.Rp, 128);
  p.status = status;
  MOE_LAUNCH(PL_GATEUP_ROUTED, st, launch_gemm(GK_MX_GATEUP, p, grid_for(cdiv(s.Rp, kBM) * cdiv(s.I, kBN / 2)), st));
  return MOE_OK;
}

// Routed down projection in MXFP8 mode, on the quantized h rows, scaled by
// the router weight of each row.
moe_status down_routed_mx(const Shape& s, const moe_weights* wts, const Routing& rt, const FwdWs& w,
                          cudaStream_t st) {
  MxWeights m;
  carve_mx(const_cast<void*>(wts->mxfp8), s, m, nullptr);
  GemmParams p;
  zero_params(p);
  MOE_TRY(qmap(&p.tmA, w.hq, s.Rp, s.I, kBM));
  MOE_TRY(qmap(&p.tmB0, m.wd, s.E * s.d, s.I, kBN / 2));
  MOE_TRY(set_mx_row_scales(p, w.hq_sf, s.Rp, m.wd_sf, nullptr, s.E * s.d, s.I));
  p.num_groups = static_cast<int>(s.E);
  p.row_start = rt.row_start;
  p.tile_start = rt.tile_start;
  p.pair_start = rt.pair_start;
  p.rem_start = rt.rem_start;
  p.counts = rt.counts;
  p.N = static_cast<int>(s.d);
  p.K = static_cast<int>(s.I);
  p.b_group_rows = static_cast<int>(s.d);
  MOE_TRY(omap(&p.tmO0, w.o, s.Rp, s.d));
  p.row_scale = rt.perm_w_pad;
  p.status = w.status;
  MOE_LAUNCH(PL_DOWN_ROUTED, st, launch_gemm(GK_MX_DOWN, p, grid_for(cdiv(s.Rp, kBM) * cdiv(s.d, kBN)), st));
  return MOE_OK;
}

// Buffers the forward's first half writes besides the activations it keeps.
struct GateUpOut {
  __nv_bfloat16* xp;    // bf16 mode: [Rp, d] x rows, when no activations are kept
  __nv_bfloat16* h;     // bf16 mode: [Rp, I] SwiGLU output
  bool shared;          // also run the shared expert's gate/up (when there is one)
  __nv_bfloat16* hs;    // [T, Is] shared expert's SwiGLU output
  __nv_bfloat16* abs;   // [T, 2Is] shared expert's a and b, or null when not kept
  uint8_t *xq, *xq_sf;  // MXFP8: [Rp, d] x rows quantized along d
  uint8_t *hq, *hq_sf;  // MXFP8: [Rp, I] h quantized along I
  int* status;
};

// The forward up to the SwiGLU activation: dispatch of x (quantized on the
// way in MXFP8 mode) and the gate/up projections with the SwiGLU epilogue,
// shared (if o.shared) and routed.  act: where the routed activations the
// backward needs go (the x rows, a and b), or null in inference.  The backward
// runs the routed part again when the saved state holds only the routing and
// the shared expert's a and b (forward activation replay).
moe_status forward_gateup(const Shape& s, const void* x, const moe_weights* wts, const Routing& rt,
                          const Acts* act, const GateUpOut& o, cudaStream_t st) {
  const int T = static_cast<int>(s.T), d = static_cast<int>(s.d), I = static_cast<int>(s.I);
  const int E = static_cast<int>(s.E);
  // dispatch: x rows into expert-grouped order (zeros in padding rows); in
  // MXFP8 mode quantized on the way, the bf16 copy kept only for training
  __nv_bfloat16* xp = act ? act->xp : o.xp;
  if (s.mx)  // along d for gate/up; in training also along the tokens for dW_gate, dW_up
    MOE_LAUNCH(PL_MX_QUANT_X, st, launch_mx_dispatch(static_cast<const __nv_bfloat16*>(x), d, T, static_cast<int>(s.k), E,
                                                     rt.perm_token_pad, rt.route_row_pad, rt.row_start, rt.counts, s.Rp,
                                                     d, o.xq, o.xq_sf, act ? act->xt : nullptr,
                                                     act ? act->xt_sf : nullptr, st));
  else
    MOE_LAUNCH(PL_PERMUTE_X, st, launch_scatter_rows(static_cast<const __nv_bfloat16*>(x), rt.route_row_pad,
                                                    rt.row_start, rt.counts, T, E, d, static_cast<int>(s.k), xp, st));
  // shared expert gate/up + SwiGLU (dense rows of x)
  if (s.S && o.shared) {
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, x, s.T, s.d, 64, kBM));
    MOE_TRY(tmap(&p.tmB0, wts->Ws_gate, s.Is, s.d, 64, kBN / 2));
    MOE_TRY(tmap(&p.tmB1, wts->Ws_up, s.Is, s.d, 64, kBN / 2));
    p.dense_rows = T;
    p.N = static_cast<int>(s.Is);
    p.K = d;
    MOE_TRY(omap(&p.tmO1, o.hs, s.T, s.Is));
    if (o.abs)
      MOE_TRY(omap(&p.tmO0, o.abs, s.T, 2 * s.Is));
    else
      p.tmO0 = p.tmO1;  // a and b are not kept in inference
    p.tmO0h = p.tmO0;  // dense rows: no tail tiles
    p.tmO1h = p.tmO1;
    p.store_ab = o.abs ? 1 : 0;
    p.I = static_cast<int>(s.Is);
    p.status = o.status;
    // Test hook for the failure path of the SM-pair kernels: with
    // MOE_DEBUG_STALL_PAIR set, the even CTA of every pair of the shared
    // expert's gate/up waits for 16 bytes that never come; both CTAs' bounded
    // waits run out and the launch records MOE_ERR_DEVICE_TIMEOUT.
    if (const char* v = getenv("MOE_DEBUG_STALL_PAIR"))
      if (v[0] && v[0] != '0') p.debug_extra_tx = 16;
    MOE_LAUNCH(PL_GATEUP_SHARED, st, launch_gemm(GK_GATEUP, p, grid_for(cdiv(s.T, kBM) * cdiv(s.Is, kBN / 2)), st));
  }
  if (s.mx) return gateup_routed_mx(s, wts, rt, act, o.xq, o.xq_sf, o.hq, o.hq_sf, o.status, st);
  // routed gate/up + SwiGLU over the expert-grouped rows
  GemmParams p;
  zero_params(p);
  MOE_TRY(tmap(&p.tmA, xp, s.Rp, s.d, 64, kBM));
  MOE_TRY(tmap(&p.tmB0, wts->W_gate, s.E * s.I, s.d, 64, kBN / 2));
  MOE_TRY(tmap(&p.tmB1, wts->W_up, s.E * s.I, s.d, 64, kBN / 2));
  p.num_groups = E;
  p.row_start = rt.row_start;
  p.counts = rt.counts;
  p.N = I;
  p.K = d;
  p.b_group_rows = I;
  MOE_TRY(omap2(&p.tmO1, &p.tmO1h, o.h, s.Rp, s.I));
  if (act) {
    MOE_TRY(omap2(&p.tmO0, &p.tmO0h, act->ab, s.Rp, 2 * s.I));
  } else {
    p.tmO0 = p.tmO1;  // a and b are not kept in inference
    p.tmO0h = p.tmO1h;
  }
  p.tile_start = rt.tile_start;
  p.pair_start = rt.pair_start;
  p.rem_start = rt.rem_start;
  p.store_ab = act ? 1 : 0;
  p.I = I;
  p.status = o.status;
  MOE_LAUNCH(PL_GATEUP_ROUTED, st, launch_gemm(GK_GATEUP, p, grid_for(cdiv(s.Rp, kBM) * cdiv(s.I, kBN / 2)), st));
  return MOE_OK;
}

// Weight gradients of the routed experts in MXFP8 mode.  Their reduction axis
// is the token rows of each expert; the operands arrive transposed and
// quantized along those rows (blocks of 32; expert groups start on 128-row
// boundaries, so a block never mixes experts):
//   dW_down[e] = dy^T (g h),  dW_gate[e] = da^T x,  dW_up[e] = db^T x
// as K-major block-scaled GEMMs over [row_start[e], row_start[e+1]).
moe_status wgrad_routed_mx(const Shape& s, const Routing& rt, const Acts& act, const BwdWs& w,
                           const moe_grads* g, cudaStream_t st) {
  constexpr int kWgradBnMx = gemm_bn<true, EPI_BF16, SCHED_WGRAD>();  // output tile width
  const int d = static_cast<int>(s.d), I = static_cast<int>(s.I), E = static_cast<int>(s.E);
  {
    GemmParams p;  // dW_down[e] = dy_rows^T . (g h)
    zero_params(p);
    MOE_TRY(qmap(&p.tmA, w.dyt, s.d, s.Rp, kBM));
    MOE_TRY(qmap(&p.tmB0, w.hgt, s.I, s.Rp, kWgradBnMx));
    set_mx_scales(p, w.dyt_sf, s.d, w.hgt_sf, nullptr, s.I);
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.M_out = d;
    p.N = I;
    MOE_TRY(omap3(&p.tmO0, g->dW_down, s.E, s.d, s.I));
    p.status = w.status;
    MOE_LAUNCH(PL_WGRAD_DOWN, st, launch_gemm(GK_MX_WGRAD, p, grid_for(s.E * cdiv(s.d, kBM) * cdiv(s.I, kWgradBnMx)), st));
  }
  for (int half = 0; half < 2; ++half) {
    GemmParams p;  // dW_gate[e] = da^T . x_rows ; dW_up[e] = db^T . x_rows
    zero_params(p);
    MOE_TRY(qmap(&p.tmA, w.dadbt, 2 * s.I, s.Rp, kBM));
    MOE_TRY(qmap(&p.tmB0, act.xt, s.d, s.Rp, kWgradBnMx));
    set_mx_scales(p, w.dadbt_sf, 2 * s.I, act.xt_sf, nullptr, s.d);
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.M_out = I;
    p.N = d;
    p.a_col_off = half ? I : 0;
    MOE_TRY(omap3(&p.tmO0, half ? g->dW_up : g->dW_gate, s.E, s.I, s.d));
    p.status = w.status;
    MOE_LAUNCH(half ? PL_WGRAD_UP : PL_WGRAD_GATE, st, launch_gemm(GK_MX_WGRAD, p, grid_for(s.E * cdiv(s.I, kBM) * cdiv(s.d, kWgradBnMx)), st));
  }
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* fwd_ws, size_t* saved, size_t* bwd_ws) {
  Shape s;
  MOE_TRY(check_config(cfg, s));
  if (fwd_ws) {
    FwdWs w;
    carve_fwd(nullptr, s, w, fwd_ws);
  }
  if (saved) {
    Saved v;
    carve_saved(nullptr, s, v, saved);
  }
  if (bwd_ws) {
    BwdWs w;
    carve_bwd(nullptr, s, w, bwd_ws);
  }
  return MOE_OK;
}

moe_status moe_mxfp8_weights_size(const moe_config* cfg, size_t* bytes) {
  Shape s;
  MOE_TRY(check_config(cfg, s));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  if (cfg->precision != MOE_MXFP8) return MOE_ERR_UNSUPPORTED;
  MxWeights m;
  carve_mx(nullptr, s, m, bytes);
  return MOE_OK;
}

moe_status moe_quantize_weights_mxfp8(const moe_config* cfg, const moe_weights* w, void* mx, void* stream) {
  Shape s;
  MOE_TRY(check_config(cfg, s));
  if (cfg->precision != MOE_MXFP8) return MOE_ERR_UNSUPPORTED;
  if (!w || !mx || !w->W_gate || !w->W_up || !w->W_down || !aligned16(mx)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MxWeights m;
  carve_mx(mx, s, m, nullptr);
  const auto* Wg = static_cast<const __nv_bfloat16*>(w->W_gate);
  const auto* Wu = static_cast<const __nv_bfloat16*>(w->W_up);
  const auto* Wd = static_cast<const __nv_bfloat16*>(w->W_down);
  const int d = static_cast<int>(s.d), I = static_cast<int>(s.I), E = static_cast<int>(s.E);
  MOE_LAUNCH(PL_MX_WEIGHTS, st, launch_mx_rows(Wg, d, s.E * s.I, d, m.wg, m.wg_sf, st));
  MOE_LAUNCH(PL_MX_WEIGHTS, st, launch_mx_rows(Wu, d, s.E * s.I, d, m.wu, m.wu_sf, st));
  MOE_LAUNCH(PL_MX_WEIGHTS, st, launch_mx_rows(Wd, I, s.E * s.d, I, m.wd, m.wd_sf, st));
  // W_down[e] is [d, I]: its transpose [I, d] quantized along d
  MOE_LAUNCH(PL_MX_WEIGHTS, st, launch_mx_cols(Wd, I, s.d * s.I, d, I, E, m.wdt, d, I, 0, m.wdt_sf, s.E * s.I, st));
  // W_gate[e], W_up[e] are [I, d]: [W_gate; W_up]^T is [d, 2I], quantized along 2I
  MOE_LAUNCH(PL_MX_WEIGHTS, st, launch_mx_cols(Wg, d, s.I * s.d, I, d, E, m.wgut, 2 * s.I, d, 0, m.wgut_sf, s.E * s.d, st));
  MOE_LAUNCH(PL_MX_WEIGHTS, st, launch_mx_cols(Wu, d, s.I * s.d, I, d, E, m.wgut, 2 * s.I, d, I, m.wgut_sf, s.E * s.d, st));
  return MOE_OK;
}

moe_status moe_route_topk(const moe_config* cfg, const void* x, const void* W_router,
                          const float* router_bias, const float* logits_in, float* logits_out,
                          int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* perm_token, int32_t* route_row, void* ws, void* stream) {
  Shape s;
  MOE_TRY(check_config(cfg, s));
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned256(ws)) return MOE_ERR_INVALID_ARG;
  if (s.T == 0) return MOE_OK;
  if (!topk_idx || !topk_w || !counts || !offsets || !perm_token || !route_row)
    return MOE_ERR_INVALID_ARG;
  if (!logits_in && (!x || !W_router || !aligned16(x) || !aligned16(W_router))) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  FwdWs w;
  carve_fwd(ws, s, w, nullptr);
  Routing rt = w.rt;
  rt.topk_idx = topk_idx;
  rt.topk_w = topk_w;
  rt.counts = counts;
  rt.offsets = offsets;
  rt.perm_token = perm_token;
  rt.route_row = route_row;
  // the fused launch writes the logits only where the caller asks for them
  float* logits = logits_out ? logits_out : w.logits;
  return run_routing(s, x, W_router, router_bias, logits_in, logits, rt, w.chunk_counts,
                     w.chunk_base, w.status, st, w.sync, false, logits_out != nullptr);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* wts, void* y,
                       void* saved, void* ws, void* stream) {
  Shape s;
  MOE_TRY(check_config(cfg, s));
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned256(ws)) return MOE_ERR_INVALID_ARG;
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_weights(s, wts, true));
  if (!x || !y || !aligned16(x) || !aligned16(y) || !aligned256(saved)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  FwdWs w;
  carve_fwd(ws, s, w, nullptr);
  Saved sv;
  Routing rt = w.rt;
  if (saved) {
    carve_saved(saved, s, sv, nullptr);
    rt = sv.rt;
  }
  // the activations the backward needs go to the saved state, unless it keeps
  // only the routing (MOE_FLAG_REPLAY) or there is none (inference)
  const bool keep_acts = saved && !s.replay;
  // the logits are not kept (the separate kernels pass them through the workspace)
  MOE_TRY(run_routing(s, x, wts->W_router, wts->router_bias, nullptr, w.logits, rt, w.chunk_counts,
                      w.chunk_base, w.status, st, w.sync, true, false));
  const int T = static_cast<int>(s.T), d = static_cast<int>(s.d), I = static_cast<int>(s.I);
  const int E = static_cast<int>(s.E);

  const GateUpOut o{w.xp, w.h, true, w.hs, saved ? sv.act.abs : nullptr, w.xq, w.xq_sf, w.hq, w.hq_sf, w.status};
  MOE_TRY(forward_gateup(s, x, wts, rt, keep_acts ? &sv.act : nullptr, o, st));
  if (s.mx) {
    MOE_TRY(down_routed_mx(s, wts, rt, w, st));
  } else {
    // routed down projection, scaled by the router weight of each row
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, w.h, s.Rp, s.I, 64, kBM));
    MOE_TRY(tmap(&p.tmB0, wts->W_down, s.E * s.d, s.I, 64, kBN / 2));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.counts = rt.counts;
    p.N = d;
    p.K = I;
    p.b_group_rows = d;
    MOE_TRY(omap2(&p.tmO0, &p.tmO0h, w.o, s.Rp, s.d));
    p.tile_start = rt.tile_start;
    p.pair_start = rt.pair_start;
    p.rem_start = rt.rem_start;
    p.row_scale = rt.perm_w_pad;
    p.status = w.status;
    MOE_LAUNCH(PL_DOWN_ROUTED, st, launch_gemm(GK_DOWN, p, grid_for(cdiv(s.Rp, kBM) * cdiv(s.d, kBN)), st));
  }
  // shared down projection
  if (s.S) {
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, w.hs, s.T, s.Is, 64, kBM));
    MOE_TRY(tmap(&p.tmB0, wts->Ws_down, s.d, s.Is, 64, kBN / 2));
    p.dense_rows = T;
    p.N = d;
    p.K = static_cast<int>(s.Is);
    MOE_TRY(omap(&p.tmO0, w.ys, s.T, s.d));
    p.tmO0h = p.tmO0;  // dense rows: no tail tiles
    p.status = w.status;
    MOE_LAUNCH(PL_DOWN_SHARED, st, launch_gemm(GK_DOWN, p, grid_for(cdiv(s.T, kBM) * cdiv(s.d, kBN)), st));
  }
  MOE_LAUNCH(PL_COMBINE, st, launch_combine(w.o, s.S ? w.ys : nullptr, rt.route_row_pad, T, d, static_cast<int>(s.k),
                          static_cast<__nv_bfloat16*>(y), st));
  return MOE_OK;
}

moe_status moe_backward(const moe_config* cfg, const void* x, const moe_weights* wts, const void* dy,
                        const void* saved, void* dx, const moe_grads* g, void* ws, void* stream) {
  Shape s;
  MOE_TRY(check_config(cfg, s));
  if (!ws) return MOE_ERR_WORKSPACE;
  if (!aligned256(ws)) return MOE_ERR_INVALID_ARG;
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_weights(s, wts, true));
  if (!x || !dy || !saved || !dx || !g || !aligned16(x) || !aligned16(dy) || !aligned16(dx) ||
      !aligned256(saved))
    return MOE_ERR_INVALID_ARG;
  if (!g->dW_router || !g->dW_gate || !g->dW_up || !g->dW_down) return MOE_ERR_INVALID_ARG;
  if (s.S && (!g->dWs_gate || !g->dWs_up || !g->dWs_down)) return MOE_ERR_INVALID_ARG;
  // the gradient buffers take TMA stores: 16-byte aligned (checked here, before anything runs)
  const void* gbufs[] = {g->dW_router, g->d_topk_w, g->dW_gate, g->dW_up, g->dW_down,
                         g->dWs_gate, g->dWs_up, g->dWs_down};
  for (const void* q : gbufs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Saved sv;
  carve_saved(const_cast<void*>(saved), s, sv, nullptr);
  const Routing& rt = sv.rt;
  BwdWs w;
  carve_bwd(ws, s, w, nullptr);
  const int T = static_cast<int>(s.T), d = static_cast<int>(s.d), I = static_cast<int>(s.I);
  const int E = static_cast<int>(s.E), k = static_cast<int>(s.k), Is = static_cast<int>(s.Is);
  // MOE_FLAG_REPLAY: the saved state holds the routing and the shared
  // expert's a and b; recompute the routed experts' forward up to the SwiGLU
  // into the workspace.  Its h outputs and quantized x rows land in buffers
  // this backward overwrites later (hg; in MXFP8 mode dadbq and dyq), the same
  // kernels on the same inputs as the forward, so a and b are bitwise those
  // the forward produced.
  Acts act = s.replay ? w.act : sv.act;
  act.abs = sv.act.abs;  // the shared expert's a and b are always saved
  if (s.replay) {
    const GateUpOut o{nullptr, w.hg, false, nullptr, nullptr, w.dyq, w.dyq_sf, w.dadbq, w.dadbq_sf, w.status};
    MOE_TRY(forward_gateup(s, x, wts, rt, &act, o, st));
  }

  MxWeights m;
  if (s.mx) carve_mx(const_cast<void*>(wts->mxfp8), s, m, nullptr);
  // dy rows into expert-grouped order (zeros in padding rows); in MXFP8 mode
  // quantized on the way (the bf16 copy feeds the transposed quantization)
  if (s.mx)  // along d for the dgrad of down, along the tokens for dW_down
    MOE_LAUNCH(PL_MX_QUANT_DY, st, launch_mx_permute_dual(static_cast<const __nv_bfloat16*>(dy), d, rt.perm_token_pad,
                                                          rt.row_start + E, s.Rp, d, w.dyq, w.dyq_sf, w.dyt,
                                                          w.dyt_sf, st));
  else
    MOE_LAUNCH(PL_PERMUTE_DY, st, launch_scatter_rows(static_cast<const __nv_bfloat16*>(dy), rt.route_row_pad,
                                                     rt.row_start, rt.counts, T, E, d, static_cast<int>(s.k), w.dyp, st));
  // dgrad of the down projection with the fused SwiGLU backward and the
  // router-weight gradient partials <h, dh> per n-tile; in MXFP8 mode the
  // epilogue also quantizes [da | db] for the gate/up dgrad
  if (s.mx) {
    GemmParams p;
    zero_params(p);
    MOE_TRY(qmap(&p.tmA, w.dyq, s.Rp, s.d, kBM));
    MOE_TRY(qmap(&p.tmB0, m.wdt, s.E * s.I, s.d, kBN / 2));
    MOE_TRY(set_mx_row_scales(p, w.dyq_sf, s.Rp, m.wdt_sf, nullptr, s.E * s.I, s.d));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.counts = rt.counts;
    p.N = I;
    p.K = d;
    p.b_group_rows = I;
    p.out3 = w.dg_part;
    p.ldo3 = static_cast<int>(s.nparts);
    p.ab = act.ab;
    p.I = I;
    p.tile_start = rt.tile_start;
    p.pair_start = rt.pair_start;
    p.rem_start = rt.rem_start;
    p.row_scale = rt.perm_w_pad;
    p.qt = w.dadbt;
    p.qt_ld = s.Rp;
    p.qt_sf = w.dadbt_sf;
    p.qt_rb = cdiv(2 * s.I, 128);
    p.qt2 = w.hgt;
    p.qt2_ld = s.Rp;
    p.qt2_sf = w.hgt_sf;
    p.qt2_rb = cdiv(s.I, 128);
    p.qout = w.dadbq;
    p.qld = 2 * s.I;
    p.qsf = w.dadbq_sf;
    p.q_rb = cdiv(s.Rp, 128);
    p.status = w.status;
    MOE_LAUNCH(PL_DGRAD_DOWN_ROUTED, st, launch_gemm(GK_MX_DGRAD_DOWN, p, grid_for(cdiv(s.Rp, kBM) * s.nparts), st));
  } else {
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, w.dyp, s.Rp, s.d, 64, kBM));
    MOE_TRY(mnmap(&p.tmB0, wts->W_down, s.E * s.d, s.I, 2));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.counts = rt.counts;
    p.N = I;
    p.K = d;
    p.b_group_rows = d;
    p.out = w.dadb;
    p.ldo = 2 * s.I;
    p.out2 = w.hg;
    p.ldo2 = s.I;
    p.out3 = w.dg_part;
    p.ldo3 = static_cast<int>(s.nparts);
    p.ab = act.ab;
    p.I = I;
    p.tile_start = rt.tile_start;
    p.pair_start = rt.pair_start;
    p.rem_start = rt.rem_start;
    p.row_scale = rt.perm_w_pad;
    p.status = w.status;
    MOE_LAUNCH(PL_DGRAD_DOWN_ROUTED, st, launch_gemm(GK_DGRAD_DOWN, p, grid_for(cdiv(s.Rp, kBM) * s.nparts), st));
  }
  if (s.S) {
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, dy, s.T, s.d, 64, kBM));
    MOE_TRY(mnmap(&p.tmB0, wts->Ws_down, s.d, s.Is, 2));
    p.dense_rows = T;
    p.N = Is;
    p.K = d;
    p.out = w.dadbs;
    p.ldo = 2 * s.Is;
    p.out2 = w.hs;
    p.ldo2 = s.Is;
    p.ab = act.abs;
    p.I = Is;
    p.status = w.status;
    MOE_LAUNCH(PL_DGRAD_DOWN_SHARED, st, launch_gemm(GK_DGRAD_DOWN, p, grid_for(cdiv(s.T, kBM) * cdiv(s.Is, kBN)), st));
  }
  MOE_LAUNCH(PL_ROUTER_GRAD, st, launch_router_grad(w.dg_part, static_cast<int>(s.nparts), rt.route_row_pad,
                                                    rt.topk_w, T, k, g->d_topk_w, w.dl_tk, w.dl_row, st));
  // dgrad of gate/up: dx_row = [da | db] . [W_gate ; W_up]
  if (s.mx) {
    GemmParams p;
    zero_params(p);
    MOE_TRY(qmap(&p.tmA, w.dadbq, s.Rp, 2 * s.I, kBM));
    MOE_TRY(qmap(&p.tmB0, m.wgut, s.E * s.d, 2 * s.I, kBN / 2));
    MOE_TRY(set_mx_row_scales(p, w.dadbq_sf, s.Rp, m.wgut_sf, nullptr, s.E * s.d, 2 * s.I));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.counts = rt.counts;
    p.N = d;
    p.K = 2 * I;
    p.b_group_rows = d;
    MOE_TRY(omap(&p.tmO0, w.dxp, s.Rp, s.d));
    p.tile_start = rt.tile_start;
    p.pair_start = rt.pair_start;
    p.rem_start = rt.rem_start;
    p.status = w.status;
    MOE_LAUNCH(PL_DGRAD_GATEUP_ROUTED, st, launch_gemm(GK_MX_DGRAD_GATEUP, p, grid_for(cdiv(s.Rp, kBM) * cdiv(s.d, kBN)), st));
  } else {
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, w.dadb, s.Rp, 2 * s.I, 64, kBM));
    MOE_TRY(mnmap(&p.tmB0, wts->W_gate, s.E * s.I, s.d, 2));
    MOE_TRY(mnmap(&p.tmB1, wts->W_up, s.E * s.I, s.d, 2));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.counts = rt.counts;
    p.N = d;
    p.K = 2 * I;
    p.b_group_rows = I;
    p.b_split = I;
    MOE_TRY(omap2(&p.tmO0, &p.tmO0h, w.dxp, s.Rp, s.d));
    p.tile_start = rt.tile_start;
    p.pair_start = rt.pair_start;
    p.rem_start = rt.rem_start;
    p.status = w.status;
    MOE_LAUNCH(PL_DGRAD_GATEUP_ROUTED, st, launch_gemm(GK_DGRAD_GATEUP, p, grid_for(cdiv(s.Rp, kBM) * cdiv(s.d, kBN)), st));
  }
  if (s.S) {
    GemmParams p;
    zero_params(p);
    MOE_TRY(tmap(&p.tmA, w.dadbs, s.T, 2 * s.Is, 64, kBM));
    MOE_TRY(mnmap(&p.tmB0, wts->Ws_gate, s.Is, s.d, 2));
    MOE_TRY(mnmap(&p.tmB1, wts->Ws_up, s.Is, s.d, 2));
    p.dense_rows = T;
    p.N = d;
    p.K = 2 * Is;
    p.b_split = Is;
    MOE_TRY(omap(&p.tmO0, w.dxs, s.T, s.d));
    p.tmO0h = p.tmO0;  // dense rows: no tail tiles
    p.status = w.status;
    MOE_LAUNCH(PL_DGRAD_GATEUP_SHARED, st, launch_gemm(GK_DGRAD_GATEUP, p, grid_for(cdiv(s.T, kBM) * cdiv(s.d, kBN)), st));
  }
  MOE_LAUNCH(PL_UNPERMUTE, st, launch_unpermute(w.dxp, s.S ? w.dxs : nullptr, rt.route_row_pad, rt.topk_idx,
                                                w.dl_tk, static_cast<const __nv_bfloat16*>(wts->W_router), T, d,
                                                k, static_cast<__nv_bfloat16*>(dx), st));
  // dx is complete: the weight gradients below do not touch it
  if (g->dx_ready) MOE_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(g->dx_ready), st));
  // dxp is no longer read: its Rp x d bf16 hold the router weight gradient's per-chunk
  // partial sums, at most (R / 128 + E + 1) x d floats (Rp >= R + 63 E)
  MOE_LAUNCH(PL_ROUTER_WGRAD, st, launch_router_wgrad(w.dl_row, rt.perm_token_pad, rt.row_start, rt.counts,
                                                      static_cast<const __nv_bfloat16*>(x), E, d, s.R,
                                                      reinterpret_cast<float*>(w.dxp), s.Rp * s.d / 2,
                                                      g->dW_router, st));
  // weight gradients, reduced over each expert's full row range (no split-K)
  if (s.mx) {
    MOE_TRY(wgrad_routed_mx(s, rt, act, w, g, st));
  } else {
  {
    GemmParams p;  // dW_down[e] = dy_rows^T . (g h)
    zero_params(p);
    MOE_TRY(mnmap(&p.tmA, w.dyp, s.Rp, s.d, 2));
    MOE_TRY(mnmap(&p.tmB0, w.hg, s.Rp, s.I, 2));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.M_out = d;
    p.N = I;
    p.wgrad_mode = wgrad_mode(s);
    p.wgrad_f32 = s.wgrad_f32 ? 1 : 0;
    MOE_TRY(s.wgrad_f32 ? omap3_f32(&p.tmO0, g->dW_down, s.E, s.d, s.I) : omap3(&p.tmO0, g->dW_down, s.E, s.d, s.I));
    p.status = w.status;
    MOE_LAUNCH(PL_WGRAD_DOWN, st, launch_gemm(GK_WGRAD, p, grid_for(s.E * cdiv(s.d, kBM) * cdiv(s.I, kBN)), st));
  }
  for (int half = 0; half < 2; ++half) {
    GemmParams p;  // dW_gate[e] = da^T . x_rows ; dW_up[e] = db^T . x_rows
    zero_params(p);
    MOE_TRY(mnmap(&p.tmA, w.dadb, s.Rp, 2 * s.I, 2));
    MOE_TRY(mnmap(&p.tmB0, act.xp, s.Rp, s.d, 2));
    p.num_groups = E;
    p.row_start = rt.row_start;
    p.M_out = I;
    p.N = d;
    p.wgrad_mode = wgrad_mode(s);
    p.a_col_off = half ? I : 0;
    void* dW = half ? g->dW_up : g->dW_gate;
    p.wgrad_f32 = s.wgrad_f32 ? 1 : 0;
    MOE_TRY(s.wgrad_f32 ? omap3_f32(&p.tmO0, dW, s.E, s.I, s.d) : omap3(&p.tmO0, dW, s.E, s.I, s.d));
    p.status = w.status;
    MOE_LAUNCH(half ? PL_WGRAD_UP : PL_WGRAD_GATE, st, launch_gemm(GK_WGRAD, p, grid_for(s.E * cdiv(s.I, kBM) * cdiv(s.d, kBN)), st));
  }
  }
  if (s.S) {
    {
      GemmParams p;  // dWs_down = dy^T . h_s
      zero_params(p);
      MOE_TRY(mnmap(&p.tmA, dy, s.T, s.d, 2));
      MOE_TRY(mnmap(&p.tmB0, w.hs, s.T, s.Is, 2));
      p.dense_rows = T;
      p.M_out = d;
      p.N = Is;
      p.wgrad_f32 = s.wgrad_f32 ? 1 : 0;
      MOE_TRY(s.wgrad_f32 ? omap_f32(&p.tmO0, g->dWs_down, s.d, s.Is) : omap(&p.tmO0, g->dWs_down, s.d, s.Is));
      p.status = w.status;
      MOE_LAUNCH(PL_WGRAD_SHARED_DOWN, st, launch_gemm(GK_WGRAD, p, grid_for(cdiv(s.d, kBM) * cdiv(s.Is, kBN)), st));
    }
    for (int half = 0; half < 2; ++half) {
      GemmParams p;  // dWs_gate = da_s^T . x ; dWs_up = db_s^T . x
      zero_params(p);
      MOE_TRY(mnmap(&p.tmA, w.dadbs, s.T, 2 * s.Is, 2));
      MOE_TRY(mnmap(&p.tmB0, x, s.T, s.d, 2));
      p.dense_rows = T;
      p.M_out = Is;
      p.N = d;
      p.a_col_off = half ? Is : 0;
      void* dWs = half ? g->dWs_up : g->dWs_gate;
      p.wgrad_f32 = s.wgrad_f32 ? 1 : 0;
      MOE_TRY(s.wgrad_f32 ? omap_f32(&p.tmO0, dWs, s.Is, s.d) : omap(&p.tmO0, dWs, s.Is, s.d));
      p.status = w.status;
      MOE_LAUNCH(half ? PL_WGRAD_SHARED_UP : PL_WGRAD_SHARED_GATE, st, launch_gemm(GK_WGRAD, p, grid_for(cdiv(s.Is, kBM) * cdiv(s.d, kBN)), st));
    }
  }
  return MOE_OK;
}

moe_status moe_read_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(v);
}

moe_status moe_profile_enable(int enable) {
  profiler().on.store(enable != 0);
  return MOE_OK;
}

moe_status moe_profile_report(char* buf, size_t buflen) {
  Profiler& P = profiler();
  std::vector<ProfRecord> recs;
  {
    std::lock_guard<std::mutex> g(P.mu);
    recs.swap(P.recs);
  }
  double total[PL_COUNT] = {0};
  long long count[PL_COUNT] = {0}, kernels[PL_COUNT] = {0};
  moe_status status = MOE_OK;
  for (const ProfRecord& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      status = MOE_ERR_CUDA;
    total[r.label] += ms;
    count[r.label] += 1;
    kernels[r.label] += r.kernels;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  std::string out;
  for (int i = 0; i < PL_COUNT; ++i) {
    if (!count[i]) continue;
    char line[128];
    snprintf(line, sizeof(line), "%s %lld %lld %.6f\n", kProfNames[i], count[i], kernels[i], total[i]);
    out += line;
  }
  if (buf && buflen) {
    const size_t n = out.size() < buflen - 1 ? out.size() : buflen - 1;
    memcpy(buf, out.data(), n);
    buf[n] = 0;
  }
  return status;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape, precision or flag";
    case MOE_ERR_WORKSPACE: return "workspace missing";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_DEVICE: return "a kernel saw an invalid value";
    case MOE_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
    default: return "unknown status";
  }
}

}  // extern "C"
