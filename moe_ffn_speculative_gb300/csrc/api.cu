// C ABI of libmoe_gb300.so: argument validation, workspace layout, TMA
// descriptors and the launch sequence of the MoE-FFN layer forward.  The
// contract of every entry point is documented in include/moe.h.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "moe.h"
#include "moe_internal.cuh"

using namespace moe;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;
constexpr int kSmemLimit = 232448;  // 227 KB of dynamic shared memory per CTA
// Above this many tokens a layer's router takes its logits from the tiled
// CUDA-core GEMM (split over H to fill the SMs) instead of the GEMV, whose
// grid no longer fits one wave there.
constexpr int kLogitsGemmMinTokens = 384;

std::atomic<int> g_sms[kMaxDevices];  // SM count per device, filled on first use (0: not yet)

thread_local void* const* t_events = nullptr;
thread_local int t_nev = 0;
thread_local int t_schedule = MOE_SCHEDULE_AUTO;
thread_local int t_overlap = 1;  // slice launches overlap the previous kernel on the stream
thread_local L2Prefetch t_prefetch = {};  // consumed by the next forward on this thread

int device_sms() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 0;
  int v = g_sms[d].load(std::memory_order_relaxed);
  if (v == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    v = n < kMaxGrid ? n : kMaxGrid;  // one GEMM CTA per SM, up to the span table's size
    g_sms[d].store(v, std::memory_order_relaxed);
  }
  return v;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor [d2][d1][d0] (d0 contiguous), loaded in boxes of 64 x 128 x 1
// with the 128-byte swizzle; out-of-range elements read as zero.
bool encode_weights_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(kHalfRows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x [T][H] bf16 in boxes of 64 columns x box_rows tokens with the 128-byte
// swizzle; rows past T read as zero.
bool encode_x_2d(CUtensorMap* m, const void* base, uint64_t H, uint64_t T, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {H, T};
  cuuint64_t strides[1] = {H * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP4 codes [d2][d1][d0 bytes] (two e2m1 codes per byte), loaded in boxes of
// 32 bytes (one 64-input k-block) x 128 rows x 1, unswizzled; out-of-range
// bytes read as zero (code 0 = 0.0).
bool encode_codes_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0, d0 * d1};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK / 2), static_cast<cuuint32_t>(kHalfRows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Block-scaled weights [d2][d1][d0 inputs]: FP4 codes (two per byte; the
// tensor map type that spaces every 16 codes over 16 bytes of shared memory,
// the operand layout of 4-bit MMA inputs) or FP8 bytes, loaded in boxes of
// 128 inputs x 128 rows x 1 with the 128-byte swizzle; rows past the matrix
// read as zero.
bool encode_mx_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, bool fp4) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t row = fp4 ? d0 / 2 : d0;  // bytes per row
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {row, row * d1};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kMxK), static_cast<cuuint32_t>(kHalfRows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// h [rows][2*I_ld] (16-bit: hi columns then lo columns), loaded in boxes of
// 64 columns x 16 rows with the 128-byte swizzle; rows past the end read as
// zero.
bool encode_h_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), 16};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_recipe(const moe_recipe* r) {
  if (!r) return MOE_ERR_INVALID_ARG;
  const int E = r->num_experts, K = r->top_k;
  if (E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > 32 || K > E) return MOE_ERR_UNSUPPORTED;
  if (r->score_fn < 0 || r->score_fn > 2) return MOE_ERR_INVALID_ARG;
  if (r->n_group < 1) return MOE_ERR_INVALID_ARG;
  if (r->n_group > 1) {
    if (r->n_group > 32 || E % r->n_group != 0) return MOE_ERR_UNSUPPORTED;
    const int gsz = E / r->n_group;
    if (r->topk_group < 1 || r->topk_group > r->n_group) return MOE_ERR_INVALID_ARG;
    if (r->group_topn < 1 || r->group_topn > gsz) return MOE_ERR_INVALID_ARG;
    if (K > r->topk_group * gsz) return MOE_ERR_UNSUPPORTED;
  }
  if (!(r->norm_eps >= 0.f) || !(r->route_scale == r->route_scale) || !(r->swiglu_limit == r->swiglu_limit))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

struct RouterGeom {
  int tb, quads, hsplit, n_eb, n_tb;
  bool fold_sh;
};

// gated: a shared-expert gate row joins the E gate rows, unless it would
// need an expert block of its own (then it is folded: fold_sh).
RouterGeom router_geometry(int T, int E, bool gated, int sms) {
  RouterGeom g;
  g.fold_sh = gated && E > 32 && ceil_div(E + 1, 32) > ceil_div(E, 32);
  const int E_tot = E + ((gated && !g.fold_sh) ? 1 : 0);
  const int qn = ceil_div(E_tot, 4);
  g.quads = 1;
  while (g.quads < qn && g.quads < 8) g.quads <<= 1;
  g.hsplit = 8 / g.quads;
  g.n_eb = ceil_div(qn, g.quads);
  // 4-token blocks when the grid would not fill the GPU with 8, and still
  // fits in one wave (a router CTA holds a whole SM's registers)
  g.tb = 8;
  if (static_cast<long long>(ceil_div(T, 8)) * g.n_eb < sms && static_cast<long long>(ceil_div(T, 4)) * g.n_eb <= sms)
    g.tb = 4;
  g.n_tb = ceil_div(T, g.tb);
  // With several expert blocks, fewer rows per block and H split over more
  // warps while the grid still fits in one wave: each warp's chain of
  // dependent gate loads gets shorter (the GEMV is bound by that latency).
  if (g.n_eb > 1) {
    while (g.quads > 1 && static_cast<long long>(g.n_tb) * ceil_div(qn, g.quads / 2) <= sms) g.quads >>= 1;
    g.hsplit = 8 / g.quads;
    g.n_eb = ceil_div(qn, g.quads);
  }
  return g;
}

// Geometry of the fused small-expert-count kernel (slice.cu).  ok: the
// layer fits it at this T.  reserve: some T' <= T does, so a workspace sized
// for T holds its regions (sized for min(T, kSliceMaxTok) tokens).
struct SlicePlan {
  bool ok, reserve;
  int n_tok, s_e, s_sh, s_max, n_units, n_mt, n_rcta, n_tg, stage_space;
  int parts;  // k-block ranges per down output tile, so that the down items occupy the SMs
};

SlicePlan slice_plan(int T, int H, int I, int Is, int E, bool gated, int sms) {
  SlicePlan s;
  memset(&s, 0, sizeof(s));
  if (T < 1 || E + (gated ? 1 : 0) > kSliceMaxExperts) return s;
  const int Tr = T < kSliceMaxTok ? T : kSliceMaxTok;
  s.n_tok = ((Tr + 15) / 16) * 16;
  s.s_e = ceil_div(I, kHalfRows);
  s.s_sh = Is > 0 ? ceil_div(Is, kHalfRows) : 0;
  s.s_max = s.s_e > s.s_sh ? s.s_e : s.s_sh;
  s.n_units = E * s.s_e + s.s_sh;
  s.n_mt = ceil_div(H, kHalfRows);
  s.n_rcta = ceil_div(Tr, kSliceTokPerTask);
  s.n_tg = ceil_div(Tr, kSliceTokPerTask);
  s.stage_space = kSmemLimit - 1024 - kSliceCtrlBytes;
  {
    const int n_es = E + (s.s_sh > 0 ? 1 : 0);
    const int s_min = s.s_sh > 0 && s.s_sh < s.s_e ? s.s_sh : s.s_e;
    const int by_sm = sms / (n_es * s.n_mt);
    s.parts = by_sm < 1 ? 1 : (by_sm < 2 * s_min ? by_sm : 2 * s_min);
  }
  // four stages at least: their token-tile parts later hold h (2 k-blocks x hi/lo)
  const bool smem_ok = s.stage_space / (2 * kTileBytesA + kSliceMaxTok * 128) >= 4;
  s.reserve = smem_ok && s.n_units + 1 <= sms &&
              kSliceSyncWords + s.n_mt + (E + 1) * s.s_max <= kSliceMaxSetWords;
  s.ok = s.reserve && T <= kSliceMaxTok && s.n_units + s.n_rcta <= sms;
  return s;
}

// The fused kernel streams every expert's gate_up weights from the start,
// before the routing is known, and stops an untouched expert once it is: it
// pays off when, under uniform routing, untouched experts are rare.
bool slice_expected(int T, int E, int K) {
  const double miss = E * pow(1.0 - static_cast<double>(K) / E, static_cast<double>(T));
  return miss <= 0.25;
}

struct Layout {
  RouterGeom rg;
  SlicePlan sp;
  int n_max, nbuf, grid, I_ld;
  uint32_t tmem_cols;
  size_t smem;
  int max_gu_tiles, max_dn_tiles, g_max;
  bool need_out;
  int lsplit;  // H ranges of the logits GEMM (layers above kLogitsGemmMinTokens tokens)
  size_t o_lpart;
  size_t o_status, o_cnt, o_tiles, o_logits, o_shl, o_shw, o_idx, o_w, o_counts, o_offsets, o_sp, o_pp, o_groups,
      o_header, o_spans, o_span_groups, o_partials, o_h, o_out, o_sync, o_hbuf, o_sout, o_xh, total;
  // block-scaled path: the token operand images (x's for gate_up, h's for
  // down) of every (token block, k-block), each expert's first token block
  size_t o_img_gu, o_img_dn, o_e2d;
  int n_dense, img_gu_rows, img_dn_rows;
};

// mx: the layout of the block-scaled path (moe_ffn_forward_mx): token tiles
// of up to kMxMaxTok, h and x as e4m3 pieces with their scales.
Layout make_layout(int T, int H, int I, int Is, int E, int K, bool gated, int sms, bool mx = false) {
  Layout L;
  L.rg = router_geometry(T, E, gated, sms);
  // Token tile width: every token of a decode-sized forward in one tile.
  // Above 128 tokens, when an expert's mean load leaves room in 128 columns,
  // about four times that load (between 64 and 128), so that routed experts
  // rarely need a second tile while the shared expert's T tokens (several
  // narrower tiles) neither size every stage of the ring for 256 columns nor
  // take the second TMEM accumulator buffer (two buffers of 2 x 128 columns
  // fill the 512).  Heavily loaded experts (a dense layer) keep one tile of
  // up to 256 columns: a second tile would stream their weights twice.
  int nm = ((T + 15) / 16) * 16;
  const long long mean = (static_cast<long long>(T) * K + E - 1) / E;
  if (T > 128 && mean + 32 <= 128) {
    const long long load4 = 4 * mean;
    const int cap = static_cast<int>(load4 < 64 ? 64 : (load4 > 128 ? 128 : ((load4 + 15) / 16) * 16));
    if (cap < nm) nm = cap;
  }
  L.n_max = nm < 16 ? 16 : (nm > 256 ? 256 : nm);
  if (mx) {
    const int t16 = ((T + 15) / 16) * 16;
    L.n_max = t16 < kMxMaxTok ? (t16 < 16 ? 16 : t16) : kMxMaxTok;
  }
  L.nbuf = (4 * L.n_max <= 512) ? 2 : 1;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(L.nbuf * 2 * L.n_max)) cols <<= 1;
  L.tmem_cols = cols;
  // all of shared memory: the kernel cuts the stage ring (two 16 KB weight
  // halves and two token tiles per stage, h as hi and lo) to the widest
  // token tile of each forward
  L.smem = kSmemLimit;
  L.grid = sms;
  const int Imax = Is > I ? Is : I;
  L.I_ld = ((Imax + 7) / 8) * 8;  // the block-scaled path needs multiples of 128 already
  const long long TK = static_cast<long long>(T) * K;
  const long long u_max = TK < E ? TK : E;
  const long long nb_sum = u_max + TK / L.n_max;
  long long gu = ceil_div(I, kHalfRows) * nb_sum, dn = ceil_div(H, 2 * kHalfRows) * nb_sum;
  if (Is > 0) {
    gu += static_cast<long long>(ceil_div(Is, kHalfRows)) * ceil_div(T, L.n_max);
    dn += static_cast<long long>(ceil_div(H, 2 * kHalfRows)) * ceil_div(T, L.n_max);
  }
  L.max_gu_tiles = static_cast<int>(gu);
  L.max_dn_tiles = static_cast<int>(dn);
  L.g_max = static_cast<int>(u_max) + (Is > 0 ? 1 : 0);
  L.need_out = (K > 1 || Is > 0);
  const size_t rows = static_cast<size_t>(TK) + T;
  // the fixed header: status block and every self-resetting counter
  L.o_status = 0;
  L.o_cnt = kRouteCntOffset;
  L.o_sync = kSliceSyncOffset;
  size_t o = kWsHeaderBytes;
  // stream-K arrival counters (gate_up, down) and gate_up readiness counters
  // (+1: the block-scaled path's count of warps that cut their share of x into pieces)
  L.o_tiles = o; o = align_up(o + 4 * static_cast<size_t>(2 * L.max_gu_tiles + L.max_dn_tiles + 1));
  L.o_logits = o; o = align_up(o + 4 * static_cast<size_t>(T) * E);
  L.o_shl = o; o = align_up(o + 4 * static_cast<size_t>(T) * (L.rg.fold_sh ? L.rg.n_eb * L.rg.hsplit : 1));
  // the logits GEMM's partial sums over its ranges of H
  const int E_tot = E + (gated ? 1 : 0);
  L.lsplit = T > kLogitsGemmMinTokens ? logits_gemm_split(T, H, E_tot, sms) : 1;
  L.o_lpart = o;
  if (L.lsplit > 1) o = align_up(o + 4 * static_cast<size_t>(L.lsplit) * T * E_tot);
  L.o_shw = o; o = align_up(o + 4 * static_cast<size_t>(T));
  L.o_idx = o; o = align_up(o + 4 * static_cast<size_t>(TK));
  L.o_w = o; o = align_up(o + 4 * static_cast<size_t>(TK));
  L.o_counts = o; o = align_up(o + 4 * static_cast<size_t>(E));
  L.o_offsets = o; o = align_up(o + 4 * static_cast<size_t>(E + 1));
  L.o_sp = o; o = align_up(o + 4 * static_cast<size_t>(TK));
  L.o_pp = o; o = align_up(o + 4 * static_cast<size_t>(TK));
  L.o_groups = o; o = align_up(o + sizeof(GroupEntry) * static_cast<size_t>(L.g_max + 1));
  L.o_header = o; o = align_up(o + sizeof(GemmHeader));
  L.o_spans = o; o = align_up(o + 8 * 2 * static_cast<size_t>(L.grid + 1));
  L.o_span_groups = o; o = align_up(o + 4 * 2 * static_cast<size_t>(L.grid + 1));
  L.o_partials = o; o = align_up(o + 4 * static_cast<size_t>(L.grid) * 4 * 2 * L.n_max * 128);
  L.o_h = L.o_img_gu = L.o_img_dn = L.o_e2d = L.o_xh = 0;
  L.n_dense = L.img_gu_rows = L.img_dn_rows = 0;
  if (mx) {
    // token blocks: the routed groups' (at most u_max + TK / n_max) and the
    // shared expert's
    L.n_dense = static_cast<int>(u_max + TK / L.n_max) + (Is > 0 ? ceil_div(T, L.n_max) : 0);
    L.img_gu_rows = ((kMxPx * L.n_max + 15) / 16) * 16;
    L.img_dn_rows = ((kMxPh * L.n_max + 15) / 16) * 16;
    const size_t slot_gu = static_cast<size_t>(L.img_gu_rows) * 128 + kMxSfBytes;
    const size_t slot_dn = static_cast<size_t>(L.img_dn_rows) * 128 + kMxSfBytes;
    const int Imx = Is > I ? Is : I;
    L.o_img_gu = o; o = align_up(o + static_cast<size_t>(L.n_dense) * (H / kMxK) * slot_gu);
    L.o_img_dn = o; o = align_up(o + static_cast<size_t>(L.n_dense) * (Imx / kMxK) * slot_dn);
    L.o_e2d = o; o = align_up(o + 4 * static_cast<size_t>(E));
  } else {
    L.o_h = o; o = align_up(o + 2 * 2 * rows * L.I_ld);
    L.o_xh = o; o = align_up(o + 2 * static_cast<size_t>(T) * H);  // f16 copy of x (FP4 experts)
  }
  L.o_out = o;
  if (L.need_out) o = align_up(o + 4 * rows * H);
  // fused small-expert-count kernel: counters and the per-slice partial outputs
  L.sp = slice_plan(T, H, I, Is, E, gated, sms);
  L.o_hbuf = L.o_sout = 0;
  if (mx) L.sp.reserve = L.sp.ok = false;
  if (L.sp.reserve) {
    // every expert's h tiles (2 per slice, each 2*n_tok rows of 128 bytes)
    // and the pair outputs for the combine; the counter sets are in the header
    const int Tr = T < kSliceMaxTok ? T : kSliceMaxTok;
    const size_t slots = static_cast<size_t>(Tr) * K + Tr;
    const size_t n_es = static_cast<size_t>(E) + 1;
    L.o_hbuf = o; o = align_up(o + n_es * 2 * L.sp.s_max * 2 * static_cast<size_t>(L.sp.n_tok) * 128);
    L.o_sout = o;
    if (K > 1 || Is > 0 || L.sp.parts > 1) o = align_up(o + 4 * slots * H * static_cast<size_t>(L.sp.parts));
  }
  L.total = o;
  return L;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool use_slice(const Layout& L, int T, int E, int K) {
  if (!L.sp.ok || t_schedule == MOE_SCHEDULE_STREAM_K) return false;
  if (t_schedule == MOE_SCHEDULE_SLICE) return true;
  // automatic: untouched experts rare, and enough down items (output tiles
  // x k-block parts) to occupy three quarters of the CTAs
  const int n_es = E + (L.sp.s_sh > 0 ? 1 : 0);
  return slice_expected(T, E, K) && 4 * n_es * L.sp.n_mt * L.sp.parts >= 3 * L.grid;
}

// Inside a stream capture the event becomes an event-record node of the
// graph (recorded on every replay), so kernels can be timed in graph replay.
void record_event_on(int i, cudaStream_t s) {
  if (!t_events || i >= 2 * t_nev || !t_events[i]) return;
  cudaEvent_t ev = static_cast<cudaEvent_t>(t_events[i]);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

namespace moe {

moe_status route_check_args(const moe_bf16* x, int T, int H, const moe_bf16* gate, const moe_recipe* recipe,
                            const int32_t* topk_idx, const float* topk_w) {
  const moe_status st = check_recipe(recipe);
  if (st != MOE_OK) return st;
  if (T < 0 || H < 8 || H % 8 != 0) return H % 8 != 0 && H >= 8 ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
  if (H > 65536 || T > 65536) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !gate || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(gate)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace moe

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_RANGE: return "MOE_ERR_DEVICE_RANGE";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_route_workspace_bytes(int T, int E) {
  if (T < 0 || E < 1) return 0;
  // [status block][token-block counters for any T][logits T x E]
  return kRouteCntOffset + kRouteCntBytes + align_up(4 * static_cast<size_t>(T) * E);
}

moe_status moe_route(const moe_bf16* x, int T, int H, const moe_bf16* gate, const float* router_bias,
                     const float* expert_bias, const moe_recipe* recipe, float* logits_out, int32_t* topk_idx,
                     float* topk_w, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const moe_status st = moe::route_check_args(x, T, H, gate, recipe, topk_idx, topk_w);
  if (st != MOE_OK || T == 0) return st;
  const int E = recipe->num_experts;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < moe_route_workspace_bytes(T, E))
    return MOE_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const RouterGeom rg = router_geometry(T, E, false, sms);
  char* w = static_cast<char*>(ws);
  const size_t o_cnt = kRouteCntOffset;
  const size_t o_logits = kRouteCntOffset + kRouteCntBytes;
  RouteParams p;
  memset(&p, 0, sizeof(p));
  p.x = x; p.gate = gate; p.router_bias = router_bias; p.expert_bias = expert_bias; p.sh_gate = nullptr;
  p.T = T; p.H = H; p.E = E; p.K = recipe->top_k;
  p.score_fn = recipe->score_fn; p.n_group = recipe->n_group; p.topk_group = recipe->topk_group;
  p.group_topn = recipe->group_topn; p.renorm = recipe->norm_topk_prob; p.eps = recipe->norm_eps;
  p.scale = recipe->route_scale;
  p.quads = rg.quads; p.hsplit = rg.hsplit; p.n_eb = rg.n_eb; p.n_tb = rg.n_tb;
  p.logits = logits_out ? logits_out : reinterpret_cast<float*>(w + o_logits);
  p.idx = topk_idx; p.w = topk_w;
  p.tb_counter = reinterpret_cast<int32_t*>(w + o_cnt);
  p.glob_counter = p.tb_counter + ceil_div(T, 4);
  p.do_permute = 0;
  if (T > 1024) {
    // many tokens: the logits by the tiled CUDA-core GEMM, then selection only
    const cudaError_t e = launch_logits_gemm(x, gate, nullptr, router_bias, T, H, E, p.logits, nullptr, 1, nullptr, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    p.logits_given = 1;
    p.n_eb = 1;
    p.n_tb = ceil_div(T, 8);
    return cuda_status(launch_route(p, 8, stream));
  }
  return cuda_status(launch_route(p, rg.tb, stream));
}

moe_status moe_route_from_logits(const float* logits, int T, const float* expert_bias, const moe_recipe* recipe,
                                 int32_t* topk_idx, float* topk_w, cudaStream_t stream) {
  moe_status st = check_recipe(recipe);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T > 65536) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_select_from_logits(logits, T, recipe->num_experts, recipe->top_k, expert_bias,
                                               recipe->score_fn, recipe->n_group, recipe->topk_group,
                                               recipe->group_topn, recipe->norm_topk_prob, recipe->norm_eps,
                                               recipe->route_scale, topk_idx, topk_w, stream));
}

moe_status moe_permute(const int32_t* topk_idx, int T, int K, int E, int32_t* counts, int32_t* offsets,
                       int32_t* sorted_pair, int32_t* pair_pos, void* ws, size_t ws_bytes, cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  if (T < 0 || K < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > E || T > 65536) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !sorted_pair || !pair_pos)) return MOE_ERR_INVALID_ARG;
  // T == 0 still defines counts and offsets (all zero)
  return cuda_status(launch_permute(topk_idx, T, K, E, counts, offsets, sorted_pair, pair_pos, stream));
}

size_t moe_ffn_workspace_bytes(int T, int H, int I, int Is, const moe_recipe* recipe) {
  if (check_recipe(recipe) != MOE_OK || T < 0 || H < 8 || I < 8 || Is < 0) return 0;
  const int sms = device_sms();
  if (sms <= 0) return 0;
  // the gated/ungated choice changes only the router's geometry: size for the
  // larger; where the block-scaled path takes the shape, for its layout too
  size_t n = 0;
  for (int mx = 0; mx < 2; ++mx) {
    if (mx && (H % kMxK != 0 || I % kMxK != 0 || Is % kMxK != 0)) continue;
    for (int gated = 0; gated < 2; ++gated) {
      const Layout L = make_layout(T, H, I, Is, recipe->num_experts, recipe->top_k, gated != 0, sms, mx != 0);
      if (L.total > n) n = L.total;
    }
  }
  return n;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

}  // extern "C"

namespace {

// FP4 routed experts of one forward (null: bf16 experts).
struct Fp4Experts {
  const uint8_t* gu_q;
  const uint8_t* dn_q;
  const uint8_t* scales;  // prepared by moe_fp4_prepare_scales()
};

moe_status ffn_forward(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate, const float* router_bias,
                       const float* expert_bias, const moe_bf16* w_gate_up, const moe_bf16* w_down,
                       const moe_bf16* sh_gate_up, const moe_bf16* sh_down, int Is, const moe_bf16* sh_gate,
                       const moe_recipe* recipe, void* ws, size_t ws_bytes, moe_bf16* y, int32_t* topk_idx_out,
                       float* topk_w_out, int32_t* counts_out, cudaStream_t stream, const Fp4Experts* fp4) {
  // the next-layer prefetch setting is consumed by this call, whatever it runs
  const L2Prefetch pf = t_prefetch;
  t_prefetch.n = 0;
  moe_status st = check_recipe(recipe);
  if (st != MOE_OK) return st;
  if (T < 0 || H < 8 || I < 8 || Is < 0) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || I % 8 != 0 || Is % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (H > 65536 || I > 16384 || Is > 16384 || T > 65536) return MOE_ERR_UNSUPPORTED;
  if ((sh_gate_up == nullptr) != (Is == 0) || (Is > 0 && sh_down == nullptr)) return MOE_ERR_INVALID_ARG;
  if (sh_gate && Is == 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !gate || !w_gate_up || !w_down || !y) return MOE_ERR_INVALID_ARG;
  if (fp4 && !aligned16(fp4->scales)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(gate) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y) ||
      (sh_gate_up && !aligned16(sh_gate_up)) || (sh_down && !aligned16(sh_down)) || (sh_gate && !aligned16(sh_gate)))
    return MOE_ERR_INVALID_ARG;
  const size_t xy_bytes = static_cast<size_t>(T) * H * 2;
  if (overlaps(x, xy_bytes, y, xy_bytes)) return MOE_ERR_INVALID_ARG;
  // a workspace that cannot even hold the fixed header is refused before any device query
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
  const int E = recipe->num_experts, K = recipe->top_k;
  const int sms = device_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const Layout L = make_layout(T, H, I, Is, E, K, sh_gate != nullptr, sms);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w + L.o_status);
  int32_t* idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t*>(w + L.o_idx);
  float* wts = topk_w_out ? topk_w_out : reinterpret_cast<float*>(w + L.o_w);
  int32_t* counts = counts_out ? counts_out : reinterpret_cast<int32_t*>(w + L.o_counts);
  int32_t* sorted_pair = reinterpret_cast<int32_t*>(w + L.o_sp);
  int32_t* pair_pos = reinterpret_cast<int32_t*>(w + L.o_pp);
  float* sh_w = reinterpret_cast<float*>(w + L.o_shw);
  GroupEntry* groups = reinterpret_cast<GroupEntry*>(w + L.o_groups);
  GemmHeader* header = reinterpret_cast<GemmHeader*>(w + L.o_header);
  int32_t* tiles = reinterpret_cast<int32_t*>(w + L.o_tiles);
  uint16_t* h = reinterpret_cast<uint16_t*>(w + L.o_h);
  float* out_ws = reinterpret_cast<float*>(w + L.o_out);

  if (!fp4 && use_slice(L, T, E, K)) {
    // ---- fused small-expert-count schedule: one launch
    CUtensorMap tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, tm_x;
    if (!encode_weights_3d(&tm_gu, w_gate_up, H, I, 2ull * E) || !encode_weights_3d(&tm_dn, w_down, I, H, E) ||
        !encode_x_2d(&tm_x, x, H, T, static_cast<uint32_t>(L.sp.n_tok)))
      return MOE_ERR_CUDA;
    if (Is > 0) {
      if (!encode_weights_3d(&tm_gu_sh, sh_gate_up, H, Is, 2) || !encode_weights_3d(&tm_dn_sh, sh_down, Is, H, 1))
        return MOE_ERR_CUDA;
    } else {
      tm_gu_sh = tm_gu;
      tm_dn_sh = tm_dn;
    }
    SliceParams sp;
    memset(&sp, 0, sizeof(sp));
    sp.x = x; sp.gate = gate; sp.router_bias = router_bias; sp.sh_gate = sh_gate;
    sp.sel = SelCfg{E, K, recipe->score_fn, recipe->n_group, recipe->topk_group, recipe->group_topn,
                    recipe->norm_topk_prob, recipe->norm_eps, recipe->route_scale, expert_bias};
    sp.T = T; sp.H = H; sp.E = E; sp.K = K; sp.TK = T * K;
    sp.n_tok = L.sp.n_tok; sp.s_e = L.sp.s_e; sp.s_sh = L.sp.s_sh; sp.s_max = L.sp.s_max;
    sp.n_units = L.sp.n_units; sp.n_mt = L.sp.n_mt; sp.n_rcta = L.sp.n_rcta; sp.n_tg = L.sp.n_tg;
    sp.stage_space = L.sp.stage_space;
    sp.swiglu_limit = recipe->swiglu_limit;
    sp.logits = reinterpret_cast<float*>(w + L.o_logits);
    sp.idx = idx; sp.w = wts; sp.sh_w = sh_w; sp.counts = counts;
    sp.hbuf = reinterpret_cast<uint8_t*>(w + L.o_hbuf);
    sp.out = reinterpret_cast<float*>(w + L.o_sout);
    sp.parts = L.sp.parts;
    sp.direct_y = (K == 1 && Is == 0 && L.sp.parts == 1) ? 1 : 0;
    sp.y = y;
    sp.sync = reinterpret_cast<int32_t*>(w + L.o_sync);
    sp.set_words = kSliceMaxSetWords;
    sp.status = status;
    record_event_on(0, stream);
    record_event_on(1, stream);
    record_event_on(2, stream);
    const cudaError_t e =
        launch_slice(tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, tm_x, sp, L.grid, kSmemLimit, t_overlap != 0, stream);
    record_event_on(3, stream);
    return cuda_status(e);
  }

  // ---- 1. router + permutation + work list
  RouteParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.x = x; rp.gate = gate; rp.router_bias = router_bias; rp.expert_bias = expert_bias; rp.sh_gate = sh_gate;
  rp.T = T; rp.H = H; rp.E = E; rp.K = K;
  rp.score_fn = recipe->score_fn; rp.n_group = recipe->n_group; rp.topk_group = recipe->topk_group;
  rp.group_topn = recipe->group_topn; rp.renorm = recipe->norm_topk_prob; rp.eps = recipe->norm_eps;
  rp.scale = recipe->route_scale;
  rp.quads = L.rg.quads; rp.hsplit = L.rg.hsplit; rp.n_eb = L.rg.n_eb; rp.n_tb = L.rg.n_tb;
  rp.fold_sh = L.rg.fold_sh ? 1 : 0;
  rp.logits = reinterpret_cast<float*>(w + L.o_logits);
  rp.sh_logit = reinterpret_cast<float*>(w + L.o_shl);
  rp.idx = idx; rp.w = wts; rp.sh_w = Is > 0 ? sh_w : nullptr;
  rp.tb_counter = reinterpret_cast<int32_t*>(w + L.o_cnt);
  rp.glob_counter = rp.tb_counter + L.rg.n_tb;
  rp.do_permute = 1;
  rp.counts = counts; rp.offsets = reinterpret_cast<int32_t*>(w + L.o_offsets);
  rp.sorted_pair = sorted_pair; rp.pair_pos = pair_pos;
  rp.groups = groups; rp.header = header;
  rp.spans = reinterpret_cast<int64_t*>(w + L.o_spans);
  rp.span_groups = reinterpret_cast<int32_t*>(w + L.o_span_groups);
  rp.grid = L.grid;
  rp.I = I; rp.Is = Is; rp.n_max = L.n_max;
  rp.zero_ptr = tiles; rp.zero_count = 2 * L.max_gu_tiles + L.max_dn_tiles + 1;
  uint16_t* xh = reinterpret_cast<uint16_t*>(w + L.o_xh);
  if (fp4) {
    rp.fp4 = 1;
    rp.xh = xh;
    rp.status = status;
  }
  record_event_on(0, stream);
  cudaError_t e = cudaSuccess;
  int tb = L.rg.tb;
  if (T > kLogitsGemmMinTokens && !fp4) {
    // many tokens: the logits by a tiled CUDA-core GEMM, H cut into enough
    // ranges (partial sums the router launch adds in order) that its 128 x
    // 64 tiles fill the SMs, then the router launch only selects, permutes
    // and builds the work list (one CTA per 8 tokens)
    e = launch_logits_gemm(x, gate, sh_gate, router_bias, T, H, E, rp.logits, rp.sh_logit, L.lsplit,
                           reinterpret_cast<float*>(w + L.o_lpart), stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    rp.logits_given = 1;
    rp.lsplit = L.lsplit;
    rp.lpart = reinterpret_cast<const float*>(w + L.o_lpart);
    rp.fold_sh = 0;
    rp.n_eb = 1;
    tb = 8;
    rp.n_tb = ceil_div(T, tb);
  }
  e = launch_route(rp, tb, stream);
  record_event_on(1, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // ---- 2. both grouped GEMMs, one persistent cooperative launch
  CUtensorMap tm_gu, tm_gu_sh, tm_dn, tm_dn_sh;
  if (fp4) {
    if (!encode_codes_3d(&tm_gu, fp4->gu_q, H / 2, I, 2ull * E) || !encode_codes_3d(&tm_dn, fp4->dn_q, I / 2, H, E))
      return MOE_ERR_CUDA;
  } else if (!encode_weights_3d(&tm_gu, w_gate_up, H, I, 2ull * E) || !encode_weights_3d(&tm_dn, w_down, I, H, E)) {
    return MOE_ERR_CUDA;
  }
  if (Is > 0) {
    if (!encode_weights_3d(&tm_gu_sh, sh_gate_up, H, Is, 2) || !encode_weights_3d(&tm_dn_sh, sh_down, Is, H, 1))
      return MOE_ERR_CUDA;
  } else {
    tm_gu_sh = tm_gu;
    tm_dn_sh = tm_dn;
  }
  GemmParams gp;
  memset(&gp, 0, sizeof(gp));
  gp.groups = groups; gp.header = header; gp.sorted_pair = sorted_pair;
  gp.spans = rp.spans; gp.span_groups = rp.span_groups;
  gp.x = x; gp.h = h;
  gp.T = T; gp.K = K; gp.TK = T * K; gp.H = H; gp.I_ld = L.I_ld;
  gp.n_max = L.n_max; gp.stage_space = kSmemLimit - 1024 - kCtrlBytes; gp.nbuf = L.nbuf;
  gp.tmem_cols = L.tmem_cols;
  gp.swiglu_limit = recipe->swiglu_limit;
  gp.out_ws = out_ws; gp.y = y; gp.direct_y = L.need_out ? 0 : 1;
  gp.topk_w = wts; gp.sh_w = (Is > 0 && sh_gate) ? sh_w : nullptr;
  gp.partials = reinterpret_cast<float*>(w + L.o_partials);
  gp.status = status;
  gp.tile_counters_gu = tiles;
  gp.tile_counters_dn = tiles + L.max_gu_tiles;
  gp.ready = tiles + L.max_gu_tiles + L.max_dn_tiles;
  gp.I = I;
  gp.E = E;
  gp.g_max = L.g_max;
  gp.max_gu_tiles = L.max_gu_tiles;
  gp.max_dn_tiles = L.max_dn_tiles;
  {
    const int Imax = Is > I ? Is : I;
    gp.max_gu_iters = static_cast<long long>(L.max_gu_tiles) * ceil_div(H, kBlockK);
    gp.max_dn_iters = static_cast<long long>(L.max_dn_tiles) * ceil_div(Imax, kBlockK);
  }
  if (fp4) {
    gp.xh = xh;
    gp.gu_scale = fp4->scales;
    gp.dn_scale = fp4->scales;  // one buffer: the down blocks follow the gate_up blocks
  }
  gp.pf = pf;
  // the down GEMM's token rows by TMA when every k-block is whole
  CUtensorMap tm_h = tm_dn;
  if (I % kBlockK == 0 && Is % kBlockK == 0) {
    if (!encode_h_2d(&tm_h, h, 2ull * L.I_ld, static_cast<uint64_t>(T) * K + T)) return MOE_ERR_CUDA;
    gp.h_tma = 1;
  }
  record_event_on(2, stream);
  e = launch_experts(tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, tm_h, gp, L.grid, L.smem, stream, fp4 != nullptr);
  record_event_on(3, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // ---- 4. weighted combine (+ shared expert)
  if (L.need_out) {
    record_event_on(4, stream);
    e = launch_combine(out_ws, pair_pos, T, K, H, Is > 0 ? 1 : 0, y, stream);
    record_event_on(5, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// ---- block-scaled experts (FP4 or FP8 routed, FP8 shared): router, one
// persistent launch of both GEMMs on the block-scaled MMA, combine
bool mx_shape_ok(int E, int H, int I, int Is) {
  return E >= 1 && E <= 1024 && H >= kMxK && I >= kMxK && H % kMxK == 0 && I % kMxK == 0 && Is % kMxK == 0 &&
         H <= 65536 && I <= 16384 && Is <= 16384;
}

size_t mx_scales_bytes(int E, int H, int I, int Is) {
  return mx_scale_offset(E, H, I, Is, 1, -1, 0, 0) + static_cast<size_t>(ceil_div(H, 2 * kHalfRows)) * (Is / kMxK) * 1024;
}

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

moe_status ffn_forward_mx(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate, const float* router_bias,
                          const float* expert_bias, int routed_fmt, const uint8_t* w_gate_up_q,
                          const uint8_t* w_down_q, const uint8_t* sh_gate_up_q, const uint8_t* sh_down_q, int Is,
                          const moe_bf16* sh_gate, const void* scales, size_t scales_bytes,
                          const moe_recipe* recipe, void* ws, size_t ws_bytes, moe_bf16* y, int32_t* topk_idx_out,
                          float* topk_w_out, int32_t* counts_out, cudaStream_t stream) {
  const L2Prefetch pf = t_prefetch;
  t_prefetch.n = 0;
  moe_status st = check_recipe(recipe);
  if (st != MOE_OK) return st;
  if (routed_fmt != MOE_FMT_FP4 && routed_fmt != MOE_FMT_FP8) return MOE_ERR_INVALID_ARG;
  if (T < 0 || H < 8 || I < 8 || Is < 0) return MOE_ERR_INVALID_ARG;
  if (T > 65536 || !mx_shape_ok(recipe->num_experts, H, I, Is)) return MOE_ERR_UNSUPPORTED;
  if ((sh_gate_up_q == nullptr) != (Is == 0) || (Is > 0 && sh_down_q == nullptr)) return MOE_ERR_INVALID_ARG;
  if (sh_gate && Is == 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !gate || !w_gate_up_q || !w_down_q || !scales || !y) return MOE_ERR_INVALID_ARG;
  const bool fp4 = routed_fmt == MOE_FMT_FP4;
  // FP4 codes go through the packed tensor-map type, which needs 32-byte alignment
  const bool wq_ok = fp4 ? (aligned32(w_gate_up_q) && aligned32(w_down_q))
                         : (aligned16(w_gate_up_q) && aligned16(w_down_q));
  if (!aligned16(x) || !aligned16(gate) || !aligned16(y) || !aligned16(scales) || !wq_ok ||
      (sh_gate_up_q && !aligned16(sh_gate_up_q)) || (sh_down_q && !aligned16(sh_down_q)) ||
      (sh_gate && !aligned16(sh_gate)))
    return MOE_ERR_INVALID_ARG;
  const int E = recipe->num_experts, K = recipe->top_k;
  if (scales_bytes < mx_scales_bytes(E, H, I, Is)) return MOE_ERR_INVALID_ARG;
  const size_t xy_bytes = static_cast<size_t>(T) * H * 2;
  if (overlaps(x, xy_bytes, y, xy_bytes)) return MOE_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < kWsHeaderBytes) return MOE_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MOE_ERR_CUDA;
  const Layout L = make_layout(T, H, I, Is, E, K, sh_gate != nullptr, sms, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w + L.o_status);
  int32_t* idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t*>(w + L.o_idx);
  float* wts = topk_w_out ? topk_w_out : reinterpret_cast<float*>(w + L.o_w);
  int32_t* counts = counts_out ? counts_out : reinterpret_cast<int32_t*>(w + L.o_counts);
  int32_t* sorted_pair = reinterpret_cast<int32_t*>(w + L.o_sp);
  int32_t* pair_pos = reinterpret_cast<int32_t*>(w + L.o_pp);
  float* sh_w = reinterpret_cast<float*>(w + L.o_shw);
  GroupEntry* groups = reinterpret_cast<GroupEntry*>(w + L.o_groups);
  GemmHeader* header = reinterpret_cast<GemmHeader*>(w + L.o_header);
  int32_t* tiles = reinterpret_cast<int32_t*>(w + L.o_tiles);
  float* out_ws = reinterpret_cast<float*>(w + L.o_out);

  // ---- 1. router + permutation + work list (128-input k-blocks, 32-token tiles)
  RouteParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.x = x; rp.gate = gate; rp.router_bias = router_bias; rp.expert_bias = expert_bias; rp.sh_gate = sh_gate;
  rp.T = T; rp.H = H; rp.E = E; rp.K = K;
  rp.score_fn = recipe->score_fn; rp.n_group = recipe->n_group; rp.topk_group = recipe->topk_group;
  rp.group_topn = recipe->group_topn; rp.renorm = recipe->norm_topk_prob; rp.eps = recipe->norm_eps;
  rp.scale = recipe->route_scale;
  rp.quads = L.rg.quads; rp.hsplit = L.rg.hsplit; rp.n_eb = L.rg.n_eb; rp.n_tb = L.rg.n_tb;
  rp.fold_sh = L.rg.fold_sh ? 1 : 0;
  rp.logits = reinterpret_cast<float*>(w + L.o_logits);
  rp.sh_logit = reinterpret_cast<float*>(w + L.o_shl);
  rp.idx = idx; rp.w = wts; rp.sh_w = Is > 0 ? sh_w : nullptr;
  rp.tb_counter = reinterpret_cast<int32_t*>(w + L.o_cnt);
  rp.glob_counter = rp.tb_counter + L.rg.n_tb;
  rp.do_permute = 1;
  rp.counts = counts; rp.offsets = reinterpret_cast<int32_t*>(w + L.o_offsets);
  rp.sorted_pair = sorted_pair; rp.pair_pos = pair_pos;
  rp.groups = groups; rp.header = header;
  rp.spans = reinterpret_cast<int64_t*>(w + L.o_spans);
  rp.span_groups = reinterpret_cast<int32_t*>(w + L.o_span_groups);
  rp.grid = L.grid;
  rp.I = I; rp.Is = Is; rp.n_max = L.n_max;
  rp.fmt = fp4 ? kFmtMxFp4 : kFmtMxFp8;
  rp.sh_fmt = kFmtMxFp8;
  rp.kblk = kMxK;
  rp.e2d = reinterpret_cast<int32_t*>(w + L.o_e2d);
  // the tile counters, readiness counters and the x-pieces counter
  rp.zero_ptr = tiles; rp.zero_count = 2 * L.max_gu_tiles + L.max_dn_tiles + 1;
  record_event_on(0, stream);
  cudaError_t e = cudaSuccess;
  int tb = L.rg.tb;
  if (T > kLogitsGemmMinTokens) {
    e = launch_logits_gemm(x, gate, sh_gate, router_bias, T, H, E, rp.logits, rp.sh_logit, L.lsplit,
                           reinterpret_cast<float*>(w + L.o_lpart), stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    rp.logits_given = 1;
    rp.lsplit = L.lsplit;
    rp.lpart = reinterpret_cast<const float*>(w + L.o_lpart);
    rp.fold_sh = 0;
    rp.n_eb = 1;
    tb = 8;
    rp.n_tb = ceil_div(T, tb);
  }
  e = launch_route(rp, tb, stream);
  record_event_on(1, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // ---- 2. both grouped GEMMs on the block-scaled MMA, one persistent launch
  CUtensorMap tm_gu, tm_gu_sh, tm_dn, tm_dn_sh;
  if (!encode_mx_3d(&tm_gu, w_gate_up_q, H, I, 2ull * E, fp4) || !encode_mx_3d(&tm_dn, w_down_q, I, H, E, fp4))
    return MOE_ERR_CUDA;
  if (Is > 0) {
    if (!encode_mx_3d(&tm_gu_sh, sh_gate_up_q, H, Is, 2, false) || !encode_mx_3d(&tm_dn_sh, sh_down_q, Is, H, 1, false))
      return MOE_ERR_CUDA;
  } else {
    tm_gu_sh = tm_gu;
    tm_dn_sh = tm_dn;
  }
  MxParams mp;
  memset(&mp, 0, sizeof(mp));
  mp.groups = groups; mp.header = header; mp.spans = rp.spans; mp.span_groups = rp.span_groups;
  mp.x = x;
  mp.sorted_pair = sorted_pair;
  mp.idx = idx;
  mp.pair_pos = pair_pos;
  mp.offsets = rp.offsets;
  mp.e2d = rp.e2d;
  mp.img_gu = reinterpret_cast<uint8_t*>(w + L.o_img_gu);
  mp.img_dn = reinterpret_cast<uint8_t*>(w + L.o_img_dn);
  mp.img_gu_rows = L.img_gu_rows;
  mp.img_dn_rows = L.img_dn_rows;
  mp.kb_gu = H / kMxK;
  mp.kb_dn = (Is > I ? Is : I) / kMxK;
  mp.mb0 = ceil_div(I, kHalfRows);
  mp.n_dense = L.n_dense;
  mp.img_ready = tiles + 2 * L.max_gu_tiles + L.max_dn_tiles;
  mp.T = T; mp.K = K; mp.TK = T * K; mp.H = H; mp.I_ld = Is > I ? Is : I;
  mp.n_max = L.n_max;
  mp.stage_space = kSmemLimit - 1024 - kCtrlBytes;
  mp.swiglu_limit = recipe->swiglu_limit;
  mp.out_ws = out_ws; mp.y = y; mp.direct_y = L.need_out ? 0 : 1;
  mp.topk_w = wts; mp.sh_w = (Is > 0 && sh_gate) ? sh_w : nullptr;
  mp.partials = reinterpret_cast<float*>(w + L.o_partials);
  mp.tile_counters_gu = tiles;
  mp.tile_counters_dn = tiles + L.max_gu_tiles;
  mp.ready = tiles + L.max_gu_tiles + L.max_dn_tiles;
  mp.status = status;
  mp.scales = static_cast<const uint8_t*>(scales);
  mp.I = I; mp.Is = Is; mp.E = E;
  mp.routed_fp4 = fp4 ? 1 : 0;
  mp.g_max = L.g_max;
  mp.max_gu_tiles = L.max_gu_tiles;
  mp.max_dn_tiles = L.max_dn_tiles;
  mp.max_gu_iters = static_cast<long long>(L.max_gu_tiles) * ceil_div(H, kMxK);
  mp.max_dn_iters = static_cast<long long>(L.max_dn_tiles) * ceil_div(mp.I_ld, kMxK);
  mp.pf = pf;
  record_event_on(2, stream);
  e = launch_mx(tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, mp, L.grid, kSmemLimit, stream);
  record_event_on(3, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // ---- 3. weighted combine (+ shared expert)
  if (L.need_out) {
    record_event_on(4, stream);
    e = launch_combine(out_ws, pair_pos, T, K, H, Is > 0 ? 1 : 0, y, stream);
    record_event_on(5, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

size_t fp4_scales_bytes(int E, int H, int I) {
  const size_t mb0 = ceil_div(I, kHalfRows), kb0 = H / kBlockK;
  const size_t mb1 = ceil_div(H, 2 * kHalfRows), kb1 = I / kBlockK;
  return static_cast<size_t>(E) * (mb0 * kb0 + mb1 * kb1) * 512;
}

bool fp4_shape_ok(int E, int H, int I) {
  return E >= 1 && E <= 1024 && H >= 64 && I >= 64 && H % 64 == 0 && I % 64 == 0 && H <= 65536 && I <= 16384;
}

}  // namespace

extern "C" {

moe_status moe_ffn_forward(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate, const float* router_bias,
                           const float* expert_bias, const moe_bf16* w_gate_up, const moe_bf16* w_down,
                           const moe_bf16* sh_gate_up, const moe_bf16* sh_down, int Is, const moe_bf16* sh_gate,
                           const moe_recipe* recipe, void* ws, size_t ws_bytes, moe_bf16* y,
                           int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out, cudaStream_t stream) {
  return ffn_forward(x, T, H, I, gate, router_bias, expert_bias, w_gate_up, w_down, sh_gate_up, sh_down, Is, sh_gate,
                     recipe, ws, ws_bytes, y, topk_idx_out, topk_w_out, counts_out, stream, nullptr);
}

size_t moe_fp4_scales_bytes(int E, int H, int I) { return fp4_shape_ok(E, H, I) ? fp4_scales_bytes(E, H, I) : 0; }

moe_status moe_fp4_prepare_scales(const uint8_t* w_gate_up_s, const uint8_t* w_down_s, int E, int H, int I,
                                  void* scales, size_t scales_bytes, cudaStream_t stream) {
  if (E < 1 || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (!fp4_shape_ok(E, H, I)) return MOE_ERR_UNSUPPORTED;
  if (!w_gate_up_s || !w_down_s || !scales || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
  if (scales_bytes < fp4_scales_bytes(E, H, I)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_fp4_scales(w_gate_up_s, w_down_s, E, H, I, static_cast<uint8_t*>(scales), stream));
}

moe_status moe_ffn_forward_fp4(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate,
                               const float* router_bias, const float* expert_bias, const uint8_t* w_gate_up_q,
                               const uint8_t* w_down_q, const void* scales, size_t scales_bytes,
                               const moe_bf16* sh_gate_up, const moe_bf16* sh_down, int Is, const moe_bf16* sh_gate,
                               const moe_recipe* recipe, void* ws, size_t ws_bytes, moe_bf16* y,
                               int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out, cudaStream_t stream) {
  if (check_recipe(recipe) != MOE_OK) return check_recipe(recipe);
  if (T < 0 || H < 8 || I < 8 || Is < 0) return MOE_ERR_INVALID_ARG;
  if (!fp4_shape_ok(recipe->num_experts, H, I)) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!w_gate_up_q || !w_down_q || !scales)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && scales_bytes < fp4_scales_bytes(recipe->num_experts, H, I)) return MOE_ERR_INVALID_ARG;
  const Fp4Experts f{w_gate_up_q, w_down_q, static_cast<const uint8_t*>(scales)};
  return ffn_forward(x, T, H, I, gate, router_bias, expert_bias, reinterpret_cast<const moe_bf16*>(w_gate_up_q),
                     reinterpret_cast<const moe_bf16*>(w_down_q), sh_gate_up, sh_down, Is, sh_gate, recipe, ws,
                     ws_bytes, y, topk_idx_out, topk_w_out, counts_out, stream, &f);
}

size_t moe_mx_scales_bytes(int routed_fmt, int E, int H, int I, int Is) {
  if ((routed_fmt != MOE_FMT_FP4 && routed_fmt != MOE_FMT_FP8) || Is < 0 || !mx_shape_ok(E, H, I, Is)) return 0;
  return mx_scales_bytes(E, H, I, Is);
}

moe_status moe_mx_prepare_scales(int routed_fmt, const uint8_t* w_gate_up_s, const uint8_t* w_down_s, int E, int H,
                                 int I, const uint8_t* sh_gate_up_s, const uint8_t* sh_down_s, int Is, void* scales,
                                 size_t scales_bytes, cudaStream_t stream) {
  if (routed_fmt != MOE_FMT_FP4 && routed_fmt != MOE_FMT_FP8) return MOE_ERR_INVALID_ARG;
  if (E < 1 || H < 1 || I < 1 || Is < 0) return MOE_ERR_INVALID_ARG;
  if (!mx_shape_ok(E, H, I, Is)) return MOE_ERR_UNSUPPORTED;
  if (!w_gate_up_s || !w_down_s || !scales || !aligned16(scales)) return MOE_ERR_INVALID_ARG;
  if (Is > 0 && (!sh_gate_up_s || !sh_down_s)) return MOE_ERR_INVALID_ARG;
  if (scales_bytes < mx_scales_bytes(E, H, I, Is)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_mx_scales(routed_fmt == MOE_FMT_FP4 ? 1 : 0, w_gate_up_s, w_down_s, E, H, I, sh_gate_up_s,
                                      sh_down_s, Is, static_cast<uint8_t*>(scales), stream));
}

moe_status moe_ffn_forward_mx(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate, const float* router_bias,
                              const float* expert_bias, int routed_fmt, const uint8_t* w_gate_up_q,
                              const uint8_t* w_down_q, const uint8_t* sh_gate_up_q, const uint8_t* sh_down_q, int Is,
                              const moe_bf16* sh_gate, const void* scales, size_t scales_bytes,
                              const moe_recipe* recipe, void* ws, size_t ws_bytes, moe_bf16* y,
                              int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out, cudaStream_t stream) {
  return ffn_forward_mx(x, T, H, I, gate, router_bias, expert_bias, routed_fmt, w_gate_up_q, w_down_q, sh_gate_up_q,
                        sh_down_q, Is, sh_gate, scales, scales_bytes, recipe, ws, ws_bytes, y, topk_idx_out,
                        topk_w_out, counts_out, stream);
}

moe_status moe_get_device_status(void* ws, cudaStream_t stream, int32_t* info_out) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t words[2] = {0, 0};
  if (cudaMemcpy(words, ws, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (info_out) *info_out = words[1];
  if (words[0] != 0 && cudaMemset(ws, 0, sizeof(words)) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(words[0]);
}

moe_status moe_set_schedule(int schedule) {
  if (schedule != MOE_SCHEDULE_AUTO && schedule != MOE_SCHEDULE_STREAM_K && schedule != MOE_SCHEDULE_SLICE)
    return MOE_ERR_INVALID_ARG;
  t_schedule = schedule;
  return MOE_OK;
}

moe_status moe_set_launch_overlap(int enable) {
  if (enable != 0 && enable != 1) return MOE_ERR_INVALID_ARG;
  t_overlap = enable;
  return MOE_OK;
}

int moe_ffn_schedule(int T, int H, int I, int Is, const moe_recipe* recipe, int gated) {
  if (check_recipe(recipe) != MOE_OK || T < 0 || H < 8 || I < 8 || Is < 0) return -1;
  const int sms = device_sms();
  if (sms <= 0) return -1;
  const int E = recipe->num_experts, K = recipe->top_k;
  const Layout L = make_layout(T, H, I, Is, E, K, gated != 0 && Is > 0, sms);
  return use_slice(L, T, E, K) ? MOE_SCHEDULE_SLICE : MOE_SCHEDULE_STREAM_K;
}

moe_status moe_set_l2_prefetch(const void* const* ptrs, const size_t* bytes, int n) {
  if (n < 0 || n > kMaxPrefetch || (n > 0 && (!ptrs || !bytes))) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return MOE_ERR_INVALID_ARG;
  L2Prefetch pf = {};
  for (int i = 0; i < n; ++i) {
    pf.ptr[i] = static_cast<const uint8_t*>(ptrs[i]);
    pf.bytes[i] = static_cast<long long>(bytes[i] & ~static_cast<size_t>(15));
  }
  pf.n = n;
  t_prefetch = pf;
  return MOE_OK;
}

void moe_set_profile_events(void* const* events, int n_pairs) {
  t_events = events;
  t_nev = events ? n_pairs : 0;
}

}  // extern "C"
