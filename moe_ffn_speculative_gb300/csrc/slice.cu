// Fused MoE-FFN forward for layers with few experts that every forward
// touches (e.g. 8 experts, top-1, a verify batch of 72 tokens): router,
// grouped SwiGLU experts, shared expert and weighted combine in one
// persistent launch.
//
// Sources (web pages): SpecForge PR #1033 "MoE FFN for DFlash-family drafts:
// the module", section "Router" (score -> select -> routing_weights);
// SpecForge PR #1073 "MoE drafts: DeepSeek-V4.1's own DSpark draft" (fused
// gate_up_proj [E,2I,H] and down_proj [E,H,I]; rows [0,I) of gate_up are the
// gate); SpecForge PR #941's follow-up comment (clamped SwiGLU); sglang PR
// #48763 "[Feat] dflash: Serve MoE FFN drafts for DFlash and DSpark", commit
// note on DraftMoE forward (routing weight times each expert's output, plus
// the shared expert).
//
// Work split.  CTA u < n_units owns unit (expert, s): slice s of 128 rows of
// the expert's intermediate dimension in the gate_up GEMM, and a share of
// the expert's 128-row output tiles in the down GEMM, so each unit streams
// about the same weight bytes and every weight byte is streamed once.
//   gate_up: 2 x 128 gate/up rows over H for ALL T tokens (x comes from L2
//     by TMA; the tensor pipe has room to spare).  It needs no routing and
//     starts at once, while the router runs on the CTAs after the units.  The
//     routing then picks the expert's tokens: their h = SwiGLU(gate, up) goes
//     to a global buffer, as the bf16 pair hi + lo already laid out as the
//     down GEMM's shared-memory operand, and the slice is flagged ready.
//   down: each output tile accumulates over the expert's whole intermediate
//     dimension, starting with the unit's own slice, the other slices' h
//     fetched (bulk copy) once their units flag them.  The epilogue applies
//     the routing weight and writes y directly (top-1, no shared expert) or
//     the pair's fp32 output row.
// An expert that no token picked stops streaming as soon as the routing is
// known and skips its down GEMM.  With top-k > 1 or a shared expert, combine
// tasks (output tile, group of tokens), taken in tile order by every CTA
// without other work, wait until every expert has finished the tile and sum
// the pair outputs in slot order: the result does not depend on timing.
//
// Consecutive forwards on a stream overlap: a launch lets the next one place
// its CTAs on the SMs it leaves (programmatic dependent launch); those CTAs
// load their first ring-full of gate/up weights and prefetch the next
// weights into L2 while the previous forward's last output tiles are being
// computed, and read x and the workspace only once it has completed.
//
// Unit CTA warp roles (224 threads): warp 0 issues the weight TMA loads,
// warp 1 allocates TMEM and issues the MMAs, warp 2 builds the unit's token
// list, then fetches the down GEMM's h tiles and publishes finished output
// tiles; warps 3..6 drain TMEM (SwiGLU into h, then the outputs).
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int kSliceThreads = 224;  // 7 warps
constexpr uint32_t kSliceTmemCols = 512;
// L2 prefetch at the start of a launch, while the previous launch on the
// stream ends: a unit's gate/up k-blocks after its first ring-full, a
// helper's first down k-blocks (up to 16 per output tile, 32 boxes of 16 KB).
constexpr int kSlicePrefetchGu = 6;
constexpr int kSlicePrefetchDnKb = 16;
constexpr int kSlicePrefetchDnBoxes = 32;

static_assert(kSliceTokPerTask == kSliceThreads / 32, "one combine token per warp");

struct SliceSmem {
  uint8_t* base;   // stage rings (gate_up and down use the same memory in turn)
  uint8_t* bbase;  // gate_up: the token tiles after the S weight parts
  uint32_t b_bytes;
  int S;
  uint64_t *full, *empty, *fullB, *emptyB, *acca, *accf, *acce, *routed, *drain, *hread;
  volatile int* abort_flag;
  volatile int* kb_stop;  // first gate_up k-block the producer did not issue
  volatile int* n_e;      // tokens routed to this unit's expert
  volatile int* task;
  int* grp_cnt;           // epilogue threads' count of finished down chunks
  int32_t* ss;            // this forward's counter set (router done, combine task, exit, -, tile counts)
  int32_t* ready;         // this forward's slice-ready flags
  uint32_t* tmem_slot;
  int* c_tok;    // [kSliceMaxTok] token of each down-GEMM column
  int* c_slot;   // [kSliceMaxTok] its output slot (pair t*K+k, or T*K+t for the shared expert)
  float* c_w;    // [kSliceMaxTok] its routing weight (or shared-expert gate)
  float* s_log;  // router: [7][33] logits of the CTA's tokens
};

__device__ __forceinline__ void carve(uint8_t* ctrl, SliceSmem& sm) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(ctrl);
  sm.full = bars;
  sm.empty = bars + 8;
  sm.fullB = bars + 16;
  sm.emptyB = bars + 24;
  sm.acca = bars + 32;
  sm.accf = bars + 33;
  sm.acce = bars + 34;
  sm.routed = bars + 35;
  sm.drain = bars + 36;
  sm.hread = bars + 37;  // the epilogue has read the gate_up accumulators
  int* words = reinterpret_cast<int*>(ctrl + 320);
  sm.tmem_slot = reinterpret_cast<uint32_t*>(words);
  sm.abort_flag = words + 1;
  sm.kb_stop = words + 2;
  sm.n_e = words + 3;
  sm.task = words + 4;
  sm.grp_cnt = words + 5;
  sm.c_tok = reinterpret_cast<int*>(ctrl + 512);
  sm.c_slot = sm.c_tok + kSliceMaxTok;
  sm.c_w = reinterpret_cast<float*>(sm.c_slot + kSliceMaxTok);
  sm.s_log = sm.c_w + kSliceMaxTok;
  sm.base = ctrl + kSliceCtrlBytes;
}
static_assert(512 + 3 * 4 * kSliceMaxTok + 4 * 7 * 33 <= kSliceCtrlBytes, "slice control block");

// Bounded wait until *p >= target.  Gives up (false) after about a second,
// or at once when another CTA has already recorded a failure.
__device__ bool wait_count(const int32_t* p, int target, const int32_t* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
    if (*reinterpret_cast<const volatile int32_t*>(status) != 0) return false;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// True on every epilogue thread (named barrier 1, 128 threads) when `v` is
// true on any of them: the four warps take each decision together.
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- router CTA
// Warp w routes token rc*7 + w: fp32 logits over the gate rows (and the
// shared-expert gate row), then score -> select -> weights.  The CTA's x rows
// and the gate rows are bulk-copied to shared memory in chunks of H (two
// buffers), so every load of a chunk is in flight at once: the router runs
// beside CTAs that keep HBM saturated, where a chain of dependent loads
// would wait behind them.
__device__ void route_tokens(const SliceParams& p, const SliceSmem& sm, int rc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = rc * kSliceTokPerTask;
  const int nt = min(kSliceTokPerTask, p.T - t0);
  const int E_tot = p.E + (p.sh_gate ? 1 : 0);
  const int rows = kSliceTokPerTask + E_tot;  // smem rows per buffer: x rows, then gate rows
  int hc = (p.stage_space / (2 * rows * 2)) / kBlockK * kBlockK;
  hc = min(hc, p.H);
  const int nchunks = ceil_div(p.H, hc);
  uint16_t* buf[2] = {reinterpret_cast<uint16_t*>(sm.base),
                      reinterpret_cast<uint16_t*>(sm.base) + static_cast<size_t>(rows) * hc};
  auto issue = [&](int c) {
    const int h0 = c * hc, len = min(hc, p.H - h0);
    uint16_t* dst = buf[c & 1];
    uint64_t* bar = &sm.full[c & 1];
    const uint32_t bytes = static_cast<uint32_t>(len) * 2u;
    mbar_arrive_expect_tx(bar, bytes * static_cast<uint32_t>(nt + E_tot));
    for (int i = 0; i < nt; ++i)
      bulk_load(dst + static_cast<size_t>(i) * hc, p.x + static_cast<size_t>(t0 + i) * p.H + h0, bytes, bar);
    for (int e = 0; e < E_tot; ++e) {
      const uint16_t* src = e < p.E ? p.gate + static_cast<size_t>(e) * p.H : p.sh_gate;
      bulk_load(dst + static_cast<size_t>(kSliceTokPerTask + e) * hc, src + h0, bytes, bar);
    }
  };
  if (threadIdx.x == 0) {
    issue(0);
    if (nchunks > 1) issue(1);
  }
  float acc[kSliceMaxExperts];
#pragma unroll
  for (int e = 0; e < kSliceMaxExperts; ++e) acc[e] = 0.f;
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    ok = ok && mbar_wait(&sm.full[c & 1], static_cast<uint32_t>(c >> 1) & 1u, sm.abort_flag);
    if (ok && warp < nt) {
      const int len = min(hc, p.H - c * hc);
      const uint16_t* xs = buf[c & 1] + static_cast<size_t>(warp) * hc;
      const uint16_t* gs = buf[c & 1] + static_cast<size_t>(kSliceTokPerTask) * hc;
      for (int i = lane * 8; i < len; i += 256) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + i);
#pragma unroll
        for (int e = 0; e < kSliceMaxExperts; ++e)
          if (e < E_tot) acc[e] = dot8(xv, *reinterpret_cast<const uint4*>(gs + static_cast<size_t>(e) * hc + i), acc[e]);
      }
    }
    ok = __syncthreads_and(ok) != 0;  // buffer c & 1 is free again; every thread takes the same way
    if (threadIdx.x == 0 && ok && c + 2 < nchunks) issue(c + 2);
  }
  if (!ok) {
    if (threadIdx.x == 0) record_failure(p.status, sm.abort_flag, kInfoRouter);
    return;
  }
  if (warp < nt) {
    const int t = t0 + warp;
    float* lrow = sm.s_log + warp * 33;
#pragma unroll
    for (int e = 0; e < kSliceMaxExperts; ++e) {
      if (e < E_tot) {
        float v = acc[e];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) {
          if (e < p.E) {
            if (p.router_bias) v += __ldg(p.router_bias + e);
            lrow[e] = v;
            p.logits[static_cast<size_t>(t) * p.E + e] = v;
          } else {
            p.sh_w[t] = 1.f / (1.f + expf(-v));
          }
        }
      }
    }
    if (lane == 0 && p.s_sh > 0 && !p.sh_gate) p.sh_w[t] = 1.f;
    __syncwarp();
    select_token<1, true>(lrow, p.sel, p.idx + static_cast<size_t>(t) * p.K, p.w + static_cast<size_t>(t) * p.K);
  }
  __syncthreads();
  if (threadIdx.x == 0) red_release_add(sm.ss + 0, 1);
}

// ---------------------------------------------------------------- unit CTA roles
// A CTA's share of the experts' work.  A unit (has_a) owns slice s of an
// expert in the gate_up GEMM; every CTA that is not a unit (the router CTAs
// once routing is done, and the rest) is a down-only helper of one expert.
// An expert's down work is n_mt 128-row output tiles, each cut into
// p.parts ranges of its k-blocks (items, tile-major); the items are split
// evenly over the expert's units and helpers.
struct Unit {
  bool has_a;   // runs the gate_up GEMM for slice s
  bool shared;
  int e, s;     // expert (-1: shared) and slice (units)
  int es;       // expert slot of the h buffer and ready flags: e, or E for the shared expert
  int nkb;      // gate_up k-blocks: ceil(H / 64), 0 for helpers
  int nkb_d;    // down k-blocks: 2 per slice of the expert
  int kstart;   // first down k-block: the unit's own slice, 0 for helpers
  int i0, ni;   // the CTA's down items [i0, i0 + ni)
};

__device__ __forceinline__ Unit make_unit(const SliceParams& p, int bid) {
  Unit u;
  const int n_es = p.E + (p.s_sh > 0 ? 1 : 0);  // experts with units, the shared one last
  const int n_help = static_cast<int>(gridDim.x) - p.n_units;
  int w;  // worker index within the expert: units first, then helpers
  if (bid < p.n_units) {
    u.has_a = true;
    u.shared = bid >= p.E * p.s_e;
    u.es = u.shared ? p.E : bid / max(p.s_e, 1);
    u.s = u.shared ? bid - p.E * p.s_e : bid % max(p.s_e, 1);
    w = u.s;
  } else {
    const int h = bid - p.n_units;
    u.has_a = false;
    u.es = h % n_es;
    u.shared = u.es == p.E;
    u.s = -1;
    w = (u.shared ? p.s_sh : p.s_e) + h / n_es;
  }
  u.e = u.shared ? -1 : u.es;
  const int su = u.shared ? p.s_sh : p.s_e;
  const int workers = su + (n_help > u.es ? (n_help - 1 - u.es) / n_es + 1 : 0);
  u.nkb = u.has_a ? ceil_div(p.H, kBlockK) : 0;
  u.nkb_d = 2 * su;
  u.kstart = u.has_a ? 2 * u.s : 0;
  const int items = p.n_mt * p.parts;
  u.i0 = items * w / workers;
  u.ni = items * (w + 1) / workers - u.i0;
  return u;
}

// h tile (expert slot es, down k-block kb): 2*n_tok rows of 128 bytes, the
// K-major 128-byte-swizzled image of the MMA operand; rows [0, n16) hold
// h_hi of the expert's picked tokens, rows [n16, 2*n16) their h_lo, so one
// MMA of width 2*n16 computes W*h_hi and W*h_lo side by side.
__device__ __forceinline__ uint8_t* h_tile(const SliceParams& p, int es, int kb) {
  return p.hbuf + (static_cast<size_t>(es) * 2 * p.s_max + kb) * 2 * p.n_tok * 128;
}

// Down-GEMM geometry of a chunk of output tiles: how many tiles share one
// pass over the k-blocks (TMEM columns and stage size), and the stage size.
struct DownGeom {
  int cj;            // tiles per chunk
  uint32_t hbytes;   // h tile bytes: 2*n16 rows
  uint32_t stage;    // bytes per stage: cj weight boxes + the h tile
  int S;             // stages
};

__device__ __forceinline__ DownGeom down_geom(const SliceParams& p, const Unit& u, int n) {
  DownGeom g;
  const int n16 = (n + 15) & ~15;
  g.hbytes = static_cast<uint32_t>(2 * n16 * 128);
  const int by_tmem = static_cast<int>(kSliceTmemCols) / (2 * n16);
  const int by_smem = (p.stage_space / 3 - static_cast<int>(g.hbytes)) / kTileBytesA;
  g.cj = p.parts == 1 ? max(1, min(u.ni, min(by_tmem, by_smem))) : 1;
  g.stage = static_cast<uint32_t>(g.cj) * kTileBytesA + g.hbytes;
  g.S = min(8, p.stage_space / static_cast<int>(g.stage));
  return g;
}

// One pass of the down GEMM over a range of k-blocks for cj output tiles
// together (one TMEM accumulator each).  With one part per tile a pass is a
// chunk of whole tiles over every k-block, a unit's own slice first; with
// several parts a pass is one item: a tile over its part's k-blocks.
struct Pass {
  int j0, cj;    // output tiles [j0, j0 + cj)
  int ka, kn;    // k-blocks [ka, ka + kn)
  int rot;       // taken from ka + rot on, wrapping
  int part;
};

__device__ __forceinline__ int n_passes(const SliceParams& p, const Unit& u, const DownGeom& g) {
  return p.parts == 1 ? ceil_div(u.ni, g.cj) : u.ni;
}

__device__ __forceinline__ Pass down_pass(const SliceParams& p, const Unit& u, const DownGeom& g, int pi) {
  Pass ps;
  if (p.parts == 1) {
    ps.j0 = u.i0 + pi * g.cj;
    ps.cj = min(g.cj, u.ni - pi * g.cj);
    ps.ka = 0;
    ps.kn = u.nkb_d;
    ps.rot = u.kstart;
    ps.part = 0;
  } else {
    const int it = u.i0 + pi;
    ps.j0 = it / p.parts;
    ps.cj = 1;
    ps.part = it - ps.j0 * p.parts;
    ps.ka = u.nkb_d * ps.part / p.parts;
    ps.kn = u.nkb_d * (ps.part + 1) / p.parts - ps.ka;
    ps.rot = 0;
  }
  return ps;
}

// k-block q of a pass
__device__ __forceinline__ int pass_kb(const Pass& ps, int q) {
  const int k = q + ps.rot;
  return ps.ka + (k < ps.kn ? k : k - ps.kn);
}

// The loads of gate_up k-block kb into its (free) stage: the slice's gate and
// up rows and (with_x) every token's x; without x, the caller loads the
// x tile later on the same barrier.
__device__ __forceinline__ void unit_load_gu(const SliceParams& p, const SliceSmem& sm, const Unit& u,
                                             const CUtensorMap* tm_gu, const CUtensorMap* tm_gu_sh,
                                             const CUtensorMap* tm_x, int kb, int stage, bool with_x = true) {
  const CUtensorMap* gu = u.shared ? tm_gu_sh : tm_gu;
  const int zg = u.shared ? 0 : 2 * u.e;
  uint8_t* st = sm.base + stage * 2 * kTileBytesA;
  uint64_t* bar = &sm.full[stage];
  mbar_arrive_expect_tx(bar, 2 * kTileBytesA + sm.b_bytes);
  // weights are streamed once: evict-first, so that L2 keeps x, h and the
  // router's operands
  const uint64_t pol = l2_evict_first_policy();
  tma_load_3d_hint(st, gu, bar, kb * kBlockK, u.s * kHalfRows, zg, pol);                    // gate rows
  tma_load_3d_hint(st + kTileBytesA, gu, bar, kb * kBlockK, u.s * kHalfRows, zg + 1, pol);  // up rows
  if (with_x) tma_load_2d(sm.bbase + stage * sm.b_bytes, tm_x, bar, kb * kBlockK, 0);       // every token
}

// L2 prefetch of the weights the CTA streams first after its ring-full: a
// unit's next gate/up k-blocks; a helper's first down k-blocks, in the order
// its passes take them (its output tiles are fixed before the routing is
// known, only the tokens it multiplies are not).
__device__ void prefetch_first_weights(const SliceParams& p, const Unit& u, const CUtensorMap* tm_gu,
                                       const CUtensorMap* tm_gu_sh, const CUtensorMap* tm_dn,
                                       const CUtensorMap* tm_dn_sh, int kb_first) {
  if (u.has_a) {
    const CUtensorMap* gu = u.shared ? tm_gu_sh : tm_gu;
    const int zg = u.shared ? 0 : 2 * u.e;
    for (int kb = kb_first; kb < min(u.nkb, kb_first + kSlicePrefetchGu); ++kb) {
      tma_prefetch_l2_3d(gu, kb * kBlockK, u.s * kHalfRows, zg);
      tma_prefetch_l2_3d(gu, kb * kBlockK, u.s * kHalfRows, zg + 1);
    }
    return;
  }
  if (u.ni == 0) return;
  const CUtensorMap* dn = u.shared ? tm_dn_sh : tm_dn;
  const int zd = u.shared ? 0 : u.e;
  if (p.parts == 1) {
    const int kq = min(u.nkb_d, min(kSlicePrefetchDnKb, kSlicePrefetchDnBoxes / u.ni));
    for (int q = 0; q < kq; ++q) {
      const int kbd = (q + u.kstart) % u.nkb_d;
      for (int jj = 0; jj < u.ni; ++jj) tma_prefetch_l2_3d(dn, kbd * kBlockK, (u.i0 + jj) * kHalfRows, zd);
    }
  } else {
    int boxes = kSlicePrefetchDnBoxes;
    for (int it = u.i0; it < u.i0 + u.ni && boxes > 0; ++it) {
      const int j = it / p.parts, part = it - j * p.parts;
      const int ka = u.nkb_d * part / p.parts, kn = u.nkb_d * (part + 1) / p.parts - ka;
      for (int q = 0; q < kn && boxes > 0; ++q, --boxes) tma_prefetch_l2_3d(dn, (ka + q) * kBlockK, j * kHalfRows, zd);
    }
  }
}

// k-blocks [0, kb_first) were issued into the fresh ring by the prologue.
__device__ void unit_produce(const SliceParams& p, const SliceSmem& sm, const Unit& u, const CUtensorMap* tm_gu,
                             const CUtensorMap* tm_gu_sh, const CUtensorMap* tm_dn, const CUtensorMap* tm_dn_sh,
                             const CUtensorMap* tm_x, int kb_first) {
  if (u.has_a && !wait_start_gate(p.status)) {
    // the start gate stayed closed: the MMAs stop after the prologue's loads
    record_failure(p.status, sm.abort_flag, kInfoHold);
    *sm.kb_stop = kb_first;
    return;
  }
  Ring ring;
  for (int i = 0; i < kb_first; ++i) ring.next(sm.S);
  int kb = kb_first;
  for (; kb < u.nkb; ++kb) {
    // an expert no token picked stops streaming once the routing is known
    if (!u.shared && mbar_test_wait(sm.routed, 0) && *sm.n_e == 0) break;
    if (!mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag)) {
      record_failure(p.status, sm.abort_flag, kInfoEmpty);
      break;
    }
    unit_load_gu(p, sm, u, tm_gu, tm_gu_sh, tm_x, kb, ring.stage);
    ring.next(sm.S);
  }
  if (kb < u.nkb) {
    *sm.kb_stop = kb;
    return;
  }
  if (!mbar_wait(sm.routed, 0, sm.abort_flag)) return;
  const int n = *sm.n_e;
  if (n == 0 || u.ni == 0) return;
  // The down ring reuses the gate_up ring's memory once the MMAs have read
  // every gate_up stage.
  for (int i = 0; i < sm.S; ++i) {
    if (!mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag)) {
      record_failure(p.status, sm.abort_flag, kInfoEmpty);
      return;
    }
    ring.next(sm.S);
  }
  const DownGeom g = down_geom(p, u, n);
  const CUtensorMap* dn = u.shared ? tm_dn_sh : tm_dn;
  const int zd = u.shared ? 0 : u.e;
  const uint64_t pol = l2_evict_first_policy();
  Ring rb;
  const int np = n_passes(p, u, g);
  for (int pi = 0; pi < np; ++pi) {
    const Pass ps = down_pass(p, u, g, pi);
    for (int q = 0; q < ps.kn; ++q) {
      const int kbd = pass_kb(ps, q);
      if (!mbar_wait(&sm.emptyB[rb.stage], rb.phase ^ 1u, sm.abort_flag)) {
        record_failure(p.status, sm.abort_flag, kInfoEmpty);
        return;
      }
      uint8_t* st = sm.base + rb.stage * g.stage;
      uint64_t* bar = &sm.fullB[rb.stage];
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ps.cj) * kTileBytesA);
      for (int jj = 0; jj < ps.cj; ++jj)
        tma_load_3d_hint(st + jj * kTileBytesA, dn, bar, kbd * kBlockK, (ps.j0 + jj) * kHalfRows, zd, pol);
      rb.next(g.S);
    }
  }
}

__device__ void unit_mma(const SliceParams& p, const SliceSmem& sm, const Unit& u, uint32_t tmem) {
  Ring ring;
  const uint32_t idesc_a = idesc_bf16(kHalfRows, p.n_tok);
  const uint32_t d_gate = tmem, d_up = tmem + 128;
  bool ok = true;
  for (int kb = 0; kb < u.nkb; ++kb) {
    // the stage, or the news that the producer stopped before it
    bool got = mbar_try_wait(&sm.full[ring.stage], ring.phase);
    if (!got) {
      const long long t0 = clock64();
      while (true) {
        if (mbar_try_wait(&sm.full[ring.stage], ring.phase)) { got = true; break; }
        if (*sm.kb_stop <= kb || *sm.abort_flag) break;
        if (clock64() - t0 > kWaitLimitCycles) {
          record_failure(p.status, sm.abort_flag, kInfoFull);
          break;
        }
      }
    }
    if (!got) { ok = false; break; }
    tc_fence_after();
    const uint32_t a0 = smem_u32(sm.base + ring.stage * 2 * kTileBytesA);
    const uint32_t a1 = a0 + kTileBytesA, b = smem_u32(sm.bbase + ring.stage * sm.b_bytes);
#pragma unroll
    for (int ks = 0; ks < kBlockK / 16; ++ks) {
      const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
      const uint64_t bd = sw128_desc(b + ks * 32);
      mma_bf16(d_gate, sw128_desc(a0 + ks * 32), bd, idesc_a, acc);
      mma_bf16(d_up, sw128_desc(a1 + ks * 32), bd, idesc_a, acc);
    }
    mma_commit(&sm.empty[ring.stage]);
    ring.next(sm.S);
  }
  mma_commit(sm.acca);
  if (ok && mbar_wait(sm.routed, 0, sm.abort_flag) && *sm.n_e > 0 && u.ni > 0) {
    const int n = *sm.n_e;
    const int n16 = (n + 15) & ~15;
    const DownGeom g = down_geom(p, u, n);
    const uint32_t idesc_b = idesc_bf16(kHalfRows, 2 * n16);
    Ring rb;
    const int np = n_passes(p, u, g);
    for (int pi = 0; pi < np && ok; ++pi) {
      const Pass ps = down_pass(p, u, g, pi);
      const int cj = ps.cj;
      // The TMEM accumulators are free once the epilogue drained the last
      // pass; a unit's first pass waits until its epilogue has read the
      // gate_up accumulators (helpers have none).
      if (pi > 0) {
        if (!mbar_wait(sm.acce, static_cast<uint32_t>(pi - 1) & 1u, sm.abort_flag)) {
          record_failure(p.status, sm.abort_flag, kInfoAccEmpty);
          break;
        }
        tc_fence_after();
      } else if (u.has_a) {
        // the down accumulators overwrite the gate_up ones: after the epilogue read them
        if (!mbar_wait(sm.hread, 0, sm.abort_flag)) {
          record_failure(p.status, sm.abort_flag, kInfoHReady);
          break;
        }
        tc_fence_after();
      }
      for (int q = 0; q < ps.kn; ++q) {
        if (!mbar_wait(&sm.fullB[rb.stage], rb.phase, sm.abort_flag)) {
          record_failure(p.status, sm.abort_flag, kInfoFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sm.base + rb.stage * g.stage);
        const uint32_t hb = a0 + static_cast<uint32_t>(cj) * kTileBytesA;
        for (int jj = 0; jj < cj; ++jj) {
          const uint32_t d = tmem + static_cast<uint32_t>(jj * 2 * n16);
#pragma unroll
          for (int ks = 0; ks < kBlockK / 16; ++ks)
            mma_bf16(d, sw128_desc(a0 + jj * kTileBytesA + ks * 32), sw128_desc(hb + ks * 32), idesc_b,
                     (q > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(&sm.emptyB[rb.stage]);
        rb.next(g.S);
      }
      mma_commit(sm.accf);
    }
  }
  // every MMA issued above has completed once `drain` flips
  mma_commit(sm.drain);
  if (!mbar_wait(sm.drain, 0, nullptr)) record_failure(p.status, sm.abort_flag, kInfoDrain);
}

// Release-publish output tiles [j0, j1) as finished (combine counters).
__device__ __forceinline__ void publish_tiles(const SliceSmem& sm, int j0, int j1) {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  for (int j = j0; j < j1; ++j)
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(sm.ss + kSliceSyncWords + j) : "memory");
}

// Each of the CTA's down items counts once for its tile.
__device__ __forceinline__ void publish_items(const SliceParams& p, const SliceSmem& sm, const Unit& u) {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  for (int i = u.i0; i < u.i0 + u.ni; ++i)
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(sm.ss + kSliceSyncWords + i / p.parts) : "memory");
}

// Warp 2: the unit's token list once the router CTAs have finished; then
// (lane 0) the down GEMM's h tiles, fetched as their slices are flagged, and
// the release of finished output tiles to the combine.
__device__ void unit_tokens(const SliceParams& p, const SliceSmem& sm, const Unit& u) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0) ok = wait_count(sm.ss + 0, p.n_rcta, p.status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();  // orders every lane's reads of the routing after lane 0's acquire
  if (!ok) {
    if (lane == 0) {
      record_failure(p.status, sm.abort_flag, kInfoRouter);
      *sm.n_e = 0;
      mbar_arrive(sm.routed);
    }
    return;
  }
  int n = 0;
  if (u.shared) {
    for (int t = lane; t < p.T; t += 32) {
      sm.c_tok[t] = t;
      sm.c_slot[t] = p.TK + t;
      sm.c_w[t] = __ldcg(p.sh_w + t);
    }
    n = p.T;
  } else {
    // pairs in (token, slot) order; a token picks an expert at most once
    for (int base = 0; base < p.TK; base += 32) {
      const int pr = base + lane;
      const bool hit = pr < p.TK && __ldcg(p.idx + pr) == u.e;
      const uint32_t mask = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        const int c = n + __popc(mask & ((1u << lane) - 1u));
        if (c < kSliceMaxTok) {
          sm.c_tok[c] = pr / p.K;
          sm.c_slot[c] = pr;
          sm.c_w[c] = __ldcg(p.w + pr);
        }
      }
      n += __popc(mask);
    }
    n = min(n, kSliceMaxTok);
    if (u.s == 0 && lane == 0) p.counts[u.e] = n;
  }
  __syncwarp();
  if (lane == 0) {
    *sm.n_e = n;
    mbar_arrive(sm.routed);
  }
  if (lane != 0) return;
  if (n == 0 || u.ni == 0) {
    // nothing to add to this unit's output tiles
    if (!p.direct_y && !*sm.abort_flag) publish_items(p, sm, u);
    return;
  }
  // The down ring aliases the gate_up ring: a unit's h fetches must wait
  // until its MMAs have read every gate_up stage (and so every gate_up load
  // has landed), however early the other slices are flagged ready.
  if (u.has_a && !mbar_wait(sm.acca, 0, sm.abort_flag)) {
    record_failure(p.status, sm.abort_flag, kInfoAccFull);
    return;
  }
  const DownGeom g = down_geom(p, u, n);
  Ring rb;
  const int np = n_passes(p, u, g);
  for (int pi = 0; pi < np; ++pi) {
    const Pass ps = down_pass(p, u, g, pi);
    const int cj = ps.cj;
    int seen = -1;  // last slice found ready
    int q = 0;
    if (pi == 0 && u.has_a && p.parts == 1) {
      // the epilogue fills the first two stages with the unit's own slice
      rb.next(g.S);
      rb.next(g.S);
      q = 2;
    }
    for (; q < ps.kn; ++q) {
      const int kbd = pass_kb(ps, q);
      const int sl = kbd >> 1;
      if (sl != seen) {
        if (!wait_count(sm.ready + u.es * p.s_max + sl, 1, p.status)) {
          record_failure(p.status, sm.abort_flag, kInfoReady);
          return;
        }
        // the slice's h was written by generic stores: order them before the bulk copy
        asm volatile("fence.proxy.async.global;" ::: "memory");
        seen = sl;
      }
      if (!mbar_wait(&sm.emptyB[rb.stage], rb.phase ^ 1u, sm.abort_flag)) {
        record_failure(p.status, sm.abort_flag, kInfoGatherEmpty);
        return;
      }
      uint8_t* st = sm.base + rb.stage * g.stage + cj * kTileBytesA;
      uint64_t* bar = &sm.fullB[rb.stage];
      mbar_arrive_expect_tx(bar, g.hbytes);
      bulk_load(st, h_tile(p, u.es, kbd), g.hbytes, bar);
      rb.next(g.S);
    }
    if (!p.direct_y) {
      // the pass's outputs are stored once every epilogue thread has counted it
      const uint32_t target = 128u * static_cast<uint32_t>(pi + 1);
      const long long t0 = clock64();
      while (true) {
        uint32_t v;
        asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(sm.grp_cnt)) : "memory");
        if (v >= target) break;
        if (*sm.abort_flag) return;
        if (clock64() - t0 > kWaitLimitCycles) {
          record_failure(p.status, sm.abort_flag, kInfoAccFull);
          return;
        }
      }
      publish_tiles(sm, ps.j0, ps.j0 + cj);
    }
  }
}

// Warps 3..6: SwiGLU of the picked tokens into the h buffer, then the down
// GEMM's weighted outputs, one chunk of output tiles at a time.
__device__ void unit_epilogue(const SliceParams& p, const SliceSmem& sm, const Unit& u, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;  // TMEM lane: slice row (gate_up) / row in the output tile (down)
  const bool leader = (warp == 3 && lane == 0);
  const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
  if (epi_any(!mbar_wait(sm.routed, 0, sm.abort_flag) || *sm.abort_flag)) return;
  const int n = *sm.n_e;
  if (n == 0) return;
  const int n16 = (n + 15) & ~15;
  const DownGeom g = down_geom(p, u, n);
  if (u.has_a) {
  if (epi_any(!mbar_wait(sm.acca, 0, sm.abort_flag))) {
    if (leader) record_failure(p.status, sm.abort_flag, kInfoAccFull);
    return;
  }
  tc_fence_after();
  // The down GEMM takes the unit's own slice first: its two k-blocks are
  // the first two stages of the down ring, whose h parts this epilogue
  // fills directly (the gate_up stages are all read by now), besides the
  // global copy the expert's other units fetch.
  const bool local = u.ni > 0 && p.parts == 1;
  {
    const float lim = p.swiglu_limit;
    const int k2 = r >> 6, kin = r & 63;
    uint8_t* th = h_tile(p, u.es, 2 * u.s + k2);
    uint8_t* tl = th + n16 * 128;
    uint8_t* sh = sm.base + k2 * g.stage + min(g.cj, u.ni) * kTileBytesA;
    for (int c0 = 0; c0 < n; c0 += 8) {
      uint32_t g[8], v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int tok = sm.c_tok[min(c0 + i, n - 1)];
        g[i] = tmem_ld1(tmem + lanes + static_cast<uint32_t>(tok));
        v[i] = tmem_ld1(tmem + lanes + 128u + static_cast<uint32_t>(tok));
      }
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + i;
        if (c < n) {
          float gv = __uint_as_float(g[i]), uv = __uint_as_float(v[i]);
          if (lim > 0.f) {
            gv = fminf(gv, lim);
            uv = fminf(fmaxf(uv, -lim), lim);
          }
          const float hv = gv / (1.f + expf(-gv)) * uv;
          const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
          const float lo = hv - __bfloat162float(hi);
          // row c, column kin of a K-major tile with the 128-byte swizzle
          // (n16 is a multiple of 8: the lo rows keep the same swizzle phase)
          const uint32_t off = static_cast<uint32_t>(c * 128 + ((((kin >> 3) ^ (c & 7)) << 4) | ((kin & 7) * 2)));
          const uint16_t hb = __bfloat16_as_ushort(hi), lb = f2bf(lo);
          *reinterpret_cast<uint16_t*>(th + off) = hb;
          *reinterpret_cast<uint16_t*>(tl + off) = lb;
          if (local) {
            *reinterpret_cast<uint16_t*>(sh + off) = hb;
            *reinterpret_cast<uint16_t*>(sh + n16 * 128 + off) = lb;
          }
        }
      }
    }
  }
  // the TMEM accumulators are read: the down GEMM may overwrite them
  tc_fence_before();
  // publish the slice's h: every thread's stores precede the leader's
  // release (global copy) and its arrivals on the first two down stages
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  epi_sync();
  if (leader) {
    mbar_arrive(sm.hread);
    if (local) {
      mbar_arrive(&sm.fullB[0]);
      mbar_arrive(&sm.fullB[1]);
    }
    red_release_add(sm.ready + u.es * p.s_max + u.s, 1);
  }
  }  // has_a
  if (u.ni == 0) return;
  // a part's fp32 partials go to its own plane of the pair outputs
  float* out = p.out;
  const int np = n_passes(p, u, g);
  for (int pi = 0; pi < np; ++pi) {
    const Pass ps = down_pass(p, u, g, pi);
    const int cj = ps.cj;
    if (p.parts > 1) out = p.out + static_cast<size_t>(ps.part) * (p.TK + p.T) * p.H;
    if (epi_any(!mbar_wait(sm.accf, static_cast<uint32_t>(pi) & 1u, sm.abort_flag))) {
      if (leader) record_failure(p.status, sm.abort_flag, kInfoAccFull);
      return;
    }
    tc_fence_after();
    for (int jj = 0; jj < cj; ++jj) {
      const int row = (ps.j0 + jj) * kHalfRows + r;
      const uint32_t d = tmem + lanes + static_cast<uint32_t>(jj * 2 * n16);
      for (int c0 = 0; c0 < n16; c0 += 16) {
        uint32_t vh[16], vl[16];
        tmem_ld16(d + static_cast<uint32_t>(c0), vh);        // W * h_hi
        tmem_ld16(d + static_cast<uint32_t>(n16 + c0), vl);  // W * h_lo
        tmem_ld_wait();
        if (row < p.H) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (c < n) {
              const float v = sm.c_w[c] * (__uint_as_float(vh[i]) + __uint_as_float(vl[i]));
              if (p.direct_y)
                p.y[static_cast<size_t>(sm.c_tok[c]) * p.H + row] = f2bf(v);
              else
                __stcg(out + static_cast<size_t>(sm.c_slot[c]) * p.H + row, v);
            }
          }
        }
      }
    }
    tc_fence_before();
    mbar_arrive(sm.acce);
    if (!p.direct_y)
      asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" ::"r"(smem_u32(sm.grp_cnt)) : "memory");
  }
}

// ---------------------------------------------------------------- combine
// Task (m, g): y[t, m*128 : m*128+128] for the 7 tokens of group g, once
// every expert (and the shared expert) has finished every part of tile m.
// Warp w sums token g*7+w in (slot, part) order; lane l four rows.
__device__ void combine_tasks(const SliceParams& p, const SliceSmem& sm) {
  if (p.direct_y) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tasks = p.n_mt * p.n_tg;
  const int target = (p.E + (p.s_sh > 0 ? 1 : 0)) * p.parts;
  int32_t* tile_cnt = sm.ss + kSliceSyncWords;
  while (true) {
    if (threadIdx.x == 0) {
      int task = atomicAdd(sm.ss + 1, 1);
      if (task < n_tasks && !wait_count(tile_cnt + task / p.n_tg, target, p.status)) {
        record_failure(p.status, sm.abort_flag, kInfoTileCount);
        task = n_tasks;
      }
      *sm.task = task;
    }
    __syncthreads();
    const int task = *sm.task;
    __syncthreads();
    if (task >= n_tasks) break;
    const int m = task / p.n_tg, tg = task - m * p.n_tg;
    const int t = tg * kSliceTokPerTask + warp;
    const int row = m * kHalfRows + lane * 4;
    if (t < p.T && row < p.H) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      const int nslot = p.K + (p.s_sh > 0 ? 1 : 0);
      for (int k = 0; k < nslot; ++k) {
        const int slot = k < p.K ? t * p.K + k : p.TK + t;
        for (int part = 0; part < p.parts; ++part) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(
              p.out + (static_cast<size_t>(part) * (p.TK + p.T) + slot) * p.H + row));
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
      }
      uint2 o;
      o.x = static_cast<uint32_t>(f2bf(acc.x)) | (static_cast<uint32_t>(f2bf(acc.y)) << 16);
      o.y = static_cast<uint32_t>(f2bf(acc.z)) | (static_cast<uint32_t>(f2bf(acc.w)) << 16);
      *reinterpret_cast<uint2*>(p.y + static_cast<size_t>(t) * p.H + row) = o;
    }
  }
}

__global__ void __launch_bounds__(kSliceThreads, 1)
    moe_slice_kernel(const __grid_constant__ CUtensorMap tm_gu, const __grid_constant__ CUtensorMap tm_gu_sh,
                     const __grid_constant__ CUtensorMap tm_dn, const __grid_constant__ CUtensorMap tm_dn_sh,
                     const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ SliceParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ctrl = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  SliceSmem sm;
  carve(ctrl, sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bid = static_cast<int>(blockIdx.x);
  const bool is_unit = bid < p.n_units;
  const Unit u = make_unit(p, bid);
  sm.b_bytes = static_cast<uint32_t>(p.n_tok) * 128u;
  sm.S = min(8, p.stage_space / static_cast<int>(2 * kTileBytesA + sm.b_bytes));
  sm.bbase = sm.base + sm.S * 2 * kTileBytesA;
  int kb_first = 0;  // gate_up k-blocks issued by the prologue (thread 0 is the producer)
  if (threadIdx.x == 0) {
    for (int s = 0; s < 8; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
      mbar_init(&sm.fullB[s], 2);  // weight loads and h fetch arrive separately
      mbar_init(&sm.emptyB[s], 1);
    }
    mbar_init(sm.acca, 1);
    mbar_init(sm.accf, 1);
    mbar_init(sm.acce, 128);
    mbar_init(sm.routed, 1);
    mbar_init(sm.drain, 1);
    mbar_init(sm.hread, 1);
    *sm.abort_flag = 0;
    *sm.kb_stop = u.nkb;
    *sm.n_e = 0;
    *sm.grp_cnt = 0;
    fence_barrier_init();
    fence_proxy_async();
    if (is_unit) {
      // the first ring-full of gate/up weights goes out before the rest of
      // the prologue, and before the previous launch on the stream has
      // ended (a forward never writes weights); their x tiles once it has
      kb_first = min(sm.S, u.nkb);
      for (int kb = 0; kb < kb_first; ++kb) unit_load_gu(p, sm, u, &tm_gu, &tm_gu_sh, &tm_x, kb, kb, false);
    }
    prefetch_first_weights(p, u, &tm_gu, &tm_gu_sh, &tm_dn, &tm_dn_sh, kb_first);
  }
  const bool works = is_unit || u.ni > 0;
  if (works && warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_gu);
    tma_prefetch_desc(&tm_dn);
    tma_prefetch_desc(&tm_x);
    if (p.s_sh > 0) {
      tma_prefetch_desc(&tm_gu_sh);
      tma_prefetch_desc(&tm_dn_sh);
    }
  }
  if (works && warp == 1) {
    tmem_alloc(sm.tmem_slot, kSliceTmemCols);
    tmem_relinquish();
  }
  // The next forward on the stream may place its CTAs on the SMs this one
  // leaves and start streaming its weights; everything that reads what the
  // previous launch wrote (x, the workspace, the counter sets) waits until
  // that launch has completed.
  griddep_launch_dependents();
  griddep_wait();
  if (threadIdx.x == 0)
    for (int kb = 0; kb < kb_first; ++kb) tma_load_2d(sm.bbase + kb * sm.b_bytes, &tm_x, &sm.full[kb], kb * kBlockK, 0);
  // Counter sets alternate between forwards: the previous forward flipped
  // the parity word as it ended; this one clears the set the previous one
  // used, which the next one will use.
  const int par = *reinterpret_cast<const volatile int32_t*>(p.sync) & 1;
  sm.ss = p.sync + 1 + par * p.set_words;
  sm.ready = sm.ss + kSliceSyncWords + p.n_mt;
  if (bid == static_cast<int>(gridDim.x) - 1) {
    int32_t* other = p.sync + 1 + (par ^ 1) * p.set_words;
    for (int i = threadIdx.x; i < p.set_words; i += blockDim.x) other[i] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // router CTAs route first, then help with the down GEMM
  if (!is_unit && bid - p.n_units < p.n_rcta) route_tokens(p, sm, bid - p.n_units);
  if (works) {
    const uint32_t tmem = *sm.tmem_slot;
    if (warp == 0) {
      if (lane == 0) unit_produce(p, sm, u, &tm_gu, &tm_gu_sh, &tm_dn, &tm_dn_sh, &tm_x, kb_first);
    } else if (warp == 1) {
      if (lane == 0) unit_mma(p, sm, u, tmem);
    } else if (warp == 2) {
      unit_tokens(p, sm, u);
    } else {
      unit_epilogue(p, sm, u, tmem);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*sm.abort_flag) {
      // let loads already issued land before the shared memory goes away
      const long long t0 = clock64();
      while (clock64() - t0 < 4000000ll) {}
    }
    if (warp == 1) tmem_dealloc(tmem, kSliceTmemCols);
  }

  combine_tasks(p, sm);

  // the last CTA out (every CTA has read the parity word) flips it
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(sm.ss + 2, 1);
    if (old == static_cast<int>(gridDim.x) - 1) *reinterpret_cast<volatile int32_t*>(p.sync) = par ^ 1;
  }
}

}  // namespace

cudaError_t launch_slice(const CUtensorMap& tm_gu, const CUtensorMap& tm_gu_sh, const CUtensorMap& tm_dn,
                         const CUtensorMap& tm_dn_sh, const CUtensorMap& tm_x, const SliceParams& p, int grid,
                         size_t smem_bytes, bool overlap, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(moe_slice_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSliceThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  // With overlap, not a cooperative launch: the grid is one CTA per SM and
  // every CTA takes an SM's whole shared memory, so once the previous launch
  // on the stream has ended every CTA is resident (and every cross-CTA wait
  // is bounded in any case).  Programmatic serialization lets this launch's
  // CTAs start on the SMs the previous forward leaves, overlapping its tail.
  // Without, a cooperative launch (griddepcontrol.wait is then a no-op).
  cudaLaunchAttribute attr[1];
  if (overlap) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_slice_kernel, tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, tm_x, p);
}

}  // namespace moe
