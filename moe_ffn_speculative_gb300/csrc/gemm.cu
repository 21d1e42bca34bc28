// Grouped expert GEMMs of the MoE-FFN layer on the 5th-generation tensor
// cores (tcgen05.mma, fp32 accumulators in TMEM), and the weighted combine.
//
// Experts are SwiGLU MLPs with fused gate_up_proj [E,2I,H] and down_proj
// [E,H,I] (SpecForge PR #1073 "MoE drafts: DeepSeek-V4.1's own DSpark draft",
// commit note on the fused expert layout; rows [0,I) of gate_up are the gate);
// DeepSeek's clamped SwiGLU per SpecForge PR #941's follow-up comment; the
// routing weight multiplies each expert's output and the shared expert is
// added (sglang PR #48763 "[Feat] dflash: Serve MoE FFN drafts for DFlash and
// DSpark", commit note on DraftMoE forward).
//
// Decode-sized token counts make the layer weight-bandwidth bound, so the
// GEMMs are "swap-AB": the weight rows fill the 128-row M side of the MMA and
// an expert's few tokens are the N side.  Every (expert, 256-row tile,
// 64-wide k-block) weight block is streamed from HBM exactly once, by one CTA:
// the k-block iterations of all tiles of all touched experts are laid end to
// end and split evenly over a persistent grid of one CTA per SM (stream-K).
// A tile cut by a CTA boundary is finished by whichever of its CTAs arrives
// last, which sums the partial accumulators in CTA order (deterministic).
//
// Both GEMMs run in one persistent launch: each CTA streams its share of the
// gate_up iterations, then its share of the down iterations; a down tile's
// token rows are gathered once the gate_up tiles that write them signal.
//
// Warp roles (224 threads): warp 0 issues the weight TMA loads, warp 1
// allocates TMEM and issues the MMAs, warp 2 fills the 128-byte-swizzled B
// tile (gate_up: the expert's token rows of x by cp.async; down: its rows of
// h, consecutive, by TMA), warps 3..6 drain TMEM in the epilogue (SwiGLU for
// gate_up; routing weight and store for down).
//
// FP4 routed experts (SpecForge PR #1073, commit note on the official
// checkpoint's formats: each byte packs the e2m1 codes of two consecutive
// inputs, the even one in its low four bits; 32 inputs share an e8m0 scale): warp 0 streams the packed codes (8 KB
// per k-block) and the k-block's 512 bytes of block scales into a deeper ring
// of their own; four more warps (352 threads) expand them with the hardware
// e2m1 -> f16 conversion, multiply by the scale (exact in f16 for scales in
// [2^-23, 2^13]) and write the 128-byte-swizzled f16 A tile the MMA reads.
// Those groups multiply in f16 (x as its f16 copy, h as an f16 hi + lo pair);
// the bf16 shared expert goes through unchanged.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {


struct Seg {
  int expert, row_base, count, idim;
  int m, n, k0, len, kb, tile, n_cnt;
  int ready_idx;  // readiness counter of (expert group, token block) = its first gate_up tile + n
  long long tile_iter0;
};

// Walks one CTA's contiguous range [begin, end) of the concatenated k-block
// iterations, one (tile, k-range) segment at a time.
struct Sched {
  const GroupEntry* groups;
  int ngroups, phase, H, n_max, g, rows, idim_max;
  long long end, it;
  bool bad;  // a group entry outside the forward's bounds: the walk stops there

  __device__ long long iter_of(int gi) const { return phase == 0 ? groups[gi].gu_iter : groups[gi].dn_iter; }

  // [b, e): the CTA's iterations; g0: the group holding iteration b
  __device__ void init(const GemmParams& p, int ng, int ph, long long b, long long e, int g0) {
    groups = p.groups; ngroups = ng; phase = ph; H = p.H; n_max = p.n_max; it = b; end = e; g = g0;
    rows = p.TK + p.T;
    idim_max = p.I_ld;
    bad = false;
  }

  __device__ bool next(Seg& s) {
    if (it >= end || bad) return false;
    while (g + 1 < ngroups && iter_of(g + 1) <= it) ++g;
    const GroupEntry ge = groups[g];
    const long long start = phase == 0 ? ge.gu_iter : ge.dn_iter;
    if (g < 0 || g >= ngroups || ge.count < 1 || ge.row_base < 0 || ge.count > rows - ge.row_base ||
        ge.idim < 1 || ge.idim > idim_max || start < 0 || start > it) {
      bad = true;
      return false;
    }
    int mb, nb, kb;
    group_geometry(phase, ge.count, ge.idim, H, n_max, mb, nb, kb);
    const long long local = it - start;
    if (local >= static_cast<long long>(mb) * nb * kb) {
      bad = true;
      return false;
    }
    const int tile_in = static_cast<int>(local / kb);
    const int k0 = static_cast<int>(local % kb);
    const long long left = end - it;
    const int len = left < static_cast<long long>(kb - k0) ? static_cast<int>(left) : kb - k0;
    s.expert = ge.expert;
    s.row_base = ge.row_base;
    s.count = ge.count;
    s.idim = ge.idim;
    s.m = tile_in / nb;
    s.n = tile_in % nb;
    s.k0 = k0;
    s.len = len;
    s.kb = kb;
    s.tile = (phase == 0 ? ge.gu_tile : ge.dn_tile) + tile_in;
    s.tile_iter0 = start + static_cast<long long>(tile_in) * kb;
    s.n_cnt = min(n_max, ge.count - s.n * n_max);
    s.ready_idx = ge.gu_tile + s.n;
    it += len;
    return true;
  }
};

// The CTA whose iteration range [span[c], span[c+1]) holds iteration i
// (span: this GEMM's table, staged in shared memory).
__device__ __forceinline__ int cta_of(const long long* span, int grid, long long i) {
  int lo = 0, hi = grid - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (span[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// --------------------------------------------------------------------------
// epilogues of one 16-column chunk; a[i], b[i] = half-0 / half-1 accumulator
// of row r (TMEM lane) and token column j0 + i
// --------------------------------------------------------------------------
template <int PHASE, bool kFp4>
__device__ __forceinline__ void finish_chunk(const GemmParams& p, const Seg& sg, int r, int j0, const float* a,
                                             const float* b, const float* col_w, const int* col_tok) {
  if (PHASE == 0) {
    // SwiGLU: h = silu(gate) * up, with the clamp when a limit is set
    const int row = sg.m * kHalfRows + r;
    if (row >= sg.idim) return;
    // h is kept as a compensated pair hi + lo of bf16 (about 16 significant
    // bits): row r holds hi in [0, I_ld) and lo in [I_ld, 2*I_ld)
    uint16_t* hp = p.h + static_cast<size_t>(sg.row_base + sg.n * p.n_max) * (2 * p.I_ld) + row;
    const float lim = p.swiglu_limit;
    const bool half16 = kFp4 && sg.expert >= 0;  // the pair in f16 for the FP4 down GEMM
    bool over = false;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int j = j0 + i;
      if (j < sg.n_cnt) {
        float g = a[i], u = b[i];
        if (lim > 0.f) {
          g = fminf(g, lim);
          u = fminf(fmaxf(u, -lim), lim);
        }
        const float hv = g / (1.f + expf(-g)) * u;
        uint16_t whi, wlo;
        if (half16) {
          const __half hi = __float2half_rn(hv);
          whi = __half_as_ushort(hi);
          wlo = __half_as_ushort(__float2half_rn(hv - __half2float(hi)));
          over |= !(fabsf(hv) < 65520.f);
        } else {
          const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
          whi = __bfloat16_as_ushort(hi);
          wlo = f2bf(hv - __bfloat162float(hi));
        }
        hp[static_cast<size_t>(j) * (2 * p.I_ld)] = whi;
        hp[static_cast<size_t>(j) * (2 * p.I_ld) + p.I_ld] = wlo;
      }
    }
    if (over) record_range(p.status, kInfoHRange);
  } else {
    // routing weight (or shared-expert gate) times the expert output
    const int row0 = sg.m * 2 * kHalfRows + r;
    const int row1 = row0 + kHalfRows;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int j = j0 + i;
      if (j < sg.n_cnt) {
        const int sr = sg.row_base + sg.n * p.n_max + j;
        const float wt = col_w[j];
        const int tok = col_tok[j];
        if (p.direct_y) {
          uint16_t* yr = p.y + static_cast<size_t>(tok) * p.H;
          if (row0 < p.H) yr[row0] = f2bf(wt * a[i]);
          if (row1 < p.H) yr[row1] = f2bf(wt * b[i]);
        } else {
          float* orow = p.out_ws + static_cast<size_t>(sr) * p.H;
          if (row0 < p.H) __stcg(orow + row0, wt * a[i]);
          if (row1 < p.H) __stcg(orow + row1, wt * b[i]);
        }
      }
    }
  }
}

__device__ __forceinline__ void u32_to_f32(const uint32_t (&u)[16], float (&f)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(u[i]);
}


// The CTA's shared memory: S stages of [A gate|A up or two 128-row output
// halves (16 KB each) | B tile (n_max x 64 bf16) | second B tile (h_lo)],
// then barriers and small control words.
struct Smem {
  uint8_t* base;
  uint32_t stage_bytes, b_bytes;
  int S;
  uint64_t *full, *empty, *accf, *acce, *drain;
  volatile int* abort_flag;
  int* bcast;
  int* s_ok;
  long long* rowoff;
  long long* span;  // [2][grid+1] CTA spans of both GEMMs
  float* col_w;     // [n_max] down epilogue: routing weight of each token column
  int* col_tok;     // [n_max] down epilogue: token of each column
  // FP4: SP stages of packed codes (8 KB) and of block scales (512 B)
  uint8_t* pbase;
  uint8_t* sbase;
  uint64_t *pfull, *pempty;
  int SP;
};

// ---------------------------------------------------------------- TMA producer (weights)
// One CTA's weight k-blocks in the order it consumes them: its gate_up span,
// then its down span.
struct WeightCursor {
  Sched sc0, sc1;
  Seg sg;
  int ph, kk;
  bool valid;

  __device__ void init(const GemmParams& p, int ngroups, const long long (&b)[2], const long long (&e)[2],
                       const int (&g)[2]) {
    sc0.init(p, ngroups, 0, b[0], e[0], g[0]);
    sc1.init(p, ngroups, 1, b[1], e[1], g[1]);
    ph = 0;
    kk = 0;
    valid = false;
    next_segment();
  }
  __device__ void next_segment() {
    while (ph < 2) {
      if (ph == 0 ? sc0.next(sg) : sc1.next(sg)) {
        kk = 0;
        valid = true;
        return;
      }
      ++ph;
    }
    valid = false;
  }
  __device__ void step() {
    if (++kk >= sg.len) next_segment();
  }
  // tensor map and box coordinates of half h of the current k-block (FP4
  // codes: the routed maps are byte tensors, 32 bytes per k-block)
  template <bool kFp4>
  __device__ const CUtensorMap* box(const CUtensorMap* tm_gu, const CUtensorMap* tm_gu_sh, const CUtensorMap* tm_dn,
                                    const CUtensorMap* tm_dn_sh, int h, int& c0, int& c1, int& c2) const {
    const int plane = sg.expert >= 0 ? sg.expert : 0;
    c0 = (sg.k0 + kk) * ((kFp4 && sg.expert >= 0) ? kBlockK / 2 : kBlockK);
    if (ph == 0) {
      c1 = sg.m * kHalfRows;
      c2 = 2 * plane + h;
    } else {
      c1 = sg.m * 2 * kHalfRows + h * kHalfRows;
      c2 = plane;
    }
    if (ph == 0) return sg.expert >= 0 ? tm_gu : tm_gu_sh;
    return sg.expert >= 0 ? tm_dn : tm_dn_sh;
  }
};

// Byte offset of the prepared block scales of (expert, tile m, k-block kb):
// 512 bytes each, gate_up blocks of all experts first, then down blocks.
__device__ __forceinline__ size_t fp4_scale_offset(const GemmParams& p, int phase, int e, int m, int kb) {
  const int mb0 = ceil_div(p.I, kHalfRows), kb0 = p.H / kBlockK;
  if (phase == 0) return ((static_cast<size_t>(e) * mb0 + m) * kb0 + kb) * 512;
  const int mb1 = ceil_div(p.H, 2 * kHalfRows), kb1 = p.I / kBlockK;
  return static_cast<size_t>(p.E) * mb0 * kb0 * 512 + ((static_cast<size_t>(e) * mb1 + m) * kb1 + kb) * 512;
}

template <bool kFp4>
__device__ bool produce(const Smem& sm, const GemmParams& p, int ngroups, const long long (&b)[2],
                        const long long (&e)[2], const int (&g)[2], const CUtensorMap* tm_gu,
                        const CUtensorMap* tm_gu_sh, const CUtensorMap* tm_dn, const CUtensorMap* tm_dn_sh,
                        Ring& ring, int32_t* status) {
  // Weights are streamed once: evict them first, so that L2 keeps what the
  // layer reuses (x, h, partials, the next kernels' code and metadata).
  const uint64_t pol = l2_evict_first_policy();
  if (!wait_start_gate(status)) {
    record_failure(status, sm.abort_flag, kInfoHold);
    return false;
  }
  WeightCursor ld;
  ld.init(p, ngroups, b, e, g);
  Ring pring;  // FP4 code stages
  // FP4: routed k-blocks advance this warp's A-ring cursor without waiting
  // on the A ring (only on the deeper code ring), so the cursor can run more
  // than one phase of an `empty` barrier ahead of the MMAs, where a parity
  // wait no longer tells the phases apart.  Before the next bf16 k-block the
  // converter must have taken the last routed one (it waited on that A stage
  // in order), which brings the cursor back within one phase.
  int last_ps = -1;
  uint32_t last_pphase = 0;
  while (ld.valid) {
    if (kFp4 && ld.sg.expert < 0 && last_ps >= 0) {
      if (!mbar_wait(&sm.pempty[last_ps], last_pphase, sm.abort_flag)) {
        record_failure(status, sm.abort_flag, kInfoEmpty);
        return false;
      }
      last_ps = -1;
    }
    if (kFp4 && ld.sg.expert >= 0) {
      // packed codes and block scales of a routed k-block; the converter
      // warps turn them into the A stage
      if (!mbar_wait(&sm.pempty[pring.stage], pring.phase ^ 1u, sm.abort_flag)) {
        record_failure(status, sm.abort_flag, kInfoEmpty);
        return false;
      }
      uint64_t* bar = &sm.pfull[pring.stage];
      mbar_arrive_expect_tx(bar, kPackedBytes + 512);
      int c0, c1, c2;
      for (int h = 0; h < 2; ++h) {
        const CUtensorMap* tm = ld.box<kFp4>(tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, h, c0, c1, c2);
        tma_load_3d_hint(sm.pbase + pring.stage * kPackedBytes + h * (kPackedBytes / 2), tm, bar, c0, c1, c2, pol);
      }
      const uint8_t* sc = ld.ph == 0 ? p.gu_scale : p.dn_scale;
      bulk_load_hint(sm.sbase + pring.stage * 512,
                     sc + fp4_scale_offset(p, ld.ph, ld.sg.expert, ld.sg.m, ld.sg.k0 + ld.kk), 512, bar, pol);
      last_ps = pring.stage;
      last_pphase = pring.phase;
      pring.next(sm.SP);
      ld.step();
      ring.next(sm.S);  // the A ring advances for every k-block
      continue;
    }
    if (!mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag)) {
      record_failure(status, sm.abort_flag, kInfoEmpty);
      return false;
    }
    uint8_t* a0 = sm.base + ring.stage * sm.stage_bytes;
    uint64_t* bar = &sm.full[ring.stage];
    mbar_arrive_expect_tx(bar, 2 * kTileBytesA);
    int c0, c1, c2;
    for (int h = 0; h < 2; ++h) {
      const CUtensorMap* tm = ld.box<kFp4>(tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, h, c0, c1, c2);
      tma_load_3d_hint(a0 + h * kTileBytesA, tm, bar, c0, c1, c2, pol);
    }
    ld.step();
    ring.next(sm.S);
  }
  if (ld.sc0.bad || ld.sc1.bad) {
    record_failure(status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  // every weight load of this CTA is issued: its share of the next layer's
  // routing-independent bytes goes to L2 while the layer's tail runs
  prefetch_share_l2(p.pf);
  return true;
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <int PHASE, bool kFp4>
__device__ bool issue_mma(const Smem& sm, const GemmParams& p, int ngroups, long long begin, long long end, int g0,
                          uint32_t tmem_base, Ring& ring, int& seg_i, int32_t* status) {
  Sched sc;
  sc.init(p, ngroups, PHASE, begin, end, g0);
  Seg sg;
  while (sc.next(sg)) {
    const int buf = seg_i % p.nbuf;
    const uint32_t use = static_cast<uint32_t>(seg_i / p.nbuf);
    if (!mbar_wait(&sm.acce[buf], (use & 1u) ^ 1u, sm.abort_flag)) {
      record_failure(status, sm.abort_flag, kInfoAccEmpty);
      return false;
    }
    tc_fence_after();
    const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * 2 * p.n_max);
    const uint32_t d1 = d0 + static_cast<uint32_t>(p.n_max);
    const int nmma = max(16, (sg.n_cnt + 15) & ~15);
    // FP4 routed groups: f16 weights (expanded) and f16 token rows
    const uint32_t idesc = (kFp4 && sg.expert >= 0) ? idesc_f16(kHalfRows, nmma) : idesc_bf16(kHalfRows, nmma);
    for (int kk = 0; kk < sg.len; ++kk) {
      if (!mbar_wait(&sm.full[ring.stage], ring.phase, sm.abort_flag)) {
        record_failure(status, sm.abort_flag, kInfoFull);
        return false;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(sm.base + ring.stage * sm.stage_bytes);
      const uint32_t a1 = a0 + kTileBytesA;
      const uint32_t bb = a0 + 2 * kTileBytesA;
#pragma unroll
      for (int ks = 0; ks < kBlockK / 16; ++ks) {
        const uint32_t acc = (kk > 0 || ks > 0) ? 1u : 0u;
        const uint64_t bd = sw128_desc(bb + ks * 32);
        const uint64_t ad0 = sw128_desc(a0 + ks * 32), ad1 = sw128_desc(a1 + ks * 32);
        mma_bf16(d0, ad0, bd, idesc, acc);
        mma_bf16(d1, ad1, bd, idesc, acc);
        if (PHASE == 1) {  // + W * h_lo
          const uint64_t bl = sw128_desc(bb + sm.b_bytes + ks * 32);
          mma_bf16(d0, ad0, bl, idesc, 1u);
          mma_bf16(d1, ad1, bl, idesc, 1u);
        }
      }
      mma_commit(&sm.empty[ring.stage]);
      ring.next(sm.S);
    }
    mma_commit(&sm.accf[buf]);
    ++seg_i;
  }
  if (sc.bad) {
    record_failure(status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- token-row gather (B), one warp
// gate_up: rows of x for the expert's tokens; down: the expert's h rows (hi and
// lo), after the gate_up tiles that write them have signalled.
template <int PHASE, bool kFp4>
__device__ bool gather(const Smem& sm, const GemmParams& p, int ngroups, long long begin, long long end, int g0,
                       Ring& ring, int& pending, int& arr_stage, int lag, const CUtensorMap* tm_h,
                       int32_t* status) {
  const int lane = threadIdx.x & 31;
  // The down GEMM's token rows (h hi and lo) of one (expert, token block)
  // are consecutive rows of h: loaded by TMA in boxes of 16 rows x 64
  // columns, lane 0 counting their bytes on the stage's barrier.
  const bool h_tma = PHASE == 1 && p.h_tma != 0;
  if (h_tma) {
    // copies of the gate_up phase still in flight land and count first
    cp_async_wait<0>();
    fence_proxy_async();
    while (pending > 0) {
      mbar_arrive(&sm.full[arr_stage]);
      if (++arr_stage == sm.S) arr_stage = 0;
      --pending;
    }
  }
  Sched sc;
  sc.init(p, ngroups, PHASE, begin, end, g0);
  constexpr int kBTiles = PHASE == 0 ? 1 : 2;
  Seg sg;
  while (sc.next(sg)) {
    const uint16_t* bsrc = PHASE == 0 ? ((kFp4 && sg.expert >= 0) ? p.xh : p.x) : p.h;
    const int nrows = max(16, (sg.n_cnt + 15) & ~15);
    const int kdim = PHASE == 0 ? p.H : sg.idim;
    __syncwarp();
    for (int j = lane; j < nrows; j += 32) {
      long long off = -1;
      if (j < sg.n_cnt) {
        const int r = sg.n * p.n_max + j;
        if (PHASE == 0) {
          const int tok = sg.expert >= 0 ? __ldg(p.sorted_pair + sg.row_base + r) / p.K : r;
          off = static_cast<long long>(tok) * p.H;
        } else {
          off = static_cast<long long>(sg.row_base + r) * (2 * p.I_ld);
        }
      }
      sm.rowoff[j] = off;
    }
    if (PHASE == 1) {
      // h of this (expert, token block) is complete once every gate_up tile
      // of it has signalled
      const int target = ceil_div(sg.idim, kHalfRows);
      const int32_t* rp = p.ready + sg.ready_idx;
      int ready = lane == 0 ? (ld_acquire_gpu(rp) >= target) : 0;
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) {
        // Release every stage this warp still holds first: the missing tiles
        // may be this CTA's own last gate_up tiles, whose MMAs wait on them.
        cp_async_wait<0>();
        fence_proxy_async();
        while (pending > 0) {
          mbar_arrive(&sm.full[arr_stage]);
          if (++arr_stage == sm.S) arr_stage = 0;
          --pending;
        }
        int okr = 1;
        if (lane == 0) {
          const long long t0 = clock64();
          while (ld_acquire_gpu(rp) < target) {
            if (*sm.abort_flag || clock64() - t0 > kWaitLimitCycles) { okr = 0; break; }
            __nanosleep(64);
          }
        }
        okr = __shfl_sync(0xffffffffu, okr, 0);
        if (!okr) {
          if (lane == 0) record_failure(status, sm.abort_flag, kInfoReady);
          return false;
        }
      }
      // rows written by other CTAs' generic stores, read by TMA below
      if (h_tma) asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
    for (int kk = 0; kk < sg.len; ++kk) {
      const int kx = (sg.k0 + kk) * kBlockK;
      const bool got = mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) record_failure(status, sm.abort_flag, kInfoGatherEmpty);
        return false;
      }
      const uint32_t bbase = smem_u32(sm.base + ring.stage * sm.stage_bytes) + 2 * kTileBytesA;
      if (h_tma) {
        uint64_t* bar = &sm.full[ring.stage];
        if (lane == 0) {
          const int nb = nrows / 16;
          const int row0 = sg.row_base + sg.n * p.n_max;
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(2 * nb * 2048));
          uint8_t* b0 = sm.base + ring.stage * sm.stage_bytes + 2 * kTileBytesA;
          for (int t = 0; t < 2; ++t)
            for (int i = 0; i < nb; ++i)
              tma_load_2d(b0 + t * sm.b_bytes + i * 2048, tm_h, bar, t * p.I_ld + kx, row0 + 16 * i);
        } else {
          mbar_arrive(bar);
        }
        ring.next(sm.S);
        continue;
      }
      for (int q = lane; q < nrows * 8 * kBTiles; q += 32) {
        const int t = (kBTiles == 2 && q >= nrows * 8) ? 1 : 0;  // 0: x or h_hi, 1: h_lo
        const int qq = q - t * nrows * 8;
        const int j = qq >> 3, c = qq & 7;
        const long long off = sm.rowoff[j];
        const int col = kx + c * 8;
        const bool valid = off >= 0 && col < kdim;
        const uint16_t* src = valid ? bsrc + off + t * p.I_ld + col : bsrc;
        cp_async_16(bbase + t * sm.b_bytes + j * 128 + ((c ^ (j & 7)) << 4), src, valid ? 16u : 0u);
      }
      cp_async_commit();
      ++pending;
      if (pending > lag) {
        if (lag >= 2) cp_async_wait<2>(); else cp_async_wait<1>();
        fence_proxy_async();
        mbar_arrive(&sm.full[arr_stage]);
        if (++arr_stage == sm.S) arr_stage = 0;
        --pending;
      }
      ring.next(sm.S);
    }
  }
  if (sc.bad) {
    if (lane == 0) record_failure(status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- FP4 expansion (4 warps)
// All 128 converter threads vote; every one of them must call it.
__device__ __forceinline__ bool conv_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

// 2^(s - 127) as an f16 pair, for s in [kFp4ScaleMin, kFp4ScaleMax] (normal
// f16 down to 2^-14, subnormal below).
__device__ __forceinline__ uint32_t e8m0_to_h2(uint32_t s) {
  const int e = static_cast<int>(s) - 127;
  const uint32_t b = e >= -14 ? static_cast<uint32_t>(e + 15) << 10 : 1u << (e + 24);
  return b | (b << 16);
}

// Eight e2m1 codes (byte j: inputs 2j in the low nibble, 2j+1 in the high
// one) -> eight f16 times the scale pair sc, in input order.
__device__ __forceinline__ uint4 expand8(uint32_t w, uint32_t sc) {
  uint4 o;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
      "mul.rn.f16x2 %0, %0, %5;\n\t"
      "mul.rn.f16x2 %1, %1, %5;\n\t"
      "mul.rn.f16x2 %2, %2, %5;\n\t"
      "mul.rn.f16x2 %3, %3, %5;\n\t"
      "}"
      : "=&r"(o.x), "=&r"(o.y), "=&r"(o.z), "=&r"(o.w)
      : "r"(w), "r"(sc));
  return o;
}

// Walks the CTA's k-blocks in the producer's order; for every routed one,
// waits for its codes and a free A stage, and writes row r of both halves of
// the A stage: the 64 inputs of the k-block as f16, 128-byte swizzled.
__device__ bool convert(const Smem& sm, const GemmParams& p, int ngroups, const long long (&b)[2],
                        const long long (&e)[2], const int (&g)[2], int32_t* status) {
  const int r = threadIdx.x - 7 * 32;
  WeightCursor ld;
  ld.init(p, ngroups, b, e, g);
  Ring ring, pring;
  bool range_ok = true;
  while (ld.valid) {
    if (ld.sg.expert < 0) {  // a bf16 k-block the producer loads itself
      ld.step();
      ring.next(sm.S);
      continue;
    }
    // Codes first: the producer issues them only after its own wait on the
    // A stage before this one (or, after routed k-blocks, after this warp's
    // last release), so the MMAs are then at most one phase of this stage's
    // `empty` barrier behind, which the parity wait needs; bf16 k-blocks
    // skipped above would otherwise leave this warp several phases ahead.
    bool ok = mbar_wait(&sm.pfull[pring.stage], pring.phase, sm.abort_flag) &&
              mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag);
    if (ok) {
      const uint8_t* cs = sm.pbase + pring.stage * kPackedBytes + r * 32;
      const uint16_t* ss = reinterpret_cast<const uint16_t*>(sm.sbase + pring.stage * 512);
      uint8_t* a = sm.base + ring.stage * sm.stage_bytes + r * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t s2 = ss[h * kHalfRows + r];  // scales of inputs [0,32) and [32,64)
        const uint32_t s0 = s2 & 0xffu, s1 = s2 >> 8;
        range_ok &= s0 >= kFp4ScaleMin && s0 <= kFp4ScaleMax && s1 >= kFp4ScaleMin && s1 <= kFp4ScaleMax;
        const uint32_t sc0 = e8m0_to_h2(min(max(s0, static_cast<uint32_t>(kFp4ScaleMin)), static_cast<uint32_t>(kFp4ScaleMax)));
        const uint32_t sc1 = e8m0_to_h2(min(max(s1, static_cast<uint32_t>(kFp4ScaleMin)), static_cast<uint32_t>(kFp4ScaleMax)));
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int q = qq ^ ((r >> 2) & 1);  // spreads the rows' 16-byte reads over the banks
          const uint4 w = *reinterpret_cast<const uint4*>(cs + h * (kPackedBytes / 2) + q * 16);
          const uint32_t sc = q ? sc1 : sc0;
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = q * 4 + j;  // 16-byte chunk of the 128-byte row
            *reinterpret_cast<uint4*>(a + h * kTileBytesA + ((c ^ (r & 7)) << 4)) = expand8(wv[j], sc);
          }
        }
      }
      fence_proxy_async();
    }
    if (!conv_all(ok)) {
      if (r == 0) record_failure(status, sm.abort_flag, kInfoFull);
      return false;
    }
    if (r == 0) {
      mbar_arrive(&sm.pempty[pring.stage]);
      mbar_arrive(&sm.full[ring.stage]);
    }
    pring.next(sm.SP);
    ld.step();
    ring.next(sm.S);
  }
  if (!range_ok) record_range(status, kInfoScaleRange);
  if (ld.sc0.bad || ld.sc1.bad) {
    if (r == 0) record_failure(status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- epilogue (4 warps)
template <int PHASE, bool kFp4>
__device__ bool epilogue(const Smem& sm, const GemmParams& p, int ngroups, long long begin, long long end, int g0,
                         uint32_t tmem_base, int& seg_i, int32_t* tile_counters, int32_t* status) {
  Sched sc;
  sc.init(p, ngroups, PHASE, begin, end, g0);
  const long long* span = sm.span + PHASE * (gridDim.x + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;  // accumulator row = TMEM lane
  const bool leader = (warp == 3 && lane == 0);
  const int grid = gridDim.x;
  Seg sg;
  while (sc.next(sg)) {
    const int buf = seg_i % p.nbuf;
    const uint32_t use = static_cast<uint32_t>(seg_i / p.nbuf);
    if (PHASE == 1) {
      // each column's routing weight (or shared-expert gate) and token, loaded
      // in parallel while the MMAs of this segment still run
      const int epi_t = (warp - 3) * 32 + lane;
      for (int j = epi_t; j < sg.n_cnt; j += 128) {
        const int sr = sg.row_base + sg.n * p.n_max + j;
        if (sg.expert >= 0) {
          const int pr = __ldg(p.sorted_pair + sr);
          sm.col_w[j] = __ldg(p.topk_w + pr);
          sm.col_tok[j] = pr / p.K;
        } else {
          const int tok = sr - p.TK;
          sm.col_w[j] = p.sh_w ? __ldg(p.sh_w + tok) : 1.f;
          sm.col_tok[j] = tok;
        }
      }
    }
    // one thread waits, the four warps leave or go on together
    if (leader) {
      const bool got = mbar_wait(&sm.accf[buf], use & 1u, sm.abort_flag);
      if (!got) record_failure(status, sm.abort_flag, kInfoAccFull);
      *sm.s_ok = got ? 1 : 0;
    }
    epi_sync();
    if (!*reinterpret_cast<volatile int*>(sm.s_ok)) return false;
    tc_fence_after();
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                          static_cast<uint32_t>(buf * 2 * p.n_max);
    const bool whole = (sg.k0 == 0 && sg.len == sg.kb);
    bool done = false;  // this CTA finished the tile's output
    uint32_t ua[16], ub[16];
    float fa[16], fb[16];
    if (whole) {
      for (int j0 = 0; j0 < sg.n_cnt; j0 += 16) {
        tmem_ld16(tacc + j0, ua);
        tmem_ld16(tacc + p.n_max + j0, ub);
        tmem_ld_wait();
        u32_to_f32(ua, fa);
        u32_to_f32(ub, fb);
        finish_chunk<PHASE, kFp4>(p, sg, r, j0, fa, fb, sm.col_w, sm.col_tok);
      }
      tc_fence_before();
      mbar_arrive(&sm.acce[buf]);
      done = true;
    } else if (sg.k0 > 0) {
      // A later part of a split tile: hand the partial sums to the CTA that
      // holds the tile's first k-block.  A CTA's span can start inside at
      // most one tile, so it writes at most one partial per GEMM.
      float* mine = p.partials + static_cast<size_t>(blockIdx.x * 4 + PHASE * 2) * 2 * p.n_max * 128;
      for (int j0 = 0; j0 < sg.n_cnt; j0 += 16) {
        tmem_ld16(tacc + j0, ua);
        tmem_ld16(tacc + p.n_max + j0, ub);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (j0 + i < sg.n_cnt) {
            __stcg(mine + static_cast<size_t>(j0 + i) * 128 + r, __uint_as_float(ua[i]));
            __stcg(mine + static_cast<size_t>(p.n_max + j0 + i) * 128 + r, __uint_as_float(ub[i]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acce[buf]);
      __threadfence();
      epi_sync();
      if (leader) atomicAdd(tile_counters + sg.tile, sg.len);
    } else {
      // The first part of a split tile: this CTA finishes it.  The later
      // parts were processed at the start of their CTAs' spans, so their
      // partials are normally there already; wait (bounded) until all are
      // counted, then add them to the accumulator in CTA order.
      if (leader) {
        const int32_t* cnt = tile_counters + sg.tile;
        const int target = sg.kb - sg.len;
        bool got = ld_acquire_gpu(cnt) >= target;
        if (!got) {
          const long long t0 = clock64();
          while (!(got = ld_acquire_gpu(cnt) >= target)) {
            if (*sm.abort_flag || clock64() - t0 > kWaitLimitCycles) break;
            __nanosleep(32);
          }
        }
        if (got) atomicExch(tile_counters + sg.tile, 0);
        else record_failure(status, sm.abort_flag, kInfoFixup);
        *sm.s_ok = got ? 1 : 0;
      }
      epi_sync();
      if (!*reinterpret_cast<volatile int*>(sm.s_ok)) return false;
      __threadfence();
      const int c1 = cta_of(span, grid, sg.tile_iter0 + sg.kb - 1);
      for (int j0 = 0; j0 < sg.n_cnt; j0 += 16) {
        tmem_ld16(tacc + j0, ua);
        tmem_ld16(tacc + p.n_max + j0, ub);
        tmem_ld_wait();
        u32_to_f32(ua, fa);
        u32_to_f32(ub, fb);
        for (int c = blockIdx.x + 1; c <= c1; ++c) {
          if (span[c] == span[c + 1]) continue;  // CTA with an empty range
          const float* pp = p.partials + static_cast<size_t>(c * 4 + PHASE * 2) * 2 * p.n_max * 128;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (j0 + i < sg.n_cnt) {
              fa[i] += __ldcg(pp + static_cast<size_t>(j0 + i) * 128 + r);
              fb[i] += __ldcg(pp + static_cast<size_t>(p.n_max + j0 + i) * 128 + r);
            }
          }
        }
        finish_chunk<PHASE, kFp4>(p, sg, r, j0, fa, fb, sm.col_w, sm.col_tok);
      }
      tc_fence_before();
      mbar_arrive(&sm.acce[buf]);
      done = true;
    }
    if (PHASE == 0 && done) {
      // this gate_up tile's h rows are written: count it towards its
      // (expert, token block); the down GEMM may read them by TMA
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __threadfence();
      epi_sync();
      if (leader) atomicAdd(p.ready + sg.ready_idx, 1);
    }
    epi_sync();
    ++seg_i;
  }
  if (sc.bad) {
    if (leader) record_failure(status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

// One persistent CTA per SM runs the gate_up GEMM over its share of the
// gate_up k-block iterations, then the down GEMM over its share of the down
// iterations.  The launch is cooperative (every CTA resident), so the down
// phase's bounded waits on the gate_up tiles of other CTAs always resolve.
template <bool kFp4>
__global__ void __launch_bounds__(kFp4 ? kGemmThreadsFp4 : kGemmThreads, 1)
    moe_experts_kernel(const __grid_constant__ CUtensorMap tm_gu, const __grid_constant__ CUtensorMap tm_gu_sh,
                       const __grid_constant__ CUtensorMap tm_dn, const __grid_constant__ CUtensorMap tm_dn_sh,
                       const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  // [control words | stages]: the control block comes first so that the
  // barriers exist before the stage size is known
  uint8_t* ctrl = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  sm.base = ctrl + kCtrlBytes;
  sm.full = reinterpret_cast<uint64_t*>(ctrl);
  sm.empty = sm.full + kMaxStages;
  sm.accf = sm.empty + kMaxStages;
  sm.acce = sm.accf + 2;
  sm.drain = sm.acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.drain + 1);
  sm.abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  sm.bcast = reinterpret_cast<int*>(tmem_slot + 2);
  sm.s_ok = reinterpret_cast<int*>(tmem_slot + 3);
  sm.rowoff = reinterpret_cast<long long*>(ctrl + kCtrlRowOff);
  sm.span = reinterpret_cast<long long*>(ctrl + kCtrlSpans);
  sm.col_w = reinterpret_cast<float*>(ctrl + kCtrlCols);
  sm.col_tok = reinterpret_cast<int*>(ctrl + kCtrlCols + 4 * 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&sm.full[s], 1 + 32);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.accf[b], 1);
      mbar_init(&sm.acce[b], 128);
    }
    mbar_init(sm.drain, 1);
    if (kFp4) {
      // the FP4 rings' barriers open the stage region
      uint64_t* pb = reinterpret_cast<uint64_t*>(ctrl + kCtrlBytes);
      for (int s = 0; s < kMaxPStages; ++s) {
        mbar_init(pb + s, 1);
        mbar_init(pb + kMaxPStages + s, 1);
      }
    }
    *sm.abort_flag = 0;
    *sm.bcast = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_gu);
    tma_prefetch_desc(&tm_gu_sh);
    tma_prefetch_desc(&tm_dn);
    tma_prefetch_desc(&tm_dn_sh);
    if (p.h_tma) tma_prefetch_desc(&tm_h);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < 2 * (static_cast<int>(gridDim.x) + 1); i += blockDim.x) sm.span[i] = p.spans[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // The router's work list, checked against the host's bounds (every thread
  // reads the same words, so the decision is uniform): a list outside them
  // -- a workspace that was not zero-filled, or was overwritten -- is
  // refused instead of streamed.
  const GemmHeader hd = *p.header;
  const int G1 = gridDim.x + 1;
  const long long bs[2] = {sm.span[blockIdx.x], sm.span[G1 + blockIdx.x]};
  const long long es[2] = {sm.span[blockIdx.x + 1], sm.span[G1 + blockIdx.x + 1]};
  const int gs[2] = {p.span_groups[blockIdx.x], p.span_groups[G1 + blockIdx.x]};
  const bool list_ok = hd.ngroups >= 0 && hd.ngroups <= p.g_max && hd.gu_tiles >= 0 &&
                       hd.gu_tiles <= p.max_gu_tiles && hd.dn_tiles >= 0 && hd.dn_tiles <= p.max_dn_tiles &&
                       hd.n_eff >= 16 && hd.n_eff <= p.n_max && (hd.n_eff & 15) == 0 && hd.gu_iters >= 0 &&
                       hd.gu_iters <= p.max_gu_iters && hd.dn_iters >= 0 && hd.dn_iters <= p.max_dn_iters &&
                       bs[0] >= 0 && bs[0] <= es[0] && es[0] <= hd.gu_iters && bs[1] >= 0 && bs[1] <= es[1] &&
                       es[1] <= hd.dn_iters && gs[0] >= 0 && gs[0] <= hd.ngroups && gs[1] >= 0 &&
                       gs[1] <= hd.ngroups;
  if (!list_ok && threadIdx.x == 0) record_failure(p.status, sm.abort_flag, kInfoWorkList);
  const int ng = hd.ngroups;
  // Stages are sized for the widest token tile this forward actually has,
  // so narrow tiles (decode) get more stages in the same shared memory.
  sm.b_bytes = (list_ok ? hd.n_eff : 16) * 128;
  sm.stage_bytes = 2 * kTileBytesA + 2 * sm.b_bytes;
  sm.S = min(kMaxStages, p.stage_space / static_cast<int>(sm.stage_bytes));
  if (kFp4) {
    // [barriers 1 KB | SP x 8 KB codes | SP x 512 B scales (1 KB aligned) |
    //  S A stages]: three A stages where the codes keep four stages or more
    const int st = static_cast<int>(sm.stage_bytes), ps = kPackedBytes + 512;
    const int space = p.stage_space - 2048;
    sm.S = (3 * st + 4 * ps <= space) ? 3 : 2;
    sm.SP = min(kMaxPStages, (space - sm.S * st) / ps);
    sm.pfull = reinterpret_cast<uint64_t*>(ctrl + kCtrlBytes);
    sm.pempty = sm.pfull + kMaxPStages;
    sm.pbase = ctrl + kCtrlBytes + 1024;
    sm.sbase = sm.pbase + sm.SP * kPackedBytes;
    sm.base = sm.sbase + ((sm.SP * 512 + 1023) & ~1023);
  }
  if (!list_ok) {
    // nothing issued: every thread goes straight to the teardown
  } else if (warp == 0) {
    if (lane == 0) {
      Ring ring;
      const bool ok = produce<kFp4>(sm, p, ng, bs, es, gs, &tm_gu, &tm_gu_sh, &tm_dn, &tm_dn_sh, ring, p.status);
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000ll) {}
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      Ring ring;
      int seg_i = 0;
      if (issue_mma<0, kFp4>(sm, p, ng, bs[0], es[0], gs[0], tmem_base, ring, seg_i, p.status))
        issue_mma<1, kFp4>(sm, p, ng, bs[1], es[1], gs[1], tmem_base, ring, seg_i, p.status);
      // every MMA issued above has completed once `drain` flips
      mma_commit(sm.drain);
      if (!mbar_wait(sm.drain, 0, nullptr)) record_failure(p.status, sm.abort_flag, kInfoDrain);
    }
  } else if (warp == 2) {
    Ring ring;
    int pending = 0, arr_stage = 0;
    // copies kept in flight before arriving; below the stage count, so the
    // stage this warp waits to refill never depends on an arrival it holds.
    // FP4 k-blocks stream in a quarter of a bf16 one's time: one group in
    // flight, so that a stage's arrival waits for the MMAs two k-blocks
    // back rather than the previous one's and two k-blocks' MMAs overlap.
    const int lag = kFp4 ? 1 : (kGatherLag < sm.S - 1 ? kGatherLag : sm.S - 1);
    if (gather<0, kFp4>(sm, p, ng, bs[0], es[0], gs[0], ring, pending, arr_stage, lag, &tm_h, p.status))
      gather<1, kFp4>(sm, p, ng, bs[1], es[1], gs[1], ring, pending, arr_stage, lag, &tm_h, p.status);
    cp_async_wait<0>();
    fence_proxy_async();
    while (pending > 0) {
      mbar_arrive(&sm.full[arr_stage]);
      if (++arr_stage == sm.S) arr_stage = 0;
      --pending;
    }
  } else if (warp < 7) {
    int seg_i = 0;
    if (epilogue<0, kFp4>(sm, p, ng, bs[0], es[0], gs[0], tmem_base, seg_i, p.tile_counters_gu, p.status))
      epilogue<1, kFp4>(sm, p, ng, bs[1], es[1], gs[1], tmem_base, seg_i, p.tile_counters_dn, p.status);
  } else if (kFp4) {
    convert(sm, p, ng, bs, es, gs, p.status);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// y[t] = sum_k out[pair_pos[t*K+k]] (+ out[T*K + t] for the shared expert),
// summed in slot order, rounded to bf16.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ out_ws,
                                                      const int32_t* __restrict__ pair_pos, int T, int K, int H,
                                                      int has_shared, uint16_t* __restrict__ y) {
  const int t = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (c >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < K; ++k) {
    const int pos = __ldg(pair_pos + t * K + k);
    const float4 v = __ldcg(reinterpret_cast<const float4*>(out_ws + static_cast<size_t>(pos) * H + c));
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  if (has_shared) {
    const float4 v =
        __ldcg(reinterpret_cast<const float4*>(out_ws + static_cast<size_t>(T * K + t) * H + c));
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  uint2 o;
  o.x = static_cast<uint32_t>(f2bf(acc.x)) | (static_cast<uint32_t>(f2bf(acc.y)) << 16);
  o.y = static_cast<uint32_t>(f2bf(acc.z)) | (static_cast<uint32_t>(f2bf(acc.w)) << 16);
  *reinterpret_cast<uint2*>(y + static_cast<size_t>(t) * H + c) = o;
}

// Re-lays e8m0 block scales [E,2I,H/32] and [E,H,I/32] into the blocks the
// FP4 expert kernel copies whole: for every (expert, tile, k-block) the two
// 128-row halves' scale pairs, 512 bytes (rows past the matrix: scale 1).
__global__ void __launch_bounds__(256) fp4_scales_kernel(const uint8_t* __restrict__ gu_s,
                                                         const uint8_t* __restrict__ dn_s, int E, int H, int I,
                                                         uint8_t* __restrict__ out) {
  const int mb0 = ceil_div(I, kHalfRows), kb0 = H / kBlockK;
  const int mb1 = ceil_div(H, 2 * kHalfRows), kb1 = I / kBlockK;
  const long long n0 = static_cast<long long>(E) * mb0 * kb0 * 256;  // scale pairs
  const long long n = n0 + static_cast<long long>(E) * mb1 * kb1 * 256;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += static_cast<long long>(gridDim.x) * 256) {
    const bool dn = i >= n0;
    const long long j = dn ? i - n0 : i;
    const int r = static_cast<int>(j % kHalfRows), h = static_cast<int>((j / kHalfRows) % 2);
    const long long blk = j / 256;  // (e, m, kb)
    const int kbs = dn ? kb1 : kb0, mbs = dn ? mb1 : mb0;
    const int kb = static_cast<int>(blk % kbs), m = static_cast<int>((blk / kbs) % mbs);
    const int e = static_cast<int>(blk / (static_cast<long long>(kbs) * mbs));
    uint16_t v = 0x7f7f;
    if (!dn) {
      const int row = m * kHalfRows + r;
      if (row < I) {
        const uint8_t* src = gu_s + (static_cast<size_t>(e) * 2 * I + h * I + row) * (H / 32) + kb * 2;
        v = static_cast<uint16_t>(src[0] | (src[1] << 8));
      }
    } else {
      const int row = m * 2 * kHalfRows + h * kHalfRows + r;
      if (row < H) {
        const uint8_t* src = dn_s + (static_cast<size_t>(e) * H + row) * (I / 32) + kb * 2;
        v = static_cast<uint16_t>(src[0] | (src[1] << 8));
      }
    }
    reinterpret_cast<uint16_t*>(out)[i] = v;
  }
}

}  // namespace

cudaError_t launch_fp4_scales(const uint8_t* gu_s, const uint8_t* dn_s, int E, int H, int I, uint8_t* out,
                              cudaStream_t s) {
  fp4_scales_kernel<<<4 * 152, 256, 0, s>>>(gu_s, dn_s, E, H, I, out);
  return cudaGetLastError();
}

cudaError_t launch_experts(const CUtensorMap& tm_gu, const CUtensorMap& tm_gu_sh, const CUtensorMap& tm_dn,
                           const CUtensorMap& tm_dn_sh, const CUtensorMap& tm_h, const GemmParams& p, int grid,
                           size_t smem_bytes, cudaStream_t s, bool fp4) {
  auto kern = fp4 ? moe_experts_kernel<true> : moe_experts_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(fp4 ? kGemmThreadsFp4 : kGemmThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, tm_h, p);
}

cudaError_t launch_combine(const float* out_ws, const int32_t* pair_pos, int T, int K, int H, int has_shared,
                           uint16_t* y, cudaStream_t s) {
  dim3 grid(ceil_div(H, 4 * 256), T);
  combine_kernel<<<grid, 256, 0, s>>>(out_ws, pair_pos, T, K, H, has_shared, y);
  return cudaGetLastError();
}

}  // namespace moe
