// Router of the MoE-FFN layer: fp32 gate logits on CUDA cores, score ->
// select -> routing_weights per token, and the token-to-expert permutation
// plus the grouped-GEMM work list.
//
// Sources (web pages): SpecForge PR #1033 "MoE FFN for DFlash-family drafts:
// the module", section "Router" (the score -> select -> routing_weights
// template; weights gathered from the unshifted scores, renormalised with
// DeepSeek's 1e-20, times route_scale); sglang PR #48763 "[Feat] dflash: Serve
// MoE FFN drafts for DFlash and DSpark" (fp32 router logits, int32 ids);
// SpecForge PR #941 (folded router bias on the logits; DeepSeek-V4 follow-up:
// sqrtsoftplus, selection-only bias, groups); SpecForge PR #1073 "MoE drafts:
// DeepSeek-V4.1's own DSpark draft" (the expert bias shifts the picks, never
// the weights; select sees the shifted scores; tokens_per_expert counts).
#include <float.h>
#include <math.h>

#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
constexpr int kMaxExperts = 1024;
// Counting-sort permutation of the (token, slot) pairs by expert, stable in
// the pair index p = t*K + k, and (optionally) the grouped-GEMM work list.
// Run by one whole CTA of kRouteThreads threads.  Up to kPermStaged ids are
// first copied to shared memory; then each warp counts and scatters its own
// contiguous chunk of pairs (per-warp cursors), so the stable order needs no
// serial pass.  Larger inputs take one warp through all pairs.
constexpr int kPermStaged = 4096;
constexpr int kPermWarps = kRouteThreads / 32;
// shared buffer: the staged ids, later the two cost prefixes of the work list
constexpr int kPermBuf = 2080;  // long longs: >= kPermStaged / 2 and >= 2 * 1040

// Exclusive prefix sum of in[0, n) into out (n <= 4 * blockDim.x); every
// thread of the CTA calls it.  Thread t owns elements [per*t, per*t + per).
__device__ void block_scan_excl(const int* in, int* out, int n, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = tid * per;
  int loc[4], sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = i0 + j;
    loc[j] = (j < per && i < n) ? in[i] : 0;
    sum += loc[j];
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += s_warp[w];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = i0 + j;
    if (j < per && i < n) {
      out[i] = run;
      run += loc[j];
    }
  }
  __syncthreads();
}

__device__ void permute_block(const int32_t* idx, int T, int K, int E, int32_t* counts, int32_t* offsets,
                              int32_t* sorted_pair, int32_t* pair_pos, GroupEntry* groups, GemmHeader* header,
                              int H, int I, int Is, int n_max, int* s_cnt, int* s_cur, long long* s_buf,
                              uint16_t* s_wc, int64_t* spans, int32_t* span_groups, int grid, int fmt,
                              int sh_fmt, int kblk, int32_t* e2d) {
  __shared__ int s_warp[kPermWarps];
  int* s_idx = reinterpret_cast<int*>(s_buf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int TK = T * K;
  const bool staged = TK <= kPermStaged;
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  if (staged) {
    for (int q = tid; q < TK; q += blockDim.x) s_idx[q] = __ldcg(idx + q);
    for (int q = tid; q < kPermWarps * E; q += blockDim.x) s_wc[q] = 0;
  }
  __syncthreads();
  // ids outside [0, E) are not counted and get no row
  const int chunk = (TK + kPermWarps - 1) / kPermWarps;
  const int p0 = warp * chunk, p1 = min(TK, p0 + chunk);
  uint16_t* wc = s_wc + warp * E;  // this warp's per-expert counts, then cursors
  if (staged) {
    // count the warp's chunk: one leader per expert and batch adds the batch's count
    for (int base = p0; base < p1; base += 32) {
      const int q = base + lane;
      const int ev = q < p1 ? s_idx[q] : -1;
      const bool act = static_cast<unsigned>(ev) < static_cast<unsigned>(E);
      const uint32_t peers = __match_any_sync(0xffffffffu, act ? ev : -1 - lane);
      if (act && lane == __ffs(peers) - 1) wc[ev] = static_cast<uint16_t>(wc[ev] + __popc(peers));
      __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
      int c = 0;
      for (int w = 0; w < kPermWarps; ++w) c += s_wc[w * E + e];
      s_cnt[e] = c;
    }
  } else {
    for (int q = tid; q < TK; q += blockDim.x) {
      const int e = __ldcg(idx + q);
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&s_cnt[e], 1);
    }
  }
  __syncthreads();
  block_scan_excl(s_cnt, s_cur, E, s_warp);  // s_cur[e]: first row of expert e
  if (staged) {
    // each warp's rows of expert e follow those of the warps before it
    for (int e = tid; e < E; e += blockDim.x) {
      int run = s_cur[e];
      for (int w = 0; w < kPermWarps; ++w) {
        const int c = s_wc[w * E + e];
        s_wc[w * E + e] = static_cast<uint16_t>(run);
        run += c;
      }
    }
    __syncthreads();
    for (int base = p0; base < p1; base += 32) {
      const int q = base + lane;
      const int ev = q < p1 ? s_idx[q] : -1;
      const bool act = static_cast<unsigned>(ev) < static_cast<unsigned>(E);
      const uint32_t peers = __match_any_sync(0xffffffffu, act ? ev : -1 - lane);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int leader = __ffs(peers) - 1;
      int bpos = (act && lane == leader) ? static_cast<int>(wc[ev]) : 0;
      bpos = __shfl_sync(0xffffffffu, bpos, leader);
      if (act) {
        sorted_pair[bpos + rank] = q;
        pair_pos[q] = bpos + rank;
      }
      __syncwarp();
      if (act && lane == leader) wc[ev] = static_cast<uint16_t>(bpos + __popc(peers));
      __syncwarp();
    }
  } else {
    // inputs too large to stage at once: chunks of kPermStaged ids in order,
    // each scattered like the staged case by all warps (a warp's rows of an
    // expert follow those of the warps before it and of the chunks before);
    // the warps' cursors count from the expert's rows so far (16 bits hold a
    // chunk), s_cur advances by each chunk's counts
    for (int c0 = 0; c0 < TK; c0 += kPermStaged) {
      const int cn = min(kPermStaged, TK - c0);
      __syncthreads();  // the previous chunk is scattered and counted in s_cur
      for (int q = tid; q < cn; q += blockDim.x) s_idx[q] = __ldcg(idx + c0 + q);
      for (int q = tid; q < kPermWarps * E; q += blockDim.x) s_wc[q] = 0;
      __syncthreads();
      const int ch = (cn + kPermWarps - 1) / kPermWarps;
      const int q0 = warp * ch, q1 = min(cn, q0 + ch);
      for (int base = q0; base < q1; base += 32) {
        const int q = base + lane;
        const int ev = q < q1 ? s_idx[q] : -1;
        const bool act = static_cast<unsigned>(ev) < static_cast<unsigned>(E);
        const uint32_t peers = __match_any_sync(0xffffffffu, act ? ev : -1 - lane);
        if (act && lane == __ffs(peers) - 1) wc[ev] = static_cast<uint16_t>(wc[ev] + __popc(peers));
        __syncwarp();
      }
      __syncthreads();
      for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < kPermWarps; ++w) {
          const int c = s_wc[w * E + e];
          s_wc[w * E + e] = static_cast<uint16_t>(run);
          run += c;
        }
      }
      __syncthreads();
      for (int base = q0; base < q1; base += 32) {
        const int q = base + lane;
        const int ev = q < q1 ? s_idx[q] : -1;
        const bool act = static_cast<unsigned>(ev) < static_cast<unsigned>(E);
        const uint32_t peers = __match_any_sync(0xffffffffu, act ? ev : -1 - lane);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int leader = __ffs(peers) - 1;
        int rel = (act && lane == leader) ? static_cast<int>(wc[ev]) : 0;
        rel = __shfl_sync(0xffffffffu, rel, leader);
        if (act) {
          const int pos = s_cur[ev] + rel + rank;
          sorted_pair[pos] = c0 + q;
          pair_pos[c0 + q] = pos;
        }
        __syncwarp();
        if (act && lane == leader) wc[ev] = static_cast<uint16_t>(rel + __popc(peers));
        __syncwarp();
      }
      __syncthreads();
      // the last warp's cursor ends at the chunk's count of the expert
      for (int e = tid; e < E; e += blockDim.x) s_cur[e] += s_wc[(kPermWarps - 1) * E + e];
    }
  }
  __syncthreads();
  if (!staged) {  // the chunks advanced s_cur to the ends: back to the starts
    for (int e = tid; e < E; e += blockDim.x) s_cur[e] -= s_cnt[e];
    __syncthreads();
  }
  for (int e = tid; e < E; e += blockDim.x) {
    if (counts) counts[e] = s_cnt[e];
    if (offsets) offsets[e + 1] = s_cur[e] + s_cnt[e];
  }
  if (tid == 0 && offsets) offsets[0] = 0;
  if (groups == nullptr) return;
  // ---- work list: one group per touched expert (expert order), then the
  // shared expert; prefix sums of tiles, k-block iterations and k-block costs
  // per GEMM.  Thread t owns experts [per*t, per*t + per); one block-wide
  // scan gives every prefix.  The cost prefixes go to shared memory (the
  // staged ids are no longer needed) for the span computation below.
  long long* s_cost0 = s_buf;              // [groups + 1]
  long long* s_cost1 = s_buf + 1040;       // [groups + 1]
  __shared__ int s_ngroups;
  __shared__ int s_neff;
  __shared__ long long s_tot[4];           // gate_up iters, down iters, gate_up cost, down cost
  __shared__ long long s_wtot[kPermWarps][4];
  if (tid == 0) s_neff = 16;
  __syncthreads();
  // widest token tile: the largest count (capped at n_max), shared expert
  // included; reduced within each warp first, so one shared atomic per warp
  {
    int wmax = (tid == 0 && Is > 0) ? min(n_max, (T + 15) & ~15) : 16;
    for (int e = tid; e < E; e += blockDim.x)
      if (s_cnt[e] > 0) wmax = max(wmax, min(n_max, (s_cnt[e] + 15) & ~15));
    wmax = __reduce_max_sync(0xffffffffu, wmax);
    if (lane == 0) atomicMax(&s_neff, wmax);
  }
  // geometry of a routed expert's tiles (every routed expert has the same I)
  const int mb0 = ceil_div(I, kHalfRows), kb0 = ceil_div(H, kblk);
  const int mb1 = ceil_div(H, 2 * kHalfRows), kb1 = ceil_div(I, kblk);
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = tid * per;
  // this thread's sums: touched experts, token blocks, gate_up cost, down cost
  long long v[4] = {0, 0, 0, 0};
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    const int c = e < E ? s_cnt[e] : 0;
    if (c > 0) {
      const int nb = ceil_div(c, n_max);
      const int nmma = max(16, min(n_max, (c + 15) & ~15));
      v[0] += 1;
      v[1] += nb;
      v[2] += static_cast<long long>(nb) * mb0 * kb0 * kblock_cost(0, nmma, fmt);
      v[3] += static_cast<long long>(nb) * mb1 * kb1 * kblock_cost(1, nmma, fmt);
    }
  }
  long long incl[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const long long o = __shfl_up_sync(0xffffffffu, incl[q], off);
      if (lane >= off) incl[q] += o;
    }
  }
  if (lane == 31)
    for (int q = 0; q < 4; ++q) s_wtot[warp][q] = incl[q];
  __syncthreads();
  long long run[4], tot[4];
  for (int q = 0; q < 4; ++q) {
    run[q] = incl[q] - v[q];
    tot[q] = 0;
  }
  for (int w = 0; w < kPermWarps; ++w)
    for (int q = 0; q < 4; ++q) {
      if (w < warp) run[q] += s_wtot[w][q];
      tot[q] += s_wtot[w][q];
    }
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    const int c = e < E ? s_cnt[e] : 0;
    if (c > 0) {
      const int nb = ceil_div(c, n_max);
      const int nmma = max(16, min(n_max, (c + 15) & ~15));
      const int gi = static_cast<int>(run[0]);
      const int w0 = kblock_cost(0, nmma, fmt), w1 = kblock_cost(1, nmma, fmt);
      GroupEntry ge;
      ge.expert = e;
      ge.row_base = s_cur[e];
      ge.count = c;
      ge.idim = I;
      ge.gu_tile = static_cast<int>(run[1]) * mb0;
      ge.dn_tile = static_cast<int>(run[1]) * mb1;
      ge.gu_w = w0;
      ge.dn_w = w1;
      ge.gu_iter = run[1] * mb0 * kb0;
      ge.dn_iter = run[1] * mb1 * kb1;
      groups[gi] = ge;
      if (e2d) e2d[e] = static_cast<int32_t>(run[1]);  // the expert's first token block, counted over all groups
      s_cost0[gi] = run[2];
      s_cost1[gi] = run[3];
      run[0] += 1;
      run[1] += nb;
      run[2] += static_cast<long long>(nb) * mb0 * kb0 * w0;
      run[3] += static_cast<long long>(nb) * mb1 * kb1 * w1;
    }
  }
  __syncthreads();  // s_neff is final
  if (tid == 0) {
    int g = static_cast<int>(tot[0]);
    int gu_t = static_cast<int>(tot[1]) * mb0, dn_t = static_cast<int>(tot[1]) * mb1;
    long long gu_i = tot[1] * mb0 * kb0, dn_i = tot[1] * mb1 * kb1, gu_c = tot[2], dn_c = tot[3];
    if (Is > 0) {
      int mb, nb, kb;
      const int nmma = max(16, min(n_max, (T + 15) & ~15));
      const int w0 = kblock_cost(0, nmma, sh_fmt), w1 = kblock_cost(1, nmma, sh_fmt);
      GroupEntry ge;
      ge.expert = -1;
      ge.row_base = TK;
      ge.count = T;
      ge.idim = Is;
      ge.gu_tile = gu_t;
      ge.dn_tile = dn_t;
      ge.gu_w = w0;
      ge.dn_w = w1;
      ge.gu_iter = gu_i;
      ge.dn_iter = dn_i;
      groups[g] = ge;
      s_cost0[g] = gu_c;
      s_cost1[g] = dn_c;
      group_geometry(0, T, Is, H, n_max, mb, nb, kb, kblk);
      gu_t += mb * nb;
      gu_i += static_cast<long long>(mb) * nb * kb;
      gu_c += static_cast<long long>(mb) * nb * kb * w0;
      group_geometry(1, T, Is, H, n_max, mb, nb, kb, kblk);
      dn_t += mb * nb;
      dn_i += static_cast<long long>(mb) * nb * kb;
      dn_c += static_cast<long long>(mb) * nb * kb * w1;
      ++g;
    }
    GemmHeader hd;
    hd.ngroups = g;
    hd.gu_tiles = gu_t;
    hd.dn_tiles = dn_t;
    hd.n_eff = s_neff;
    hd.gu_iters = gu_i;
    hd.dn_iters = dn_i;
    *header = hd;
    s_ngroups = g;
    s_tot[0] = gu_i;
    s_tot[1] = dn_i;
    s_tot[2] = gu_c;
    s_tot[3] = dn_c;
  }
  __syncthreads();
  // ---- CTA spans: cut each GEMM's total cost into `grid` equal parts and
  // round every cut to a whole k-block iteration.
  const int ng = s_ngroups;
  for (int q = tid; q < 2 * (grid + 1); q += blockDim.x) {
    const int ph = q / (grid + 1), c = q % (grid + 1);
    const long long* cs = ph == 0 ? s_cost0 : s_cost1;
    const long long total_cost = s_tot[2 + ph], total_it = s_tot[ph];
    const long long pos = total_cost * c / grid;
    long long it = total_it;
    int gsel = ng;
    if (pos < total_cost && ng > 0) {
      int lo = 0, hi = ng - 1;  // last group whose cost starts at or before pos
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cs[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      const GroupEntry& ge = groups[lo];
      const long long w = ph == 0 ? ge.gu_w : ge.dn_w;
      const long long i0 = ph == 0 ? ge.gu_iter : ge.dn_iter;
      it = i0 + (pos - cs[lo] + w - 1) / w;
      const long long next = lo + 1 < ng ? (ph == 0 ? groups[lo + 1].gu_iter : groups[lo + 1].dn_iter) : total_it;
      gsel = it < next ? lo : lo + 1;
    }
    spans[q] = it;
    span_groups[q] = gsel;
  }
}

// One launch: every CTA computes a TB-token x (4*quads)-row block of the fp32
// logits (row E is the shared-expert gate when present); the last CTA of a
// token block selects its tokens; the last token block builds the
// permutation and the work list.
// Two bf16 values -> two f16 values (round to nearest even); `over` is set
// when one leaves the f16 range.
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w, bool& over) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
  over |= !(fabsf(lo) < 65520.f) || !(fabsf(hi) < 65520.f);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int TB, int NJ>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteParams p) {
  __shared__ float red[8][TB][4];
  __shared__ float s_log[TB][33];  // the block's logits when it covers every expert (E <= 32)
  __shared__ int s_flag;
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_cur[kMaxExperts];
  __shared__ long long s_buf[kPermBuf];
  __shared__ uint16_t s_wc[kPermWarps * kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tbi = blockIdx.x, ebi = blockIdx.y;
  // The shared-expert gate is one more row of the GEMV, unless that row
  // would add an expert block (fold_sh): then the quad-0 warps of every
  // block add x.sh_gate over a disjoint subset of H steps and leave partial
  // sums that the selecting warp adds in block order.
  const bool fold = p.fold_sh != 0;
  const int E_tot = p.E + ((p.sh_gate && !fold) ? 1 : 0);
  {  // clear the GEMM tile counters for this forward
    const int nthr = gridDim.x * gridDim.y * kRouteThreads;
    const int gid = (blockIdx.y * gridDim.x + blockIdx.x) * kRouteThreads + threadIdx.x;
    for (int i = gid; i < p.zero_count; i += nthr) p.zero_ptr[i] = 0;
  }
  const int t0 = tbi * TB;
  const SelCfg sel{p.E, p.K, p.score_fn, p.n_group, p.topk_group, p.group_topn, p.renorm, p.eps, p.scale,
                   p.expert_bias};
  if (p.logits_given) {
    // the logits (and the shared-gate logit) come from logits_gemm_kernel:
    // warp w routes token t0 + w
    if (warp < TB && t0 + warp < p.T) {
      const int tok = t0 + warp;
      if (p.lsplit > 1) {
        // the GEMM's partial sums of this token's logits, added in split order
        const int E_tot = p.E + (p.sh_gate ? 1 : 0);
        for (int e = lane; e < E_tot; e += 32) {
          float v = 0.f;
          for (int zz = 0; zz < p.lsplit; ++zz)
            v += __ldcg(p.lpart + (static_cast<size_t>(zz) * p.T + tok) * E_tot + e);
          if (e < p.E) {
            if (p.router_bias) v += __ldg(p.router_bias + e);
            p.logits[static_cast<size_t>(tok) * p.E + e] = v;
          } else {
            p.sh_logit[tok] = v;
          }
        }
        __syncwarp();
      }
      select_token<NJ, false>(p.logits + static_cast<size_t>(tok) * p.E, sel,
                              p.idx + static_cast<size_t>(tok) * p.K, p.w + static_cast<size_t>(tok) * p.K);
      if (lane == 0 && p.sh_w) p.sh_w[tok] = p.sh_gate ? 1.f / (1.f + expf(-__ldcg(p.sh_logit + tok))) : 1.f;
    }
  } else {
  // ---- logits block
  const int quad = warp / p.hsplit, hs = warp % p.hsplit;
  const int e0 = (ebi * p.quads + quad) * 4;
  const uint16_t* rows[4];
  bool ev[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = e0 + q;
    ev[q] = quad < p.quads && e < E_tot;
    rows[q] = e < p.E ? p.gate + static_cast<size_t>(e) * p.H : p.sh_gate;
  }
  const int hs_len = ceil_div(ceil_div(p.H, p.hsplit), 8) * 8;
  const int h_lo = hs * hs_len;
  const int h_hi = min(p.H, h_lo + hs_len);
  float acc[TB][4], acc_sh[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    acc_sh[t] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[t][q] = 0.f;
  }
  const bool do_sh = fold && quad == 0;
  // FP4 experts multiply in f16: the quad-0 warps of expert block 0 (which
  // cover H once) also write the f16 copy of their x columns
  const bool xh_w = p.xh != nullptr && ebi == 0 && quad == 0;
  // D - 1 steps of loads stay in flight while a step is multiplied (two
  // for 4-token blocks; one for 8-token blocks, whose registers are full)
  constexpr int D = TB <= 4 ? 3 : 2;
  uint4 gb[D][4], xb[D][TB], sb[D];
  auto load_step = [&](int c, int step, uint4 (&g)[4], uint4 (&xx)[TB], uint4& sg) {
#pragma unroll
    for (int q = 0; q < 4; ++q) g[q] = ev[q] ? ldg128(rows[q] + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int t = 0; t < TB; ++t)
      xx[t] = (t0 + t < p.T) ? ldg128(p.x + static_cast<size_t>(t0 + t) * p.H + c) : make_uint4(0, 0, 0, 0);
    sg = (do_sh && step % p.n_eb == ebi) ? ldg128(p.sh_gate + c) : make_uint4(0, 0, 0, 0);
  };
  const int c0 = h_lo + lane * 8;
#pragma unroll
  for (int d = 0; d + 1 < D; ++d)
    if (c0 + d * 256 < h_hi) load_step(c0 + d * 256, d, gb[d], xb[d], sb[d]);
  for (int base = 0; c0 + base * 256 < h_hi; base += D) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int step = base + d;
      const int c = c0 + step * 256;
      if (c < h_hi) {
        const int dn = (d + D - 1) % D;  // the slot freed one step ago
        if (c + (D - 1) * 256 < h_hi) load_step(c + (D - 1) * 256, step + D - 1, gb[dn], xb[dn], sb[dn]);
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[t][q] = dot8(xb[d][t], gb[d][q], acc[t][q]);
        if (do_sh && step % p.n_eb == ebi) {
#pragma unroll
          for (int t = 0; t < TB; ++t) acc_sh[t] = dot8(xb[d][t], sb[d], acc_sh[t]);
        }
        if (xh_w) {
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            if (t0 + t < p.T) {
              bool over = false;
              uint4 o;
              o.x = bf2_to_h2(xb[d][t].x, over);
              o.y = bf2_to_h2(xb[d][t].y, over);
              o.z = bf2_to_h2(xb[d][t].z, over);
              o.w = bf2_to_h2(xb[d][t].w, over);
              *reinterpret_cast<uint4*>(p.xh + static_cast<size_t>(t0 + t) * p.H + c) = o;
              if (over) record_range(p.status, kInfoXRange);
            }
          }
        }
      }
    }
  }
  if (do_sh) {
    // this block's partial of x.sh_gate for each token: slot ebi*hsplit + hs
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      float v = acc_sh[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && t0 + t < p.T)
        p.sh_logit[static_cast<size_t>(t0 + t) * p.n_eb * p.hsplit + ebi * p.hsplit + hs] = v;
    }
  }
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v = acc[t][q];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[t][q] = v;
    }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) red[warp][t][q] = acc[t][q];
  }
  __syncthreads();
  for (int o = threadIdx.x; o < p.quads * 4 * TB; o += kRouteThreads) {
    const int qd = o / (4 * TB), rem = o % (4 * TB), t = rem / 4, q = rem % 4;
    const int e = (ebi * p.quads + qd) * 4 + q, tok = t0 + t;
    if (e < E_tot && tok < p.T) {
      float v = red[qd * p.hsplit][t][q];
      for (int h2 = 1; h2 < p.hsplit; ++h2) v += red[qd * p.hsplit + h2][t][q];
      if (e < p.E) {
        if (p.router_bias) v += __ldg(p.router_bias + e);
        p.logits[static_cast<size_t>(tok) * p.E + e] = v;
      } else {
        p.sh_logit[tok] = v;
      }
      if (p.n_eb == 1) s_log[t][e] = v;
    }
  }
  if (p.n_eb == 1) {
    // this block holds every expert's logit of its tokens: select from shared memory
    __syncthreads();
    if (warp < TB && t0 + warp < p.T) {
      const int tok = t0 + warp;
      if (NJ == 1)
        select_token<1, true>(s_log[warp], sel, p.idx + static_cast<size_t>(tok) * p.K,
                              p.w + static_cast<size_t>(tok) * p.K);
      if (lane == 0 && p.sh_w) p.sh_w[tok] = p.sh_gate ? 1.f / (1.f + expf(-s_log[warp][p.E])) : 1.f;
    }
  } else {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int old = atomicAdd(&p.tb_counter[tbi], 1);
      const int last = (old == p.n_eb - 1);
      if (last) p.tb_counter[tbi] = 0;
      s_flag = last;
    }
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    // ---- selection: warp w routes token t0 + w
    if (warp < TB && t0 + warp < p.T) {
      const int tok = t0 + warp;
      select_token<NJ, false>(p.logits + static_cast<size_t>(tok) * p.E, sel,
                              p.idx + static_cast<size_t>(tok) * p.K, p.w + static_cast<size_t>(tok) * p.K);
      if (lane == 0 && p.sh_w) {
        float v = 0.f;
        if (fold) {  // the blocks' partials of x.sh_gate, in block order
          const int np = p.n_eb * p.hsplit;
          for (int i = 0; i < np; ++i) v += __ldcg(p.sh_logit + static_cast<size_t>(tok) * np + i);
        } else if (p.sh_gate) {
          v = __ldcg(p.sh_logit + tok);
        }
        p.sh_w[tok] = p.sh_gate ? 1.f / (1.f + expf(-v)) : 1.f;
      }
    }
  }
  }  // logits computed here
  if (!p.do_permute) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(p.glob_counter, 1);
    const int last = (old == p.n_tb - 1);
    if (last) *p.glob_counter = 0;
    s_flag = last;
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  permute_block(p.idx, p.T, p.K, p.E, p.counts, p.offsets, p.sorted_pair, p.pair_pos, p.groups, p.header, p.H,
                p.I, p.Is, p.n_max, s_cnt, s_cur, s_buf, s_wc, p.spans, p.span_groups, p.grid,
                p.fmt != 0 ? p.fmt : (p.fp4 ? kFmtFp4Conv : kFmtBf16), p.sh_fmt, p.kblk > 0 ? p.kblk : kBlockK, p.e2d);
}

// logits = x . gate^T (+ router_bias) for many tokens: a CTA computes a
// 128-token x 64-expert tile with x and gate staged through shared memory as
// fp32, each thread an 8 x 4 block accumulated over its range of H in
// increasing order (fp32 fused multiply-adds of the exact bf16 products);
// with one range the tile is the logits, with several each range's partial
// sums go to `part` for the router launch to add in range order.  Column E
// is the shared-expert gate when sh_gate is given (-> sh_logit).
constexpr int kLgBM = 128, kLgBN = 64, kLgBK = 32;

__global__ void __launch_bounds__(256) logits_gemm_kernel(const uint16_t* __restrict__ x,
                                                          const uint16_t* __restrict__ gate,
                                                          const uint16_t* __restrict__ sh_gate,
                                                          const float* __restrict__ router_bias, int T, int H, int E,
                                                          float* __restrict__ logits, float* __restrict__ sh_logit,
                                                          int split, float* __restrict__ part) {
  // x and gate chunks as fp32, k-major; row k starts 8*(k/8) words further
  // than its stride alone would place it, so that the four lanes storing one
  // token's (or gate row's) 8 inputs hit four different banks
  __shared__ __align__(16) float As[kLgBK * (kLgBM + 4) + 24];
  __shared__ __align__(16) float Bs[kLgBK * (kLgBN + 4) + 24];
  auto a_at = [](int k, int t) { return k * (kLgBM + 4) + ((k >> 3) << 3) + t; };
  auto b_at = [](int k, int e) { return k * (kLgBN + 4) + ((k >> 3) << 3) + e; };
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * kLgBM, e0 = blockIdx.y * kLgBN;
  const int E_tot = E + (sh_gate ? 1 : 0);
  // this slice's range of H: chunks [nch*z/split, nch*(z+1)/split) of 32 inputs
  const int nch = ceil_div(H, kLgBK), z = blockIdx.z;
  const int h_lo = nch * z / split * kLgBK, h_hi = min(H, nch * (z + 1) / split * kLgBK);
  // loader: x rows lr and lr + 64, gate row lr; 8 consecutive h at lc
  const int lr = tid >> 2, lc = (tid & 3) * 8;
  const uint16_t* xrow0 = t0 + lr < T ? x + static_cast<size_t>(t0 + lr) * H : nullptr;
  const uint16_t* xrow1 = t0 + lr + 64 < T ? x + static_cast<size_t>(t0 + lr + 64) * H : nullptr;
  const int ex = e0 + lr;
  const uint16_t* grow = ex < E ? gate + static_cast<size_t>(ex) * H : (ex < E_tot ? sh_gate : nullptr);
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  uint4 xv0 = (xrow0 && h_lo + lc < h_hi) ? ldg128(xrow0 + h_lo + lc) : zero;
  uint4 xv1 = (xrow1 && h_lo + lc < h_hi) ? ldg128(xrow1 + h_lo + lc) : zero;
  uint4 gv = (grow && h_lo + lc < h_hi) ? ldg128(grow + h_lo + lc) : zero;
  for (int h0 = h_lo; h0 < h_hi; h0 += kLgBK) {
    __syncthreads();  // the previous chunk is read
    const uint32_t x0w[4] = {xv0.x, xv0.y, xv0.z, xv0.w}, x1w[4] = {xv1.x, xv1.y, xv1.z, xv1.w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      As[a_at(lc + 2 * i, lr)] = bf_lo(x0w[i]);
      As[a_at(lc + 2 * i + 1, lr)] = bf_hi(x0w[i]);
      As[a_at(lc + 2 * i, lr + 64)] = bf_lo(x1w[i]);
      As[a_at(lc + 2 * i + 1, lr + 64)] = bf_hi(x1w[i]);
      Bs[b_at(lc + 2 * i, lr)] = bf_lo(gw[i]);
      Bs[b_at(lc + 2 * i + 1, lr)] = bf_hi(gw[i]);
    }
    __syncthreads();
    const int hn = h0 + kLgBK + lc;  // the next chunk's loads overlap this chunk's products
    xv0 = (xrow0 && hn < h_hi) ? ldg128(xrow0 + hn) : zero;
    xv1 = (xrow1 && hn < h_hi) ? ldg128(xrow1 + hn) : zero;
    gv = (grow && hn < h_hi) ? ldg128(grow + hn) : zero;
#pragma unroll
    for (int k = 0; k < kLgBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[a_at(k, ty * 8)]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[a_at(k, ty * 8 + 4)]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[b_at(k, tx * 4)]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (split > 1) {
        if (e < E_tot) part[(static_cast<size_t>(z) * T + t) * E_tot + e] = acc[i][j];
      } else if (e < E) {
        logits[static_cast<size_t>(t) * E + e] = acc[i][j] + (router_bias ? __ldg(router_bias + e) : 0.f);
      } else if (e < E_tot) {
        sh_logit[t] = acc[i][j];
      }
    }
  }
}

template <int NJ>
__global__ void __launch_bounds__(kRouteThreads) select_kernel(const float* logits, int T, SelCfg c, int32_t* idx,
                                                               float* w) {
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tok >= T) return;
  select_token<NJ, false>(logits + static_cast<size_t>(tok) * c.E, c, idx + static_cast<size_t>(tok) * c.K,
                          w + static_cast<size_t>(tok) * c.K);
}

__global__ void __launch_bounds__(kRouteThreads) permute_kernel(const int32_t* idx, int T, int K, int E,
                                                                int32_t* counts, int32_t* offsets,
                                                                int32_t* sorted_pair, int32_t* pair_pos) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_cur[kMaxExperts];
  __shared__ long long s_buf[kPermBuf];
  __shared__ uint16_t s_wc[kPermWarps * kMaxExperts];
  permute_block(idx, T, K, E, counts, offsets, sorted_pair, pair_pos, nullptr, nullptr, 0, 0, 0, 1, s_cnt, s_cur,
                s_buf, s_wc, nullptr, nullptr, 0, kFmtBf16, kFmtBf16, kBlockK, nullptr);
}

}  // namespace

cudaError_t launch_logits_gemm(const uint16_t* x, const uint16_t* gate, const uint16_t* sh_gate,
                               const float* router_bias, int T, int H, int E, float* logits, float* sh_logit,
                               int split, float* part, cudaStream_t s) {
  const int E_tot = E + (sh_gate ? 1 : 0);
  dim3 grid(ceil_div(T, kLgBM), ceil_div(E_tot, kLgBN), split);
  logits_gemm_kernel<<<grid, 256, 0, s>>>(x, gate, sh_gate, router_bias, T, H, E, logits, sh_logit, split, part);
  return cudaGetLastError();
}

int logits_gemm_split(int T, int H, int E_tot, int sms) {
  const int tiles = ceil_div(T, kLgBM) * ceil_div(E_tot, kLgBN);
  const int by_sm = 3 * sms / tiles, by_h = ceil_div(H, kLgBK) / 8;
  const int s = by_sm < by_h ? by_sm : by_h;
  return s < 1 ? 1 : s;
}

namespace {

int nj_for(int E) {
  const int nj = ceil_div(E, 32);
  if (nj <= 1) return 1;
  if (nj <= 2) return 2;
  if (nj <= 4) return 4;
  if (nj <= 8) return 8;
  if (nj <= 16) return 16;
  return 32;
}

template <int TB>
cudaError_t launch_route_tb(const RouteParams& p, cudaStream_t s) {
  dim3 grid(p.n_tb, p.n_eb);
  switch (nj_for(p.E)) {
    case 1: route_kernel<TB, 1><<<grid, kRouteThreads, 0, s>>>(p); break;
    case 2: route_kernel<TB, 2><<<grid, kRouteThreads, 0, s>>>(p); break;
    case 4: route_kernel<TB, 4><<<grid, kRouteThreads, 0, s>>>(p); break;
    case 8: route_kernel<TB, 8><<<grid, kRouteThreads, 0, s>>>(p); break;
    case 16: route_kernel<TB, 16><<<grid, kRouteThreads, 0, s>>>(p); break;
    default: route_kernel<TB, 32><<<grid, kRouteThreads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, int tb, cudaStream_t s) {
  return tb == 4 ? launch_route_tb<4>(p, s) : launch_route_tb<8>(p, s);
}

cudaError_t launch_select_from_logits(const float* logits, int T, int E, int K, const float* expert_bias,
                                      int score_fn, int n_group, int topk_group, int group_topn, int renorm,
                                      float eps, float scale, int32_t* idx, float* w, cudaStream_t s) {
  SelCfg c{E, K, score_fn, n_group, topk_group, group_topn, renorm, eps, scale, expert_bias};
  const int grid = ceil_div(T, 8);
  switch (nj_for(E)) {
    case 1: select_kernel<1><<<grid, kRouteThreads, 0, s>>>(logits, T, c, idx, w); break;
    case 2: select_kernel<2><<<grid, kRouteThreads, 0, s>>>(logits, T, c, idx, w); break;
    case 4: select_kernel<4><<<grid, kRouteThreads, 0, s>>>(logits, T, c, idx, w); break;
    case 8: select_kernel<8><<<grid, kRouteThreads, 0, s>>>(logits, T, c, idx, w); break;
    case 16: select_kernel<16><<<grid, kRouteThreads, 0, s>>>(logits, T, c, idx, w); break;
    default: select_kernel<32><<<grid, kRouteThreads, 0, s>>>(logits, T, c, idx, w); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* idx, int T, int K, int E, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* pair_pos, cudaStream_t s) {
  permute_kernel<<<1, kRouteThreads, 0, s>>>(idx, T, K, E, counts, offsets, sorted_pair, pair_pos);
  return cudaGetLastError();
}

}  // namespace moe
