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

#include "moe_internal.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
constexpr int kMaxExperts = 1024;
// Counting-sort permutation of the (token, slot) pairs by expert, stable in
// the pair index p = t*K + k, and (optionally) the grouped-GEMM work list.
// Run by one whole CTA.  Up to kPermStaged ids are first copied to shared
// memory in one parallel pass, so the serial scatter reads them from there.
constexpr int kPermStaged = 4096;
// shared buffer: the staged ids, later the two cost prefixes of the work list
constexpr int kPermBuf = 2080;  // long longs: >= kPermStaged / 2 and >= 2 * 1040

__device__ void permute_block(const int32_t* idx, int T, int K, int E, int32_t* counts, int32_t* offsets,
                              int32_t* sorted_pair, int32_t* pair_pos, GroupEntry* groups, GemmHeader* header,
                              int H, int I, int Is, int n_max, int* s_cnt, int* s_cur, long long* s_buf,
                              int64_t* spans, int32_t* span_groups, int grid) {
  int* s_idx = reinterpret_cast<int*>(s_buf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int TK = T * K;
  const bool staged = TK <= kPermStaged;
  for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
  if (staged)
    for (int p = tid; p < TK; p += blockDim.x) s_idx[p] = __ldcg(idx + p);
  __syncthreads();
  // ids outside [0, E) are not counted and get no row
  for (int p = tid; p < TK; p += blockDim.x) {
    const int e = staged ? s_idx[p] : __ldcg(idx + p);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int v = e < E ? s_cnt[e] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
      }
      if (e < E) s_cur[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    for (int base = 0; base < TK; base += 32) {
      const int p = base + lane;
      const int ev = p < TK ? (staged ? s_idx[p] : __ldcg(idx + p)) : -1;
      const bool act = static_cast<unsigned>(ev) < static_cast<unsigned>(E);
      const int e = act ? ev : -1 - lane;
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int leader = __ffs(peers) - 1;
      int bpos = (act && lane == leader) ? s_cur[e] : 0;
      bpos = __shfl_sync(0xffffffffu, bpos, leader);
      if (act) {
        sorted_pair[bpos + rank] = p;
        pair_pos[p] = bpos + rank;
      }
      __syncwarp();
      if (act && lane == leader) s_cur[e] = bpos + __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  // s_cur[e] now holds the end of expert e's rows
  for (int e = tid; e < E; e += blockDim.x) {
    if (counts) counts[e] = s_cnt[e];
    if (offsets) offsets[e + 1] = s_cur[e];
  }
  if (tid == 0 && offsets) offsets[0] = 0;
  if (groups == nullptr) return;
  // ---- work list: one group per touched expert (expert order), then the
  // shared expert; prefix sums of tiles, k-block iterations and k-block costs
  // per GEMM.  The cost prefix goes to shared memory (the staged ids are no
  // longer needed) for the span computation below.
  long long* s_cost0 = s_buf;              // [groups + 1]
  long long* s_cost1 = s_buf + 1040;       // [groups + 1]
  __shared__ int s_ngroups;
  __shared__ int s_neff;
  __shared__ long long s_tot[4];           // gate_up iters, down iters, gate_up cost, down cost
  if (tid == 0) s_neff = 16;
  __syncthreads();
  // widest token tile: the largest count (capped at n_max), shared expert included
  for (int e = tid; e < E; e += blockDim.x)
    if (s_cnt[e] > 0) atomicMax(&s_neff, min(n_max, (s_cnt[e] + 15) & ~15));
  if (tid == 0 && Is > 0) atomicMax(&s_neff, min(n_max, (T + 15) & ~15));
  __syncthreads();
  if (warp == 0) {
    int g = 0, gu_t = 0, dn_t = 0;
    long long gu_i = 0, dn_i = 0, gu_c = 0, dn_c = 0;
    auto geometry = [&](int c, int idim, int& gut, int& dnt, long long& gui, long long& dni, int& w0, int& w1) {
      int mb, nb, kb;
      const int nmma = max(16, min(n_max, (c + 15) & ~15));
      group_geometry(0, c, idim, H, n_max, mb, nb, kb);
      gut = mb * nb;
      gui = static_cast<long long>(gut) * kb;
      group_geometry(1, c, idim, H, n_max, mb, nb, kb);
      dnt = mb * nb;
      dni = static_cast<long long>(dnt) * kb;
      w0 = kblock_cost(0, nmma);
      w1 = kblock_cost(1, nmma);
    };
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? s_cnt[e] : 0;
      const bool touched = c > 0;
      const uint32_t m = __ballot_sync(0xffffffffu, touched);
      int gut = 0, dnt = 0, w0 = 0, w1 = 0;
      long long gui = 0, dni = 0;
      if (touched) geometry(c, I, gut, dnt, gui, dni, w0, w1);
      const long long guc = gui * w0, dnc = dni * w1;
      int a = gut, b = dnt;
      long long ci = gui, di = dni, cc = guc, dc = dnc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int na = __shfl_up_sync(0xffffffffu, a, off);
        const int nb2 = __shfl_up_sync(0xffffffffu, b, off);
        const long long nci = __shfl_up_sync(0xffffffffu, ci, off);
        const long long ndi = __shfl_up_sync(0xffffffffu, di, off);
        const long long ncc = __shfl_up_sync(0xffffffffu, cc, off);
        const long long ndc = __shfl_up_sync(0xffffffffu, dc, off);
        if (lane >= off) { a += na; b += nb2; ci += nci; di += ndi; cc += ncc; dc += ndc; }
      }
      if (touched) {
        const int gi = g + __popc(m & ((1u << lane) - 1u));
        GroupEntry ge;
        ge.expert = e;
        ge.row_base = s_cur[e] - c;
        ge.count = c;
        ge.idim = I;
        ge.gu_tile = gu_t + a - gut;
        ge.dn_tile = dn_t + b - dnt;
        ge.gu_w = w0;
        ge.dn_w = w1;
        ge.gu_iter = gu_i + ci - gui;
        ge.dn_iter = dn_i + di - dni;
        groups[gi] = ge;
        s_cost0[gi] = gu_c + cc - guc;
        s_cost1[gi] = dn_c + dc - dnc;
      }
      g += __popc(m);
      gu_t += __shfl_sync(0xffffffffu, a, 31);
      dn_t += __shfl_sync(0xffffffffu, b, 31);
      gu_i += __shfl_sync(0xffffffffu, ci, 31);
      dn_i += __shfl_sync(0xffffffffu, di, 31);
      gu_c += __shfl_sync(0xffffffffu, cc, 31);
      dn_c += __shfl_sync(0xffffffffu, dc, 31);
    }
    if (lane == 0) {
      if (Is > 0) {
        int gut, dnt, w0, w1;
        long long gui, dni;
        geometry(T, Is, gut, dnt, gui, dni, w0, w1);
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
        gu_t += gut;
        dn_t += dnt;
        gu_i += gui;
        dn_i += dni;
        gu_c += gui * w0;
        dn_c += dni * w1;
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
template <int TB, int NJ>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteParams p) {
  __shared__ float red[8][TB][4];
  __shared__ float s_log[TB][33];  // the block's logits when it covers every expert (E <= 32)
  __shared__ int s_flag;
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_cur[kMaxExperts];
  __shared__ long long s_buf[kPermBuf];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tbi = blockIdx.x, ebi = blockIdx.y;
  const int E_tot = p.E + (p.sh_gate ? 1 : 0);
  {  // clear the GEMM tile counters for this forward
    const int nthr = gridDim.x * gridDim.y * kRouteThreads;
    const int gid = (blockIdx.y * gridDim.x + blockIdx.x) * kRouteThreads + threadIdx.x;
    for (int i = gid; i < p.zero_count; i += nthr) p.zero_ptr[i] = 0;
  }
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
  const int t0 = tbi * TB;
  const int hs_len = ceil_div(ceil_div(p.H, p.hsplit), 8) * 8;
  const int h_lo = hs * hs_len;
  const int h_hi = min(p.H, h_lo + hs_len);
  float acc[TB][4];
#pragma unroll
  for (int t = 0; t < TB; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[t][q] = 0.f;
  // one step of loads stays in flight while the previous step is multiplied
  uint4 gv[4], xv[TB];
  auto load_step = [&](int c, uint4 (&g)[4], uint4 (&xx)[TB]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) g[q] = ev[q] ? ldg128(rows[q] + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int t = 0; t < TB; ++t)
      xx[t] = (t0 + t < p.T) ? ldg128(p.x + static_cast<size_t>(t0 + t) * p.H + c) : make_uint4(0, 0, 0, 0);
  };
  int c = h_lo + lane * 8;
  if (c < h_hi) load_step(c, gv, xv);
  while (c < h_hi) {
    const int cn = c + 256;
    uint4 gn[4], xn[TB];
    if (cn < h_hi) load_step(cn, gn, xn);
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[t][q] = dot8(xv[t], gv[q], acc[t][q]);
    if (cn < h_hi) {
#pragma unroll
      for (int q = 0; q < 4; ++q) gv[q] = gn[q];
#pragma unroll
      for (int t = 0; t < TB; ++t) xv[t] = xn[t];
    }
    c = cn;
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
  const SelCfg sel{p.E, p.K, p.score_fn, p.n_group, p.topk_group, p.group_topn, p.renorm, p.eps, p.scale,
                   p.expert_bias};
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
      if (lane == 0 && p.sh_w) p.sh_w[tok] = p.sh_gate ? 1.f / (1.f + expf(-__ldcg(p.sh_logit + tok))) : 1.f;
    }
  }
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
                p.I, p.Is, p.n_max, s_cnt, s_cur, s_buf, p.spans, p.span_groups, p.grid);
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
  permute_block(idx, T, K, E, counts, offsets, sorted_pair, pair_pos, nullptr, nullptr, 0, 0, 0, 1, s_cnt, s_cur,
                s_buf, nullptr, nullptr, 0);
}

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
