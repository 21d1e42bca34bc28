// Per-token routing on CUDA cores, shared by the router kernel and the
// fused small-expert-count kernel: bf16 dot products for the fp32 gate
// logits, and score -> select -> routing_weights by one warp per token.
//
// Sources (web pages): SpecForge PR #1033 "MoE FFN for DFlash-family drafts:
// the module", section "Router" (the score -> select -> routing_weights
// template; weights gathered from the unshifted scores, renormalised with
// DeepSeek's 1e-20, times route_scale); SpecForge PR #941's DeepSeek-V4
// follow-up (sqrtsoftplus, selection-only bias, groups); SpecForge PR #1073
// "MoE drafts: DeepSeek-V4.1's own DSpark draft" (the expert bias shifts the
// picks, never the weights).
#pragma once

#include <float.h>
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr float kNegInf = -INFINITY;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// acc += sum_i a_i * b_i over 8 bf16 pairs, one fused multiply-add at a time
// (bf16 x bf16 products are exact in fp32).
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  acc = fmaf(bf_lo(a.x), bf_lo(b.x), acc);
  acc = fmaf(bf_hi(a.x), bf_hi(b.x), acc);
  acc = fmaf(bf_lo(a.y), bf_lo(b.y), acc);
  acc = fmaf(bf_hi(a.y), bf_hi(b.y), acc);
  acc = fmaf(bf_lo(a.z), bf_lo(b.z), acc);
  acc = fmaf(bf_hi(a.z), bf_hi(b.z), acc);
  acc = fmaf(bf_lo(a.w), bf_lo(b.w), acc);
  acc = fmaf(bf_hi(a.w), bf_hi(b.w), acc);
  return acc;
}

__device__ __forceinline__ uint4 ldg128(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Order-preserving image of a float in the unsigned integers (larger float,
// larger image; -inf maps below every finite value; -0 and +0 map alike, as
// they compare equal).  NaN never reaches it.
__device__ __forceinline__ uint32_t ord_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value, index) maximum over the warp; ties go to the lower index.  The
// order is total, so every lane ends with the same winner.  Two warp-wide
// reductions (the largest value, then the smallest index holding it) and one
// shuffle of the winner's carried value; an index is lane + 32*j, so the
// winner's lane is its index mod 32.
__device__ __forceinline__ void warp_argmax(float& v, int& ix, float& carry) {
  const uint32_t k = ord_key(v);
  const uint32_t best = __reduce_max_sync(0xffffffffu, k);
  const uint32_t cand = (k == best) ? static_cast<uint32_t>(ix) : 0xffffffffu;
  const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
  carry = __shfl_sync(0xffffffffu, carry, static_cast<int>(win & 31u));
  v = __shfl_sync(0xffffffffu, v, static_cast<int>(win & 31u));
  ix = static_cast<int>(win);
}


// score -> select -> routing_weights for one token, by one warp.  Lane l
// holds experts l, l+32, ..., (NJ per lane).  Writes idx_out[0..K) and
// w_out[0..K).
template <int NJ, bool kShared>
__device__ void select_token(const float* lrow, const SelCfg& c, int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  float l[NJ], s[NJ], key[NJ], eb[NJ];
  // the logits and the expert bias are loaded together, before any scoring
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    l[j] = e < c.E ? (kShared ? lrow[e] : __ldcg(lrow + e)) : kNegInf;
    eb[j] = (c.expert_bias && e < c.E) ? __ldg(c.expert_bias + e) : 0.f;
  }
  // ---- score (fp32)
  if (c.score_fn == 0) {  // softmax
    float m = kNegInf;
#pragma unroll
    for (int j = 0; j < NJ; ++j) m = fmaxf(m, l[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      s[j] = (lane + 32 * j < c.E) ? expf(l[j] - m) : 0.f;
      sum += s[j];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
#pragma unroll
    for (int j = 0; j < NJ; ++j) s[j] = s[j] / sum;
  } else if (c.score_fn == 1) {  // sigmoid
#pragma unroll
    for (int j = 0; j < NJ; ++j) s[j] = (lane + 32 * j < c.E) ? 1.f / (1.f + expf(-l[j])) : 0.f;
  } else {  // sqrt(softplus)
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      s[j] = (lane + 32 * j < c.E) ? sqrtf(fmaxf(l[j], 0.f) + log1pf(expf(-fabsf(l[j])))) : 0.f;
  }
  // ---- selection key.  All three scores are strictly increasing in the
  // logit, so without an expert bias and without groups the selection is
  // made on the fp32 logits themselves (the exact order of the scores).
  // A NaN key becomes the lowest finite value, so every pick stays a valid
  // expert id (-inf marks only experts that may not be picked).
  const bool on_logits = (c.expert_bias == nullptr && c.n_group == 1);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    float v;
    if (e >= c.E) v = kNegInf;
    else if (on_logits) v = l[j];
    else v = c.expert_bias ? s[j] + eb[j] : s[j];
    key[j] = (v != v) ? -FLT_MAX : v;
  }
  // ---- group-limited select: keep the topk_group groups with the best sum
  // of their group_topn largest keys; the other experts become unselectable.
  if (c.n_group > 1) {
    const int gsz = c.E / c.n_group;
    float my_gs = kNegInf;
    for (int g = 0; g < c.n_group; ++g) {
      float tmp[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        tmp[j] = (e < c.E && e / gsz == g) ? key[j] : kNegInf;
      }
      float gsum = 0.f;
      for (int r = 0; r < c.group_topn; ++r) {
        float bv = kNegInf;
        int bj = -1;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          if (tmp[j] > bv) { bv = tmp[j]; bj = j; }
        int ix = bj >= 0 ? lane + 32 * bj : 0x7fffffff;
        float dummy = 0.f;
        warp_argmax(bv, ix, dummy);
        gsum = (r == 0) ? bv : gsum + bv;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          if (lane + 32 * j == ix) tmp[j] = kNegInf;
      }
      if (lane == g) my_gs = gsum;
    }
    uint32_t keep = 0;
    float gv = my_gs;
    for (int r = 0; r < c.topk_group; ++r) {
      float v = gv;
      int ix = lane < c.n_group ? lane : 0x7fffffff;
      float dummy = 0.f;
      warp_argmax(v, ix, dummy);
      keep |= 1u << ix;
      if (lane == ix) gv = kNegInf;
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < c.E && !((keep >> (e / gsz)) & 1u)) key[j] = kNegInf;
    }
  }
  // ---- K rounds of warp argmax; lane k keeps the k-th pick and its score.
  int my_e = -1;
  float my_s = 0.f;
  for (int k = 0; k < c.K; ++k) {
    float bv = kNegInf, bs = 0.f;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (key[j] > bv) { bv = key[j]; bj = j; bs = s[j]; }
    int ix = bj >= 0 ? lane + 32 * bj : 0x7fffffff;
    warp_argmax(bv, ix, bs);
    if (lane == k) { my_e = ix; my_s = bs; }
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (lane + 32 * j == ix) key[j] = kNegInf;
  }
  // ---- routing weights from the unshifted scores
  float sum = 0.f;
  for (int k = 0; k < c.K; ++k) sum += __shfl_sync(0xffffffffu, my_s, k);
  if (lane < c.K) {
    float wv = my_s;
    if (c.renorm) wv = wv / (sum + c.eps);
    wv = wv * c.scale;
    idx_out[lane] = my_e;
    w_out[lane] = wv;
  }
}

}  // namespace
}  // namespace moe
