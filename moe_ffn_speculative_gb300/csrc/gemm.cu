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
// Warp roles (224 threads): warp 0 issues the weight TMA loads, warp 1
// allocates TMEM and issues the MMAs, warp 2 gathers the token rows with
// cp.async into the 128-byte-swizzled B tile, warps 3..6 drain TMEM in the
// epilogue (SwiGLU for gate_up; routing weight and store for down).
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint16_t f2bf(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void record_failure(int32_t* status, volatile int* abort_flag, int32_t info) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) atomicExch(status + 1, info);
  *abort_flag = 1;
}

struct Seg {
  int expert, row_base, count, idim;
  int m, n, k0, len, kb, tile, n_cnt;
  long long tile_iter0;
};

// Walks one CTA's contiguous range [begin, end) of the concatenated k-block
// iterations, one (tile, k-range) segment at a time.
struct Sched {
  const GroupEntry* groups;
  int ngroups, phase, H, n_max, g;
  long long end, it;

  __device__ long long iter_of(int gi) const { return phase == 0 ? groups[gi].gu_iter : groups[gi].dn_iter; }

  __device__ void init(const GroupEntry* gs, int ng, int ph, int H_, int nmax, long long b, long long e) {
    groups = gs; ngroups = ng; phase = ph; H = H_; n_max = nmax; it = b; end = e; g = 0;
    if (b < e) {
      int lo = 0, hi = ng - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (iter_of(mid) <= b) lo = mid; else hi = mid - 1;
      }
      g = lo;
    }
  }

  __device__ bool next(Seg& s) {
    if (it >= end) return false;
    while (g + 1 < ngroups && iter_of(g + 1) <= it) ++g;
    const GroupEntry ge = groups[g];
    int mb, nb, kb;
    group_geometry(phase, ge.count, ge.idim, H, n_max, mb, nb, kb);
    const long long start = phase == 0 ? ge.gu_iter : ge.dn_iter;
    const long long local = it - start;
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
    it += len;
    return true;
  }
};

__device__ __forceinline__ long long cta_begin(long long c, long long total, long long grid) {
  return c * total / grid;
}
// The CTA whose iteration range holds iteration i.
__device__ __forceinline__ int cta_of(long long i, long long total, long long grid) {
  return static_cast<int>(((i + 1) * grid + total - 1) / total - 1);
}

// --------------------------------------------------------------------------
// epilogues of one 16-column chunk; a[i], b[i] = half-0 / half-1 accumulator
// of row r (TMEM lane) and token column j0 + i
// --------------------------------------------------------------------------
template <int PHASE>
__device__ __forceinline__ void finish_chunk(const GemmParams& p, const Seg& sg, int r, int j0, const float* a,
                                             const float* b) {
  if (PHASE == 0) {
    // SwiGLU: h = silu(gate) * up, with the clamp when a limit is set
    const int row = sg.m * kHalfRows + r;
    if (row >= sg.idim) return;
    // h is kept as a compensated pair hi + lo of bf16 (about 16 significant
    // bits): row r holds hi in [0, I_ld) and lo in [I_ld, 2*I_ld)
    uint16_t* hp = p.h + static_cast<size_t>(sg.row_base + sg.n * p.n_max) * (2 * p.I_ld) + row;
    const float lim = p.swiglu_limit;
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
        const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
        const float lo = hv - __bfloat162float(hi);
        hp[static_cast<size_t>(j) * (2 * p.I_ld)] = __bfloat16_as_ushort(hi);
        hp[static_cast<size_t>(j) * (2 * p.I_ld) + p.I_ld] = f2bf(lo);
      }
    }
  } else {
    // routing weight (or shared-expert gate) times the expert output
    const int row0 = sg.m * 2 * kHalfRows + r;
    const int row1 = row0 + kHalfRows;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int j = j0 + i;
      if (j < sg.n_cnt) {
        const int sr = sg.row_base + sg.n * p.n_max + j;
        float wt;
        int tok;
        if (sg.expert >= 0) {
          const int pr = __ldg(p.sorted_pair + sr);
          wt = __ldg(p.topk_w + pr);
          tok = pr / p.K;
        } else {
          tok = sr - p.TK;
          wt = p.sh_w ? __ldg(p.sh_w + tok) : 1.f;
        }
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

template <int PHASE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_routed, const __grid_constant__ CUtensorMap tm_shared,
                    const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = p.stages;
  constexpr int kBTiles = PHASE == 0 ? 1 : 2;  // down: B = h_hi and h_lo
  const uint32_t b_bytes = p.n_max * 128;
  const uint32_t stage_bytes = 2 * kTileBytesA + kBTiles * b_bytes;
  uint8_t* ctrl = smem + S * stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accf = empty + kMaxStages;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bcast = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_ok = reinterpret_cast<int*>(tmem_slot + 3);
  long long* rowoff = reinterpret_cast<long long*>(ctrl + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + 32);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *bcast = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_routed);
    tma_prefetch_desc(&tm_shared);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const GemmHeader hd = *p.header;
  const long long total = PHASE == 0 ? hd.gu_iters : hd.dn_iters;
  const long long grid = gridDim.x;
  const long long begin = cta_begin(blockIdx.x, total, grid);
  const long long end = cta_begin(blockIdx.x + 1, total, grid);
  Sched sc;
  sc.init(p.groups, hd.ngroups, PHASE, p.H, p.n_max, begin, end);
  Seg sg;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (weights)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      while (ok && sc.next(sg)) {
        const CUtensorMap* tm = sg.expert >= 0 ? &tm_routed : &tm_shared;
        const int plane = sg.expert >= 0 ? sg.expert : 0;
        for (int kk = 0; kk < sg.len; ++kk) {
          const int kx = (sg.k0 + kk) * kBlockK;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            record_failure(p.status, abort_flag, kInfoEmpty);
            ok = false;
            break;
          }
          uint8_t* a0 = smem + stage * stage_bytes;
          mbar_arrive_expect_tx(&full[stage], 2 * kTileBytesA);
          if (PHASE == 0) {
            tma_load_3d(a0, tm, &full[stage], kx, sg.m * kHalfRows, 2 * plane);
            tma_load_3d(a0 + kTileBytesA, tm, &full[stage], kx, sg.m * kHalfRows, 2 * plane + 1);
          } else {
            tma_load_3d(a0, tm, &full[stage], kx, sg.m * 2 * kHalfRows, plane);
            tma_load_3d(a0 + kTileBytesA, tm, &full[stage], kx, sg.m * 2 * kHalfRows + kHalfRows, plane);
          }
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA can exit
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000ll) {}
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, seg_i = 0;
      uint32_t phase = 0;
      bool ok = true;
      while (ok && sc.next(sg)) {
        const int buf = seg_i % p.nbuf;
        const uint32_t use = static_cast<uint32_t>(seg_i / p.nbuf);
        if (!mbar_wait(&acce[buf], (use & 1u) ^ 1u, abort_flag)) {
          record_failure(p.status, abort_flag, kInfoAccEmpty);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * 2 * p.n_max);
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.n_max);
        const int nmma = max(16, (sg.n_cnt + 15) & ~15);
        const uint32_t idesc = idesc_bf16(kHalfRows, nmma);
        for (int kk = 0; kk < sg.len; ++kk) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            record_failure(p.status, abort_flag, kInfoFull);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * stage_bytes);
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
              const uint64_t bl = sw128_desc(bb + b_bytes + ks * 32);
              mma_bf16(d0, ad0, bl, idesc, 1u);
              mma_bf16(d1, ad1, bl, idesc, 1u);
            }
          }
          mma_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&accf[buf]);
        ++seg_i;
      }
      // every MMA issued above has completed once `drain` flips
      mma_commit(drain);
      if (!mbar_wait(drain, 0, nullptr)) record_failure(p.status, abort_flag, kInfoDrain);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ token-row gather (B)
    int stage = 0, arr_stage = 0, pending = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int K = p.K, H = p.H;
    // copies kept in flight before arriving; below the stage count, so the
    // stage this warp waits to refill never depends on an arrival it holds
    const int lag = kGatherLag < S - 1 ? kGatherLag : S - 1;
    while (ok && sc.next(sg)) {
      const int nrows = max(16, (sg.n_cnt + 15) & ~15);
      const int kdim = PHASE == 0 ? H : sg.idim;
      __syncwarp();
      for (int j = lane; j < nrows; j += 32) {
        long long off = -1;
        if (j < sg.n_cnt) {
          const int r = sg.n * p.n_max + j;
          if (PHASE == 0) {
            const int tok = sg.expert >= 0 ? __ldg(p.sorted_pair + sg.row_base + r) / K : r;
            off = static_cast<long long>(tok) * H;
          } else {
            off = static_cast<long long>(sg.row_base + r) * (2 * p.I_ld);
          }
        }
        rowoff[j] = off;
      }
      __syncwarp();
      for (int kk = 0; kk < sg.len; ++kk) {
        const int kx = (sg.k0 + kk) * kBlockK;
        const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) record_failure(p.status, abort_flag, kInfoGatherEmpty);
          ok = false;
          break;
        }
        const uint32_t bbase = smem_u32(smem + stage * stage_bytes) + 2 * kTileBytesA;
        for (int q = lane; q < nrows * 8 * kBTiles; q += 32) {
          const int t = (kBTiles == 2 && q >= nrows * 8) ? 1 : 0;  // 0: x or h_hi, 1: h_lo
          const int qq = q - t * nrows * 8;
          const int j = qq >> 3, c = qq & 7;
          const long long off = rowoff[j];
          const int col = kx + c * 8;
          const bool valid = off >= 0 && col < kdim;
          const uint16_t* src = valid ? p.bsrc + off + t * p.I_ld + col : p.bsrc;
          cp_async_16(bbase + t * b_bytes + j * 128 + ((c ^ (j & 7)) << 4), src, valid ? 16u : 0u);
        }
        cp_async_commit();
        ++pending;
        if (pending > lag) {
          if (lag >= 2) cp_async_wait<2>(); else cp_async_wait<1>();
          fence_proxy_async();
          mbar_arrive(&full[arr_stage]);
          if (++arr_stage == S) arr_stage = 0;
          --pending;
        }
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    while (pending > 0) {
      mbar_arrive(&full[arr_stage]);
      if (++arr_stage == S) arr_stage = 0;
      --pending;
    }
  } else {
    // ------------------------------------------------ epilogue (warps 3..6)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // accumulator row = TMEM lane
    const bool leader = (warp == 3 && lane == 0);
    int seg_i = 0;
    while (sc.next(sg)) {
      const int buf = seg_i % p.nbuf;
      const uint32_t use = static_cast<uint32_t>(seg_i / p.nbuf);
      // one thread waits, the four warps leave or go on together
      if (leader) {
        const bool got = mbar_wait(&accf[buf], use & 1u, abort_flag);
        if (!got) record_failure(p.status, abort_flag, kInfoAccFull);
        *s_ok = got ? 1 : 0;
      }
      epi_sync();
      if (!*reinterpret_cast<volatile int*>(s_ok)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                            static_cast<uint32_t>(buf * 2 * p.n_max);
      const bool whole = (sg.k0 == 0 && sg.len == sg.kb);
      uint32_t ua[16], ub[16];
      float fa[16], fb[16];
      if (whole) {
        for (int j0 = 0; j0 < sg.n_cnt; j0 += 16) {
          tmem_ld16(tacc + j0, ua);
          tmem_ld16(tacc + p.n_max + j0, ub);
          tmem_ld_wait();
          u32_to_f32(ua, fa);
          u32_to_f32(ub, fb);
          finish_chunk<PHASE>(p, sg, r, j0, fa, fb);
        }
        tc_fence_before();
        mbar_arrive(&acce[buf]);
      } else {
        const int slot = (begin >= sg.tile_iter0) ? 0 : 1;
        float* mine = p.partials + static_cast<size_t>(blockIdx.x * 2 + slot) * 2 * p.n_max * 128;
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
        mbar_arrive(&acce[buf]);
        __threadfence();
        epi_sync();
        if (leader) {
          const int old = atomicAdd(p.tile_counters + sg.tile, sg.len);
          const int last = (old + sg.len == sg.kb);
          if (last) atomicExch(p.tile_counters + sg.tile, 0);
          *bcast = last;
        }
        epi_sync();
        const int last = *reinterpret_cast<volatile int*>(bcast);
        if (last) {
          __threadfence();
          const int c0 = cta_of(sg.tile_iter0, total, grid);
          const int c1 = cta_of(sg.tile_iter0 + sg.kb - 1, total, grid);
          for (int j0 = 0; j0 < sg.n_cnt; j0 += 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) { fa[i] = 0.f; fb[i] = 0.f; }
            for (int c = c0; c <= c1; ++c) {
              const long long bc = cta_begin(c, total, grid);
              if (bc == cta_begin(c + 1, total, grid)) continue;  // CTA with an empty range
              const int sl = (bc >= sg.tile_iter0) ? 0 : 1;
              const float* pp = p.partials + static_cast<size_t>(c * 2 + sl) * 2 * p.n_max * 128;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                if (j0 + i < sg.n_cnt) {
                  fa[i] += __ldcg(pp + static_cast<size_t>(j0 + i) * 128 + r);
                  fb[i] += __ldcg(pp + static_cast<size_t>(p.n_max + j0 + i) * 128 + r);
                }
              }
            }
            finish_chunk<PHASE>(p, sg, r, j0, fa, fb);
          }
        }
      }
      epi_sync();
      ++seg_i;
    }
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

}  // namespace

cudaError_t launch_gemm(int phase, const CUtensorMap& tm_routed, const CUtensorMap& tm_shared, const GemmParams& p,
                        int grid, size_t smem_bytes, cudaStream_t s) {
  if (phase == 0) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes));
    if (e != cudaSuccess) return e;
    moe_gemm_kernel<0><<<grid, kGemmThreads, smem_bytes, s>>>(tm_routed, tm_shared, p);
  } else {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes));
    if (e != cudaSuccess) return e;
    moe_gemm_kernel<1><<<grid, kGemmThreads, smem_bytes, s>>>(tm_routed, tm_shared, p);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* out_ws, const int32_t* pair_pos, int T, int K, int H, int has_shared,
                           uint16_t* y, cudaStream_t s) {
  dim3 grid(ceil_div(H, 4 * 256), T);
  combine_kernel<<<grid, 256, 0, s>>>(out_ws, pair_pos, T, K, H, has_shared, y);
  return cudaGetLastError();
}

}  // namespace moe
