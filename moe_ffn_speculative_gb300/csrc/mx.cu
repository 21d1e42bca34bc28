// Block-scaled expert GEMMs of the MoE-FFN layer: the routed experts' weights
// stay in the format of DeepSeek-V4.1's official draft checkpoint (SpecForge
// PR #1073 "MoE drafts: DeepSeek-V4.1's own DSpark draft", commit note on its
// export formats) -- FP4 routed experts (two e2m1 codes per byte along the
// input, the even input in the low nibble, one e8m0 scale per 32 inputs) or
// FP8 (e4m3 with one e8m0 scale per 32 x 32 block, the format of its other
// linears, which the shared expert takes) -- and are multiplied on the tensor
// cores by the block-scaled MMA (tcgen05.mma kind::mxf8f6f4.block_scale),
// which applies one scale of each operand per 32 products.  The products are
// those of the exactly dequantized weights, as the bf16 draft the import
// builds computes them.
//
// The other operand (x for gate_up, h for down) enters as a sum of e4m3
// pieces: piece p of a 32-input block is the block's remaining value rounded
// to e4m3 after dividing by 2^s_p, where s_p puts the block's largest
// remaining magnitude in [128, 256).  Three pieces carry a bf16 x (8
// significant bits) and four carry h (about 16 bits, as the bf16 path's hi+lo
// pair); each piece is one more MMA column of the token, with its own scales,
// and the epilogue adds a token's pieces.  The pieces are written once,
// straight into the shared-memory image of the B tile of every (token block,
// k-block) -- x's by the kernel's prologue, h's by the gate_up epilogue -- so
// a stage's token operand is two bulk copies that complete on the stage's
// barrier: no warp waits on the L2 round trip of scattered rows.
//
// Layout and schedule follow the stream-K bf16 kernel (gemm.cu): swap-AB
// tiles of 256 weight rows (two M=128 MMAs into two TMEM accumulators) by up
// to 24 tokens, the k-block iterations of all tiles of all touched experts
// cut into one contiguous span per SM, split tiles finished by the CTA that
// holds their first k-block, both GEMMs in one persistent launch.  A k-block
// is 128 inputs: the weight halves arrive by TMA in the MMA's K-major
// 128-byte-swizzled layout (FP4 codes through the tensor map type that
// spaces 16 codes over 16 bytes, the operand layout of 4-bit types), their
// scale chunks by a bulk copy, the token pieces and their scales by the
// gather warp; tcgen05.cp moves the stage's scale chunks to TMEM.
//
// Warp roles (224 threads): warp 0 issues the weight loads, warp 1 allocates
// TMEM and issues tcgen05.cp and the MMAs, warp 2 issues the token images'
// bulk copies, warps 3..6 drain TMEM; at the start warps 2..6 of every CTA
// cut their share of x into pieces and write them into the gate_up images.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kHalfBytes = kHalfRows * kMxK;  // one 128-row half of a k-block in shared memory: 16 KB
constexpr uint32_t kSfCols = 16;              // TMEM columns per stage for its scale chunks
constexpr int kQuantWarps = 5;                // warps 2..6 cut x into pieces
constexpr int kImgBlocks = 16;                // 32-input blocks of one token per prologue work item

struct Seg {
  int expert, row_base, count, idim;
  int m, n, k0, len, kb, tile, n_cnt;
  int ready_idx;
  int dense;  // token block over all groups: its image slots
  long long tile_iter0;
};

// Walks one CTA's range [begin, end) of the concatenated k-block iterations
// of one GEMM; a group entry outside the forward's bounds stops the walk.
struct Sched {
  const GroupEntry* groups;
  int ngroups, phase, H, n_max, g, rows, idim_max, mb0, n_dense;
  long long end, it;
  bool bad;

  __device__ long long iter_of(int gi) const { return phase == 0 ? groups[gi].gu_iter : groups[gi].dn_iter; }

  __device__ void init(const MxParams& p, int ng, int ph, long long b, long long e, int g0) {
    groups = p.groups; ngroups = ng; phase = ph; H = p.H; n_max = p.n_max; it = b; end = e; g = g0;
    rows = p.TK + p.T;
    idim_max = p.I_ld;
    mb0 = p.mb0;
    n_dense = p.n_dense;
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
    group_geometry(phase, ge.count, ge.idim, H, n_max, mb, nb, kb, kMxK);
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
    s.dense = ge.gu_tile / mb0 + s.n;
    if (ge.gu_tile % mb0 != 0 || s.dense >= n_dense) {
      bad = true;
      return false;
    }
    it += len;
    return true;
  }
};

__device__ __forceinline__ int cta_of(const long long* span, int grid, long long i) {
  int lo = 0, hi = grid - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (span[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// MMA columns of a segment: its tokens' pieces, token-major (column j*P + p),
// rounded up to the MMA's multiple of 16.
__device__ __forceinline__ int mx_cols(int phase, int n_cnt) {
  const int P = phase == 0 ? kMxPx : kMxPh;
  return max(16, (P * n_cnt + 15) & ~15);
}

struct Smem {
  uint8_t* base;
  uint32_t stage_bytes, b_bytes;
  int S;
  uint64_t *full, *empty, *accf, *acce, *drain;
  volatile int* abort_flag;
  int* s_ok;
  long long* span;
  float* col_w;
  int* col_tok;
};

// Image slot of (token block d, k-block kb): rows x 128 bytes, then the
// 512-byte scale chunk.
__device__ __forceinline__ uint8_t* img_slot(uint8_t* base, int rows, int kbs, int d, int kb) {
  return base + (static_cast<size_t>(d) * kbs + kb) * (static_cast<size_t>(rows) * 128 + kMxSfBytes);
}

// Byte of input i (0..127) in row c of a K-major 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int c, int i) {
  return static_cast<uint32_t>(c * 128 + ((((i >> 4) ^ (c & 7)) << 4) | (i & 15)));
}

// Byte of column c's scale of input chunk j in a 512-byte scale chunk.
__device__ __forceinline__ uint32_t sf_byte(int c, int j) {
  return static_cast<uint32_t>(16 * (c & 31) + 4 * (c >> 5) + j);
}

// offsets within a stage
__device__ __forceinline__ uint8_t* st_a(const Smem& sm, int s) { return sm.base + s * sm.stage_bytes; }
__device__ __forceinline__ uint8_t* st_b(const Smem& sm, int s) { return st_a(sm, s) + 2 * kHalfBytes; }
__device__ __forceinline__ uint8_t* st_sfa(const Smem& sm, int s) { return st_b(sm, s) + sm.b_bytes; }
__device__ __forceinline__ uint8_t* st_sfb(const Smem& sm, int s) { return st_sfa(sm, s) + 2 * kMxSfBytes; }

// Shared-memory descriptor of a 32-row x 16-byte scale chunk (no swizzle:
// 8-row core matrices 128 bytes apart), the source of tcgen05.cp.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// The 512-byte chunk (32 lines x 16 bytes; line r holds rows r, r+32, r+64,
// r+96, each with its four 32-input scales) copied to every 32-lane quarter
// of TMEM; the MMA reads row m's scale of input chunk j at column m / 32,
// byte j (the scale ID of the instruction).
__device__ __forceinline__ void sf_copy(uint32_t taddr, uint32_t saddr) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sf_desc(saddr)) : "memory");
}

// Instruction descriptor of kind::mxf8f6f4.block_scale: fp32 accumulator,
// A e2m1 (5) or e4m3 (0), B e4m3, both K-major, e8m0 scales, M = 128, N
// columns, scale IDs (the 32-input chunk within the 128-input k-block).
__device__ __forceinline__ uint32_t idesc_mx(bool a_fp4, int N, uint32_t chunk) {
  return (chunk << 4) | ((a_fp4 ? 5u : 0u) << 7) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(kHalfRows >> 4) << 24) | (chunk << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// ---------------------------------------------------------------- e4m3 pieces
// One piece of a 32-value block held one value per lane: the block's scale
// exponent e (its largest remaining magnitude over 2^e in [128, 256); 0 for
// an all-zero block), the value's e4m3 code at that scale, and the remainder
// for the next piece.
__device__ __forceinline__ uint8_t cut_piece(float& r, int& e_out) {
  // the block's largest magnitude in one warp reduction: the bits of a
  // non-negative float order as the unsigned integers they spell
  const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(r))));
  int e = 0;
  if (m > 0.f) {
    int k;
    frexpf(m, &k);  // m in [2^(k-1), 2^k)
    e = max(-127, min(127, k - 8));
  }
  const float q = ldexpf(r, -e);  // exact: a power-of-two scaling
  const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(c, __NV_E4M3);
  r -= ldexpf(__half2float(__half(hr)), e);
  e_out = e;
  return static_cast<uint8_t>(c);
}

// Warps 2..6 of every CTA: the CTA's share of (token, 16 blocks of 32
// inputs) items.  Each block of x is cut into kMxPx pieces once and written
// into the gate_up image of every token block that holds the token (its K
// routed experts' and the shared expert's), as row j*kMxPx + p with its
// scale; then one arrival per warp on the grid-wide counter.
__device__ void build_gu_images(const MxParams& p, int qw, int ngroups) {
  const int lane = threadIdx.x & 31;
  const int hb = p.H / 32;
  const int per_tok = ceil_div(hb, kImgBlocks);
  const long long items = static_cast<long long>(p.T) * per_tok;
  const long long w0 = static_cast<long long>(blockIdx.x) * kQuantWarps + qw;
  const long long nw = static_cast<long long>(gridDim.x) * kQuantWarps;
  const int nd = p.K + (p.Is > 0 ? 1 : 0);  // destinations of a token (<= 33)
  for (long long it = w0; it < items; it += nw) {
    const int t = static_cast<int>(it / per_tok), jb0 = static_cast<int>(it % per_tok) * kImgBlocks;
    // destination q of this token (q < K: its slot-q expert; q == K: the
    // shared expert): token block d, row group j; lane q holds q, lane 0
    // also q = 32
    int dq[2] = {-1, -1}, jq[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = lane + 32 * h;
      if (q < nd) {
        int d = -1, j = 0;
        if (q < p.K) {
          const int pr = t * p.K + q;
          const int e = __ldg(p.idx + pr);
          if (static_cast<unsigned>(e) < static_cast<unsigned>(p.E)) {
            const int pos = __ldg(p.pair_pos + pr) - __ldg(p.offsets + e);
            d = __ldg(p.e2d + e) + pos / p.n_max;
            j = pos % p.n_max;
          }
        } else {
          const GroupEntry& sh = p.groups[ngroups - 1];
          d = sh.gu_tile / p.mb0 + t / p.n_max;
          j = t % p.n_max;
        }
        if (d >= 0 && d < p.n_dense && j >= 0) { dq[h] = d; jq[h] = j; }
      }
    }
    // the item's inputs at once (one L2 round trip, not one per block);
    // then one k-block (four blocks) at a time: the four blocks' pieces are
    // cut side by side, so their warp reductions overlap, and each
    // destination is visited once per k-block (a rolled outer loop keeps
    // the code small for the warps that share the SM's instruction cache)
    uint16_t xv[kImgBlocks];
#pragma unroll
    for (int b = 0; b < kImgBlocks; ++b)
      xv[b] = jb0 + b < hb ? __ldg(p.x + static_cast<size_t>(t) * p.H + (jb0 + b) * 32 + lane) : 0;
#pragma unroll 1
    for (int b0 = 0; b0 < kImgBlocks && jb0 + b0 < hb; b0 += 4) {
      const int kb = (jb0 + b0) >> 2;  // H is a multiple of 128: the k-block's four blocks are all here
      float r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) r[u] = __bfloat162float(__ushort_as_bfloat16(xv[b0 + u]));
      uint8_t c[kMxPx][4];
      uint32_t sfw[kMxPx];  // the four blocks' scale bytes of each piece, block u in byte u
#pragma unroll
      for (int pc = 0; pc < kMxPx; ++pc) {
        sfw[pc] = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          int e;
          c[pc][u] = cut_piece(r[u], e);
          sfw[pc] |= static_cast<uint32_t>(127 + e) << (8 * u);
        }
      }
      for (int q = 0; q < nd; ++q) {
        const int d = __shfl_sync(0xffffffffu, q < 32 ? dq[0] : dq[1], q & 31);
        const int j = __shfl_sync(0xffffffffu, q < 32 ? jq[0] : jq[1], q & 31);
        if (d < 0) continue;  // warp-uniform
        uint8_t* sl = img_slot(p.img_gu, p.img_gu_rows, p.kb_gu, d, kb);
#pragma unroll
        for (int pc = 0; pc < kMxPx; ++pc) {
          const int row = j * kMxPx + pc;
#pragma unroll
          for (int u = 0; u < 4; ++u) sl[swz(row, u * 32 + lane)] = c[pc][u];
          // the row's four scale bytes are adjacent: one aligned word
          if (lane == 0)
            *reinterpret_cast<uint32_t*>(sl + p.img_gu_rows * 128 + sf_byte(row, 0)) = sfw[pc];
        }
      }
    }
  }
  // the images are read by bulk copies (the async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicAdd(p.img_ready, 1);
}

// ---------------------------------------------------------------- TMA producer (weights)
struct WeightCursor {
  Sched sc0, sc1;
  Seg sg;
  int ph, kk;
  bool valid;

  __device__ void init(const MxParams& p, int ngroups, const long long (&b)[2], const long long (&e)[2],
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
};

template <bool kFp4>
__device__ bool produce(const Smem& sm, const MxParams& p, int ngroups, const long long (&b)[2],
                        const long long (&e)[2], const int (&g)[2], const CUtensorMap* tm_gu,
                        const CUtensorMap* tm_gu_sh, const CUtensorMap* tm_dn, const CUtensorMap* tm_dn_sh) {
  const uint64_t pol = l2_evict_first_policy();
  if (!wait_start_gate(p.status)) {
    record_failure(p.status, sm.abort_flag, kInfoHold);
    return false;
  }
  WeightCursor ld;
  ld.init(p, ngroups, b, e, g);
  Ring ring;
  while (ld.valid) {
    if (!mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag)) {
      record_failure(p.status, sm.abort_flag, kInfoEmpty);
      return false;
    }
    const Seg& sg = ld.sg;
    const bool routed = sg.expert >= 0;
    // FP4 codes count their packed bytes (64 per row), FP8 128 per row
    const uint32_t abytes = (kFp4 && routed) ? kHalfBytes / 2 : kHalfBytes;
    uint64_t* bar = &sm.full[ring.stage];
    mbar_arrive_expect_tx(bar, 2 * abytes + 2 * kMxSfBytes);
    const int plane = routed ? sg.expert : 0;
    const int kb = sg.k0 + ld.kk;
    const CUtensorMap* tm = ld.ph == 0 ? (routed ? tm_gu : tm_gu_sh) : (routed ? tm_dn : tm_dn_sh);
    uint8_t* a = st_a(sm, ring.stage);
    for (int h = 0; h < 2; ++h) {
      int c1, c2;
      if (ld.ph == 0) { c1 = sg.m * kHalfRows; c2 = 2 * plane + h; }
      else            { c1 = sg.m * 2 * kHalfRows + h * kHalfRows; c2 = plane; }
      tma_load_3d_hint(a + h * kHalfBytes, tm, bar, kb * kMxK, c1, c2, pol);
    }
    // the weights' scale chunks are streamed once too: evict-first, like the
    // codes, so that they do not push the router's and the next layer's
    // operands out of L2
    bulk_load_hint(st_sfa(sm, ring.stage),
                   p.scales + mx_scale_offset(p.E, p.H, p.I, p.Is, ld.ph, sg.expert, sg.m, kb), 2 * kMxSfBytes,
                   bar, pol);
    ld.step();
    ring.next(sm.S);
  }
  if (ld.sc0.bad || ld.sc1.bad) {
    record_failure(p.status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  // every weight load of this CTA is issued: its share of the next layer's
  // routing-independent bytes goes to L2 while the layer's tail runs
  prefetch_share_l2(p.pf);
  return true;
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <int PHASE, bool kFp4>
__device__ bool issue_mma(const Smem& sm, const MxParams& p, int ngroups, long long begin, long long end, int g0,
                          uint32_t tmem_base, int nbuf, int n_eff_cols, uint32_t sf_base, Ring& ring, int& seg_i) {
  Sched sc;
  sc.init(p, ngroups, PHASE, begin, end, g0);
  Seg sg;
  while (sc.next(sg)) {
    const int buf = seg_i % nbuf;
    const uint32_t use = static_cast<uint32_t>(seg_i / nbuf);
    if (!mbar_wait(&sm.acce[buf], (use & 1u) ^ 1u, sm.abort_flag)) {
      record_failure(p.status, sm.abort_flag, kInfoAccEmpty);
      return false;
    }
    tc_fence_after();
    const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * 2 * n_eff_cols);
    const uint32_t d1 = d0 + static_cast<uint32_t>(n_eff_cols);
    const int N = mx_cols(PHASE, sg.n_cnt);
    const bool a_fp4 = kFp4 && sg.expert >= 0;
    for (int kk = 0; kk < sg.len; ++kk) {
      if (!mbar_wait(&sm.full[ring.stage], ring.phase, sm.abort_flag)) {
        record_failure(p.status, sm.abort_flag, kInfoFull);
        return false;
      }
      tc_fence_after();
      const uint32_t sf = tmem_base + sf_base + static_cast<uint32_t>(ring.stage) * kSfCols;
      const uint32_t sfa = smem_u32(st_sfa(sm, ring.stage));
      sf_copy(sf, sfa);                        // weight half 0
      sf_copy(sf + 4, sfa + kMxSfBytes);       // weight half 1
      sf_copy(sf + 8, smem_u32(st_sfb(sm, ring.stage)));  // token pieces
      const uint32_t a0 = smem_u32(st_a(sm, ring.stage)), a1 = a0 + kHalfBytes;
      const uint32_t bb = smem_u32(st_b(sm, ring.stage));
#pragma unroll
      for (int ks = 0; ks < kMxK / 32; ++ks) {
        const uint32_t acc = (kk > 0 || ks > 0) ? 1u : 0u;
        const uint32_t idesc = idesc_mx(a_fp4, N, static_cast<uint32_t>(ks));
        const uint64_t bd = sw128_desc(bb + ks * 32);
        mma_mx(d0, sw128_desc(a0 + ks * 32), bd, idesc, sf, sf + 8, acc);
        mma_mx(d1, sw128_desc(a1 + ks * 32), bd, idesc, sf + 4, sf + 8, acc);
      }
      mma_commit(&sm.empty[ring.stage]);
      ring.next(sm.S);
    }
    mma_commit(&sm.accf[buf]);
    ++seg_i;
  }
  if (sc.bad) {
    record_failure(p.status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- token images (B), lane 0 of warp 2
// Every k-block's B tile and its scale chunk are two bulk copies of the
// (token block, k-block) image, counted on the stage's barrier.
template <int PHASE>
__device__ bool gather(const Smem& sm, const MxParams& p, int ngroups, long long begin, long long end, int g0,
                       Ring& ring) {
  if (PHASE == 0) {
    // every CTA's share of the gate_up images is written before the first copy
    const int target = kQuantWarps * static_cast<int>(gridDim.x);
    const long long t0 = clock64();
    while (ld_acquire_gpu(p.img_ready) < target) {
      if (*sm.abort_flag || clock64() - t0 > kWaitLimitCycles) {
        record_failure(p.status, sm.abort_flag, kInfoReady);
        return false;
      }
      __nanosleep(64);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  Sched sc;
  sc.init(p, ngroups, PHASE, begin, end, g0);
  uint8_t* const base = PHASE == 0 ? p.img_gu : p.img_dn;
  const int rows = PHASE == 0 ? p.img_gu_rows : p.img_dn_rows;
  const int kbs = PHASE == 0 ? p.kb_gu : p.kb_dn;
  Seg sg;
  while (sc.next(sg)) {
    const int N = mx_cols(PHASE, sg.n_cnt);
    if (PHASE == 1) {
      // the down images of this token block are complete once every gate_up
      // tile of it has signalled
      const int target = ceil_div(sg.idim, kHalfRows);
      const int32_t* rp = p.ready + sg.ready_idx;
      if (ld_acquire_gpu(rp) < target) {
        const long long t0 = clock64();
        while (ld_acquire_gpu(rp) < target) {
          if (*sm.abort_flag || clock64() - t0 > kWaitLimitCycles) {
            record_failure(p.status, sm.abort_flag, kInfoReady);
            return false;
          }
          __nanosleep(64);
        }
      }
      // written by other CTAs' generic stores, read by bulk copies below
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    for (int kk = 0; kk < sg.len; ++kk) {
      if (!mbar_wait(&sm.empty[ring.stage], ring.phase ^ 1u, sm.abort_flag)) {
        record_failure(p.status, sm.abort_flag, kInfoGatherEmpty);
        return false;
      }
      const uint8_t* sl = img_slot(base, rows, kbs, sg.dense, sg.k0 + kk);
      uint64_t* bar = &sm.full[ring.stage];
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(N) * 128u + kMxSfBytes);
      bulk_load(st_b(sm, ring.stage), sl, static_cast<uint32_t>(N) * 128u, bar);
      bulk_load(st_sfb(sm, ring.stage), sl + static_cast<size_t>(rows) * 128, kMxSfBytes, bar);
      ring.next(sm.S);
    }
  }
  if (sc.bad) {
    record_failure(p.status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- epilogue (4 warps)
// Token j's accumulator of one half: the sum of its P piece columns.
template <int P>
__device__ __forceinline__ void load_tokens4(uint32_t tacc, int j0, int n_cnt, float (&v)[4]) {
  uint32_t u[4][P];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int q = 0; q < P; ++q)  // j0 and n_cnt are warp-uniform: the loads stay .sync.aligned
      u[t][q] = j0 + t < n_cnt ? tmem_ld1(tacc + static_cast<uint32_t>((j0 + t) * P + q)) : 0u;
  tmem_ld_wait();
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < P; ++q) s += __uint_as_float(u[t][q]);
    v[t] = s;
  }
}

// gate_up: SwiGLU (with the clamp) into h's pieces, written into the down
// image of k-block m (the tile's 128 rows of the intermediate dimension are
// the down GEMM's k-block m); every lane of a warp holds one of 32
// consecutive rows, i.e. one 32-input chunk (the warp's quarter) of h for
// each token.
__device__ __forceinline__ void finish_gu(const MxParams& p, const Seg& sg, int r, int j0, const float (&a)[4],
                                          const float (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const float lim = p.swiglu_limit;
  uint8_t* sl = img_slot(p.img_dn, p.img_dn_rows, p.kb_dn, sg.dense, sg.m);
  // the four tokens' h values, cut into pieces side by side so that their
  // warp reductions overlap (columns past the tile's tokens cut zeros and
  // store nothing; the count is uniform over the warp)
  float rem[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    float g = a[t], u = b[t];
    if (lim > 0.f) {
      g = fminf(g, lim);
      u = fminf(fmaxf(u, -lim), lim);
    }
    rem[t] = j0 + t < sg.n_cnt ? g / (1.f + expf(-g)) * u : 0.f;
  }
#pragma unroll
  for (int q = 0; q < kMxPh; ++q) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      int e;
      const uint8_t c = cut_piece(rem[t], e);
      if (j0 + t < sg.n_cnt) {
        const int row = (j0 + t) * kMxPh + q;
        sl[swz(row, r)] = c;
        if (lane == 0) sl[p.img_dn_rows * 128 + sf_byte(row, r >> 5)] = static_cast<uint8_t>(127 + e);
      }
    }
  }
}

// down: routing weight (or shared-expert gate) times the expert output
__device__ __forceinline__ void finish_dn(const MxParams& p, const Seg& sg, int r, int j0, const float (&a)[4],
                                          const float (&b)[4], const float* col_w, const int* col_tok) {
  const int row0 = sg.m * 2 * kHalfRows + r;
  const int row1 = row0 + kHalfRows;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int j = j0 + t;
    if (j >= sg.n_cnt) break;
    const int sr = sg.row_base + sg.n * p.n_max + j;
    const float wt = col_w[j];
    if (p.direct_y) {
      uint16_t* yr = p.y + static_cast<size_t>(col_tok[j]) * p.H;
      if (row0 < p.H) yr[row0] = f2bf(wt * a[t]);
      if (row1 < p.H) yr[row1] = f2bf(wt * b[t]);
    } else {
      float* orow = p.out_ws + static_cast<size_t>(sr) * p.H;
      if (row0 < p.H) __stcg(orow + row0, wt * a[t]);
      if (row1 < p.H) __stcg(orow + row1, wt * b[t]);
    }
  }
}

template <int PHASE>
__device__ bool epilogue(const Smem& sm, const MxParams& p, int ngroups, long long begin, long long end, int g0,
                         uint32_t tmem_base, int nbuf, int n_eff_cols, int& seg_i, int32_t* tile_counters) {
  constexpr int P = PHASE == 0 ? kMxPx : kMxPh;
  Sched sc;
  sc.init(p, ngroups, PHASE, begin, end, g0);
  const long long* span = sm.span + PHASE * (gridDim.x + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const bool leader = (warp == 3 && lane == 0);
  const int grid = gridDim.x;
  Seg sg;
  while (sc.next(sg)) {
    const int buf = seg_i % nbuf;
    const uint32_t use = static_cast<uint32_t>(seg_i / nbuf);
    if (PHASE == 1) {
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
    if (leader) {
      const bool got = mbar_wait(&sm.accf[buf], use & 1u, sm.abort_flag);
      if (!got) record_failure(p.status, sm.abort_flag, kInfoAccFull);
      *sm.s_ok = got ? 1 : 0;
    }
    epi_sync();
    if (!*reinterpret_cast<volatile int*>(sm.s_ok)) return false;
    tc_fence_after();
    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                          static_cast<uint32_t>(buf * 2 * n_eff_cols);
    const bool whole = (sg.k0 == 0 && sg.len == sg.kb);
    bool done = false;
    float fa[4], fb[4];
    if (whole) {
      for (int j0 = 0; j0 < sg.n_cnt; j0 += 4) {
        load_tokens4<P>(tacc, j0, sg.n_cnt, fa);
        load_tokens4<P>(tacc + n_eff_cols, j0, sg.n_cnt, fb);
        if (PHASE == 0) finish_gu(p, sg, r, j0, fa, fb);
        else finish_dn(p, sg, r, j0, fa, fb, sm.col_w, sm.col_tok);
      }
      tc_fence_before();
      mbar_arrive(&sm.acce[buf]);
      done = true;
    } else if (sg.k0 > 0) {
      // a later part of a split tile: its token sums go to this CTA's
      // partial slot for the CTA holding the tile's first k-block
      float* mine = p.partials + static_cast<size_t>(blockIdx.x * 4 + PHASE * 2) * 2 * p.n_max * 128;
      for (int j0 = 0; j0 < sg.n_cnt; j0 += 4) {
        load_tokens4<P>(tacc, j0, sg.n_cnt, fa);
        load_tokens4<P>(tacc + n_eff_cols, j0, sg.n_cnt, fb);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (j0 + t < sg.n_cnt) {
            __stcg(mine + static_cast<size_t>(j0 + t) * 128 + r, fa[t]);
            __stcg(mine + static_cast<size_t>(p.n_max + j0 + t) * 128 + r, fb[t]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.acce[buf]);
      __threadfence();
      epi_sync();
      if (leader) atomicAdd(tile_counters + sg.tile, sg.len);
    } else {
      // the first part of a split tile: wait (bounded) for the later parts'
      // partials, then add them in CTA order and finish the tile
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
        else record_failure(p.status, sm.abort_flag, kInfoFixup);
        *sm.s_ok = got ? 1 : 0;
      }
      epi_sync();
      if (!*reinterpret_cast<volatile int*>(sm.s_ok)) return false;
      __threadfence();
      const int c1 = cta_of(span, grid, sg.tile_iter0 + sg.kb - 1);
      for (int j0 = 0; j0 < sg.n_cnt; j0 += 4) {
        load_tokens4<P>(tacc, j0, sg.n_cnt, fa);
        load_tokens4<P>(tacc + n_eff_cols, j0, sg.n_cnt, fb);
        for (int c = blockIdx.x + 1; c <= c1; ++c) {
          if (span[c] == span[c + 1]) continue;
          const float* pp = p.partials + static_cast<size_t>(c * 4 + PHASE * 2) * 2 * p.n_max * 128;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (j0 + t < sg.n_cnt) {
              fa[t] += __ldcg(pp + static_cast<size_t>(j0 + t) * 128 + r);
              fb[t] += __ldcg(pp + static_cast<size_t>(p.n_max + j0 + t) * 128 + r);
            }
          }
        }
        if (PHASE == 0) finish_gu(p, sg, r, j0, fa, fb);
        else finish_dn(p, sg, r, j0, fa, fb, sm.col_w, sm.col_tok);
      }
      tc_fence_before();
      mbar_arrive(&sm.acce[buf]);
      done = true;
    }
    if (PHASE == 0 && done) {
      // this tile's k-block of the down images is written: count it towards
      // its token block, whose images the down GEMM reads by bulk copies
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __threadfence();
      epi_sync();
      if (leader) atomicAdd(p.ready + sg.ready_idx, 1);
    }
    epi_sync();
    ++seg_i;
  }
  if (sc.bad) {
    if (leader) record_failure(p.status, sm.abort_flag, kInfoWorkList);
    return false;
  }
  return true;
}

template <bool kFp4>
__global__ void __launch_bounds__(kMxThreads, 1)
    moe_mx_kernel(const __grid_constant__ CUtensorMap tm_gu, const __grid_constant__ CUtensorMap tm_gu_sh,
                  const __grid_constant__ CUtensorMap tm_dn, const __grid_constant__ CUtensorMap tm_dn_sh,
                  const __grid_constant__ MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  uint8_t* ctrl = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  sm.base = ctrl + kCtrlBytes;
  sm.full = reinterpret_cast<uint64_t*>(ctrl);
  sm.empty = sm.full + kMaxStages;
  sm.accf = sm.empty + kMaxStages;
  sm.acce = sm.accf + 2;
  sm.drain = sm.acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.drain + 1);
  sm.abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  sm.s_ok = reinterpret_cast<int*>(tmem_slot + 3);
  sm.span = reinterpret_cast<long long*>(ctrl + kCtrlSpans);
  sm.col_w = reinterpret_cast<float*>(ctrl + kCtrlCols);
  sm.col_tok = reinterpret_cast<int*>(ctrl + kCtrlCols + 4 * 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&sm.full[s], 2);  // the weight loads and the token image copies
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.accf[b], 1);
      mbar_init(&sm.acce[b], 128);
    }
    mbar_init(sm.drain, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_gu);
    tma_prefetch_desc(&tm_gu_sh);
    tma_prefetch_desc(&tm_dn);
    tma_prefetch_desc(&tm_dn_sh);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < 2 * (static_cast<int>(gridDim.x) + 1); i += blockDim.x) sm.span[i] = p.spans[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // the router's work list, checked against the host's bounds (uniform)
  const GemmHeader hd = *p.header;
  const int G1 = gridDim.x + 1;
  const long long bs[2] = {sm.span[blockIdx.x], sm.span[G1 + blockIdx.x]};
  const long long es[2] = {sm.span[blockIdx.x + 1], sm.span[G1 + blockIdx.x + 1]};
  const int gs[2] = {p.span_groups[blockIdx.x], p.span_groups[G1 + blockIdx.x]};
  const bool list_ok = hd.ngroups >= 0 && hd.ngroups <= p.g_max && hd.gu_tiles >= 0 &&
                       hd.gu_tiles <= p.max_gu_tiles && hd.dn_tiles >= 0 && hd.dn_tiles <= p.max_dn_tiles &&
                       hd.n_eff >= 8 && hd.n_eff <= p.n_max && (hd.n_eff & 7) == 0 && hd.gu_iters >= 0 &&
                       hd.gu_iters <= p.max_gu_iters && hd.dn_iters >= 0 && hd.dn_iters <= p.max_dn_iters &&
                       bs[0] >= 0 && bs[0] <= es[0] && es[0] <= hd.gu_iters && bs[1] >= 0 && bs[1] <= es[1] &&
                       es[1] <= hd.dn_iters && gs[0] >= 0 && gs[0] <= hd.ngroups && gs[1] >= 0 &&
                       gs[1] <= hd.ngroups;
  if (!list_ok && threadIdx.x == 0) record_failure(p.status, sm.abort_flag, kInfoWorkList);
  const int ng = hd.ngroups;
  // stages sized for the widest token tile of this forward: kMxPh pieces of
  // n_eff tokens as B rows of 128 bytes; TMEM holds two accumulator buffers
  // (2 x 2 halves x <= 96 columns), then every stage's scale chunks
  const int n_eff_cols = (kMxPh * (list_ok ? hd.n_eff : 16) + 15) & ~15;
  sm.b_bytes = static_cast<uint32_t>(n_eff_cols) * 128u;
  sm.stage_bytes = (2 * kHalfBytes + sm.b_bytes + 3 * kMxSfBytes + 1023u) & ~1023u;
  sm.S = min(kMaxStages, p.stage_space / static_cast<int>(sm.stage_bytes));
  const int nbuf = 2;
  const uint32_t sf_base = static_cast<uint32_t>(nbuf * 2 * n_eff_cols);

  if (!list_ok) {
    // nothing issued: every thread goes straight to the teardown
  } else if (warp == 0) {
    if (lane == 0) {
      const bool ok = produce<kFp4>(sm, p, ng, bs, es, gs, &tm_gu, &tm_gu_sh, &tm_dn, &tm_dn_sh);
      if (!ok) {
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000ll) {}
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      Ring ring;
      int seg_i = 0;
      if (issue_mma<0, kFp4>(sm, p, ng, bs[0], es[0], gs[0], tmem_base, nbuf, n_eff_cols, sf_base, ring, seg_i))
        issue_mma<1, kFp4>(sm, p, ng, bs[1], es[1], gs[1], tmem_base, nbuf, n_eff_cols, sf_base, ring, seg_i);
      mma_commit(sm.drain);
      if (!mbar_wait(sm.drain, 0, nullptr)) record_failure(p.status, sm.abort_flag, kInfoDrain);
    }
  } else if (warp == 2) {
    build_gu_images(p, 0, ng);
    if (lane == 0) {
      Ring ring;
      if (gather<0>(sm, p, ng, bs[0], es[0], gs[0], ring)) gather<1>(sm, p, ng, bs[1], es[1], gs[1], ring);
    }
  } else {
    build_gu_images(p, warp - 2, ng);
    int seg_i = 0;
    if (epilogue<0>(sm, p, ng, bs[0], es[0], gs[0], tmem_base, nbuf, n_eff_cols, seg_i, p.tile_counters_gu))
      epilogue<1>(sm, p, ng, bs[1], es[1], gs[1], tmem_base, nbuf, n_eff_cols, seg_i, p.tile_counters_dn);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// Weight scales -> the chunks the MMA reads: for every (group, 256-row tile,
// 128-input k-block) the two 128-row halves, each 512 bytes with byte
// 16*(r%32) + 4*(r/32) + j the scale of row r, input chunk j.  FP4 scales
// [.., rows, K/32] give each row its own; FP8 scales [.., rows/32, K/32]
// (32 x 32 blocks) repeat for the block's 32 rows.  Rows past the matrix
// take scale 1 (their weights load as zero).
__global__ void __launch_bounds__(256) mx_scales_kernel(int routed_fp4, const uint8_t* __restrict__ gu_s,
                                                        const uint8_t* __restrict__ dn_s, int E, int H, int I,
                                                        const uint8_t* __restrict__ sh_gu_s,
                                                        const uint8_t* __restrict__ sh_dn_s, int Is,
                                                        uint8_t* __restrict__ out) {
  // one thread per (block of 1 KB, half, row r): 4 bytes
  const int mb0 = ceil_div(I, kHalfRows), kb0 = H / kMxK, mb1 = ceil_div(H, 2 * kHalfRows), kb1 = I / kMxK;
  const long long n_rgu = static_cast<long long>(E) * mb0 * kb0, n_rdn = static_cast<long long>(E) * mb1 * kb1;
  const long long n_sgu = Is > 0 ? static_cast<long long>(ceil_div(Is, kHalfRows)) * kb0 : 0;
  const long long n_sdn = Is > 0 ? static_cast<long long>(mb1) * (Is / kMxK) : 0;
  const long long nblk = n_rgu + n_rdn + n_sgu + n_sdn;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < nblk * 256; i += static_cast<long long>(gridDim.x) * 256) {
    const long long blk = i / 256;
    const int h = static_cast<int>((i / kHalfRows) % 2), r = static_cast<int>(i % kHalfRows);
    long long b = blk;
    int phase, e = -1, m, kb;
    bool fp4;
    if (b < n_rgu) {
      phase = 0; fp4 = routed_fp4 != 0;
      e = static_cast<int>(b / (static_cast<long long>(mb0) * kb0)); b %= static_cast<long long>(mb0) * kb0;
      m = static_cast<int>(b / kb0); kb = static_cast<int>(b % kb0);
    } else if ((b -= n_rgu) < n_rdn) {
      phase = 1; fp4 = routed_fp4 != 0;
      e = static_cast<int>(b / (static_cast<long long>(mb1) * kb1)); b %= static_cast<long long>(mb1) * kb1;
      m = static_cast<int>(b / kb1); kb = static_cast<int>(b % kb1);
    } else if ((b -= n_rdn) < n_sgu) {
      phase = 0; fp4 = false;
      m = static_cast<int>(b / kb0); kb = static_cast<int>(b % kb0);
    } else {
      b -= n_sgu;
      phase = 1; fp4 = false;
      m = static_cast<int>(b / (Is / kMxK)); kb = static_cast<int>(b % (Is / kMxK));
    }
    const int idim = e >= 0 ? I : Is;
    const int kdim = phase == 0 ? H : idim;  // inputs per weight row
    int row, nrows;
    if (phase == 0) { row = h * idim + m * kHalfRows + r; nrows = 2 * idim; }
    else            { row = m * 2 * kHalfRows + h * kHalfRows + r; nrows = H; }
    const bool in = phase == 0 ? (m * kHalfRows + r < idim) : (row < H);
    uint32_t v = 0x7F7F7F7Fu;
    if (in) {
      const uint8_t* src;
      if (e >= 0) src = phase == 0 ? gu_s : dn_s;
      else src = phase == 0 ? sh_gu_s : sh_dn_s;
      const size_t mat = e >= 0 ? static_cast<size_t>(e) : 0;
      v = 0;
      for (int j = 0; j < 4; ++j) {
        const int c = kb * 4 + j;  // 32-input chunk along the row
        uint8_t sv;
        if (fp4) sv = src[(mat * nrows + row) * static_cast<size_t>(kdim / 32) + c];
        else sv = src[(mat * ceil_div(nrows, 32) + row / 32) * static_cast<size_t>(kdim / 32) + c];
        v |= static_cast<uint32_t>(sv) << (8 * j);
      }
    }
    uint8_t* dst = out + blk * 1024 + h * kMxSfBytes + 16 * (r % 32) + 4 * (r / 32);
    *reinterpret_cast<uint32_t*>(dst) = v;
  }
}

}  // namespace

cudaError_t launch_mx(const CUtensorMap& tm_gu, const CUtensorMap& tm_gu_sh, const CUtensorMap& tm_dn,
                      const CUtensorMap& tm_dn_sh, const MxParams& p, int grid, size_t smem_bytes, cudaStream_t s) {
  auto kern = p.routed_fp4 ? moe_mx_kernel<true> : moe_mx_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMxThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_gu, tm_gu_sh, tm_dn, tm_dn_sh, p);
}

cudaError_t launch_mx_scales(int routed_fp4, const uint8_t* gu_s, const uint8_t* dn_s, int E, int H, int I,
                             const uint8_t* sh_gu_s, const uint8_t* sh_dn_s, int Is, uint8_t* out, cudaStream_t s) {
  mx_scales_kernel<<<4 * 152, 256, 0, s>>>(routed_fp4, gu_s, dn_s, E, H, I, sh_gu_s, sh_dn_s, Is, out);
  return cudaGetLastError();
}

}  // namespace moe
