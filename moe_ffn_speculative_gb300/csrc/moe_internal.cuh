// Internal declarations shared by the kernels and the host layer of
// libmoe_gb300.so: work-list structures, launch parameter blocks and the
// inline-PTX wrappers for sm_103a (mbarrier, TMA, cp.async, tcgen05/TMEM).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"
#ifdef __CUDACC__
#include <cuda_bf16.h>
#endif

namespace moe {

// ----------------------------------------------------------------------------
// status word (first 8 bytes of every workspace): {code, info}
// ----------------------------------------------------------------------------
enum : int32_t { kStatusTimeout = 5, kStatusRange = 6 };
// info values: which wait ran out
enum : int32_t {
  kInfoEmpty = 1, kInfoFull = 2, kInfoAccFull = 3, kInfoAccEmpty = 4,
  kInfoGatherEmpty = 5, kInfoDrain = 6, kInfoReady = 7, kInfoFixup = 8,
  kInfoRouter = 9, kInfoTileCount = 10, kInfoHReady = 11,
  // range errors (kStatusRange): an FP4 block scale outside [104, 140], or a
  // value of x or h outside the f16 range of the FP4 experts' MMAs
  kInfoScaleRange = 12, kInfoXRange = 13, kInfoHRange = 14,
  // the start gate (status word 2) stayed closed for the whole wait
  kInfoHold = 15,
  // the router's work list is outside the bounds the host computed (a
  // workspace that was not zero-filled before its first use, or overwritten)
  kInfoWorkList = 16
};

// ----------------------------------------------------------------------------
// Expert-group work list written by the router's last CTA and read by the
// grouped GEMMs.  Group g is one touched expert (expert >= 0, in expert
// order) or the shared expert (expert == -1, always last).  Its rows are the
// sorted (token, slot) pairs [row_base, row_base + count) of the expert, or
// for the shared expert the T tokens in order at row_base = T*K.
// ----------------------------------------------------------------------------
struct GroupEntry {
  int32_t expert;
  int32_t row_base;
  int32_t count;
  int32_t idim;     // I of this expert (I or Is)
  int32_t gu_tile;  // first tile index of the group in the gate_up GEMM
  int32_t dn_tile;  // first tile index of the group in the down GEMM
  int32_t gu_w;     // cost of one gate_up k-block of this group (quarter k-blocks)
  int32_t dn_w;     // cost of one down k-block
  int64_t gu_iter;  // first k-block iteration of the group (gate_up)
  int64_t dn_iter;  // first k-block iteration of the group (down)
};
static_assert(sizeof(GroupEntry) == 48, "group entry layout");

struct GemmHeader {
  int32_t ngroups;
  int32_t gu_tiles;
  int32_t dn_tiles;
  int32_t n_eff;  // widest token tile of this forward (multiple of 16, <= n_max)
  int64_t gu_iters;
  int64_t dn_iters;
};

// Tile geometry.  A "tile" is 256 weight rows (two 128-row MMA halves) by up
// to n_max tokens; one k-block is 64 elements of the reduction dimension.
//   gate_up: half 0 = gate rows [m*128, m*128+128), half 1 = the matching up
//            rows; m-blocks = ceil(I/128); K = H.
//   down:    half 0 = output rows [m*256, m*256+128), half 1 = the next 128;
//            m-blocks = ceil(H/256); K = I.
constexpr int kBlockK = 64;
constexpr int kHalfRows = 128;
constexpr int kTileBytesA = kHalfRows * kBlockK * 2;  // one half, bf16: 16 KB
constexpr int kGemmThreads = 224;                     // 7 warps
constexpr int kGemmThreadsFp4 = 352;                  // + 4 warps that expand FP4 weights
constexpr int kPackedBytes = 2 * kHalfRows * kBlockK / 2;  // FP4 codes of one k-block, both halves: 8 KB
constexpr int kMaxPStages = 16;                       // stages of FP4 codes
// e8m0 block scales whose products with every e2m1 value are exact in f16
constexpr int kFp4ScaleMin = 104, kFp4ScaleMax = 140;
constexpr int kMaxStages = 8;
// shared-memory control block: barriers and flags, the gather's row table
// (<= 256 rows), both GEMMs' CTA span tables (<= kMaxGrid CTAs) and the
// down epilogue's per-column weight and token (<= 256 columns)
constexpr int kCtrlBytes = 8192;
constexpr int kCtrlRowOff = 256;
constexpr int kCtrlSpans = 256 + 256 * 8;
constexpr int kCtrlCols = 6144;
constexpr int kMaxGrid = (kCtrlCols - kCtrlSpans) / 16 - 1;
constexpr int kGatherLag = 1;                         // cp.async groups in flight (<= stages - 1)

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Weight formats of a group's k-blocks, for the work list's cost model:
// bf16 (64 inputs, 32 KB), FP4 expanded by converter warps (64 inputs, 8.5
// KB), and the block-scaled formats read by the MMA directly (128 inputs:
// FP4 codes 16 KB + 1 KB of scales, FP8 codes 32 KB + 1 KB).
enum : int { kFmtBf16 = 0, kFmtFp4Conv = 1, kFmtMxFp4 = 2, kFmtMxFp8 = 3 };

// Relative cost of one k-block of a group whose tiles carry `nmma` token
// columns, in quarters of a weight-streaming k-block: up to 16 columns a
// k-block costs what its 32 KB of weights take to stream; wider tiles
// (the shared expert, large token counts) add MMA, gather and epilogue
// work, more in the down GEMM (h as hi and lo doubles its MMAs and gathers).
// The slopes are fitted to per-CTA timings of 16- and 80-column tiles.
// An FP4 k-block streams about a quarter of the bytes (8.5 KB); a
// block-scaled FP4 k-block half (17 KB), an FP8 one about the same (33 KB).
__host__ __device__ inline int kblock_cost(int phase, int nmma, int fmt = kFmtBf16) {
  const int base = fmt == kFmtFp4Conv ? 1 : (fmt == kFmtMxFp4 ? 2 : 4);
  return phase == 0 ? base + ((nmma - 16) * 3 + 80) / 160 : base + ((nmma - 16) * 7 + 20) / 40;
}

// Tiles of a group: nb token blocks of up to n_max tokens, mb 256-row weight
// tiles, kb k-blocks of `kblk` inputs (64 for bf16 operands, 128 for the
// block-scaled 8-bit and FP4 operands).
__host__ __device__ inline void group_geometry(int phase, int count, int idim, int H, int n_max,
                                               int& mb, int& nb, int& kb, int kblk = kBlockK) {
  nb = ceil_div(count, n_max);
  if (phase == 0) { mb = ceil_div(idim, kHalfRows); kb = ceil_div(H, kblk); }
  else            { mb = ceil_div(H, 2 * kHalfRows); kb = ceil_div(idim, kblk); }
}

// Byte ranges (16-byte aligned; sizes rounded down to 16) that an expert
// kernel prefetches into L2 once every CTA has issued its own weight loads:
// CTA c takes the c-th of `grid` equal shares of their concatenation.
constexpr int kMaxPrefetch = 8;
struct L2Prefetch {
  const uint8_t* ptr[kMaxPrefetch];
  long long bytes[kMaxPrefetch];
  int n;
};

struct GemmParams {
  const GroupEntry* groups;
  const GemmHeader* header;
  const int64_t* spans;        // [2][grid+1] first k-block iteration of every CTA, per phase
  const int32_t* span_groups;  // [2][grid+1] work-list group holding that iteration
  const uint16_t* x;           // [T,H] (gate_up token rows)
  const int32_t* sorted_pair;  // [T*K]
  int T, K, TK, H, I_ld;
  int n_max;                   // token tile width, multiple of 16, <= 256
  int stage_space;             // shared-memory bytes for the stage ring
  int nbuf;                    // TMEM accumulator buffers (1 or 2)
  uint32_t tmem_cols;
  float swiglu_limit;
  uint16_t* h;                 // gate_up output / down input [T*K + T, 2*I_ld] bf16 hi | lo
  float* out_ws;               // down output [T*K + T, H] fp32 (weighted)
  uint16_t* y;                 // down output when direct_y: [T, H] bf16
  int direct_y;
  const float* topk_w;         // [T*K]
  const float* sh_w;           // [T] shared-expert gate (nullable = 1)
  float* partials;             // [grid, 2 phases x 2 slots, 2 halves, n_max, 128] fp32
  int32_t* tile_counters_gu;   // [gate_up tiles] stream-K arrivals
  int32_t* tile_counters_dn;   // [down tiles]
  int32_t* ready;              // [gate_up tiles] finished gate_up tiles per (group, token block)
  int32_t* status;
  // FP4 routed experts (moe_ffn_forward_fp4): codes come through the tensor
  // maps, the e8m0 scales are read here; routed groups multiply in f16
  const uint16_t* xh;          // [T,H] f16 copy of x
  const uint8_t* gu_scale;     // prepared scale blocks (moe_fp4_prepare_scales): 512 bytes per
  const uint8_t* dn_scale;     // (expert, tile, k-block), gate_up blocks first, then down
  int I, E;                    // routed experts' I, expert count
  int h_tma;                   // the down GEMM loads h rows by TMA (I, Is multiples of 64)
  // host-computed bounds of the router's work list, checked before use
  int g_max, max_gu_tiles, max_dn_tiles;
  long long max_gu_iters, max_dn_iters;
  L2Prefetch pf;               // byte ranges to prefetch into L2 in the launch's tail
};

// Block-scaled expert GEMMs (mx.cu): routed experts as FP4 (e2m1 codes with
// an e8m0 scale per 32 inputs) or FP8 (e4m3 codes with an e8m0 scale per
// 32 x 32 block), the shared expert as FP8, both multiplied by the tensor
// cores' block-scaled MMA (kind::mxf8f6f4) on k-blocks of 128 inputs.  The
// activations x and h enter as sums of e4m3 pieces, each piece with its own
// e8m0 scale per 32 inputs.
constexpr int kMxK = 128;        // inputs per k-block
constexpr int kMxPx = 3;         // e4m3 pieces of x
constexpr int kMxPh = 4;         // e4m3 pieces of h
constexpr int kMxMaxTok = 24;    // token tile: kMxPh x 24 = 96 MMA columns, two accumulator buffers in TMEM
constexpr int kMxSfBytes = 512;  // one scale chunk: 128 rows x 4 inputs-chunks of 32
constexpr int kMxThreads = 224;

struct MxParams {
  const GroupEntry* groups;
  const GemmHeader* header;
  const int64_t* spans;
  const int32_t* span_groups;
  const uint16_t* x;           // [T,H] bf16
  const int32_t* sorted_pair;
  const int32_t* idx;          // [T*K] routing of every (token, slot)
  const int32_t* pair_pos;     // [T*K] its row among the sorted pairs
  const int32_t* offsets;      // [E+1] first sorted row of every expert
  const int32_t* e2d;          // [E] first token block of every touched expert (router)
  // Operand images: for every token block of every group (dense index: the
  // group's first gate_up tile / mb0 + block) and every k-block, the B tile
  // the MMA reads (rows of 128 bytes in the 128-byte-swizzled K-major layout,
  // token j's piece p in row j*P + p) followed by its 512-byte scale chunk.
  // The gate_up images (pieces of x) are written by the kernel's prologue,
  // the down images (pieces of h) by the gate_up epilogue.
  uint8_t* img_gu;
  uint8_t* img_dn;
  int img_gu_rows, img_dn_rows;  // rows of an image slot
  int kb_gu, kb_dn;            // k-blocks per token block: H/128, I_ld/128
  int mb0;                     // routed gate_up m-blocks, ceil(I/128)
  int n_dense;                 // token blocks of all groups (bound)
  int32_t* img_ready;          // warps that finished their share of the gate_up images (zeroed by the router)
  int T, K, TK, H, I_ld;       // I_ld = max(I, Is)
  int n_max;                   // token tile width (16 or 24)
  int stage_space;
  float swiglu_limit;
  float* out_ws;               // [T*K + T, H] fp32 weighted outputs (unless direct_y)
  uint16_t* y;
  int direct_y;
  const float* topk_w;
  const float* sh_w;
  float* partials;             // [grid][4][2][n_max][128] fp32
  int32_t* tile_counters_gu;
  int32_t* tile_counters_dn;
  int32_t* ready;
  int32_t* status;
  const uint8_t* scales;       // prepared weight scale chunks (moe_mx_prepare_scales)
  int I, Is, E;
  int routed_fp4;              // routed weights are FP4 (else FP8)
  int g_max, max_gu_tiles, max_dn_tiles;
  long long max_gu_iters, max_dn_iters;
  L2Prefetch pf;
};

// Byte offsets of the prepared weight scales: for every (expert, 256-row
// tile, 128-input k-block) 1 KB, the two 128-row halves' chunks; routed
// gate_up, routed down, shared gate_up, shared down, in that order.
__host__ __device__ inline size_t mx_scale_offset(int E, int H, int I, int Is, int phase, int e, int m, int kb) {
  const size_t mb0 = ceil_div(I, kHalfRows), kb0 = H / kMxK, mb1 = ceil_div(H, 2 * kHalfRows), kb1 = I / kMxK;
  const size_t r_gu = static_cast<size_t>(E) * mb0 * kb0, r_dn = static_cast<size_t>(E) * mb1 * kb1;
  const size_t s_gu = static_cast<size_t>(ceil_div(Is, kHalfRows)) * kb0;
  if (e >= 0) {
    if (phase == 0) return ((static_cast<size_t>(e) * mb0 + m) * kb0 + kb) * 1024;
    return (r_gu + (static_cast<size_t>(e) * mb1 + m) * kb1 + kb) * 1024;
  }
  if (phase == 0) return (r_gu + r_dn + static_cast<size_t>(m) * kb0 + kb) * 1024;
  return (r_gu + r_dn + s_gu + static_cast<size_t>(m) * (Is / kMxK) + kb) * 1024;
}

// Routing recipe as the selection code reads it (score_fn 0 softmax,
// 1 sigmoid, 2 sqrt(softplus); renorm = norm_topk_prob).
struct SelCfg {
  int E, K, score_fn, n_group, topk_group, group_topn, renorm;
  float eps, scale;
  const float* expert_bias;
};

struct RouteParams {
  const uint16_t* x;
  const uint16_t* gate;
  const float* router_bias;
  const float* expert_bias;
  const uint16_t* sh_gate;
  int T, H, E, K;
  int score_fn, n_group, topk_group, group_topn, renorm;
  float eps, scale;
  int quads, hsplit, n_eb, n_tb;
  float* logits;               // [T, E]
  float* sh_logit;             // [T] (when sh_gate), or [T][n_eb*hsplit] partial sums (fold_sh)
  int fold_sh;                 // the shared-gate row is folded into per-block partials
  int32_t* idx;                // [T*K]
  float* w;                    // [T*K]
  float* sh_w;                 // [T] (nullable)
  int32_t* tb_counter;         // [n_tb]
  int32_t* glob_counter;       // [1]
  // optional permutation and GEMM work list (do_permute)
  int do_permute;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_pair;
  int32_t* pair_pos;
  GroupEntry* groups;          // nullable
  GemmHeader* header;
  int64_t* spans;              // [2][grid+1] cost-balanced CTA spans for the GEMM
  int32_t* span_groups;        // [2][grid+1]
  int grid;                    // CTAs of the GEMM launch
  int I, Is, n_max;
  int32_t* zero_ptr;           // GEMM tile counters cleared by this launch
  int zero_count;
  int fp4;                     // routed experts are FP4: their k-blocks cost less
  int fmt, sh_fmt;             // cost-model formats of the routed and the shared groups (kFmt*)
  int kblk;                    // inputs per k-block of the work list (64, or 128 block-scaled)
  int32_t* e2d;                // [E] (nullable) each touched expert's first token block over all groups
  int logits_given;            // logits (and sh_logit) were computed by logits_gemm_kernel: route only
  int lsplit;                  // > 1: the GEMM left lsplit partial sums over ranges of H in lpart
  const float* lpart;          // [lsplit][T][E (+1 with sh_gate)] fp32, summed in split order
  uint16_t* xh;                // [T,H] f16 copy of x written for FP4 experts (nullable)
  int32_t* status;             // range errors of that copy
};

// Fused small-expert-count forward (slice.cu): one CTA per (expert, 128-row
// slice of its intermediate dimension), the router on spare CTAs.
struct SliceParams {
  const uint16_t* x;           // [T,H]
  const uint16_t* gate;        // [E,H]
  const float* router_bias;    // [E] (nullable)
  const uint16_t* sh_gate;     // [H] (nullable)
  SelCfg sel;
  int T, H, E, K, TK;
  int n_tok;                   // gate_up MMA width: T rounded up to 16 (<= kSliceMaxTok)
  int s_e, s_sh;               // 128-row slices of a routed expert / of the shared expert (0: none)
  int s_max;                   // max(s_e, s_sh)
  int n_units;                 // E * s_e + s_sh
  int n_mt;                    // 128-row output tiles: ceil(H / 128)
  int n_rcta;                  // router CTAs (after the unit CTAs)
  int n_tg;                    // token groups of the combine (kSliceTokPerTask tokens each)
  int stage_space;             // shared-memory bytes for the stage rings
  int parts;                   // k-block ranges per down output tile (fp32 partials when > 1)
  int direct_y;                // top-1, no shared expert, one part: the down epilogue writes y
  float swiglu_limit;
  float* logits;               // [T,E]
  int32_t* idx;                // [T*K]
  float* w;                    // [T*K]
  float* sh_w;                 // [T] shared-expert weight (gate, or 1)
  int32_t* counts;             // [E]
  uint8_t* hbuf;               // [(E+1) * 2*s_max] h tiles of 2*n_tok rows x 128 B (see slice.cu)
  float* out;                  // [parts][T*K + T, H] fp32 weighted expert outputs (unless direct_y)
  uint16_t* y;                 // [T,H]
  // [1 + 2 * set_words]: a parity word, then two counter sets used by
  // alternate forwards; a set is kSliceSyncWords words (router done, combine
  // task, exit count, -), n_mt output-tile counts, (E+1)*s_max slice-ready flags
  int32_t* sync;
  int set_words;               // stride of the two sets (kSliceMaxSetWords); a set is cleared whole
  int32_t* status;
};
constexpr int kSliceMaxTok = 128;
constexpr int kSliceMaxExperts = 16;  // routed experts + the shared-expert gate row
constexpr int kSliceTokPerTask = 7;   // one token per warp of a reduction task
constexpr int kSliceSyncWords = 4;
constexpr int kSliceCtrlBytes = 4096;  // control block at the start of shared memory
// Words of one slice counter set for the largest shape the entry points
// accept (H <= 65536: 512 output tiles; E + 1 <= 17 expert slots; I, Is <=
// 16384: 128 slices): every shape's set fits, so the sets sit at fixed
// offsets whatever the shape.
constexpr int kSliceMaxSetWords = kSliceSyncWords + 512 + (kSliceMaxExperts + 1) * 128;

// ---------------------------------------------------------------------------
// Fixed workspace header (every workspace of moe_route / moe_ffn_forward):
// the status block, then every counter that returns to zero by itself after
// a call, at offsets that depend on neither the token count nor the shape,
// so one zero-filled workspace serves calls of any size it is large enough
// for.  Everything after the header is data a call writes before it reads.
//   [0, 256)                   status block: {code, info, hold, -}
//   [256, 256 + kRouteCntBytes)  router token-block counters + completion
//                              counter (4-token blocks of up to 65536 tokens)
//   [.., + kSliceSyncBytes)    fused kernel: parity word + two counter sets
// ---------------------------------------------------------------------------
constexpr size_t kWsAlign = 256;
constexpr size_t ws_align_up(size_t v) { return (v + kWsAlign - 1) / kWsAlign * kWsAlign; }
constexpr int kMaxTokens = 65536;
constexpr size_t kRouteCntOffset = kWsAlign;
constexpr size_t kRouteCntBytes = ws_align_up(4 * (kMaxTokens / 4 + 1));
constexpr size_t kSliceSyncOffset = kRouteCntOffset + kRouteCntBytes;
constexpr size_t kSliceSyncBytes = ws_align_up(4 * (1 + 2 * static_cast<size_t>(kSliceMaxSetWords)));
constexpr size_t kWsHeaderBytes = kSliceSyncOffset + kSliceSyncBytes;
// Word 2 of the status block: the start gate.  While it is non-zero the
// expert kernels wait at their start (bounded), then record
// MOE_ERR_DEVICE_TIMEOUT with info kInfoHold and abort the forward.
constexpr int kStatusHoldWord = 2;

// Host-side argument checks of the router entry points (api.cu): MOE_OK
// when the call may proceed (T == 0 included), else the status to return.
// Nothing touches a device before they pass.
moe_status route_check_args(const uint16_t* x, int T, int H, const uint16_t* gate, const moe_recipe* recipe,
                            const int32_t* topk_idx, const float* topk_w);

// launchers (route.cu, gemm.cu, combine.cu); return cudaError_t
cudaError_t launch_route(const RouteParams& p, int tb, cudaStream_t s);
// Tiled CUDA-core logits GEMM for many tokens (the router's first step).
// split > 1: H is cut into split ranges of 32-input chunks, one grid slice
// each, which write their partial sums (no router bias) to part
// [split][T][E (+1)]; the router launch adds them in split order.
cudaError_t launch_logits_gemm(const uint16_t* x, const uint16_t* gate, const uint16_t* sh_gate,
                               const float* router_bias, int T, int H, int E, float* logits, float* sh_logit,
                               int split, float* part, cudaStream_t s);
// H ranges of the logits GEMM for a layer's router with T tokens: enough
// slices to fill the SMs about three times, each at least 8 chunks of 32.
int logits_gemm_split(int T, int H, int E_tot, int sms);
cudaError_t launch_select_from_logits(const float* logits, int T, int E, int K, const float* expert_bias,
                                      int score_fn, int n_group, int topk_group, int group_topn,
                                      int renorm, float eps, float scale, int32_t* idx, float* w,
                                      cudaStream_t s);
cudaError_t launch_permute(const int32_t* idx, int T, int K, int E, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* pair_pos, cudaStream_t s);
cudaError_t launch_experts(const CUtensorMap& tm_gu, const CUtensorMap& tm_gu_sh, const CUtensorMap& tm_dn,
                           const CUtensorMap& tm_dn_sh, const CUtensorMap& tm_h, const GemmParams& p, int grid,
                           size_t smem_bytes, cudaStream_t s, bool fp4);
// FP4 block scales re-laid into 512-byte (expert, tile, k-block) blocks.
cudaError_t launch_fp4_scales(const uint8_t* gu_s, const uint8_t* dn_s, int E, int H, int I, uint8_t* out,
                              cudaStream_t s);
// overlap: programmatic stream serialization, else a cooperative launch
cudaError_t launch_slice(const CUtensorMap& tm_gu, const CUtensorMap& tm_gu_sh, const CUtensorMap& tm_dn,
                         const CUtensorMap& tm_dn_sh, const CUtensorMap& tm_x, const SliceParams& p, int grid,
                         size_t smem_bytes, bool overlap, cudaStream_t s);
cudaError_t launch_combine(const float* out_ws, const int32_t* pair_pos, int T, int K, int H,
                           int has_shared, uint16_t* y, cudaStream_t s);
cudaError_t launch_mx(const CUtensorMap& tm_gu, const CUtensorMap& tm_gu_sh, const CUtensorMap& tm_dn,
                      const CUtensorMap& tm_dn_sh, const MxParams& p, int grid, size_t smem_bytes, cudaStream_t s);
// Weight scales re-laid into the chunks the block-scaled MMA reads
// (routed_fp4: one scale per 32 inputs; else one per 32 x 32 block).
cudaError_t launch_mx_scales(int routed_fp4, const uint8_t* gu_s, const uint8_t* dn_s, int E, int H, int I,
                             const uint8_t* sh_gu_s, const uint8_t* sh_dn_s, int Is, uint8_t* out, cudaStream_t s);

// ----------------------------------------------------------------------------
// inline PTX (device only)
// ----------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// A bounded wait gives up after this many SM clock cycles (about 1 s).
constexpr long long kWaitLimitCycles = 2000000000ll;

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `parity` to complete; returns false if the CTA's
// abort flag (when given) is raised or the wait runs past kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA: 3-D tiled load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// The same with an L2 cache policy (createpolicy), e.g. evict-first for
// weights that are streamed once.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                                 int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Contiguous bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// The same copy with an L2 cache-eviction policy (data streamed once).
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// L2 prefetch of a contiguous range (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// This CTA's share of the ranges of `pf`, prefetched into L2 in 64 KB pieces.
__device__ __forceinline__ void prefetch_share_l2(const L2Prefetch& pf) {
  long long total = 0;
  for (int i = 0; i < pf.n; ++i) total += pf.bytes[i];
  if (total <= 0) return;
  long long a = (total * blockIdx.x / gridDim.x) & ~15ll, b = (total * (blockIdx.x + 1) / gridDim.x) & ~15ll;
  long long base = 0;
  for (int i = 0; i < pf.n && a < b; ++i) {
    const long long lo = a > base ? a : base, hi = b < base + pf.bytes[i] ? b : base + pf.bytes[i];
    for (long long o = lo; o < hi; o += 65536) {
      const long long n = hi - o < 65536 ? hi - o : 65536;
      if (n >= 16) bulk_prefetch_l2(pf.ptr[i] + (o - base), static_cast<uint32_t>(n & ~15ll));
    }
    base += pf.bytes[i];
  }
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// L2 prefetch of one tile box of a 3-D tensor map.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Programmatic dependent launch: let the next launch on the stream (made
// with the programmatic-serialization attribute) start its CTAs, and wait
// until the previous launch on the stream has completed with its memory
// visible (a no-op when the launch does not depend on one programmatically).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// cp.async (16 bytes, L2 only); src_bytes == 0 zero-fills the destination.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// cp.async of 4 bytes (through L1); src_bytes == 0 zero-fills the destination.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05.mma issued so far by this thread is complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x one 32-bit column.
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 128 bytes (64 bf16), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// ---- small helpers shared by the GEMM kernels
__device__ __forceinline__ uint16_t f2bf(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void record_failure(int32_t* status, volatile int* abort_flag, int32_t info) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) atomicExch(status + 1, info);
  *abort_flag = 1;
}

// A value outside the exact range of the computation: recorded, the forward
// runs on (its output is not exact).
__device__ __forceinline__ void record_range(int32_t* status, int32_t info) {
  if (atomicCAS(status, 0, kStatusRange) == 0) atomicExch(status + 1, info);
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The start gate (status word kStatusHoldWord): true once it is zero; false
// when it stays non-zero past kGateLimitCycles or another CTA has already
// recorded a failure.  The limit is a quarter of every other wait's, so a
// closed gate is always the first failure a forward records.
constexpr long long kGateLimitCycles = kWaitLimitCycles / 4;
__device__ __forceinline__ bool wait_start_gate(const int32_t* status) {
  if (ld_acquire_gpu(status + kStatusHoldWord) == 0) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(256);
    if (ld_acquire_gpu(status + kStatusHoldWord) == 0) return true;
    if (*reinterpret_cast<const volatile int32_t*>(status) != 0) return false;
    if (clock64() - t0 > kGateLimitCycles) return false;
  }
}

// Position in the ring of shared-memory stages (each role keeps its own).
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ void next(int S) {
    if (++stage == S) { stage = 0; phase ^= 1u; }
  }
};

#endif  // __CUDACC__

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A
// and B, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with f16 A and B (type fields 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace moe
