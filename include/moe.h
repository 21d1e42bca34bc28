/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE-FFN layer forward used by
 * DFlash / DSpark block-diffusion draft models.
 *
 * The layer (sources are web pages, cited by title and section):
 *   1. Router, the score -> select -> routing_weights template of SpecForge
 *      PR #1033 "MoE FFN for DFlash-family drafts: the module", section
 *      "Router": fp32 logits of a linear gate (sglang PR #48763 "[Feat]
 *      dflash: Serve MoE FFN drafts for DFlash and DSpark", commit note on
 *      the router's fp32 logits), optionally with a folded router
 *      bias added to the logits (SpecForge PR #941 "SGLang draft classes for
 *      the Qwen3.8-27B DSpark MoE drafter", section "What"); softmax, sigmoid
 *      or sqrt(softplus) scores; a selection-only expert bias (SpecForge PR
 *      #1073 "MoE drafts: DeepSeek-V4.1's own DSpark draft", expert-bias
 *      commit note); plain or group-limited top-k; weights gathered from the
 *      unshifted scores, renormalised with +1e-20 and times route_scale.
 *   2. Token-to-expert grouped SwiGLU experts (fused gate_up_proj [E,2I,H],
 *      down_proj [E,H,I]; PR #1073 commit note on the fused expert layout),
 *      with DeepSeek's optional clamp (PR #941 follow-up comment).
 *   3. An optional shared expert, sigmoid-gated (Qwen, PR #941 "What") or
 *      ungated (DeepSeek), added to the weighted combine of the routed
 *      experts (PR #48763 commit note on DraftMoE forward).
 *
 * Conventions (every entry point):
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; tensors are
 *     contiguous, row-major.  bf16 tensors are passed as raw 16-bit words.
 *     Indices are int32 (PR #48763: the fused routers' id type).
 *   - Calls are asynchronous on `stream` and never synchronise the host, so a
 *     sequence of them can be captured in a CUDA graph.  The library performs
 *     no device allocation; scratch space is the caller's workspace.
 *   - Argument errors are returned synchronously, before any launch.  Errors
 *     found on the device (a bounded wait that ran out) are recorded in the
 *     workspace's status word and read with moe_get_device_status().
 *   - T == 0 returns MOE_OK and launches nothing (PR #48763: an empty batch gives
 *     an empty routing).
 *   - x is only read; y must not alias x (PR #48763 fix: the shared expert
 *     must read x before in-place experts overwrite it).
 *   - Requested features are never silently dropped (PR #48763 fixed an
 *     ignored expert bias and a routed_scaling_factor that was never applied):
 *     what the kernels cannot do is refused with MOE_ERR_UNSUPPORTED.
 *   - Limits: 1 <= E <= 1024, 1 <= K <= min(E, 32), H and I multiples of 8,
 *     8 <= H <= 65536, 8 <= I <= 16384, T <= 65536, n_group <= 32 and
 *     divides E, K <= topk_group * (E / n_group).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* raw bfloat16 bits */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null required pointer, negative size, ...  */
  MOE_ERR_UNSUPPORTED = 2,    /* well-formed but outside the kernels' limits */
  MOE_ERR_WORKSPACE = 3,      /* workspace missing, too small or misaligned  */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime call failed                  */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait ran out          */
  MOE_ERR_DEVICE_RANGE = 6    /* an input outside the exact range of the FP4
                                 path (a block scale, or x / h beyond f16);
                                 recorded on the device, the output is not
                                 exact                                       */
} moe_status;

typedef enum {
  MOE_SCORE_SOFTMAX = 0,
  MOE_SCORE_SIGMOID = 1,
  MOE_SCORE_SQRTSOFTPLUS = 2
} moe_score_fn;

/* The routing recipe (PR #1033 "Router" table; the HF keys num_experts,
 * num_experts_per_tok, scoring_func, n_group / topk_group, norm_topk_prob,
 * routed_scaling_factor, swiglu_limit map onto these fields). */
typedef struct {
  int32_t num_experts;    /* E                                                  */
  int32_t top_k;          /* K                                                  */
  int32_t score_fn;       /* moe_score_fn                                       */
  int32_t n_group;        /* 1 = plain top-k; > 1 = group-limited select        */
  int32_t topk_group;     /* groups kept by group-limited select                */
  int32_t group_topn;     /* a group's score = sum of its group_topn best (2)   */
  int32_t norm_topk_prob; /* 1: renormalise the K gathered scores               */
  float norm_eps;         /* added to the renormalisation sum (1e-20)           */
  float route_scale;      /* route_scale == routed_scaling_factor (routed only) */
  float swiglu_limit;     /* > 0: clamped SwiGLU (routed and shared experts)    */
} moe_recipe;

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(moe_status s);

/* Bytes of workspace moe_route() needs for T tokens and E experts: the fixed
 * header (status block, token-block completion counters sized for any T) and
 * the [T,E] fp32 logits (used when logits_out is NULL). */
MOE_API size_t moe_route_workspace_bytes(int T, int E);

/* Router: logits = x . gate^T (+ router_bias), fp32 accumulation of the exact
 * bf16 products; scores; select over scores + expert_bias; weights.
 *   x           [T,H] bf16            gate        [E,H] bf16
 *   router_bias [E] fp32 or NULL      added to the logits (moves weights too)
 *   expert_bias [E] fp32 or NULL      added to the scores for selection only
 *   logits_out  [T,E] fp32 or NULL    the fp32 logits
 *   topk_idx    [T,K] int32           descending shifted score, ties -> lower e
 *   topk_w      [T,K] fp32            routing weights
 *   ws          workspace of >= moe_route_workspace_bytes(T, E) bytes,
 *               256-byte aligned, zero-filled once before its first use
 *               (moe_workspace_init).  Its counters sit at fixed offsets and
 *               every call leaves them at zero, so the workspace then serves
 *               any later call it is large enough for, whatever its T; after
 *               a device-side error (moe_get_device_status) zero-fill it again.
 */
MOE_API moe_status moe_route(const moe_bf16* x, int T, int H, const moe_bf16* gate,
                     const float* router_bias, const float* expert_bias,
                     const moe_recipe* recipe, float* logits_out,
                     int32_t* topk_idx, float* topk_w,
                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_route() without a workspace, for callers that cannot allocate device
 * memory when they call it (a serving engine whose pool has reserved the whole
 * device up front, code that must not re-enter its allocator, a plain C
 * caller with no device allocator).  The pages have no counterpart: this is a
 * packaging variant of moe_route().
 *   Same arguments and results as moe_route() minus ws / ws_bytes.
 *   Scratch: one file-scope device array of about 1.1 MB inside the library
 *     (moe_route's workspace for the largest call it takes: the token-block
 *     counters and the [T,E] fp32 logits, which hold the logits when
 *     logits_out is NULL), held on every GPU that loads the library until the
 *     process exits.  No cudaMalloc / cudaFree or other allocating call is
 *     made.
 *   Arguments are checked as moe_route() checks them before the array is
 *     touched: a refused call leaves it as it was.
 *   Limits: T <= MOE_NOALLOC_MAX_TOKENS and T*E <= MOE_NOALLOC_MAX_LOGITS,
 *     else MOE_ERR_UNSUPPORTED before anything runs.
 *   The first call on each device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   Every call shares the one array: the call clears its counters (they must
 *     start at zero) on `stream`, and two calls that may overlap on the GPU
 *     (other streams, other host threads) race on it. */
#define MOE_NOALLOC_MAX_TOKENS 4096
#define MOE_NOALLOC_MAX_LOGITS 262144
MOE_API moe_status moe_route_noalloc(const moe_bf16* x, int T, int H, const moe_bf16* gate,
                                     const float* router_bias, const float* expert_bias,
                                     const moe_recipe* recipe, float* logits_out,
                                     int32_t* topk_idx, float* topk_w, cudaStream_t stream);

/* Router steps score -> select -> routing_weights on given fp32 logits [T,E]
 * (the same logits fed to another implementation give the same selection).
 * Needs no workspace. */
MOE_API moe_status moe_route_from_logits(const float* logits, int T,
                                 const float* expert_bias,
                                 const moe_recipe* recipe,
                                 int32_t* topk_idx, float* topk_w,
                                 cudaStream_t stream);

/* Token-to-expert grouping (SpecForge grouped_mm experts, PR #1033; the
 * tokens_per_expert counts of PR #1073):
 *   counts[e]   = #{(t,k) : topk_idx[t,k] == e}                 [E]   int32
 *   offsets     = exclusive prefix sum of counts                [E+1] int32
 *   sorted_pair = pairs p = t*K + k, stably sorted by expert   [T*K] int32
 *   pair_pos    = inverse permutation of sorted_pair            [T*K] int32
 * Needs no workspace (ws may be NULL). */
MOE_API moe_status moe_permute(const int32_t* topk_idx, int T, int K, int E,
                       int32_t* counts, int32_t* offsets,
                       int32_t* sorted_pair, int32_t* pair_pos,
                       void* ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes for moe_ffn_forward() of exactly T tokens on the CURRENT
 * device (the size depends on its SM count).  Is = 0 means no shared expert.
 * Returns 0 for an invalid recipe.  The size is not monotone in T (above 128
 * tokens the token tile narrows to about four times an expert's mean load):
 * a workspace meant for every T up to a maximum takes the largest value over
 * that range. */
MOE_API size_t moe_ffn_workspace_bytes(int T, int H, int I, int Is, const moe_recipe* recipe);

/* Zero-fill a workspace (required once before its first use, and again after
 * a device-side error). */
MOE_API moe_status moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* The whole layer: y = sum_k w_tk * Expert_{idx_tk}(x_t) + g_t * Shared(x_t).
 *   x          [T,H] bf16
 *   gate       [E,H] bf16; router_bias, expert_bias as in moe_route()
 *   w_gate_up  [E,2I,H] bf16: rows [0,I) gate (w1), rows [I,2I) up (w3)
 *   w_down     [E,H,I] bf16
 *   sh_gate_up [2Is,H] bf16 or NULL (no shared expert; then Is must be 0)
 *   sh_down    [H,Is] bf16
 *   sh_gate    [H] bf16 or NULL: g_t = sigmoid(x_t . sh_gate), else g_t = 1
 *   ws         >= moe_ffn_workspace_bytes(T,H,I,Is,recipe) bytes, 256-byte
 *              aligned, zero-filled once before its first use
 *              (moe_workspace_init).  Every counter the kernels keep sits in
 *              a fixed header whose offsets depend on neither T nor the shape,
 *              and every call leaves it at zero, so the workspace then serves
 *              any later call (another T, shape or recipe) it is large enough
 *              for; after a device-side error (moe_get_device_status)
 *              zero-fill it again.  One workspace must not be used by two
 *              calls that may overlap on the GPU.  A workspace smaller than
 *              the call needs is refused with MOE_ERR_WORKSPACE.
 *   y          [T,H] bf16 output (round to nearest even from fp32)
 *   topk_idx_out [T,K] int32, topk_w_out [T,K] fp32, counts_out [E] int32:
 *              optional copies of the routing (each may be NULL).
 */
MOE_API moe_status moe_ffn_forward(const moe_bf16* x, int T, int H, int I,
                           const moe_bf16* gate, const float* router_bias,
                           const float* expert_bias,
                           const moe_bf16* w_gate_up, const moe_bf16* w_down,
                           const moe_bf16* sh_gate_up, const moe_bf16* sh_down,
                           int Is, const moe_bf16* sh_gate,
                           const moe_recipe* recipe, void* ws, size_t ws_bytes,
                           moe_bf16* y, int32_t* topk_idx_out, float* topk_w_out,
                           int32_t* counts_out, cudaStream_t stream);

/* Expert schedules of moe_ffn_forward():
 *   MOE_SCHEDULE_STREAM_K  a router launch (logits, top-k, permutation, work
 *       list); one persistent launch of both expert GEMMs that streams the
 *       touched experts' weight k-blocks split evenly over the SMs; the
 *       weighted combine (skipped for K == 1 without a shared expert).
 *   MOE_SCHEDULE_SLICE     one persistent launch for layers with few experts
 *       that every forward touches: one CTA per (expert, 128-row slice of I),
 *       the gate_up GEMM over all T tokens started before the routing is
 *       known, the router on spare CTAs, and a deterministic sum of the
 *       per-slice partial outputs.  An expert no token picked stops streaming
 *       once the routing is known.  Shape limits: T <= 128, E (+1 with
 *       sh_gate) <= 16, E*ceil(I/128) + ceil(Is/128) + ceil(T/7) <= SMs.
 *       The launch is made with programmatic stream serialization: its
 *       CTAs may start on the SMs that the previous kernel on the stream
 *       leaves (when that kernel allows it, as this one does) and stream
 *       their first weights into shared memory and L2 there; everything
 *       they read that a kernel writes (x, the workspace) waits until the
 *       previous kernel has completed.  So a CTA of the launch may wait for
 *       another to be placed (bounded, MOE_ERR_DEVICE_TIMEOUT on expiry): the
 *       grid assumes the SMs are not held by other work for long, and
 *       moe_set_launch_overlap(0) makes it a cooperative launch instead.
 *   MOE_SCHEDULE_AUTO      SLICE where the shape fits, the expected number
 *       of untouched experts under uniform routing, E*(1-K/E)^T, is at most
 *       0.25, and the down GEMM's work items (128-row output tiles, each cut
 *       into up to 2*ceil(I/128) k-block ranges so that the items do not
 *       outnumber the SMs) occupy at least three quarters of the SMs;
 *       STREAM_K otherwise.
 * Both give the same routing; outputs agree to fp32 summation order. */
typedef enum {
  MOE_SCHEDULE_AUTO = 0,
  MOE_SCHEDULE_STREAM_K = 1,
  MOE_SCHEDULE_SLICE = 2
} moe_schedule;

/* Per calling thread: the schedule later moe_ffn_forward() calls use.  A
 * forced MOE_SCHEDULE_SLICE still runs STREAM_K where the shape does not fit.
 * Returns MOE_ERR_INVALID_ARG for an unknown value. */
MOE_API moe_status moe_set_schedule(int schedule);

/* Per calling thread: how later MOE_SCHEDULE_SLICE launches start.  1 (the
 * default): with programmatic stream serialization, overlapping the end of
 * the previous kernel on the stream (see MOE_SCHEDULE_SLICE above).  0: as
 * cooperative launches, which start once every CTA of the grid can be
 * resident -- for streams whose kernels may run beside other work that holds
 * SMs.  Both compute the same bits.  Returns MOE_ERR_INVALID_ARG for a value
 * other than 0 or 1. */
MOE_API moe_status moe_set_launch_overlap(int enable);

/* The schedule moe_ffn_forward() would run for this shape on the current
 * device under the calling thread's setting: MOE_SCHEDULE_STREAM_K or
 * MOE_SCHEDULE_SLICE, or -1 for invalid arguments.  gated != 0 when sh_gate
 * will be passed. */
MOE_API int moe_ffn_schedule(int T, int H, int I, int Is, const moe_recipe* recipe, int gated);

/* ---- FP4 routed experts.  The format of DeepSeek-V4.1's official checkpoint
 * (SpecForge PR #1073, commit note on its export formats): every routed
 * expert weight is stored as e2m1 codes, two per byte along the input
 * dimension with the even input in the low nibble, and one e8m0 scale byte
 * (value 2^(s-127)) per 32 consecutive inputs; the MXFP4 tensors of
 * MoE-Infinity PR #143 have the same output-major layout:
 *   w_gate_up_q [E,2I,H/2] uint8   w_gate_up_s [E,2I,H/32] uint8
 *   w_down_q    [E,H,I/2]  uint8   w_down_s    [E,H,I/32]  uint8
 * The layer computes with the exactly dequantized weights (code value x
 * scale), as the bf16 draft those weights import into does.
 * Limits: H and I multiples of 64 (whole 64-input k-blocks), H <= 65536,
 * I <= 16384. */

/* Bytes of the prepared block scales of one layer (0 for unsupported
 * shapes). */
MOE_API size_t moe_fp4_scales_bytes(int E, int H, int I);

/* Re-lays the two scale tensors into the blocks the expert kernel copies
 * whole (for every expert, 256-row tile and 64-input k-block, the 128-row
 * halves' scale pairs: 512 bytes).  Once per set of weights, e.g. at load
 * time; asynchronous on `stream`.
 *   scales   device buffer of >= moe_fp4_scales_bytes(E,H,I) bytes, 16-byte
 *            aligned, owned by the caller and passed to every
 *            moe_ffn_forward_fp4() with these weights.
 * Returns MOE_ERR_WORKSPACE when scales_bytes is too small. */
MOE_API moe_status moe_fp4_prepare_scales(const uint8_t* w_gate_up_s, const uint8_t* w_down_s, int E, int H,
                                          int I, void* scales, size_t scales_bytes, cudaStream_t stream);

/* moe_ffn_forward() with FP4 routed experts: w_gate_up_q, w_down_q as above
 * (16-byte aligned), `scales` from moe_fp4_prepare_scales().  Router, shared
 * expert (bf16), workspace (moe_ffn_workspace_bytes), outputs and errors as in
 * moe_ffn_forward().  Always the STREAM_K schedule.
 * Arithmetic: the routed experts' products are exact f16 x f16 -> fp32 on the
 * tensor cores, so they need every e8m0 scale in [104, 140] (2^-23 .. 2^13,
 * where code x scale is exact in f16), |x| < 65520 and |h| < 65520 (the SwiGLU
 * output, carried as an f16 hi + lo pair); anything outside is recorded as
 * MOE_ERR_DEVICE_RANGE in the workspace status (moe_get_device_status).  x
 * values below 2^-17 in magnitude round to the f16 grid (error < 2^-25).
 * H and I must be multiples of 64 (else MOE_ERR_UNSUPPORTED). */
MOE_API moe_status moe_ffn_forward_fp4(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate,
                                       const float* router_bias, const float* expert_bias,
                                       const uint8_t* w_gate_up_q, const uint8_t* w_down_q, const void* scales,
                                       size_t scales_bytes, const moe_bf16* sh_gate_up, const moe_bf16* sh_down,
                                       int Is, const moe_bf16* sh_gate, const moe_recipe* recipe, void* ws,
                                       size_t ws_bytes, moe_bf16* y, int32_t* topk_idx_out, float* topk_w_out,
                                       int32_t* counts_out, cudaStream_t stream);

/* ---- Block-scaled experts: the weights stay in the formats of DeepSeek-V4.1's
 * official draft checkpoint (SpecForge PR #1073, commit note on its export
 * formats) and the tensor cores' block-scaled MMA multiplies them directly.
 *   routed_fmt MOE_FMT_FP4: the FP4 layout above (e2m1 codes, the even input
 *       in the low nibble, one e8m0 scale per 32 inputs):
 *         w_gate_up_q [E,2I,H/2], w_gate_up_s [E,2I,H/32],
 *         w_down_q    [E,H,I/2],  w_down_s    [E,H,I/32]
 *   routed_fmt MOE_FMT_FP8: e4m3 codes with one e8m0 scale per 32 x 32 block
 *       of the weight (the checkpoint's format for its other linears):
 *         w_gate_up_q [E,2I,H],   w_gate_up_s [E,2I/32,H/32],
 *         w_down_q    [E,H,I],    w_down_s    [E,H/32,I/32]
 *   shared expert, when present, always FP8 in that block format:
 *         sh_gate_up_q [2Is,H], sh_gate_up_s [2Is/32,H/32],
 *         sh_down_q    [H,Is],  sh_down_s    [H/32,Is/32]
 * The layer computes with the exactly dequantized weights (code x scale), as
 * the bf16 draft those weights import into does: the MMA applies both
 * operands' scales per 32 products, and x and h enter as sums of e4m3 pieces
 * (three for x, four for h, each piece with its own scale per 32 inputs) that
 * reproduce them to within 2^-13 (x) and 2^-17 (h) of a 32-input block's
 * largest magnitude (a bf16 x whose block spans a few binades exactly).
 * Limits: H, I and Is multiples of 128, H <= 65536, I, Is <= 16384; FP4 code
 * tensors 32-byte aligned, every other pointer 16-byte aligned. */
#define MOE_FMT_FP4 1
#define MOE_FMT_FP8 2

/* Bytes of the prepared weight scales of one layer (0 for an invalid format
 * or unsupported shape). */
MOE_API size_t moe_mx_scales_bytes(int routed_fmt, int E, int H, int I, int Is);

/* Re-lays the weight scales into the chunks the block-scaled MMA reads: for
 * every (expert, 256-row tile, 128-input k-block) 1 KB.  Once per set of
 * weights (load time); asynchronous on `stream`.  sh_* may be NULL when
 * Is == 0.  scales: device buffer of >= moe_mx_scales_bytes() bytes, 16-byte
 * aligned, owned by the caller and passed to every moe_ffn_forward_mx() with
 * these weights.  Returns MOE_ERR_WORKSPACE when scales_bytes is too small. */
MOE_API moe_status moe_mx_prepare_scales(int routed_fmt, const uint8_t* w_gate_up_s, const uint8_t* w_down_s, int E,
                                         int H, int I, const uint8_t* sh_gate_up_s, const uint8_t* sh_down_s, int Is,
                                         void* scales, size_t scales_bytes, cudaStream_t stream);

/* moe_ffn_forward() with block-scaled experts: router, workspace
 * (moe_ffn_workspace_bytes), outputs and errors as in moe_ffn_forward();
 * always the stream-K schedule, with token tiles of up to 24 tokens (an
 * expert with more tokens streams its weights once per tile).
 *   routed_fmt   MOE_FMT_FP4 or MOE_FMT_FP8
 *   w_gate_up_q, w_down_q   the routed experts' codes (layouts above)
 *   sh_gate_up_q, sh_down_q the shared expert's FP8 codes, or NULL (Is = 0)
 *   scales       from moe_mx_prepare_scales() */
MOE_API moe_status moe_ffn_forward_mx(const moe_bf16* x, int T, int H, int I, const moe_bf16* gate,
                                      const float* router_bias, const float* expert_bias, int routed_fmt,
                                      const uint8_t* w_gate_up_q, const uint8_t* w_down_q,
                                      const uint8_t* sh_gate_up_q, const uint8_t* sh_down_q, int Is,
                                      const moe_bf16* sh_gate, const void* scales, size_t scales_bytes,
                                      const moe_recipe* recipe, void* ws, size_t ws_bytes, moe_bf16* y,
                                      int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out,
                                      cudaStream_t stream);

/* Synchronises `stream`, reads the device status word of a workspace used by
 * moe_route() or moe_ffn_forward(), and clears it.  Returns MOE_OK or the
 * first device-side error recorded (MOE_ERR_DEVICE_TIMEOUT, or
 * MOE_ERR_DEVICE_RANGE from the FP4 path); *info_out (if not NULL) receives
 * the kernel-specific detail word (for MOE_ERR_DEVICE_TIMEOUT: which wait
 * ran out; MOE_INFO_HOLD for the start gate below).
 *
 * Start gate: the int32 at byte offset MOE_WS_HOLD_OFFSET of a workspace.
 * While it is non-zero, the expert kernels of moe_ffn_forward(),
 * moe_ffn_forward_fp4() and moe_ffn_forward_mx() wait at their start; once it
 * is zero they go on.  A
 * wait that lasts past a quarter of the device wait limit (about a quarter
 * second of SM clocks; every other device wait gives up after about one
 * second) ends the forward with MOE_ERR_DEVICE_TIMEOUT / MOE_INFO_HOLD: every CTA
 * lets its issued copies land, releases its tensor memory and returns, so
 * the context stays usable and the next forward on the same workspace is
 * correct.  The gate lets a host hold a queued forward from outside (and
 * exercises that failure path); it is zero in a zero-filled workspace and
 * the library never writes it. */
#define MOE_WS_HOLD_OFFSET 8
#define MOE_INFO_HOLD 15
MOE_API moe_status moe_get_device_status(void* ws, cudaStream_t stream, int32_t* info_out);

/* Route-ahead of the routing-independent part of the next layer (MoE-Infinity
 * PR #143 "converge DFlash spec-decode stack", route-ahead commit note:
 * bring what the next step needs close before it runs).  Which experts the
 * next layer touches depends on its input, but its router gate (and biases)
 * and its shared expert do not.  The next moe_ffn_forward(),
 * moe_ffn_forward_fp4() or moe_ffn_forward_mx() on the calling thread on the
 * stream-K schedule takes these n <= 8 byte ranges (16-byte aligned; sizes
 * rounded down to 16): once every CTA of its expert kernel has issued its own
 * weight loads, it prefetches its share of them into L2, so the prefetch
 * rides the layer's tail.  The setting is consumed by that call (also when
 * the call runs the fused schedule, which ignores it); n = 0 clears it.
 * Whether the bytes are still in L2 when the next layer runs depends on what
 * runs in between (an attention step that streams more than L2 evicts them).
 * Returns MOE_ERR_INVALID_ARG for n outside [0, 8] or a NULL / unaligned
 * pointer. */
MOE_API moe_status moe_set_l2_prefetch(const void* const* ptrs, const size_t* bytes, int n);

/* Profiling hook: when `events` is not NULL, moe_ffn_forward() records
 * events[2*i] / events[2*i+1] (cudaEvent_t) around its i-th kernel launch,
 * for i < n_pairs, on its stream.  Per calling thread; NULL turns it off.
 * The launch order is: router, expert GEMMs (gate_up and down in one
 * persistent launch), combine (skipped when K == 1 and there is no shared
 * expert).  Under MOE_SCHEDULE_SLICE the one fused launch is recorded as the
 * expert-GEMM pair; the router pair is recorded empty (both events at the
 * same point) and the combine pair not at all.  During a stream capture the
 * events are recorded as external event-record nodes of the graph, so every
 * replay records them. */
MOE_API void moe_set_profile_events(void* const* events, int n_pairs);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
