/*
 * mok.h -- C ABI of libmok.so: one Mixture-of-Experts layer, forward and
 * backward, on one GB300 (sm_103a).
 *
 * What the layer computes follows three news pages on Cursor's
 * "Mixture-of-Kittens" (MoK) MoE kernel; they give prose, not formulas:
 *   [kucoin] "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
 *            NVL72" (kucoin.com flash, Arabic), sections 01, 02, 03;
 *   [miku]   "Mixture of kittens: how Cursor opened a kernel that speeds up
 *            AI training by up to 2.4x" (miku-ai.ru);
 *   [qvib]   "Mixture-of-Kittens (MoK) open source" (qvib.pro news).
 * [kucoin] §03 names the steps of the measured layer: routing, the expert
 * FFN, combine and the final weighted combine; §01 adds per-expert counts and
 * placement (layout) before the grouped GEMM; §02 gives pull dispatch / push
 * combine (and the reverse pair in backward) and MXFP8 quantisation fused into
 * dispatch, the grouped GEMM and SwiGLU.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are caller-owned device memory; pointers marked
 *     "host" are read before the call returns.  The library never allocates,
 *     never frees and never synchronises the host inside a call: work is
 *     enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     So the layer calls can be captured into a CUDA graph and replayed,
 *     once each kind of call has run outside the capture (the first call
 *     of a kind sets its kernels' launch attributes, once per process).
 *   - Return value: MOK_OK, or a host-detectable error code (nothing was
 *     enqueued).  Errors found on the device (a bounded wait that ran out)
 *     land in the status word of the workspace; read them with
 *     mok_get_device_status.
 *   - Notation: T tokens, d = d_model, E experts, k = top_k, F = d_ff,
 *     S = T*k slots.  BF16 values are stored as raw 16-bit patterns.
 *   - Expert-ordered row buffers (xe, h, saved a/b/h, dy/dx rows) use the
 *     PADDED layout: expert e owns rows [pad_offsets[e], pad_offsets[e] +
 *     counts[e]) and pad_offsets[e+1] - pad_offsets[e] = counts[e] rounded up
 *     to MOK_ROW_ALIGN; the rows in between are padding with unspecified
 *     contents.  A buffer of mok_max_padded_rows(cfg) rows always suffices.
 *   - MXFP8 tensors are E4M3 codes (one byte each, row-major [rows, K]) plus
 *     E8M0 scales (one byte per 32 consecutive elements along K) in the MX
 *     SCALE TILE LAYOUT: for rows a multiple of 128 and K a multiple of 128,
 *     the 32-bit word of (k-group g = K/128 index, row r) sits at word index
 *        (g * rows/128 + r/128) * 128 + (r % 32) * 4 + (r % 128) / 32
 *     and its byte b (0..3, little-endian) is the scale of K-block 4g + b.
 *     Total size rows * K / 32 bytes.
 */
#ifndef MOK_H
#define MOK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MOK_OK = 0,
    MOK_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, bad enum */
    MOK_ERR_UNSUPPORTED = 2,   /* shape the kernels do not handle (see mok_config) */
    MOK_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    MOK_ERR_TIMEOUT = 4        /* device: a bounded wait gave up */
};

enum { MOK_ROUTER_SOFTMAX = 0, MOK_ROUTER_SIGMOID = 1 };
enum { MOK_BF16 = 0, MOK_MXFP8 = 1 };
/* Tile choice of the tensor-core GEMMs: one CTA per 128-row tile, or CTA
 * pairs (cta_group::2, 256-row tiles shared by two SMs).  Results are
 * bit-identical either way; only the speed differs. */
enum { MOK_PAIRS_AUTO = 0, MOK_PAIRS_ON = 1, MOK_PAIRS_OFF = 2 };

#define MOK_ROW_ALIGN 128      /* expert segment alignment of row buffers */
#define MOK_MAX_SOURCES 64     /* simulated expert-parallel source buffers */
#define MOK_MAX_EXPERTS 1024
#define MOK_MAX_TOPK 8

/*
 * Layer configuration.  Supported: 0 <= T, 1 <= E <= MOK_MAX_EXPERTS,
 * 1 <= k <= min(E, MOK_MAX_TOPK), d and F multiples of 128 (the MXFP8 block
 * of 32 and the 128-wide tiles), S + 128 E < 2^31, and for n_sources > 1 every
 * source_rows[s] a multiple of 128 (one router row tile never spans two
 * sources).  Anything else returns MOK_ERR_UNSUPPORTED.
 *
 * T = 0 is an empty batch (n_sources must be 1): every call returns MOK_OK
 * and launches no kernel, and pointers to arrays with T (or T*k) rows may be
 * NULL.  What is still written follows from the definitions with no tokens:
 * mok_route_layout, mok_layout_static and a training mok_moe_forward (into
 * its saved context) set counts to 0 and offsets, pad_offsets to 0;
 * mok_moe_backward sets the three weight gradients and dW_r to 0 (empty
 * sums); the forward, fused and backward calls clear their workspace's status
 * word.  Nothing is enqueued but those memsets.
 */
typedef struct {
    int T, d_model, n_experts, top_k, d_ff;
    int router;                    /* MOK_ROUTER_SOFTMAX | MOK_ROUTER_SIGMOID */
    int dtype;                     /* MOK_BF16 | MOK_MXFP8 (expert GEMM operands) */
    int n_sources;                 /* 1: x is one [T,d] buffer; >1: token t lives in
                                      source s at row r, sources in token order */
    const int *source_rows;        /* host [n_sources] rows per source (NULL if 1) */
    int minibatch_rows;            /* rows per hand-off chunk of the fused forward:
                                      64 | 128 | 256 (0 = from the shape) */
    float gather_sm_fraction;      /* SMs given to the gather/combine role in the
                                      fused forward (0 = automatic; 1 = every CTA
                                      gathers the tokens first, then every CTA runs
                                      the GEMM role -- needs an uncapped ring) */
    size_t ring_bytes;             /* token ring of the fused forward (0 = no cap) */
    unsigned long long wait_limit_ns; /* device spin give-up (0 = 2 s) */
    int fused_cta_pairs;           /* GEMM role of the fused forward on CTA pairs:
                                      MOK_PAIRS_AUTO (from the shape, see
                                      mok_fused_plan), MOK_PAIRS_ON (wherever the
                                      shape allows), MOK_PAIRS_OFF */
    int gemm_cta_pairs;            /* the separate expert FFN (mok_expert_ffn) and
                                      the weight-gradient GEMMs on CTA pairs:
                                      MOK_PAIRS_AUTO (= on) / ON / OFF; pairs
                                      need the tile's dimensions to be
                                      multiples of 256, else one CTA per tile */
} mok_config;

/* Expert weights.  Masters are BF16; the MXFP8 copies are made by
 * mok_quantize_mx from the masters (forward blocking along each forward
 * GEMM's K; "_t" copies are the transposes blocked along the backward dgrad
 * GEMMs' K).  Unused members may be NULL. */
typedef struct {
    const void *w_gate;            /* device BF16 [E, F, d] */
    const void *w_up;              /* device BF16 [E, F, d] */
    const void *w_down;            /* device BF16 [E, d, F] */
    const uint8_t *q_gate, *q_up, *q_down;     /* device E4M3, same shapes */
    const uint32_t *s_gate, *s_up, *s_down;    /* device scales, tile layout */
    const uint8_t *qt_gate, *qt_up;            /* device E4M3 [E, d, F] (W_g^T, W_u^T) */
    const uint8_t *qt_down;                    /* device E4M3 [E, F, d] (W_d^T) */
    const uint32_t *st_gate, *st_up, *st_down; /* device scales of the transposes */
    const void *wt_gate, *wt_up;               /* device BF16 [E, d, F] (BF16 backward) */
    const void *wt_down;                       /* device BF16 [E, F, d] (BF16 backward) */
} mok_weights;

typedef struct {
    void *d_gate;                  /* device BF16 [E, F, d] */
    void *d_up;                    /* device BF16 [E, F, d] */
    void *d_down;                  /* device BF16 [E, d, F] */
} mok_weight_grads;

/* Byte offsets of the fields of the forward's saved context (for backward and
 * for inspection).  All offsets are 256-byte aligned. */
typedef struct {
    size_t ids, gates, sel_scores, counts, offsets, pad_offsets, slot_pos,
           row_tok, row_j, logits, a, b, h, ystage, total;
} mok_ctx_layout;

/* Upper bound on padded expert-ordered rows: S + E*(MOK_ROW_ALIGN-1),
 * rounded up to 256.  Returns 0 on a bad config. */
int64_t mok_max_padded_rows(const mok_config *cfg);

/* Workspace sizes in bytes: fwd_ws for mok_moe_forward and the step calls,
 * saved_ctx for the forward's saved context, bwd_ws for mok_moe_backward.
 * Any output pointer may be NULL. */
int mok_workspace_size(const mok_config *cfg, size_t *fwd_ws, size_t *saved_ctx,
                       size_t *bwd_ws);

/* Offsets of the saved-context fields for this config. */
int mok_saved_ctx_layout(const mok_config *cfg, mok_ctx_layout *out);

/* Byte offsets of the backward workspace's intermediate rows, for
 * inspection after mok_moe_backward: the status word, dy rows (BF16
 * [rows_pad, d], B1's output in the padded expert order), da and db (BF16
 * [rows_pad, F], B2's output), dx rows (BF16 [rows_pad, d], B3's output) and
 * the chosen experts' logit gradients (fp32 [T, k]).  256-byte aligned. */
typedef struct {
    size_t status, dy, da, db, dx, dl_sel, total;
} mok_bwd_layout;
int mok_bwd_ws_layout(const mok_config *cfg, mok_bwd_layout *out);

/*
 * A1 + A2: router top-k and layout ([kucoin] §01: the router decides each
 * token's experts at every step; the layout counts tokens per expert and
 * places one expert's tokens together for the grouped GEMM).
 *   logits = x W_r^T (+ bias); scores = softmax over E (MOK_ROUTER_SOFTMAX)
 *   or sigmoid; top-k by logit, ties to the lower expert id, slot j = 0 the
 *   largest; gates = chosen scores / their sum.  Layout = stable counting
 *   sort of slot t*k+j by expert.
 * x_src      host array [n_sources] of device BF16 [source_rows[s], d]
 * W_r        device fp32 [E, d];  bias device fp32 [E] or NULL
 * ids        device int32 [T, k];   gates device fp32 [T, k]
 * sel_scores device fp32 [T, k] chosen scores (softmax or sigmoid), or NULL
 * logits     device fp32 [T, E] or NULL
 * counts     device int32 [E];  offsets, pad_offsets device int32 [E+1]
 * slot_pos   device int32 [T, k] dense row of slot (t, j)
 * row_tok    device int32 [S];  row_j device uint8 [S]  (dense rows)
 * ws         device workspace of at least fwd_ws bytes
 */
int mok_route_layout(const mok_config *cfg, const void *const *x_src, const float *W_r,
                     const float *bias, int32_t *ids, float *gates, float *sel_scores,
                     float *logits, int32_t *counts, int32_t *offsets,
                     int32_t *pad_offsets, int32_t *slot_pos, int32_t *row_tok,
                     uint8_t *row_j, void *ws, void *stream);

/*
 * A3: pull dispatch ([kucoin] §02: the expert side reads the tokens it needs
 * by (source, position in source) and lays them out in its own expert order;
 * MXFP8 quantisation fused into dispatch).  Row pad_offsets[e] + i of xe is
 * token row_tok[offsets[e] + i].  BF16: xe is BF16 [rows, d].  MXFP8: xe is
 * E4M3 [rows, d] and xe_scales the tile-layout scales (rows =
 * mok_max_padded_rows).  ids/offsets/pad_offsets/row_tok as produced by
 * mok_route_layout.
 */
int mok_dispatch(const mok_config *cfg, const void *const *x_src, const int32_t *ids,
                 const int32_t *offsets, const int32_t *pad_offsets,
                 const int32_t *row_tok, const uint8_t *row_j, void *xe,
                 uint32_t *xe_scales, void *stream);

/*
 * A3 with one read per token: the same bytes as mok_dispatch (xe, and the
 * xe_scales when MXFP8), but each token's row is read from its source once
 * (and quantised once) and written into each of its k slot rows:
 * pad_offsets[e] + slot_pos[t, j] - offsets[e] for e = ids[t, j].  [kucoin]
 * §02's pull with one request per token instead of one per slot (on several
 * GPUs: one pull per token and destination rank, placed into every local
 * expert the token selected).  HBM reads drop from T*k rows to T rows.
 * slot_pos: device int32 [T, k] from mok_route_layout; other arguments as
 * mok_dispatch.
 */
int mok_dispatch_by_token(const mok_config *cfg, const void *const *x_src, const int32_t *ids,
                          const int32_t *slot_pos, const int32_t *offsets,
                          const int32_t *pad_offsets, void *xe, uint32_t *xe_scales, void *stream);

/*
 * A4 + A5: per-expert SwiGLU FFN as grouped GEMMs on the tensor cores
 * ([kucoin] §01: grouped GEMM over organised input; §02: MXFP8 fused into
 * the grouped GEMM and SwiGLU; push combine: each result goes straight to
 * its token).  a = xe W_g^T, b = xe W_u^T (fp32 accumulate), h = silu(a) b
 * stored as BF16 (BF16) or MXFP8 along F (MXFP8), y = h W_d^T stored as
 * BF16 into ystage[row_tok[p], row_j[p]].
 * ystage   device BF16 [T, k, d]
 * saved_a, saved_b, saved_h  device BF16 [rows, F] (padded layout) or NULL
 * ws       device workspace (fwd_ws bytes) holding h
 */
int mok_expert_ffn(const mok_config *cfg, const void *xe, const uint32_t *xe_scales,
                   const mok_weights *w, const int32_t *offsets,
                   const int32_t *pad_offsets, const int32_t *row_tok,
                   const uint8_t *row_j, void *ystage, void *saved_a, void *saved_b,
                   void *saved_h, void *ws, void *stream);

/*
 * A6: final weighted combine ([kucoin] §03).  out[t] = BF16 of the fp32
 * fused multiply-add fold over j = 0..k-1 of gates[t,j] * ystage[t,j],
 * starting from 0 -- a fixed order, so results are bit-reproducible.
 * ystage device BF16 [T,k,d]; gates device fp32 [T,k]; out device BF16 [T,d].
 */
int mok_combine(const mok_config *cfg, const void *ystage, const float *gates,
                void *out, void *stream);

/*
 * A3-A5 as ONE persistent cooperative kernel, then A6 ([kucoin] §02: the megakernel
 * splits the SMs between dispatch/combine/state and the expert FFN, hands
 * minibatches over through on-GPU counters and reuses a fixed-size token ring
 * buffer as soon as the experts are done with it).  From a layout made by
 * mok_route_layout: cfg->gather_sm_fraction of the SMs (0: chosen from the
 * shape, see mok_fused_plan) start pulling rows (quantised when MXFP8) into a
 * token ring of cfg->ring_bytes (0: no cap; it must hold 256 rows) in
 * minibatches of cfg->minibatch_rows (0: chosen from the shape);
 * the other SMs run the FFN1 and FFN2 tiles as rows arrive; the weighted
 * combine follows as the mok_combine kernel on the same stream (launched by
 * this call).  The result is bit-identical to mok_dispatch + mok_expert_ffn +
 * mok_combine for every split, minibatch and ring size.  With a gather share
 * of 1 (uncapped ring only) the call first runs the mok_dispatch_by_token
 * kernel -- each row read once and quantised once, written into its k slot
 * rows -- and the fused kernel then runs the GEMM role on every CTA.  ids/gates/counts/offsets/pad_offsets/slot_pos/row_tok/
 * row_j as produced by mok_route_layout; ystage: device BF16 [T,k,d]; out:
 * device BF16 [T,d]; ws: fwd_ws bytes.  A ring below 256 rows, or a gather
 * share of 1 with a capped ring, returns MOK_ERR_INVALID_ARG; a bounded device
 * wait that runs out sets MOK_ERR_TIMEOUT in the status word.
 */
int mok_moe_fused(const mok_config *cfg, const void *const *x_src, const mok_weights *w,
                  const int32_t *ids, const float *gates, const int32_t *counts,
                  const int32_t *offsets, const int32_t *pad_offsets, const int32_t *slot_pos,
                  const int32_t *row_tok, const uint8_t *row_j, void *ystage, void *out, void *ws,
                  void *stream);

/*
 * The launch plan of the fused forward for this config on the current device,
 * host only (no device work): its CTAs (at most one per SM), whether its
 * GEMM role runs on CTA pairs (1) or one CTA per tile (0), the CTAs that
 * start in the gather role, the minibatch (rows per hand-off) and the token
 * ring's rows.  CTA pairs need d a multiple of 256 and an uncapped ring or
 * one of at least 512 rows; cfg->fused_cta_pairs = MOK_PAIRS_ON / OFF forces
 * either where the shape allows, MOK_PAIRS_AUTO takes them for BF16 layers and
 * for MXFP8 layers whose experts average at least 384 rows (T*k >= 384 E).
 * A knob the config
 * leaves 0 is chosen from the shape ([kucoin] §03: the right minibatch and
 * number of communication SMs change with the hidden size, top-k and expert
 * size; §02: one minibatch should give the expert GEMM two full waves of
 * tiles): gather CTAs from the ratio of the per-row gather time to the
 * per-row FFN1 time on one SM (twice that ratio, within 1/16..1/3 of the
 * SMs; even when the GEMM role runs on CTA pairs); minibatch = the smallest
 * of 64, 128, 256 rows for which one round of the gather role (one
 * minibatch per gather CTA, every 128-row tile released as soon as it has
 * landed) hands over two waves of FFN1 tiles to the GEMM CTAs, else 256.
 * With an uncapped ring and a share of 1/8 of the CTAs or more by that rule,
 * or a config share of 1, every CTA gathers first instead (gather CTAs =
 * CTAs, minibatch 0; see mok_moe_fused).  Any output may be NULL.
 */
int mok_fused_plan(const mok_config *cfg, int *ctas, int *cta_pairs, int *gather_ctas,
                   int *minibatch_rows, int64_t *ring_rows);

/*
 * The whole forward layer: mok_route_layout then the fused persistent kernel
 * of mok_moe_fused, enqueued back to back on one stream with no host round
 * trip.  saved_ctx: device buffer of saved_ctx bytes (training: a, b, h,
 * ystage and the routing are kept for mok_moe_backward) or NULL (inference).
 */
int mok_moe_forward(const mok_config *cfg, const void *const *x_src, const float *W_r,
                    const float *bias, const mok_weights *w, void *out, void *saved_ctx,
                    void *ws, void *stream);

/*
 * n independent forward layer calls back to back, inference (macrobatch
 * pipelining: [kucoin] §02, the token ring lets the combine of one macrobatch
 * overlap the dispatch and expert work of the next).  Call i computes
 * out[i] from x_src[i] exactly as mok_moe_forward (the same bits), with its
 * own workspace ws[i] (fwd_ws bytes).  Call i's weighted combine is not run
 * after its own fused kernel: call i+1's fused kernel runs it, in chunks (one
 * token per epilogue warp) spread among its FFN1 tiles, so the epilogue warps
 * do that HBM-bound work while the same SMs' MMAs run; the last call's combine
 * follows its kernel as in mok_moe_forward.  Everything is
 * enqueued on `stream` in call order, so out[i] is complete once call i+1's
 * kernel has run.  Adjacent calls need different workspaces and outputs (two
 * workspaces alternating suffice); otherwise MOK_ERR_INVALID_ARG.
 * x_src  host array [n] of the calls' host source arrays (as mok_moe_forward)
 * out    host array [n] of device BF16 [T, d];  ws host array [n] of workspaces
 */
int mok_moe_forward_chain(const mok_config *cfg, int n, const void *const *const *x_src,
                          const float *W_r, const float *bias, const mok_weights *w,
                          void *const *out, void *const *ws, void *stream);

/*
 * Backward of mok_moe_forward ([kucoin] §01: backward runs two more rounds
 * of communication in reverse; §02: pull reverse-combine, push
 * reverse-dispatch).  saved_ctx is the forward's saved context (the forward
 * must have been called with it); x_src and W_r are the forward's inputs.
 * MXFP8 layers need w->qt_* / st_* (mok_quantize_mx, transpose = 1); BF16
 * layers need w->wt_* (mok_transpose_bf16).  ws: bwd_ws bytes.
 * Gradients of L = <dY, out>:
 *   dy_slot = g dY[t] (BF16), dgates = <dY[t], y_tj>; dh = dy W_d; SwiGLU
 *   backward with the saved a, b; dx_slot = da W_g + db W_u; dW_d = dy^T h,
 *   dW_g = da^T xe, dW_u = db^T xe per expert (BF16); dlogits through the
 *   renormalised top-k gates; dW_r = dlogits^T x; dX = sum_j dx_slot +
 *   dlogits W_r (BF16).
 * dY device BF16 [T,d]; dX device BF16 [T,d]; dgates device fp32 [T,k];
 * dlogits device fp32 [T,E] or NULL; dW_r device fp32 [E,d].
 */
int mok_moe_backward(const mok_config *cfg, const void *const *x_src, const float *W_r,
                     const void *saved_ctx, const void *dY, const mok_weights *w,
                     void *dX, mok_weight_grads *dw, float *dgates, float *dlogits,
                     float *dW_r, void *ws, void *stream);

/*
 * MXFP8 quantiser (OCP MX v1.0: scale X = clamp(floor(log2 amax) - 8, -127,
 * 127), E8M0 byte X + 127, elements E4M3 round-to-nearest-even of v / 2^X,
 * saturating at +-448).  src is `batch` BF16 matrices [rows, K], rows and K
 * multiples of 128.  transpose = 0: blocks run along K; codes [batch, rows, K],
 * scales in tile layout for a matrix of batch*rows rows and K columns.
 * transpose = 1: each matrix is transposed first; codes [batch, K, rows],
 * scales for batch*K rows and `rows` columns.
 */
int mok_quantize_mx(const void *src, int64_t batch, int64_t rows, int64_t K,
                    int transpose, uint8_t *codes, uint32_t *scales, void *stream);

/*
 * The expert GEMM's SwiGLU and MXFP8 quantisation of h, on fp32 inputs
 * ([kucoin] §02: MXFP8 quantisation fused into SwiGLU).  h = silu(a) * b in
 * fp32, quantised in blocks of 32 along F, by the same device code the FFN1
 * epilogue runs on its fp32 accumulators -- so for given fp32 a, b the codes
 * and scales are the ones the fused forward writes.  For checking the
 * epilogue's quantiser against a reference on known inputs.
 * a, b   device fp32 [rows, F];  h device fp32 [rows, F] (the fp32 SwiGLU
 *        output) or NULL;  codes device E4M3 [rows, F];  scales device, tile
 *        layout for a [rows, F] matrix.  rows and F multiples of 128.
 */
int mok_swiglu_quantize_mx(const float *a, const float *b, int64_t rows, int64_t F, float *h,
                           uint8_t *codes, uint32_t *scales, void *stream);

/* BF16 transpose of `batch` matrices [rows, K] into [K, rows] each (the
 * transposed weights of the BF16 backward).  rows, K >= 1. */
int mok_transpose_bf16(const void *src, int64_t batch, int64_t rows, int64_t K, void *dst,
                       void *stream);

/*
 * Layout step without any caller-provided scratch.  No passage of the pages
 * corresponds to this call: it is a convenience of this library.
 *
 * Who it is for: callers that cannot allocate device memory when they need
 * the layout -- a host callback or a runtime that forbids CUDA API calls that
 * synchronise the device (cudaMalloc and cudaFree may), an embedding that
 * hands the library a fixed set of buffers with a hard memory budget, or a
 * hot path that must not grow its allocator.  mok_route_layout needs a
 * workspace for two per-chunk tables; this call keeps them in one 1 MiB array
 * owned by the library instead, so it needs no workspace at all.
 *
 * Computes exactly what the layout part of mok_route_layout computes, from
 * the routing ids [T, k] (device int32): counts, offsets, pad_offsets,
 * slot_pos, row_tok, row_j, with the same layouts and the same bits.
 *
 * Precondition: every id lies in [0, E).  The kernels check it: an id
 * outside that range is counted for no expert and placed in no row, its
 * slot_pos is set to -1, and offsets[E] is set to -1 instead of T*k (the
 * other outputs then describe the valid slots only).  Check offsets[E]
 * before using the layout when the ids come from outside mok_route_layout.
 *
 * Limit: 2 * ceil(T*k / 256) * E <= 262144 (for example T*k = 131072 slots
 * with E = 256 experts); larger layers return MOK_ERR_UNSUPPORTED and enqueue
 * nothing.  The call itself allocates nothing and calls no allocating
 * routine, with one exception on its first call on each device: it looks up
 * the array's device address with that device current, and under CUDA's lazy
 * module loading (the default) that lookup also loads this part of the
 * library's device code onto the device, which allocates device memory (the
 * 1 MiB array among it) and may synchronise the device.  So make the first
 * call on each device during set-up, before any stream capture and before
 * the point where allocation is not allowed; every later call on that device
 * is allocation-free.  Every GPU that loads the library holds the 1 MiB until
 * the process exits.  All calls on a device share the one array, and each call
 * overwrites what the previous one left there (nothing in it needs to start
 * at zero), so two calls that can run at the same time on the GPU -- on
 * different streams without ordering between them -- race and give wrong
 * results; order them on one stream.
 */
int mok_layout_static(const mok_config *cfg, const int32_t *ids, int32_t *counts,
                      int32_t *offsets, int32_t *pad_offsets, int32_t *slot_pos,
                      int32_t *row_tok, uint8_t *row_j, void *stream);

/* Clears the device status word of a workspace (enqueued on stream). */
int mok_reset_device_status(void *ws, void *stream);

/* Synchronises `stream` and returns the device status word of `ws`:
 * MOK_OK or MOK_ERR_TIMEOUT (a bounded device wait gave up). */
int mok_get_device_status(const void *ws, void *stream);

/* Human-readable name of a status code (static string). */
const char *mok_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOK_H */
