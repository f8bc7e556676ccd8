// mok_internal.h -- declarations shared by the library's translation units:
// the source-buffer table, workspace carving and kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mok.h"

namespace mok {

// Largest source count the per-source tensor-map table of the router GEMM
// carries in its kernel parameters (64 maps = 8 KB of parameters).
constexpr int kMaxRouterSources = 64;

// Token t lives in source s = the last s with row_start[s] <= t, at row
// t - row_start[s].
struct Sources {
    const uint16_t *ptr[MOK_MAX_SOURCES];
    int row_start[MOK_MAX_SOURCES + 1];
    int n;
};

__host__ __device__ inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Byte layout of the forward workspace (all offsets 256-aligned).
struct FwdWs {
    size_t status;          // uint32 status word
    size_t chunk_counts;    // int32 [nchunks, E]
    size_t chunk_base;      // int32 [nchunks, E]
    size_t w3;              // BF16 [E_pad, 3d]: router weights split hi/mid/lo
    size_t route;           // start of the route outputs block (when no saved ctx)
    size_t xe, xe_scales;   // expert-ordered activations (padded rows)
    size_t h, h_scales;     // SwiGLU output (padded rows)
    size_t ystage;          // BF16 [T, k, d] (when no saved ctx)
    size_t counters;        // int32 hand-off counters of the fused forward
    size_t total;
};

struct Dims {
    int T, d, E, k, F;
    int router, dtype;
    int64_t S;              // T * k
    int64_t rows_pad;       // padded expert-ordered rows bound
    int E_pad;              // E rounded up to 128 (router GEMM N)
    int nchunks;            // layout chunks of kLayoutChunk slots
    bool gemm_pairs;        // separate expert FFN / weight-gradient GEMMs may use CTA pairs
};

constexpr int kLayoutChunk = 256;

// Device buffers of the backward (carved from the backward workspace).
struct BwdBufs {
    uint16_t *dy;                 // BF16 [rows_pad, d] dy of each slot row
    uint8_t *dy_q;                // MXFP8 codes of dy along d
    uint32_t *dy_s;
    const uint16_t *saved_a, *saved_b, *saved_h;  // BF16 [rows_pad, F] from the forward
    uint16_t *da, *db;            // BF16 [rows_pad, F]
    uint8_t *da_q, *db_q;         // MXFP8 along F
    uint32_t *da_s, *db_s;
    uint16_t *dx;                 // BF16 [rows_pad, d]
    void *dyT, *hT, *daT, *dbT, *xT;              // [X, rows_pad] wgrad operands
    uint32_t *dyT_s, *hT_s, *daT_s, *dbT_s, *xT_s;
    float *dl_sel;                // [T, k] logit gradients of the chosen experts
};

struct BwdWs {
    size_t status, dy, dy_q, dy_s, da, db, da_q, db_q, da_s, db_s, dx, dyT, hT, daT, dbT, xT,
        dyT_s, hT_s, daT_s, dbT_s, xT_s, dl_sel, total;
};

int check_config(const mok_config *cfg, Dims *dm);
// counts = 0, offsets = pad_offsets = 0 on st (the layout of an empty batch)
int empty_layout(const Dims &dm, int32_t *counts, int32_t *offsets, int32_t *pad_offsets, cudaStream_t st);
void bwd_ws_layout(const Dims &dm, BwdWs *w);
void fwd_ws_layout(const Dims &dm, FwdWs *w);
void ctx_layout(const Dims &dm, mok_ctx_layout *c);
int make_sources(const mok_config *cfg, const Dims &dm, const void *const *x_src, Sources *s);

// ---- launchers (return cudaSuccess or the launch error) ----
cudaError_t launch_router_split(const float *Wr, int E, int E_pad, int d, uint16_t *w3,
                                cudaStream_t st);
cudaError_t launch_router_gemm(const Dims &dm, const Sources &src, const uint16_t *w3,
                               const float *bias, float *logits, uint32_t *status,
                               uint64_t wait_ns, cudaStream_t st);
cudaError_t launch_topk(const Dims &dm, const float *logits, int32_t *ids, float *gates,
                        float *sel_scores, cudaStream_t st);
cudaError_t launch_layout(const Dims &dm, const int32_t *ids, int32_t *counts, int32_t *offsets,
                          int32_t *pad_offsets, int32_t *slot_pos, int32_t *row_tok,
                          uint8_t *row_j, int32_t *chunk_counts, int32_t *chunk_base,
                          cudaStream_t st);
cudaError_t launch_counts_from_offsets(const int32_t *offsets, int E, int32_t *counts,
                                       cudaStream_t st);
cudaError_t launch_dispatch(const Dims &dm, const Sources &src, const int32_t *ids,
                            const int32_t *offsets, const int32_t *pad_offsets,
                            const int32_t *row_tok, const uint8_t *row_j, void *xe,
                            uint32_t *xe_scales, cudaStream_t st);
cudaError_t launch_dispatch_by_token(const Dims &dm, const Sources &src, const int32_t *ids,
                                     const int32_t *slot_pos, const int32_t *offsets,
                                     const int32_t *pad_offsets, void *xe, uint32_t *xe_scales,
                                     cudaStream_t st);
cudaError_t launch_combine(const Dims &dm, const uint16_t *ystage, const float *gates,
                           uint16_t *out, cudaStream_t st);
cudaError_t launch_quant_mx(const uint16_t *src, int64_t batch, int64_t rows, int64_t K,
                            int transpose, uint8_t *codes, uint32_t *scales, cudaStream_t st);
cudaError_t launch_ffn(const Dims &dm, const void *xe, const uint32_t *xe_scales,
                       const mok_weights *w, const int32_t *counts, const int32_t *offsets,
                       const int32_t *pad_offsets, const int32_t *row_tok,
                       const uint8_t *row_j, void *h, uint32_t *h_scales, uint16_t *ystage,
                       uint16_t *saved_a, uint16_t *saved_b, uint16_t *saved_h,
                       uint32_t *status, uint64_t wait_ns, cudaStream_t st);

#ifdef __CUDACC__
__device__ __forceinline__ const uint16_t *source_row(const Sources &src, int t, int d)
{
    int lo = 0, hi = src.n;  // last s with row_start[s] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (src.row_start[mid] <= t) lo = mid;
        else hi = mid;
    }
    return src.ptr[lo] + static_cast<int64_t>(t - src.row_start[lo]) * d;
}
#endif

cudaError_t launch_dgrad(const Dims &dm, const BwdBufs &b, const mok_weights *w,
                         const int32_t *counts, const int32_t *pad_offsets, uint32_t *status,
                         uint64_t wait_ns, cudaStream_t st);
cudaError_t launch_wgrad(const Dims &dm, const void *A_T, const uint32_t *A_s, int64_t a_rows,
                         const void *B_T, const uint32_t *B_s, int64_t b_rows,
                         const int32_t *pad_offsets, uint16_t *dW, uint32_t *status,
                         uint64_t wait_ns, cudaStream_t st);
cudaError_t launch_rev_combine(const Dims &dm, const uint16_t *dY, const float *gates,
                               const float *sel_scores, const int32_t *ids,
                               const int32_t *slot_pos, const int32_t *offsets,
                               const int32_t *pad_offsets, const uint16_t *ystage,
                               const BwdBufs &b, float *dgates, float *dlogits, cudaStream_t st);
cudaError_t launch_transpose_rows(const Dims &dm, const uint16_t *in, const Sources *src, int C,
                                  const int32_t *counts, const int32_t *offsets,
                                  const int32_t *pad_offsets, const int32_t *row_tok, void *out,
                                  uint32_t *out_s, cudaStream_t st);
cudaError_t launch_rev_dispatch(const Dims &dm, const int32_t *ids, const int32_t *slot_pos,
                                const int32_t *offsets, const int32_t *pad_offsets,
                                const uint16_t *dx_rows, const float *dl_sel, const float *W_r,
                                uint16_t *dX, cudaStream_t st);
cudaError_t launch_router_wgrad(const Dims &dm, const Sources &src, const int32_t *offsets,
                                const int32_t *row_tok, const uint8_t *row_j, const float *dl_sel,
                                float *dW_r, cudaStream_t st);
cudaError_t launch_swiglu_quant(const float *a, const float *b, int64_t rows, int64_t F, float *h,
                                uint8_t *codes, uint32_t *scales, cudaStream_t st);
cudaError_t launch_transpose_bf16(const uint16_t *src, int64_t batch, int64_t rows, int64_t K,
                                  uint16_t *dst, cudaStream_t st);

// Buffers of the fused persistent forward.
struct FusedIo {
    const int32_t *ids, *counts, *offsets, *pad_offsets, *slot_pos, *row_tok;
    const uint8_t *row_j;
    const float *gates;
    void *ring;               // token ring (a prefix of the xe buffer)
    uint32_t *ring_scales;
    void *h;
    uint32_t *h_scales;
    uint16_t *ystage, *out, *saved_a, *saved_b, *saved_h;
    int *counters;            // fused_counter_ints(dm) ints
    // chained calls: the previous call's combine (prev_T = 0: none), and whether
    // this call leaves its own combine to the next call
    const uint16_t *prev_ystage;
    const float *prev_gates;
    uint16_t *prev_out;
    int prev_T;
    bool skip_combine;
};
int64_t fused_ring_rows(const Dims &dm, size_t ring_bytes);
// Defaults of the fused forward's knobs when the config leaves them 0.
int auto_gather_ctas(const Dims &dm, int sms);
int auto_minibatch_rows(const Dims &dm, int gather_ctas, int gemm_ctas);
// Whether every CTA gathers the tokens first (a gather share of 1; see fused_knobs).
bool fused_gathers_first(const Dims &dm, const mok_config *cfg, int ctas);
// Whether the fused forward runs its GEMM role on CTA pairs (d a multiple of
// 256 and an uncapped ring or one of at least 4 row tiles, as
// cfg->fused_cta_pairs allows), and its CTAs.
bool fused_uses_pairs(const Dims &dm, const mok_config *cfg);
int fused_ctas(const Dims &dm, const mok_config *cfg, int sms);
// The knobs one fused launch of `ctas` CTAs uses: gather CTAs and minibatch rows
// (gather CTAs == ctas: every CTA gathers the tokens first, then every CTA
// runs the GEMM role; minibatch rows then 0).
void fused_knobs(const Dims &dm, const mok_config *cfg, int ctas, int *gather_ctas, int *minibatch_rows);
int fused_counter_ints(const Dims &dm);
cudaError_t launch_fused(const Dims &dm, const mok_config *cfg, const Sources &src, const FusedIo &io,
                         const mok_weights *w, uint32_t *status, uint64_t wait_ns, cudaStream_t st);

int num_sms();
// Encodes a 2-D tiled tensor map with 128-byte swizzle; returns 0 on success.
int encode_tmap_2d(CUtensorMap *m, const void *base, bool fp8, uint64_t inner_elems,
                   uint64_t rows, uint32_t box_inner, uint32_t box_rows);
// Encodes a map over an MX scale array of a [rows, K] matrix viewed as
// [(K/128) * (rows/128), 128] 32-bit words: map row i is the 512-byte scale
// tile i (k-group i / (rows/128), row tile i % (rows/128)); box = one tile.
int encode_tmap_scales(CUtensorMap *m, const uint32_t *base, uint64_t rows, uint64_t K);

}  // namespace mok
