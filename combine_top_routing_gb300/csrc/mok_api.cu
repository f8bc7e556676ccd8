// mok_api.cu -- the C ABI of libmok.so (declared in include/mok.h): argument
// checks, workspace carving, tensor-map encoding and the order of launches.
// No entry point allocates, frees or synchronises the host, except
// mok_get_device_status, which synchronises by contract.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mok.h"
#include "mok_internal.h"

namespace mok {

static constexpr size_t kAlign = 256;

static size_t take(size_t *cursor, size_t bytes)
{
    const size_t off = (*cursor + kAlign - 1) / kAlign * kAlign;
    *cursor = off + bytes;
    return off;
}

int check_config(const mok_config *cfg, Dims *dm)
{
    if (!cfg) return MOK_ERR_INVALID_ARG;
    const int T = cfg->T, d = cfg->d_model, E = cfg->n_experts, k = cfg->top_k, F = cfg->d_ff;
    // T = 0 is an empty batch: every call is then a no-op apart from the
    // per-expert outputs it defines (see empty_layout and mok_moe_backward)
    if (T < 0 || d < 1 || E < 1 || k < 1 || F < 1) return MOK_ERR_INVALID_ARG;
    if (T == 0 && cfg->n_sources != 1) return MOK_ERR_INVALID_ARG;
    if (cfg->router != MOK_ROUTER_SOFTMAX && cfg->router != MOK_ROUTER_SIGMOID) return MOK_ERR_INVALID_ARG;
    if (cfg->dtype != MOK_BF16 && cfg->dtype != MOK_MXFP8) return MOK_ERR_INVALID_ARG;
    if (cfg->n_sources < 1 || cfg->n_sources > MOK_MAX_SOURCES) return MOK_ERR_INVALID_ARG;
    if (cfg->n_sources > 1 && !cfg->source_rows) return MOK_ERR_INVALID_ARG;
    if (cfg->minibatch_rows != 0 && cfg->minibatch_rows != 64 && cfg->minibatch_rows != 128 &&
        cfg->minibatch_rows != 256)
        return MOK_ERR_INVALID_ARG;
    if (!(cfg->gather_sm_fraction >= 0.0f && cfg->gather_sm_fraction <= 1.0f)) return MOK_ERR_INVALID_ARG;
    for (const int v : {cfg->fused_cta_pairs, cfg->gemm_cta_pairs})
        if (v != MOK_PAIRS_AUTO && v != MOK_PAIRS_ON && v != MOK_PAIRS_OFF) return MOK_ERR_INVALID_ARG;
    if (E > MOK_MAX_EXPERTS || k > MOK_MAX_TOPK || k > E) return MOK_ERR_UNSUPPORTED;
    if (d % 128 != 0 || F % 128 != 0) return MOK_ERR_UNSUPPORTED;
    const int64_t S = static_cast<int64_t>(T) * k;
    if (S + static_cast<int64_t>(E) * MOK_ROW_ALIGN > (int64_t{1} << 31) - 1) return MOK_ERR_UNSUPPORTED;
    if (cfg->n_sources > 1) {
        int64_t sum = 0;
        for (int s = 0; s < cfg->n_sources; ++s) {
            if (cfg->source_rows[s] < 1) return MOK_ERR_INVALID_ARG;
            if (cfg->source_rows[s] % 128 != 0) return MOK_ERR_UNSUPPORTED;
            sum += cfg->source_rows[s];
        }
        if (sum != T) return MOK_ERR_INVALID_ARG;
    }
    if (dm) {
        dm->T = T;
        dm->d = d;
        dm->E = E;
        dm->k = k;
        dm->F = F;
        dm->router = cfg->router;
        dm->dtype = cfg->dtype;
        dm->S = S;
        dm->rows_pad = round_up(S + static_cast<int64_t>(E) * (MOK_ROW_ALIGN - 1), 256);
        dm->E_pad = static_cast<int>(round_up(E, 128));
        dm->nchunks = static_cast<int>((S + kLayoutChunk - 1) / kLayoutChunk);
        dm->gemm_pairs = cfg->gemm_cta_pairs != MOK_PAIRS_OFF;
    }
    return MOK_OK;
}

void ctx_layout(const Dims &dm, mok_ctx_layout *c)
{
    size_t cur = 0;
    const size_t S = static_cast<size_t>(dm.S);
    c->ids = take(&cur, S * 4);
    c->gates = take(&cur, S * 4);
    c->sel_scores = take(&cur, S * 4);
    c->counts = take(&cur, static_cast<size_t>(dm.E) * 4);
    c->offsets = take(&cur, static_cast<size_t>(dm.E + 1) * 4);
    c->pad_offsets = take(&cur, static_cast<size_t>(dm.E + 1) * 4);
    c->slot_pos = take(&cur, S * 4);
    c->row_tok = take(&cur, S * 4);
    c->row_j = take(&cur, S);
    c->logits = take(&cur, static_cast<size_t>(dm.T) * dm.E * 4);
    const size_t rowsF = static_cast<size_t>(dm.rows_pad) * dm.F * 2;
    c->a = take(&cur, rowsF);
    c->b = take(&cur, rowsF);
    c->h = take(&cur, rowsF);
    c->ystage = take(&cur, S * dm.d * 2);
    c->total = (cur + kAlign - 1) / kAlign * kAlign;
}

void fwd_ws_layout(const Dims &dm, FwdWs *w)
{
    size_t cur = 0;
    const size_t esize = dm.dtype == MOK_MXFP8 ? 1 : 2;
    w->status = take(&cur, 256);
    w->chunk_counts = take(&cur, static_cast<size_t>(dm.nchunks) * dm.E * 4);
    w->chunk_base = take(&cur, static_cast<size_t>(dm.nchunks) * dm.E * 4);
    w->w3 = take(&cur, static_cast<size_t>(dm.E_pad) * 3 * dm.d * 2);
    mok_ctx_layout c;
    ctx_layout(dm, &c);
    w->route = take(&cur, c.a);  // ids .. logits, same sub-layout as the saved context
    w->xe = take(&cur, static_cast<size_t>(dm.rows_pad) * dm.d * esize);
    w->xe_scales = take(&cur, dm.dtype == MOK_MXFP8 ? static_cast<size_t>(dm.rows_pad) * dm.d / 32 : 0);
    w->h = take(&cur, static_cast<size_t>(dm.rows_pad) * dm.F * esize);
    w->h_scales = take(&cur, dm.dtype == MOK_MXFP8 ? static_cast<size_t>(dm.rows_pad) * dm.F / 32 : 0);
    w->ystage = take(&cur, static_cast<size_t>(dm.S) * dm.d * 2);
    w->counters = take(&cur, static_cast<size_t>(fused_counter_ints(dm)) * 4);
    w->total = (cur + kAlign - 1) / kAlign * kAlign;
}

void bwd_ws_layout(const Dims &dm, BwdWs *w)
{
    size_t cur = 0;
    const bool mx = dm.dtype == MOK_MXFP8;
    const size_t R = static_cast<size_t>(dm.rows_pad), d = dm.d, F = dm.F;
    const size_t esize = mx ? 1 : 2;
    w->status = take(&cur, 256);
    w->dy = take(&cur, R * d * 2);
    w->dy_q = take(&cur, mx ? R * d : 0);
    w->dy_s = take(&cur, mx ? R * d / 32 : 0);
    w->da = take(&cur, R * F * 2);
    w->db = take(&cur, R * F * 2);
    w->da_q = take(&cur, mx ? R * F : 0);
    w->db_q = take(&cur, mx ? R * F : 0);
    w->da_s = take(&cur, mx ? R * F / 32 : 0);
    w->db_s = take(&cur, mx ? R * F / 32 : 0);
    w->dx = take(&cur, R * d * 2);
    w->dyT = take(&cur, d * R * esize);
    w->hT = take(&cur, F * R * esize);
    w->daT = take(&cur, F * R * esize);
    w->dbT = take(&cur, F * R * esize);
    w->xT = take(&cur, d * R * esize);
    w->dyT_s = take(&cur, mx ? d * R / 32 : 0);
    w->hT_s = take(&cur, mx ? F * R / 32 : 0);
    w->daT_s = take(&cur, mx ? F * R / 32 : 0);
    w->dbT_s = take(&cur, mx ? F * R / 32 : 0);
    w->xT_s = take(&cur, mx ? d * R / 32 : 0);
    w->dl_sel = take(&cur, static_cast<size_t>(dm.S) * 4);
    w->total = (cur + kAlign - 1) / kAlign * kAlign;
}

int make_sources(const mok_config *cfg, const Dims &dm, const void *const *x_src, Sources *s)
{
    if (!x_src) return MOK_ERR_INVALID_ARG;
    s->n = cfg->n_sources;
    int run = 0;
    for (int i = 0; i < s->n; ++i) {
        if (!x_src[i]) return MOK_ERR_INVALID_ARG;
        s->ptr[i] = static_cast<const uint16_t *>(x_src[i]);
        s->row_start[i] = run;
        run += s->n == 1 ? dm.T : cfg->source_rows[i];
    }
    s->row_start[s->n] = run;
    return MOK_OK;
}

int num_sms()
{
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int encode_tmap_2d(CUtensorMap *m, const void *base, bool fp8, uint64_t inner_elems,
                   uint64_t rows, uint32_t box_inner, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15)) return 1;
    const uint64_t esize = fp8 ? 1 : 2;
    cuuint64_t dims[2] = {inner_elems, rows};
    cuuint64_t strides[1] = {inner_elems * esize};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 1;
}

int encode_tmap_scales(CUtensorMap *m, const uint32_t *base, uint64_t rows, uint64_t K)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15) || rows % 128 || K % 128) return 1;
    cuuint64_t dims[2] = {128, (K / 128) * (rows / 128)};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 1;
}

static uint64_t wait_ns(const mok_config *cfg)
{
    return cfg->wait_limit_ns ? cfg->wait_limit_ns : 2000000000ull;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA; }

// The layout of an empty batch: no expert has a row, every offset is 0.
int empty_layout(const Dims &dm, int32_t *counts, int32_t *offsets, int32_t *pad_offsets, cudaStream_t st)
{
    if (!counts || !offsets || !pad_offsets) return MOK_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(counts, 0, static_cast<size_t>(dm.E) * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, static_cast<size_t>(dm.E + 1) * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(pad_offsets, 0, static_cast<size_t>(dm.E + 1) * 4, st);
    return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}

template <typename T>
static T *at(void *base, size_t off)
{
    return reinterpret_cast<T *>(static_cast<uint8_t *>(base) + off);
}

struct RouteOut {
    int32_t *ids;
    float *gates, *sel_scores, *logits;
    int32_t *counts, *offsets, *pad_offsets, *slot_pos, *row_tok;
    uint8_t *row_j;
};

static RouteOut route_in(void *base, const mok_ctx_layout &c)
{
    RouteOut r;
    r.ids = at<int32_t>(base, c.ids);
    r.gates = at<float>(base, c.gates);
    r.sel_scores = at<float>(base, c.sel_scores);
    r.logits = at<float>(base, c.logits);
    r.counts = at<int32_t>(base, c.counts);
    r.offsets = at<int32_t>(base, c.offsets);
    r.pad_offsets = at<int32_t>(base, c.pad_offsets);
    r.slot_pos = at<int32_t>(base, c.slot_pos);
    r.row_tok = at<int32_t>(base, c.row_tok);
    r.row_j = at<uint8_t>(base, c.row_j);
    return r;
}

static int route_layout_impl(const mok_config *cfg, const Dims &dm, const Sources &src,
                             const float *W_r, const float *bias, const RouteOut &o, void *ws,
                             cudaStream_t st)
{
    FwdWs w;
    fwd_ws_layout(dm, &w);
    uint16_t *w3 = at<uint16_t>(ws, w.w3);
    cudaError_t e = launch_router_split(W_r, dm.E, dm.E_pad, dm.d, w3, st);
    if (e == cudaSuccess)
        e = launch_router_gemm(dm, src, w3, bias, o.logits, at<uint32_t>(ws, w.status), wait_ns(cfg), st);
    if (e == cudaSuccess) e = launch_topk(dm, o.logits, o.ids, o.gates, o.sel_scores, st);
    if (e == cudaSuccess)
        e = launch_layout(dm, o.ids, o.counts, o.offsets, o.pad_offsets, o.slot_pos, o.row_tok,
                          o.row_j, at<int32_t>(ws, w.chunk_counts), at<int32_t>(ws, w.chunk_base), st);
    return cuda_status(e);
}

}  // namespace mok

using namespace mok;

extern "C" {

int64_t mok_max_padded_rows(const mok_config *cfg)
{
    Dims dm;
    if (check_config(cfg, &dm) != MOK_OK) return 0;
    return dm.rows_pad;
}

int mok_workspace_size(const mok_config *cfg, size_t *fwd_ws, size_t *saved_ctx, size_t *bwd_ws)
{
    Dims dm;
    const int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    FwdWs w;
    fwd_ws_layout(dm, &w);
    mok_ctx_layout c;
    ctx_layout(dm, &c);
    BwdWs bw;
    bwd_ws_layout(dm, &bw);
    if (fwd_ws) *fwd_ws = w.total;
    if (saved_ctx) *saved_ctx = c.total;
    if (bwd_ws) *bwd_ws = bw.total;
    return MOK_OK;
}

int mok_saved_ctx_layout(const mok_config *cfg, mok_ctx_layout *out)
{
    Dims dm;
    const int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    if (!out) return MOK_ERR_INVALID_ARG;
    ctx_layout(dm, out);
    return MOK_OK;
}

int mok_route_layout(const mok_config *cfg, const void *const *x_src, const float *W_r,
                     const float *bias, int32_t *ids, float *gates, float *sel_scores,
                     float *logits, int32_t *counts, int32_t *offsets, int32_t *pad_offsets,
                     int32_t *slot_pos, int32_t *row_tok, uint8_t *row_j, void *ws, void *stream)
{
    Dims dm;
    int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    if (dm.T == 0) return empty_layout(dm, counts, offsets, pad_offsets, static_cast<cudaStream_t>(stream));
    if (!W_r || !ids || !gates || !counts || !offsets || !pad_offsets || !slot_pos || !row_tok ||
        !row_j || !ws)
        return MOK_ERR_INVALID_ARG;
    Sources src;
    if ((rc = make_sources(cfg, dm, x_src, &src)) != MOK_OK) return rc;
    FwdWs w;
    fwd_ws_layout(dm, &w);
    mok_ctx_layout c;
    ctx_layout(dm, &c);
    RouteOut o;
    o.ids = ids;
    o.gates = gates;
    o.sel_scores = sel_scores ? sel_scores : at<float>(ws, w.route + c.sel_scores);
    o.logits = logits ? logits : at<float>(ws, w.route + c.logits);
    o.counts = counts;
    o.offsets = offsets;
    o.pad_offsets = pad_offsets;
    o.slot_pos = slot_pos;
    o.row_tok = row_tok;
    o.row_j = row_j;
    return route_layout_impl(cfg, dm, src, W_r, bias, o, ws, static_cast<cudaStream_t>(stream));
}

int mok_dispatch(const mok_config *cfg, const void *const *x_src, const int32_t *ids,
                 const int32_t *offsets, const int32_t *pad_offsets, const int32_t *row_tok,
                 const uint8_t *row_j, void *xe, uint32_t *xe_scales, void *stream)
{
    Dims dm;
    int rc = check_config(cfg, &dm);
    if (rc != MOK_OK || dm.T == 0) return rc;
    if (!ids || !offsets || !pad_offsets || !row_tok || !row_j || !xe) return MOK_ERR_INVALID_ARG;
    if (dm.dtype == MOK_MXFP8 && !xe_scales) return MOK_ERR_INVALID_ARG;
    Sources src;
    if ((rc = make_sources(cfg, dm, x_src, &src)) != MOK_OK) return rc;
    return cuda_status(launch_dispatch(dm, src, ids, offsets, pad_offsets, row_tok, row_j, xe,
                                       xe_scales, static_cast<cudaStream_t>(stream)));
}

int mok_dispatch_by_token(const mok_config *cfg, const void *const *x_src, const int32_t *ids,
                          const int32_t *slot_pos, const int32_t *offsets, const int32_t *pad_offsets,
                          void *xe, uint32_t *xe_scales, void *stream)
{
    Dims dm;
    int rc = check_config(cfg, &dm);
    if (rc != MOK_OK || dm.T == 0) return rc;
    if (!ids || !slot_pos || !offsets || !pad_offsets || !xe) return MOK_ERR_INVALID_ARG;
    if (dm.dtype == MOK_MXFP8 && !xe_scales) return MOK_ERR_INVALID_ARG;
    Sources src;
    if ((rc = make_sources(cfg, dm, x_src, &src)) != MOK_OK) return rc;
    return cuda_status(launch_dispatch_by_token(dm, src, ids, slot_pos, offsets, pad_offsets, xe, xe_scales,
                                                static_cast<cudaStream_t>(stream)));
}

int mok_expert_ffn(const mok_config *cfg, const void *xe, const uint32_t *xe_scales,
                   const mok_weights *w, const int32_t *offsets, const int32_t *pad_offsets,
                   const int32_t *row_tok, const uint8_t *row_j, void *ystage, void *saved_a,
                   void *saved_b, void *saved_h, void *ws, void *stream)
{
    Dims dm;
    int rc = check_config(cfg, &dm);
    if (rc != MOK_OK || dm.T == 0) return rc;
    if (!xe || !w || !offsets || !pad_offsets || !row_tok || !row_j || !ystage || !ws)
        return MOK_ERR_INVALID_ARG;
    const bool mx = dm.dtype == MOK_MXFP8;
    if (mx && (!xe_scales || !w->q_gate || !w->q_up || !w->q_down || !w->s_gate || !w->s_up || !w->s_down))
        return MOK_ERR_INVALID_ARG;
    if (!mx && (!w->w_gate || !w->w_up || !w->w_down)) return MOK_ERR_INVALID_ARG;
    FwdWs fw;
    fwd_ws_layout(dm, &fw);
    // per-expert counts follow from the dense offsets; derive them into ws
    mok_ctx_layout c;
    ctx_layout(dm, &c);
    int32_t *counts = at<int32_t>(ws, fw.route + c.counts);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_counts_from_offsets(offsets, dm.E, counts, st);
    if (e == cudaSuccess)
        e = launch_ffn(dm, xe, xe_scales, w, counts, offsets, pad_offsets, row_tok, row_j,
                       at<void>(ws, fw.h), mx ? at<uint32_t>(ws, fw.h_scales) : nullptr,
                       static_cast<uint16_t *>(ystage), static_cast<uint16_t *>(saved_a),
                       static_cast<uint16_t *>(saved_b), static_cast<uint16_t *>(saved_h),
                       at<uint32_t>(ws, fw.status), wait_ns(cfg), st);
    return cuda_status(e);
}

int mok_combine(const mok_config *cfg, const void *ystage, const float *gates, void *out,
                void *stream)
{
    Dims dm;
    const int rc = check_config(cfg, &dm);
    if (rc != MOK_OK || dm.T == 0) return rc;
    if (!ystage || !gates || !out) return MOK_ERR_INVALID_ARG;
    return cuda_status(launch_combine(dm, static_cast<const uint16_t *>(ystage), gates,
                                      static_cast<uint16_t *>(out), static_cast<cudaStream_t>(stream)));
}

namespace {

// The previous call of a chain, whose combine the next call's fused kernel runs.
struct ChainPrev {
    const uint16_t *ystage = nullptr;
    const float *gates = nullptr;
    uint16_t *out = nullptr;
    int T = 0;
};

int check_forward_args(const mok_config *cfg, Dims *dm, const float *W_r, const mok_weights *w,
                       const void *out, const void *ws)
{
    int rc = check_config(cfg, dm);
    if (rc != MOK_OK) return rc;
    if (!W_r || !w || (!out && dm->T > 0) || !ws) return MOK_ERR_INVALID_ARG;
    const bool mx = dm->dtype == MOK_MXFP8;
    if (mx && (!w->q_gate || !w->q_up || !w->q_down || !w->s_gate || !w->s_up || !w->s_down))
        return MOK_ERR_INVALID_ARG;
    if (!mx && (!w->w_gate || !w->w_up || !w->w_down)) return MOK_ERR_INVALID_ARG;
    // the token ring must hold at least one minibatch of every size (256 rows)
    const int64_t ring_rows = fused_ring_rows(*dm, cfg->ring_bytes);
    if (ring_rows < 256) return MOK_ERR_INVALID_ARG;
    // every CTA gathering first needs a ring that holds every row
    if (cfg->gather_sm_fraction >= 1.0f && ring_rows < dm->rows_pad) return MOK_ERR_INVALID_ARG;
    return MOK_OK;
}

// Router + layout, then the fused kernel; `prev` / `skip_combine` chain calls.
int forward_impl(const mok_config *cfg, const Dims &dm, const Sources &src, const float *W_r,
                 const float *bias, const mok_weights *w, void *out, void *saved_ctx, void *ws,
                 cudaStream_t st, const ChainPrev &prev, bool skip_combine, const float **gates_out,
                 uint16_t **ystage_out)
{
    const bool mx = dm.dtype == MOK_MXFP8;
    FwdWs fw;
    fwd_ws_layout(dm, &fw);
    mok_ctx_layout c;
    ctx_layout(dm, &c);
    void *rbase = saved_ctx ? saved_ctx : at<void>(ws, fw.route);
    RouteOut o = route_in(rbase, c);
    uint16_t *ystage = saved_ctx ? at<uint16_t>(saved_ctx, c.ystage) : at<uint16_t>(ws, fw.ystage);
    uint32_t *status = at<uint32_t>(ws, fw.status);
    cudaError_t e = cudaMemsetAsync(status, 0, 4, st);
    if (e != cudaSuccess) return MOK_ERR_CUDA;
    if (gates_out) *gates_out = o.gates;
    if (ystage_out) *ystage_out = ystage;
    // an empty batch: the saved routing says that no expert has a row
    if (dm.T == 0) return saved_ctx ? empty_layout(dm, o.counts, o.offsets, o.pad_offsets, st) : MOK_OK;
    int rc = route_layout_impl(cfg, dm, src, W_r, bias, o, ws, st);
    if (rc != MOK_OK) return rc;
    // dispatch, expert FFN and combine: one persistent kernel (role split,
    // token ring, on-GPU hand-off counters)
    FusedIo io = {};
    io.ids = o.ids;
    io.counts = o.counts;
    io.offsets = o.offsets;
    io.pad_offsets = o.pad_offsets;
    io.slot_pos = o.slot_pos;
    io.row_tok = o.row_tok;
    io.row_j = o.row_j;
    io.gates = o.gates;
    io.ring = at<void>(ws, fw.xe);
    io.ring_scales = mx ? at<uint32_t>(ws, fw.xe_scales) : nullptr;
    io.h = at<void>(ws, fw.h);
    io.h_scales = mx ? at<uint32_t>(ws, fw.h_scales) : nullptr;
    io.ystage = ystage;
    io.out = static_cast<uint16_t *>(out);
    io.saved_a = saved_ctx ? at<uint16_t>(saved_ctx, c.a) : nullptr;
    io.saved_b = saved_ctx ? at<uint16_t>(saved_ctx, c.b) : nullptr;
    io.saved_h = saved_ctx ? at<uint16_t>(saved_ctx, c.h) : nullptr;
    io.counters = at<int>(ws, fw.counters);
    io.prev_ystage = prev.ystage;
    io.prev_gates = prev.gates;
    io.prev_out = prev.out;
    io.prev_T = prev.T;
    io.skip_combine = skip_combine;
    return cuda_status(launch_fused(dm, cfg, src, io, w, status, wait_ns(cfg), st));
}

}  // namespace

int mok_moe_forward(const mok_config *cfg, const void *const *x_src, const float *W_r,
                    const float *bias, const mok_weights *w, void *out, void *saved_ctx, void *ws,
                    void *stream)
{
    Dims dm;
    int rc = check_forward_args(cfg, &dm, W_r, w, out, ws);
    if (rc != MOK_OK) return rc;
    Sources src = {};
    if (dm.T > 0 && (rc = make_sources(cfg, dm, x_src, &src)) != MOK_OK) return rc;
    return forward_impl(cfg, dm, src, W_r, bias, w, out, saved_ctx, ws, static_cast<cudaStream_t>(stream),
                        ChainPrev(), false, nullptr, nullptr);
}

int mok_moe_forward_chain(const mok_config *cfg, int n, const void *const *const *x_src,
                          const float *W_r, const float *bias, const mok_weights *w,
                          void *const *out, void *const *ws, void *stream)
{
    Dims dm;
    if (n < 1 || !x_src || !out || !ws) return MOK_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const int rc = check_forward_args(cfg, &dm, W_r, w, out[i], ws[i]);
        if (rc != MOK_OK) return rc;
        Sources src;
        const int rs = dm.T > 0 ? make_sources(cfg, dm, x_src[i], &src) : MOK_OK;
        if (rs != MOK_OK) return rs;
        // call i's combine runs in call i + 1's kernel from call i's workspace
        if (i > 0 && (ws[i] == ws[i - 1] || (dm.T > 0 && out[i] == out[i - 1]))) return MOK_ERR_INVALID_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ChainPrev prev;
    for (int i = 0; i < n; ++i) {
        Sources src = {};
        if (dm.T > 0) make_sources(cfg, dm, x_src[i], &src);
        const float *gates = nullptr;
        uint16_t *ystage = nullptr;
        const int rc = forward_impl(cfg, dm, src, W_r, bias, w, out[i], nullptr, ws[i], st, prev, i + 1 < n,
                                    &gates, &ystage);
        if (rc != MOK_OK) return rc;
        prev.ystage = ystage;
        prev.gates = gates;
        prev.out = static_cast<uint16_t *>(out[i]);
        prev.T = dm.T;
    }
    return MOK_OK;
}

int mok_fused_plan(const mok_config *cfg, int *ctas, int *cta_pairs, int *gather_ctas,
                   int *minibatch_rows, int64_t *ring_rows)
{
    Dims dm;
    const int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    int ng, mb;
    const int grid = fused_ctas(dm, cfg, num_sms());
    fused_knobs(dm, cfg, grid, &ng, &mb);
    if (ctas) *ctas = grid;
    if (cta_pairs) *cta_pairs = fused_uses_pairs(dm, cfg) ? 1 : 0;
    if (gather_ctas) *gather_ctas = ng;
    if (minibatch_rows) *minibatch_rows = mb;
    if (ring_rows) *ring_rows = fused_ring_rows(dm, cfg->ring_bytes);
    return MOK_OK;
}

int mok_moe_fused(const mok_config *cfg, const void *const *x_src, const mok_weights *w,
                  const int32_t *ids, const float *gates, const int32_t *counts,
                  const int32_t *offsets, const int32_t *pad_offsets, const int32_t *slot_pos,
                  const int32_t *row_tok, const uint8_t *row_j, void *ystage, void *out, void *ws,
                  void *stream)
{
    Dims dm;
    int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    if (dm.T == 0) {
        // an empty batch: nothing to move or compute; the status word reads OK
        if (!ws) return MOK_ERR_INVALID_ARG;
        FwdWs fw;
        fwd_ws_layout(dm, &fw);
        return cuda_status(cudaMemsetAsync(at<uint32_t>(ws, fw.status), 0, 4, static_cast<cudaStream_t>(stream)));
    }
    if (!w || !ids || !gates || !counts || !offsets || !pad_offsets || !slot_pos || !row_tok ||
        !row_j || !ystage || !out || !ws)
        return MOK_ERR_INVALID_ARG;
    const bool mx = dm.dtype == MOK_MXFP8;
    if (mx && (!w->q_gate || !w->q_up || !w->q_down || !w->s_gate || !w->s_up || !w->s_down))
        return MOK_ERR_INVALID_ARG;
    if (!mx && (!w->w_gate || !w->w_up || !w->w_down)) return MOK_ERR_INVALID_ARG;
    if (fused_ring_rows(dm, cfg->ring_bytes) < 256) return MOK_ERR_INVALID_ARG;
    if (cfg->gather_sm_fraction >= 1.0f && fused_ring_rows(dm, cfg->ring_bytes) < dm.rows_pad)
        return MOK_ERR_INVALID_ARG;
    Sources src;
    if ((rc = make_sources(cfg, dm, x_src, &src)) != MOK_OK) return rc;
    FwdWs fw;
    fwd_ws_layout(dm, &fw);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *status = at<uint32_t>(ws, fw.status);
    if (cudaMemsetAsync(status, 0, 4, st) != cudaSuccess) return MOK_ERR_CUDA;
    FusedIo io = {};
    io.ids = ids;
    io.counts = counts;
    io.offsets = offsets;
    io.pad_offsets = pad_offsets;
    io.slot_pos = slot_pos;
    io.row_tok = row_tok;
    io.row_j = row_j;
    io.gates = gates;
    io.ring = at<void>(ws, fw.xe);
    io.ring_scales = mx ? at<uint32_t>(ws, fw.xe_scales) : nullptr;
    io.h = at<void>(ws, fw.h);
    io.h_scales = mx ? at<uint32_t>(ws, fw.h_scales) : nullptr;
    io.ystage = static_cast<uint16_t *>(ystage);
    io.out = static_cast<uint16_t *>(out);
    io.counters = at<int>(ws, fw.counters);
    return cuda_status(launch_fused(dm, cfg, src, io, w, status, wait_ns(cfg), st));
}

int mok_moe_backward(const mok_config *cfg, const void *const *x_src, const float *W_r,
                     const void *saved_ctx, const void *dY, const mok_weights *w, void *dX,
                     mok_weight_grads *dw, float *dgates, float *dlogits, float *dW_r, void *ws,
                     void *stream)
{
    Dims dm;
    int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    if (dm.T == 0) {
        // an empty batch: every weight gradient is an empty sum, so zero
        if (!dw || !dw->d_gate || !dw->d_up || !dw->d_down || !dW_r || !ws) return MOK_ERR_INVALID_ARG;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        BwdWs bw;
        bwd_ws_layout(dm, &bw);
        const size_t wbytes = static_cast<size_t>(dm.E) * dm.F * dm.d * 2;
        cudaError_t e = cudaMemsetAsync(at<uint32_t>(ws, bw.status), 0, 4, st);
        for (void *g : {dw->d_gate, dw->d_up, dw->d_down})
            if (e == cudaSuccess) e = cudaMemsetAsync(g, 0, wbytes, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dW_r, 0, static_cast<size_t>(dm.E) * dm.d * 4, st);
        return cuda_status(e);
    }
    if (!W_r || !saved_ctx || !dY || !w || !dX || !dw || !dw->d_gate || !dw->d_up || !dw->d_down ||
        !dgates || !dW_r || !ws)
        return MOK_ERR_INVALID_ARG;
    const bool mx = dm.dtype == MOK_MXFP8;
    if (mx && (!w->qt_gate || !w->qt_up || !w->qt_down || !w->st_gate || !w->st_up || !w->st_down))
        return MOK_ERR_INVALID_ARG;
    if (!mx && (!w->wt_gate || !w->wt_up || !w->wt_down)) return MOK_ERR_INVALID_ARG;
    Sources src;
    if ((rc = make_sources(cfg, dm, x_src, &src)) != MOK_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    mok_ctx_layout c;
    ctx_layout(dm, &c);
    BwdWs bw;
    bwd_ws_layout(dm, &bw);
    void *ctx = const_cast<void *>(saved_ctx);
    RouteOut o = route_in(ctx, c);
    BwdBufs b;
    b.dy = at<uint16_t>(ws, bw.dy);
    b.dy_q = at<uint8_t>(ws, bw.dy_q);
    b.dy_s = at<uint32_t>(ws, bw.dy_s);
    b.saved_a = at<uint16_t>(ctx, c.a);
    b.saved_b = at<uint16_t>(ctx, c.b);
    b.saved_h = at<uint16_t>(ctx, c.h);
    b.da = at<uint16_t>(ws, bw.da);
    b.db = at<uint16_t>(ws, bw.db);
    b.da_q = at<uint8_t>(ws, bw.da_q);
    b.db_q = at<uint8_t>(ws, bw.db_q);
    b.da_s = at<uint32_t>(ws, bw.da_s);
    b.db_s = at<uint32_t>(ws, bw.db_s);
    b.dx = at<uint16_t>(ws, bw.dx);
    b.dyT = at<void>(ws, bw.dyT);
    b.hT = at<void>(ws, bw.hT);
    b.daT = at<void>(ws, bw.daT);
    b.dbT = at<void>(ws, bw.dbT);
    b.xT = at<void>(ws, bw.xT);
    b.dyT_s = at<uint32_t>(ws, bw.dyT_s);
    b.hT_s = at<uint32_t>(ws, bw.hT_s);
    b.daT_s = at<uint32_t>(ws, bw.daT_s);
    b.dbT_s = at<uint32_t>(ws, bw.dbT_s);
    b.xT_s = at<uint32_t>(ws, bw.xT_s);
    b.dl_sel = at<float>(ws, bw.dl_sel);
    uint32_t *status = at<uint32_t>(ws, bw.status);
    const uint64_t wns = wait_ns(cfg);
    cudaError_t e = cudaMemsetAsync(status, 0, 4, st);
    // B1 reverse combine (+ gate and chosen-logit gradients)
    if (e == cudaSuccess)
        e = launch_rev_combine(dm, static_cast<const uint16_t *>(dY), o.gates, o.sel_scores, o.ids,
                               o.slot_pos, o.offsets, o.pad_offsets, at<uint16_t>(ctx, c.ystage), b,
                               dgates, dlogits, st);
    // B2 + B3 dgrad GEMMs
    if (e == cudaSuccess) e = launch_dgrad(dm, b, w, o.counts, o.pad_offsets, status, wns, st);
    // B4 wgrad operands (token dimension innermost) and GEMMs
    if (e == cudaSuccess)
        e = launch_transpose_rows(dm, b.dy, nullptr, dm.d, o.counts, o.offsets, o.pad_offsets,
                                  o.row_tok, b.dyT, b.dyT_s, st);
    if (e == cudaSuccess)
        e = launch_transpose_rows(dm, b.saved_h, nullptr, dm.F, o.counts, o.offsets, o.pad_offsets,
                                  o.row_tok, b.hT, b.hT_s, st);
    if (e == cudaSuccess)
        e = launch_transpose_rows(dm, b.da, nullptr, dm.F, o.counts, o.offsets, o.pad_offsets,
                                  o.row_tok, b.daT, b.daT_s, st);
    if (e == cudaSuccess)
        e = launch_transpose_rows(dm, b.db, nullptr, dm.F, o.counts, o.offsets, o.pad_offsets,
                                  o.row_tok, b.dbT, b.dbT_s, st);
    if (e == cudaSuccess)
        e = launch_transpose_rows(dm, nullptr, &src, dm.d, o.counts, o.offsets, o.pad_offsets,
                                  o.row_tok, b.xT, b.xT_s, st);
    if (e == cudaSuccess)
        e = launch_wgrad(dm, b.dyT, b.dyT_s, dm.d, b.hT, b.hT_s, dm.F, o.pad_offsets,
                         static_cast<uint16_t *>(dw->d_down), status, wns, st);
    if (e == cudaSuccess)
        e = launch_wgrad(dm, b.daT, b.daT_s, dm.F, b.xT, b.xT_s, dm.d, o.pad_offsets,
                         static_cast<uint16_t *>(dw->d_gate), status, wns, st);
    if (e == cudaSuccess)
        e = launch_wgrad(dm, b.dbT, b.dbT_s, dm.F, b.xT, b.xT_s, dm.d, o.pad_offsets,
                         static_cast<uint16_t *>(dw->d_up), status, wns, st);
    // B5 reverse dispatch (+ router dX), B6 router weight gradient
    if (e == cudaSuccess)
        e = launch_rev_dispatch(dm, o.ids, o.slot_pos, o.offsets, o.pad_offsets, b.dx, b.dl_sel, W_r,
                                static_cast<uint16_t *>(dX), st);
    if (e == cudaSuccess)
        e = launch_router_wgrad(dm, src, o.offsets, o.row_tok, o.row_j, b.dl_sel, dW_r, st);
    return cuda_status(e);
}

int mok_transpose_bf16(const void *src, int64_t batch, int64_t rows, int64_t K, void *dst,
                       void *stream)
{
    if (!src || !dst || batch < 1 || rows < 1 || K < 1) return MOK_ERR_INVALID_ARG;
    return cuda_status(launch_transpose_bf16(static_cast<const uint16_t *>(src), batch, rows, K,
                                             static_cast<uint16_t *>(dst),
                                             static_cast<cudaStream_t>(stream)));
}

int mok_quantize_mx(const void *src, int64_t batch, int64_t rows, int64_t K, int transpose,
                    uint8_t *codes, uint32_t *scales, void *stream)
{
    if (!src || !codes || !scales || batch < 1 || rows < 1 || K < 1) return MOK_ERR_INVALID_ARG;
    if (rows % 128 != 0 || K % 128 != 0) return MOK_ERR_UNSUPPORTED;
    if (transpose != 0 && transpose != 1) return MOK_ERR_INVALID_ARG;
    return cuda_status(launch_quant_mx(static_cast<const uint16_t *>(src), batch, rows, K, transpose,
                                       codes, scales, static_cast<cudaStream_t>(stream)));
}

int mok_swiglu_quantize_mx(const float *a, const float *b, int64_t rows, int64_t F, float *h,
                           uint8_t *codes, uint32_t *scales, void *stream)
{
    if (!a || !b || !codes || !scales || rows < 1 || F < 1) return MOK_ERR_INVALID_ARG;
    if (rows % 128 != 0 || F % 128 != 0) return MOK_ERR_UNSUPPORTED;
    return cuda_status(launch_swiglu_quant(a, b, rows, F, h, codes, scales, static_cast<cudaStream_t>(stream)));
}

int mok_bwd_ws_layout(const mok_config *cfg, mok_bwd_layout *out)
{
    Dims dm;
    const int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    if (!out) return MOK_ERR_INVALID_ARG;
    BwdWs w;
    bwd_ws_layout(dm, &w);
    out->status = w.status;
    out->dy = w.dy;
    out->da = w.da;
    out->db = w.db;
    out->dx = w.dx;
    out->dl_sel = w.dl_sel;
    out->total = w.total;
    return MOK_OK;
}

int mok_reset_device_status(void *ws, void *stream)
{
    if (!ws) return MOK_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(ws, 0, 4, static_cast<cudaStream_t>(stream)));
}

int mok_get_device_status(const void *ws, void *stream)
{
    if (!ws) return MOK_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOK_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOK_ERR_CUDA;
    return static_cast<int>(v);
}

const char *mok_status_string(int status)
{
    switch (status) {
    case MOK_OK: return "MOK_OK";
    case MOK_ERR_INVALID_ARG: return "MOK_ERR_INVALID_ARG";
    case MOK_ERR_UNSUPPORTED: return "MOK_ERR_UNSUPPORTED";
    case MOK_ERR_CUDA: return "MOK_ERR_CUDA";
    case MOK_ERR_TIMEOUT: return "MOK_ERR_TIMEOUT";
    default: return "MOK_ERR_UNKNOWN";
    }
}

}  // extern "C"
