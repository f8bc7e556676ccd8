// mok_bwd.cu -- the HBM-bound steps of the backward layer.
//
// [kucoin] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72" (kucoin.com flash, Arabic).  §01: training runs two more rounds of
// exchange in the reverse direction; §02: backward uses a pull
// reverse-combine (each slot pulls dY of its token) and a push
// reverse-dispatch (each slot's input gradient goes back to its token).
//
//   k_rev_combine    B1 + B6 (gate part): dy_slot = bf16(g dY[t]) into the
//                    padded expert-ordered rows (and MXFP8 along d), dgates =
//                    <dY[t], y_tj>, dlogits of the chosen experts;
//   k_transpose_rows wgrad operands: a padded row buffer (or x gathered by
//                    token) transposed to [X, rows] with padding rows zeroed,
//                    BF16 or MXFP8 along the token dimension;
//   k_rev_dispatch   B5 + router dX: dX[t] = sum_j dx_slot + sum_j dl_j W_r[e_j];
//   k_router_wgrad   B6: dW_r[e] = sum over e's rows of dl * x[t].
// Every reduction runs in a fixed order (no atomics), so results are
// bit-reproducible.
#include <cuda_bf16.h>

#include "mok_internal.h"
#include "mok_ptx.cuh"

namespace mok {

// padded row of slot (t, j)
__device__ __forceinline__ int64_t slot_row(const int32_t *ids, const int32_t *slot_pos,
                                            const int32_t *offsets, const int32_t *pad_offsets,
                                            int64_t i)
{
    const int e = ids[i];
    return pad_offsets[e] + (slot_pos[i] - offsets[e]);
}

// ---------------------------------------------------------------------------
// B1: one warp per token.  Lane l owns columns [8l + 256 i, +8).
// ---------------------------------------------------------------------------
template <bool MX>
__global__ void __launch_bounds__(256) k_rev_combine(
    int T, int d, int k, int E, int kind, const uint16_t *__restrict__ dY,
    const float *__restrict__ gates, const float *__restrict__ sel_scores,
    const int32_t *__restrict__ ids, const int32_t *__restrict__ slot_pos,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ pad_offsets,
    const uint16_t *__restrict__ ystage, uint16_t *__restrict__ dy_rows, uint8_t *__restrict__ dy_q,
    uint32_t *__restrict__ dy_s, int64_t rows_pad, float *__restrict__ dgates,
    float *__restrict__ dlogits, float *__restrict__ dl_sel)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint4 *dyrow = reinterpret_cast<const uint4 *>(dY + static_cast<int64_t>(t) * d);
    // one pass over the columns: the token's dY chunk is read once and the k
    // slot rows' chunks are all in flight before they are used; the dot
    // products run per slot over the columns in order, as before
    float dg[MOK_MAX_TOPK], g[MOK_MAX_TOPK];
    int64_t q[MOK_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOK_MAX_TOPK; ++j) {
        dg[j] = 0.0f;
        if (j < k) {
            const int64_t i = static_cast<int64_t>(t) * k + j;
            g[j] = gates[i];
            q[j] = slot_row(ids, slot_pos, offsets, pad_offsets, i);
        }
    }
    for (int c0 = 0; c0 < d; c0 += 256) {
        const int nvalid = d - c0 >= 256 ? 32 : 16;
        uint4 a = make_uint4(0, 0, 0, 0), y[MOK_MAX_TOPK];
        if (lane < nvalid) a = __ldg(dyrow + (c0 >> 3) + lane);
#pragma unroll
        for (int j = 0; j < MOK_MAX_TOPK; ++j)
            if (j < k && lane < nvalid)
                y[j] = __ldg(reinterpret_cast<const uint4 *>(ystage + (static_cast<int64_t>(t) * k + j) * d) +
                             (c0 >> 3) + lane);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < MOK_MAX_TOPK; ++j) {
            if (j >= k) break;
            uint4 out = make_uint4(0, 0, 0, 0);
            if (lane < nvalid) {
                const uint32_t yv[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
                uint32_t ov[4];
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {
                    const float d0 = bf16_bits_to_float(av[q2] & 0xFFFFu);
                    const float d1 = bf16_bits_to_float(av[q2] >> 16);
                    dg[j] = fmaf(d0, bf16_bits_to_float(yv[q2] & 0xFFFFu), dg[j]);
                    dg[j] = fmaf(d1, bf16_bits_to_float(yv[q2] >> 16), dg[j]);
                    ov[q2] = pack_bf16x2(g[j] * d0, g[j] * d1);
                }
                out = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                reinterpret_cast<uint4 *>(dy_rows + q[j] * d)[(c0 >> 3) + lane] = out;
            }
            if (MX) mx_quant_stretch(out, lane, nvalid, dy_q + q[j] * d, c0, dy_s, q[j], rows_pad);
        }
    }
#pragma unroll
    for (int j = 0; j < MOK_MAX_TOPK; ++j) {
        if (j >= k) break;
#pragma unroll
        for (int o = 16; o; o >>= 1) dg[j] += __shfl_xor_sync(0xffffffffu, dg[j], o);
    }
    // gradients through the renormalised top-k gates to the chosen logits
    // (loops unrolled to the bound on k, so that the per-slot values stay in registers)
    float G = 0.0f, ssum = 0.0f;
#pragma unroll
    for (int j = 0; j < MOK_MAX_TOPK; ++j) {
        if (j >= k) break;
        G += dg[j] * g[j];
        ssum += sel_scores[static_cast<int64_t>(t) * k + j];
    }
    float dl[MOK_MAX_TOPK];
    int sel[MOK_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOK_MAX_TOPK; ++j) {
        if (j >= k) break;
        const int64_t i = static_cast<int64_t>(t) * k + j;
        sel[j] = ids[i];
        if (kind == MOK_ROUTER_SOFTMAX) {
            dl[j] = g[j] * (dg[j] - G);
        } else {
            const float sc = sel_scores[i];
            dl[j] = (dg[j] - G) / ssum * sc * (1.0f - sc);
        }
        if (lane == 0) {
            dgates[i] = dg[j];
            dl_sel[i] = dl[j];
        }
    }
    if (dlogits) {
        for (int e = lane; e < E; e += 32) {
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < MOK_MAX_TOPK; ++j)
                if (j < k && sel[j] == e) v = dl[j];
            dlogits[static_cast<int64_t>(t) * E + e] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// wgrad operands: out[c, q] = in[q, c] for the padded rows q of one 256-row
// tile, zero where q is a padding row; GATHER reads row q from the token it
// holds (x via the sources) instead of from a row buffer.
// ---------------------------------------------------------------------------
template <bool MX, bool GATHER>
__global__ void __launch_bounds__(256, 3) k_transpose_rows(
    const uint16_t *__restrict__ in, Sources src, int C, int E, const int32_t *__restrict__ counts,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ pad_offsets,
    const int32_t *__restrict__ row_tok, int64_t rows_pad, void *out, uint32_t *__restrict__ out_s,
    int col_tiles)
{
    // A 256-row tile and col_tiles 64-column tiles of it, one after the other.
    // Every row read is one 128-byte line.  A thread holds 8 columns of two
    // adjacent rows and writes them transposed as 32-bit (row 2p, row 2p + 1)
    // pairs: shared word (c, p) sits at c * 128 + (p ^ 4 * ((c / 8) % 8)), so
    // that the 32 lanes of a transposing store (4 row pairs x 8 column groups)
    // and of a 16-byte read along one column (32 aligned groups of 4 pairs)
    // each hit 32 different banks.  The next column tile's loads are in flight
    // while this one is written.
    __shared__ __align__(16) uint32_t tileT[64][128];
    __shared__ const uint16_t *s_row[256];
    __shared__ int s_seg[2];
    const int64_t q0 = static_cast<int64_t>(blockIdx.y) * 256;
    const int64_t pad_end = pad_offsets[E];
    if (q0 >= pad_end) return;  // beyond the last expert segment: never read
    // The expert segments holding rows q0 and q0 + 128: segments start on
    // 128-row boundaries, so each 128-row half lies in one.  One round of loads,
    // every thread testing a few experts, instead of a binary search per row.
    if (threadIdx.x < 2) s_seg[threadIdx.x] = -1;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int lo = pad_offsets[e], hi = pad_offsets[e + 1];
        if (lo <= q0 && q0 < hi) s_seg[0] = e;
        if (lo <= q0 + 128 && q0 + 128 < hi) s_seg[1] = e;
    }
    __syncthreads();
    {
        // source row of padded row q0 + threadIdx.x (null: padding, reads as zeros)
        const int64_t q = q0 + threadIdx.x;
        const int e = s_seg[threadIdx.x >> 7];
        const uint16_t *row = nullptr;
        if (e >= 0) {
            const int64_t local = q - pad_offsets[e];
            if (local < counts[e]) {
                if (GATHER) row = source_row(src, row_tok[offsets[e] + local], C);
                else row = in + q * C;
            }
        }
        s_row[threadIdx.x] = row;
    }
    __syncthreads();
    // 8 threads per row pair (16 bytes of each row), 32 row pairs per pass, all
    // 4 passes (8 rows of 16 bytes) in flight
    const int cg = threadIdx.x & 7;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ct0 = blockIdx.x * col_tiles;
    const int nct = min(col_tiles, C / 64 - ct0);
    uint4 v[8];
    auto load = [&](int c0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rp = i * 32 + (threadIdx.x >> 3);
            const uint16_t *r0 = s_row[2 * rp], *r1 = s_row[2 * rp + 1];
            v[2 * i] = r0 ? __ldg(reinterpret_cast<const uint4 *>(r0 + c0 + cg * 8)) : make_uint4(0, 0, 0, 0);
            v[2 * i + 1] = r1 ? __ldg(reinterpret_cast<const uint4 *>(r1 + c0 + cg * 8)) : make_uint4(0, 0, 0, 0);
        }
    };
    load(ct0 * 64);
    for (int t = 0; t < nct; ++t) {
        const int c0 = (ct0 + t) * 64;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rp = i * 32 + (threadIdx.x >> 3);
            const uint32_t a[4] = {v[2 * i].x, v[2 * i].y, v[2 * i].z, v[2 * i].w};
            const uint32_t b[4] = {v[2 * i + 1].x, v[2 * i + 1].y, v[2 * i + 1].z, v[2 * i + 1].w};
            const int sw = rp ^ (4 * cg);  // (c / 8) % 8 == cg for the thread's 8 columns
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = cg * 8 + 2 * j;
                tileT[c][sw] = (a[j] & 0xFFFFu) | (b[j] << 16);
                tileT[c + 1][sw] = (a[j] >> 16) | (b[j] & 0xFFFF0000u);
            }
        }
        __syncthreads();
        if (t + 1 < nct) load(c0 + 64);
        for (int oc = warp; oc < 64; oc += blockDim.x >> 5) {
            const int64_t orow = c0 + oc;
            const uint4 raw = *reinterpret_cast<const uint4 *>(&tileT[oc][4 * (lane ^ ((oc >> 3) & 7))]);
            if (MX) {
                mx_quant_stretch(raw, lane, 32, static_cast<uint8_t *>(out) + orow * rows_pad, q0, out_s,
                                 orow, C);
            } else {
                reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + orow * rows_pad + q0)[lane] = raw;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// B5: dX[t] = bf16( sum_j dx_rows[slot row] + sum_j dl_tj W_r[e_tj] ), both
// sums in j order in fp32.  One warp per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rev_dispatch(
    int T, int d, int k, const int32_t *__restrict__ ids, const int32_t *__restrict__ slot_pos,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ pad_offsets,
    const uint16_t *__restrict__ dx_rows, const float *__restrict__ dl_sel,
    const float *__restrict__ W_r, uint16_t *__restrict__ dX)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    // the token's slot rows and router terms (k values, registers)
    int64_t q[MOK_MAX_TOPK];
    float dl[MOK_MAX_TOPK];
    int eid[MOK_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOK_MAX_TOPK; ++j) {
        if (j < k) {
            const int64_t i = static_cast<int64_t>(t) * k + j;
            q[j] = slot_row(ids, slot_pos, offsets, pad_offsets, i);
            dl[j] = dl_sel[i];
            eid[j] = ids[i];
        }
    }
    for (int c0 = lane * 8; c0 < d; c0 += 256) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        // all k slot-row loads in flight, then the sums in j order
        uint4 v[MOK_MAX_TOPK];
#pragma unroll
        for (int j = 0; j < MOK_MAX_TOPK; ++j)
            if (j < k) v[j] = __ldg(reinterpret_cast<const uint4 *>(dx_rows + q[j] * d + c0));
#pragma unroll
        for (int j = 0; j < MOK_MAX_TOPK; ++j) {
            if (j >= k) break;
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += bf16_bits_to_float(w[i] & 0xFFFFu);
                acc[2 * i + 1] += bf16_bits_to_float(w[i] >> 16);
            }
        }
#pragma unroll
        for (int j = 0; j < MOK_MAX_TOPK; ++j) {
            if (j >= k) break;
            const float4 *wr = reinterpret_cast<const float4 *>(W_r + static_cast<int64_t>(eid[j]) * d + c0);
            const float4 w0 = __ldg(wr), w1 = __ldg(wr + 1);
            acc[0] = fmaf(dl[j], w0.x, acc[0]);
            acc[1] = fmaf(dl[j], w0.y, acc[1]);
            acc[2] = fmaf(dl[j], w0.z, acc[2]);
            acc[3] = fmaf(dl[j], w0.w, acc[3]);
            acc[4] = fmaf(dl[j], w1.x, acc[4]);
            acc[5] = fmaf(dl[j], w1.y, acc[5]);
            acc[6] = fmaf(dl[j], w1.z, acc[6]);
            acc[7] = fmaf(dl[j], w1.w, acc[7]);
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4 *>(dX + static_cast<int64_t>(t) * d + c0) = o;
    }
}

// ---------------------------------------------------------------------------
// B6: dW_r[e, c] = sum over e's dense rows p (in order) of dl(p) x[t(p), c].
// Block (512 columns, expert e); two columns per thread.  The rows' source
// pointers and dl values are staged 256 rows at a time in shared memory, so
// that the x loads of 8 rows are in flight at once instead of one row's
// chain of dependent loads (row -> token -> dl -> x) at a time.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_router_wgrad(
    Sources src, int d, int k, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ row_tok, const uint8_t *__restrict__ row_j,
    const float *__restrict__ dl_sel, float *__restrict__ dW_r)
{
    __shared__ const uint16_t *s_x[256];
    __shared__ float s_dl[256];
    const int e = blockIdx.y;
    const int c = (blockIdx.x * 256 + threadIdx.x) * 2;
    const int p0 = offsets[e], p1 = offsets[e + 1];
    float acc0 = 0.0f, acc1 = 0.0f;
    for (int pc = p0; pc < p1; pc += 256) {
        const int n = min(256, p1 - pc);
        __syncthreads();  // the previous chunk's rows are consumed
        if (threadIdx.x < n) {
            const int p = pc + threadIdx.x;
            const int t = row_tok[p];
            s_dl[threadIdx.x] = dl_sel[static_cast<int64_t>(t) * k + row_j[p]];
            s_x[threadIdx.x] = source_row(src, t, d);
        }
        __syncthreads();
        if (c < d) {
            int r = 0;
            for (; r + 8 <= n; r += 8) {
                uint32_t xv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) xv[u] = __ldg(reinterpret_cast<const uint32_t *>(s_x[r + u] + c));
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    acc0 = fmaf(s_dl[r + u], bf16_bits_to_float(xv[u] & 0xFFFFu), acc0);
                    acc1 = fmaf(s_dl[r + u], bf16_bits_to_float(xv[u] >> 16), acc1);
                }
            }
            for (; r < n; ++r) {
                const uint32_t xv = __ldg(reinterpret_cast<const uint32_t *>(s_x[r] + c));
                acc0 = fmaf(s_dl[r], bf16_bits_to_float(xv & 0xFFFFu), acc0);
                acc1 = fmaf(s_dl[r], bf16_bits_to_float(xv >> 16), acc1);
            }
        }
    }
    if (c < d) *reinterpret_cast<float2 *>(dW_r + static_cast<int64_t>(e) * d + c) = make_float2(acc0, acc1);
}

// ---------------------------------------------------------------------------
// BF16 transpose of `batch` matrices [rows, K] -> [K, rows] (weights for the
// BF16 backward GEMMs).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_transpose_bf16(const uint16_t *__restrict__ src,
                                                        int64_t rows, int64_t K,
                                                        uint16_t *__restrict__ dst)
{
    __shared__ uint16_t tile[32][33];
    const int64_t b = blockIdx.z;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, k0 = static_cast<int64_t>(blockIdx.x) * 32;
    const uint16_t *s = src + b * rows * K;
    uint16_t *o = dst + b * rows * K;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8)
        if (r0 + i < rows && k0 + tx < K) tile[i][tx] = s[(r0 + i) * K + k0 + tx];
    __syncthreads();
    for (int i = ty; i < 32; i += 8)
        if (k0 + i < K && r0 + tx < rows) o[(k0 + i) * rows + r0 + tx] = tile[tx][i];
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_rev_combine(const Dims &dm, const uint16_t *dY, const float *gates,
                               const float *sel_scores, const int32_t *ids,
                               const int32_t *slot_pos, const int32_t *offsets,
                               const int32_t *pad_offsets, const uint16_t *ystage,
                               const BwdBufs &b, float *dgates, float *dlogits, cudaStream_t st)
{
    const int blocks = (dm.T + 7) / 8;
    if (dm.dtype == MOK_MXFP8)
        k_rev_combine<true><<<blocks, 256, 0, st>>>(dm.T, dm.d, dm.k, dm.E, dm.router, dY, gates,
                                                   sel_scores, ids, slot_pos, offsets, pad_offsets,
                                                   ystage, b.dy, b.dy_q, b.dy_s, dm.rows_pad, dgates,
                                                   dlogits, b.dl_sel);
    else
        k_rev_combine<false><<<blocks, 256, 0, st>>>(dm.T, dm.d, dm.k, dm.E, dm.router, dY, gates,
                                                    sel_scores, ids, slot_pos, offsets, pad_offsets,
                                                    ystage, b.dy, nullptr, nullptr, dm.rows_pad,
                                                    dgates, dlogits, b.dl_sel);
    return cudaGetLastError();
}

cudaError_t launch_transpose_rows(const Dims &dm, const uint16_t *in, const Sources *src, int C,
                                  const int32_t *counts, const int32_t *offsets,
                                  const int32_t *pad_offsets, const int32_t *row_tok, void *out,
                                  uint32_t *out_s, cudaStream_t st)
{
    constexpr int kColTiles = 4;  // 64-column tiles per block (the row segments found once)
    dim3 grid(static_cast<unsigned>((C / 64 + kColTiles - 1) / kColTiles), static_cast<unsigned>(dm.rows_pad / 256));
    const bool mx = dm.dtype == MOK_MXFP8;
    Sources empty_src = {};
    const Sources &s = src ? *src : empty_src;
    if (mx && src)
        k_transpose_rows<true, true><<<grid, 256, 0, st>>>(in, s, C, dm.E, counts, offsets, pad_offsets,
                                                          row_tok, dm.rows_pad, out, out_s, kColTiles);
    else if (mx)
        k_transpose_rows<true, false><<<grid, 256, 0, st>>>(in, s, C, dm.E, counts, offsets, pad_offsets,
                                                           row_tok, dm.rows_pad, out, out_s, kColTiles);
    else if (src)
        k_transpose_rows<false, true><<<grid, 256, 0, st>>>(in, s, C, dm.E, counts, offsets, pad_offsets,
                                                           row_tok, dm.rows_pad, out, out_s, kColTiles);
    else
        k_transpose_rows<false, false><<<grid, 256, 0, st>>>(in, s, C, dm.E, counts, offsets,
                                                            pad_offsets, row_tok, dm.rows_pad, out, out_s, kColTiles);
    return cudaGetLastError();
}

cudaError_t launch_rev_dispatch(const Dims &dm, const int32_t *ids, const int32_t *slot_pos,
                                const int32_t *offsets, const int32_t *pad_offsets,
                                const uint16_t *dx_rows, const float *dl_sel, const float *W_r,
                                uint16_t *dX, cudaStream_t st)
{
    k_rev_dispatch<<<(dm.T + 7) / 8, 256, 0, st>>>(dm.T, dm.d, dm.k, ids, slot_pos, offsets,
                                                   pad_offsets, dx_rows, dl_sel, W_r, dX);
    return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const Dims &dm, const Sources &src, const int32_t *offsets,
                                const int32_t *row_tok, const uint8_t *row_j, const float *dl_sel,
                                float *dW_r, cudaStream_t st)
{
    dim3 grid(static_cast<unsigned>((dm.d / 2 + 255) / 256), static_cast<unsigned>(dm.E));
    k_router_wgrad<<<grid, 256, 0, st>>>(src, dm.d, dm.k, offsets, row_tok, row_j, dl_sel, dW_r);
    return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const uint16_t *src, int64_t batch, int64_t rows, int64_t K,
                                  uint16_t *dst, cudaStream_t st)
{
    dim3 grid(static_cast<unsigned>((K + 31) / 32), static_cast<unsigned>((rows + 31) / 32),
              static_cast<unsigned>(batch));
    k_transpose_bf16<<<grid, 256, 0, st>>>(src, rows, K, dst);
    return cudaGetLastError();
}

}  // namespace mok
