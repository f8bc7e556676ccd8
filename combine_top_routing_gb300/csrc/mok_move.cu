// mok_move.cu -- HBM-bound row movement: A3 pull dispatch (with fused MXFP8
// quantisation), A6 final weighted combine, and the MXFP8 quantiser.
//
// [kucoin] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72" (kucoin.com flash, Arabic).  §02: dispatch is a pull -- the expert
// side reads each token it needs from (source, position in source) and places
// it in its own expert order; MXFP8 activation quantisation is fused into
// dispatch so no separate quantise pass touches HBM.  §03: the measured layer
// ends with the final weighted combine.
//
// All kernels move 16-byte vectors per lane with rows spread over warps; a
// warp owns whole rows so reads and writes are fully coalesced.
#include <cuda_bf16.h>

#include "mok_gather.cuh"
#include "mok_internal.h"
#include "mok_ptx.cuh"

namespace mok {

// ---------------------------------------------------------------------------
// A3 dispatch.  Dense layout row p holds slot (t = row_tok[p], j = row_j[p]) of
// expert e = ids[t*k+j]; it is written to padded row pad_offsets[e] + p -
// offsets[e].  One warp per row, grid-stride over rows.
// ---------------------------------------------------------------------------
template <bool MX>
__global__ void __launch_bounds__(256) k_dispatch(const Sources src, int64_t S, int d, int k,
                                                  const int32_t *__restrict__ ids,
                                                  const int32_t *__restrict__ offsets,
                                                  const int32_t *__restrict__ pad_offsets,
                                                  const int32_t *__restrict__ row_tok,
                                                  const uint8_t *__restrict__ row_j, void *xe,
                                                  uint32_t *__restrict__ xe_scales,
                                                  int64_t rows_pad)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t p = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); p < S;
         p += warps) {
        const int t = row_tok[p];
        const int e = ids[static_cast<int64_t>(t) * k + row_j[p]];
        const int64_t q = pad_offsets[e] + (p - offsets[e]);
        const uint4 *in = reinterpret_cast<const uint4 *>(source_row(src, t, d));
        if (!MX) {
            uint4 *out = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(xe) + q * d);
            for (int c = lane; c < d / 8; c += 32) out[c] = __ldg(in + c);
        } else {
            uint8_t *codes_row = static_cast<uint8_t *>(xe) + q * d;
            // four 256-element stretches per step: their loads are in flight together
            for (int c0 = 0; c0 < d; c0 += 1024) {
                uint4 raw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cu = c0 + 256 * u;
                    const int nvalid = cu >= d ? 0 : (d - cu >= 256 ? 32 : 16);
                    raw[u] = lane < nvalid ? __ldg(in + (cu >> 3) + lane) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cu = c0 + 256 * u;
                    if (cu < d)
                        mx_quant_stretch(raw[u], lane, d - cu >= 256 ? 32 : 16, codes_row, cu,
                                         xe_scales, q, rows_pad);
                }
            }
        }
    }
}

cudaError_t launch_dispatch(const Dims &dm, const Sources &src, const int32_t *ids,
                            const int32_t *offsets, const int32_t *pad_offsets,
                            const int32_t *row_tok, const uint8_t *row_j, void *xe,
                            uint32_t *xe_scales, cudaStream_t st)
{
    const int threads = 256;
    const int64_t need = (dm.S + 7) / 8;
    const int blocks = static_cast<int>(need < 32 * num_sms() ? need : 32 * num_sms());
    if (dm.dtype == MOK_MXFP8)
        k_dispatch<true><<<blocks, threads, 0, st>>>(src, dm.S, dm.d, dm.k, ids, offsets,
                                                     pad_offsets, row_tok, row_j, xe, xe_scales,
                                                     dm.rows_pad);
    else
        k_dispatch<false><<<blocks, threads, 0, st>>>(src, dm.S, dm.d, dm.k, ids, offsets,
                                                      pad_offsets, row_tok, row_j, xe, xe_scales,
                                                      dm.rows_pad);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// A3 with one read per token: warp w takes token t, reads its row from its
// source once (and quantises it once, MXFP8) and writes it into each of the
// token's k slot rows.  This is the receiver's pull with one request per token
// instead of one per slot -- on several GPUs, one pull per (token, destination
// rank) placed into every local expert the token selected.  The output bytes
// are k_dispatch's; HBM reads drop from S rows to T rows.
// ---------------------------------------------------------------------------
template <bool MX>
__global__ void __launch_bounds__(256) k_dispatch_by_token(const Sources src, int T, int d, int k,
                                                           const int32_t *__restrict__ ids,
                                                           const int32_t *__restrict__ slot_pos,
                                                           const int32_t *__restrict__ offsets,
                                                           const int32_t *__restrict__ pad_offsets,
                                                           void *xe, uint32_t *__restrict__ xe_scales,
                                                           int64_t rows_pad)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps)
        dispatch_token<MX>(src, t, d, k, ids, slot_pos, offsets, pad_offsets, xe, xe_scales, rows_pad, lane);
}

cudaError_t launch_dispatch_by_token(const Dims &dm, const Sources &src, const int32_t *ids,
                                     const int32_t *slot_pos, const int32_t *offsets,
                                     const int32_t *pad_offsets, void *xe, uint32_t *xe_scales,
                                     cudaStream_t st)
{
    const int threads = 256;
    const int64_t need = (static_cast<int64_t>(dm.T) + 7) / 8;
    const int blocks = static_cast<int>(need < 32 * num_sms() ? need : 32 * num_sms());
    if (dm.dtype == MOK_MXFP8)
        k_dispatch_by_token<true><<<blocks, threads, 0, st>>>(src, dm.T, dm.d, dm.k, ids, slot_pos, offsets,
                                                              pad_offsets, xe, xe_scales, dm.rows_pad);
    else
        k_dispatch_by_token<false><<<blocks, threads, 0, st>>>(src, dm.T, dm.d, dm.k, ids, slot_pos, offsets,
                                                               pad_offsets, xe, xe_scales, dm.rows_pad);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// A6 combine: out[t, c] = bf16( fold_j fmaf(g_tj, y_tj[c], acc) ), acc from 0,
// j = 0..k-1 in order.  One thread per 16 columns of one token; KMAX >= k
// sizes the register buffer of slot loads.
// ---------------------------------------------------------------------------
template <int KMAX>
__global__ void __launch_bounds__(256) k_combine(const uint16_t *__restrict__ ystage,
                                                 const float *__restrict__ gates, int T, int k,
                                                 int d, uint16_t *__restrict__ out)
{
    // two adjacent 8-column vectors per thread: 2k slot loads in flight
    const int64_t vec_per_tok = d / 16;
    const int64_t n = static_cast<int64_t>(T) * vec_per_tok;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / vec_per_tok;
        const int64_t c = (i % vec_per_tok) * 2;
        uint4 y[KMAX][2];
        float g[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < k) {
                g[j] = __ldg(gates + t * k + j);
                const uint4 *row = reinterpret_cast<const uint4 *>(ystage + (t * k + j) * d) + c;
                y[j][0] = __ldg(row);
                y[j][1] = __ldg(row + 1);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < k) {
                    const uint32_t w[4] = {y[j][h].x, y[j][h].y, y[j][h].z, y[j][h].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = fmaf(g[j], bf16_bits_to_float(w[q] & 0xFFFFu), acc[2 * q]);
                        acc[2 * q + 1] = fmaf(g[j], bf16_bits_to_float(w[q] >> 16), acc[2 * q + 1]);
                    }
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            reinterpret_cast<uint4 *>(out + t * d)[c + h] = o;
        }
    }
}

cudaError_t launch_combine(const Dims &dm, const uint16_t *ystage, const float *gates,
                           uint16_t *out, cudaStream_t st)
{
    const int64_t n = static_cast<int64_t>(dm.T) * (dm.d / 16);
    const int threads = 256;
    const int64_t need = (n + threads - 1) / threads;
    const int blocks = static_cast<int>(need < 64 * num_sms() ? need : 64 * num_sms());
    if (dm.k <= 2) k_combine<2><<<blocks, threads, 0, st>>>(ystage, gates, dm.T, dm.k, dm.d, out);
    else if (dm.k <= 4) k_combine<4><<<blocks, threads, 0, st>>>(ystage, gates, dm.T, dm.k, dm.d, out);
    else k_combine<MOK_MAX_TOPK><<<blocks, threads, 0, st>>>(ystage, gates, dm.T, dm.k, dm.d, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// MXFP8 quantiser of BF16 matrices (weights and backward operands).
// transpose = 0: rows of [rows, K] along K; one warp per row.
// transpose = 1: the transpose [K, rows] along rows; a 256 x 32 tile of the
// source goes through shared memory so that reads and writes stay coalesced.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quant_rows(const uint16_t *__restrict__ src, int64_t R,
                                                    int64_t K, uint8_t *__restrict__ codes,
                                                    uint32_t *__restrict__ scales)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < R;
         r += warps) {
        const uint4 *in = reinterpret_cast<const uint4 *>(src + r * K);
        for (int64_t c0 = 0; c0 < K; c0 += 256) {
            const int nvalid = K - c0 >= 256 ? 32 : 16;
            const uint4 raw = lane < nvalid ? __ldg(in + (c0 >> 3) + lane) : make_uint4(0, 0, 0, 0);
            mx_quant_stretch(raw, lane, nvalid, codes + r * K, c0, scales, r, R);
        }
    }
}

// Source matrix b: [rows, K] BF16 at src + b*rows*K; output row (b*K + c) is
// source column c, quantised along the source rows.
__global__ void __launch_bounds__(256) k_quant_cols(const uint16_t *__restrict__ src, int64_t rows,
                                                    int64_t K, uint8_t *__restrict__ codes,
                                                    uint32_t *__restrict__ scales, int64_t R_out)
{
    __shared__ uint16_t tile[32][256 + 8];
    const int64_t b = blockIdx.z;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32;   // source columns -> output rows
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 256;  // source rows -> output columns
    const uint16_t *s = src + b * rows * K;
    // load 256 source rows x 32 columns: each thread reads 8 columns (16 bytes)
    const int64_t nrows = rows - r0 < 256 ? rows - r0 : 256;
    for (int i = threadIdx.x; i < 256 * 4; i += blockDim.x) {
        const int rr = i >> 2, cc = (i & 3) * 8;
        const uint4 v = rr < nrows
                            ? __ldg(reinterpret_cast<const uint4 *>(s + (r0 + rr) * K + c0 + cc))
                            : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            tile[cc + 2 * q][rr] = static_cast<uint16_t>(w[q] & 0xFFFFu);
            tile[cc + 2 * q + 1][rr] = static_cast<uint16_t>(w[q] >> 16);
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int oc = warp; oc < 32; oc += blockDim.x >> 5) {
        const int64_t orow = b * K + c0 + oc;
        uint4 raw;
        const uint16_t *t = &tile[oc][8 * lane];
        raw.x = t[0] | (static_cast<uint32_t>(t[1]) << 16);
        raw.y = t[2] | (static_cast<uint32_t>(t[3]) << 16);
        raw.z = t[4] | (static_cast<uint32_t>(t[5]) << 16);
        raw.w = t[6] | (static_cast<uint32_t>(t[7]) << 16);
        mx_quant_stretch(raw, lane, nrows >= 256 ? 32 : 16, codes + orow * rows, r0, scales, orow,
                         R_out);
    }
}

cudaError_t launch_quant_mx(const uint16_t *src, int64_t batch, int64_t rows, int64_t K,
                            int transpose, uint8_t *codes, uint32_t *scales, cudaStream_t st)
{
    if (!transpose) {
        const int64_t R = batch * rows;
        const int64_t need = (R + 7) / 8;
        const int blocks = static_cast<int>(need < 32 * num_sms() ? need : 32 * num_sms());
        k_quant_rows<<<blocks, 256, 0, st>>>(src, R, K, codes, scales);
    } else {
        dim3 grid(static_cast<unsigned>(K / 32), static_cast<unsigned>((rows + 255) / 256),
                  static_cast<unsigned>(batch));
        k_quant_cols<<<grid, 256, 0, st>>>(src, rows, K, codes, scales, batch * K);
    }
    return cudaGetLastError();
}

}  // namespace mok
