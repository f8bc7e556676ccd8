// mok_route.cu -- A1 router top-k and A2 layout.
//
// [kucoin] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72" (kucoin.com flash, Arabic).  §01: at every step the router decides
// again which experts each token goes to; before the grouped GEMM the
// system counts tokens per expert, decides where each lands and keeps one
// expert's tokens together.  The logits GEMM itself runs on the tensor cores
// (mok_gemm.cu); this file holds the fp32 -> 3 x BF16 weight split it uses,
// the warp-per-token top-k and the three integer layout kernels.
#include <cuda_bf16.h>

#include "mok_internal.h"
#include "mok_ptx.cuh"

namespace mok {

// ---------------------------------------------------------------------------
// Router weights for the tensor-core logits GEMM: W_r (fp32) = hi + mid + lo
// with each term BF16 (the split-BF16 method of Henry, Tang & Heinecke,
// "Leveraging the bfloat16 Artificial Intelligence Datatype For
// Higher-Precision Computations", 2019).  Three BF16 terms carry all 24
// significand bits of an fp32 value, and x is BF16, so every product x*term
// is exact and the logits equal an fp32-accumulated x.W_r.  Layout: row e of
// w3 is [hi(W_r[e]) | mid(W_r[e]) | lo(W_r[e])] (3d BF16); rows E..E_pad-1 are
// zero.
// ---------------------------------------------------------------------------
__global__ void k_router_split(const float *__restrict__ Wr, int E, int E_pad, int d,
                               uint16_t *__restrict__ w3)
{
    const int64_t n = static_cast<int64_t>(E_pad) * d;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int e = static_cast<int>(i / d);
        const int c = static_cast<int>(i % d);
        float v = e < E ? Wr[i] : 0.0f;
        const uint32_t hi = float_to_bf16_bits(v);
        const float r1 = v - bf16_bits_to_float(hi);
        const uint32_t mid = float_to_bf16_bits(r1);
        const float r2 = r1 - bf16_bits_to_float(mid);
        const uint32_t lo = float_to_bf16_bits(r2);
        uint16_t *row = w3 + static_cast<int64_t>(e) * 3 * d;
        row[c] = static_cast<uint16_t>(hi);
        row[d + c] = static_cast<uint16_t>(mid);
        row[2 * d + c] = static_cast<uint16_t>(lo);
    }
}

cudaError_t launch_router_split(const float *Wr, int E, int E_pad, int d, uint16_t *w3,
                                cudaStream_t st)
{
    const int64_t n = static_cast<int64_t>(E_pad) * d;
    const int threads = 256;
    const int blocks = static_cast<int>((n + threads - 1) / threads < 4096 ? (n + threads - 1) / threads : 4096);
    k_router_split<<<blocks, threads, 0, st>>>(Wr, E, E_pad, d, w3);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Top-k: one warp per token.  Lane l holds logits l, l+32, ...; k rounds of a
// warp arg-max (larger logit wins, equal logits go to the lower id).  Scores
// are softmax over E or sigmoid; both are monotone in the logit, so choosing
// by logit is choosing by score.  gates = chosen scores / their sum.
// ---------------------------------------------------------------------------
template <int EPL>
__global__ void __launch_bounds__(256) k_topk(const float *__restrict__ logits, int T, int E,
                                              int k, int kind, int32_t *__restrict__ ids,
                                              float *__restrict__ gates,
                                              float *__restrict__ sel_scores)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + static_cast<int64_t>(t) * E;
    float v[EPL];
    float vmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? row[e] : -INFINITY;
        vmax = fmaxf(vmax, v[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    float z = 0.0f;  // softmax normaliser over all E
    if (kind == MOK_ROUTER_SOFTMAX) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (lane + 32 * i < E) z += __expf(v[i] - vmax);
#pragma unroll
        for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    }
    uint32_t taken = 0;
    float sel_l[MOK_MAX_TOPK];
    int sel_e[MOK_MAX_TOPK];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < be))) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        sel_l[j] = bv;
        sel_e[j] = be;
    }
    if (lane == 0) {
        float s[MOK_MAX_TOPK];
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) {
            s[j] = kind == MOK_ROUTER_SOFTMAX ? __expf(sel_l[j] - vmax) / z
                                              : 1.0f / (1.0f + __expf(-sel_l[j]));
            sum += s[j];
        }
        for (int j = 0; j < k; ++j) {
            ids[t * k + j] = sel_e[j];
            gates[t * k + j] = s[j] / sum;
            if (sel_scores) sel_scores[t * k + j] = s[j];
        }
    }
}

cudaError_t launch_topk(const Dims &dm, const float *logits, int32_t *ids, float *gates,
                        float *sel_scores, cudaStream_t st)
{
    const int warps = 8;
    const int blocks = (dm.T + warps - 1) / warps;
    const int epl = (dm.E + 31) / 32;
#define MOK_TOPK_CASE(N)                                                                  \
    if (epl <= N) {                                                                       \
        k_topk<N><<<blocks, warps * 32, 0, st>>>(logits, dm.T, dm.E, dm.k, dm.router, ids, \
                                                 gates, sel_scores);                      \
        return cudaGetLastError();                                                        \
    }
    MOK_TOPK_CASE(1)
    MOK_TOPK_CASE(2)
    MOK_TOPK_CASE(4)
    MOK_TOPK_CASE(8)
    MOK_TOPK_CASE(16)
    MOK_TOPK_CASE(32)
#undef MOK_TOPK_CASE
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Layout: a stable counting sort of the S = T*k slots by expert, in integer
// passes over chunks of kLayoutChunk consecutive slots.  The per-chunk tables
// are expert-major ([E][nchunks]) so that one expert's chunks are contiguous.
//   count        : per-chunk histogram (shared-memory integer atomics);
//   scan_chunks  : one block per expert, exclusive prefix over its chunks
//                  (relative to the expert's first row) and its total count;
//   scan_experts : dense offsets and padded offsets (segments rounded up to
//                  MOK_ROW_ALIGN rows) from the counts;
//   place        : one warp walks its chunk 32 slots at a time in slot order;
//                  lanes with equal expert get consecutive ranks (match +
//                  popc), so a slot's row is offsets[e] + (slots of e before
//                  it) -- stable by t*k+j.
// Everything is integer, so the result is the same on every run.  An id
// outside [0, E) (possible only when the caller supplies the ids) is counted
// nowhere and placed nowhere: its slot_pos is -1, and offsets[E] becomes -1
// instead of T*k, so the error is visible and no table is indexed with it.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_layout_count(const int32_t *__restrict__ ids, int64_t S,
                                                      int E, int nchunks,
                                                      int32_t *__restrict__ chunk_counts)
{
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * kLayoutChunk;
    const int64_t hi = lo + kLayoutChunk < S ? lo + kLayoutChunk : S;
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const int e = ids[i];
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[static_cast<int64_t>(e) * nchunks + blockIdx.x] = hist[e];
}

// Block-wide exclusive scan of `v` (256 threads); returns the block total.
__device__ __forceinline__ int32_t block_excl_scan256(int32_t v, int32_t *excl, int32_t *s_warp)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    int32_t base = 0, total = 0;
    for (int w = 0; w < 8; ++w) {
        if (w < wid) base += s_warp[w];
        total += s_warp[w];
    }
    __syncthreads();
    *excl = base + incl - v;
    return total;
}

__global__ void __launch_bounds__(256) k_layout_scan_chunks(const int32_t *__restrict__ chunk_counts,
                                                            int nchunks,
                                                            int32_t *__restrict__ chunk_base,
                                                            int32_t *__restrict__ counts)
{
    __shared__ int32_t s_warp[8];
    const int e = blockIdx.x;
    const int32_t *cc = chunk_counts + static_cast<int64_t>(e) * nchunks;
    int32_t *cb = chunk_base + static_cast<int64_t>(e) * nchunks;
    int32_t carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 256) {
        const int c = c0 + threadIdx.x;
        const int32_t v = c < nchunks ? cc[c] : 0;
        int32_t excl;
        const int32_t total = block_excl_scan256(v, &excl, s_warp);
        if (c < nchunks) cb[c] = carry + excl;
        carry += total;
    }
    if (threadIdx.x == 0) counts[e] = carry;
}

__global__ void __launch_bounds__(1024) k_layout_scan_experts(const int32_t *__restrict__ counts,
                                                              int E, int64_t S,
                                                              int32_t *__restrict__ offsets,
                                                              int32_t *__restrict__ pad_offsets)
{
    __shared__ int32_t s_warp[2][32];
    const int e = threadIdx.x;
    const int32_t cnt = e < E ? counts[e] : 0;
    const int32_t pad = static_cast<int32_t>(round_up(cnt, MOK_ROW_ALIGN));
    const int lane = e & 31, wid = e >> 5;
    int32_t ic = cnt, ip = pad;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t a = __shfl_up_sync(0xffffffffu, ic, o);
        const int32_t b = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) {
            ic += a;
            ip += b;
        }
    }
    if (lane == 31) {
        s_warp[0][wid] = ic;
        s_warp[1][wid] = ip;
    }
    __syncthreads();
    if (wid == 0) {
        int32_t a = s_warp[0][lane];
        int32_t b = s_warp[1][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t x = __shfl_up_sync(0xffffffffu, a, o);
            const int32_t y = __shfl_up_sync(0xffffffffu, b, o);
            if (lane >= o) {
                a += x;
                b += y;
            }
        }
        s_warp[0][lane] = a;
        s_warp[1][lane] = b;
    }
    __syncthreads();
    const int32_t excl_c = (wid ? s_warp[0][wid - 1] : 0) + ic - cnt;
    const int32_t excl_p = (wid ? s_warp[1][wid - 1] : 0) + ip - pad;
    if (e < E) {
        offsets[e] = excl_c;
        pad_offsets[e] = excl_p;
        if (e == E - 1) {
            // fewer counted slots than T*k: some id was outside [0, E)
            offsets[E] = excl_c + cnt == S ? excl_c + cnt : -1;
            pad_offsets[E] = excl_p + pad;
        }
    }
}

__global__ void __launch_bounds__(32) k_layout_place(const int32_t *__restrict__ ids, int64_t S,
                                                     int k, int E, int nchunks,
                                                     const int32_t *__restrict__ chunk_base,
                                                     const int32_t *__restrict__ offsets,
                                                     int32_t *__restrict__ slot_pos,
                                                     int32_t *__restrict__ row_tok,
                                                     uint8_t *__restrict__ row_j)
{
    extern __shared__ int32_t run[];
    const int lane = threadIdx.x;
    for (int e = lane; e < E; e += 32)
        run[e] = offsets[e] + chunk_base[static_cast<int64_t>(e) * nchunks + blockIdx.x];
    __syncwarp();
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * kLayoutChunk;
    const int64_t hi = lo + kLayoutChunk < S ? lo + kLayoutChunk : S;
    for (int64_t i0 = lo; i0 < hi; i0 += 32) {
        const int64_t i = i0 + lane;
        const bool act = i < hi;
        const uint32_t active = __ballot_sync(0xffffffffu, act);
        if (act) {
            const int e = ids[i];
            const bool ok = static_cast<unsigned>(e) < static_cast<unsigned>(E);
            const uint32_t peers = __match_any_sync(active, ok ? e : -1);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            if (ok) {
                const int pos = run[e] + rank;
                slot_pos[i] = pos;
                row_tok[pos] = static_cast<int32_t>(i / k);
                row_j[pos] = static_cast<uint8_t>(i % k);
            } else {
                slot_pos[i] = -1;
            }
            __syncwarp(active);
            if (ok && rank == 0) run[e] += __popc(peers);
        }
        __syncwarp();
    }
}

cudaError_t launch_layout(const Dims &dm, const int32_t *ids, int32_t *counts, int32_t *offsets,
                          int32_t *pad_offsets, int32_t *slot_pos, int32_t *row_tok,
                          uint8_t *row_j, int32_t *chunk_counts, int32_t *chunk_base,
                          cudaStream_t st)
{
    const size_t hist_bytes = static_cast<size_t>(dm.E) * sizeof(int32_t);
    k_layout_count<<<dm.nchunks, 256, hist_bytes, st>>>(ids, dm.S, dm.E, dm.nchunks, chunk_counts);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    k_layout_scan_chunks<<<dm.E, 256, 0, st>>>(chunk_counts, dm.nchunks, chunk_base, counts);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    k_layout_scan_experts<<<1, 1024, 0, st>>>(counts, dm.E, dm.S, offsets, pad_offsets);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    k_layout_place<<<dm.nchunks, 32, hist_bytes, st>>>(ids, dm.S, dm.k, dm.E, dm.nchunks, chunk_base,
                                                        offsets, slot_pos, row_tok, row_j);
    return cudaGetLastError();
}

__global__ void k_counts_from_offsets(const int32_t *__restrict__ offsets, int E,
                                      int32_t *__restrict__ counts)
{
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
        counts[e] = offsets[e + 1] - offsets[e];
}

cudaError_t launch_counts_from_offsets(const int32_t *offsets, int E, int32_t *counts,
                                       cudaStream_t st)
{
    k_counts_from_offsets<<<(E + 255) / 256, 256, 0, st>>>(offsets, E, counts);
    return cudaGetLastError();
}

}  // namespace mok
