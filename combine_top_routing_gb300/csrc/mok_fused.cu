// mok_fused.cu -- A7: dispatch, the grouped SwiGLU FFN and the weighted
// combine of the forward layer as ONE persistent cooperative kernel.
//
// [kucoin] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72" (kucoin.com flash, Arabic), §02: the megakernel splits the SMs into
// a part that runs dispatch, combine and state management and a part that
// runs the expert FFN; the communication side tells the compute side through
// a local on-GPU counter when a full set of tokens has arrived, and the
// compute side tells it back when results can go out; the minibatch (tokens
// handed over per step) trades early start against GEMM efficiency; a
// fixed-size token ring buffer is filled by dispatch and reused as soon as
// the experts are done with it, with no CPU in the loop.  [miku]: results are
// bit-identical whatever the schedule.
//
// On one GPU this becomes:
//   * gather role (the first n_gather CTAs): pull each expert-ordered row from
//     its (source, row), quantise it (MXFP8) and write it into the token ring
//     (ring row = padded row mod ring_rows); after each minibatch of mb rows,
//     bump ready[row tile] (release).  Before reusing ring rows it waits until
//     every FFN1 tile that read their previous occupant has loaded them
//     (consumed[row tile] == FFN1 N tiles).  When the gather is done these
//     CTAs join the GEMM role.
//   * GEMM role: a dynamic scheduler (one global atomic) hands out all FFN1
//     tiles, then all FFN2 tiles, expert by expert in bands of row tiles
//     (N tile by N tile, the band's row tiles innermost; one band per expert
//     unless the ring is capped, then half the ring per band).  An FFN1 tile
//     waits for ready[m], loads A from the ring, and signals consumed[m] once
//     its loads have landed; its epilogue writes h and bumps h_done[m] (once
//     per epilogue warp).  An FFN2 tile waits until all FFN1 N tiles of m are
//     in h and pushes y rows to their token slots (ystage).
//   * combine: the separate combine kernel, launched right after this one on
//     the same stream (with seven warps per SM this kernel's threads did the
//     same reads 1.4x slower than the combine kernel at full occupancy).
//   * gather first (uncapped ring only, chosen by the plan where the split
//     would give the gather role many SMs): the by-token dispatch kernel pulls
//     whole tokens into their k ring rows (one read per token) right before
//     this kernel on the same stream, and every CTA runs the GEMM role from
//     the start.  (A gather prologue inside this kernel, seven warps per SM,
//     took 0.30 ms where the dispatch kernel at full occupancy takes 0.24.)
//   * chained calls (macrobatch pipelining): the previous call's weighted
//     combine runs in this kernel, its tokens in chunks (one token per
//     epilogue warp) whose queue ids sit evenly among the FFN1 tiles; the
//     scheduler hands them out like tiles, so they fill the epilogue warps'
//     gaps while the MMAs of the next tiles run.
// Each tile is computed by exactly one CTA with the same instruction sequence
// as the separate-kernel path, so the output is bit-identical to it for every
// SM split, minibatch and ring size.  Every wait is bounded (wait_ns): on
// expiry the status word gets MOK_ERR_TIMEOUT and the kernel winds down.
// Deadlock-free: the ring fills strictly in row-tile order and holds two
// bands, the rows a gather waits for belong to a band whose tiles all precede
// the tiles that wait for that gather, and every CTA processes its tiles in
// schedule order (cooperative launch: all CTAs are resident).
#include <cuda_bf16.h>

#include <mutex>

#include "mok_internal.h"
#include "mok_ptx.cuh"
#include "mok_tc.cuh"

namespace mok {

namespace {

constexpr int kTQ = 2;  // depth of the tile-id queue from the scheduler thread to MMA / epilogue
// 7 warps: 0 TMA producer (and tile scheduler), 1 MMA issue, 2-5 epilogue (one
// TMEM lane quarter each), 6 MXFP8 scale copies into TMEM (idle for BF16)
constexpr int kFThreads = 224;
constexpr int kScaleWarp = 6;

// Tensor maps of both fused kernels.  ring64 / h64 cover the same tensors as
// ring / h with 64-row boxes: a row tile whose expert has 64 valid rows or
// fewer in it loads only those (the rows past an expert's count are padding,
// whose results are discarded).  The scale-tile maps serve the pair kernel.
struct FusedMaps {
    CUtensorMap ring, ring64, g, u, h, h64, dn;   // operands
    CUtensorMap s_ring, s_g, s_u, s_h, s_dn;      // MX scale tiles (MXFP8, CTA pairs)
};

// Rows of A a 128-row tile loads: all, its first 64, or none (rows past the
// expert's count are padding; the MMA reads stale shared memory there, which
// only reaches the discarded rows of the accumulator).  rel = first row of the
// tile relative to the expert's first row.
__device__ __forceinline__ int a_rows_to_load(int count, int64_t rel)
{
    const int64_t v = count - rel;
    return v <= 0 ? 0 : (v <= 64 ? 64 : kBM);
}

struct FusedArgs {
    int E, T, k, d, F;
    const int32_t *ids, *counts, *offsets, *pad_offsets, *slot_pos, *row_tok;
    const uint8_t *row_j;
    const float *gates;
    Sources src;
    uint8_t *ring;            // [ring_rows, d] BF16 or E4M3
    uint32_t *ring_scales;    // MX scale tile layout, rows = ring_rows, K = d
    int64_t ring_rows;        // multiple of 256 (holds any minibatch)
    void *h;                  // [h_rows, F]
    uint32_t *h_scales;
    int64_t h_rows;
    const uint32_t *s_gate, *s_up, *s_down;
    int64_t EF, Ed;
    uint16_t *ystage, *out;
    uint16_t *saved_a, *saved_b, *saved_h;
    int mb;                   // minibatch rows per hand-off (64, 128, 256)
    int n_gather;             // CTAs that start in the gather role
    int prologue;             // 1: the rows are in the ring already (gathered by the dispatch kernel)
    // the previous call of a chain: its weighted combine runs here, in chunks
    // interleaved among this call's FFN1 tiles (prev_chunks = 0: none)
    const uint16_t *prev_ystage;
    const float *prev_gates;
    uint16_t *prev_out;
    int prev_T, prev_chunks;
    int NT1, NT2, BN2, k1, k2;
    int band1;                // row tiles per band of the FFN1 order (ring-bounded)
    int *counters;            // zeroed: [0] next tile, [1] next minibatch, [2] unused,
                              // then ready[mt], consumed[mt], h_done[mt]
    int max_mt;
    uint32_t *status;
    uint64_t wait_ns;
};

// Bounded spin until *p >= target (acquire).
__device__ __forceinline__ bool spin_ge(const int *p, int target, const FusedArgs &a,
                                        volatile int *abort_flag)
{
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire_gpu(p) >= target) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > a.wait_ns) {
                report_timeout(a.status, abort_flag);
                return false;
            }
        }
        __nanosleep(64);
    }
}

// Tile order of one phase (FFN1 or FFN2, NT N tiles per row tile): expert by
// expert; inside an expert, bands of up to `band` row tiles; inside a band,
// N tile by N tile with the band's row tiles innermost, so the CTAs running
// side by side share a weight tile through L2 and a band's ring rows are
// released by tiles that all come before the next band's.
struct PTile {
    int m, n;
};
__device__ __forceinline__ PTile decode_phase_tile(int t, const int *s_pad, int E, int NT, int band)
{
    int lo = 0, hi = E;  // last expert whose first tile index <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((s_pad[mid] / 128) * NT <= t) lo = mid;
        else hi = mid;
    }
    const int m0 = s_pad[lo] / 128;
    const int mt = s_pad[lo + 1] / 128 - m0;
    const int b = band < mt ? band : mt;  // b * NT <= the expert's tile count
    const int local = t - m0 * NT;
    const int j = local / (b * NT);
    const int bm = mt - j * b < b ? mt - j * b : b;
    const int ll = local - j * b * NT;
    PTile r;
    r.n = ll / bm;
    r.m = m0 + j * b + ll % bm;
    return r;
}

// index of the MX scale tile of (k element x, row y) in a [rows, K] matrix
__device__ __forceinline__ int sf_tile(int x, int y, int64_t rows)
{
    return static_cast<int>((x >> 7) * (rows >> 7) + (y >> 7));
}

// expert whose padded segment holds row q (last e with pad[e] <= q)
__device__ __forceinline__ int expert_of_row(const int *s_pad, int E, int64_t q)
{
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pad[mid] <= q) lo = mid;
        else hi = mid;
    }
    return lo;
}

// MXFP8 quantisation of elements [c0, c0 + 1024) of a BF16 row held in shared
// memory, one MX block of 32 per lane (the arithmetic of mx_quant_stretch,
// laid out for instruction-level parallelism): lane l reads block l as four
// 16-byte pieces in a rotated order (conflict-free: each read by the warp is
// four wavefronts), takes the block's amax in registers, writes its 32 codes
// and, with two shuffles, lanes 4g write the scale words of the chunk's
// k-groups.  A tail chunk (d - c0 < 1024) leaves the lanes past it idle
// except for the shuffles.
__device__ __forceinline__ void mx_quant_block_per_lane(const uint8_t *row, int c0, int d, int lane,
                                                        uint8_t *codes_row, uint32_t *scales,
                                                        int64_t scale_row, int64_t scale_rows)
{
    const int nblk = (d - c0) >= 1024 ? 32 : (d - c0) / 32;
    const bool on = lane < nblk;
    const int rot = (lane >> 1) & 3;
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[q] = make_uint4(0, 0, 0, 0);
        if (on) v[q] = *reinterpret_cast<const uint4 *>(row + (c0 + 32 * lane) * 2 + 16 * ((q + rot) & 3));
    }
    float f[32];
#pragma unroll
    for (int p2 = 0; p2 < 4; ++p2) {
        const int qp = (p2 - rot) & 3;  // the read that fetched piece p2
        uint4 src = v[0];
        if (qp == 1) src = v[1];
        if (qp == 2) src = v[2];
        if (qp == 3) src = v[3];
        const uint32_t w[4] = {src.x, src.y, src.z, src.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[8 * p2 + 2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
            f[8 * p2 + 2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
    const int x = mx_scale_exp(amax);
    const float inv = mx_inv_scale(x);
    uint32_t code[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        code[i] = pack_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv) |
                  (pack_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
    if (on) {
        uint4 *o = reinterpret_cast<uint4 *>(codes_row + c0 + 32 * lane);
        o[0] = make_uint4(code[0], code[1], code[2], code[3]);
        o[1] = make_uint4(code[4], code[5], code[6], code[7]);
    }
    // scale byte of block l at byte l % 4 of the word of k-group (c0 + 32 l) / 128
    uint32_t word = static_cast<uint32_t>(x + 127) << (8 * (lane & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    if (on && (lane & 3) == 0)
        scales[mx_word_index((c0 + 32 * lane) >> 7, scale_row, scale_rows)] = word;
}

// Gather role of the fused forward: pull expert-ordered rows into the token
// ring (quantised when MXFP8) in minibatches claimed from a global counter,
// after the ring rows' previous occupants were loaded by every FFN1 tile, and
// publish each 64-row half of a row tile in ready[].  Every thread of the CTA
// calls it.
//
// Rows are staged through shared memory: the GEMM stage buffers (`stage`,
// unused while this CTA gathers) hold up to 16 source rows, each fetched by
// one bulk copy completing on its own mbarrier, so ~190 KB of row reads are in
// flight per SM while the six warps quantise (MXFP8) or copy (BF16) the rows
// already landed.  A row too large for two slots is read directly.
template <bool MX>
__device__ __forceinline__ void gather_rows(const FusedArgs &a, const int *s_pad, int64_t pad_end, int *s_unit,
                                            volatile int *abort_flag, int *next_unit, int *ready,
                                            int *consumed, int warp, int lane, int nwarps,
                                            uint8_t *stage, int stage_bytes)
{
    const int units = static_cast<int>((pad_end + a.mb - 1) / a.mb);
    const int ring_tiles = static_cast<int>(a.ring_rows / kBM);
    // staging layout: 16 mbarriers, the unit's row and token lists, then slots
    constexpr int kHdr = 2304;
    const int row_bytes = a.d * 2;
    const int slot_bytes = (row_bytes + 127) & ~127;
    int ns = (stage_bytes - kHdr) / slot_bytes;
    ns = ns > 16 ? 16 : ns;
    const bool staged = ns >= 2;
    uint64_t *gbar = reinterpret_cast<uint64_t *>(stage);
    int *lst_q = reinterpret_cast<int *>(stage + 128);  // [256] padded rows of the unit with a token
    int *lst_t = lst_q + 256;                            // [256] their tokens
    int *s_n = lst_t + 256;
    uint8_t *slots = stage + kHdr;
    if (staged) {
        if (threadIdx.x == 0) {
            for (int j = 0; j < ns; ++j) mbar_init(&gbar[j], 1);
            fence_barrier_init();
        }
        __syncthreads();
    }
    uint32_t base = 0;  // rows this CTA has staged so far: slot = base % ns, parity = (base / ns) & 1
    for (;;) {
        if (threadIdx.x == 0) *s_unit = atomicAdd(next_unit, 1);
        __syncthreads();
        const int u = *s_unit;
        if (u >= units || *abort_flag) break;
        const int64_t r0 = static_cast<int64_t>(u) * a.mb;
        const int64_t r1 = r0 + a.mb < pad_end ? r0 + a.mb : pad_end;
        if (threadIdx.x == 0) {
            // the ring rows' previous occupants must have been loaded by every FFN1 tile
            for (int64_t q = r0; q < r1; q += kBM) {
                const int m_prev = static_cast<int>(q / kBM) - ring_tiles;
                if (m_prev >= 0 && !spin_ge(&consumed[m_prev], a.NT1, a, abort_flag)) break;
            }
        }
        __syncthreads();
        if (*abort_flag) break;
        if (staged) {
            // the unit's rows that hold a token (padding rows: nothing to pull)
            if (threadIdx.x == 0) *s_n = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < static_cast<int>(r1 - r0); i += blockDim.x) {
                const int64_t q = r0 + i;
                const int e = expert_of_row(s_pad, a.E, q);
                const int64_t local = q - s_pad[e];
                if (local < a.counts[e]) {
                    const int idx = atomicAdd(s_n, 1);
                    lst_q[idx] = static_cast<int>(q);
                    lst_t[idx] = a.row_tok[a.offsets[e] + local];
                }
            }
            __syncthreads();
            const int n = *s_n;
            auto issue = [&](int i) {
                const int slot = static_cast<int>((base + static_cast<uint32_t>(i)) % static_cast<uint32_t>(ns));
                mbar_arrive_expect_tx(&gbar[slot], static_cast<uint32_t>(row_bytes));
                bulk_load(slots + slot * slot_bytes, source_row(a.src, lst_t[i], a.d), static_cast<uint32_t>(row_bytes),
                          &gbar[slot]);
            };
            if (threadIdx.x == 0)
                for (int i = 0; i < n && i < ns; ++i) issue(i);
            for (int i = warp; i < n; i += nwarps) {
                const uint32_t g = base + static_cast<uint32_t>(i);
                const int slot = static_cast<int>(g % static_cast<uint32_t>(ns));
                if (!wait_bar(&gbar[slot], (g / static_cast<uint32_t>(ns)) & 1u, a.status, a.wait_ns, abort_flag)) break;
                const uint8_t *row = slots + slot * slot_bytes;
                const int64_t rr = lst_q[i] % a.ring_rows;
                if (!MX) {
                    uint4 *o = reinterpret_cast<uint4 *>(a.ring + rr * a.d * 2);
                    const uint4 *in = reinterpret_cast<const uint4 *>(row);
                    for (int c = lane; c < a.d / 8; c += 32) o[c] = in[c];
                } else {
                    uint8_t *codes_row = a.ring + rr * a.d;
                    for (int c0 = 0; c0 < a.d; c0 += 1024)
                        mx_quant_block_per_lane(row, c0, a.d, lane, codes_row, a.ring_scales, rr, a.ring_rows);
                }
                // this warp's reads of the slot come before the next bulk copy into it
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0 && i + ns < n) issue(i + ns);
            }
            base += static_cast<uint32_t>(n);
        } else {
            for (int64_t q = r0 + warp; q < r1; q += nwarps) {
                const int e = expert_of_row(s_pad, a.E, q);
                const int64_t local = q - s_pad[e];
                if (local >= a.counts[e]) continue;  // padding row: nothing to pull
                const int t = a.row_tok[a.offsets[e] + local];
                const uint4 *in = reinterpret_cast<const uint4 *>(source_row(a.src, t, a.d));
                const int64_t rr = q % a.ring_rows;
                // 16 vectors of 16 bytes per lane in flight (8 KB per warp): a gather
                // CTA runs six warps and the row reads miss L2, so the loads in
                // flight set the gather rate
                if (!MX) {
                    uint4 *o = reinterpret_cast<uint4 *>(a.ring + rr * a.d * 2);
                    for (int c0 = 0; c0 < a.d / 8; c0 += 512) {
                        uint4 v[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int c = c0 + 32 * u + lane;
                            v[u] = c < a.d / 8 ? __ldg(in + c) : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int c = c0 + 32 * u + lane;
                            if (c < a.d / 8) o[c] = v[u];
                        }
                    }
                } else {
                    uint8_t *codes_row = a.ring + rr * a.d;
                    for (int c0 = 0; c0 < a.d; c0 += 4096) {
                        uint4 raw[16];
#pragma unroll
                        for (int w = 0; w < 16; ++w) {
                            const int cu = c0 + 256 * w;
                            const int nvalid = cu >= a.d ? 0 : (a.d - cu >= 256 ? 32 : 16);
                            raw[w] = lane < nvalid ? __ldg(in + (cu >> 3) + lane) : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int w = 0; w < 16; ++w) {
                            const int cu = c0 + 256 * w;
                            if (cu < a.d)
                                mx_quant_stretch(raw[w], lane, a.d - cu >= 256 ? 32 : 16, codes_row, cu,
                                                 a.ring_scales, rr, a.ring_rows);
                        }
                    }
                }
            }
        }
        fence_proxy_async_global();
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            for (int64_t q = r0; q < r1; q += 64)  // hand over in 64-row halves of row tiles
                red_release_gpu_add(&ready[q / kBM], 1);
        }
    }
    __syncthreads();
    if (staged) {
        // the staging bytes go back to the GEMM role's TMA loads
        if (threadIdx.x == 0 && !*abort_flag)
            for (int j = 0; j < ns; ++j) mbar_inval(&gbar[j]);
        fence_proxy_async_shared();
        __syncthreads();
    }
}

// Ids in the tile queue: with a previous call to combine, its C combine chunks
// sit among the FFN1 tiles, one every s = (T1 + C) / C ids (id c*s + s - 1 is
// chunk c); every other id is GEMM tile `tile` in the usual order.  Returns the
// chunk index, or -1 with *tile set.
__device__ __forceinline__ int split_queue_id(int id, int T1, int C, int *tile)
{
    if (C > 0) {
        const int s = (T1 + C) / C;
        if (id < C * s) {
            if (id % s == s - 1) return id / s;
            *tile = id - (id + 1) / s;
            return -1;
        }
        *tile = id - C;
        return -1;
    }
    *tile = id;
    return -1;
}

// One token of the weighted combine by one warp: out[t] = BF16 of the fmaf fold
// over j = 0..k-1 of g_tj * y_tj from 0 -- the separate combine kernel's order
// and access pattern (16 columns a lane, all 2k slot loads in flight).
__device__ __forceinline__ void combine_token_warp(const uint16_t *ystage, const float *gates, uint16_t *out,
                                                   int64_t t, int k, int d, int lane)
{
    for (int64_t c = 2 * lane; c < d / 8; c += 64) {
        uint4 y[MOK_MAX_TOPK][2];
        float g[MOK_MAX_TOPK];
#pragma unroll
        for (int j = 0; j < MOK_MAX_TOPK; ++j) {
            if (j < k) {
                g[j] = gates[t * k + j];
                const uint4 *row = reinterpret_cast<const uint4 *>(ystage + (t * k + j) * d) + c;
                y[j][0] = row[0];
                y[j][1] = row[1];
            }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int j = 0; j < MOK_MAX_TOPK; ++j) {
                if (j < k) {
                    const uint32_t w[4] = {y[j][hh].x, y[j][hh].y, y[j][hh].z, y[j][hh].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = fmaf(g[j], bf16_bits_to_float(w[q] & 0xFFFFu), acc[2 * q]);
                        acc[2 * q + 1] = fmaf(g[j], bf16_bits_to_float(w[q] >> 16), acc[2 * q + 1]);
                    }
                }
            }
            reinterpret_cast<uint4 *>(out + t * d)[c + hh] =
                make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                           pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
        }
    }
}

template <bool MX>
__global__ void __launch_bounds__(kFThreads, 1)
    k_moe_fused(const __grid_constant__ FusedMaps pm, const __grid_constant__ FusedArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = sA + kStages * kAStage;
    uint8_t *sSF = sB + kStages * kBStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSF + (MX ? kStages * (kSfaBytes + kSfbBytes) : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + kStages;
    uint64_t *sf_ready = bars + 2 * kStages;  // MXFP8: the stage's scales are in TMEM
    uint64_t *sf_full = bars + 3 * kStages;   // MXFP8: the stage's scale bytes have landed
    uint64_t *acc_full = bars + 4 * kStages;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *tq_full = acc_empty + 1;
    uint64_t *tq_empty = tq_full + kTQ;
    int *tq = reinterpret_cast<int *>(tq_empty + kTQ);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(tq + kTQ);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *s_unit = reinterpret_cast<int *>(tmem_holder + 2);
    int *s_pad = reinterpret_cast<int *>(tmem_holder + 4);  // [E + 1]
    uint32_t *stage_out = reinterpret_cast<uint32_t *>(s_pad + MOK_MAX_EXPERTS + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int *next_tile = a.counters;
    int *next_unit = a.counters + 1;
    int *ready = a.counters + 3;
    int *consumed = ready + a.max_mt;
    int *h_done = consumed + a.max_mt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 1);
            mbar_init(&sf_full[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        for (int i = 0; i < kTQ; ++i) {
            mbar_init(&tq_full[i], 1);
            mbar_init(&tq_empty[i], MX ? 6 : 5);  // MMA, 4 epilogue warps (+ scale copier)
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&pm.ring);
        prefetch_tmap(&pm.g);
        prefetch_tmap(&pm.u);
        prefetch_tmap(&pm.h);
        prefetch_tmap(&pm.dn);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) s_pad[e] = a.pad_offsets[e];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int64_t pad_end = s_pad[a.E];
    const int total_mt = static_cast<int>(pad_end / kBM);
    const int T1 = total_mt * a.NT1;
    const int total_tiles = T1 + total_mt * a.NT2;
    const int total_ids = total_tiles + a.prev_chunks;  // GEMM tiles and the previous call's combine chunks
    constexpr int kE = MX ? 128 : 64;

    // ---------------------------------------------------------- gather role
    if (!a.prologue && static_cast<int>(blockIdx.x) < a.n_gather)
        gather_rows<MX>(a, s_pad, pad_end, s_unit, abort_flag, next_unit, ready, consumed, warp, lane,
                        kFThreads / 32, smem, kStages * (kAStage + kBStage));

    // ------------------------------------------------------------ GEMM role
    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, qs = 0, qphase = 0;
            for (;;) {
                int qid = *abort_flag ? -1 : atomicAdd(next_tile, 1);
                if (qid >= total_ids) qid = -1;
                if (!wait_bar(&tq_empty[qs], qphase ^ 1u, a.status, a.wait_ns, abort_flag)) break;
                tq[qs] = qid;
                mbar_arrive(&tq_full[qs]);
                if (++qs == kTQ) {
                    qs = 0;
                    qphase ^= 1u;
                }
                if (qid < 0) break;
                int tile;
                if (split_queue_id(qid, T1, a.prev_chunks, &tile) >= 0) continue;  // a combine chunk: no loads
                const bool f1 = tile < T1;
                const PTile pt = f1 ? decode_phase_tile(tile, s_pad, a.E, a.NT1, a.band1)
                                    : decode_phase_tile(tile - T1, s_pad, a.E, a.NT2, 1 << 30);
                const int m = pt.m, n = pt.n;
                if (m < 0 || m >= total_mt || n < 0 || n >= (f1 ? a.NT1 : a.NT2)) {
                    report_timeout(a.status, abort_flag);  // a schedule bug: stop, touch nothing
                    break;
                }
                const int e = expert_of_row(s_pad, a.E, static_cast<int64_t>(m) * kBM);
                const int cnt_e = a.counts[e];
                if (f1 ? !(a.prologue || spin_ge(&ready[m], 2, a, abort_flag))
                       : !spin_ge(&h_done[m], 4 * a.NT1, a, abort_flag))
                    break;
                fence_proxy_async_global();
                const int BN = f1 ? 256 : a.BN2;
                // every tile holds at least one of its expert's rows: 64 or 128 to load
                const int arows = a_rows_to_load(cnt_e, static_cast<int64_t>(m) * kBM - s_pad[e]);
                const uint32_t stage_bytes = arows * kBKBytes + (BN / 128) * 16384;
                const uint32_t sf_bytes = kSfaBytes + (BN / 128) * 512;
                const int kst = f1 ? a.k1 : a.k2;
                const int ya = f1 ? static_cast<int>((static_cast<int64_t>(m) * kBM) % a.ring_rows) : m * kBM;
                const int yb = f1 ? e * a.F + n * 128 : e * a.d + n * BN;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&empty[stage], phase ^ 1u, a.status, a.wait_ns, abort_flag)) goto producer_done;
                    uint8_t *dA = sA + stage * kAStage;
                    uint8_t *dB = sB + stage * kBStage;
                    const int x = ks * kE;
                    if constexpr (MX) {
                        // the scales first, on their own barrier: the copier copies them
                        // into TMEM as soon as they land, so the copies (which the tensor
                        // pipe runs in order with the MMAs already issued) are done before
                        // the stage's operands arrive
                        uint8_t *dS = sSF + stage * (kSfaBytes + kSfbBytes);
                        mbar_arrive_expect_tx(&sf_full[stage], sf_bytes);
                        if (f1) {
                            bulk_load(dS, a.ring_scales + scale_word(x, ya, a.ring_rows), kSfaBytes, &sf_full[stage]);
                            bulk_load(dS + kSfaBytes, a.s_gate + scale_word(x, yb, a.EF), 512, &sf_full[stage]);
                            bulk_load(dS + kSfaBytes + 512, a.s_up + scale_word(x, yb, a.EF), 512, &sf_full[stage]);
                        } else {
                            bulk_load(dS, a.h_scales + scale_word(x, ya, a.h_rows), kSfaBytes, &sf_full[stage]);
                            bulk_load(dS + kSfaBytes, a.s_down + scale_word(x, yb, a.Ed), (BN / 128) * 512,
                                      &sf_full[stage]);
                        }
                    }
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    if (f1) {
                        tma_load_2d(dA, arows == kBM ? &pm.ring : &pm.ring64, &full[stage], x, ya);
                        tma_load_2d(dB, &pm.g, &full[stage], x, yb);
                        tma_load_2d(dB + 16384, &pm.u, &full[stage], x, yb);
                    } else {
                        tma_load_2d(dA, arows == kBM ? &pm.h : &pm.h64, &full[stage], x, ya);
                        tma_load_2d(dB, &pm.dn, &full[stage], x, yb);
                        if (BN == 256) tma_load_2d(dB + 16384, &pm.dn, &full[stage], x, yb + 128);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc_phase = 0, qs = 0, qphase = 0;
            const uint64_t adesc0 = sdesc_k_sw128(smem_u32(sA));
            const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(sB));
            for (;;) {
                if (!wait_bar(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
                const int qid = tq[qs];
                mbar_arrive(&tq_empty[qs]);
                if (++qs == kTQ) {
                    qs = 0;
                    qphase ^= 1u;
                }
                if (qid < 0) break;
                int tile;
                if (split_queue_id(qid, T1, a.prev_chunks, &tile) >= 0) continue;
                const bool f1 = tile < T1;
                const int m = f1 ? decode_phase_tile(tile, s_pad, a.E, a.NT1, a.band1).m : 0;
                const int BN = f1 ? 256 : a.BN2;
                const int kst = f1 ? a.k1 : a.k2;
                // MXFP8: the scale-factor byte selectors (bits 4-5 and 29-30) are or-ed in per MMA
                const uint32_t idesc = MX ? idesc_mxf8(kBM, BN, 0, 0) : idesc_bf16(kBM, BN);
                if (!wait_bar(acc_empty, acc_phase ^ 1u, a.status, a.wait_ns, abort_flag)) break;
                tc_fence_after();
                for (int ks = 0; ks < kst; ++ks) {
                    // the operands, and (MXFP8) the stage's scales in TMEM (sf_ready)
                    if (!wait_bar(&full[stage], phase, a.status, a.wait_ns, abort_flag)) goto mma_done;
                    if (MX && !wait_bar(&sf_ready[stage], phase, a.status, a.wait_ns, abort_flag)) goto mma_done;
                    tc_fence_after();
                    if (f1 && ks == kst - 1) {
                        // every ring row of row tile m this tile needs is now in shared memory
                        __threadfence();
                        red_release_gpu_add(&consumed[m], 1);
                    }
                    // descriptors: the stage's base plus 32 bytes of K per MMA (address >> 4
                    // in the low bits; every shared address here is below 256 KB, so no carry)
                    const uint64_t ad0 = adesc0 + static_cast<uint64_t>((stage * kAStage) >> 4);
                    const uint64_t bd0 = bdesc0 + static_cast<uint64_t>((stage * kBStage) >> 4);
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
                        if (MX)
                            mma_mxf8(tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc | (kk << 4) | (kk << 29), sfa_col,
                                     sfb_col, accum);
                        else mma_bf16(tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc, accum);
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit(acc_full);
                acc_phase ^= 1u;
            }
        mma_done:;
        }
    } else if (warp == kScaleWarp) {
        if (MX && lane == 0) {
            // ------------------------------------------------ scale copier
            // the same tile and stage sequence as the MMA issuer: once a stage's
            // scale bytes have landed (sf_full), copy its A and B scales into the
            // stage's TMEM columns and commit to sf_ready (a scale slot is refilled
            // only after empty[stage], i.e. after the MMAs that read it completed)
            uint32_t stage = 0, phase = 0, qs = 0, qphase = 0;
            const uint64_t sfdesc0 = sdesc_sf(smem_u32(sSF));
            for (;;) {
                if (!wait_bar(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
                const int qid = tq[qs];
                mbar_arrive(&tq_empty[qs]);
                if (++qs == kTQ) {
                    qs = 0;
                    qphase ^= 1u;
                }
                if (qid < 0) break;
                int tile;
                if (split_queue_id(qid, T1, a.prev_chunks, &tile) >= 0) continue;
                const bool f1 = tile < T1;
                const int BN = f1 ? 256 : a.BN2;
                const int kst = f1 ? a.k1 : a.k2;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&sf_full[stage], phase, a.status, a.wait_ns, abort_flag)) goto copier_done;
                    tc_fence_after();
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
                    const uint64_t sd = sfdesc0 + static_cast<uint64_t>((stage * (kSfaBytes + kSfbBytes)) >> 4);
                    tmem_cp_32x128b_warpx4(sfa_col, sd);
                    tmem_cp_32x128b_warpx4(sfb_col, sd + (kSfaBytes >> 4));
                    if (BN == 256) tmem_cp_32x128b_warpx4(sfb_col + 4, sd + ((kSfaBytes + 512) >> 4));
                    tc_commit(&sf_ready[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        copier_done:;
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        uint32_t acc_phase = 0, qs = 0, qphase = 0;
        for (;;) {
            if (!wait_bar(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
            const int qid = tq[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive(&tq_empty[qs]);
            if (++qs == kTQ) {
                qs = 0;
                qphase ^= 1u;
            }
            if (qid < 0) break;
            int tile;
            const int chunk = split_queue_id(qid, T1, a.prev_chunks, &tile);
            if (chunk >= 0) {
                // the previous call's combine: one token per epilogue warp
                const int64_t t = static_cast<int64_t>(chunk) * 4 + (warp - 2);
                if (t < a.prev_T) combine_token_warp(a.prev_ystage, a.prev_gates, a.prev_out, t, a.k, a.d, lane);
                continue;
            }
            const bool f1 = tile < T1;
            const PTile pt = f1 ? decode_phase_tile(tile, s_pad, a.E, a.NT1, a.band1)
                                : decode_phase_tile(tile - T1, s_pad, a.E, a.NT2, 1 << 30);
            const int m = pt.m, n = pt.n;
            if (m < 0 || m >= total_mt || n < 0 || n >= (f1 ? a.NT1 : a.NT2)) {
                report_timeout(a.status, abort_flag);
                break;
            }
            const int64_t q = static_cast<int64_t>(m) * kBM + r;   // padded row of this thread
            const int e = expert_of_row(s_pad, a.E, static_cast<int64_t>(m) * kBM);
            const int64_t row_in_e = q - s_pad[e];
            const bool valid = row_in_e < a.counts[e];
            // FFN2: this row's token slot in ystage, looked up while the tile's MMAs
            // run (the accumulator is handed back only after the lookup)
            uint16_t *dst = nullptr;
            if (!f1 && valid) {
                const int64_t p = a.offsets[e] + row_in_e;
                dst = a.ystage + (static_cast<int64_t>(a.row_tok[p]) * a.k + a.row_j[p]) * a.d + n * a.BN2;
            }
            if (!wait_bar(acc_full, acc_phase, a.status, a.wait_ns, abort_flag)) break;
            tc_fence_after();
            bool released = false;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(acc_empty);
                released = true;
            };
            if (f1) {
                epi_ffn1<MX>(trow, valid, q, n * 128, a.F, a.h, a.h_scales, a.h_rows, a.saved_a, a.saved_b,
                             a.saved_h, stage_out + (warp - 2) * kStageWords, lane, release);
            } else {
                epi_rows_bf16(trow, a.BN2, false, valid, dst, stage_out + (warp - 2) * kStageWords, lane,
                              release);
            }
            if (!released) release();
            acc_phase ^= 1u;
            // an FFN1 tile publishes this warp's quarter of its h rows for the FFN2
            // tiles (TMA reads them); each epilogue warp counts for itself, so no
            // barrier ties the four warps together.  FFN2 tiles' ystage rows are read
            // by the combine kernel that follows this one on the stream.
            if (f1) {
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    red_release_gpu_add(&h_done[m], 1);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }

}

// ---------------------------------------------------------------------------
// The same forward with the GEMM role on CTA pairs (cta_group::2): clusters of
// two CTAs compute 256-row x 256-column tiles -- two consecutive 128-row tiles
// of one expert, each CTA loading its own rows and one half of B (FFN1: the
// even CTA the W_g rows, the odd CTA the W_u rows; FFN2: 128 rows of W_d
// each), with every load counted on the even CTA's barrier.  Per flop each SM
// loads a third fewer bytes than with one CTA per tile.  The even CTA's
// scheduler thread claims pair tiles from the global counter and hands their
// ids to both CTAs through a cluster-wide queue; the even CTA issues the MMAs
// and scale copies; both CTAs run the epilogue of their own rows.  When an
// expert has an odd number of row tiles its last pair tile has a ghost odd
// half: the odd CTA loads only its half of B (its A rows in shared memory are
// stale; their results are discarded), stores nothing and signals no counter.
// A half with 64 valid rows or fewer loads only those 64 rows of A.  Gather CTAs come in pairs and a pair
// enters the GEMM role only once both of its CTAs have finished gathering, so
// a pair never holds a tile while one of its CTAs waits in the gather role.
// Tiles keep the single-CTA kernel's per-row arithmetic, so results are
// bit-identical to it.
// ---------------------------------------------------------------------------
constexpr int kFPStages = 6;
constexpr int kFPStage = kAStage + 128 * kBKBytes;  // 32 KB: A rows + one half of B


// Pair tile t of one phase (NT N tiles per pair row): expert e, pair row j of
// that expert (row tiles 2j and 2j + 1 of its segment), N tile n; the same
// expert / band / N-tile / row order as decode_phase_tile, in pair rows.
struct PPTile {
    int e, j, n;
};
__device__ __forceinline__ PPTile decode_pair_tile(int t, const int *s_pp, int E, int NT, int band)
{
    int lo = 0, hi = E;  // last expert whose first tile index <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pp[mid] * NT <= t) lo = mid;
        else hi = mid;
    }
    const int pr = s_pp[lo + 1] - s_pp[lo];
    const int b = band < pr ? band : pr;
    const int local = t - s_pp[lo] * NT;
    const int jb = local / (b * NT);
    const int bm = pr - jb * b < b ? pr - jb * b : b;
    const int ll = local - jb * b * NT;
    PPTile r;
    r.e = lo;
    r.n = ll / bm;
    r.j = jb * b + ll % bm;
    return r;
}

template <bool MX>
__global__ void __launch_bounds__(kFThreads, 1)
    k_moe_fused_pair(const __grid_constant__ FusedMaps pm, const __grid_constant__ FusedArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sT = smem;
    uint8_t *sSF = sT + kFPStages * kFPStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSF + (MX ? kFPStages * (kSfaBytes + kSfbBytes) : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + kFPStages;
    uint64_t *sf_ready = bars + 2 * kFPStages;  // MXFP8, even CTA: the stage's scales are in TMEM
    uint64_t *sf_full = bars + 3 * kFPStages;   // MXFP8, even CTA: both CTAs' scale bytes have landed
    uint64_t *acc_full = bars + 4 * kFPStages;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *tq_full = acc_empty + 1;
    uint64_t *tq_empty = tq_full + kTQ;
    int *tq = reinterpret_cast<int *>(tq_empty + kTQ);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(tq + kTQ);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *s_unit = reinterpret_cast<int *>(tmem_holder + 2);
    int *s_pad = reinterpret_cast<int *>(tmem_holder + 4);   // [E + 1]
    int *s_pp = s_pad + MOK_MAX_EXPERTS + 4;                 // [E + 1] pair-row prefix
    uint32_t *stage_out = reinterpret_cast<uint32_t *>(s_pp + MOK_MAX_EXPERTS + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    int *next_tile = a.counters;
    int *next_unit = a.counters + 1;
    int *ready = a.counters + 3;
    int *consumed = ready + a.max_mt;
    int *h_done = consumed + a.max_mt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 1);
            mbar_init(&sf_full[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 8);  // four epilogue warps of each CTA
        for (int i = 0; i < kTQ; ++i) {
            mbar_init(&tq_full[i], 1);
            // even: MMA + 4 epilogue warps (+ scale copier); odd: producer + 4 epilogue warps
            mbar_init(&tq_empty[i], MX ? 11 : 10);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&pm.ring);
        prefetch_tmap(&pm.g);
        prefetch_tmap(&pm.u);
        prefetch_tmap(&pm.h);
        prefetch_tmap(&pm.dn);
    }
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) s_pad[e] = a.pad_offsets[e];
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive, store or load
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, kTmemCols);
        tmem_relinquish_pair();
    }
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < a.E; ++e) {
            s_pp[e] = run;
            run += ((s_pad[e + 1] - s_pad[e]) / kBM + 1) / 2;
        }
        s_pp[a.E] = run;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int64_t pad_end = s_pad[a.E];
    const int total_mt = static_cast<int>(pad_end / kBM);
    const int total_pr = s_pp[a.E];
    const int T1 = total_pr * a.NT1;
    const int total_tiles = T1 + total_pr * a.NT2;
    const int total_ids = total_tiles + a.prev_chunks;  // pair tiles and the previous call's combine chunks
    constexpr int kE = MX ? 128 : 64;
    const int bandp = a.band1 >= (1 << 29) ? (1 << 30) : (a.band1 / 2 > 0 ? a.band1 / 2 : 1);

    // ---------------------------------------------------------- gather role
    if (!a.prologue && static_cast<int>(blockIdx.x) < a.n_gather) {
        gather_rows<MX>(a, s_pad, pad_end, s_unit, abort_flag, next_unit, ready, consumed, warp, lane,
                        kFThreads / 32, smem, kFPStages * kFPStage);
        cluster_sync_all();  // the pair joins the GEMM role together
    }

    // what a pair tile means for this CTA: its row tile m (ghost: none), N tile
    struct Job {
        bool f1, ghost, ghost_odd;
        int e, m0, n;
    };
    auto job_of = [&](int tile) {
        Job jb;
        jb.f1 = tile < T1;
        const PPTile pt = jb.f1 ? decode_pair_tile(tile, s_pp, a.E, a.NT1, bandp)
                                : decode_pair_tile(tile - T1, s_pp, a.E, a.NT2, 1 << 30);
        jb.e = pt.e;
        jb.n = pt.n;
        jb.m0 = s_pad[pt.e] / kBM + 2 * pt.j;
        jb.ghost_odd = jb.m0 + 1 >= s_pad[pt.e + 1] / kBM;
        jb.ghost = rank == 1 && jb.ghost_odd;
        return jb;
    };
    const uint32_t full0 = mapa_shared(smem_u32(full), 0);
    const uint32_t sf_full0 = mapa_shared(smem_u32(sf_full), 0);

    // ------------------------------------------------------------ GEMM role
    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, qs = 0, qphase = 0;
            const uint32_t tq_full_odd = mapa_shared(smem_u32(tq_full), 1);
            const uint32_t tq_odd = mapa_shared(smem_u32(tq), 1);
            const uint32_t tq_empty_even = mapa_shared(smem_u32(tq_empty), 0);
            for (;;) {
                int tile;
                if (rank == 0) {
                    // scheduler: claim the next pair tile and hand it to both CTAs
                    tile = *abort_flag ? -1 : atomicAdd(next_tile, 1);
                    if (tile >= total_ids) tile = -1;
                    if (!wait_bar(&tq_empty[qs], qphase ^ 1u, a.status, a.wait_ns, abort_flag)) tile = -1;
                    tq[qs] = tile;
                    st_shared_cluster(tq_odd + qs * 4, static_cast<uint32_t>(tile));
                    mbar_arrive(&tq_full[qs]);
                    mbar_arrive_remote(tq_full_odd + qs * 8);
                } else {
                    if (!wait_bar_cluster(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
                    tile = tq[qs];
                    mbar_arrive_remote(tq_empty_even + qs * 8);
                }
                if (++qs == kTQ) {
                    qs = 0;
                    qphase ^= 1u;
                }
                if (tile < 0) break;
                if (split_queue_id(tile, T1, a.prev_chunks, &tile) >= 0) continue;  // a combine chunk: no loads
                const Job jb = job_of(tile);
                const int m = jb.m0 + static_cast<int>(rank);
                if (jb.e < 0 || jb.e >= a.E || m >= total_mt + 1 || jb.n < 0 || jb.n >= (jb.f1 ? a.NT1 : a.NT2)) {
                    report_timeout(a.status, abort_flag);  // a schedule bug: stop, touch nothing
                    break;
                }
                // rows of A each half loads (a ghost half none: it only loads its half of
                // B, and its results are discarded); the even CTA's barrier counts both
                const int cnt_e = a.counts[jb.e];
                const int64_t rel0 = static_cast<int64_t>(jb.m0) * kBM - s_pad[jb.e];
                const int rows0 = a_rows_to_load(cnt_e, rel0), rows1 = a_rows_to_load(cnt_e, rel0 + kBM);
                const int my_rows = rank ? rows1 : rows0;
                const uint32_t tx = 2u * 128 * kBKBytes + static_cast<uint32_t>((rows0 + rows1) * kBKBytes);
                const uint32_t tx_sf = 2u * kSfbBytes + (rows0 ? kSfaBytes : 0) + (rows1 ? kSfaBytes : 0);
                if (my_rows > 0 && (jb.f1 ? !(a.prologue || spin_ge(&ready[m], 2, a, abort_flag))
                                          : !spin_ge(&h_done[m], 4 * a.NT1, a, abort_flag)))
                    break;
                fence_proxy_async_global();
                const int kst = jb.f1 ? a.k1 : a.k2;
                const int64_t arows = jb.f1 ? a.ring_rows : a.h_rows;
                const int ya = jb.f1 ? static_cast<int>((static_cast<int64_t>(m) * kBM) % a.ring_rows) : m * kBM;
                const CUtensorMap *amap = jb.f1 ? (my_rows == kBM ? &pm.ring : &pm.ring64)
                                                : (my_rows == kBM ? &pm.h : &pm.h64);
                // B rows of this CTA's half, and the first B row of the tile (scales)
                const int yb_tile = jb.f1 ? jb.e * a.F + jb.n * 128 : jb.e * a.d + jb.n * 256;
                const int yb = jb.f1 ? yb_tile : yb_tile + static_cast<int>(rank) * 128;
                const CUtensorMap *bmap = jb.f1 ? (rank ? &pm.u : &pm.g) : &pm.dn;
                const CUtensorMap *samap = jb.f1 ? &pm.s_ring : &pm.s_h;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&empty[stage], phase ^ 1u, a.status, a.wait_ns, abort_flag)) goto producer_done;
                    uint8_t *dA = sT + stage * kFPStage;
                    const int x = ks * kE;
                    const uint32_t fb = full0 + stage * 8;
                    if constexpr (MX) {
                        // the scales first, on their own barrier (see k_moe_fused)
                        const uint32_t sfb = sf_full0 + stage * 8;
                        uint8_t *dS = sSF + stage * (kSfaBytes + kSfbBytes);
                        if (rank == 0) mbar_arrive_expect_tx(&sf_full[stage], tx_sf);
                        if (my_rows > 0) tma_load_2d_pair(dS, samap, sfb, 0, sf_tile(x, ya, arows));
                        if (jb.f1) {
                            tma_load_2d_pair(dS + kSfaBytes, &pm.s_g, sfb, 0, sf_tile(x, yb_tile, a.EF));
                            tma_load_2d_pair(dS + kSfaBytes + 512, &pm.s_u, sfb, 0, sf_tile(x, yb_tile, a.EF));
                        } else {
                            tma_load_2d_pair(dS + kSfaBytes, &pm.s_dn, sfb, 0, sf_tile(x, yb_tile, a.Ed));
                            tma_load_2d_pair(dS + kSfaBytes + 512, &pm.s_dn, sfb, 0, sf_tile(x, yb_tile + 128, a.Ed));
                        }
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], tx);
                    if (my_rows > 0) tma_load_2d_pair(dA, amap, fb, x, ya);
                    tma_load_2d_pair(dA + kAStage, bmap, fb, x, yb);
                    if (++stage == kFPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------------------------------- even CTA: MMA issue for the pair
            uint32_t stage = 0, phase = 0, acc_phase = 0, qs = 0, qphase = 0;
            const uint64_t tdesc0 = sdesc_k_sw128(smem_u32(sT));
            for (;;) {
                if (!wait_bar(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
                int tile = tq[qs];
                mbar_arrive(&tq_empty[qs]);
                if (++qs == kTQ) {
                    qs = 0;
                    qphase ^= 1u;
                }
                if (tile < 0) break;
                if (split_queue_id(tile, T1, a.prev_chunks, &tile) >= 0) continue;
                const Job jb = job_of(tile);
                const int kst = jb.f1 ? a.k1 : a.k2;
                const uint32_t idesc = MX ? idesc_mxf8(2 * kBM, 256, 0, 0) : idesc_bf16(2 * kBM, 256);
                if (!wait_bar(acc_empty, acc_phase ^ 1u, a.status, a.wait_ns, abort_flag)) break;
                tc_fence_after();
                for (int ks = 0; ks < kst; ++ks) {
                    // both CTAs' operands, and (MXFP8) the stage's scales in TMEM
                    if (!wait_bar(&full[stage], phase, a.status, a.wait_ns, abort_flag)) goto mma_done;
                    if (MX && !wait_bar(&sf_ready[stage], phase, a.status, a.wait_ns, abort_flag)) goto mma_done;
                    tc_fence_after();
                    if (jb.f1 && ks == kst - 1) {
                        // every ring row of the pair's row tiles is now in shared memory
                        __threadfence();
                        red_release_gpu_add(&consumed[jb.m0], 1);
                        if (!jb.ghost_odd) red_release_gpu_add(&consumed[jb.m0 + 1], 1);
                    }
                    // descriptors: the stage's base plus 32 bytes of K per MMA (see k_moe_fused)
                    const uint64_t ad0 = tdesc0 + static_cast<uint64_t>((stage * kFPStage) >> 4);
                    const uint64_t bd0 = ad0 + (kAStage >> 4);
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
                        if (MX)
                            mma_mxf8_pair(tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc | (kk << 4) | (kk << 29), sfa_col,
                                          sfb_col, accum);
                        else mma_bf16_pair(tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc, accum);
                    }
                    tc_commit_pair(&empty[stage], 0x3);
                    if (++stage == kFPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit_pair(acc_full, 0x3);
                acc_phase ^= 1u;
            }
        mma_done:;
        }
    } else if (warp == kScaleWarp) {
        if (MX && lane == 0 && rank == 0) {
            // ---------------------------------- even CTA: scale copier for the pair
            // once a stage's scale bytes (both CTAs') have landed, copy them into
            // both CTAs' TMEM and commit to sf_ready (see k_moe_fused)
            uint32_t stage = 0, phase = 0, qs = 0, qphase = 0;
            const uint64_t sfdesc0 = sdesc_sf(smem_u32(sSF));
            for (;;) {
                if (!wait_bar(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
                int tile = tq[qs];
                mbar_arrive(&tq_empty[qs]);
                if (++qs == kTQ) {
                    qs = 0;
                    qphase ^= 1u;
                }
                if (tile < 0) break;
                if (split_queue_id(tile, T1, a.prev_chunks, &tile) >= 0) continue;
                const int kst = tile < T1 ? a.k1 : a.k2;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&sf_full[stage], phase, a.status, a.wait_ns, abort_flag)) goto copier_done;
                    tc_fence_after();
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
                    const uint64_t sd = sfdesc0 + static_cast<uint64_t>((stage * (kSfaBytes + kSfbBytes)) >> 4);
                    tmem_cp_32x128b_warpx4_pair(sfa_col, sd);
                    tmem_cp_32x128b_warpx4_pair(sfb_col, sd + (kSfaBytes >> 4));
                    tmem_cp_32x128b_warpx4_pair(sfb_col + 4, sd + ((kSfaBytes + 512) >> 4));
                    tc_commit_pair(&sf_ready[stage], 0x1);
                    if (++stage == kFPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        copier_done:;
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t acc_empty_even = mapa_shared(smem_u32(acc_empty), 0);
        const uint32_t tq_empty_even = mapa_shared(smem_u32(tq_empty), 0);
        uint32_t acc_phase = 0, qs = 0, qphase = 0;
        for (;;) {
            if (!wait_bar_cluster(&tq_full[qs], qphase, a.status, a.wait_ns, abort_flag)) break;
            int tile = tq[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tq_empty_even + qs * 8);
            if (++qs == kTQ) {
                qs = 0;
                qphase ^= 1u;
            }
            if (tile < 0) break;
            const int chunk = split_queue_id(tile, T1, a.prev_chunks, &tile);
            if (chunk >= 0) {
                // the previous call's combine: one token per epilogue warp of the pair
                const int64_t t = static_cast<int64_t>(chunk) * 8 + rank * 4 + (warp - 2);
                if (t < a.prev_T) combine_token_warp(a.prev_ystage, a.prev_gates, a.prev_out, t, a.k, a.d, lane);
                continue;
            }
            const Job jb = job_of(tile);
            const int m = jb.m0 + static_cast<int>(rank);
            const int64_t q = static_cast<int64_t>(m) * kBM + r;  // padded row of this thread
            const int64_t row_in_e = q - s_pad[jb.e];
            const bool valid = !jb.ghost && row_in_e < a.counts[jb.e];
            // FFN2: this row's token slot in ystage, looked up while the tile's MMAs run
            uint16_t *dst = nullptr;
            if (!jb.f1 && valid) {
                const int64_t p = a.offsets[jb.e] + row_in_e;
                dst = a.ystage + (static_cast<int64_t>(a.row_tok[p]) * a.k + a.row_j[p]) * a.d + jb.n * 256;
            }
            if (!wait_bar(acc_full, acc_phase, a.status, a.wait_ns, abort_flag)) break;
            tc_fence_after();
            bool released = false;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(acc_empty_even);
                released = true;
            };
            if (jb.f1) {
                epi_ffn1<MX>(trow, valid, q, jb.n * 128, a.F, a.h, a.h_scales, a.h_rows, a.saved_a, a.saved_b,
                             a.saved_h, stage_out + (warp - 2) * kStageWords, lane, release);
            } else {
                epi_rows_bf16(trow, 256, false, valid, dst, stage_out + (warp - 2) * kStageWords, lane, release);
            }
            if (!released) release();
            acc_phase ^= 1u;
            // an FFN1 tile publishes this warp's quarter of its h rows (a ghost half
            // has none); FFN2 tiles' ystage rows go to the combine kernel that follows
            if (jb.f1 && !jb.ghost) {
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    red_release_gpu_add(&h_done[m], 1);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no more remote arrives, stores, loads or multicast commits into either CTA
    if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }

}

template <bool MX>
constexpr size_t fused_pair_smem_bytes()
{
    return 1024 + kFPStages * kFPStage + (MX ? kFPStages * (kSfaBytes + kSfbBytes) : 0) +
           (4 * kFPStages + 2 + 2 * kTQ) * 8 + kTQ * 4 + 16 + 2 * (MOK_MAX_EXPERTS + 4) * 4 + kStageBytes;
}

// Launch configuration of the pair kernel: its attributes are set once and its
// grid is the number of CTA pairs that can be resident at once (the roles
// wait on one another, so every CTA must be resident), at most one per SM.
template <bool MX>
cudaError_t fused_pair_setup(int *grid_out)
{
    constexpr size_t smem = fused_pair_smem_bytes<MX>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int grid = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(k_moe_fused_pair<MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kFThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms() / 2 * 2));
        int clusters = 0;
        if (attr_err == cudaSuccess) attr_err = cudaOccupancyMaxActiveClusters(&clusters, k_moe_fused_pair<MX>, &cfg);
        grid = clusters * 2 <= num_sms() ? clusters * 2 : num_sms() / 2 * 2;
        if (attr_err == cudaSuccess && grid < 4) attr_err = cudaErrorInvalidConfiguration;
    });
    *grid_out = grid;
    return attr_err;
}

template <bool MX>
cudaError_t launch_fused_pair_t(const FusedMaps &pm, const FusedArgs &args, int grid, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = fused_pair_smem_bytes<MX>();
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_moe_fused_pair<MX>, pm, args);
}

template <bool MX>
constexpr size_t fused_smem_bytes()
{
    return 1024 + kStages * (kAStage + kBStage) + (MX ? kStages * (kSfaBytes + kSfbBytes) : 0) +
           (4 * kStages + 2 + 2 * kTQ) * 8 + kTQ * 4 + 16 + (MOK_MAX_EXPERTS + 4) * 4 + kStageBytes;
}

template <bool MX>
cudaError_t launch_fused_t(const FusedMaps &pm, const FusedArgs &args, cudaStream_t st)
{
    constexpr size_t smem = fused_smem_bytes<MX>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(k_moe_fused<MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
        int per_sm = 0;
        if (attr_err == cudaSuccess)
            attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_moe_fused<MX>, kFThreads, smem);
        if (attr_err == cudaSuccess && per_sm < 1) attr_err = cudaErrorInvalidConfiguration;
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms()));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_moe_fused<MX>, pm, args);
}

int gather_ctas(int sms, float frac)
{
    const int ng = static_cast<int>(frac * static_cast<float>(sms) + 0.5f);
    return ng < 1 ? 1 : (ng > sms - 1 ? sms - 1 : ng);
}

}  // namespace

// Shape-driven defaults of the fused forward's two knobs.  [kucoin] §03: when
// the hidden size, top-k or expert size changes, the right minibatch and the
// number of SMs on the communication side change with them; §02: one
// minibatch should give the expert GEMM at least two full waves of tiles.
//
// Gather CTAs: the GEMM role must never wait for rows in FFN1.  Per padded row
// the gather moves 2d bytes in and d (1 + 1/32) (MXFP8) or 2d (BF16) bytes
// out, at about kGatherBytesPerSm per second on one gathering SM (the pull
// dispatch measured on its own on GB300, all SMs pulling); FFN1 spends 4dF
// flops on the row at about kGemmFlopsPerSm per second on one GEMM SM (the
// fused forward measured on GB300).  n_gather / n_gemm must exceed the ratio
// of the two per-row times; the default takes twice that ratio, clamped to
// [1/16, 1/3] of the SMs (the gather CTAs join the GEMM role once the gather
// is done, so a generous share costs little).
int auto_gather_ctas(const Dims &dm, int sms)
{
    constexpr double kGatherBytesPerSm = 21e9;
    const double gemm_flops_per_sm = dm.dtype == MOK_MXFP8 ? 9.4e12 : 8.6e12;
    const double row_bytes = 2.0 * dm.d + (dm.dtype == MOK_MXFP8 ? dm.d * (1.0 + 1.0 / 32) : 2.0 * dm.d);
    const double t_gather = row_bytes / kGatherBytesPerSm;
    const double t_gemm = 4.0 * dm.d * static_cast<double>(dm.F) / gemm_flops_per_sm;
    const double q = 2.0 * t_gather / t_gemm;  // n_gather / n_gemm
    double frac = q / (1.0 + q);
    frac = frac < 1.0 / 16 ? 1.0 / 16 : (frac > 1.0 / 3 ? 1.0 / 3 : frac);
    return gather_ctas(sms, static_cast<float>(frac));
}

// Minibatch: [kucoin] wants one minibatch to give the expert GEMM two full
// waves of tiles.  Here every 128-row tile is released as soon as its rows
// have landed, and the gather CTAs each work on their own minibatch, so one
// round of the gather role hands over n_gather minibatches, worth
// n_gather * (mb / 128) * (F / 128) FFN1 tiles; the default is the smallest
// hand-off (64, 128 or 256 rows) for which a round covers two waves of the
// GEMM CTAs, else 256.  Smaller hand-offs let the first tiles start sooner.
int auto_minibatch_rows(const Dims &dm, int gather_ctas, int gemm_ctas)
{
    const int64_t tiles_per_row_tile = dm.F / 128;
    for (int mb = 64; mb < 256; mb *= 2)
        if (static_cast<int64_t>(gather_ctas) * mb * tiles_per_row_tile >= 2LL * 128 * gemm_ctas) return mb;
    return 256;
}

// CTA pairs need d a multiple of 256 (FFN2 pair tiles are 256 columns of d)
// and, when the token ring is capped, a ring of at least four row tiles.  A
// pair tile needs two row tiles that can straddle two gather units, and a
// gather unit may only overwrite ring rows once every FFN1 tile of their band
// has loaded them; with bands of B pair rows the wait is acyclic when
// 2B <= R - U + 1 (R ring row tiles, U <= 2 row tiles per unit), which
// B = R / 4 >= 1 satisfies for R >= 4.  Smaller rings run one CTA per tile.
// Default: pairs for BF16 layers; for MXFP8 layers pairs when the average
// expert holds at least 384 rows (three row tiles), one CTA per tile below.
// An expert with an odd number of row tiles ends in a pair tile with a ghost
// half, which still loads its half of B; the pair kernel (with its scale
// copies on their own thread) loads a third fewer bytes per SM-stage but
// completes a stage only when both SMs' loads have landed.  Measured on GB300,
// fused kernel, router routing: DeepSeek-V3 shape at 16384 tokens (512 rows
// per expert) 6.00 vs 6.08 ms, at 8192 tokens (256) 3.56 vs 3.47 ms, skewed
// layer with a capped ring 6.55 vs 6.59 ms; Mixtral shape 3.75 vs 3.81 ms.
// cfg->fused_cta_pairs = MOK_PAIRS_ON / OFF forces either.
bool fused_uses_pairs(const Dims &dm, const mok_config *cfg)
{
    if (dm.d % 256 != 0 || cfg->fused_cta_pairs == MOK_PAIRS_OFF) return false;
    if (cfg->fused_cta_pairs == MOK_PAIRS_AUTO && dm.dtype == MOK_MXFP8 && dm.S < 384LL * dm.E) return false;
    const int64_t ring_rows = fused_ring_rows(dm, cfg->ring_bytes);
    return ring_rows >= dm.rows_pad || ring_rows / 128 >= 4;
}

int fused_ctas(const Dims &dm, const mok_config *cfg, int sms)
{
    if (!fused_uses_pairs(dm, cfg)) return sms;
    int dev_count = 0, grid = 0;
    if (cudaGetDeviceCount(&dev_count) == cudaSuccess && dev_count > 0 &&
        (dm.dtype == MOK_MXFP8 ? fused_pair_setup<true>(&grid) : fused_pair_setup<false>(&grid)) == cudaSuccess)
        return grid;
    cudaGetLastError();  // no device here: clear the error, plan for every SM paired
    return sms / 2 * 2;
}

// ctas: the CTAs of the launch (for the pair kernel, its grid)
// A gather share of 1 (every token pulled first, by the dispatch kernel, then
// every CTA of the fused kernel runs the GEMM role) when the config asks for
// it, or automatically when the ring is uncapped and the split rule would give
// the gather role at least 1/8 of the CTAs: the split keeps that share away
// from the GEMM role for as long as it takes a fraction of the SMs to pull the
// rows (one read per slot); gathering first takes every SM for the time the
// whole GPU needs to pull them (one read per token).  Measured on GB300
// (DeepSeek-V3 MXFP8 shape, 38 of 152 CTAs by the split rule): 6.43 -> 6.09
// ms; Mixtral shape (10 of 152): 3.66 vs 3.68 ms, so the split stays there.
bool fused_gathers_first(const Dims &dm, const mok_config *cfg, int ctas)
{
    if (fused_ring_rows(dm, cfg->ring_bytes) < dm.rows_pad) return false;
    if (cfg->gather_sm_fraction >= 1.0f) return true;
    return cfg->gather_sm_fraction == 0.0f && 8 * auto_gather_ctas(dm, ctas) >= ctas;
}

void fused_knobs(const Dims &dm, const mok_config *cfg, int ctas, int *gather, int *mb)
{
    if (fused_gathers_first(dm, cfg, ctas)) {
        *gather = ctas;
        *mb = 0;
        return;
    }
    *gather = cfg->gather_sm_fraction > 0.0f ? gather_ctas(ctas, cfg->gather_sm_fraction)
                                             : auto_gather_ctas(dm, ctas);
    if (fused_uses_pairs(dm, cfg)) {
        // gather CTAs come in pairs; at least one pair stays in the GEMM role
        *gather = (*gather + 1) / 2 * 2;
        if (*gather > ctas - 2) *gather = ctas - 2;
        if (*gather < 2) *gather = 2;
    }
    *mb = cfg->minibatch_rows ? cfg->minibatch_rows : auto_minibatch_rows(dm, *gather, ctas - *gather);
}

int64_t fused_ring_rows(const Dims &dm, size_t ring_bytes)
{
    if (ring_bytes == 0) return dm.rows_pad;
    const int64_t row_bytes = dm.dtype == MOK_MXFP8 ? dm.d + dm.d / 32 : 2 * static_cast<int64_t>(dm.d);
    int64_t rows = static_cast<int64_t>(ring_bytes) / row_bytes / 256 * 256;
    return rows < dm.rows_pad ? rows : dm.rows_pad;
}

int fused_counter_ints(const Dims &dm) { return 3 + 3 * static_cast<int>(dm.rows_pad / 128); }

cudaError_t launch_fused(const Dims &dm, const mok_config *cfg, const Sources &src, const FusedIo &io,
                         const mok_weights *w, uint32_t *status, uint64_t wait_ns, cudaStream_t st)
{
    const bool mx = dm.dtype == MOK_MXFP8;
    const uint32_t box = mx ? 128 : 64;
    const int64_t ring_rows = fused_ring_rows(dm, cfg->ring_bytes);
    if (ring_rows < 256) return cudaErrorInvalidValue;
    const uint64_t EF = static_cast<uint64_t>(dm.E) * dm.F;
    const uint64_t Ed = static_cast<uint64_t>(dm.E) * dm.d;
    FusedMaps pm = {};
    if (encode_tmap_2d(&pm.ring, io.ring, mx, dm.d, ring_rows, box, kBM) ||
        encode_tmap_2d(&pm.ring64, io.ring, mx, dm.d, ring_rows, box, 64) ||
        encode_tmap_2d(&pm.g, mx ? static_cast<const void *>(w->q_gate) : w->w_gate, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&pm.u, mx ? static_cast<const void *>(w->q_up) : w->w_up, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&pm.h, io.h, mx, dm.F, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&pm.h64, io.h, mx, dm.F, dm.rows_pad, box, 64) ||
        encode_tmap_2d(&pm.dn, mx ? static_cast<const void *>(w->q_down) : w->w_down, mx, dm.F, Ed, box, 128))
        return cudaErrorInvalidValue;
    FusedArgs a = {};
    a.E = dm.E;
    a.T = dm.T;
    a.k = dm.k;
    a.d = dm.d;
    a.F = dm.F;
    a.ids = io.ids;
    a.counts = io.counts;
    a.offsets = io.offsets;
    a.pad_offsets = io.pad_offsets;
    a.slot_pos = io.slot_pos;
    a.row_tok = io.row_tok;
    a.row_j = io.row_j;
    a.gates = io.gates;
    a.src = src;
    a.ring = static_cast<uint8_t *>(io.ring);
    a.ring_scales = io.ring_scales;
    a.ring_rows = ring_rows;
    a.h = io.h;
    a.h_scales = io.h_scales;
    a.h_rows = dm.rows_pad;
    a.s_gate = w->s_gate;
    a.s_up = w->s_up;
    a.s_down = w->s_down;
    a.EF = static_cast<int64_t>(EF);
    a.Ed = static_cast<int64_t>(Ed);
    a.ystage = io.ystage;
    a.out = io.out;
    a.saved_a = io.saved_a;
    a.saved_b = io.saved_b;
    a.saved_h = io.saved_h;
    const bool pair = fused_uses_pairs(dm, cfg);
    int grid = num_sms();
    if (pair) {
        const cudaError_t ge = mx ? fused_pair_setup<true>(&grid) : fused_pair_setup<false>(&grid);
        if (ge != cudaSuccess) return ge;
    }
    fused_knobs(dm, cfg, grid, &a.n_gather, &a.mb);
    a.prologue = a.n_gather >= grid ? 1 : 0;
    if (a.prologue && ring_rows < dm.rows_pad) return cudaErrorInvalidValue;
    a.NT1 = dm.F / 128;
    a.BN2 = dm.d % 256 == 0 ? 256 : 128;
    a.NT2 = dm.d / a.BN2;
    a.k1 = dm.d / static_cast<int>(box);
    a.k2 = dm.F / static_cast<int>(box);
    // an uncapped ring never wraps: one band per expert (the separate-kernel
    // order); a capped ring holds two bands, so a band is always free to fill
    // (CTA pairs: bands of ring/4 pair rows, see fused_uses_pairs)
    a.band1 = ring_rows >= dm.rows_pad ? (1 << 30)
                                       : static_cast<int>(pair ? ring_rows / 128 / 4 * 2 : ring_rows / 128 / 2);
    a.counters = io.counters;
    a.max_mt = static_cast<int>(dm.rows_pad / 128);
    a.prev_ystage = io.prev_ystage;
    a.prev_gates = io.prev_gates;
    a.prev_out = io.prev_out;
    a.prev_T = io.prev_T;
    // one token per epilogue warp: four per chunk on one CTA, eight on a pair
    a.prev_chunks = io.prev_T > 0 ? (io.prev_T + (pair ? 8 : 4) - 1) / (pair ? 8 : 4) : 0;
    a.status = status;
    a.wait_ns = wait_ns;
    if (pair) {
        if (mx && (encode_tmap_scales(&pm.s_ring, io.ring_scales, static_cast<uint64_t>(ring_rows), dm.d) ||
                   encode_tmap_scales(&pm.s_g, w->s_gate, EF, dm.d) ||
                   encode_tmap_scales(&pm.s_u, w->s_up, EF, dm.d) ||
                   encode_tmap_scales(&pm.s_h, io.h_scales, dm.rows_pad, dm.F) ||
                   encode_tmap_scales(&pm.s_dn, w->s_down, Ed, dm.F)))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaMemsetAsync(io.counters, 0, sizeof(int) * fused_counter_ints(dm), st);
    if (e != cudaSuccess) return e;
    if (a.prologue) {
        // gather first: every token's row read once, quantised once, placed into
        // its k rows of the (uncapped) ring, by the dispatch kernel
        e = launch_dispatch_by_token(dm, src, io.ids, io.slot_pos, io.offsets, io.pad_offsets, io.ring,
                                     io.ring_scales, st);
        if (e != cudaSuccess) return e;
    }
    e = pair ? (mx ? launch_fused_pair_t<true>(pm, a, grid, st) : launch_fused_pair_t<false>(pm, a, grid, st))
             : (mx ? launch_fused_t<true>(pm, a, st) : launch_fused_t<false>(pm, a, st));
    if (e != cudaSuccess || io.skip_combine) return e;
    // the weighted combine of this call's tokens, by the separate combine kernel
    return launch_combine(dm, io.ystage, io.gates, io.out, st);
}

}  // namespace mok
