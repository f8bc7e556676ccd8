// mok_gemm.cu -- tcgen05 grouped GEMMs of the MoE layer on sm_103a.
//
// [kucoin] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72" (kucoin.com flash, Arabic).  §01: the grouped GEMM needs each
// expert's tokens organised together before it can feed the tensor cores,
// and backward runs the exchange again in reverse; §02: MXFP8 activation
// quantisation is fused into the grouped GEMM and SwiGLU, and combine is a
// push -- each result goes straight to the token it came from.
//
// One persistent kernel template, one CTA per SM, 6 warps:
//   warp 0      TMA producer: A tile (128 rows) and B tile (128 or 256 rows)
//               of 128 bytes along K per stage, plus MX scale tiles (bulk
//               copies), into a 4-stage shared-memory ring (mbarrier
//               full/empty pairs);
//   warp 1      allocates TMEM and issues tcgen05.mma from one thread into a
//               128 x N fp32 accumulator (N = 256 or 128);
//   warps 2..5  epilogue: each thread owns one accumulator row (its TMEM
//               lane) and runs the mode's epilogue straight from registers.
// Modes (C = A B^T, both operands K-major):
//   ROUTER  x . [W_hi | W_mid | W_lo]^T over the token rows of each source
//           buffer (A's K wraps three times); fp32 logits (+ bias);
//   FFN1    per expert, B = 128 rows of W_g and the same 128 rows of W_u, so
//           one tile holds a and b for 128 columns of F: h = silu(a) b, stored
//           BF16 or MXFP8 (blocks of 32 along F, quantised in registers);
//   FFN2    per expert, y = h W_d^T stored BF16 into ystage[token, j];
//   DGRAD2  per expert, dh = dy W_d (B = W_d^T rows); SwiGLU backward with the
//           saved a, b in the epilogue -> da, db (BF16, and MXFP8 along F);
//   DGRAD1  per expert, dx = da W_g + db W_u as one K = 2F loop over
//           (da, W_g^T) then (db, W_u^T); BF16 rows;
//   WGRAD   per expert, dW = A^T B over the expert's token rows: A and B are
//           the transposed operands [X, rows] whose K range is the expert's
//           padded row segment; BF16 out, zeros for an expert without rows.
// Tiles are ordered group by group, N-tile by N-tile, with the group's row
// tiles innermost, and dealt round-robin to the CTAs: concurrently running
// CTAs share B tiles and the group's rows through L2.
#include <cuda_bf16.h>

#include <mutex>

#include "mok_internal.h"
#include "mok_ptx.cuh"
#include "mok_tc.cuh"

namespace mok {

namespace {

#ifndef MOK_GEMM_CLUSTER
#define MOK_GEMM_CLUSTER 1
#endif
constexpr int kCluster = MOK_GEMM_CLUSTER;  // CTAs per cluster of the GEMM launch
enum { MODE_ROUTER = 0, MODE_FFN1, MODE_FFN2, MODE_DGRAD2, MODE_DGRAD1, MODE_WGRAD };
// Epilogue staging: four warps of 32 rows x 33 words, or DGRAD2's eight warps
// of 32 rows x 17 words (64-byte row segments)
constexpr int kD2StageWords = 32 * 17;
constexpr size_t kGemmStageBytes =
    kStageBytes > 8 * kD2StageWords * 4 ? kStageBytes : static_cast<size_t>(8 * kD2StageWords * 4);

template <int NA>
struct AMaps {
    CUtensorMap m[NA];
    int mt_start[NA + 1];   // router: first row tile of each source
    int row_start[NA + 1];  // router: first token of each source
    int rows[NA];           // router: rows of each source
    int n;
};

struct GemmArgs {
    int E;                  // groups (experts); router: sources
    const int32_t *counts;
    const int32_t *offsets;
    const int32_t *pad_offsets;
    int n_tiles;            // N tiles per group
    int BN;                 // MMA N: 128 or 256
    int k_stages;           // K / (128 bytes) (not WGRAD)
    int a_k_stages;         // router: K stages of A before it wraps
    int ks_half;            // DGRAD1: K stages of each of the two segments
    int b_rows_per_group;   // rows of B per expert
    int m_rows;             // WGRAD: output rows per expert (multiple of 128)
    // MX scales (tile layout) of A maps 0/1 and B maps 0/1
    const uint32_t *sfa[2];
    int64_t sfa_rows[2];
    const uint32_t *sfb[2];
    int64_t sfb_rows[2];
    // epilogue
    int F, d, k_top, T;
    float *logits;
    const float *bias;
    int E_valid;
    void *h;
    uint32_t *h_scales;
    int64_t h_rows;
    uint16_t *saved_a, *saved_b, *saved_h;
    uint16_t *ystage;
    const int32_t *row_tok;
    const uint8_t *row_j;
    // backward
    const uint16_t *in_a, *in_b;     // DGRAD2: saved a, b
    uint16_t *out_da, *out_db;       // DGRAD2: BF16 da, db
    uint8_t *q_da, *q_db;            // DGRAD2 (MX): codes of da, db along F
    uint32_t *s_da, *s_db;           // DGRAD2 (MX): their scales
    uint16_t *out_rows;              // DGRAD1: dx rows; WGRAD: dW [E * m_rows, N]
    int64_t out_ld;                  // WGRAD: columns of dW
    uint32_t *status;
    uint64_t wait_ns;
};

struct Tile {
    int group, m_blk, n_blk;
};

__device__ __forceinline__ Tile decode_tile(int tile, const int *prefix, int E, int n_tiles)
{
    int lo = 0, hi = E;  // last group with prefix[g] <= tile
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile) lo = mid;
        else hi = mid;
    }
    const int mt = (prefix[lo + 1] - prefix[lo]) / n_tiles;
    const int local = tile - prefix[lo];
    Tile t;
    t.group = lo;
    t.n_blk = local / mt;
    t.m_blk = local % mt;
    return t;
}

template <int MODE>
__device__ __forceinline__ int group_row_tiles(const AMaps<MODE == MODE_ROUTER ? 64 : 2> &am,
                                               const GemmArgs &a, int g)
{
    if constexpr (MODE == MODE_ROUTER) return am.mt_start[g + 1] - am.mt_start[g];
    else if constexpr (MODE == MODE_WGRAD) return a.m_rows / kBM;
    else return (a.pad_offsets[g + 1] - a.pad_offsets[g]) / kBM;
}

template <int MODE, bool MX>
__device__ __forceinline__ int tile_k_stages(const GemmArgs &a, int g)
{
    if constexpr (MODE == MODE_WGRAD)
        return (a.pad_offsets[g + 1] - a.pad_offsets[g]) / (MX ? 128 : 64);
    else return a.k_stages;
}

// Epilogue warps of the single-CTA GEMM per mode: the data-gradient SwiGLU
// backward (DGRAD2) is long arithmetic per accumulator column with the MMA
// waiting for it, so it runs on two warps per TMEM lane quarter (128 columns
// each); the other modes on one.
template <int MODE>
struct GemmShape {
    static constexpr int kEpiWarps = MODE == MODE_DGRAD2 ? 8 : 4;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
};

template <int MODE, bool MX>
__global__ void __launch_bounds__(GemmShape<MODE>::kThreads, 1)
    k_gemm(const __grid_constant__ AMaps<MODE == MODE_ROUTER ? 64 : 2> am,
           const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
           const GemmArgs a)
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
    uint64_t *acc_full = bars + 2 * kStages;
    uint64_t *acc_empty = acc_full + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(acc_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *prefix = reinterpret_cast<int *>(tmem_holder + 4);  // [groups + 1]
    uint32_t *stage_out = reinterpret_cast<uint32_t *>(prefix + MOK_MAX_EXPERTS + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int groups = MODE == MODE_ROUTER ? am.n : a.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, GemmShape<MODE>::kEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        const int na = MODE == MODE_ROUTER ? am.n : (MODE == MODE_DGRAD1 ? 2 : 1);
        for (int i = 0; i < na; ++i) prefetch_tmap(&am.m[i]);
        prefetch_tmap(&tmB0);
        prefetch_tmap(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2) {
        // exclusive prefix over groups of (row tiles x N tiles)
        const int per = (groups + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int g = g0; g < g0 + per && g < groups; ++g)
            local += group_row_tiles<MODE>(am, a, g) * a.n_tiles;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int g = g0; g < g0 + per && g < groups; ++g) {
            prefix[g] = run;
            run += group_row_tiles<MODE>(am, a, g) * a.n_tiles;
        }
        if (lane == 31) prefix[groups] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = prefix[groups];
    const int BN = a.BN;
    constexpr int kE = MX ? 128 : 64;  // elements per 128-byte K stage

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t stage = 0, phase = 0;
            const uint32_t stage_bytes = kAStage + (BN / 128) * 16384 +
                                         (MX ? kSfaBytes + (BN / 128) * 512 : 0);
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                const Tile tl = decode_tile(tile, prefix, groups, a.n_tiles);
                const int g = tl.group;
                const int kst = tile_k_stages<MODE, MX>(a, g);
                for (int ks = 0; ks < kst; ++ks) {
                    // coordinates of this stage: A map / (x, y), B maps / (x, y0, y1)
                    int ai = 0, xa, ya, bi0 = 0, bi1 = 0, xb, yb0, yb1;
                    if constexpr (MODE == MODE_ROUTER) {
                        ai = g;
                        xa = (ks % a.a_k_stages) * kE;
                        ya = tl.m_blk * kBM;
                        xb = ks * kE;
                        yb0 = tl.n_blk * BN;
                        yb1 = yb0 + 128;
                    } else if constexpr (MODE == MODE_FFN1) {
                        xa = ks * kE;
                        ya = a.pad_offsets[g] + tl.m_blk * kBM;
                        xb = ks * kE;
                        yb0 = g * a.b_rows_per_group + tl.n_blk * 128;
                        yb1 = yb0;
                        bi1 = 1;
                    } else if constexpr (MODE == MODE_DGRAD1) {
                        const int seg = ks >= a.ks_half;
                        const int kk = ks - seg * a.ks_half;
                        ai = bi0 = bi1 = seg;
                        xa = kk * kE;
                        ya = a.pad_offsets[g] + tl.m_blk * kBM;
                        xb = kk * kE;
                        yb0 = g * a.b_rows_per_group + tl.n_blk * BN;
                        yb1 = yb0 + 128;
                    } else if constexpr (MODE == MODE_WGRAD) {
                        xa = a.pad_offsets[g] + ks * kE;
                        ya = tl.m_blk * kBM;
                        xb = xa;
                        yb0 = tl.n_blk * BN;
                        yb1 = yb0 + 128;
                    } else {  // FFN2, DGRAD2
                        xa = ks * kE;
                        ya = a.pad_offsets[g] + tl.m_blk * kBM;
                        xb = ks * kE;
                        yb0 = g * a.b_rows_per_group + tl.n_blk * BN;
                        yb1 = yb0 + 128;
                    }
                    if (!wait_bar(&empty[stage], phase ^ 1u, a.status, a.wait_ns, abort_flag)) goto producer_done;
                    uint8_t *dA = sA + stage * kAStage;
                    uint8_t *dB = sB + stage * kBStage;
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    tma_load_2d(dA, &am.m[ai], &full[stage], xa, ya);
                    tma_load_2d(dB, bi0 ? &tmB1 : &tmB0, &full[stage], xb, yb0);
                    if (BN == 256) tma_load_2d(dB + 16384, bi1 ? &tmB1 : &tmB0, &full[stage], xb, yb1);
                    if constexpr (MX) {
                        uint8_t *dS = sSF + stage * (kSfaBytes + kSfbBytes);
                        bulk_load(dS, a.sfa[ai] + scale_word(xa, ya, a.sfa_rows[ai]), kSfaBytes, &full[stage]);
                        bulk_load(dS + kSfaBytes, a.sfb[bi0] + scale_word(xb, yb0, a.sfb_rows[bi0]), 512,
                                  &full[stage]);
                        if (BN == 256)
                            bulk_load(dS + kSfaBytes + 512,
                                      a.sfb[bi1] + scale_word(xb, yb1, a.sfb_rows[bi1]), 512, &full[stage]);
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
            // ------------------------------------------------ MMA issuer
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            // MXFP8: the scale-factor byte selectors (bits 4-5 and 29-30) are or-ed in per MMA
            const uint32_t idesc = MX ? idesc_mxf8(kBM, BN, 0, 0) : idesc_bf16(kBM, BN);
            const uint64_t adesc0 = sdesc_k_sw128(smem_u32(sA));
            const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(sB));
            const uint64_t sfdesc0 = sdesc_sf(smem_u32(sSF));
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                const Tile tl = decode_tile(tile, prefix, groups, a.n_tiles);
                const int kst = tile_k_stages<MODE, MX>(a, tl.group);
                if (!wait_bar(acc_empty, acc_phase ^ 1u, a.status, a.wait_ns, abort_flag)) break;
                tc_fence_after();
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&full[stage], phase, a.status, a.wait_ns, abort_flag)) goto mma_done;
                    tc_fence_after();
                    // descriptors: the stage's base plus 32 bytes of K per MMA (address >> 4
                    // in the low bits; every shared address here is below 256 KB, so no carry)
                    const uint64_t ad0 = adesc0 + static_cast<uint64_t>((stage * kAStage) >> 4);
                    const uint64_t bd0 = bdesc0 + static_cast<uint64_t>((stage * kBStage) >> 4);
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
                    if (MX) {
                        const uint64_t sd = sfdesc0 + static_cast<uint64_t>((stage * (kSfaBytes + kSfbBytes)) >> 4);
                        tmem_cp_32x128b_warpx4(sfa_col, sd);
                        tmem_cp_32x128b_warpx4(sfb_col, sd + (kSfaBytes >> 4));
                        if (BN == 256) tmem_cp_32x128b_warpx4(sfb_col + 4, sd + ((kSfaBytes + 512) >> 4));
                    }
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
    } else {
        // ---------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile tl = decode_tile(tile, prefix, groups, a.n_tiles);
            // What this thread's row needs from global memory is looked up while
            // the tile's MMAs run, not after the accumulator is full: the expert's
            // counts and offsets, FFN2's token slot, DGRAD2's first 32 columns of
            // the saved a, b.  (Prefetching the rest of the row into L2 here read
            // it from DRAM twice -- the K loop's weights evict it before the
            // epilogue -- and bought no time.)
            const int e = tl.group;
            const int row_in_e = tl.m_blk * kBM + r;
            bool valid = true;
            int64_t grow = 0;
            uint16_t *dst = nullptr;
            bool empty_k = false;
            uint4 na[4], nb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) na[q] = nb[q] = make_uint4(0, 0, 0, 0);
            int c_begin = 0, c_end = 0, f0 = 0;
            if constexpr (MODE == MODE_FFN1 || MODE == MODE_FFN2 || MODE == MODE_DGRAD2 || MODE == MODE_DGRAD1) {
                valid = row_in_e < a.counts[e];
                grow = a.pad_offsets[e] + row_in_e;
            }
            if constexpr (MODE == MODE_FFN2) {
                if (valid) {
                    const int64_t p = a.offsets[e] + row_in_e;
                    const int64_t t = a.row_tok[p];
                    const int64_t j = a.row_j[p];
                    dst = a.ystage + (t * a.k_top + j) * a.d + tl.n_blk * BN;
                }
            } else if constexpr (MODE == MODE_DGRAD1) {
                dst = a.out_rows + grow * a.d + tl.n_blk * BN;
            } else if constexpr (MODE == MODE_WGRAD) {
                empty_k = a.pad_offsets[e + 1] == a.pad_offsets[e];
                dst = a.out_rows + (static_cast<int64_t>(e) * a.m_rows + tl.m_blk * kBM + r) * a.out_ld +
                      tl.n_blk * BN;
            } else if constexpr (MODE == MODE_DGRAD2) {
                // warps 2-5 take accumulator columns [0, 128), warps 6-9 [128, 256)
                // (nothing when BN = 128): whole 128-column MX scale groups each
                c_begin = ((warp - 2) >> 2) * 128;
                c_end = min(BN, c_begin + 128);
                f0 = tl.n_blk * BN + c_begin;
                if (valid && c_begin < c_end) {
                    const uint4 *pa = reinterpret_cast<const uint4 *>(a.in_a + grow * a.F + f0);
                    const uint4 *pb = reinterpret_cast<const uint4 *>(a.in_b + grow * a.F + f0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        na[q] = __ldg(pa + q);
                        nb[q] = __ldg(pb + q);
                    }
                }
            }
            if (!wait_bar(acc_full, acc_phase, a.status, a.wait_ns, abort_flag)) break;
            tc_fence_after();
            // Hands the accumulator back to the MMA warp; epilogues that first
            // drain their row into registers call it before their global stores,
            // so the stores overlap the next tile's main loop.
            bool released = false;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_relaxed(acc_empty);
                released = true;
            };
            if constexpr (MODE == MODE_ROUTER) {
                const int lrow = tl.m_blk * kBM + r;
                const bool valid = lrow < am.rows[tl.group];
                const int64_t tok = am.row_start[tl.group] + lrow;
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32(trow + c, v);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int col = tl.n_blk * BN + c + i;
                            if (col < a.E_valid)
                                a.logits[tok * a.E_valid + col] =
                                    __uint_as_float(v[i]) + (a.bias ? a.bias[col] : 0.0f);
                        }
                    }
                }
            } else if constexpr (MODE == MODE_FFN1) {
                epi_ffn1<MX>(trow, valid, grow, tl.n_blk * 128, a.F, a.h, a.h_scales, a.h_rows, a.saved_a,
                             a.saved_b, a.saved_h, stage_out + (warp - 2) * kStageWords, lane, release);
            } else if constexpr (MODE == MODE_FFN2) {
                epi_rows_bf16(trow, BN, false, valid, dst, stage_out + (warp - 2) * kStageWords, lane,
                              release);
            } else if constexpr (MODE == MODE_DGRAD2) {
                // dh -> SwiGLU backward with the saved (BF16) a, b:
                //   s = sigmoid(a), da = dh b s (1 + a (1 - s)), db = dh a s
                // (the first 32 columns of a, b are in na / nb; each chunk loads the
                // next one's while it is processed)
                // Every lane computes (rows past the expert's count on zeros) and
                // takes part in the staged stores, which write whole row segments;
                // only valid rows are stored.
                uint32_t wa = 0, wb = 0;
                uint32_t *stg = stage_out + (warp - 2) * kD2StageWords;
                for (int c = 0; c < c_end - c_begin; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32(trow + c_begin + c, v);
                    tmem_ld_wait();
                    const int64_t off = grow * a.F + f0 + c;
                    float av[32], bv[32], da[32], db[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t ua[4] = {na[q].x, na[q].y, na[q].z, na[q].w};
                        const uint32_t ub[4] = {nb[q].x, nb[q].y, nb[q].z, nb[q].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            av[8 * q + 2 * i] = bf16_bits_to_float(ua[i] & 0xFFFFu);
                            av[8 * q + 2 * i + 1] = bf16_bits_to_float(ua[i] >> 16);
                            bv[8 * q + 2 * i] = bf16_bits_to_float(ub[i] & 0xFFFFu);
                            bv[8 * q + 2 * i + 1] = bf16_bits_to_float(ub[i] >> 16);
                        }
                    }
                    if (valid && c + 32 < c_end - c_begin) {
                        const uint4 *pa = reinterpret_cast<const uint4 *>(a.in_a + off + 32);
                        const uint4 *pb = reinterpret_cast<const uint4 *>(a.in_b + off + 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            na[q] = __ldg(pa + q);
                            nb[q] = __ldg(pb + q);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float dh = __uint_as_float(v[i]);
                        const float s = 1.0f / (1.0f + __expf(-av[i]));
                        da[i] = dh * bv[i] * s * (1.0f + av[i] * (1.0f - s));
                        db[i] = dh * av[i] * s;
                    }
                    uint32_t pk[16];
                    pack_bf16x32(da, pk);
                    store_rows_staged_n<16>(pk, valid ? a.out_da + off : nullptr, stg, lane);
                    pack_bf16x32(db, pk);
                    store_rows_staged_n<16>(pk, valid ? a.out_db + off : nullptr, stg, lane);
                    if constexpr (MX) {
                        // quantise the BF16-rounded values (the stored da, db)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            da[i] = bf16_bits_to_float(float_to_bf16_bits(da[i]));
                            db[i] = bf16_bits_to_float(float_to_bf16_bits(db[i]));
                        }
                        const int sh = 8 * ((c >> 5) & 3);
                        uint32_t qc[8];
                        wa |= mx_block32(da, qc) << sh;
                        store_rows_staged_n<8>(qc, valid ? a.q_da + off : nullptr, stg, lane);
                        wb |= mx_block32(db, qc) << sh;
                        store_rows_staged_n<8>(qc, valid ? a.q_db + off : nullptr, stg, lane);
                        if ((c & 127) == 96) {
                            if (valid) {
                                const int64_t wi = scale_word_row((f0 + c) >> 7, grow, a.h_rows);
                                a.s_da[wi] = wa;
                                a.s_db[wi] = wb;
                            }
                            wa = wb = 0;
                        }
                    }
                }
            } else if constexpr (MODE == MODE_DGRAD1) {
                epi_rows_bf16(trow, BN, false, valid, dst, stage_out + (warp - 2) * kStageWords, lane,
                              release);
            } else {  // MODE_WGRAD
                epi_rows_bf16(trow, BN, empty_k, true, dst, stage_out + (warp - 2) * kStageWords, lane,
                              release);
            }
            if (!released) release();
            acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // let copies and MMAs already in flight land before the CTA exits
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant of FFN1 / FFN2 (cta_group::2): clusters of two CTAs compute
// a 256 x 256 tile -- each CTA loads its own 128 rows of A and one half of B
// (FFN1: CTA 0 the 128 W_g rows, CTA 1 the 128 W_u rows; FFN2: 128 rows of
// W_d each) into 32 KB stages, six stages deep, plus (MXFP8) its A rows'
// scale tile and the scale tiles of all 256 B rows.  Every load of both CTAs
// is a tensor-map copy whose completion is counted on the even CTA's "full"
// barrier, which the even CTA arms for the bytes of both; the even CTA issues
// the MMAs and scale copies for the pair; the MMA commits release the stage
// and publish the accumulator in both CTAs (multicast); both CTAs' epilogue
// warps hand the accumulator back to the even CTA.  Every CTA of a pair walks
// the same tile sequence; an odd last row tile of an expert is computed and
// discarded (its A rows and scales beyond the matrix read as zeros).
// ---------------------------------------------------------------------------
constexpr int kPStage = kAStage + 128 * kBKBytes;  // 32 KB

// Shape of the pair kernel per mode.  WGRAD tiles have a K of only the
// expert's token rows (~2-3 stages) and a 64 KB output per CTA, so they are
// paced by the epilogue: 8 epilogue warps (two per TMEM lane quarter, 128
// columns each) and 4 stages; the other modes run 4 epilogue warps and 6 stages.
template <int MODE>
struct PairShape {
    static constexpr int kEpiWarps = MODE == MODE_WGRAD ? 8 : 4;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kStages = MODE == MODE_WGRAD ? 5 : 6;
};

struct PairMaps {
    CUtensorMap a, b0, b1;     // A rows; B rows (FFN1: W_g, W_u; FFN2: W_d twice)
    CUtensorMap sa, sb0, sb1;  // scale tiles of A and of B (MXFP8 only)
    CUtensorMap out;           // WGRAD: dW [E * m_rows, N] BF16, 32-row x 64-column boxes
};

// WGRAD epilogue: every epilogue warp owns 32 dW rows x (256 / (warps / 4))
// columns per tile, stored 64 columns at a time through one shared-memory box
// of 32 x 64 BF16 (4 KB, 128-byte swizzled) by TMA.  Box bytes per warp:
template <int MODE>
constexpr int pair_box_bytes()
{
    return MODE == MODE_WGRAD ? 4096 : 0;
}

// index of the scale tile of (k element x, row y) in a [rows, K] matrix
__device__ __forceinline__ int sf_tile(int x, int y, int64_t rows)
{
    return static_cast<int>((x >> 7) * (rows >> 7) + (y >> 7));
}

template <int MODE, bool MX>
__global__ void __launch_bounds__(PairShape<MODE>::kThreads, 1)
    k_gemm_pair(const __grid_constant__ PairMaps pm, const GemmArgs a)
{
    constexpr int kPStages = PairShape<MODE>::kStages;
    constexpr int kEpiWarps = PairShape<MODE>::kEpiWarps;
    static_assert(MODE == MODE_FFN1 || MODE == MODE_FFN2 || MODE == MODE_WGRAD, "pair path: FFN1, FFN2, WGRAD");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sT = smem;  // stage s: A at s*32K, B half at s*32K + 16K
    uint8_t *sOut = sT + kPStages * kPStage;  // WGRAD output boxes (1024-byte aligned)
    uint8_t *sSF = sOut + kEpiWarps * pair_box_bytes<MODE>();
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSF + (MX ? kPStages * (kSfaBytes + kSfbBytes) : 0));
    uint64_t *full = bars;
    uint64_t *empty = bars + kPStages;
    uint64_t *acc_full = bars + 2 * kPStages;
    uint64_t *acc_empty = acc_full + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(acc_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *prefix = reinterpret_cast<int *>(tmem_holder + 4);
    uint32_t *stage_out = reinterpret_cast<uint32_t *>(prefix + MOK_MAX_EXPERTS + 4);  // FFN epilogues
    int *s_pad = prefix + MOK_MAX_EXPERTS + 4;  // WGRAD: the experts' K ranges (pad_offsets)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int groups = a.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&pm.a);
        prefetch_tmap(&pm.b0);
        prefetch_tmap(&pm.b1);
        if (MX) {
            prefetch_tmap(&pm.sa);
            prefetch_tmap(&pm.sb0);
            prefetch_tmap(&pm.sb1);
        }
    }
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or load
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 2) {
        const int per = (groups + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        // WGRAD: a fixed (X / 256) x (Y / 256) tiles per expert; FFN: pair rows x N tiles
        auto pair_tiles = [&](int g) {
            if constexpr (MODE == MODE_WGRAD) return a.m_rows / (2 * kBM) * a.n_tiles;
            else return ((a.pad_offsets[g + 1] - a.pad_offsets[g]) / kBM + 1) / 2 * a.n_tiles;
        };
        for (int g = g0; g < g0 + per && g < groups; ++g) local += pair_tiles(g);
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int g = g0; g < g0 + per && g < groups; ++g) {
            prefix[g] = run;
            run += pair_tiles(g);
        }
        if (lane == 31) prefix[groups] = incl;
        if constexpr (MODE == MODE_WGRAD)
            for (int g = lane; g <= groups; g += 32) s_pad[g] = a.pad_offsets[g];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = prefix[groups];
    constexpr int kE = MX ? 128 : 64;
    // bytes one CTA lands per stage; the even CTA's barrier counts both CTAs'
    const uint32_t cta_bytes = kPStage + (MX ? kSfaBytes + kSfbBytes : 0);
    // Tile and K stages of a tile index.  WGRAD: every expert has the same
    // (X / 256) x (Y / 256) tiles, so the expert is one division away and its K
    // range sits in shared memory (a few stages per tile leave no room for a
    // global load on the issue path).
    const int wmt = MODE == MODE_WGRAD ? a.m_rows / (2 * kBM) : 1;
    const int wper = wmt * a.n_tiles;
    auto locate = [&](int tile) {
        Tile t;
        if constexpr (MODE == MODE_WGRAD) {
            t.group = tile / wper;
            const int local = tile - t.group * wper;
            t.m_blk = local / a.n_tiles;
            t.n_blk = local - t.m_blk * a.n_tiles;
        } else {
            t = decode_tile(tile, prefix, groups, a.n_tiles);
        }
        return t;
    };
    auto k_stages_of = [&](int g) {
        if constexpr (MODE == MODE_WGRAD) return (s_pad[g + 1] - s_pad[g]) / kE;
        else return a.k_stages;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- TMA producer (both CTAs)
            uint32_t stage = 0, phase = 0;
            const uint32_t full0 = mapa_shared(smem_u32(full), 0);
            for (int tile = pair; tile < total; tile += npairs) {
                const Tile tl = locate(tile);
                const int g = tl.group;
                const int kst = k_stages_of(g);
                // WGRAD: A rows over X, B rows over Y, K along the expert's token rows
                const int x0 = MODE == MODE_WGRAD ? s_pad[g] : 0;
                const int ya = MODE == MODE_WGRAD ? (2 * tl.m_blk + static_cast<int>(rank)) * kBM
                                                  : a.pad_offsets[g] + (2 * tl.m_blk + static_cast<int>(rank)) * kBM;
                int yb, ysf;
                const CUtensorMap *bmap;
                if constexpr (MODE == MODE_WGRAD) {
                    ysf = tl.n_blk * 256;
                    yb = ysf + static_cast<int>(rank) * 128;
                    bmap = &pm.b0;
                } else if constexpr (MODE == MODE_FFN1) {
                    yb = g * a.b_rows_per_group + tl.n_blk * 128;
                    ysf = yb;
                    bmap = rank ? &pm.b1 : &pm.b0;
                } else {
                    ysf = g * a.b_rows_per_group + tl.n_blk * 256;
                    yb = ysf + static_cast<int>(rank) * 128;
                    bmap = &pm.b0;
                }
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&empty[stage], phase ^ 1u, a.status, a.wait_ns, abort_flag)) goto producer_done;
                    uint8_t *dA = sT + stage * kPStage;
                    const int x = x0 + ks * kE;
                    const uint32_t fb = full0 + stage * 8;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * cta_bytes);
                    tma_load_2d_pair(dA, &pm.a, fb, x, ya);
                    tma_load_2d_pair(dA + kAStage, bmap, fb, x, yb);
                    if constexpr (MX) {
                        uint8_t *dS = sSF + stage * (kSfaBytes + kSfbBytes);
                        tma_load_2d_pair(dS, &pm.sa, fb, 0, sf_tile(x, ya, a.sfa_rows[0]));
                        if constexpr (MODE == MODE_FFN1) {
                            tma_load_2d_pair(dS + kSfaBytes, &pm.sb0, fb, 0, sf_tile(x, ysf, a.sfb_rows[0]));
                            tma_load_2d_pair(dS + kSfaBytes + 512, &pm.sb1, fb, 0, sf_tile(x, ysf, a.sfb_rows[1]));
                        } else {
                            tma_load_2d_pair(dS + kSfaBytes, &pm.sb0, fb, 0, sf_tile(x, ysf, a.sfb_rows[0]));
                            tma_load_2d_pair(dS + kSfaBytes + 512, &pm.sb0, fb, 0,
                                             sf_tile(x, ysf + 128, a.sfb_rows[0]));
                        }
                    }
                    if (++stage == kPStages) {
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
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            const uint32_t idesc = MX ? idesc_mxf8(2 * kBM, 256, 0, 0) : idesc_bf16(2 * kBM, 256);
            const uint64_t tdesc0 = sdesc_k_sw128(smem_u32(sT));
            const uint64_t sfdesc0 = sdesc_sf(smem_u32(sSF));
            for (int tile = pair; tile < total; tile += npairs) {
                const int kst = k_stages_of(locate(tile).group);
                if (!wait_bar(acc_empty, acc_phase ^ 1u, a.status, a.wait_ns, abort_flag)) break;
                tc_fence_after();
                for (int ks = 0; ks < kst; ++ks) {
                    if (!wait_bar(&full[stage], phase, a.status, a.wait_ns, abort_flag)) goto mma_done;
                    tc_fence_after();
                    // descriptors: the stage's base plus 32 bytes of K per MMA (see k_gemm)
                    const uint64_t ad0 = tdesc0 + static_cast<uint64_t>((stage * kPStage) >> 4);
                    const uint64_t bd0 = ad0 + (kAStage >> 4);
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
                    if (MX) {
                        const uint64_t sd = sfdesc0 + static_cast<uint64_t>((stage * (kSfaBytes + kSfbBytes)) >> 4);
                        tmem_cp_32x128b_warpx4_pair(sfa_col, sd);
                        tmem_cp_32x128b_warpx4_pair(sfb_col, sd + (kSfaBytes >> 4));
                        tmem_cp_32x128b_warpx4_pair(sfb_col + 4, sd + ((kSfaBytes + 512) >> 4));
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
                        if (MX)
                            mma_mxf8_pair(tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc | (kk << 4) | (kk << 29), sfa_col,
                                          sfb_col, accum);
                        else mma_bf16_pair(tmem, ad0 + 2 * kk, bd0 + 2 * kk, idesc, accum);
                    }
                    tc_commit_pair(&empty[stage], 0x3);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit_pair(acc_full, 0x3);
                acc_phase ^= 1u;
            }
        mma_done:;
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        // 8 epilogue warps: warps 2-5 take columns [0, 128), warps 6-9 [128, 256)
        const int ecol = kEpiWarps == 8 ? ((warp - 2) >> 2) * 128 : 0;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(ecol);
        const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
        uint32_t acc_phase = 0;
        for (int tile = pair; tile < total; tile += npairs) {
            const Tile tl = locate(tile);
            const int e = tl.group;
            const int row_in_e = (2 * tl.m_blk + static_cast<int>(rank)) * kBM + r;
            // FFN1 / FFN2: the row's counts, offsets and token slot, looked up while
            // the tile's MMAs run
            bool valid = true;
            int64_t grow = 0;
            uint16_t *dst = nullptr;
            if constexpr (MODE != MODE_WGRAD) {
                valid = row_in_e < a.counts[e];
                grow = a.pad_offsets[e] + row_in_e;
                if (MODE == MODE_FFN2 && valid) {
                    const int64_t p = a.offsets[e] + row_in_e;
                    dst = a.ystage + (static_cast<int64_t>(a.row_tok[p]) * a.k_top + a.row_j[p]) * a.d +
                          tl.n_blk * 256;
                }
            }
            if (!wait_bar(acc_full, acc_phase, a.status, a.wait_ns, abort_flag)) break;
            tc_fence_after();
            bool released = false;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote_relaxed(acc_empty_leader);
                released = true;
            };
            if constexpr (MODE == MODE_WGRAD) {
                // dW rows (expert e) x this warp's columns; zeros for an expert without rows.
                // The accumulator is released once it is in registers; the rows go to this
                // warp's boxes (lane = row, 16-byte chunk c of a 128-byte box row at
                // c ^ (row & 7): the SWIZZLE_128B layout) and leave by TMA stores.
                constexpr int kCols = 256 / (kEpiWarps / 4);
                constexpr int kBoxes = kCols / 64;
                const bool empty_k = s_pad[e + 1] == s_pad[e];
                uint32_t pk[128];
                drain_row_bf16(trow, kCols, empty_k, pk);
                release();
                uint8_t *box = sOut + (warp - 2) * pair_box_bytes<MODE>();
                const uint32_t rbase = smem_u32(box) + static_cast<uint32_t>(lane) * 128u;
                const int x = tl.n_blk * 256 + ecol;
                const int y = e * a.m_rows + (2 * tl.m_blk + static_cast<int>(rank)) * kBM + quarter * 32;
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx) {
                    if (lane == 0) bulk_wait_group_read<0>();  // the box's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(rbase + ((c ^ (lane & 7)) << 4), pk[bx * 32 + 4 * c], pk[bx * 32 + 4 * c + 1],
                                     pk[bx * 32 + 4 * c + 2], pk[bx * 32 + 4 * c + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&pm.out, box, x + 64 * bx, y);
                        bulk_commit_group();
                    }
                }
            } else if constexpr (MODE == MODE_FFN1) {
                epi_ffn1<MX>(trow, valid, grow, tl.n_blk * 128, a.F, a.h, a.h_scales, a.h_rows, a.saved_a,
                             a.saved_b, a.saved_h, stage_out + (warp - 2) * kStageWords, lane, release);
            } else {
                epi_rows_bf16(trow, 256, false, valid, dst, stage_out + (warp - 2) * kStageWords, lane,
                              release);
            }
            if (!released) release();
            acc_phase ^= 1u;
        }
        if constexpr (MODE == MODE_WGRAD) {
            if (lane == 0) bulk_wait_group<0>();  // this warp's dW stores are complete
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no more remote arrives, loads or multicast commits into either CTA
    if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

template <int MODE, bool MX>
constexpr size_t pair_smem_bytes()
{
    constexpr int st = PairShape<MODE>::kStages;
    constexpr int ew = PairShape<MODE>::kEpiWarps;
    return 1024 + st * kPStage + ew * pair_box_bytes<MODE>() + (MX ? st * (kSfaBytes + kSfbBytes) : 0) +
           (2 * st + 2) * 8 + 16 + (MOK_MAX_EXPERTS + 4) * 4 +
           (MODE == MODE_WGRAD ? (MOK_MAX_EXPERTS + 4) * 4 : ew * kStageWords * 4);
}

template <int MODE, bool MX>
cudaError_t launch_gemm_pair(const PairMaps &pm, const GemmArgs &args, cudaStream_t st)
{
    constexpr size_t smem = pair_smem_bytes<MODE, MX>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int grid = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(PairShape<MODE>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(k_gemm_pair<MODE, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms() / 2 * 2));
        int clusters = 0;
        if (attr_err == cudaSuccess)
            attr_err = cudaOccupancyMaxActiveClusters(&clusters, k_gemm_pair<MODE, MX>, &cfg);
        grid = clusters * 2;
        if (attr_err == cudaSuccess && grid == 0) attr_err = cudaErrorInvalidConfiguration;
    });
    if (attr_err != cudaSuccess) return attr_err;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, k_gemm_pair<MODE, MX>, pm, args);
}

template <bool MX>
constexpr size_t smem_bytes()
{
    return 1024 + kStages * (kAStage + kBStage) + (MX ? kStages * (kSfaBytes + kSfbBytes) : 0) +
           (2 * kStages + 2) * 8 + 16 + (MOK_MAX_EXPERTS + 4) * 4 + kGemmStageBytes;
}

template <int MODE, bool MX>
cudaError_t launch_gemm(const AMaps<MODE == MODE_ROUTER ? 64 : 2> &am, const CUtensorMap &b0,
                        const CUtensorMap &b1, const GemmArgs &args, cudaStream_t st)
{
    constexpr size_t smem = smem_bytes<MX>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int grid = 0;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(k_gemm<MODE, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
        grid = num_sms();
        if (attr_err == cudaSuccess && kCluster > 1) {
            // CTAs of a cluster share a GPC (so one die and its L2 partition):
            // consecutive tiles -- the row tiles of one weight tile -- run side
            // by side there.  The grid is the number of clusters that fit at once.
            attr_err = cudaFuncSetAttribute(k_gemm<MODE, MX>,
                                            cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = kCluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(grid / kCluster * kCluster));
            cfg.blockDim = dim3(GemmShape<MODE>::kThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (attr_err == cudaSuccess)
                attr_err = cudaOccupancyMaxActiveClusters(&clusters, k_gemm<MODE, MX>, &cfg);
            if (attr_err == cudaSuccess) grid = clusters > 0 ? clusters * kCluster : 0;
            if (grid == 0) attr_err = cudaErrorInvalidConfiguration;
        }
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (kCluster > 1) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(GemmShape<MODE>::kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, k_gemm<MODE, MX>, am, b0, b1, args);
    }
    k_gemm<MODE, MX><<<grid, GemmShape<MODE>::kThreads, smem, st>>>(am, b0, b1, args);
    return cudaGetLastError();
}

GemmArgs base_args(const Dims &dm, uint32_t *status, uint64_t wait_ns)
{
    GemmArgs g = {};
    g.E = dm.E;
    g.F = dm.F;
    g.d = dm.d;
    g.k_top = dm.k;
    g.T = dm.T;
    g.status = status;
    g.wait_ns = wait_ns;
    return g;
}

}  // namespace

static_assert(kMaxRouterSources == 64, "router tensor-map table size");

cudaError_t launch_router_gemm(const Dims &dm, const Sources &src, const uint16_t *w3,
                               const float *bias, float *logits, uint32_t *status,
                               uint64_t wait_ns, cudaStream_t st)
{
    static AMaps<64> am;  // large: keep off the stack
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (src.n > kMaxRouterSources) return cudaErrorInvalidValue;
    am.n = src.n;
    int mt = 0;
    for (int s = 0; s < src.n; ++s) {
        const int rows = src.row_start[s + 1] - src.row_start[s];
        if (encode_tmap_2d(&am.m[s], src.ptr[s], false, dm.d, rows, 64, kBM)) return cudaErrorInvalidValue;
        am.mt_start[s] = mt;
        am.row_start[s] = src.row_start[s];
        am.rows[s] = rows;
        mt += (rows + kBM - 1) / kBM;
    }
    am.mt_start[src.n] = mt;
    am.row_start[src.n] = src.row_start[src.n];
    CUtensorMap b;
    if (encode_tmap_2d(&b, w3, false, 3 * static_cast<uint64_t>(dm.d), dm.E_pad, 64, 128))
        return cudaErrorInvalidValue;
    GemmArgs g = base_args(dm, status, wait_ns);
    g.E = src.n;
    g.BN = dm.E_pad >= 256 ? 256 : 128;
    g.n_tiles = dm.E_pad / g.BN;
    g.k_stages = 3 * dm.d / 64;
    g.a_k_stages = dm.d / 64;
    g.logits = logits;
    g.bias = bias;
    g.E_valid = dm.E;
    return launch_gemm<MODE_ROUTER, false>(am, b, b, g, st);
}

cudaError_t launch_ffn(const Dims &dm, const void *xe, const uint32_t *xe_scales,
                       const mok_weights *w, const int32_t *counts, const int32_t *offsets,
                       const int32_t *pad_offsets, const int32_t *row_tok,
                       const uint8_t *row_j, void *h, uint32_t *h_scales, uint16_t *ystage,
                       uint16_t *saved_a, uint16_t *saved_b, uint16_t *saved_h,
                       uint32_t *status, uint64_t wait_ns, cudaStream_t st)
{
    const bool mx = dm.dtype == MOK_MXFP8;
    const uint32_t box = mx ? 128 : 64;
    const uint64_t EF = static_cast<uint64_t>(dm.E) * dm.F;
    const uint64_t Ed = static_cast<uint64_t>(dm.E) * dm.d;
    AMaps<2> a1 = {}, a2 = {};
    CUtensorMap bg, bu, bd;
    if (encode_tmap_2d(&a1.m[0], xe, mx, dm.d, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&bg, mx ? static_cast<const void *>(w->q_gate) : w->w_gate, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&bu, mx ? static_cast<const void *>(w->q_up) : w->w_up, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&a2.m[0], h, mx, dm.F, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&bd, mx ? static_cast<const void *>(w->q_down) : w->w_down, mx, dm.F, Ed, box, 128))
        return cudaErrorInvalidValue;
    a1.n = a2.n = 1;

    GemmArgs g = base_args(dm, status, wait_ns);
    g.counts = counts;
    g.offsets = offsets;
    g.pad_offsets = pad_offsets;

    // GEMM1 + SwiGLU: N tile = 128 columns of F, as 128 gate + 128 up rows of B
    GemmArgs g1 = g;
    g1.BN = 256;
    g1.n_tiles = dm.F / 128;
    g1.k_stages = dm.d / static_cast<int>(box);
    g1.b_rows_per_group = dm.F;
    g1.sfa[0] = xe_scales;
    g1.sfa_rows[0] = dm.rows_pad;
    g1.sfb[0] = w->s_gate;
    g1.sfb[1] = w->s_up;
    g1.sfb_rows[0] = g1.sfb_rows[1] = static_cast<int64_t>(EF);
    g1.h = h;
    g1.h_scales = h_scales;
    g1.h_rows = dm.rows_pad;
    g1.saved_a = saved_a;
    g1.saved_b = saved_b;
    g1.saved_h = saved_h;
    // CTA pairs unless the config turns them off (MXFP8 expert FFN of the
    // DeepSeek-V3 shape 7.5 vs 8.0 ms, BF16 Mixtral shape 4.2 vs 4.3 ms on GB300)
    const bool pair = dm.gemm_pairs;
    PairMaps p1 = {}, p2 = {};
    if (pair) {
        p1.a = a1.m[0];
        p1.b0 = bg;
        p1.b1 = bu;
        p2.a = a2.m[0];
        p2.b0 = p2.b1 = bd;
        if (mx && (encode_tmap_scales(&p1.sa, xe_scales, dm.rows_pad, dm.d) ||
                   encode_tmap_scales(&p1.sb0, w->s_gate, EF, dm.d) ||
                   encode_tmap_scales(&p1.sb1, w->s_up, EF, dm.d) ||
                   encode_tmap_scales(&p2.sa, h_scales, dm.rows_pad, dm.F) ||
                   encode_tmap_scales(&p2.sb0, w->s_down, Ed, dm.F)))
            return cudaErrorInvalidValue;
        p2.sb1 = p2.sb0;
        if (!mx) p1.sa = p1.sb0 = p1.sb1 = p2.sa = p2.sb0 = p2.sb1 = bd;  // unused
    }
    cudaError_t err;
    if (pair)
        err = mx ? launch_gemm_pair<MODE_FFN1, true>(p1, g1, st) : launch_gemm_pair<MODE_FFN1, false>(p1, g1, st);
    else
        err = mx ? launch_gemm<MODE_FFN1, true>(a1, bg, bu, g1, st)
                 : launch_gemm<MODE_FFN1, false>(a1, bg, bu, g1, st);
    if (err != cudaSuccess) return err;

    // GEMM2: y = h W_d^T scattered to ystage
    GemmArgs g2 = g;
    g2.BN = dm.d % 256 == 0 ? 256 : 128;
    g2.n_tiles = dm.d / g2.BN;
    g2.k_stages = dm.F / static_cast<int>(box);
    g2.b_rows_per_group = dm.d;
    g2.sfa[0] = h_scales;
    g2.sfa_rows[0] = dm.rows_pad;
    g2.sfb[0] = g2.sfb[1] = w->s_down;
    g2.sfb_rows[0] = g2.sfb_rows[1] = static_cast<int64_t>(Ed);
    g2.ystage = ystage;
    g2.row_tok = row_tok;
    g2.row_j = row_j;
    if (pair && g2.BN == 256)
        return mx ? launch_gemm_pair<MODE_FFN2, true>(p2, g2, st) : launch_gemm_pair<MODE_FFN2, false>(p2, g2, st);
    return mx ? launch_gemm<MODE_FFN2, true>(a2, bd, bd, g2, st)
              : launch_gemm<MODE_FFN2, false>(a2, bd, bd, g2, st);
}

cudaError_t launch_dgrad(const Dims &dm, const BwdBufs &b, const mok_weights *w,
                         const int32_t *counts, const int32_t *pad_offsets, uint32_t *status,
                         uint64_t wait_ns, cudaStream_t st)
{
    const bool mx = dm.dtype == MOK_MXFP8;
    const uint32_t box = mx ? 128 : 64;
    const uint64_t EF = static_cast<uint64_t>(dm.E) * dm.F;
    const uint64_t Ed = static_cast<uint64_t>(dm.E) * dm.d;
    const void *wdT = mx ? static_cast<const void *>(w->qt_down) : w->wt_down;
    const void *wgT = mx ? static_cast<const void *>(w->qt_gate) : w->wt_gate;
    const void *wuT = mx ? static_cast<const void *>(w->qt_up) : w->wt_up;
    AMaps<2> a2 = {}, a1 = {};
    CUtensorMap bdT, bgT, buT;
    if (encode_tmap_2d(&a2.m[0], mx ? static_cast<const void *>(b.dy_q) : b.dy, mx, dm.d, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&bdT, wdT, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&a1.m[0], mx ? static_cast<const void *>(b.da_q) : b.da, mx, dm.F, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&a1.m[1], mx ? static_cast<const void *>(b.db_q) : b.db, mx, dm.F, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&bgT, wgT, mx, dm.F, Ed, box, 128) ||
        encode_tmap_2d(&buT, wuT, mx, dm.F, Ed, box, 128))
        return cudaErrorInvalidValue;
    a2.n = 1;
    a1.n = 2;
    GemmArgs g = base_args(dm, status, wait_ns);
    g.counts = counts;
    g.pad_offsets = pad_offsets;

    // dh = dy W_d (K = d) -> SwiGLU backward -> da, db
    GemmArgs g2 = g;
    g2.BN = dm.F % 256 == 0 ? 256 : 128;
    g2.n_tiles = dm.F / g2.BN;
    g2.k_stages = dm.d / static_cast<int>(box);
    g2.b_rows_per_group = dm.F;
    g2.sfa[0] = b.dy_s;
    g2.sfa_rows[0] = dm.rows_pad;
    g2.sfb[0] = g2.sfb[1] = w->st_down;
    g2.sfb_rows[0] = g2.sfb_rows[1] = static_cast<int64_t>(EF);
    g2.in_a = b.saved_a;
    g2.in_b = b.saved_b;
    g2.out_da = b.da;
    g2.out_db = b.db;
    g2.q_da = b.da_q;
    g2.q_db = b.db_q;
    g2.s_da = b.da_s;
    g2.s_db = b.db_s;
    g2.h_rows = dm.rows_pad;
    cudaError_t err = mx ? launch_gemm<MODE_DGRAD2, true>(a2, bdT, bdT, g2, st)
                         : launch_gemm<MODE_DGRAD2, false>(a2, bdT, bdT, g2, st);
    if (err != cudaSuccess) return err;

    // dx = da W_g + db W_u (K = 2F)
    GemmArgs g1 = g;
    g1.BN = dm.d % 256 == 0 ? 256 : 128;
    g1.n_tiles = dm.d / g1.BN;
    g1.ks_half = dm.F / static_cast<int>(box);
    g1.k_stages = 2 * g1.ks_half;
    g1.b_rows_per_group = dm.d;
    g1.sfa[0] = b.da_s;
    g1.sfa[1] = b.db_s;
    g1.sfa_rows[0] = g1.sfa_rows[1] = dm.rows_pad;
    g1.sfb[0] = w->st_gate;
    g1.sfb[1] = w->st_up;
    g1.sfb_rows[0] = g1.sfb_rows[1] = static_cast<int64_t>(Ed);
    g1.out_rows = b.dx;
    return mx ? launch_gemm<MODE_DGRAD1, true>(a1, bgT, buT, g1, st)
              : launch_gemm<MODE_DGRAD1, false>(a1, bgT, buT, g1, st);
}

cudaError_t launch_wgrad(const Dims &dm, const void *A_T, const uint32_t *A_s, int64_t a_rows,
                         const void *B_T, const uint32_t *B_s, int64_t b_rows,
                         const int32_t *pad_offsets, uint16_t *dW, uint32_t *status,
                         uint64_t wait_ns, cudaStream_t st)
{
    const bool mx = dm.dtype == MOK_MXFP8;
    const uint32_t box = mx ? 128 : 64;
    AMaps<2> am = {};
    CUtensorMap bm;
    if (encode_tmap_2d(&am.m[0], A_T, mx, dm.rows_pad, a_rows, box, kBM) ||
        encode_tmap_2d(&bm, B_T, mx, dm.rows_pad, b_rows, box, 128))
        return cudaErrorInvalidValue;
    am.n = 1;
    GemmArgs g = base_args(dm, status, wait_ns);
    g.pad_offsets = pad_offsets;
    if (dm.gemm_pairs && a_rows % 256 == 0 && b_rows % 256 == 0) {
        // CTA pairs: 256 dW rows x 256 columns per pair tile
        PairMaps pm = {};
        pm.a = am.m[0];
        pm.b0 = pm.b1 = bm;
        if (mx && (encode_tmap_scales(&pm.sa, A_s, static_cast<uint64_t>(a_rows), static_cast<uint64_t>(dm.rows_pad)) ||
                   encode_tmap_scales(&pm.sb0, B_s, static_cast<uint64_t>(b_rows), static_cast<uint64_t>(dm.rows_pad))))
            return cudaErrorInvalidValue;
        pm.sb1 = pm.sb0;
        if (!mx) pm.sa = pm.sb0 = pm.sb1 = bm;  // unused
        if (encode_tmap_2d(&pm.out, dW, false, static_cast<uint64_t>(b_rows),
                           static_cast<uint64_t>(dm.E) * static_cast<uint64_t>(a_rows), 64, 32))
            return cudaErrorInvalidValue;
        g.BN = 256;
        g.n_tiles = static_cast<int>(b_rows / 256);
        g.m_rows = static_cast<int>(a_rows);
        g.sfa_rows[0] = a_rows;
        g.sfb_rows[0] = g.sfb_rows[1] = b_rows;
        g.out_rows = dW;
        g.out_ld = b_rows;
        return mx ? launch_gemm_pair<MODE_WGRAD, true>(pm, g, st) : launch_gemm_pair<MODE_WGRAD, false>(pm, g, st);
    }
    g.BN = b_rows % 256 == 0 ? 256 : 128;
    g.n_tiles = static_cast<int>(b_rows / g.BN);
    g.m_rows = static_cast<int>(a_rows);
    g.sfa[0] = A_s;
    g.sfa_rows[0] = a_rows;
    g.sfb[0] = g.sfb[1] = B_s;
    g.sfb_rows[0] = g.sfb_rows[1] = b_rows;
    g.out_rows = dW;
    g.out_ld = b_rows;
    return mx ? launch_gemm<MODE_WGRAD, true>(am, bm, bm, g, st)
              : launch_gemm<MODE_WGRAD, false>(am, bm, bm, g, st);
}

// ---------------------------------------------------------------------------
// The FFN1 epilogue's SwiGLU and MXFP8 quantisation of h, run on fp32 a, b
// read from memory (mok_swiglu_quantize_mx): one thread per row and block of
// 32 columns along F, through the same swiglu_f32 and mx_block32 as the
// epilogues, so the codes and scales it writes are the ones the expert GEMM
// writes for the same fp32 accumulator values.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_swiglu_quant(const float *__restrict__ a,
                                                      const float *__restrict__ b, int64_t rows, int F,
                                                      float *__restrict__ h, uint8_t *__restrict__ codes,
                                                      uint32_t *__restrict__ scales)
{
    const int64_t nblk = F / 32;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * nblk) return;
    const int64_t r = i / nblk;
    const int c = static_cast<int>(i % nblk) * 32;
    const int64_t off = r * F + c;
    float hv[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) hv[j] = swiglu_f32(a[off + j], b[off + j]);
    if (h) {
#pragma unroll
        for (int j = 0; j < 32; ++j) h[off + j] = hv[j];
    }
    uint32_t q[8];
    const uint32_t sb = mx_block32(hv, q);
    uint4 *o = reinterpret_cast<uint4 *>(codes + off);
    o[0] = make_uint4(q[0], q[1], q[2], q[3]);
    o[1] = make_uint4(q[4], q[5], q[6], q[7]);
    // byte (c / 32) % 4 of the word of k-group c / 128 holds this block's scale
    reinterpret_cast<uint8_t *>(scales + scale_word_row(c >> 7, r, rows))[(c >> 5) & 3] =
        static_cast<uint8_t>(sb);
}

cudaError_t launch_swiglu_quant(const float *a, const float *b, int64_t rows, int64_t F, float *h,
                                uint8_t *codes, uint32_t *scales, cudaStream_t st)
{
    const int64_t threads = rows * (F / 32);
    k_swiglu_quant<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(
        a, b, rows, static_cast<int>(F), h, codes, scales);
    return cudaGetLastError();
}

}  // namespace mok
