// mok_gemm.cu -- tcgen05 grouped GEMMs of the MoE layer on sm_103a.
//
// [kucoin] = "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
// NVL72" (kucoin.com flash, Arabic).  §01: the grouped GEMM needs each
// expert's tokens organised together before it can feed the tensor cores;
// §02: MXFP8 activation quantisation is fused into the grouped GEMM and
// SwiGLU, and combine is a push -- each result goes straight to the token it
// came from.
//
// One persistent kernel template, one CTA per SM, 6 warps:
//   warp 0      TMA producer: A tile (128 rows) and B tile (128 or 256 rows)
//               of 128 bytes along K per stage, plus MX scale tiles, into a
//               4-stage shared-memory ring (mbarrier full/empty pairs);
//   warp 1      allocates TMEM and issues tcgen05.mma from one thread into a
//               128 x N fp32 accumulator (N = 256 or 128);
//   warps 2..5  epilogue: each thread owns one accumulator row (its TMEM
//               lane) and runs the mode's epilogue straight from registers.
// Modes:
//   ROUTER  plain GEMM x . [W_hi | W_mid | W_lo]^T over the token rows of each
//           source buffer (A's K wraps three times), fp32 logits (+ bias);
//   FFN1    per expert, B = 128 rows of W_g and the same 128 rows of W_u, so
//           one tile holds a and b for 128 columns of F: h = silu(a) b, stored
//           BF16 or MXFP8 (blocks of 32 along F, quantised in registers);
//   FFN2    per expert, y = h W_d^T stored BF16 into ystage[token, j].
// Tiles are ordered expert by expert, N-tile by N-tile, with the expert's row
// tiles innermost, and dealt round-robin to the CTAs: concurrently running
// CTAs share B tiles and the expert's rows through L2.
#include <cuda_bf16.h>

#include <mutex>

#include "mok_internal.h"
#include "mok_ptx.cuh"

namespace mok {

namespace {

constexpr int kThreads = 192;
constexpr int kStages = 4;
constexpr int kBM = 128;
constexpr int kBKBytes = 128;
constexpr int kAStage = kBM * kBKBytes;   // 16 KB
constexpr int kBStage = 256 * kBKBytes;   // 32 KB
constexpr int kSfaBytes = 512;            // 128 rows x 4 scale bytes
constexpr int kSfbBytes = 1024;           // 256 rows x 4 scale bytes
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;          // scale columns: 16 per stage after the accumulator

enum { MODE_ROUTER = 0, MODE_FFN1 = 1, MODE_FFN2 = 2 };

template <int NA>
struct AMaps {
    CUtensorMap m[NA];
    int mt_start[NA + 1];   // router: first row tile of each source
    int row_start[NA + 1];  // router: first token of each source
    int rows[NA];           // router: rows of each source
    int n;
};

struct GemmArgs {
    int E;                  // groups (experts); router: 1
    const int32_t *counts;
    const int32_t *offsets;
    const int32_t *pad_offsets;
    int n_tiles;            // N tiles per group
    int BN;                 // MMA N: 128 or 256
    int k_stages;           // K / (128 bytes)
    int a_k_stages;         // K stages of A before it wraps (router), else k_stages
    int b_rows_per_group;   // rows of B per expert
    // MX scales (tile layout)
    const uint32_t *sfa;
    int64_t sfa_rows;
    const uint32_t *sfb0, *sfb1;
    int64_t sfb_rows;
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

__device__ __noinline__ void report_timeout(uint32_t *status, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (status) atomicMax(status, static_cast<uint32_t>(MOK_ERR_TIMEOUT));
}

// Bounded mbarrier wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, const GemmArgs &a,
                                         volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > a.wait_ns) {
                report_timeout(a.status, abort_flag);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void store_bf16x32(uint16_t *dst, const float *v)
{
    uint4 *o = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        o[q] = w;
    }
}

template <int MODE, bool MX, int NA>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm(const __grid_constant__ AMaps<NA> am, const __grid_constant__ CUtensorMap tmB0,
           const __grid_constant__ CUtensorMap tmB1, const GemmArgs a)
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

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int groups = MODE == MODE_ROUTER ? am.n : a.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < (MODE == MODE_ROUTER ? am.n : 1); ++i) prefetch_tmap(&am.m[i]);
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
        for (int g = g0; g < g0 + per && g < groups; ++g) {
            int mt;
            if (MODE == MODE_ROUTER) mt = am.mt_start[g + 1] - am.mt_start[g];
            else mt = (a.pad_offsets[g + 1] - a.pad_offsets[g]) / kBM;
            local += mt * a.n_tiles;
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int g = g0; g < g0 + per && g < groups; ++g) {
            prefix[g] = run;
            int mt;
            if (MODE == MODE_ROUTER) mt = am.mt_start[g + 1] - am.mt_start[g];
            else mt = (a.pad_offsets[g + 1] - a.pad_offsets[g]) / kBM;
            run += mt * a.n_tiles;
        }
        if (lane == 31) prefix[groups] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int total = prefix[groups];
    const int BN = a.BN;
    constexpr int kElemsPerStage = MX ? 128 : 64;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t stage = 0, phase = 0;
            const uint32_t stage_bytes = kAStage + (BN / 128) * 16384 +
                                         (MX ? kSfaBytes + (BN / 128) * 512 : 0);
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                const Tile tl = decode_tile(tile, prefix, groups, a.n_tiles);
                int a_row, b_row, ai = 0;
                if (MODE == MODE_ROUTER) {
                    ai = tl.group;
                    a_row = tl.m_blk * kBM;
                    b_row = tl.n_blk * BN;
                } else {
                    a_row = a.pad_offsets[tl.group] + tl.m_blk * kBM;
                    b_row = tl.group * a.b_rows_per_group + tl.n_blk * (MODE == MODE_FFN1 ? 128 : BN);
                }
                for (int ks = 0; ks < a.k_stages; ++ks) {
                    if (!wait_bar(&empty[stage], phase ^ 1u, a, abort_flag)) goto producer_done;
                    uint8_t *dA = sA + stage * kAStage;
                    uint8_t *dB = sB + stage * kBStage;
                    const int ka = (ks % a.a_k_stages) * kElemsPerStage;
                    const int kb = ks * kElemsPerStage;
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    tma_load_2d(dA, &am.m[ai], &full[stage], ka, a_row);
                    tma_load_2d(dB, &tmB0, &full[stage], kb, b_row);
                    if (BN == 256) {
                        if (MODE == MODE_FFN1) tma_load_2d(dB + 16384, &tmB1, &full[stage], kb, b_row);
                        else tma_load_2d(dB + 16384, &tmB0, &full[stage], kb, b_row + 128);
                    }
                    if (MX) {
                        uint8_t *dS = sSF + stage * (kSfaBytes + kSfbBytes);
                        const uint32_t *sa = a.sfa + (static_cast<int64_t>(ks) * (a.sfa_rows >> 7) + (a_row >> 7)) * 128;
                        bulk_load(dS, sa, kSfaBytes, &full[stage]);
                        const uint32_t *sb = a.sfb0 + (static_cast<int64_t>(ks) * (a.sfb_rows >> 7) + (b_row >> 7)) * 128;
                        if (MODE == MODE_FFN1) {
                            bulk_load(dS + kSfaBytes, sb, 512, &full[stage]);
                            const uint32_t *su = a.sfb1 + (static_cast<int64_t>(ks) * (a.sfb_rows >> 7) + (b_row >> 7)) * 128;
                            bulk_load(dS + kSfaBytes + 512, su, 512, &full[stage]);
                        } else {
                            bulk_load(dS + kSfaBytes, sb, (BN / 128) * 512, &full[stage]);
                        }
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
            const uint32_t idesc = idesc_bf16(kBM, BN);
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                if (!wait_bar(acc_empty, acc_phase ^ 1u, a, abort_flag)) break;
                tc_fence_after();
                for (int ks = 0; ks < a.k_stages; ++ks) {
                    if (!wait_bar(&full[stage], phase, a, abort_flag)) goto mma_done;
                    tc_fence_after();
                    const uint32_t aaddr = smem_u32(sA + stage * kAStage);
                    const uint32_t baddr = smem_u32(sB + stage * kBStage);
                    const uint32_t sfa_col = tmem + kSfCol + stage * 16;
                    const uint32_t sfb_col = sfa_col + 4;
                    if (MX) {
                        const uint32_t sbase = smem_u32(sSF + stage * (kSfaBytes + kSfbBytes));
                        tmem_cp_32x128b_warpx4(sfa_col, sdesc_sf(sbase));
                        tmem_cp_32x128b_warpx4(sfb_col, sdesc_sf(sbase + kSfaBytes));
                        if (BN == 256) tmem_cp_32x128b_warpx4(sfb_col + 4, sdesc_sf(sbase + kSfaBytes + 512));
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_k_sw128(aaddr + kk * 32);
                        const uint64_t bd = sdesc_k_sw128(baddr + kk * 32);
                        const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
                        if (MX) mma_mxf8(tmem, ad, bd, idesc_mxf8(kBM, BN, kk, kk), sfa_col, sfb_col, accum);
                        else mma_bf16(tmem, ad, bd, idesc, accum);
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
            if (!wait_bar(acc_full, acc_phase, a, abort_flag)) break;
            tc_fence_after();
            if (MODE == MODE_ROUTER) {
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
            } else if (MODE == MODE_FFN1) {
                const int e = tl.group;
                const int row_in_e = tl.m_blk * kBM + r;
                const bool valid = row_in_e < a.counts[e];
                const int64_t grow = a.pad_offsets[e] + row_in_e;
                const int f0 = tl.n_blk * 128;
                uint32_t sword = 0;
                for (int c = 0; c < 128; c += 32) {
                    uint32_t gv[32], uv[32];
                    tmem_ld_32x32(trow + c, gv);
                    tmem_ld_32x32(trow + 128 + c, uv);
                    tmem_ld_wait();
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float av = __uint_as_float(gv[i]);
                        const float bv = __uint_as_float(uv[i]);
                        hv[i] = av / (1.0f + __expf(-av)) * bv;
                    }
                    if (valid) {
                        const int64_t off = grow * a.F + f0 + c;
                        if (a.saved_a) {
                            float t[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(gv[i]);
                            store_bf16x32(a.saved_a + off, t);
                        }
                        if (a.saved_b) {
                            float t[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(uv[i]);
                            store_bf16x32(a.saved_b + off, t);
                        }
                        if (!MX) {
                            store_bf16x32(static_cast<uint16_t *>(a.h) + off, hv);
                            if (a.saved_h) store_bf16x32(a.saved_h + off, hv);
                        } else {
                            float amax = 0.0f;
#pragma unroll
                            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
                            const int x = mx_scale_exp(amax);
                            const float inv = mx_inv_scale(x);
                            uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.h) + off);
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                uint4 w;
                                const float *s = hv + 16 * q;
                                w.x = pack_e4m3x2(s[0] * inv, s[1] * inv) | (pack_e4m3x2(s[2] * inv, s[3] * inv) << 16);
                                w.y = pack_e4m3x2(s[4] * inv, s[5] * inv) | (pack_e4m3x2(s[6] * inv, s[7] * inv) << 16);
                                w.z = pack_e4m3x2(s[8] * inv, s[9] * inv) | (pack_e4m3x2(s[10] * inv, s[11] * inv) << 16);
                                w.w = pack_e4m3x2(s[12] * inv, s[13] * inv) | (pack_e4m3x2(s[14] * inv, s[15] * inv) << 16);
                                o[q] = w;
                            }
                            sword |= static_cast<uint32_t>(x + 127) << (8 * (c >> 5));
                            if (a.saved_h) store_bf16x32(a.saved_h + off, hv);
                        }
                    }
                }
                if (MX && valid) {
                    const int64_t g = f0 >> 7;
                    a.h_scales[(g * (a.h_rows >> 7) + (grow >> 7)) * 128 + (grow & 31) * 4 + ((grow & 127) >> 5)] = sword;
                }
            } else {
                const int e = tl.group;
                const int row_in_e = tl.m_blk * kBM + r;
                const bool valid = row_in_e < a.counts[e];
                uint16_t *dst = nullptr;
                if (valid) {
                    const int64_t p = a.offsets[e] + row_in_e;
                    const int64_t t = a.row_tok[p];
                    const int64_t j = a.row_j[p];
                    dst = a.ystage + (t * a.k_top + j) * a.d + tl.n_blk * BN;
                }
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32(trow + c, v);
                    tmem_ld_wait();
                    if (valid) {
                        float f[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
                        store_bf16x32(dst + c, f);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
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

template <int MODE, bool MX, int NA>
constexpr size_t smem_bytes()
{
    return 1024 + kStages * (kAStage + kBStage) + (MX ? kStages * (kSfaBytes + kSfbBytes) : 0) +
           (2 * kStages + 2) * 8 + 16 + (MOK_MAX_EXPERTS + 1) * 4;
}

template <int MODE, bool MX, int NA>
cudaError_t launch_gemm(const AMaps<NA> &am, const CUtensorMap &b0, const CUtensorMap &b1,
                        const GemmArgs &args, cudaStream_t st)
{
    constexpr size_t smem = smem_bytes<MODE, MX, NA>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(k_gemm<MODE, MX, NA>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    k_gemm<MODE, MX, NA><<<num_sms(), kThreads, smem, st>>>(am, b0, b1, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_gemm(const Dims &dm, const Sources &src, const uint16_t *w3,
                               const float *bias, float *logits, uint32_t *status,
                               uint64_t wait_ns, cudaStream_t st)
{
    static AMaps<kMaxRouterSources> am;  // large: keep off the stack
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
    GemmArgs g = {};
    g.E = 1;
    g.BN = dm.E_pad >= 256 ? 256 : 128;
    g.n_tiles = dm.E_pad / g.BN;
    g.k_stages = 3 * dm.d / 64;
    g.a_k_stages = dm.d / 64;
    g.T = dm.T;
    g.logits = logits;
    g.bias = bias;
    g.E_valid = dm.E;
    g.status = status;
    g.wait_ns = wait_ns;
    return launch_gemm<MODE_ROUTER, false, kMaxRouterSources>(am, b, b, g, st);
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
    AMaps<1> a1 = {}, a2 = {};
    CUtensorMap bg, bu, bd;
    if (encode_tmap_2d(&a1.m[0], xe, mx, dm.d, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&bg, mx ? static_cast<const void *>(w->q_gate) : w->w_gate, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&bu, mx ? static_cast<const void *>(w->q_up) : w->w_up, mx, dm.d, EF, box, 128) ||
        encode_tmap_2d(&a2.m[0], h, mx, dm.F, dm.rows_pad, box, kBM) ||
        encode_tmap_2d(&bd, mx ? static_cast<const void *>(w->q_down) : w->w_down, mx, dm.F, Ed, box, 128))
        return cudaErrorInvalidValue;
    a1.n = a2.n = 1;

    GemmArgs g = {};
    g.E = dm.E;
    g.counts = counts;
    g.offsets = offsets;
    g.pad_offsets = pad_offsets;
    g.F = dm.F;
    g.d = dm.d;
    g.k_top = dm.k;
    g.T = dm.T;
    g.status = status;
    g.wait_ns = wait_ns;

    // GEMM1 + SwiGLU: N tile = 128 columns of F, as 128 gate + 128 up rows of B
    GemmArgs g1 = g;
    g1.BN = 256;
    g1.n_tiles = dm.F / 128;
    g1.k_stages = dm.d / static_cast<int>(box);
    g1.a_k_stages = g1.k_stages;
    g1.b_rows_per_group = dm.F;
    g1.sfa = xe_scales;
    g1.sfa_rows = dm.rows_pad;
    g1.sfb0 = w->s_gate;
    g1.sfb1 = w->s_up;
    g1.sfb_rows = static_cast<int64_t>(EF);
    g1.h = h;
    g1.h_scales = h_scales;
    g1.h_rows = dm.rows_pad;
    g1.saved_a = saved_a;
    g1.saved_b = saved_b;
    g1.saved_h = saved_h;
    cudaError_t err = mx ? launch_gemm<MODE_FFN1, true, 1>(a1, bg, bu, g1, st)
                         : launch_gemm<MODE_FFN1, false, 1>(a1, bg, bu, g1, st);
    if (err != cudaSuccess) return err;

    // GEMM2: y = h W_d^T scattered to ystage
    GemmArgs g2 = g;
    g2.BN = dm.d % 256 == 0 ? 256 : 128;
    g2.n_tiles = dm.d / g2.BN;
    g2.k_stages = dm.F / static_cast<int>(box);
    g2.a_k_stages = g2.k_stages;
    g2.b_rows_per_group = dm.d;
    g2.sfa = h_scales;
    g2.sfa_rows = dm.rows_pad;
    g2.sfb0 = w->s_down;
    g2.sfb1 = w->s_down;
    g2.sfb_rows = static_cast<int64_t>(Ed);
    g2.ystage = ystage;
    g2.row_tok = row_tok;
    g2.row_j = row_j;
    return mx ? launch_gemm<MODE_FFN2, true, 1>(a2, bd, bd, g2, st)
              : launch_gemm<MODE_FFN2, false, 1>(a2, bd, bd, g2, st);
}

}  // namespace mok
