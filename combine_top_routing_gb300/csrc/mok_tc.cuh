// mok_tc.cuh -- building blocks shared by the tcgen05 GEMM kernels: tile and
// pipeline constants, bounded waits, and the register-level epilogue helpers
// (BF16 packing, MXFP8 block quantisation, MX scale tile addressing).
#pragma once

#include "mok.h"
#include "mok_ptx.cuh"

namespace mok {

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


static __device__ __noinline__ void report_timeout(uint32_t *status, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (status) atomicMax(status, static_cast<uint32_t>(MOK_ERR_TIMEOUT));
}

// Bounded mbarrier wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, uint32_t *status,
                                         uint64_t wait_ns, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > wait_ns) {
                report_timeout(status, abort_flag);
                return false;
            }
        }
    }
}

// wait_bar with cluster-scope acquire (barriers another CTA arrives on after
// writing into this CTA's shared memory).
__device__ __forceinline__ bool wait_bar_cluster(uint64_t *bar, uint32_t parity, uint32_t *status,
                                                 uint64_t wait_ns, volatile int *abort_flag)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > wait_ns) {
                report_timeout(status, abort_flag);
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

__device__ __forceinline__ void load_bf16x32(const uint16_t *src, float *v)
{
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 w = p[q];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * q + 2 * i] = bf16_bits_to_float(u[i] & 0xFFFFu);
            v[8 * q + 2 * i + 1] = bf16_bits_to_float(u[i] >> 16);
        }
    }
}

// SwiGLU of one accumulator element pair: h = silu(a) b, silu(a) = a / (1 + e^-a),
// the quotient by the fast reciprocal (a few ulp in fp32, far below the BF16 or
// MXFP8 rounding of h that follows; for a < -88, 1 + e^-a is infinite and
// silu(a) is -0).
__device__ __forceinline__ float swiglu_f32(float a, float b) { return __fdividef(a, 1.0f + __expf(-a)) * b; }

// 32 fp32 values -> one MX block: 32 E4M3 codes packed four per word into q;
// returns the E8M0 scale byte.  Every MXFP8 quantisation of h (the FFN1
// epilogues and mok_swiglu_quantize_mx) runs this function.
__device__ __forceinline__ uint32_t mx_block32(const float (&v)[32], uint32_t (&q)[8])
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int x = mx_scale_exp(amax);
    const float inv = mx_inv_scale(x);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        q[i] = pack_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
               (pack_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
    return static_cast<uint32_t>(x + 127);
}

// 32 fp32 values -> one MX block: 32 E4M3 codes at dst (16-byte aligned);
// returns the E8M0 scale byte.
__device__ __forceinline__ uint32_t quant_mx32(const float (&v)[32], uint8_t *dst)
{
    uint32_t q[8];
    const uint32_t s = mx_block32(v, q);
    uint4 *o = reinterpret_cast<uint4 *>(dst);
    o[0] = make_uint4(q[0], q[1], q[2], q[3]);
    o[1] = make_uint4(q[4], q[5], q[6], q[7]);
    return s;
}

__device__ __forceinline__ int64_t scale_word(int64_t x_elem, int64_t row, int64_t rows)
{
    return ((x_elem >> 7) * (rows >> 7) + (row >> 7)) * 128;
}

__device__ __forceinline__ int64_t scale_word_row(int64_t g, int64_t r, int64_t rows)
{
    return (g * (rows >> 7) + (r >> 7)) * 128 + (r & 31) * 4 + ((r & 127) >> 5);
}

// Reads BN (<= 256) fp32 accumulator columns of this thread's TMEM lane into
// packed BF16 pairs (zeros when `zero`), 64 columns per TMEM wait.
__device__ __forceinline__ void drain_row_bf16(uint32_t trow, int BN, bool zero, uint32_t (&pk)[128])
{
#pragma unroll
    for (int c = 0; c < 256; c += 64) {
        if (c < BN) {
            uint32_t v0[32], v1[32];
            if (!zero) {
                tmem_ld_32x32(trow + c, v0);
                tmem_ld_32x32(trow + c + 32, v1);
                tmem_ld_wait();
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                pk[c / 2 + i] = zero ? 0u : pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
                pk[c / 2 + 16 + i] =
                    zero ? 0u : pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
            }
        }
    }
}

// Shared-memory staging for epilogue stores: 32 rows x 33 words per warp
// (one padding word per row keeps the row-wise writes conflict-free).
constexpr int kStageWords = 32 * 33;
constexpr int kStageBytes = 4 * kStageWords * 4;  // four epilogue warps

// Writes each lane's row -- nwords 32-bit words of pk (nwords a multiple of
// 32) -- to dst (nullptr: skip the row) as contiguous 128-byte segments: one
// 128-byte column slice of the warp's 32 rows at a time goes through `stage`,
// then eight lanes store one row's slice, four rows per instruction.
template <int MAXW>
__device__ __forceinline__ void store_rows_staged(const uint32_t (&pk)[MAXW], int nwords, void *dst,
                                                  uint32_t *stage, int lane)
{
    const unsigned long long d64 = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
    for (int c0 = 0; c0 < MAXW; c0 += 32) {
        if (c0 < nwords) {
#pragma unroll
            for (int i = 0; i < 32; ++i) stage[lane * 33 + i] = pk[c0 + i];
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int row = j * 4 + (lane >> 3);
                const int w = (lane & 7) * 4;
                const unsigned long long rd = __shfl_sync(0xffffffffu, d64, row);
                if (rd) {
                    const uint32_t *sp = stage + row * 33 + w;
                    *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(rd) + (c0 + w) * 4) =
                        make_uint4(sp[0], sp[1], sp[2], sp[3]);
                }
            }
            __syncwarp();
        }
    }
}

// Stores NW words (NW * 4 bytes at a 16-byte aligned dst) of each of the
// warp's 32 rows (lane = row; a null dst stores nothing for that row) through
// `stage` (32 rows of NW + 1 words): NW / 4 lanes then write one row's words,
// 16 bytes each, so a store instruction covers 128 / NW rows' whole segments
// instead of 32 rows' 16-byte pieces.  Every lane of the warp calls it.
template <int NW>
__device__ __forceinline__ void store_rows_staged_n(const uint32_t (&pk)[NW], void *dst, uint32_t *stage, int lane)
{
    static_assert(NW == 8 || NW == 16 || NW == 32, "row segment of 32, 64 or 128 bytes");
    constexpr int kStride = NW + 1;  // odd: the per-lane writes hit distinct banks
    constexpr int kLanesPerRow = NW / 4;
    constexpr int kRowsPerStore = 32 / kLanesPerRow;
    const unsigned long long d64 = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
    for (int i = 0; i < NW; ++i) stage[lane * kStride + i] = pk[i];
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kLanesPerRow; ++j) {
        const int row = j * kRowsPerStore + lane / kLanesPerRow;
        const int w = (lane % kLanesPerRow) * 4;
        const unsigned long long rd = __shfl_sync(0xffffffffu, d64, row);
        if (rd) {
            const uint32_t *sp = stage + row * kStride + w;
            *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(rd) + w * 4) =
                make_uint4(sp[0], sp[1], sp[2], sp[3]);
        }
    }
    __syncwarp();
}

// 32 fp32 values -> 16 BF16 pairs (round to nearest even, as store_bf16x32).
__device__ __forceinline__ void pack_bf16x32(const float (&v)[32], uint32_t (&pk)[16])
{
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}

// Stores BN packed BF16 values (16-byte stores).
__device__ __forceinline__ void store_row_bf16(uint16_t *dst, int BN, const uint32_t (&pk)[128])
{
    uint4 *o = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int c = 0; c < 256; c += 8)
        if (c < BN) o[c / 8] = make_uint4(pk[c / 2], pk[c / 2 + 1], pk[c / 2 + 2], pk[c / 2 + 3]);
}

// FFN1 epilogue of one accumulator row (TMEM lane): columns [0,128) hold
// a = x W_g^T and [128,256) b = x W_u^T for 128 columns of F starting at f0.
// h = silu(a) b is stored BF16 or MXFP8 (one block of 32 along F per chunk,
// quantised in registers) at row `grow` of h; training also stores a, b, h in
// BF16.  Inference drains h into registers and calls release() before the
// global stores.
template <bool MX, typename Release>
__device__ __forceinline__ void epi_ffn1(uint32_t trow, bool valid, int64_t grow, int f0, int F,
                                         void *h, uint32_t *h_scales, int64_t h_rows,
                                         uint16_t *saved_a, uint16_t *saved_b, uint16_t *saved_h,
                                         uint32_t *stage, int lane, Release &&release)
{
    uint32_t sword = 0;
    if (!saved_a && !saved_b && !saved_h) {
        // inference: h for the row's 128 columns into registers, release, store
        uint32_t hq[64];  // BF16 pairs (64) or E4M3 quads (32)
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
            uint32_t gv[32], uv[32];
            tmem_ld_32x32(trow + c, gv);
            tmem_ld_32x32(trow + 128 + c, uv);
            tmem_ld_wait();
            float hv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) hv[i] = swiglu_f32(__uint_as_float(gv[i]), __uint_as_float(uv[i]));
            if (!MX) {
#pragma unroll
                for (int i = 0; i < 16; ++i) hq[c / 2 + i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
            } else {
                uint32_t q[8];
                sword |= mx_block32(hv, q) << (8 * (c >> 5));
#pragma unroll
                for (int i = 0; i < 8; ++i) hq[c / 4 + i] = q[i];
            }
        }
        release();
        const int64_t off = grow * F + f0;
        void *dst = valid ? (MX ? static_cast<void *>(static_cast<uint8_t *>(h) + off)
                                : static_cast<void *>(static_cast<uint16_t *>(h) + off))
                          : nullptr;
        store_rows_staged(hq, MX ? 32 : 64, dst, stage, lane);
        if (MX && valid) h_scales[scale_word_row(f0 >> 7, grow, h_rows)] = sword;
        return;
    }
    // training: a, b, h also stored (BF16); stores happen before the release.
    // BF16 layers stage the rows through shared memory so each store writes whole
    // row segments (Mixtral shape: forward 4.1 -> 4.0 ms); MXFP8 layers store
    // from registers, which measured faster there (3.84 vs 3.94 ms at T 8192)
    for (int c = 0; c < 128; c += 32) {
        uint32_t gv[32], uv[32];
        tmem_ld_32x32(trow + c, gv);
        tmem_ld_32x32(trow + 128 + c, uv);
        tmem_ld_wait();
        float hv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) hv[i] = swiglu_f32(__uint_as_float(gv[i]), __uint_as_float(uv[i]));
        const int64_t off = grow * F + f0 + c;
        if constexpr (MX) {
            if (valid) {
                if (saved_a) {
                    float t[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(gv[i]);
                    store_bf16x32(saved_a + off, t);
                }
                if (saved_b) {
                    float t[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(uv[i]);
                    store_bf16x32(saved_b + off, t);
                }
                if (saved_h) store_bf16x32(saved_h + off, hv);
                sword |= quant_mx32(hv, static_cast<uint8_t *>(h) + off) << (8 * (c >> 5));
            }
        } else {
            uint32_t pk[16];
            if (saved_a) {
                float t[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(gv[i]);
                pack_bf16x32(t, pk);
                store_rows_staged_n<16>(pk, valid ? saved_a + off : nullptr, stage, lane);
            }
            if (saved_b) {
                float t[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(uv[i]);
                pack_bf16x32(t, pk);
                store_rows_staged_n<16>(pk, valid ? saved_b + off : nullptr, stage, lane);
            }
            if (saved_h) {
                pack_bf16x32(hv, pk);
                store_rows_staged_n<16>(pk, valid ? saved_h + off : nullptr, stage, lane);
            }
            pack_bf16x32(hv, pk);
            store_rows_staged_n<16>(pk, valid ? static_cast<uint16_t *>(h) + off : nullptr, stage, lane);
        }
    }
    if (MX && valid) h_scales[scale_word_row(f0 >> 7, grow, h_rows)] = sword;
}

// Plain row epilogue: BN fp32 columns -> BF16 at dst (zeros when `zero`),
// TMEM released before the (staged, coalesced) stores.
template <typename Release>
__device__ __forceinline__ void epi_rows_bf16(uint32_t trow, int BN, bool zero, bool valid,
                                              uint16_t *dst, uint32_t *stage, int lane,
                                              Release &&release)
{
    uint32_t pk[128];
    drain_row_bf16(trow, BN, zero, pk);
    release();
    store_rows_staged(pk, BN / 2, valid ? dst : nullptr, stage, lane);
}

}  // namespace mok
