// mok_gather.cuh -- the pull of one token ([kucoin] = "Cursor's MoK achieves
// 2.37x performance boost on NVIDIA GB300 NVL72", kucoin.com, §02: the expert
// side pulls each token it needs by (source, position) and places it in its
// own expert order, with MXFP8 quantisation fused in): one warp reads token
// t's row from its source once, quantises it once (MXFP8) and writes it into
// each of the token's k slot rows of the expert-ordered buffer.  Shared by the
// by-token dispatch kernel (which the fused forward also runs first when its
// plan gathers every token before the GEMM role).
#pragma once

#include "mok_internal.h"
#include "mok_ptx.cuh"

namespace mok {

// Padded expert-ordered row of slot (t, j): pad_offsets[e] + slot_pos - offsets[e].
// xe: BF16 [rows, d] or E4M3 [rows, d]; xe_scales: tile layout for `rows` rows.
template <bool MX>
__device__ __forceinline__ void dispatch_token(const Sources &src, int64_t t, int d, int k,
                                               const int32_t *__restrict__ ids,
                                               const int32_t *__restrict__ slot_pos,
                                               const int32_t *__restrict__ offsets,
                                               const int32_t *__restrict__ pad_offsets, void *xe,
                                               uint32_t *__restrict__ xe_scales, int64_t rows, int lane)
{
    int64_t q[MOK_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOK_MAX_TOPK; ++j) {
        if (j < k) {
            const int e = ids[t * k + j];
            q[j] = pad_offsets[e] + (slot_pos[t * k + j] - offsets[e]);
        }
    }
    const uint4 *in = reinterpret_cast<const uint4 *>(source_row(src, static_cast<int>(t), d));
    // 16 vectors of 16 bytes per lane (8 KB per warp) in flight before any is stored; 8 when
    // quantising, whose registers also hold the block's codes
    if (!MX) {
        for (int c0 = 0; c0 < d / 8; c0 += 512) {
            uint4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int c = c0 + 32 * u + lane;
                v[u] = c < d / 8 ? __ldg(in + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < MOK_MAX_TOPK; ++j) {
                if (j < k) {
                    uint4 *out = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(xe) + q[j] * d);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int c = c0 + 32 * u + lane;
                        if (c < d / 8) out[c] = v[u];
                    }
                }
            }
        }
    } else {
        for (int c0 = 0; c0 < d; c0 += 2048) {
            uint4 raw[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int cu = c0 + 256 * u;
                const int nvalid = cu >= d ? 0 : (d - cu >= 256 ? 32 : 16);
                raw[u] = lane < nvalid ? __ldg(in + (cu >> 3) + lane) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int cu = c0 + 256 * u;
                if (cu >= d) continue;
                const int nvalid = d - cu >= 256 ? 32 : 16;
                uint2 codes;
                uint32_t word;
                mx_quant8(raw[u], lane, codes, word);
#pragma unroll
                for (int j = 0; j < MOK_MAX_TOPK; ++j) {
                    if (j < k) {
                        uint8_t *row = static_cast<uint8_t *>(xe) + q[j] * d;
                        if (lane < nvalid) *reinterpret_cast<uint2 *>(row + cu + 8 * lane) = codes;
                        if ((lane & 15) == 0 && lane < nvalid)
                            xe_scales[mx_word_index((cu + 8 * lane) >> 7, q[j], rows)] = word;
                    }
                }
            }
        }
    }
}

}  // namespace mok
