// mok_noalloc.cu -- mok_layout_static: the layout step (per-expert counts,
// offsets, padded offsets, slot positions) for callers that cannot allocate
// device memory.
//
// The regular layout kernels keep two per-chunk tables (chunk histograms and
// chunk bases) in the caller's workspace.  Here those tables live in one
// fixed array owned by the library, so the caller passes only the routing
// ids and the output buffers.  The array is sized for kStaticLayoutWords
// 32-bit words (1 MiB): a layer fits when 2 * ceil(T*k / 256) * E <= 262144.
// Every GPU that loads the library holds that 1 MiB until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "mok.h"
#include "mok_internal.h"

namespace mok {

namespace {

constexpr int64_t kStaticLayoutWords = 262144;

// File-scope scratch.  In host code this name is only a stand-in for the
// symbol, never a device address: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_layout_scratch[kStaticLayoutWords];

constexpr int kMaxDevices = 64;
int32_t *g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
int scratch_for_current_device(int32_t **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOK_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || !p) return MOK_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOK_OK;
}

}  // namespace

}  // namespace mok

using namespace mok;

extern "C" int mok_layout_static(const mok_config *cfg, const int32_t *ids, int32_t *counts,
                                 int32_t *offsets, int32_t *pad_offsets, int32_t *slot_pos,
                                 int32_t *row_tok, uint8_t *row_j, void *stream)
{
    Dims dm;
    const int rc = check_config(cfg, &dm);
    if (rc != MOK_OK) return rc;
    if (dm.T == 0) return empty_layout(dm, counts, offsets, pad_offsets, static_cast<cudaStream_t>(stream));
    if (!ids || !counts || !offsets || !pad_offsets || !slot_pos || !row_tok || !row_j)
        return MOK_ERR_INVALID_ARG;
    const int64_t words = 2 * static_cast<int64_t>(dm.nchunks) * dm.E;
    if (words > kStaticLayoutWords) return MOK_ERR_UNSUPPORTED;
    int32_t *scratch = nullptr;
    const int src = scratch_for_current_device(&scratch);
    if (src != MOK_OK) return src;
    int32_t *chunk_counts = scratch;
    int32_t *chunk_base = scratch + static_cast<int64_t>(dm.nchunks) * dm.E;
    const cudaError_t e = launch_layout(dm, ids, counts, offsets, pad_offsets, slot_pos, row_tok,
                                        row_j, chunk_counts, chunk_base,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOK_OK : MOK_ERR_CUDA;
}
