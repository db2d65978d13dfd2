// dsa_index_noalloc: dsa_index for callers that cannot allocate device memory.
//
// dsa_index needs a scratch workspace that the caller allocates.  Some
// callers cannot: plugin and custom-op hosts that pass the library only its
// input and output buffers and own every other byte of device memory,
// serving runtimes whose memory pools are sized once at start-up and refuse
// later requests, and latency-bound loops that must not call cudaMalloc
// because it can block until the device is idle.  For them this entry point
// runs the same indexer as dsa_index with its scratch in one fixed-size array
// that is part of the library's device code.  The pages describe no such
// call; it is an addition of this library.
//
// Limits: T <= 4096 tokens, n_docs <= 256 documents, H_i * d_i <= 4096.
// The array (about 26 MB) is reserved on every GPU where this file's device
// code is loaded and stays there until the process exits.
#include <cstdint>
#include <mutex>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {
namespace {

constexpr int NOALLOC_MAX_T = 4096;
constexpr int NOALLOC_MAX_DOCS = 256;
constexpr int NOALLOC_MAX_HD = 4096;      // H_i * d_i
constexpr int NOALLOC_MAX_HI = 64;
constexpr int NOALLOC_MAX_DI = 128;

constexpr size_t up256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t pairs_upto(size_t T) {   // sum over r < T of floor((r+1)/4)
    return 2 * (T / 4) * (T / 4 - 1) + (T / 4) * (T % 4 + 1);
}
// Upper bound of the dsa_index workspace for every size within the limits.
constexpr size_t NOALLOC_BYTES =
    up256((size_t)NOALLOC_MAX_T * NOALLOC_MAX_HD) + up256((size_t)NOALLOC_MAX_T * NOALLOC_MAX_HI * 4) +
    up256((size_t)NOALLOC_MAX_T / 4 * NOALLOC_MAX_DI) + up256((size_t)NOALLOC_MAX_T / 4 * 4) +
    up256((size_t)(NOALLOC_MAX_DOCS + 1) * 8) + up256((size_t)(NOALLOC_MAX_DOCS + 1) * 4) +
    up256(pairs_upto(NOALLOC_MAX_T) * 4);

}  // namespace
}  // namespace kpool

// The scratch itself.  In host code this name is only a stand-in for the
// device array: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_kpool_noalloc_scratch[kpool::NOALLOC_BYTES];

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_ptr[MAX_DEVICES] = {nullptr};

// Device address of the scratch on the current device, looked up once per
// device (the lookup loads this file's device code on that device) and kept
// for the process.  A reset of the device's context can move the array, so
// the kept address is valid only until such a reset.
int scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KPOOL_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kpool_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return KPOOL_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KPOOL_OK;
}
}  // namespace

extern "C" int dsa_index_noalloc(const void* q_idx, const float* w, const float* kpool, const kpool_layout* layout,
                                 int32_t topk, const kpool_params* p, int32_t* indices, int32_t W,
                                 kpool_stream_t stream) {
    using namespace kpool;
    if (!p || !layout) return KPOOL_ERR_INVALID_ARG;
    if (layout->T > NOALLOC_MAX_T || layout->n_docs > NOALLOC_MAX_DOCS ||
        (int64_t)p->n_idx_heads * p->d_idx > NOALLOC_MAX_HD || p->n_idx_heads > NOALLOC_MAX_HI ||
        p->d_idx > NOALLOC_MAX_DI)
        return KPOOL_ERR_SHAPE;
    if (layout->T >= 0 && layout->n_docs >= 1 && p->n_idx_heads >= 1 && p->d_idx >= 1 &&
        ws_layout(layout->T, layout->n_docs, layout->T / KPOOL, p->n_idx_heads, p->d_idx).total > NOALLOC_BYTES)
        return KPOOL_ERR_SHAPE;
    void* scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != KPOOL_OK) return rc;
    return dsa_index(q_idx, w, kpool, layout, topk, p, scratch, NOALLOC_BYTES, indices, W, stream);
}
