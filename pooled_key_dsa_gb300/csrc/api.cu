// C ABI of the KPool-DSA forward: argument checks, workspace geometry and the
// launch sequence of each call on the caller's stream.
#include <cstdint>
#include <cstring>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int T, int n_docs, int max_pools, int n_idx_heads, int d_idx) {
    WsLayout w{};
    size_t off = 0;
    w.q8 = off;        off = align256(off + (size_t)T * n_idx_heads * d_idx);
    w.ws = off;        off = align256(off + (size_t)T * n_idx_heads * sizeof(float));
    w.k8 = off;        off = align256(off + (size_t)max_pools * d_idx);
    w.s_k = off;       off = align256(off + (size_t)max_pools * sizeof(float));
    w.pair_base = off; off = align256(off + (size_t)(n_docs + 1) * sizeof(int64_t));
    w.sched = off;     off = align256(off + (size_t)(n_docs + 1) * sizeof(int32_t));
    w.scores = off;    off = align256(off + (size_t)pairs_before(T) * sizeof(float));
    w.total = off;
    return w;
}

static bool params_ok(const kpool_params* p) {
    return p && p->kpool == KPOOL && p->topk >= 1 && p->n_idx_heads >= 1 && p->n_idx_heads <= 64 &&
           (p->d_idx == 64 || p->d_idx == 128) && p->n_heads >= 1 && p->n_heads <= 64 && p->d_lat == D_LAT;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static cudaEvent_t g_stage_events[4];
static int g_n_stage_events = 0;

static int stage_mark(int k, cudaStream_t s) {
    if (k < g_n_stage_events && cudaEventRecord(g_stage_events[k], s) != cudaSuccess) {
        cudaGetLastError();
        return KPOOL_ERR_CUDA;
    }
    return KPOOL_OK;
}

static bool layout_ok(const kpool_layout* L) {
    return L && L->n_docs >= 1 && L->T >= 0 && L->max_pools >= L->T / KPOOL && L->cu_seqlens && L->cu_pools &&
           L->pool_tok_start && L->tok_doc && L->status;
}

}  // namespace kpool

using namespace kpool;

extern "C" {

size_t kpool_workspace_bytes(const kpool_params* p, int32_t T, int32_t n_docs) {
    if (!params_ok(p) || T < 0 || n_docs < 1) return 0;
    return ws_layout(T, n_docs, T / KPOOL, p->n_idx_heads, p->d_idx).total;
}

int kpool_workspace_offsets(const kpool_params* p, int32_t T, int32_t n_docs, kpool_ws_offsets* out) {
    if (!params_ok(p) || T < 0 || n_docs < 1 || !out) return KPOOL_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(T, n_docs, T / KPOOL, p->n_idx_heads, p->d_idx);
    out->q8 = w.q8;
    out->ws = w.ws;
    out->k8 = w.k8;
    out->s_k = w.s_k;
    out->pair_base = w.pair_base;
    out->sched = w.sched;
    out->scores = w.scores;
    out->total = w.total;
    return KPOOL_OK;
}

int kpool_build(const void* k, const float* gate, const float* ape, const int32_t* cu_seqlens, int32_t n_docs,
                int32_t T, const kpool_params* p, float* kpool_out, kpool_layout* layout, kpool_stream_t stream) {
    if (!params_ok(p)) return KPOOL_ERR_INVALID_ARG;
    if (!layout_ok(layout) || layout->n_docs != n_docs || layout->T != T || layout->cu_seqlens != cu_seqlens)
        return KPOOL_ERR_INVALID_ARG;
    if (!cu_seqlens || !ape || !kpool_out || (T > 0 && (!k || !gate))) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(k, 8) || !aligned(gate, 16) || !aligned(ape, 16) || !aligned(kpool_out, 16))
        return KPOOL_ERR_ALIGN;
    return launch_kpool_build(k, gate, ape, *layout, p->d_idx, kpool_out, reinterpret_cast<cudaStream_t>(stream));
}

int dsa_index(const void* q_idx, const float* w, const float* kpool, const kpool_layout* layout, int32_t topk,
              const kpool_params* p, void* workspace, size_t workspace_bytes, int32_t* indices, int32_t W,
              kpool_stream_t stream) {
    if (!params_ok(p) || !layout_ok(layout)) return KPOOL_ERR_INVALID_ARG;
    const int tk = topk > 0 ? topk : p->topk;
    const int T = layout->T;
    if (T > 0 && (!q_idx || !w || !kpool || !indices)) return KPOOL_ERR_INVALID_ARG;
    if ((int64_t)W < (int64_t)KPOOL * tk + KPOOL - 1 || W % 4 != 0) return KPOOL_ERR_SHAPE;
    if (!aligned(q_idx, 8) || !aligned(kpool, 16) || !aligned(indices, 16) || !aligned(workspace, 256))
        return KPOOL_ERR_ALIGN;
    const WsLayout wl = ws_layout(T, layout->n_docs, T / KPOOL, p->n_idx_heads, p->d_idx);
    if (!workspace || workspace_bytes < wl.total) return KPOOL_ERR_WORKSPACE;
    kpool_layout L = *layout;
    L.max_pools = T / KPOOL;       // every split of T tokens has at most floor(T/4) pools
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* q8 = base + wl.q8;
    float* ws = reinterpret_cast<float*>(base + wl.ws);
    uint8_t* k8 = base + wl.k8;
    float* s_k = reinterpret_cast<float*>(base + wl.s_k);
    int64_t* pair_base = reinterpret_cast<int64_t*>(base + wl.pair_base);
    int32_t* sched = reinterpret_cast<int32_t*>(base + wl.sched);
    float* scores = reinterpret_cast<float*>(base + wl.scores);
    int rc;
    if ((rc = stage_mark(0, s)) != KPOOL_OK) return rc;
    if ((rc = launch_index_prep(L, tk, scoring_group(p->n_idx_heads, p->d_idx), pair_base, sched, s)) != KPOOL_OK)
        return rc;
    if ((rc = launch_hadamard_fp8(q_idx, true, (int64_t)T * p->n_idx_heads, p->d_idx, nullptr, w, q8, nullptr, ws,
                                  s)) != KPOOL_OK)
        return rc;
    if ((rc = launch_hadamard_fp8(kpool, false, L.max_pools, p->d_idx, L.cu_pools + L.n_docs, nullptr, k8, s_k,
                                  nullptr, s)) != KPOOL_OK)
        return rc;
    if ((rc = stage_mark(1, s)) != KPOOL_OK) return rc;
    if ((rc = launch_score(q8, ws, k8, s_k, L, pair_base, sched, tk, p->n_idx_heads, p->d_idx, scores, s)) !=
        KPOOL_OK)
        return rc;
    if ((rc = stage_mark(2, s)) != KPOOL_OK) return rc;
    if ((rc = launch_select(scores, pair_base, L, tk, indices, W, s)) != KPOOL_OK) return rc;
    return stage_mark(3, s);
}

int sparse_mla_fwd(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W, int32_t T,
                   int32_t n_heads, float scale, void* out, float* lse, int32_t* status, kpool_stream_t stream) {
    if (T < 0 || W < 1 || n_heads < 1 || n_heads > 64) return KPOOL_ERR_SHAPE;
    if (T > 0 && (!q_lat || !kv_lat || !indices || !out || !lse)) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(q_lat, 16) || !aligned(kv_lat, 16) || !aligned(out, 16) || !aligned(indices, 4))
        return KPOOL_ERR_ALIGN;
    if (!(scale == scale)) return KPOOL_ERR_INVALID_ARG;
    return launch_sparse_mla(static_cast<const uint16_t*>(q_lat), static_cast<const uint16_t*>(kv_lat), indices, W, T,
                             n_heads, scale, static_cast<uint16_t*>(out), lse, status,
                             reinterpret_cast<cudaStream_t>(stream));
}

int kpool_stage_select(const float* scores, const int64_t* pair_base, const kpool_layout* layout, int32_t topk,
                       int32_t* indices, int32_t W, kpool_stream_t stream) {
    if (!layout_ok(layout) || topk < 1 || !pair_base || (layout->T > 0 && (!scores || !indices)))
        return KPOOL_ERR_INVALID_ARG;
    if ((int64_t)W < (int64_t)KPOOL * topk + KPOOL - 1 || W % 4 != 0) return KPOOL_ERR_SHAPE;
    if (!aligned(indices, 16) || !aligned(pair_base, 8)) return KPOOL_ERR_ALIGN;
    return launch_select(scores, pair_base, *layout, topk, indices, W, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_set_stage_events(kpool_event_t* events, int32_t n) {
    if (n < 0 || n > 4 || (n > 0 && !events)) return KPOOL_ERR_INVALID_ARG;
    for (int k = 0; k < n; ++k) g_stage_events[k] = reinterpret_cast<cudaEvent_t>(events[k]);
    g_n_stage_events = n;
    return KPOOL_OK;
}

int kpool_check_status(const int32_t* status, kpool_stream_t stream) {
    if (!status) return KPOOL_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return KPOOL_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KPOOL_ERR_CUDA;
    return v;
}

const char* kpool_strerror(int code) {
    switch (code) {
        case KPOOL_OK: return "ok";
        case KPOOL_ERR_INVALID_ARG: return "invalid argument";
        case KPOOL_ERR_SHAPE: return "unsupported shape";
        case KPOOL_ERR_ALIGN: return "misaligned pointer";
        case KPOOL_ERR_LAYOUT: return "invalid cu_seqlens";
        case KPOOL_ERR_INDEX_RANGE: return "index out of range";
        case KPOOL_ERR_TIMEOUT: return "device wait timed out";
        case KPOOL_ERR_CUDA: return "CUDA error";
        case KPOOL_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown error";
    }
}

// The tags after the arch name identify the kernel generations (used to match
// stored profiler counters to the code that produced them).
const char* kpool_version(void) { return "kpooldsa 0.2 sm_103a mla-tc4 score-tc1 select1"; }

}  // extern "C"
