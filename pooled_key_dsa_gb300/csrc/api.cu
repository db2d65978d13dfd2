// C ABI of the KPool-DSA forward: argument checks, workspace geometry and the
// launch sequence of each call on the caller's stream.
#include <cstdint>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

// NVTX range around the host side of one call (the enqueue of its launches), named after the
// call, so that a timeline tool can group each call's kernels under it.  Without a tool attached
// a push/pop costs a few nanoseconds.
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

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

// The buffers and shapes of one dsa_index call, checked once; its stages run whole (dsa_index) or per
// block of query rows (the host-buffer forward).
struct IndexPlan {
    const void* q_idx;
    const float* w;
    const float* kpool;
    kpool_layout L;
    const kpool_params* p;
    int topk, W, T, qg;
    int32_t* indices;
    uint8_t* q8;
    float* ws;
    uint8_t* k8;
    float* s_k;
    int64_t* pair_base;
    int32_t* sched;
    float* scores;
};

static int index_plan(const void* q_idx, const float* w, const float* kpool, const kpool_layout* layout, int32_t topk,
                      const kpool_params* p, void* workspace, size_t workspace_bytes, int32_t* indices, int32_t W,
                      IndexPlan* out) {
    if (!params_ok(p) || !layout_ok(layout)) return KPOOL_ERR_INVALID_ARG;
    const int tk = topk > 0 ? topk : p->topk;
    const int T = layout->T;
    if (T > 0 && (!q_idx || !w || !kpool || !indices)) return KPOOL_ERR_INVALID_ARG;
    if ((int64_t)W < (int64_t)KPOOL * tk + KPOOL - 1 || W % 4 != 0) return KPOOL_ERR_SHAPE;
    if (!aligned(q_idx, 8) || !aligned(kpool, 16) || !aligned(indices, 16) || !aligned(workspace, 256))
        return KPOOL_ERR_ALIGN;
    const WsLayout wl = ws_layout(T, layout->n_docs, T / KPOOL, p->n_idx_heads, p->d_idx);
    if (!workspace || workspace_bytes < wl.total) return KPOOL_ERR_WORKSPACE;
    IndexPlan& P = *out;
    P.q_idx = q_idx;
    P.w = w;
    P.kpool = kpool;
    P.L = *layout;
    P.L.max_pools = T / KPOOL;     // every split of T tokens has at most floor(T/4) pools
    P.p = p;
    P.topk = tk;
    P.W = W;
    P.T = T;
    P.qg = scoring_group(p->n_idx_heads, p->d_idx);
    P.indices = indices;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    P.q8 = base + wl.q8;
    P.ws = reinterpret_cast<float*>(base + wl.ws);
    P.k8 = base + wl.k8;
    P.s_k = reinterpret_cast<float*>(base + wl.s_k);
    P.pair_base = reinterpret_cast<int64_t*>(base + wl.pair_base);
    P.sched = reinterpret_cast<int32_t*>(base + wl.sched);
    P.scores = reinterpret_cast<float*>(base + wl.scores);
    return KPOOL_OK;
}

// Per-document score bases and work schedule, and the pooled keys' Hadamard/FP8.
static int index_setup(const IndexPlan& P, cudaStream_t s) {
    int rc = launch_index_prep(P.L, P.topk, P.qg, P.pair_base, P.sched, s);
    if (rc != KPOOL_OK) return rc;
    return launch_hadamard_fp8(P.kpool, false, P.L.max_pools, P.p->d_idx, P.L.cu_pools + P.L.n_docs, nullptr, P.k8,
                               P.s_k, nullptr, s);
}

// Query rows r0 .. r1-1: Hadamard/FP8 of their queries and head weights.
static int index_queries(const IndexPlan& P, int r0, int r1, cudaStream_t s) {
    const int64_t hv = (int64_t)P.p->n_idx_heads, e = hv * P.p->d_idx;
    return launch_hadamard_fp8(static_cast<const uint16_t*>(P.q_idx) + r0 * e, true, (int64_t)(r1 - r0) * hv,
                               P.p->d_idx, nullptr, P.w + r0 * hv, P.q8 + r0 * e, nullptr, P.ws + r0 * hv, s);
}

// Work items of the tcgen05 scoring schedule whose first query row lies below row R: documents in order,
// each with the groups of qg queries from the group holding r = 4*topk + 3 (the numbering of the schedule
// kernel), counted on the host from the host copy of cu_seqlens.
static int items_before(const int32_t* cu, int n_docs, int topk, int qg, int R) {
    int64_t acc = 0;
    const int q0 = (KPOOL * topk + KPOOL - 1) / qg;
    for (int d = 0; d < n_docs; ++d) {
        const int s = cu[d], L = cu[d + 1] - cu[d];
        if (R <= s) break;
        const int q_all = (L + qg - 1) / qg;
        const int n_d = q_all > q0 ? q_all - q0 : 0;
        if (R >= s + L) {
            acc += n_d;
            continue;
        }
        const int c = (R - s + qg - 1) / qg - q0;     // groups (q0 + k) * qg < R - s
        acc += c < 0 ? 0 : (c > n_d ? n_d : c);
        break;
    }
    return (int)acc;
}

// Row R moved down to the start of its document's query group (groups of qg rows from each document's start).
static int group_floor(const int32_t* cu, int n_docs, int qg, int R) {
    for (int d = 0; d < n_docs; ++d)
        if (R < cu[d + 1]) return cu[d] + (R - cu[d]) / qg * qg;
    return R;
}

// A host copy of cu_seqlens fit for planning row blocks: starts at 0, never decreases, ends at T.
static bool host_cu_ok(const int32_t* cu, int n_docs, int T) {
    if (!cu || cu[0] != 0 || cu[n_docs] != T) return false;
    for (int d = 0; d < n_docs; ++d)
        if (cu[d + 1] < cu[d]) return false;
    return true;
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
    const Range range("kpool_build");
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
    const Range range("dsa_index");
    IndexPlan P;
    int rc = index_plan(q_idx, w, kpool, layout, topk, p, workspace, workspace_bytes, indices, W, &P);
    if (rc != KPOOL_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = stage_mark(0, s)) != KPOOL_OK) return rc;
    if ((rc = index_setup(P, s)) != KPOOL_OK) return rc;
    if ((rc = index_queries(P, 0, P.T, s)) != KPOOL_OK) return rc;
    if ((rc = stage_mark(1, s)) != KPOOL_OK) return rc;
    if ((rc = launch_score(P.q8, P.ws, P.k8, P.s_k, P.L, P.pair_base, P.sched, P.topk, p->n_idx_heads, p->d_idx,
                           P.scores, s)) != KPOOL_OK)
        return rc;
    if ((rc = stage_mark(2, s)) != KPOOL_OK) return rc;
    if ((rc = launch_select(P.scores, P.pair_base, P.L, P.topk, P.indices, P.W, s)) != KPOOL_OK) return rc;
    return stage_mark(3, s);
}

int sparse_mla_fwd_rows(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W, int32_t n_rows,
                        int32_t T, int32_t n_heads, float scale, void* out, float* lse, int32_t* status,
                        kpool_stream_t stream) {
    const Range range("sparse_mla_fwd");
    if (n_rows < 0 || T < 0 || W < 1 || n_heads < 1 || n_heads > 64) return KPOOL_ERR_SHAPE;
    if (n_rows > 0 && (!q_lat || !kv_lat || !indices || !out || !lse)) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(q_lat, 16) || !aligned(kv_lat, 16) || !aligned(out, 16) || !aligned(indices, 4))
        return KPOOL_ERR_ALIGN;
    if (!(scale == scale)) return KPOOL_ERR_INVALID_ARG;
    return launch_sparse_mla(static_cast<const uint16_t*>(q_lat), static_cast<const uint16_t*>(kv_lat), indices, W,
                             n_rows, T, n_heads, scale, static_cast<uint16_t*>(out), lse, status,
                             reinterpret_cast<cudaStream_t>(stream));
}

int sparse_mla_fwd(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W, int32_t T,
                   int32_t n_heads, float scale, void* out, float* lse, int32_t* status, kpool_stream_t stream) {
    return sparse_mla_fwd_rows(q_lat, kv_lat, indices, W, T, T, n_heads, scale, out, lse, status, stream);
}

int sparse_mla_bwd(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W, int32_t T,
                   int32_t n_heads, float scale, const void* out, const float* lse, const void* dout, void* dq,
                   float* dkv, float* delta, int32_t* status, kpool_stream_t stream) {
    const Range range("sparse_mla_bwd");
    if (T < 0 || W < 1 || n_heads < 1 || n_heads > 64) return KPOOL_ERR_SHAPE;
    if (T > 0 && (!q_lat || !kv_lat || !indices || !out || !lse || !dout || !dq || !dkv || !delta))
        return KPOOL_ERR_INVALID_ARG;
    if (!aligned(q_lat, 16) || !aligned(kv_lat, 16) || !aligned(out, 16) || !aligned(dout, 16) || !aligned(dq, 16) ||
        !aligned(dkv, 16) || !aligned(indices, 4) || !aligned(lse, 4) || !aligned(delta, 4))
        return KPOOL_ERR_ALIGN;
    if (!(scale == scale)) return KPOOL_ERR_INVALID_ARG;
    if (T == 0) return KPOOL_OK;
    return launch_sparse_mla_bwd(static_cast<const uint16_t*>(q_lat), static_cast<const uint16_t*>(kv_lat), indices,
                                 W, T, T, n_heads, scale, static_cast<const uint16_t*>(out), lse,
                                 static_cast<const uint16_t*>(dout), static_cast<uint16_t*>(dq), dkv, delta, status,
                                 reinterpret_cast<cudaStream_t>(stream));
}

int kpool_cast_e4m3(const float* x, int64_t n, uint8_t* codes, kpool_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !codes))) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(x, 4)) return KPOOL_ERR_ALIGN;
    return launch_cast_e4m3(x, n, codes, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_debug_inject_stall(int32_t mask) {
    if (mask & ~(KPOOL_STALL_SCORE | KPOOL_STALL_SPARSE_MLA)) return KPOOL_ERR_INVALID_ARG;
    int rc = set_score_tc_stall(mask & KPOOL_STALL_SCORE);
    if (rc == KPOOL_OK) rc = set_sparse_mla_stall(mask & KPOOL_STALL_SPARSE_MLA);
    return rc;
}

int kpool_measure_l2_reduce(float* buf, int32_t rows, const int32_t* row_ids, int32_t n_ids,
                            kpool_stream_t stream) {
    if (rows < 0 || n_ids < 0) return KPOOL_ERR_SHAPE;
    if (n_ids > 0 && (!buf || !row_ids)) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(buf, 16) || !aligned(row_ids, 4)) return KPOOL_ERR_ALIGN;
    return launch_l2_reduce(buf, rows, row_ids, n_ids, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- paged decode

namespace {
struct DecodeWs {
    size_t q8, ws, scores, total;
};
DecodeWs decode_ws(int B, int n_idx_heads, int d_idx, int max_pages) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    DecodeWs w;
    w.q8 = 0;
    w.ws = up((size_t)B * n_idx_heads * d_idx);
    w.scores = w.ws + up((size_t)B * n_idx_heads * 4);
    w.total = w.scores + up((size_t)B * max_pages * 32 * 4);
    return w;
}
bool decode_shape_ok(const kpool_params* p) {
    return p && p->kpool == KPOOL && p->d_idx == 128 && (p->n_idx_heads == 16 || p->n_idx_heads == 32);
}
}  // namespace

size_t dsa_decode_workspace_bytes(const kpool_params* p, int32_t B, int32_t max_pages) {
    if (!decode_shape_ok(p) || B < 0 || max_pages < 0) return 0;
    return decode_ws(B, p->n_idx_heads, p->d_idx, max_pages).total;
}

int kpool_paged_append(const void* k, const float* gate, const float* ape, const int32_t* pool_tok,
                       const int32_t* pool_seq, const int32_t* pool_idx, int32_t n_items, const int32_t* block_table,
                       int32_t max_pages, int32_t n_pages, const kpool_params* p, uint8_t* k8_cache, float* sk_cache,
                       int32_t* status, kpool_stream_t stream) {
    const Range range("kpool_paged_append");
    if (!decode_shape_ok(p)) return p ? KPOOL_ERR_SHAPE : KPOOL_ERR_INVALID_ARG;
    if (n_items < 0 || max_pages < 1 || n_pages < 1) return KPOOL_ERR_SHAPE;
    if (n_items == 0) return KPOOL_OK;
    if (!k || !gate || !ape || !pool_tok || !pool_seq || !pool_idx || !block_table || !k8_cache || !sk_cache)
        return KPOOL_ERR_INVALID_ARG;
    if (!aligned(k, 8) || !aligned(gate, 16) || !aligned(ape, 16) || !aligned(k8_cache, 16) || !aligned(sk_cache, 4))
        return KPOOL_ERR_ALIGN;
    return launch_paged_append(k, gate, ape, pool_tok, pool_seq, pool_idx, n_items, block_table, max_pages, n_pages,
                               k8_cache, sk_cache, status, reinterpret_cast<cudaStream_t>(stream));
}

int dsa_decode_index(const void* q_idx, const float* w, const uint8_t* k8_cache, const float* sk_cache,
                     int32_t n_pages, const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                     int32_t B, int32_t topk, const kpool_params* p, void* workspace, size_t workspace_bytes,
                     int32_t* indices, int32_t W, int32_t* status, kpool_stream_t stream) {
    const Range range("dsa_decode_index");
    if (!p) return KPOOL_ERR_INVALID_ARG;
    if (!decode_shape_ok(p)) return KPOOL_ERR_SHAPE;
    if (B < 0 || max_pages < 1 || n_pages < 1 || topk < 1 || W < KPOOL * topk + KPOOL - 1 || (W & 3) != 0)
        return KPOOL_ERR_SHAPE;
    if (B == 0) return KPOOL_OK;
    if (!workspace) return KPOOL_ERR_WORKSPACE;
    if (!q_idx || !w || !k8_cache || !sk_cache || !block_table || !seq_lens || !indices) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(q_idx, 8) || !aligned(k8_cache, 16) || !aligned(workspace, 256) || !aligned(indices, 16))
        return KPOOL_ERR_ALIGN;
    const DecodeWs o = decode_ws(B, p->n_idx_heads, p->d_idx, max_pages);
    if (workspace_bytes < o.total) return KPOOL_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* q8 = base + o.q8;
    float* ws = reinterpret_cast<float*>(base + o.ws);
    float* scores = reinterpret_cast<float*>(base + o.scores);
    int rc = launch_hadamard_fp8(q_idx, true, (int64_t)B * p->n_idx_heads, p->d_idx, nullptr, w, q8, nullptr, ws, st);
    if (rc == KPOOL_OK)
        rc = launch_decode_score(q8, ws, k8_cache, sk_cache, n_pages, block_table, max_pages, seq_lens, B,
                                 p->n_idx_heads, scores, (int64_t)max_pages * 32, status, st);
    if (rc == KPOOL_OK)
        rc = launch_decode_select(scores, (int64_t)max_pages * 32, seq_lens, block_table, max_pages, B, topk, indices,
                                  W, st);
    return rc;
}

int mla_absorb_q(const void* q_nope, const void* w_kv_b, int32_t T, int32_t n_heads, int32_t d_nope, int32_t d_v,
                 void* q_lat, int32_t* status, kpool_stream_t stream) {
    const Range range("mla_absorb_q");
    if (T < 0 || !mla_proj_shape_ok(n_heads, d_nope, d_v)) return KPOOL_ERR_SHAPE;
    if (T > 0 && (!q_nope || !w_kv_b || !q_lat)) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(q_nope, 16) || !aligned(w_kv_b, 16) || !aligned(q_lat, 16)) return KPOOL_ERR_ALIGN;
    return launch_mla_proj(true, q_nope, w_kv_b, T, n_heads, d_nope, d_v, q_lat, status,
                           reinterpret_cast<cudaStream_t>(stream));
}

int mla_v_proj(const void* o_lat, const void* w_kv_b, int32_t T, int32_t n_heads, int32_t d_nope, int32_t d_v,
               void* o_v, int32_t* status, kpool_stream_t stream) {
    const Range range("mla_v_proj");
    if (T < 0 || !mla_proj_shape_ok(n_heads, d_nope, d_v)) return KPOOL_ERR_SHAPE;
    if (T > 0 && (!o_lat || !w_kv_b || !o_v)) return KPOOL_ERR_INVALID_ARG;
    if (!aligned(o_lat, 16) || !aligned(w_kv_b, 16) || !aligned(o_v, 16)) return KPOOL_ERR_ALIGN;
    return launch_mla_proj(false, o_lat, w_kv_b, T, n_heads, d_nope, d_v, o_v, status,
                           reinterpret_cast<cudaStream_t>(stream));
}

int kpool_forward_host(const kpool_host_io* h, const kpool_dev_io* d, int32_t n_docs, int32_t T,
                       const kpool_params* p, int32_t n_chunks, kpool_stream_t s_in, kpool_stream_t s_compute,
                       kpool_stream_t s_out) {
    const Range range("kpool_forward_host");
    if (!h || !d || !p || !d->layout) return KPOOL_ERR_INVALID_ARG;
    if (T < 1 || n_docs < 1 || n_chunks < 1 || n_chunks > KPOOL_MAX_CHUNKS) return KPOOL_ERR_SHAPE;
    if (!h->k || !h->gate || !h->ape || !h->cu_seqlens || !h->q_idx || !h->w || !h->q_lat || !h->kv_lat ||
        !h->out || !h->lse)
        return KPOOL_ERR_INVALID_ARG;
    if (!d->k || !d->gate || !d->ape || !d->cu_seqlens || !d->q_idx || !d->w || !d->q_lat || !d->kv_lat ||
        !d->out || !d->lse || !d->kpool || !d->workspace || !d->indices)
        return KPOOL_ERR_INVALID_ARG;
    if (d->layout->cu_seqlens != d->cu_seqlens || d->layout->T != T || d->layout->n_docs != n_docs)
        return KPOOL_ERR_INVALID_ARG;
    if (p->d_lat != D_LAT || p->kpool != KPOOL || p->n_heads < 1 || p->n_heads > 64) return KPOOL_ERR_SHAPE;
    IndexPlan P;
    int rc = index_plan(d->q_idx, d->w, d->kpool, d->layout, p->topk, p, d->workspace, d->workspace_bytes,
                        d->indices, d->W, &P);
    if (rc != KPOOL_OK) return rc;
    cudaStream_t si = reinterpret_cast<cudaStream_t>(s_in), sc = reinterpret_cast<cudaStream_t>(s_compute),
                 so = reinterpret_cast<cudaStream_t>(s_out);
    const size_t q_row = (size_t)p->n_heads * D_LAT * 2;       // bytes of one q_lat / out row
    const size_t lse_row = (size_t)p->n_heads * 4;
    const size_t qi_row = (size_t)p->n_idx_heads * p->d_idx * 2;
    const size_t w_row = (size_t)p->n_idx_heads * 4;
    // Query-row blocks.  With the tcgen05 scorer and a well-formed host cu_seqlens, each block is indexed
    // on its own (its queries' Hadamard/FP8, scores, select) as soon as its q_idx rows have arrived, so
    // the first attention block and the first copy-out start early; block edges then fall on the
    // scorer's query groups, so no work item spans two blocks.  Otherwise the indexer runs over all
    // rows before the first attention block.
    const bool blocked = P.qg > 0 && host_cu_ok(h->cu_seqlens, n_docs, T);
    int32_t edge[KPOOL_MAX_CHUNKS + 1];
    const int32_t rows_per = (T + n_chunks - 1) / n_chunks;
    n_chunks = (T + rows_per - 1) / rows_per;
    edge[0] = 0;
    for (int c = 1; c < n_chunks; ++c)
        edge[c] = blocked ? group_floor(h->cu_seqlens, n_docs, P.qg, c * rows_per) : c * rows_per;
    edge[n_chunks] = T;

    cudaEvent_t ev[2 * KPOOL_MAX_CHUNKS + 2];
    const int n_ev = 2 * n_chunks + 2;
    int made = 0;
    for (; made < n_ev; ++made)
        if (cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming) != cudaSuccess) { rc = KPOOL_ERR_CUDA; break; }
    cudaEvent_t ev_in = ev[0], ev_out = ev[1];
    cudaEvent_t* ev_q = ev + 2;
    cudaEvent_t* ev_mla = ev + 2 + n_chunks;
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        if (rc == KPOOL_OK && bytes > 0 && cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, si) != cudaSuccess)
            rc = KPOOL_ERR_CUDA;
    };
    auto d2h = [&](void* dst, const void* src, size_t bytes) {
        if (rc == KPOOL_OK && bytes > 0 && cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, so) != cudaSuccess)
            rc = KPOOL_ERR_CUDA;
    };
    auto ok = [&](cudaError_t e) {
        if (rc == KPOOL_OK && e != cudaSuccess) rc = KPOOL_ERR_CUDA;
    };
    auto rows_of = [](void* base, size_t row, int32_t r0) { return static_cast<uint8_t*>(base) + r0 * row; };
    auto crows_of = [](const void* base, size_t row, int32_t r0) { return static_cast<const uint8_t*>(base) + r0 * row; };
    // copy-in stream: keys and what every block shares, then each block's query rows
    h2d(d->cu_seqlens, h->cu_seqlens, (size_t)(n_docs + 1) * 4);
    h2d(d->k, h->k, (size_t)T * p->d_idx * 2);
    h2d(d->gate, h->gate, (size_t)T * p->d_idx * 4);
    h2d(d->ape, h->ape, (size_t)KPOOL * p->d_idx * 4);
    h2d(d->kv_lat, h->kv_lat, (size_t)T * D_LAT * 2);
    h2d(d->w, h->w, (size_t)T * w_row);
    if (!blocked) h2d(d->q_idx, h->q_idx, (size_t)T * qi_row);
    if (rc == KPOOL_OK) ok(cudaEventRecord(ev_in, si));
    for (int c = 0; c < n_chunks && rc == KPOOL_OK; ++c) {
        const int32_t r0 = edge[c], n = edge[c + 1] - edge[c];
        if (blocked) h2d(rows_of(d->q_idx, qi_row, r0), crows_of(h->q_idx, qi_row, r0), (size_t)n * qi_row);
        h2d(rows_of(d->q_lat, q_row, r0), crows_of(h->q_lat, q_row, r0), (size_t)n * q_row);
        if (rc == KPOOL_OK) ok(cudaEventRecord(ev_q[c], si));
    }
    // compute stream: pooled keys and the index schedule, then block by block (index rows when blocked)
    // and attention
    if (rc == KPOOL_OK) ok(cudaStreamWaitEvent(sc, ev_in, 0));
    if (rc == KPOOL_OK)
        rc = kpool_build(d->k, d->gate, d->ape, d->cu_seqlens, n_docs, T, p, d->kpool, d->layout, s_compute);
    if (rc == KPOOL_OK) {
        if (blocked)
            rc = index_setup(P, sc);
        else
            rc = dsa_index(d->q_idx, d->w, d->kpool, d->layout, p->topk, p, d->workspace, d->workspace_bytes,
                           d->indices, d->W, s_compute);
    }
    for (int c = 0; c < n_chunks && rc == KPOOL_OK; ++c) {
        const int32_t r0 = edge[c], r1 = edge[c + 1], n = r1 - r0;
        ok(cudaStreamWaitEvent(sc, ev_q[c], 0));
        if (blocked && rc == KPOOL_OK && n > 0) {
            rc = index_queries(P, r0, r1, sc);
            if (rc == KPOOL_OK) {
                const int j0 = items_before(h->cu_seqlens, n_docs, P.topk, P.qg, r0);
                const int j1 = items_before(h->cu_seqlens, n_docs, P.topk, P.qg, r1);
                rc = launch_score(P.q8, P.ws, P.k8, P.s_k, P.L, P.pair_base, P.sched, P.topk, p->n_idx_heads,
                                  p->d_idx, P.scores, sc, j0, j1);
            }
            if (rc == KPOOL_OK) rc = launch_select(P.scores, P.pair_base, P.L, P.topk, P.indices, P.W, sc, r0, r1);
        }
        if (rc == KPOOL_OK && n > 0)
            rc = sparse_mla_fwd_rows(crows_of(d->q_lat, q_row, r0), d->kv_lat, d->indices + (size_t)r0 * d->W, d->W,
                                     n, T, p->n_heads, p->scale, rows_of(d->out, q_row, r0),
                                     d->lse + (size_t)r0 * p->n_heads, d->layout->status, s_compute);
        if (rc == KPOOL_OK) ok(cudaEventRecord(ev_mla[c], sc));
    }
    // copy-out stream: each block's results as soon as its attention is done
    for (int c = 0; c < n_chunks && rc == KPOOL_OK; ++c) {
        const int32_t r0 = edge[c], n = edge[c + 1] - edge[c];
        ok(cudaStreamWaitEvent(so, ev_mla[c], 0));
        d2h(rows_of(h->out, q_row, r0), crows_of(d->out, q_row, r0), (size_t)n * q_row);
        d2h(rows_of(h->lse, lse_row, r0), crows_of(d->lse, lse_row, r0), (size_t)n * lse_row);
    }
    // the compute stream ends after the last copy-out
    if (rc == KPOOL_OK) ok(cudaEventRecord(ev_out, so));
    if (rc == KPOOL_OK) ok(cudaStreamWaitEvent(sc, ev_out, 0));
    for (int k = 0; k < made; ++k) cudaEventDestroy(ev[k]);   // released once their work completes
    return rc;
}

int kpool_stage_select(const float* scores, const int64_t* pair_base, const kpool_layout* layout, int32_t topk,
                       int32_t* indices, int32_t W, kpool_stream_t stream) {
    if (!layout_ok(layout) || topk < 1 || !pair_base || (layout->T > 0 && (!scores || !indices)))
        return KPOOL_ERR_INVALID_ARG;
    if ((int64_t)W < (int64_t)KPOOL * topk + KPOOL - 1 || W % 4 != 0) return KPOOL_ERR_SHAPE;
    if (!aligned(indices, 16) || !aligned(pair_base, 8) || !aligned(scores, 16)) return KPOOL_ERR_ALIGN;
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
        case KPOOL_ERR_CHECK: return "internal bounds check failed";
        default: return "unknown error";
    }
}

// The tags after the arch name identify the kernel generations (used to match
// stored profiler counters to the code that produced them).
const char* kpool_version(void) { return "kpooldsa 0.18 sm_103a mla-tc12 score-tc3 select5 proj1 bwd4 decode2 pool2 hadamard3"; }

}  // extern "C"
