/*
 * kpooldsa.h -- C ABI of the KPool-DSA forward on one GB300 (sm_103a).
 *
 * The forward of a GLM-5.3-Flash pooled-key DeepSeek-Sparse-Attention layer
 * in three calls, each asynchronous on the caller's CUDA stream:
 *
 *   kpool_build     indexer keys -> per-document pooled keys + PoolLayout
 *   dsa_index       Hadamard + FP8 queries and pooled keys, FP8 pool scores,
 *                   top-k pools per query, padded int32 index rows
 *   sparse_mla_fwd  NoPE sparse latent attention over the index rows
 *
 * Sources (page title, section):
 *   prime-rl PR "GLM-5.3-Flash text model", Summary: the k-pool indexer
 *     (pools of 4 per document from the first token, per-channel
 *     softmax(gate+ape)-weighted mean, Hadamard rotation in an fp32
 *     butterfly, FP8 scoring, complete pools ending at or before the query,
 *     top 512, own incomplete pool, rows padded to a multiple of 128,
 *     PoolLayout built once per forward).
 *   NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog and
 *     "cuDNN sparse MLA parity and performance": K absorbed into the query,
 *     attention over a shared 512-wide latent K/V, 64 heads,
 *     index_topk=2048, index_kpool=4, 2051 raw sparse slots.
 *   miles "GLM-5.3-Flash" recipe, section 1: NoPE MLA, kpool-compressed
 *     lightning indexer.
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented "device" are device pointers owned by
 *     the caller; the library allocates nothing and keeps no pointer after
 *     the call returns.
 *   - bf16 tensors are passed as `const void*` holding IEEE bfloat16.
 *   - All tensors are dense row-major (C order) with the shapes stated.
 *   - The return value is a kpool_status.  Host-side checks (null or
 *     misaligned pointers, unsupported sizes) return an error before any
 *     launch.  Checks that need device data (cu_seqlens, index values)
 *     record the first error in the caller's device status word, which
 *     kpool_check_status() reads; such a call still completes and leaves
 *     safe values (empty layouts, -1 rows, skipped slots) behind.
 *   - Every call only enqueues work; none synchronises the stream except
 *     kpool_check_status().
 */
#ifndef KPOOLDSA_H
#define KPOOLDSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* kpool_stream_t;

typedef enum {
    KPOOL_OK = 0,
    KPOOL_ERR_INVALID_ARG = 1,  /* null pointer, bad count, bad parameter   */
    KPOOL_ERR_SHAPE = 2,        /* size outside what the kernels support     */
    KPOOL_ERR_ALIGN = 3,        /* pointer not aligned as documented         */
    KPOOL_ERR_LAYOUT = 4,       /* cu_seqlens not 0 = c0 <= c1 <= ... = T    */
    KPOOL_ERR_INDEX_RANGE = 5,  /* index row entry outside [-1, T)           */
    KPOOL_ERR_TIMEOUT = 6,      /* a bounded device wait expired             */
    KPOOL_ERR_CUDA = 7,         /* a CUDA runtime call failed                */
    KPOOL_ERR_WORKSPACE = 8,    /* workspace null or too small               */
    KPOOL_ERR_CHECK = 9         /* internal bounds check failed (library
                                   built with KPOOL_CHECKED only)             */
} kpool_status;

/* Layer parameters.  kpool must be 4 (index_kpool); d_idx is 64 or 128;
 * n_idx_heads is 1..64; n_heads is 1..64; d_lat must be 512; topk >= 1. */
typedef struct {
    int32_t kpool;        /* tokens per pool (4)                          */
    int32_t topk;         /* pools kept per query (512 = 2048 positions)  */
    int32_t n_idx_heads;  /* H_i, indexer heads                           */
    int32_t d_idx;        /* d_i, indexer head width                      */
    int32_t n_heads;      /* H, attention heads                           */
    int32_t d_lat;        /* D, latent width (K and V)                    */
    float scale;          /* attention softmax scale (1/sqrt(512))        */
} kpool_params;

/* PoolLayout: per-document pool geometry of a packed (THD) row of T tokens
 * in n_docs documents.  All buffers are caller-allocated device memory,
 * filled by kpool_build and read by dsa_index.
 *   cu_seqlens     int32 [n_docs+1]  input: document starts, 0 .. T
 *   cu_pools       int32 [n_docs+1]  cu_pools[d+1] - cu_pools[d] = floor(L_d/4)
 *   pool_tok_start int32 [max_pools] first token of each pool (0 past the end)
 *   tok_doc        int32 [T]         document of each token (-1 if the layout
 *                                    is invalid)
 *   status         int32 [1]         device error word (0 = OK); the caller
 *                                    zeroes it before first use.
 * max_pools must be >= floor(T/4), which bounds the pool count of any split. */
typedef struct {
    int32_t n_docs;
    int32_t T;
    int32_t max_pools;
    const int32_t* cu_seqlens;
    int32_t* cu_pools;
    int32_t* pool_tok_start;
    int32_t* tok_doc;
    int32_t* status;
} kpool_layout;

/* Byte offsets of the intermediate tensors inside the dsa_index workspace
 * (all 256-byte aligned).  Reading them after dsa_index is allowed and is how
 * the intermediate values are inspected:
 *   q8        uint8 E4M3 [T, H_i, d_i]  rotated, quantised queries
 *   ws        fp32 [T, H_i]             w[i,h] * s_q[i,h]
 *   k8        uint8 E4M3 [floor(T/4), d_i]
 *   s_k       fp32 [floor(T/4)]         per-pool scale amax/448
 *   pair_base int64 [n_docs+1]          start of each document's scores
 *   sched     int32 [n_docs+1]          first scoring tile of each document
 *   scores    fp32, compact triangle:   query i of document d at in-document
 *             position r = i - cu_seqlens[d] has n = floor((r+1)/4) candidate
 *             pools; its scores start at pair_base[d] + G(r) with
 *             G(r) = 2a(a-1) + a(b+1), r = 4a + b, and are in pool order.
 *             Rows with n <= topk are not scored (every candidate is kept). */
typedef struct {
    size_t q8, ws, k8, s_k, pair_base, sched, scores, total;
} kpool_ws_offsets;

/* Workspace bytes dsa_index needs for T tokens in at most n_docs documents
 * (sized for the worst split: one document of T tokens).  Returns 0 on bad
 * parameters. */
size_t kpool_workspace_bytes(const kpool_params* p, int32_t T, int32_t n_docs);
int kpool_workspace_offsets(const kpool_params* p, int32_t T, int32_t n_docs, kpool_ws_offsets* out);

/* kpool_build: PoolLayout from cu_seqlens, then pooled indexer keys.
 *   k      bf16 [T, d_idx]   indexer keys              (8-byte aligned)
 *   gate   fp32 [T, d_idx]   pooling gate logits       (16-byte aligned)
 *   ape    fp32 [kpool, d_idx] per-offset bias, indexed by position in pool
 *   kpool_out fp32 [max_pools, d_idx]: row p = sum_j softmax_j(gate+ape) k,
 *             rows >= the pool count are zero.
 *   layout  filled in place; layout->cu_seqlens must equal cu_seqlens.
 * Source: prime-rl PR "GLM-5.3-Flash text model", Summary (k-pool
 * compression; PoolLayout built once per forward). */
int kpool_build(const void* k, const float* gate, const float* ape, const int32_t* cu_seqlens,
                int32_t n_docs, int32_t T, const kpool_params* p, float* kpool_out,
                kpool_layout* layout, kpool_stream_t stream);

/* dsa_index: the k-pool indexer after pooling.
 *   q_idx  bf16 [T, H_i, d_i] indexer queries           (8-byte aligned)
 *   w      fp32 [T, H_i]      per-query head weights
 *   kpool  fp32 [max_pools, d_i] from kpool_build (16-byte aligned)
 *   topk   pools kept per query (overrides p->topk when > 0)
 *   workspace  kpool_workspace_bytes(p, T, n_docs) bytes, 256-byte aligned
 *   indices    int32 [T, W]: for query i, the positions of its top-k pools
 *              (4 each) and of its own incomplete pool up to i, ascending,
 *              then -1.  W >= 4*topk + 3 and a multiple of 4 (2176 for topk
 *              512 keeps rows a multiple of 128); 16-byte aligned.
 * Score of query i for pool p: s_k[p] * sum_h w[i,h] s_q[i,h] ReLU(q8[i,h].k8[p]);
 * ties go to the lower pool index, -0 ranks as +0, and a NaN score ranks below
 * every number (-inf included).
 * Source: prime-rl PR "GLM-5.3-Flash text model", Summary. */
int dsa_index(const void* q_idx, const float* w, const float* kpool, const kpool_layout* layout,
              int32_t topk, const kpool_params* p, void* workspace, size_t workspace_bytes,
              int32_t* indices, int32_t W, kpool_stream_t stream);

/* sparse_mla_fwd: absorbed NoPE sparse latent attention.
 *   q_lat  bf16 [T, H, 512]  queries with K absorbed     (16-byte aligned)
 *   kv_lat bf16 [T, 512]     shared latent key = value   (16-byte aligned)
 *   indices int32 [T, W]     positions; -1 entries are skipped anywhere in
 *                            the row; entries outside [-1, T) are skipped and
 *                            flagged KPOOL_ERR_INDEX_RANGE in *status.
 *   out    bf16 [T, H, 512]  sum_j softmax_j(scale q.kv_j) kv_j (RNE to bf16);
 *                            16-byte aligned
 *   lse    fp32 [T, H]       ln sum_j exp(scale q.kv_j); -inf (and out = 0)
 *                            for a row with no valid slot.
 *   status int32 [1] device error word (may be NULL: errors then go unreported).
 * Source: NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog
 * (attention over the shared 512-wide latent, V projection applied after). */
int sparse_mla_fwd(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W,
                   int32_t T, int32_t n_heads, float scale, void* out, float* lse,
                   int32_t* status, kpool_stream_t stream);

/* sparse_mla_fwd_rows: sparse_mla_fwd over a block of n_rows query rows of a
 * longer sequence.  q_lat, indices, out and lse point at the block's first
 * row (shapes [n_rows, ...] as for sparse_mla_fwd); kv_lat is the whole
 * latent [T, 512] and index entries must lie in [-1, T).  Rows are
 * independent, so the blocks of a split give exactly the unsplit results.
 * sparse_mla_fwd is this call with n_rows = T. */
int sparse_mla_fwd_rows(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W,
                        int32_t n_rows, int32_t T, int32_t n_heads, float scale, void* out, float* lse,
                        int32_t* status, kpool_stream_t stream);

/* kpool_forward_host: the whole forward from host memory, with the copies
 * overlapped with the kernels.  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister); pageable buffers work but their copies
 * do not overlap.  Shapes are those of kpool_build, dsa_index and
 * sparse_mla_fwd.  No counterpart on the pages: a pipelined executor of this
 * library for callers whose inputs and outputs live on the host. */
typedef struct {
    const void* k;              /* bf16 [T, d_idx]            */
    const float* gate;          /* fp32 [T, d_idx]            */
    const float* ape;           /* fp32 [kpool, d_idx]        */
    const int32_t* cu_seqlens;  /* int32 [n_docs+1]           */
    const void* q_idx;          /* bf16 [T, H_i, d_i]         */
    const float* w;             /* fp32 [T, H_i]              */
    const void* q_lat;          /* bf16 [T, H, 512]           */
    const void* kv_lat;         /* bf16 [T, 512]              */
    void* out;                  /* bf16 [T, H, 512] (written) */
    float* lse;                 /* fp32 [T, H]      (written) */
} kpool_host_io;

/* Device buffers of one forward (caller-allocated, alignment as documented
 * for each call); layout->cu_seqlens must be cu_seqlens below and
 * layout->T / n_docs must match the call. */
typedef struct {
    void* k;
    float* gate;
    float* ape;
    int32_t* cu_seqlens;
    void* q_idx;
    float* w;
    void* q_lat;
    void* kv_lat;
    void* out;
    float* lse;
    float* kpool;               /* fp32 [max_pools, d_idx]    */
    kpool_layout* layout;
    void* workspace;            /* kpool_workspace_bytes(p, T, n_docs) */
    size_t workspace_bytes;
    int32_t* indices;           /* int32 [T, W]               */
    int32_t W;
} kpool_dev_io;

#define KPOOL_MAX_CHUNKS 64

/* Enqueues, for query rows cut into n_chunks (1..KPOOL_MAX_CHUNKS) blocks:
 *   s_in:      keys, gate, ape, kv_lat and w to the device, then each
 *              block's q_idx and q_lat rows;
 *   s_compute: kpool_build, then block by block, each after its rows have
 *              arrived: the block's index rows (Hadamard/FP8 of its queries,
 *              their scores, the select) and sparse_mla_fwd_rows;
 *   s_out:     out and lse of each block back to the host once its
 *              attention is done;
 * and makes s_compute wait for the last copy-out, so the forward is complete
 * when s_compute is.
 * Blocks are indexed one at a time when the tcgen05 scorer serves the shape
 * (d_idx = 128) and host->cu_seqlens starts at 0, never decreases and ends
 * at T. The host reads host->cu_seqlens to place each block edge on the start
 * of a scoring query group (256 / n_idx_heads rows from each document's
 * start), so blocks are near, not exactly, T / n_chunks rows. Otherwise the
 * whole dsa_index runs after all of q_idx has arrived, and blocks are
 * ceil(T / n_chunks) rows. Either way the results are those of kpool_build,
 * dsa_index and sparse_mla_fwd.
 * The three streams must be distinct, non-default streams for the copies to
 * overlap. Device errors go to layout->status. Host-side errors return before
 * or between enqueues (work already enqueued still runs). Creates and
 * releases 2*n_chunks+2 CUDA events. */
int kpool_forward_host(const kpool_host_io* host, const kpool_dev_io* dev, int32_t n_docs, int32_t T,
                       const kpool_params* p, int32_t n_chunks, kpool_stream_t s_in,
                       kpool_stream_t s_compute, kpool_stream_t s_out);

/* dsa_index_noalloc: dsa_index for callers that cannot allocate.
 * No counterpart on the pages: this call is an addition of this library.
 * dsa_index needs a caller-allocated workspace; callers that cannot allocate
 * device memory (custom-op hosts that hand over only input and output
 * buffers, runtimes with fixed memory pools, loops that must not call
 * cudaMalloc because it can block until the device is idle) use this entry
 * instead.  Arguments and results are those of dsa_index without the
 * workspace; the scratch is one static device array of 26,349,056 bytes held
 * by every GPU that loads it until the process exits.
 * Limits: layout->T <= 4096, layout->n_docs <= 256, n_idx_heads * d_idx <=
 * 4096; larger sizes return KPOOL_ERR_SHAPE before any launch.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the rest of the process; make that
 * first call before any stream capture begins.  The kept address does not
 * survive a teardown of the device's context (cudaDeviceReset): after one,
 * the array may sit elsewhere, so do not call this entry point on that
 * device again in the same process.  Every call uses the same array and leaves its contents behind
 * (each call writes every scratch byte it later reads, so nothing needs to
 * start at zero); calls that can overlap on the GPU (different streams, or
 * other threads) race on the array and must be serialised by the caller.
 * It calls no allocator (no cudaMalloc, cudaFree or library allocation). */
int dsa_index_noalloc(const void* q_idx, const float* w, const float* kpool, const kpool_layout* layout,
                      int32_t topk, const kpool_params* p, int32_t* indices, int32_t W, kpool_stream_t stream);

/* Stage entry point: top-k select + row expansion alone, fed with scores in
 * the workspace's compact layout (same rules as dsa_index's last step,
 * including the order of ties, signed zeros and NaN).
 *   scores   fp32, compact triangle as described for kpool_ws_offsets
 *            (16-byte aligned, as the workspace's scores are)
 *   pair_base int64 [n_docs+1] as described there (8-byte aligned) */
int kpool_stage_select(const float* scores, const int64_t* pair_base, const kpool_layout* layout,
                       int32_t topk, int32_t* indices, int32_t W, kpool_stream_t stream);

/* Stage timing hook.  With n = 4 events registered, every later dsa_index
 * call records events[0] before its first launch, events[1] after the
 * Hadamard/FP8 kernels, events[2] after the scoring kernel and events[3]
 * after the select kernel, all on its stream (cudaEventRecord only; nothing
 * synchronises).  events = NULL or n = 0 switches the hook off.  The events
 * are cudaEvent_t handles owned by the caller; the hook is process-wide and
 * not thread-safe. */
typedef struct CUevent_st* kpool_event_t;
int kpool_set_stage_events(kpool_event_t* events, int32_t n);

/* sparse_mla_bwd: gradients of sparse_mla_fwd.
 * NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog and
 * "cuDNN sparse MLA parity and performance": training runs the latent sparse
 * attention backward for dQ and dKV.  The latent row is both key and value,
 * so dkv sums a value term and a key term.  Per query i, head h, over the
 * valid slots j of row i (p the forward's softmax, rebuilt from lse):
 *   delta = dout[i,h] . out[i,h]
 *   dz_j  = p_j * (dout[i,h] . kv[j] - delta)
 *   dq[i,h]  = scale * sum_j dz_j kv[j]
 *   dkv[j]  += p_j dout[i,h] + scale * dz_j q[i,h]
 *   q_lat, kv_lat, indices, W, T, n_heads, scale: as for sparse_mla_fwd
 *   out     bf16 [T, n_heads, 512]  and  lse fp32 [T, n_heads]: the forward's
 *           results for these inputs
 *   dout    bf16 [T, n_heads, 512]  gradient of the loss w.r.t. out
 *   dq      bf16 [T, n_heads, 512]  written (rows with no valid slot: 0)
 *   dkv     fp32 [T, 512]           overwritten: zeroed by the call, then
 *           accumulated with fp32 atomic reductions, so the summation order
 *           (and the last bits) can differ between calls
 *   delta   fp32 [T, n_heads]       caller-allocated scratch, written
 * Alignment: q_lat, kv_lat, out, dout, dq, dkv 16 bytes; indices, lse, delta
 * 4 bytes.  Index entries outside [-1, T) are skipped and recorded as
 * KPOOL_ERR_INDEX_RANGE; KPOOL_ERR_TIMEOUT as for the forward. */
int sparse_mla_bwd(const void* q_lat, const void* kv_lat, const int32_t* indices, int32_t W, int32_t T,
                   int32_t n_heads, float scale, const void* out, const float* lse, const void* dout, void* dq,
                   float* dkv, float* delta, int32_t* status, kpool_stream_t stream);

/* ----------------------------------------------------------------------
 * Paged decode.  prime-rl PR "GLM-5.3-Flash text model", section "Patches
 * and workarounds": serving aligns hybrid KV blocks to index_kpool x 32 = 128
 * tokens, and the paged indexer kernel takes pages of 32 pools on SM100.  One
 * page id indexes three caches:
 *   k8_cache  e4m3 [n_pages, 32, d_i]   pooled-key codes (16-byte aligned)
 *   sk_cache  fp32 [n_pages, 32]        their per-vector scales
 *   kv_cache  bf16 [n_pages, 128, 512]  latent rows (read by sparse_mla_fwd_rows)
 *   block_table int32 [B, max_pages]: page of tokens 128j .. 128j+127 of sequence b
 * Sizes: d_i = 128, n_idx_heads 16 or 32, kpool 4 (else KPOOL_ERR_SHAPE).
 * Pooling, Hadamard, FP8, scoring, top-k and row rules are those of
 * kpool_build / dsa_index; a sequence is one document.
 * ---------------------------------------------------------------------- */

/* kpool_paged_append: pooled keys into the page cache.  For item v, the pool
 * of the 4 token rows pool_tok[v] .. pool_tok[v]+3 of k (bf16 [*, d_i]) and
 * gate (fp32 [*, d_i]) with ape (fp32 [4, d_i]) is Hadamard-rotated,
 * FP8-quantised and written to slot pool_idx[v] % 32 of page
 * block_table[pool_seq[v]][pool_idx[v] / 32].  Fills the cache from a prefill
 * (one item per pool) and appends the pool a decode step completes (sequences
 * whose new token makes seq_len % 4 == 0).  An item whose page is outside
 * [0, n_pages) is skipped and recorded as KPOOL_ERR_INDEX_RANGE. */
int kpool_paged_append(const void* k, const float* gate, const float* ape, const int32_t* pool_tok,
                       const int32_t* pool_seq, const int32_t* pool_idx, int32_t n_items,
                       const int32_t* block_table, int32_t max_pages, int32_t n_pages,
                       const kpool_params* p, uint8_t* k8_cache, float* sk_cache, int32_t* status,
                       kpool_stream_t stream);

/* Workspace bytes of dsa_decode_index (0 for an unsupported shape). */
size_t dsa_decode_workspace_bytes(const kpool_params* p, int32_t B, int32_t max_pages);

/* dsa_decode_index: index rows of one decode step.  The query of sequence b
 * is its newest token, at position r = seq_lens[b] - 1:
 *   q_idx bf16 [B, n_idx_heads, d_i], w fp32 [B, n_idx_heads]
 * It scores the seq_lens[b] / 4 complete pools of its pages, keeps the top
 * `topk` (higher score, then lower pool), adds its own incomplete pool, and
 * writes latent-cache slots (page * 128 + offset, i.e. rows of kv_cache seen
 * as [n_pages * 128, 512]) ascending in position, -1 padded:
 *   indices int32 [B, W], W a multiple of 4 and >= 4*topk + 3, 16-byte aligned.
 * The attention of the step is sparse_mla_fwd_rows(q_lat [B, H, 512],
 * kv_cache, indices, W, n_rows = B, T = n_pages * 128, ...).
 * workspace: >= dsa_decode_workspace_bytes(p, B, max_pages), 256-byte aligned.
 * A sequence longer than max_pages * 128 gets an all -1 row and
 * KPOOL_ERR_SHAPE in *status; a page id outside [0, n_pages) gives
 * KPOOL_ERR_INDEX_RANGE. */
int dsa_decode_index(const void* q_idx, const float* w, const uint8_t* k8_cache, const float* sk_cache,
                     int32_t n_pages, const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                     int32_t B, int32_t topk, const kpool_params* p, void* workspace, size_t workspace_bytes,
                     int32_t* indices, int32_t W, int32_t* status, kpool_stream_t stream);

/* kpool_measure_l2_reduce: measurement utility, no counterpart on the pages.
 * Adds 1.0f to each of the 512 floats of rows buf[row_ids[k]], k < n_ids,
 * with fp32 reductions in sparse_mla_bwd's dkv access pattern (each warp
 * instruction covers 128 contiguous bytes of one row), so that a caller can
 * time the reduction rate that bounds sparse_mla_bwd.
 *   buf      fp32 [rows, 512], device, 16-byte aligned
 *   row_ids  int32 [n_ids], device; ids outside [0, rows) are skipped */
int kpool_measure_l2_reduce(float* buf, int32_t rows, const int32_t* row_ids, int32_t n_ids,
                            kpool_stream_t stream);

/* kpool_debug_inject_stall: test utility, no counterpart on the pages.
 * Every wait of the tcgen05 kernels on an mbarrier is bounded: after about
 * two seconds it records KPOOL_ERR_TIMEOUT in the call's status word, every
 * warp role leaves its loop, copies and MMAs in flight are waited for and
 * TMEM is freed, so the context stays usable.  This hook makes that path run
 * on demand: with KPOOL_STALL_SCORE set, every later launch of the tcgen05
 * scoring kernel (dsa_index with d_idx = 128) first waits on a barrier that
 * nothing completes, in its TMA producer; with KPOOL_STALL_SPARSE_MLA, every
 * later sparse_mla_fwd / sparse_mla_fwd_rows launch does the same in its row
 * scanner (the barrier completes only after the kernel has aborted).  Such a launch takes about two seconds, ends with
 * KPOOL_ERR_TIMEOUT and leaves its outputs undefined.  mask = 0 restores
 * normal operation (the state at load).  The setting is per device (the
 * current one) and applies to launches enqueued after the call returns; it
 * synchronises with the device like cudaMemcpyToSymbol.
 * Returns KPOOL_ERR_INVALID_ARG for unknown bits, KPOOL_ERR_CUDA if the copy
 * fails. */
#define KPOOL_STALL_SCORE 1
#define KPOOL_STALL_SPARSE_MLA 2
int kpool_debug_inject_stall(int32_t mask);

/* kpool_cast_e4m3: test and diagnostic utility, no counterpart on the pages.
 * codes[k] = OCP E4M3 ("fn") code of x[k], k < n: round to nearest, ties to
 * even, magnitudes above 448 saturate to 448, the sign follows the input.
 * This is the conversion every FP8 quantiser of the library applies to its
 * scaled values (prime-rl PR "GLM-5.3-Flash text model", Summary: queries and
 * pooled keys are quantised to FP8), exposed so that it can be compared value
 * by value with an independent encoder.
 *   x      fp32 [n], device, 4-byte aligned
 *   codes  uint8 [n], device
 * Returns KPOOL_ERR_INVALID_ARG for null pointers with n > 0 or n < 0. */
int kpool_cast_e4m3(const float* x, int64_t n, uint8_t* codes, kpool_stream_t stream);

/* ----------------------------------------------------------------------
 * Absorbed-MLA projections either side of sparse_mla_fwd.
 * NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog: the K
 * projection is absorbed into the query, attention runs over the shared
 * 512-wide latent, and the model-owned V projection follows.  miles
 * "GLM-5.3-Flash" recipe, section 6 "LoRA RL": both use the kv_b_proj weight
 * directly instead of calling that module.
 *
 *   w_kv_b  bf16 [n_heads*(d_nope+d_v), 512], the kv_b_proj weight stored
 *           [out, in]: rows h*(d_nope+d_v) .. +d_nope-1 are head h's key
 *           rows W_UK[h], the next d_v rows its value rows W_UV[h]
 *   d_nope, d_v   64 or 128 each; n_heads 1..1024.  Other sizes return
 *           KPOOL_ERR_SHAPE before any launch.
 * Every pointer is a device pointer, 16-byte aligned (KPOOL_ERR_ALIGN).
 * Results are bf16 (round to nearest even) of fp32 sums of exact bf16
 * products.  T = 0 does nothing.  The only device error is KPOOL_ERR_TIMEOUT
 * (a bounded wait that expired), recorded in *status (which may be NULL).
 * ---------------------------------------------------------------------- */

/* mla_absorb_q: q_lat[t,h,:] = sum_n q_nope[t,h,n] * W_UK[h][n,:].
 *   q_nope  bf16 [T, n_heads, d_nope]   ->   q_lat  bf16 [T, n_heads, 512] */
int mla_absorb_q(const void* q_nope, const void* w_kv_b, int32_t T, int32_t n_heads, int32_t d_nope,
                 int32_t d_v, void* q_lat, int32_t* status, kpool_stream_t stream);

/* mla_v_proj: o_v[t,h,:] = W_UV[h] . o_lat[t,h,:] (sum over the 512 latent).
 *   o_lat   bf16 [T, n_heads, 512]      ->   o_v    bf16 [T, n_heads, d_v] */
int mla_v_proj(const void* o_lat, const void* w_kv_b, int32_t T, int32_t n_heads, int32_t d_nope,
               int32_t d_v, void* o_v, int32_t* status, kpool_stream_t stream);

/* Synchronises `stream`, then returns the device status word's value (a
 * kpool_status), or KPOOL_ERR_CUDA if the stream or copy failed. */
int kpool_check_status(const int32_t* status, kpool_stream_t stream);

/* Static, human-readable text of a kpool_status. */
const char* kpool_strerror(int code);

/* Library version string, e.g. "kpooldsa 0.1 sm_103a". */
const char* kpool_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KPOOLDSA_H */
