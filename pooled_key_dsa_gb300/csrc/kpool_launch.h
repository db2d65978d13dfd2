// Internal launch entry points behind the C ABI (one per kernel family).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kpooldsa.h"

namespace kpool {

// Workspace geometry shared by the host layer and the launchers.
struct WsLayout {
    size_t q8, ws, k8, s_k, pair_base, sched, scores, total;
};
WsLayout ws_layout(int T, int n_docs, int max_pools, int n_idx_heads, int d_idx);

int launch_kpool_build(const void* k, const float* gate, const float* ape, const kpool_layout& L, int d_idx,
                       float* kpool_out, cudaStream_t stream);

// Hadamard rotation + per-vector E4M3 quantisation of n_vec vectors of width d.
// in_bf16 selects the input type (bf16 queries or fp32 pooled keys).  If
// n_valid_dev is non-null, vectors at or past *n_valid_dev get zero codes and
// scale.  If w is non-null, ws_out[v] = w[v] * scale[v]; scales may be null.
int launch_cast_e4m3(const float* x, int64_t n, uint8_t* codes, cudaStream_t stream);
int launch_hadamard_fp8(const void* x, bool in_bf16, int64_t n_vec, int d, const int32_t* n_valid_dev,
                        const float* w, uint8_t* codes, float* scales, float* ws_out, cudaStream_t stream);

// Per-document score bases and scoring work schedule (one tiny kernel);
// qg = scoring_group(n_idx_heads, d_idx).
int launch_index_prep(const kpool_layout& L, int topk, int qg, int64_t* pair_base, int32_t* sched,
                      cudaStream_t stream);

// Queries per work item of the tcgen05 scoring kernel (256 / H_i for d_i =
// 128), or 0 when the mma.sync kernel serves the shape (d_i = 64).
int scoring_group(int n_idx_heads, int d_idx);

// FP8 pool scores into the compact triangle, for the work items j_lo .. j_hi-1 of the schedule
// (j_hi < 0: every item from j_lo on; item ranges other than the whole schedule need the tcgen05 kernel).
int launch_score(const uint8_t* q8, const float* ws, const uint8_t* k8, const float* s_k, const kpool_layout& L,
                 const int64_t* pair_base, const int32_t* sched, int topk, int n_idx_heads, int d_idx,
                 float* scores, cudaStream_t stream, int j_lo = 0, int j_hi = -1);

// The mma.sync e4m3 scoring kernel (d_i = 64 shapes).
int launch_score_mma(const uint8_t* q8, const float* ws, const uint8_t* k8, const float* s_k, const kpool_layout& L,
                     const int64_t* pair_base, const int32_t* sched, int topk, int n_idx_heads, int d_idx,
                     float* scores, cudaStream_t stream);

// Top-k select, expansion to positions, own tail, -1 padding, for the query rows row0 .. row1-1
// (row1 < 0: to the last row).
int launch_select(const float* scores, const int64_t* pair_base, const kpool_layout& L, int topk, int32_t* indices,
                  int W, cudaStream_t stream, int row0 = 0, int row1 = -1);

int launch_sparse_mla(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int n_rows,
                      int T, int n_heads, float scale, uint16_t* out, float* lse, int32_t* status,
                      cudaStream_t stream);

// Sparse latent attention backward: zeroes dkv, computes delta = rowsum(out * dout) into `delta`
// [n_rows, H], then dq (bf16) and dkv (fp32 reductions).
int launch_sparse_mla_bwd(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int n_rows,
                          int T, int n_heads, float scale, const uint16_t* out, const float* lse,
                          const uint16_t* dout, uint16_t* dq, float* dkv, float* delta, int32_t* status,
                          cudaStream_t stream);

// Test hooks of the bounded waits: nonzero makes the next launches of the kernel wait first on a barrier
// that cannot complete in time (tcgen05 scoring: its TMA producer; sparse MLA: its row scanner).
int set_score_tc_stall(int on);
int set_sparse_mla_stall(int on);

// Measurement: fp32 reductions into 512-float rows (the dKv scatter's access pattern).
int launch_l2_reduce(float* buf, int rows, const int32_t* row_ids, int n_ids, cudaStream_t stream);

// Paged decode (pages of 32 pools = 128 tokens): pooled keys into the page cache; paged FP8 scores
// scores[b * stride + p] for the complete pools of each sequence; top-k select into cache slots.
int launch_paged_append(const void* k, const float* gate, const float* ape, const int32_t* pool_tok,
                        const int32_t* pool_seq, const int32_t* pool_idx, int n_items, const int32_t* block_table,
                        int max_pages, int n_pages, uint8_t* k8_cache, float* sk_cache, int32_t* status,
                        cudaStream_t stream);
int launch_decode_score(const uint8_t* q8, const float* ws, const uint8_t* k8_cache, const float* sk_cache,
                        int n_pages, const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                        int n_idx_heads, float* scores, int64_t stride, int32_t* status, cudaStream_t stream);
int launch_decode_select(const float* scores, int64_t stride, const int32_t* seq_lens, const int32_t* block_table,
                         int max_pages, int B, int topk, int32_t* indices, int W, cudaStream_t stream);

// Absorbed-MLA projections (absorb: q_nope -> q_lat; otherwise o_lat -> o_v).
bool mla_proj_shape_ok(int n_heads, int d_nope, int d_v);
int launch_mla_proj(bool absorb, const void* act, const void* w_kv_b, int T, int n_heads, int d_nope, int d_v,
                    void* out, int32_t* status, cudaStream_t stream);

}  // namespace kpool
