// PoolLayout builder and k-pool pooling kernels.
//
// prime-rl PR "GLM-5.3-Flash text model", Summary: indexer keys are pooled per
// document in groups of 4 starting at each document's first token, as a
// per-channel softmax(gate + ape)-weighted mean; the per-document pool layout
// is built once per forward.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

// One block: validates cu_seqlens (0 = c_0 <= c_1 <= ... <= c_n = T) and writes
// cu_pools as the running sum of floor(L_d / 4).  An invalid layout is marked
// by cu_pools[n_docs] = -1 (all other entries 0) and KPOOL_ERR_LAYOUT.
__global__ void __launch_bounds__(1024) layout_scan_kernel(const int32_t* __restrict__ cu_seqlens,
                                                           int n_docs, int T,
                                                           int32_t* __restrict__ cu_pools,
                                                           int32_t* status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int bad = 0;
    for (int d = tid; d < n_docs; d += blockDim.x)
        bad |= cu_seqlens[d + 1] < cu_seqlens[d];
    if (tid == 0) bad |= (cu_seqlens[0] != 0) | (cu_seqlens[n_docs] != T);
    bad = __syncthreads_or(bad);
    if (bad) {
        for (int d = tid; d < n_docs; d += blockDim.x) cu_pools[d] = 0;
        if (tid == 0) {
            cu_pools[n_docs] = -1;
            set_status(status, KPOOL_ERR_LAYOUT);
        }
        return;
    }
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < n_docs; base += blockDim.x) {
        const int d = base + tid;
        const int v = d < n_docs ? (cu_seqlens[d + 1] - cu_seqlens[d]) / KPOOL : 0;
        int x = v;                                      // inclusive warp scan
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            warp_sums[lane] = s;                        // inclusive over warps
        }
        __syncthreads();
        const int excl = carry + (wid ? warp_sums[wid - 1] : 0) + x - v;
        if (d < n_docs) cu_pools[d] = excl;
        __syncthreads();
        if (tid == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (tid == 0) cu_pools[n_docs] = carry;
}

// One thread per token: tok_doc, and pool_tok_start for tokens that open a
// complete pool.  Thread p also zeroes pool_tok_start[p] for p past the pool
// count.
__global__ void layout_fill_kernel(const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ cu_pools,
                                   int n_docs, int T, int max_pools, int32_t* __restrict__ pool_tok_start,
                                   int32_t* __restrict__ tok_doc) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T) return;
    const int P = cu_pools[n_docs];
    if (P < 0) {
        tok_doc[i] = -1;
        if (i < max_pools) pool_tok_start[i] = 0;
        return;
    }
    if (i >= P && i < max_pools) pool_tok_start[i] = 0;
    int lo = 0, hi = n_docs - 1;                        // largest d with cu_seqlens[d] <= i
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_seqlens[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int d = lo;
    tok_doc[i] = d;
    const int r = i - cu_seqlens[d];
    const int L = cu_seqlens[d + 1] - cu_seqlens[d];
    if ((r & (KPOOL - 1)) == 0 && r + KPOOL <= L) pool_tok_start[cu_pools[d] + r / KPOOL] = i;
}

// Pooled keys: one thread per (pool, 4 channels).  The softmax and the
// weighted sum run in fp64 in a fixed order (max, exp(l - max), sequential sum,
// e/s, sequential weighted sum) and are rounded once to fp32.
__global__ void kpool_pool_kernel(const uint16_t* __restrict__ k, const float* __restrict__ gate,
                                  const float* __restrict__ ape, const int32_t* __restrict__ cu_pools,
                                  const int32_t* __restrict__ pool_tok_start, int n_docs, int max_pools,
                                  int d_idx, float* __restrict__ kpool_out, int T, int32_t* status) {
    const int groups = d_idx >> 2;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (int64_t)max_pools * groups) return;
    const int p = (int)(gid / groups);
    const int c = (int)(gid % groups) * 4;
    const int P = max(cu_pools[n_docs], 0);
    float4* dst = reinterpret_cast<float4*>(kpool_out + (int64_t)p * d_idx + c);
    if (p >= P) {
        *dst = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int t0 = pool_tok_start[p];
    if (!in_bounds(t0 >= 0 && t0 + KPOOL <= T, status)) return;
    double lg[KPOOL][4], kv[KPOOL][4];
#pragma unroll
    for (int j = 0; j < KPOOL; ++j) {
        const float4 g = *reinterpret_cast<const float4*>(gate + (int64_t)(t0 + j) * d_idx + c);
        const float4 a = *reinterpret_cast<const float4*>(ape + j * d_idx + c);
        const uint2 kb = *reinterpret_cast<const uint2*>(k + (int64_t)(t0 + j) * d_idx + c);
        lg[j][0] = __dadd_rn((double)g.x, (double)a.x);
        lg[j][1] = __dadd_rn((double)g.y, (double)a.y);
        lg[j][2] = __dadd_rn((double)g.z, (double)a.z);
        lg[j][3] = __dadd_rn((double)g.w, (double)a.w);
        kv[j][0] = (double)bf16_bits_to_float((uint16_t)(kb.x & 0xffffu));
        kv[j][1] = (double)bf16_bits_to_float((uint16_t)(kb.x >> 16));
        kv[j][2] = (double)bf16_bits_to_float((uint16_t)(kb.y & 0xffffu));
        kv[j][3] = (double)bf16_bits_to_float((uint16_t)(kb.y >> 16));
    }
    float res[4];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        double m = lg[0][ch];
        int jm = 0;                                   // first index holding the max: its weight is exp(0) = 1
#pragma unroll
        for (int j = 1; j < KPOOL; ++j) {
            jm = lg[j][ch] > m ? j : jm;
            m = fmax(m, lg[j][ch]);
        }
        // exp of the other three logits only (gathered so that every lane runs the same three exps)
        double o[KPOOL - 1];
#pragma unroll
        for (int k = 0; k < KPOOL - 1; ++k) {
            const int j = k + (k >= jm ? 1 : 0);
            double v = lg[0][ch];
#pragma unroll
            for (int jj = 1; jj < KPOOL; ++jj) v = j == jj ? lg[jj][ch] : v;
            o[k] = exp(__dsub_rn(v, m));
        }
        double e[KPOOL];
#pragma unroll
        for (int j = 0; j < KPOOL; ++j) {
            const int k = j < jm ? j : j - 1;
            double v = 1.0;
#pragma unroll
            for (int kk = 0; kk < KPOOL - 1; ++kk) v = (j != jm && k == kk) ? o[kk] : v;
            e[j] = v;
        }
        double s = 0.0;
#pragma unroll
        for (int j = 0; j < KPOOL; ++j) s = __dadd_rn(s, e[j]);
        double acc = 0.0;
#pragma unroll
        for (int j = 0; j < KPOOL; ++j) acc = __dadd_rn(acc, __dmul_rn(__ddiv_rn(e[j], s), kv[j][ch]));
        res[ch] = (float)acc;
    }
    *dst = make_float4(res[0], res[1], res[2], res[3]);
}

int launch_kpool_build(const void* k, const float* gate, const float* ape, const kpool_layout& L, int d_idx,
                       float* kpool_out, cudaStream_t stream) {
    layout_scan_kernel<<<1, 1024, 0, stream>>>(L.cu_seqlens, L.n_docs, L.T, L.cu_pools, L.status);
    if (L.T > 0)
        layout_fill_kernel<<<ceil_div(L.T, 256), 256, 0, stream>>>(L.cu_seqlens, L.cu_pools, L.n_docs, L.T,
                                                                   L.max_pools, L.pool_tok_start, L.tok_doc);
    const int64_t work = (int64_t)L.max_pools * (d_idx / 4);
    if (work > 0)
        kpool_pool_kernel<<<(unsigned)((work + 255) / 256), 256, 0, stream>>>(
            static_cast<const uint16_t*>(k), gate, ape, L.cu_pools, L.pool_tok_start, L.n_docs, L.max_pools,
            d_idx, kpool_out, L.T, L.status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
