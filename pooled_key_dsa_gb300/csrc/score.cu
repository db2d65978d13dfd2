// FP8 pool scoring for d_i = 64 (mma.sync e4m3) and the scoring schedule.
// The d_i = 128 shapes run on the tcgen05 kernel in score_tc.cu.
//
// prime-rl PR "GLM-5.3-Flash text model", Summary: each query scores the
// complete pools of its own document that end at or before it, reusing an FP8
// indexer over pools: S[i,p] = s_k[p] * sum_h ws[i,h] * ReLU(q8[i,h] . k8[p])
// with ws = w * s_q (miles "GLM-5.3-Flash" recipe, section 1: a
// kpool-compressed lightning indexer).
//
// Tiles are (document, 16 queries, 64 pools), enumerated per document over the
// causal triangle only, and only for query tiles holding a row with more than
// topk candidates (rows with fewer keep every pool and need no score).  A
// persistent grid walks the tile list.  Each of the 4 warps owns 16 pools and
// runs E4M3 tensor-core MMAs (m16n8k32, fp32 accumulate) against every query
// of the tile; the epilogue applies ReLU, the head weights, the head sum
// (thread-local plus two shuffles) and s_k, and stores into the compact
// per-row triangle.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

namespace {

constexpr int QT = 16;    // queries per tile
constexpr int PT = 64;    // pools per tile
constexpr int R = PT / (QT / KPOOL);   // query tiles per extra pool tile along the diagonal

// sum_{m=1..n} ceil(m / R)
__host__ __device__ __forceinline__ int64_t tri_tiles(int64_t n) {
    const int64_t a = n / R, b = n % R;
    return R * a * (a + 1) / 2 + b * (a + 1);
}

struct DocTiles {
    int qt0, Q;      // first scored query tile, number of query tiles
    int64_t count;   // tiles of the document
};

__device__ __forceinline__ DocTiles doc_tiles(int L, int topk) {
    DocTiles dt;
    dt.Q = (L + QT - 1) / QT;
    dt.qt0 = (KPOOL * topk + KPOOL - 1) / QT;      // tile holding r = 4*topk + 3
    const int P = L / KPOOL;
    if (dt.qt0 >= dt.Q) {
        dt.count = 0;
    } else {
        // query tiles qt0 .. Q-2 see ceil((qt+1)/R) pool tiles; the last sees ceil(P/PT)
        dt.count = tri_tiles(dt.Q - 1) - tri_tiles(dt.qt0) + (P + PT - 1) / PT;
    }
    return dt;
}

}  // namespace

// One block: pair_base[d] (start of document d's score triangle) and
// sched[d] (first work item of document d); sched[n_docs] = total items.
// qg = 0: items are the (16 queries x 64 pools) tiles of the mma.sync kernel;
// qg > 0: items are groups of qg consecutive queries (tcgen05 kernel), from
// the group holding r = 4*topk + 3 to the end of the document.
__global__ void __launch_bounds__(1024) index_prep_kernel(const int32_t* __restrict__ cu_seqlens,
                                                          const int32_t* __restrict__ cu_pools, int n_docs, int topk,
                                                          int qg, int64_t* __restrict__ pair_base,
                                                          int32_t* __restrict__ sched) {
    __shared__ int64_t wsum_p[32], wsum_t[32];
    __shared__ int64_t carry_p, carry_t;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    const bool ok = cu_pools[n_docs] >= 0;
    if (tid == 0) { carry_p = 0; carry_t = 0; }
    __syncthreads();
    for (int base = 0; base < n_docs; base += blockDim.x) {
        const int d = base + tid;
        int64_t vp = 0, vt = 0;
        if (ok && d < n_docs) {
            const int L = cu_seqlens[d + 1] - cu_seqlens[d];
            vp = pairs_before(L);
            if (qg > 0) {
                const int q_all = (L + qg - 1) / qg, q0 = (KPOOL * topk + KPOOL - 1) / qg;
                vt = q_all > q0 ? q_all - q0 : 0;
            } else {
                vt = doc_tiles(L, topk).count;
            }
        }
        int64_t xp = vp, xt = vt;
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t yp = __shfl_up_sync(0xffffffffu, xp, o);
            const int64_t yt = __shfl_up_sync(0xffffffffu, xt, o);
            if (lane >= o) { xp += yp; xt += yt; }
        }
        if (lane == 31) { wsum_p[wid] = xp; wsum_t[wid] = xt; }
        __syncthreads();
        int64_t bp = carry_p, bt = carry_t;
        for (int w = 0; w < wid; ++w) { bp += wsum_p[w]; bt += wsum_t[w]; }
        if (d < n_docs) {
            pair_base[d] = bp + xp - vp;
            sched[d] = (int32_t)(bt + xt - vt);
        }
        __syncthreads();
        if (tid == blockDim.x - 1) { carry_p = bp + xp; carry_t = bt + xt; }
        __syncthreads();
    }
    if (tid == 0) {
        pair_base[n_docs] = carry_p;
        sched[n_docs] = (int32_t)carry_t;
    }
    (void)nw;
}

__device__ __forceinline__ void mma_e4m3_16832(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int HI, int DI>
__global__ void __launch_bounds__(128) score_kernel(const uint8_t* __restrict__ q8, const float* __restrict__ ws,
                                                    const uint8_t* __restrict__ k8, const float* __restrict__ s_k,
                                                    const int32_t* __restrict__ cu_seqlens,
                                                    const int32_t* __restrict__ cu_pools, int n_docs, int max_pools,
                                                    const int64_t* __restrict__ pair_base,
                                                    const int32_t* __restrict__ sched, int topk,
                                                    float* __restrict__ scores) {
    constexpr int NT = (HI + 7) / 8;      // n8 tiles of heads
    constexpr int KS = DI / 32;           // k32 steps
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tig = lane & 3;
    const int total = sched[n_docs];
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int lo = 0, hi = n_docs - 1;                   // document: largest d with sched[d] <= tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sched[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        const int d = lo;
        const int s_d = cu_seqlens[d];
        const int L = cu_seqlens[d + 1] - s_d;
        const DocTiles dt = doc_tiles(L, topk);
        const int64_t u = tile - sched[d];
        // query tile: largest qt in [qt0, Q-1] with tri_tiles(qt) - tri_tiles(qt0) <= u
        int qlo = dt.qt0, qhi = dt.Q - 1;
        const int64_t t0 = tri_tiles(dt.qt0);
        while (qlo < qhi) {
            const int mid = (qlo + qhi + 1) >> 1;
            if (tri_tiles(mid) - t0 <= u) qlo = mid; else qhi = mid - 1;
        }
        const int qt = qlo;
        const int pt = (int)(u - (tri_tiles(qt) - t0));
        const int p0 = cu_pools[d];
        const int local0 = pt * PT + warp * 16;        // this warp's first pool (in-document)

        // A fragments: 16 pools x DI codes of this warp
        uint32_t a[KS][4];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int pool = p0 + local0 + g + 8 * half;
                const bool in = pool < max_pools;
                const uint8_t* src = k8 + (int64_t)(in ? pool : 0) * DI + ks * 32 + tig * 4;
                a[ks][half] = in ? __ldg(reinterpret_cast<const uint32_t*>(src)) : 0u;
                a[ks][2 + half] = in ? __ldg(reinterpret_cast<const uint32_t*>(src + 16)) : 0u;
            }
        }
        const int poolA = p0 + local0 + g, poolB = poolA + 8;
        const float skA = poolA < max_pools ? s_k[poolA] : 0.f;
        const float skB = poolB < max_pools ? s_k[poolB] : 0.f;

        for (int qq = 0; qq < QT; ++qq) {
            const int r = qt * QT + qq;
            if (r >= L) break;
            const int n_i = (r + 1) / KPOOL;
            if (n_i <= topk || local0 >= n_i) continue;
            const int i = s_d + r;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
                const int h = nt * 8 + g;
                const bool hv = h < HI;
                const uint8_t* qrow = q8 + ((int64_t)i * HI + (hv ? h : 0)) * DI;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const uint32_t b0 = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 32 + tig * 4)) : 0u;
                    const uint32_t b1 = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 32 + 16 + tig * 4)) : 0u;
                    mma_e4m3_16832(acc[nt], a[ks], b0, b1);
                }
            }
            float sA = 0.f, sB = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = nt * 8 + tig * 2 + e;
                    const float wv = h < HI ? __ldg(ws + (int64_t)i * HI + h) : 0.f;
                    sA += wv * fmaxf(acc[nt][e], 0.f);
                    sB += wv * fmaxf(acc[nt][2 + e], 0.f);
                }
            }
            sA += __shfl_xor_sync(0xffffffffu, sA, 1);
            sA += __shfl_xor_sync(0xffffffffu, sA, 2);
            sB += __shfl_xor_sync(0xffffffffu, sB, 1);
            sB += __shfl_xor_sync(0xffffffffu, sB, 2);
            if (tig == 0) {
                float* dst = scores + pair_base[d] + pairs_before(r);
                if (local0 + g < n_i) dst[local0 + g] = sA * skA;
                if (local0 + g + 8 < n_i) dst[local0 + g + 8] = sB * skB;
            }
        }
    }
}

int launch_index_prep(const kpool_layout& L, int topk, int qg, int64_t* pair_base, int32_t* sched,
                      cudaStream_t stream) {
    index_prep_kernel<<<1, 1024, 0, stream>>>(L.cu_seqlens, L.cu_pools, L.n_docs, topk, qg, pair_base, sched);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

template <int HI, int DI>
static void launch_score_t(const uint8_t* q8, const float* ws, const uint8_t* k8, const float* s_k,
                           const kpool_layout& L, const int64_t* pair_base, const int32_t* sched, int topk,
                           float* scores, cudaStream_t stream) {
    score_kernel<HI, DI><<<152 * 8, 128, 0, stream>>>(q8, ws, k8, s_k, L.cu_seqlens, L.cu_pools, L.n_docs,
                                                      L.max_pools, pair_base, sched, topk, scores);
}

int launch_score_mma(const uint8_t* q8, const float* ws, const uint8_t* k8, const float* s_k, const kpool_layout& L,
                     const int64_t* pair_base, const int32_t* sched, int topk, int n_idx_heads, int d_idx,
                     float* scores, cudaStream_t stream) {
#define KPOOL_SCORE_CASE(H, D)                                                                   \
    if (n_idx_heads == H && d_idx == D) {                                                        \
        launch_score_t<H, D>(q8, ws, k8, s_k, L, pair_base, sched, topk, scores, stream);        \
        return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;                    \
    }
    KPOOL_SCORE_CASE(32, 64)
    KPOOL_SCORE_CASE(16, 64)
    KPOOL_SCORE_CASE(8, 64)
    KPOOL_SCORE_CASE(4, 64)
#undef KPOOL_SCORE_CASE
    return KPOOL_ERR_SHAPE;
}

}  // namespace kpool
