// FP8 pool scoring on tcgen05 (d_i = 128).
//
// prime-rl PR "GLM-5.3-Flash text model", Summary: each query scores the
// complete pools of its own document that end at or before it with an FP8
// indexer over pools: S[i,p] = s_k[p] * sum_h ws[i,h] * ReLU(q8[i,h] . k8[p]),
// ws = w * s_q (miles "GLM-5.3-Flash" recipe, section 1: kpool-compressed
// lightning indexer).
//
// Work item = a group of QG = 256 / H_i consecutive queries of one document
// (from the group holding r = 4*topk + 3 on; earlier rows keep every pool).
// Per item the (query, head) rows form the MMA's N = 256 operand (TMA, one
// 32 KB box); the item's pools stream through a 6-stage ring of 128-pool A
// tiles (TMA, 16 KB).  Each tile is 4 tcgen05 kind::f8f6f4 MMAs (M = 128
// pools, N = 256, K = 32) into one of two TMEM accumulators, so the epilogue
// of tile t overlaps the MMAs of tile t+1.
//
// Epilogue: two groups of 4 warps; group g takes the tiles of TMEM buffer g,
// so the epilogues of consecutive tiles run side by side.  A thread owns one
// pool (its TMEM lane) and all 256 columns, read in 32-column loads issued one
// chunk ahead; ReLU, the head weights and the head sum stay thread-local
// (packed fp32 adds and FMAs, independent partial sums); one coalesced store
// per (query, pool).
// Items are spread over the persistent CTAs in a snake order (the item size
// grows along a document).  Waits are bounded (KPOOL_ERR_TIMEOUT).
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kpool_common.cuh"
#include "kpool_launch.h"
#include "tc_ptx.cuh"
#include "tmap_host.h"

namespace kpool {

namespace {

constexpr int SC_THREADS = 384;        // warp 0 TMA, warp 1 MMA, warps 4-11 epilogue
constexpr int A_STAGES = 6;
constexpr int A_BYTES = 128 * 128;     // 128 pools x 128 B
constexpr int B_BYTES = 256 * 128;     // 256 (query, head) rows x 128 B
constexpr int OFF_B = 0;
constexpr int OFF_A = OFF_B + 2 * B_BYTES;
constexpr int OFF_WS = OFF_A + A_STAGES * A_BYTES;
constexpr int OFF_SMALL = OFF_WS + 4 * 256 * 4;     // two groups x two items x 256 weights

struct ScSmall {
    uint64_t b_full[2], b_empty[2], a_full[A_STAGES], a_empty[A_STAGES], acc_full[2], acc_empty[2], drain;
    uint64_t never;                    // no thread arrives on it: the stall hook waits here
    int abort;
    uint32_t tmem;
};
constexpr int SC_SMEM = OFF_SMALL + (int)sizeof(ScSmall) + 1024;

constexpr uint32_t ID_SC = tc::idesc(128, 256, 0, 0, false, false);   // e4m3 x e4m3 -> fp32

struct Item {
    int d, s_d, L, p0, r0, ntiles;
};

__device__ __forceinline__ Item decode_item(int j, const int32_t* sched, const int32_t* cu_seqlens,
                                            const int32_t* cu_pools, int n_docs, int topk, int qg) {
    int lo = 0, hi = n_docs - 1;                 // largest d with sched[d] <= j
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sched[mid] <= j) lo = mid; else hi = mid - 1;
    }
    Item it;
    it.d = lo;
    it.s_d = cu_seqlens[lo];
    it.L = cu_seqlens[lo + 1] - it.s_d;
    it.p0 = cu_pools[lo];
    it.r0 = ((KPOOL * topk + KPOOL - 1) / qg + (j - sched[lo])) * qg;
    const int r_last = min(it.r0 + qg - 1, it.L - 1);
    const int nmax = (r_last + 1) / KPOOL;
    it.ntiles = (nmax + 127) / 128;
    return it;
}

// k-th item of this CTA in snake order over the grid (balances growing items)
__device__ __forceinline__ int item_of(int k) {
    const int G = gridDim.x, c = blockIdx.x;
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(addr, parity, abort) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Named barrier 1 + g over the 128 threads of epilogue group g, ORing a predicate.
__device__ __forceinline__ bool group_or(bool pred, int g) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(1 + g)
        : "memory");
    return r != 0;
}

// One 32-column chunk cc of a thread's row (cc is a constant after unrolling):
// res[q] = sum over the heads h of query q in this chunk of
// ws[q,h] * ReLU(acc[q,h]).  Column pairs go through packed fp32 FMAs into up
// to four independent partial sums per query (short dependency chains); a
// query spanning two chunks (H_i = 64) adds the second chunk's sum to the first.
template <int HI, int NQ>
__device__ __forceinline__ void score_chunk(const uint32_t (&v)[32], const float* __restrict__ wrow, int cc,
                                            float (&res)[NQ]) {
    constexpr int HC = HI >= 32 ? 32 : HI;           // columns of one query in this chunk
    constexpr int QPC = 32 / HC;                     // queries in this chunk
    constexpr int PPQ = HC / 2;                      // column pairs of one query
    constexpr int NP = PPQ >= 4 ? 4 : PPQ;           // partial sums per query
    const float4* w4 = reinterpret_cast<const float4*>(wrow + cc * 32);
#pragma unroll
    for (int qq = 0; qq < QPC; ++qq) {
        float2 part[NP];
#pragma unroll
        for (int jp = 0; jp < PPQ; ++jp) {
            const int c = qq * HC + 2 * jp;           // column within the chunk
            const float4 wv = w4[c >> 2];
            const float2 w2 = (c & 2) ? make_float2(wv.z, wv.w) : make_float2(wv.x, wv.y);
            // 2*ReLU(a) = a + |a|, exact (+0 for a <= 0; the accumulator is never NaN), as one packed
            // add on the FMA pipe instead of a max per element on the ALU pipe; the head weights in
            // shared memory carry the factor 1/2 (exact for normal values), so each product is ws * ReLU(a)
            const float a0 = __uint_as_float(v[c]), a1 = __uint_as_float(v[c + 1]);
            const float2 x = __fadd2_rn(make_float2(a0, a1), make_float2(fabsf(a0), fabsf(a1)));
            if (jp < NP)
                part[jp] = __fmul2_rn(x, w2);
            else
                part[jp % NP] = __ffma2_rn(x, w2, part[jp % NP]);
        }
#pragma unroll
        for (int p = 1; p < NP; ++p) part[0] = __fadd2_rn(part[0], part[p]);
        const int q = cc * 32 / HI + qq;
        const float s = part[0].x + part[0].y;
        if ((cc * 32) % HI == 0) res[q] = s;
        else res[q] += s;
    }
}

// Nonzero: the next launches stall their TMA producer on a barrier that is never
// completed (test of the bounded waits; set with set_score_tc_stall).
__device__ int g_score_tc_stall = 0;

}  // namespace

int set_score_tc_stall(int on) {
    const int v = on ? 1 : 0;
    return cudaMemcpyToSymbol(g_score_tc_stall, &v, sizeof(v)) == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

template <int HI>
__global__ void __launch_bounds__(SC_THREADS, 1) score_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k, const float* __restrict__ ws,
    const float* __restrict__ s_k, const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ cu_pools,
    int n_docs, int max_pools, int T, const int64_t* __restrict__ pair_base, const int32_t* __restrict__ sched,
    int topk, uint32_t b_box_bytes, uint32_t a_box_bytes, float* __restrict__ scores, int64_t n_scores,
    int32_t* status, int j_lo, int j_hi) {
    constexpr int QG = 256 / HI;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    ScSmall& sm = *reinterpret_cast<ScSmall*>(smem + OFF_SMALL);
    const uint32_t s_base = tc::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &sm.abort;
    // work items j_lo .. j_hi-1 of the schedule (j_hi < 0: to the last item)
    const int total = (j_hi < 0 ? sched[n_docs] : j_hi) - j_lo;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tc::smem_u32(&sm.b_full[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.b_empty[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.acc_full[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.acc_empty[b]), 4);
        }
        for (int s = 0; s < A_STAGES; ++s) {
            tc::mbar_init(tc::smem_u32(&sm.a_full[s]), 1);
            tc::mbar_init(tc::smem_u32(&sm.a_empty[s]), 1);
        }
        tc::mbar_init(tc::smem_u32(&sm.drain), 1);
        tc::mbar_init(tc::smem_u32(&sm.never), 1);
        sm.abort = 0;
        tc::mbar_init_fence();
    }
    if (warp == 1) tc::tmem_alloc(tc::smem_u32(&sm.tmem), 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp == 0) {
        // ===================================================== TMA producer
        if (lane == 0) {
            uint32_t ni = 0, na = 0;
            // test hook: with a stall injected, wait first on a barrier that nothing completes, so the
            // bounded waits of every role run out
            bool ok = g_score_tc_stall == 0 || tc::mbar_wait(tc::smem_u32(&sm.never), 0, abort_flag);
            for (int k = 0; ok; ++k, ++ni) {
                const int jj = item_of(k);
                if (jj >= total) break;
                const int j = j_lo + jj;
                const Item it = decode_item(j, sched, cu_seqlens, cu_pools, n_docs, topk, QG);
                const int ib = ni & 1;
                if (!tc::mbar_wait(tc::smem_u32(&sm.b_empty[ib]), ((ni >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
                tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.b_full[ib]), b_box_bytes);
                tc::tma_load_2d(s_base + OFF_B + ib * B_BYTES, &tmap_q, 0, (it.s_d + it.r0) * HI,
                                tc::smem_u32(&sm.b_full[ib]));
                for (int t = 0; t < it.ntiles; ++t, ++na) {
                    const int as = na % A_STAGES;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.a_empty[as]), ((na / A_STAGES) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.a_full[as]), a_box_bytes);
                    tc::tma_load_2d(s_base + OFF_A + as * A_BYTES, &tmap_k, 0, it.p0 + 128 * t,
                                    tc::smem_u32(&sm.a_full[as]));
                }
            }
            if (!ok) {
                sm.abort = 1;
                set_status(status, KPOOL_ERR_TIMEOUT);
            }
            // no TMA load may still be writing shared memory when the CTA ends: wait (bounded by the
            // full limit, whatever the outcome) for the last load issued into every buffer.  The
            // parity is that of the load's own phase; the barrier cannot have moved past it, since
            // no later load went into the same buffer.
            for (int s = 0; s < A_STAGES; ++s) {
                if ((uint32_t)s >= na) break;
                const uint32_t last = na - 1 - ((na - 1 - (uint32_t)s) % A_STAGES);   // last load into stage s
                tc::mbar_wait_for(tc::smem_u32(&sm.a_full[s]), (last / A_STAGES) & 1, tc::WAIT_LIMIT_NS);
            }
            for (uint32_t n = ni >= 2 ? ni - 2 : 0; n < ni; ++n)
                tc::mbar_wait_for(tc::smem_u32(&sm.b_full[n & 1]), (n >> 1) & 1, tc::WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        if (lane == 0) {
            uint32_t ni = 0, na = 0, nacc = 0;
            bool ok = true;
            for (int k = 0; ok && !*abort_flag; ++k, ++ni) {
                const int jj = item_of(k);
                if (jj >= total) break;
                const int j = j_lo + jj;
                const Item it = decode_item(j, sched, cu_seqlens, cu_pools, n_docs, topk, QG);
                const int ib = ni & 1;
                if (!tc::mbar_wait(tc::smem_u32(&sm.b_full[ib]), (ni >> 1) & 1, abort_flag)) { ok = false; break; }
                const uint64_t bd = tc::sw128_desc(s_base + OFF_B + ib * B_BYTES, 0, 1024);
                for (int t = 0; t < it.ntiles; ++t, ++na, ++nacc) {
                    const int as = na % A_STAGES, ab = nacc & 1;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.a_full[as]), (na / A_STAGES) & 1, abort_flag) ||
                        !tc::mbar_wait(tc::smem_u32(&sm.acc_empty[ab]), ((nacc >> 1) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint64_t ad = tc::sw128_desc(s_base + OFF_A + as * A_BYTES, 0, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_e4m3(tmem + 256 * ab, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), ID_SC,
                                     kk > 0 ? 1u : 0u);
                    tc::commit(tc::smem_u32(&sm.a_empty[as]));
                    tc::commit(tc::smem_u32(&sm.acc_full[ab]));
                }
                if (!ok) break;
                tc::commit(tc::smem_u32(&sm.b_empty[ib]));
            }
            if (!ok) {
                sm.abort = 1;
                set_status(status, KPOOL_ERR_TIMEOUT);
            }
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ===================================================== epilogue
        // group g (warps 4-7 / 8-11) takes the tiles of TMEM buffer g (running tile index of parity g), so
        // the epilogues of two consecutive tiles run at once; warp w reads TMEM lanes 32*(w%4) .., all columns
        const int g = (warp - 4) >> 2;
        const int e = tid - 128 - 128 * g;            // 0..127 within the group
        const int sp = warp & 3;                      // TMEM subpartition (lanes 32sp..)
        const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
        uint32_t ni = 0, nacc = 0;
        bool bad = false;
        for (int k = 0;; ++k, ++ni) {
            const int jj = item_of(k);
            if (jj >= total) break;
            const int j = j_lo + jj;
            const Item it = decode_item(j, sched, cu_seqlens, cu_pools, n_docs, topk, QG);
            const int i0 = it.s_d + it.r0;
            // the item's head weights (256 floats), halved, into this group's shared buffer
            float* wsb = reinterpret_cast<float*>(smem + OFF_WS) + g * 512 + (ni & 1) * 256;
            wsb[e] = (it.r0 + e / HI < it.L) ? 0.5f * ws[(int64_t)i0 * HI + e] : 0.f;
            wsb[e + 128] = (it.r0 + (e + 128) / HI < it.L) ? 0.5f * ws[(int64_t)i0 * HI + e + 128] : 0.f;
            if (group_or(bad, g)) { bad = true; break; }
            const int64_t row_base = pair_base[it.d];
            // per query: the start of its score row and its pool count (0: no scored row)
            constexpr int QS = QG <= 8 ? QG : 1;
            int64_t qbase[QS];
            int qlim[QS];
            if constexpr (QG <= 8) {
#pragma unroll
                for (int q = 0; q < QG; ++q) {
                    const int r = it.r0 + q;
                    const int n_i = (r + 1) / KPOOL;
                    qbase[q] = row_base + pairs_before(r);
                    qlim[q] = (r < it.L && n_i > topk) ? n_i : 0;
                }
            }
            for (int t = (int)((nacc & 1) != (uint32_t)g); t < it.ntiles; t += 2) {
                const uint32_t na = nacc + (uint32_t)t;      // running tile index; buffer na & 1 == g
                const int pool_local = 128 * t + 32 * sp + lane;
                const int pool = it.p0 + pool_local;
                const float sk = pool < max_pools ? s_k[pool] : 0.f;
                bad = bad || !warp_wait(tc::smem_u32(&sm.acc_full[g]), (na >> 1) & 1, abort_flag);
                if (bad) continue;                           // the group learns it at the next item
                tc::fence_after();
                // eight 32-column loads; each is issued before the previous chunk is summed
                const uint32_t tb = tmem + 256 * g + lane_base;
                float res[QG];
                auto store = [&](int q) {
                    if constexpr (QG <= 8) {
                        if (pool_local < qlim[q] && in_bounds(qbase[q] + pool_local < n_scores, status))
                            scores[qbase[q] + pool_local] = res[q] * sk;
                    } else {
                        const int r = it.r0 + q;
                        const int n_i = (r + 1) / KPOOL;
                        const int64_t o = row_base + pairs_before(r) + pool_local;
                        if (r < it.L && n_i > topk && pool_local < n_i && in_bounds(o < n_scores, status))
                            scores[o] = res[q] * sk;
                    }
                };
                if constexpr (QG <= 32) {
                    uint32_t v[2][32];
                    tc::tmem_ld32(tb, v[0]);
                    tc::tmem_wait_ld32(v[0]);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        if (cc < 7) {
                            tc::tmem_ld32(tb + 32 * (cc + 1), v[(cc + 1) & 1]);
                        } else {                              // every load of the buffer has completed
                            tc::fence_before();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.acc_empty[g]));
                        }
                        score_chunk<HI>(v[cc & 1], wsb, cc, res);
                        if (cc < 7) tc::tmem_wait_ld32(v[(cc + 1) & 1]);
                    }
#pragma unroll
                    for (int q = 0; q < QG; ++q) store(q);
                } else {                                      // H_i = 4: 64 results per thread, one buffer
                    uint32_t v[32];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        tc::tmem_ld32(tb + 32 * cc, v);
                        tc::tmem_wait_ld32(v);
                        if (cc == 7) {
                            tc::fence_before();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.acc_empty[g]));
                        }
                        score_chunk<HI>(v, wsb, cc, res);
#pragma unroll
                        for (int q = cc * QG / 8; q < (cc + 1) * QG / 8; ++q) store(q);   // queries of chunk cc
                    }
                }
            }
            nacc += (uint32_t)it.ntiles;
        }
        if (bad) {
            sm.abort = 1;
            set_status(status, KPOOL_ERR_TIMEOUT);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

int scoring_group(int n_idx_heads, int d_idx) {
    if (d_idx != 128) return 0;
    switch (n_idx_heads) {
        case 4: case 8: case 16: case 32: case 64: return 256 / n_idx_heads;
        default: return 0;
    }
}

// 2-D byte tensor [rows, 128] with 128-byte rows, 128-byte swizzle, box
// {128, box_rows}.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HI>
static int launch_tc(const uint8_t* q8, const float* ws, const uint8_t* k8, const float* s_k, const kpool_layout& L,
                     const int64_t* pair_base, const int32_t* sched, int topk, float* scores, int j_lo, int j_hi,
                     cudaStream_t stream) {
    static int n_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    if (n_sm[dev] == 0) {
        if (cudaFuncSetAttribute(score_tc_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM) !=
            cudaSuccess)
            return KPOOL_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KPOOL_ERR_CUDA;
        n_sm[dev] = sms;
    }
    const uint64_t q_rows = (uint64_t)L.T * HI;
    const uint64_t k_rows = (uint64_t)(L.max_pools > 0 ? L.max_pools : 1);
    const uint32_t b_rows = (uint32_t)(q_rows < 256 ? q_rows : 256);
    const uint32_t a_rows = (uint32_t)(k_rows < 128 ? k_rows : 128);
    CUtensorMap mq, mk;
    if (!make_map(&mq, q8, q_rows, b_rows) || !make_map(&mk, k8, k_rows, a_rows)) return KPOOL_ERR_CUDA;
    score_tc_kernel<HI><<<n_sm[dev], SC_THREADS, SC_SMEM, stream>>>(
        mq, mk, ws, s_k, L.cu_seqlens, L.cu_pools, L.n_docs, L.max_pools, L.T, pair_base, sched, topk, b_rows * 128,
        a_rows * 128, scores, pairs_before(L.T), L.status, j_lo, j_hi);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

int launch_score(const uint8_t* q8, const float* ws, const uint8_t* k8, const float* s_k, const kpool_layout& L,
                 const int64_t* pair_base, const int32_t* sched, int topk, int n_idx_heads, int d_idx,
                 float* scores, cudaStream_t stream, int j_lo, int j_hi) {
    if (L.T <= 0) return KPOOL_OK;
    if (scoring_group(n_idx_heads, d_idx) == 0) {
        if (j_lo != 0 || j_hi >= 0) return KPOOL_ERR_SHAPE;        // item ranges are a tcgen05-kernel feature
        return launch_score_mma(q8, ws, k8, s_k, L, pair_base, sched, topk, n_idx_heads, d_idx, scores, stream);
    }
    if (j_lo < 0 || (j_hi >= 0 && j_hi < j_lo)) return KPOOL_ERR_INVALID_ARG;
    if (j_hi >= 0 && j_hi == j_lo) return KPOOL_OK;
    switch (n_idx_heads) {
        case 4: return launch_tc<4>(q8, ws, k8, s_k, L, pair_base, sched, topk, scores, j_lo, j_hi, stream);
        case 8: return launch_tc<8>(q8, ws, k8, s_k, L, pair_base, sched, topk, scores, j_lo, j_hi, stream);
        case 16: return launch_tc<16>(q8, ws, k8, s_k, L, pair_base, sched, topk, scores, j_lo, j_hi, stream);
        case 32: return launch_tc<32>(q8, ws, k8, s_k, L, pair_base, sched, topk, scores, j_lo, j_hi, stream);
        case 64: return launch_tc<64>(q8, ws, k8, s_k, L, pair_base, sched, topk, scores, j_lo, j_hi, stream);
        default: return KPOOL_ERR_SHAPE;
    }
}

}  // namespace kpool
