// Sparse latent attention forward (absorbed NoPE MLA over index rows), tcgen05.
//
// NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog: the K
// projection is absorbed into the query and attention runs over the shared
// 512-wide latent, which is both key and value; the caller applies the V
// projection afterwards.  miles "GLM-5.3-Flash" recipe, section 1: NoPE MLA,
// 64 heads.
//
// Persistent CTAs (one per SM), each walking query tokens i = blockIdx.x +
// k*gridDim.x.  For one query the index row is cut into blocks of 32 slots:
//   S   = Q Kv^T      tcgen05 kind::f16, M = 64 heads, N = 32 slots, K = 512,
//                     split over two issuing warps (latent 0-255 / 256-511,
//                     two accumulators the softmax adds)
//   O^T += Kv^T P^T   tcgen05 kind::f16, M = 128 latent rows (4 tiles),
//                     N = 64 heads, K = 32 slots; A is the gathered block read
//                     MN-major, so the tile that fed S also feeds PV
// Q (64 KB) stays in shared memory for the whole query; gathered latent rows
// go through a 4-stage ring of 32 KB blocks; S (2 buffers x 2 halves x 32
// columns) and O^T (4 x 64 columns) live in TMEM.
//
// The latent gather from L2 is this kernel's binding resource (about 1 KB per
// slot, shared by nothing across queries), so four producer warps keep many
// 16-byte cp.async in flight; each lane's copies arrive on the stage's
// mbarrier when they land (cp.async.mbarrier.arrive.noinc), so no producer
// ever waits for a copy, and the MMA issuers take a proxy fence before
// reading the tile.
//
// Warp roles (384 threads):
//   warps 0-3  producers: index scan, Q, latent rows (128-byte swizzle
//              written by hand), 8 rows of every block per warp
//   warps 4-7  softmax: the M=64 accumulator sits in lanes 0-15 of each
//              warp's TMEM subpartition; after the load, lanes 16-31 take the
//              upper 16 slots of every row, so all 32 lanes work.  The running
//              max only moves (and O^T is rescaled) when a slot beats it by
//              more than 2^8; a vote on that is the only barrier of a block in
//              the common case.  P^T goes to shared memory in the operand
//              layout; the epilogue writes O^T / l as bf16 through a staging
//              tile (the P buffers, idle by then).
//   warps 8-9  S issuers (warp 8 also owns the TMEM allocation)
//   warp 10    PV issuer
// Every wait is bounded and warp-uniform (lane 0 polls, the warp takes its
// answer); on expiry the kernel records KPOOL_ERR_TIMEOUT, the softmax warps
// agree on stopping at their next named barrier, every role leaves its loop,
// in-flight copies and MMAs are drained and TMEM is freed.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"
#include "tc_ptx.cuh"

namespace kpool {

namespace {

constexpr int BN = 32;                 // slots per block
constexpr int NSTAGE = 4;              // latent-row ring depth
constexpr int NSB = 2;                 // S / P double buffers
constexpr int HP = 64;                 // head rows (M of S, N of PV)
constexpr float TAU = 8.0f;            // lazy-rescale threshold (log2 units)
constexpr int THREADS = 384;
constexpr int NPROD = 4;               // producer warps

constexpr int Q_BYTES = HP * D_LAT * 2;          // 64 KB: 8 chunks x [64 rows x 128 B]
constexpr int Q_CHUNK = HP * 128;                // 8 KB
constexpr int KV_BYTES = BN * D_LAT * 2;         // 32 KB: 8 chunks x [32 rows x 128 B]
constexpr int KV_CHUNK = BN * 128;               // 4 KB
constexpr int P_BYTES = HP * 128;                // 8 KB: [64 head rows x 128 B], first 64 B used

constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + Q_BYTES;
constexpr int OFF_P = OFF_KV + NSTAGE * KV_BYTES;        // 2 P buffers = the 16 KB epilogue staging
constexpr int OFF_SMALL = OFF_P + NSB * P_BYTES;

struct Small {
    uint64_t q_full, q_empty, o_full, o_free, drain;
    uint64_t kv_full[NSTAGE], kv_empty[NSTAGE];
    uint64_t s_full[NSB], s_free[NSB], p_full[NSB], p_empty[NSB], o_step[NSB];
    uint8_t mask[NSTAGE][NPROD];           // valid-slot bits, 8 slots per producer warp
    int nb;
    int abort;
    uint32_t tmem;
    float alpha[2][HP];
    float inv_l[HP];
};
constexpr int SMEM_BYTES = OFF_SMALL + (int)sizeof(Small) + 1024;   // + alignment slack

constexpr uint32_t TM_O = 0;           // O^T tile t at columns 64t
constexpr uint32_t TM_S = 256;         // S buffer b, latent half k at 256 + 64b + 32k
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_S = tc::idesc(64, BN, 1, 1, false, false);
constexpr uint32_t ID_PV = tc::idesc(128, HP, 1, 1, true, false);

__device__ __forceinline__ uint32_t swz(int row, int unit) { return (uint32_t)(row * 128 + ((unit ^ (row & 7)) << 4)); }

// 2^x on the SFU (ex2.approx.ftz: relative error near 2^-22; -inf -> +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void fail(Small& sm, int32_t* status) {
    sm.abort = 1;
    set_status(status, KPOOL_ERR_TIMEOUT);
}

// Named barrier 2 over the 128 softmax threads that also ORs a predicate:
// every thread gets the same answer, so decisions taken on it stay uniform.
__device__ __forceinline__ bool wg_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Warp-uniform bounded wait: lane 0 polls, every lane gets the answer.
__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(addr, parity, abort) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

}  // namespace

__global__ void __launch_bounds__(THREADS, 1) sparse_mla_tc_kernel(const uint16_t* __restrict__ q_lat,
                                                                  const uint16_t* __restrict__ kv_lat,
                                                                  const int32_t* __restrict__ indices, int W, int T,
                                                                  int H, float scale_log2,
                                                                  uint16_t* __restrict__ out,
                                                                  float* __restrict__ lse, int32_t* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    Small& sm = *reinterpret_cast<Small*>(smem + OFF_SMALL);
    const uint32_t s_base = tc::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &sm.abort;

    if (tid == 0) {
        tc::mbar_init(tc::smem_u32(&sm.q_full), NPROD * 32 + 1);      // every producer lane's copies + nb
        tc::mbar_init(tc::smem_u32(&sm.q_empty), 4);      // two S issuers, PV issuer, softmax
        tc::mbar_init(tc::smem_u32(&sm.o_full), 1);
        tc::mbar_init(tc::smem_u32(&sm.o_free), 4);
        tc::mbar_init(tc::smem_u32(&sm.drain), 3);
        for (int s = 0; s < NSTAGE; ++s) {
            tc::mbar_init(tc::smem_u32(&sm.kv_full[s]), NPROD * 32 + NPROD);   // copies + masks
            tc::mbar_init(tc::smem_u32(&sm.kv_empty[s]), 3);   // two S issuers + PV issuer
        }
        for (int b = 0; b < NSB; ++b) {
            tc::mbar_init(tc::smem_u32(&sm.s_full[b]), 2);     // both halves of S
            tc::mbar_init(tc::smem_u32(&sm.s_free[b]), 4);
            tc::mbar_init(tc::smem_u32(&sm.p_full[b]), 4);
            tc::mbar_init(tc::smem_u32(&sm.p_empty[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.o_step[b]), 1);
        }
        sm.abort = 0;
        tc::mbar_init_fence();
    }
    if (warp == 8) tc::tmem_alloc(tc::smem_u32(&sm.tmem), TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp < NPROD) {
        // ===================================================== producers
        // Warp w copies Q rows 16w..16w+15 and rows 8w..8w+7 of every block;
        // lane l copies 16-byte units l and 32+l of a row.
        uint32_t g = 0;                             // global block counter
        uint32_t qn = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < T && ok; i += gridDim.x, ++qn) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int32_t* irow = indices + (int64_t)i * W;
            // last valid slot of the row (entries outside [-1, T) are flagged and skipped)
            int last = -1;
            for (int j = lane; j < W; j += 32) {
                const int v = irow[j];
                if (v >= 0 && v < T) last = j;
                else if (v != -1 && warp == 0) set_status(status, KPOOL_ERR_INDEX_RANGE);
            }
            for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
            const int nb = (last + BN) / BN;
            // Q tile: the previous query's S MMAs and every reader of nb must be done
            if (!warp_wait(tc::smem_u32(&sm.q_empty), (qn & 1) ^ 1, abort_flag)) { ok = false; break; }
            const uint16_t* qsrc = q_lat + (int64_t)i * H * D_LAT;
#pragma unroll 2
            for (int rr = 0; rr < HP / NPROD; ++rr) {
                const int row = warp * (HP / NPROD) + rr;
                const bool v = row < H;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int u = k * 32 + lane;
                    tc::cp_async16(s_base + OFF_Q + (u >> 3) * Q_CHUNK + swz(row, u & 7),
                                   v ? (const void*)(qsrc + row * D_LAT + u * 8) : (const void*)q_lat, v);
                }
            }
            tc::cp_async_arrive_noinc(tc::smem_u32(&sm.q_full));
            if (warp == 0 && lane == 0) {
                sm.nb = nb;
                tc::mbar_arrive(tc::smem_u32(&sm.q_full));
            }
            for (int b = 0; b < nb; ++b, ++g) {
                const int s = g % NSTAGE;
                if (!warp_wait(tc::smem_u32(&sm.kv_empty[s]), ((g / NSTAGE) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                int myv = -1;                       // lane l < 8: slot 8w + l of the block
                if (lane < 8) {
                    const int slot = b * BN + warp * 8 + lane;
                    const int v = slot < W ? irow[slot] : -1;
                    myv = (v >= 0 && v < T) ? v : -1;
                }
                const uint32_t m8 = __ballot_sync(0xffffffffu, myv >= 0) & 0xffu;
                const uint32_t dst = s_base + OFF_KV + s * KV_BYTES;
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int row = warp * 8 + rr;
                    const int v = __shfl_sync(0xffffffffu, myv, rr);
                    const bool valid = v >= 0;
                    const uint16_t* src = valid ? kv_lat + (int64_t)v * D_LAT : kv_lat;
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int u = k * 32 + lane;          // one instruction = 512 contiguous bytes
                        tc::cp_async16(dst + (u >> 3) * KV_CHUNK + swz(row, u & 7), src + (valid ? u * 8 : 0), valid);
                    }
                }
                tc::cp_async_arrive_noinc(tc::smem_u32(&sm.kv_full[s]));
                if (lane == 0) {
                    sm.mask[s][warp] = (uint8_t)m8;
                    tc::mbar_arrive(tc::smem_u32(&sm.kv_full[s]));
                }
            }
        }
        tc::cp_async_wait<0>();
        if (!ok) fail(sm, status);
    } else if (warp == 8 || warp == 9) {
        // ===================================================== S issuers (latent half = warp - 8)
        const int half = warp - 8;
        if (lane == 0) {
            uint32_t g = 0, qn = 0;
            const uint32_t q_addr = s_base + OFF_Q;
            bool ok = true;
            for (int i = blockIdx.x; i < T && ok && !*abort_flag; i += gridDim.x, ++qn) {
                if (!tc::mbar_wait(tc::smem_u32(&sm.q_full), qn & 1, abort_flag)) { ok = false; break; }
                tc::fence_proxy_async();                // Q was written by cp.async (generic proxy)
                const int nb = sm.nb;
                if (nb == 0) {
                    tc::commit(tc::smem_u32(&sm.q_empty));
                    continue;
                }
                const uint64_t a0 = tc::sw128_desc(q_addr + half * 4 * Q_CHUNK, 0, 1024);
                for (int b = 0; b < nb; ++b, ++g) {
                    const int s = g % NSTAGE, sb = g % NSB;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.kv_full[s]), (g / NSTAGE) & 1, abort_flag) ||
                        !tc::mbar_wait(tc::smem_u32(&sm.s_free[sb]), ((g / NSB) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::fence_proxy_async();            // the block was written by cp.async
                    tc::fence_after();
                    const uint64_t b0 = tc::sw128_desc(s_base + OFF_KV + s * KV_BYTES + half * 4 * KV_CHUNK, 0, 1024);
                    const uint32_t d = tmem + TM_S + 64 * sb + 32 * half;
#pragma unroll
                    for (int kl = 0; kl < D_LAT / 32; ++kl)      // K steps of 16 latent columns
                        tc::mma_bf16(d, a0 + (uint64_t)((kl >> 2) * (Q_CHUNK >> 4) + (kl & 3) * 2),
                                     b0 + (uint64_t)((kl >> 2) * (KV_CHUNK >> 4) + (kl & 3) * 2), ID_S,
                                     kl > 0 ? 1u : 0u);
                    tc::commit(tc::smem_u32(&sm.s_full[sb]));
                    tc::commit(tc::smem_u32(&sm.kv_empty[s]));
                    if (b == nb - 1) tc::commit(tc::smem_u32(&sm.q_empty));
                }
            }
            if (!ok) fail(sm, status);
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else if (warp == 10) {
        // ===================================================== PV issuer
        if (lane == 0) {
            uint32_t g = 0, qn = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < T && ok && !*abort_flag; i += gridDim.x, ++qn) {
                if (!tc::mbar_wait(tc::smem_u32(&sm.q_full), qn & 1, abort_flag)) { ok = false; break; }
                const int nb = sm.nb;
                tc::mbar_arrive(tc::smem_u32(&sm.q_empty));   // nb has been read
                for (int b = 0; b < nb; ++b, ++g) {
                    const int s = g % NSTAGE, sb = g % NSB;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.p_full[sb]), (g / NSB) & 1, abort_flag) ||
                        (b == 0 && !tc::mbar_wait(tc::smem_u32(&sm.o_free), (qn & 1) ^ 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc::fence_proxy_async();
                    tc::fence_after();
                    const uint64_t a0 = tc::sw128_desc(s_base + OFF_KV + s * KV_BYTES, KV_CHUNK, 1024);
                    const uint64_t b0 = tc::sw128_desc(s_base + OFF_P + sb * P_BYTES, 0, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            tc::mma_bf16(tmem + TM_O + 64 * t,
                                         a0 + (uint64_t)(((2 * t) * KV_CHUNK + kk * 2048) >> 4),
                                         b0 + (uint64_t)(kk * 2), ID_PV, (b == 0 && kk == 0) ? 0u : 1u);
                    tc::commit(tc::smem_u32(&sm.kv_empty[s]));
                    tc::commit(tc::smem_u32(&sm.p_empty[sb]));
                    tc::commit(tc::smem_u32(&sm.o_step[sb]));
                }
                if (!ok) break;
                tc::commit(tc::smem_u32(&sm.o_full));      // once per query, also for an empty row
            }
            if (!ok) fail(sm, status);
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ===================================================== softmax / correction / epilogue
        // Row h = 16*wid + (lane & 15) (head); lane half hs = lane >> 4 owns
        // slots 16*hs .. 16*hs+15 of the block.  `bad` is sticky per thread and
        // ORed across the four warps at every named barrier (bar.red.or).
        const int wid = warp - 4;                   // TMEM subpartition
        const int hs = lane >> 4;
        const int h = wid * 16 + (lane & 15);       // head of this thread
        const uint32_t lane_base = (uint32_t)(wid * 32) << 16;
        uint32_t g = 0, qn = 0;
        bool bad = false;
        for (int i = blockIdx.x; i < T; i += gridDim.x, ++qn) {
            bad = bad || !warp_wait(tc::smem_u32(&sm.q_full), qn & 1, abort_flag);
            if (wg_or(bad)) { bad = true; break; }
            const int nb = sm.nb;
            wg_or(false);                           // every warp has read nb
            if (tid == 128) tc::mbar_arrive(tc::smem_u32(&sm.q_empty));
            float m_ref = -INFINITY, l = 0.f;       // m_ref equal in both lanes of a row; l partial
            for (int b = 0; b < nb; ++b, ++g) {
                const int s = g % NSTAGE, sb = g % NSB;
                const int cb = g & 1;
                float x[16];
                bad = bad || !warp_wait(tc::smem_u32(&sm.s_full[sb]), (g / NSB) & 1, abort_flag);
                if (!bad) {
                    tc::fence_after();
                    // lanes 0-15 hold whole rows: keep slots 0-15, hand slots 16-31 to lane + 16
                    uint32_t va[32], vb[32];
                    tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sb, va);
                    tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sb + 32, vb);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float lo = __uint_as_float(va[j]) + __uint_as_float(vb[j]);
                        const float hi = __uint_as_float(va[16 + j]) + __uint_as_float(vb[16 + j]);
                        const float up = __shfl_sync(0xffffffffu, hi, lane & 15);
                        x[j] = hs ? up : lo;
                    }
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.s_free[sb]));
                    bad = !warp_wait(tc::smem_u32(&sm.kv_full[s]), (g / NSTAGE) & 1, abort_flag);
                }
                const uint32_t mask =
                    bad ? 0u : ((*reinterpret_cast<volatile uint32_t*>(&sm.mask[s][0]) >> (16 * hs)) & 0xffffu);
                const float thr = m_ref + TAU;        // -inf for a row that has seen no valid slot yet
                bool exceed = false;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    x[j] = ((mask >> j) & 1u) ? x[j] * scale_log2 : -INFINITY;
                    exceed |= x[j] > thr;
                }
                // common case: no running max moves, one barrier per block
                if (wg_or(bad || exceed)) {
                    if (wg_or(bad)) { bad = true; break; }
                    float bmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, x[j]);
                    bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 16));
                    float alpha = 1.f;
                    bool need = false;
                    if (bmax > m_ref + TAU) {
                        if (m_ref != -INFINITY) {          // O^T holds this head's earlier slots
                            alpha = fast_exp2(m_ref - bmax);
                            l *= alpha;
                            need = true;
                        }
                        m_ref = bmax;
                    }
                    if (hs == 0) sm.alpha[cb][h] = alpha;
                    if (wg_or(need)) {
                        // O^T must hold the previous block's PV before it is rescaled
                        const uint32_t gp = g - 1;
                        bad = !warp_wait(tc::smem_u32(&sm.o_step[gp % NSB]), (gp / NSB) & 1, abort_flag);
                        if (!bad) {
                            tc::fence_after();
                            for (int t = 0; t < 4; ++t)
                                for (int c0 = 0; c0 < HP; c0 += 32) {
                                    uint32_t o[32];
                                    const uint32_t ta = tmem + lane_base + TM_O + 64 * t + c0;
                                    tc::tmem_ld32(ta, o);
                                    tc::tmem_wait_ld();
#pragma unroll
                                    for (int j = 0; j < 32; ++j)
                                        o[j] = __float_as_uint(__uint_as_float(o[j]) * sm.alpha[cb][c0 + j]);
                                    tc::tmem_st32(ta, o);
                                }
                            tc::tmem_wait_st();
                            tc::fence_before();
                        }
                    }
                }
                // P^T row h, slots 16*hs .. 16*hs+15: 32 bytes, 16-byte units 2hs, 2hs+1
                bad = bad || !warp_wait(tc::smem_u32(&sm.p_empty[sb]), ((g / NSB) & 1) ^ 1, abort_flag);
                if (!bad) {
                    uint32_t pk[8];
                    float ps = 0.f;
                    const bool live = m_ref != -INFINITY;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float p0 = live ? fast_exp2(x[j] - m_ref) : 0.f;
                        const float p1 = live ? fast_exp2(x[j + 1] - m_ref) : 0.f;
                        ps += p0 + p1;
                        pk[j >> 1] = pack_bf16(p0, p1);
                    }
                    l += ps;
                    uint8_t* prow = smem + OFF_P + sb * P_BYTES;
                    *reinterpret_cast<uint4*>(prow + swz(h, 2 * hs)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(prow + swz(h, 2 * hs + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    tc::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.p_full[sb]));
                }
            }
            if (wg_or(bad)) { bad = true; break; }
            // ---- epilogue: O^T / l -> bf16 out, lse
            bad = !warp_wait(tc::smem_u32(&sm.o_full), qn & 1, abort_flag);
            const float lt = l + __shfl_xor_sync(0xffffffffu, l, 16);
            if (hs == 0) {
                sm.inv_l[h] = lt > 0.f ? 1.f / lt : 0.f;
                if (h < H)
                    lse[(int64_t)i * H + h] = lt > 0.f ? (m_ref + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
            }
            if (wg_or(bad)) { bad = true; break; }
            tc::fence_after();
            uint16_t* orow = out + (int64_t)i * H * D_LAT;
            uint8_t* stg = smem + OFF_P + wid * (HP * 64);        // [64 heads][32 latent] bf16
            for (int t = 0; t < 4; ++t) {
                for (int c0 = 0; c0 < HP; c0 += 32) {
                    uint32_t o[32];
                    if (nb > 0) {
                        tc::tmem_ld32(tmem + lane_base + TM_O + 64 * t + c0, o);
                        tc::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float val = __uint_as_float(o[j]) * sm.inv_l[c0 + j];
                        reinterpret_cast<__nv_bfloat16*>(stg + (c0 + j) * 64)[lane] = __float2bfloat16_rn(val);
                    }
                }
                __syncwarp();
                // 64 heads x 64 B: 16-byte stores, 8 per lane
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int cidx = k * 32 + lane;        // 0..255
                    const int hh = cidx >> 2, part = cidx & 3;
                    if (hh < H) {
                        const uint4 val = *reinterpret_cast<const uint4*>(stg + hh * 64 + part * 16);
                        *reinterpret_cast<uint4*>(orow + hh * D_LAT + t * 128 + wid * 32 + part * 8) = val;
                    }
                }
                __syncwarp();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.o_free));
            wg_or(false);                           // inv_l and the staging tile are reused next query
        }
        if (bad) fail(sm, status);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 8) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, TM_COLS);
    }
}

int launch_sparse_mla(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int T,
                      int n_heads, float scale, uint16_t* out, float* lse, int32_t* status, cudaStream_t stream) {
    if (T <= 0) return KPOOL_OK;
    if (n_heads < 1 || n_heads > HP) return KPOOL_ERR_SHAPE;
    static int n_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    if (n_sm[dev] == 0) {
        if (cudaFuncSetAttribute(sparse_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
            cudaSuccess)
            return KPOOL_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KPOOL_ERR_CUDA;
        n_sm[dev] = sms;
    }
    const int grid = T < n_sm[dev] ? T : n_sm[dev];
    const float scale_log2 = scale * 1.4426950408889634f;
    sparse_mla_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(q_lat, kv_lat, indices, W, T, n_heads, scale_log2,
                                                               out, lse, status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
