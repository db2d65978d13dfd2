// Sparse latent attention forward (absorbed NoPE MLA over index rows), tcgen05.
//
// NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog: the K
// projection is absorbed into the query and attention runs over the shared
// 512-wide latent, which is both key and value; the caller applies the V
// projection afterwards.  miles "GLM-5.3-Flash" recipe, section 1: NoPE MLA,
// 64 heads.
//
// Persistent CTAs (one per SM), each walking query tokens i = blockIdx.x +
// k*gridDim.x.  For one query the index row is cut into blocks of 64 slots:
//   S   = Q Kv^T      tcgen05 kind::f16, M = 64 heads, N = 64 slots, K = 512,
//                     split over two issuing warps by latent half; A (Q) is
//                     read from TMEM, B (the gathered block) from shared memory
//   O^T += Kv^T P^T   tcgen05 kind::f16, M = 128 latent rows (4 tiles),
//                     N = 64 heads, K = 64 slots; A is the gathered block read
//                     MN-major, so the tile that fed S also feeds PV
// TMEM, 512 columns x 128 lanes:
//   columns   0-255  O^T, tile t at columns 64t (all lanes)
//   columns 256-383  Q.  An M=64 operand row r lives in lane 32*(r/16) + r%16
//                    of subpartition r/16; latent half 0 of every head sits in
//                    those lanes, latent half 1 in the 16 lanes above them.  An
//                    M=64 MMA with A in TMEM reads A from the lane half its D is
//                    written to, so each half of the K sum stays in its half.
//   columns 384-511  S, two buffers of 64 columns; K half k in lane half k
// Shared memory holds a 3-stage ring of 64 KB gathered blocks and two P^T tiles.
//
// The latent gather from L2 (about 1 KB per slot, shared by nothing across
// queries) and the MMA chain of a block bound this kernel.  Eight producer warps keep many
// 16-byte cp.async in flight; each lane's copies arrive on the stage's
// mbarrier when they land (cp.async.mbarrier.arrive.noinc), so no producer
// ever waits for a copy, and the MMA issuers take a proxy fence before
// reading the tile.  The producers also move each query's Q from global memory
// into TMEM (tcgen05.st) once the previous query's S MMAs are done; they start
// the gathers of the new query's first blocks before that and prefetch the
// next query's Q into L2, so a query boundary does not drain the ring.
//
// Warp roles (512 threads, per-warpgroup register budgets set with setmaxnreg):
//   warps 0-3, 12-15  eight producers: rows 8g..8g+7 of every block for gather
//              warp g (0-3 -> g = w, 12-15 -> g = w-8); and the Q rows of TMEM
//              subpartition w%4, warps 0-3 latent columns 0-127, warps 12-15
//              columns 128-255 of each half
//   warps 4-7  softmax: lane l < 16 loads the K-half-0 row of head 16w+l and
//              lane l+16 the K-half-1 row; a half-row exchange between the two
//              leaves lane l with slots 0-31 and lane l+16 with slots 32-63 of
//              the summed row.  The running max only moves when a slot beats it
//              by more than 2^8; each warp decides that for its own heads, with
//              no barrier between the four.  A move of a max that O^T already
//              depends on raises a flag that the PV issuer reads with the P^T
//              tile: it then asks the four warps (served inside their waits) to
//              rescale O^T after the previous PV and only then issues this one.
//              When every
//              slot of the warp's half-blocks is valid (all but a row's last
//              block), the test runs on the unscaled block max and the scale is
//              fused into the exponent's FMA.  P^T goes to
//              shared memory in the operand layout; the epilogue writes O^T / l
//              as bf16 straight from TMEM, both 32-column halves of a tile
//              loaded under one wait (lane pairs swap values so that every
//              store covers two 64-byte runs of output rows), and releases
//              O^T to the next query's PV once its last tile is in registers.
//              1/l is kept per query parity, so a query needs two named
//              barriers (its start and the end of its blocks).
//   warps 8-9  S issuers (warp 8 also owns the TMEM allocation)
//   warp 10    PV issuer
//   warp 11    row scanner: block count and range check of each query's
//              index row, two queries ahead of the producers (with one query
//              per CTA, as in a decode step, nothing hides the scan: the
//              ONE_QUERY instance reads the row with 16-byte loads)
// Every wait is bounded and warp-uniform (lane 0 polls, the warp takes its
// answer); on expiry the kernel records KPOOL_ERR_TIMEOUT, the softmax warps
// agree on stopping at the next query-level named barrier, every role leaves its loop,
// in-flight copies and MMAs are drained and TMEM is freed.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"
#include "tc_ptx.cuh"

namespace kpool {

namespace {

constexpr int BN = 64;                 // slots per block
constexpr int NSTAGE = 3;              // latent-row ring depth
constexpr int NSB = 2;                 // S / P double buffers
constexpr int HP = 64;                 // head rows (M of S, N of PV)
constexpr float TAU = 8.0f;            // lazy-rescale threshold (log2 units)
constexpr int THREADS = 512;
constexpr int NPROD = 4;               // producer warps that also load Q (warps 0-3)
constexpr int NGATH = 8;               // gather warps: 0-3 and 12-15
constexpr int ROWS_PER_PROD = BN / NGATH;

constexpr int KV_BYTES = BN * D_LAT * 2;         // 64 KB: 8 chunks x [64 rows x 128 B]
constexpr int KV_CHUNK = BN * 128;               // 8 KB
constexpr int P_BYTES = HP * 128;                // 8 KB: [64 head rows x 128 B] = 64 slots

constexpr int OFF_KV = 0;
constexpr int OFF_P = OFF_KV + NSTAGE * KV_BYTES;        // 2 P^T buffers
constexpr int OFF_SMALL = OFF_P + NSB * P_BYTES;

struct Small {
    uint64_t q_full, q_empty, o_full, o_free, drain;
    uint64_t kv_full[NSTAGE], kv_empty[NSTAGE];
    uint64_t s_full[NSB], s_free[NSB], p_full[NSB], p_empty[NSB], o_step[NSB];
    uint64_t nb_full[2], nb_empty[2];           // row-scan results, two queries deep
    alignas(8) uint8_t mask[NSTAGE][NGATH];    // valid-slot bits, 8 slots per gather warp
    int nbq[2];                                 // blocks of the scanned query (ring)
    int nb;
    int abort;
    uint32_t tmem;
    float alpha[2][HP];
    uint64_t resc_done;                         // the softmax warps have rescaled O^T for a request
    uint8_t resc_flag[NSB][4];                  // per P buffer: softmax warp w raised a head's max
    uint32_t resc_mask;                         // flags of the outstanding request
    int resc_g;                                 // block of the outstanding request
    int resc_seq;                               // requests issued so far
    alignas(16) float inv_l[2][HP];             // per query parity: 1/l of every head
};
constexpr int SMEM_BYTES = OFF_SMALL + (int)sizeof(Small) + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

constexpr uint32_t TM_O = 0;           // O^T tile t at columns 64t
constexpr uint32_t TM_Q = 256;         // Q, K step kl (16 latent) at 256 + 8kl, lane half = latent half
constexpr uint32_t TM_S = 384;         // S buffer b at 384 + 64b, lane half = latent half of the sum
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

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];\n" : "=r"(v) : "r"(tc::smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;\n" ::"r"(tc::smem_u32(p)), "r"(v) : "memory");
}

// Per-warpgroup register budgets (launch: 512 threads x 128).  Shares: the two
// producer warpgroups 104 each, softmax 168, issuers and row scanner 80 (sum 456).
template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }

// Warp-uniform bounded wait: lane 0 polls, every lane gets the answer.
__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(addr, parity, abort) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Nonzero: the next launches stall their row scanner on a barrier that cannot
// complete before the kernel aborts (test of the bounded waits; set with
// set_sparse_mla_stall).
__device__ int g_sparse_mla_stall = 0;

// A rescale request of the PV issuer: multiply the O^T columns of the heads whose running max moved
// (the flagged warps' heads; the others by 1) by their factors, once the previous block's PV has landed.
// Every softmax warp serves it on its 32 lanes (tm = the warp's TMEM lane base); the PV issuer waits
// for all four.
__device__ __forceinline__ bool serve_rescale(Small& sm, uint32_t tm, const volatile int* abort_flag) {
    const int gr = *reinterpret_cast<volatile int*>(&sm.resc_g);
    const uint32_t fm = *reinterpret_cast<volatile uint32_t*>(&sm.resc_mask);
    const uint32_t gp = (uint32_t)gr - 1u;
    if (!warp_wait(tc::smem_u32(&sm.o_step[gp % NSB]), (gp / NSB) & 1, abort_flag)) return false;
    tc::fence_after();
    const float* al = sm.alpha[gr % NSB];
    for (int t = 0; t < 4; ++t)
        for (int c0 = 0; c0 < HP; c0 += 32) {
            uint32_t o[32];
            const uint32_t ta = tm + TM_O + 64 * t + c0;
            tc::tmem_ld32(ta, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int c = c0 + j;
                const float f = ((fm >> (8 * (c >> 4))) & 1u) ? al[c] : 1.f;
                o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            }
            tc::tmem_st32(ta, o);
        }
    tc::tmem_wait_st();
    tc::fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(tc::smem_u32(&sm.resc_done));
    return true;
}

}  // namespace

int set_sparse_mla_stall(int on) {
    const int v = on ? 1 : 0;
    return cudaMemcpyToSymbol(g_sparse_mla_stall, &v, sizeof(v)) == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

template <bool ONE_QUERY>
__global__ void __launch_bounds__(THREADS, 1) sparse_mla_tc_kernel(const uint16_t* __restrict__ q_lat,
                                                                  const uint16_t* __restrict__ kv_lat,
                                                                  const int32_t* __restrict__ indices, int W,
                                                                  int n_rows, int T, int H, float scale_log2,
                                                                  uint16_t* __restrict__ out,
                                                                  float* __restrict__ lse, int32_t* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    Small& sm = *reinterpret_cast<Small*>(smem + OFF_SMALL);
    const uint32_t s_base = tc::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &sm.abort;
    // The first query's Q and the index rows of the first two queries into L2 before anything else (the
    // in-loop prefetches run ahead of later queries only).  With one query per CTA (a decode step) nothing
    // else hides their HBM latency: the row scan waits on the row and the Q store on 16 scattered loads per
    // producer lane.
    if (tid == 32 * 11) {
        const int i0 = blockIdx.x;
        tc::prefetch_l2(q_lat + (int64_t)i0 * H * D_LAT, (uint32_t)(H * D_LAT * 2));
        if ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(indices) & 15u) == 0) {
            tc::prefetch_l2(indices + (int64_t)i0 * W, (uint32_t)W * 4u);
            if (i0 + (int)gridDim.x < n_rows)
                tc::prefetch_l2(indices + (int64_t)(i0 + (int)gridDim.x) * W, (uint32_t)W * 4u);
        }
    }

    if (tid == 0) {
        tc::mbar_init(tc::smem_u32(&sm.q_full), NGATH);   // each producer warp: its Q columns stored (+ nb)
        tc::mbar_init(tc::smem_u32(&sm.q_empty), 7);      // two S issuers, PV issuer, four softmax warps
        tc::mbar_init(tc::smem_u32(&sm.o_full), 1);
        tc::mbar_init(tc::smem_u32(&sm.o_free), 4);
        tc::mbar_init(tc::smem_u32(&sm.drain), 3);
        for (int r = 0; r < 2; ++r) {
            tc::mbar_init(tc::smem_u32(&sm.nb_full[r]), 1);        // the row scanner
            tc::mbar_init(tc::smem_u32(&sm.nb_empty[r]), NGATH);   // every gather warp has read it
        }
        for (int s = 0; s < NSTAGE; ++s) {
            tc::mbar_init(tc::smem_u32(&sm.kv_full[s]), NGATH * 32 + NGATH);   // copies + masks
            tc::mbar_init(tc::smem_u32(&sm.kv_empty[s]), 3);   // two S issuers + PV issuer
        }
        for (int b = 0; b < NSB; ++b) {
            tc::mbar_init(tc::smem_u32(&sm.s_full[b]), 2);     // both halves of S
            tc::mbar_init(tc::smem_u32(&sm.s_free[b]), 4);
            tc::mbar_init(tc::smem_u32(&sm.p_full[b]), 4);
            tc::mbar_init(tc::smem_u32(&sm.p_empty[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.o_step[b]), 1);
        }
        tc::mbar_init(tc::smem_u32(&sm.resc_done), 4);
        *reinterpret_cast<uint32_t*>(&sm.resc_flag[0][0]) = 0u;
        *reinterpret_cast<uint32_t*>(&sm.resc_flag[1][0]) = 0u;
        sm.resc_seq = 0;
        sm.abort = 0;
        tc::mbar_init_fence();
    }
    if (warp == 8) tc::tmem_alloc(tc::smem_u32(&sm.tmem), TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp < NPROD || warp >= 12) {
        // ===================================================== producers (warps 0-3 also load Q)
        regs_dec<104>();
        const int gw = warp < NPROD ? warp : warp - 8;   // gather warp index 0..7
        const int qc0 = warp < NPROD ? 0 : 2;            // Q column blocks 2*gw/4.. of this warp
        // Warp w (subpartition w % 4): Q rows of heads 16(w%4)..16(w%4)+15, column blocks
        // qc0, qc0+1 (of 4), and rows 8gw..8gw+7 of every block; lane l copies 16-byte
        // units l and 32+l of a latent row.
        uint32_t g = 0;                             // global block counter
        uint32_t qn = 0;
        bool ok = true;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int qh = (warp & 3) * 16 + (lane & 15);   // head whose Q row this lane stores
        const int qhalf = lane >> 4;                // latent half it stores
        for (int i = blockIdx.x; i < n_rows && ok; i += gridDim.x, ++qn) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int32_t* irow = indices + (int64_t)i * W;
            // the row scanner's block count for this query
            if (!warp_wait(tc::smem_u32(&sm.nb_full[qn & 1]), (qn >> 1) & 1, abort_flag)) { ok = false; break; }
            const int nb = sm.nbq[qn & 1];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.nb_empty[qn & 1]));
            if (warp == 0 && lane == 0 && i + (int)gridDim.x < n_rows)
                tc::prefetch_l2(q_lat + (int64_t)(i + (int)gridDim.x) * H * D_LAT, (uint32_t)(H * D_LAT * 2));

            // Blocks 0 .. pre-1 need nothing from the previous query and go first;
            // at b == pre the query's Q is stored (after the previous query's S
            // MMAs are done).  Lane l < 16 holds the slot index of row 16w + l of
            // the block, loaded one block ahead.
            const int pre = nb < NSTAGE - 1 ? nb : NSTAGE - 1;
            auto slot_of = [&](int b) -> int {
                const int slot = b * BN + gw * ROWS_PER_PROD + lane;
                const int v = (lane < ROWS_PER_PROD && slot < W) ? irow[slot] : -1;
                return (v >= 0 && v < T) ? v : -1;
            };
            int nxt = nb > 0 ? slot_of(0) : -1;
            // this lane's Q row half (512 B), loaded before the first gathers so that
            // the load latency hides behind them; stored to TMEM at b == pre
            uint32_t qr[2][32];
            {
                const bool v = nb > 0 && qh < H;
                const uint4* qsrc = reinterpret_cast<const uint4*>(
                    q_lat + ((int64_t)i * H + (qh < H ? qh : 0)) * D_LAT + qhalf * (D_LAT / 2));
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 x = v ? __ldg(qsrc + (qc0 + c) * 8 + j) : make_uint4(0u, 0u, 0u, 0u);
                        qr[c][4 * j] = x.x;
                        qr[c][4 * j + 1] = x.y;
                        qr[c][4 * j + 2] = x.z;
                        qr[c][4 * j + 3] = x.w;
                    }
            }
            for (int b = 0; b <= nb; ++b) {
                if (b == pre) {
                    // Q: the previous query's S MMAs and every reader of nb must be done
                    if (!warp_wait(tc::smem_u32(&sm.q_empty), (qn & 1) ^ 1, abort_flag)) { ok = false; break; }
                    if (nb > 0) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) tc::tmem_st32(tmem + lane_base + TM_Q + 32 * (qc0 + c), qr[c]);
                        tc::tmem_wait_st();
                    }
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (warp == 0) sm.nb = nb;
                        tc::mbar_arrive(tc::smem_u32(&sm.q_full));
                    }
                }
                if (b == nb) break;
                const int myv = nxt;
                if (b + 1 < nb) nxt = slot_of(b + 1);
                const int s = g % NSTAGE;
                if (!warp_wait(tc::smem_u32(&sm.kv_empty[s]), ((g / NSTAGE) & 1) ^ 1, abort_flag)) { ok = false; break; }
                const uint32_t m8 = __ballot_sync(0xffffffffu, myv >= 0) & 0xffu;
                const uint32_t dst = s_base + OFF_KV + s * KV_BYTES;
#pragma unroll
                for (int rr = 0; rr < ROWS_PER_PROD; ++rr) {
                    const int row = gw * ROWS_PER_PROD + rr;
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
                    sm.mask[s][gw] = (uint8_t)m8;
                    tc::mbar_arrive(tc::smem_u32(&sm.kv_full[s]));
                }
                ++g;
            }
        }
        tc::cp_async_wait<0>();
        if (!ok) fail(sm, status);
    } else if (warp >= 8 && warp < 12) {
      regs_dec<80>();
      if (warp == 8 || warp == 9) {
        // ===================================================== S issuers (latent half = warp - 8)
        const int half = warp - 8;
        if (lane == 0) {
            uint32_t g = 0, qn = 0;
            const uint32_t lh = (uint32_t)(16 * half) << 16;    // lane half of this K half
            bool ok = true;
            for (int i = blockIdx.x; i < n_rows && ok && !*abort_flag; i += gridDim.x, ++qn) {
                if (!tc::mbar_wait(tc::smem_u32(&sm.q_full), qn & 1, abort_flag)) { ok = false; break; }
                tc::fence_after();                      // Q was stored with tcgen05.st
                const int nb = sm.nb;
                if (nb == 0) {
                    tc::commit(tc::smem_u32(&sm.q_empty));
                    continue;
                }
                const uint32_t a0 = tmem + lh + TM_Q;
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
                    const uint32_t d = tmem + lh + TM_S + 64 * sb;
#pragma unroll
                    for (int kl = 0; kl < D_LAT / 32; ++kl)      // K steps of 16 latent columns
                        tc::mma_bf16_ts(d, a0 + 8u * kl, b0 + (uint64_t)((kl >> 2) * (KV_CHUNK >> 4) + (kl & 3) * 2),
                                        ID_S, kl > 0 ? 1u : 0u);
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
            uint32_t g = 0, qn = 0, nreq = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_rows && ok && !*abort_flag; i += gridDim.x, ++qn) {
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
                    // a softmax warp raised a head's running max in this block: O^T is rescaled by the
                    // softmax warps (after the previous PV) before this PV adds to it
                    const uint32_t fl = *reinterpret_cast<volatile uint32_t*>(&sm.resc_flag[sb][0]);
                    if (fl != 0u) {
                        *reinterpret_cast<volatile uint32_t*>(&sm.resc_flag[sb][0]) = 0u;
                        sm.resc_mask = fl;
                        sm.resc_g = (int)g;
                        st_release(&sm.resc_seq, (int)++nreq);
                        if (!tc::mbar_wait(tc::smem_u32(&sm.resc_done), (nreq - 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
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
                // once per query, also for an empty row; an empty row still waits for the
                // previous epilogue so that o_full and o_free strictly alternate
                if (nb == 0 && !tc::mbar_wait(tc::smem_u32(&sm.o_free), (qn & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::commit(tc::smem_u32(&sm.o_full));
            }
            if (!ok) fail(sm, status);
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else if (warp == 11) {
        // ===================================================== row scanner
        // For each query of this CTA: the last valid slot of its index row
        // (entries outside [-1, T) are flagged and skipped) -> block count,
        // published up to two queries ahead of the producers; rows two queries
        // ahead are prefetched into L2.
        uint32_t qn = 0;
        // test hook: with a stall injected, first wait on the end-of-kernel barrier, which completes
        // only after the MMA issuers have left their loops, so the bounded waits of every role run out
        bool ok = g_sparse_mla_stall == 0 || warp_wait(tc::smem_u32(&sm.drain), 0, abort_flag);
        for (int i = blockIdx.x; i < n_rows && ok; i += gridDim.x, ++qn) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int r = qn & 1;
            if (!warp_wait(tc::smem_u32(&sm.nb_empty[r]), ((qn >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            const int64_t ahead = (int64_t)i + 2 * (int64_t)gridDim.x;
            if (lane == 0 && ahead < n_rows && (W & 3) == 0 && ((reinterpret_cast<uintptr_t>(indices) & 15u) == 0))
                tc::prefetch_l2(indices + ahead * W, (uint32_t)W * 4u);
            const int32_t* irow = indices + (int64_t)i * W;
            int last = -1;
            bool out_of_range = false;
            if (ONE_QUERY && (W & 3) == 0 && (reinterpret_cast<uintptr_t>(indices) & 15u) == 0) {
                // one query per CTA (a decode step): no scan runs ahead of it, so the scan is
                // exposed; 16-byte loads, eight in flight per lane
                const int4* irow4 = reinterpret_cast<const int4*>(irow);
#pragma unroll 8
                for (int j4 = lane; j4 < (W >> 2); j4 += 32) {
                    const int4 v4 = __ldg(irow4 + j4);
                    const int vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool valid = vv[e] >= 0 && vv[e] < T;
                        last = valid ? 4 * j4 + e : last;
                        out_of_range |= !valid && vv[e] != -1;
                    }
                }
            } else {
#pragma unroll 4
                for (int j = lane; j < W; j += 32) {
                    const int v = __ldg(irow + j);
                    const bool valid = v >= 0 && v < T;
                    last = valid ? j : last;
                    out_of_range |= !valid && v != -1;
                }
            }
            for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
            if (__any_sync(0xffffffffu, out_of_range) && lane == 0) set_status(status, KPOOL_ERR_INDEX_RANGE);
            if (lane == 0) {
                sm.nbq[r] = (last + BN) / BN;
                tc::mbar_arrive(tc::smem_u32(&sm.nb_full[r]));
            }
            __syncwarp();
        }
        if (!ok) fail(sm, status);
      }
    } else if (warp >= 4 && warp < 8) {
        // ===================================================== softmax / correction / epilogue
        regs_inc<168>();
        // Row h = 16*wid + (lane & 15) (head); lane half hs = lane >> 4 owns
        // slots 32*hs .. 32*hs+31 of the block.  `bad` is sticky per warp; a warp
        // that sees it leaves the block loop, and the four warps OR it at the
        // named barriers (bar.red.or) of every query's start and end.
        const int wid = warp - 4;                   // TMEM subpartition
        const int hs = lane >> 4;
        const int h = wid * 16 + (lane & 15);       // head of this thread
        const uint32_t lane_base = (uint32_t)(wid * 32) << 16;
        uint32_t g = 0, qn = 0;
        bool bad = false;
        int served = 0;                             // rescale requests this warp has served
        // Bounded wait of a softmax warp that serves rescale requests meanwhile (the awaited phase
        // can depend on the PV that a request holds back).
        auto sm_wait = [&](uint32_t addr, uint32_t parity) -> bool {
            const uint64_t t0 = tc::globaltimer_ns();
            for (uint32_t it = 0;; ++it) {
                uint32_t st = 0;
                if (lane == 0) {
                    st = tc::mbar_try(addr, parity) ? 1u : 0u;
                    if (!st && ld_acquire(&sm.resc_seq) != served) st = 2u;
                    if (!st && (it & 15u) == 15u && (*abort_flag || tc::globaltimer_ns() - t0 > tc::WAIT_LIMIT_NS))
                        st = 3u;
                }
                st = __shfl_sync(0xffffffffu, st, 0);
                if (st == 1u) return true;
                if (st == 3u) return false;
                if (st == 2u) {
                    if (!serve_rescale(sm, tmem + lane_base, abort_flag)) return false;
                    ++served;
                }
            }
        };
        for (int i = blockIdx.x; i < n_rows; i += gridDim.x, ++qn) {
            bad = bad || !warp_wait(tc::smem_u32(&sm.q_full), qn & 1, abort_flag);
            if (wg_or(bad)) { bad = true; break; }
            const int nb = sm.nb;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.q_empty));   // this warp has read nb
            float m_ref = -INFINITY, l = 0.f;       // m_ref equal in both lanes of a row; l partial
            for (int b = 0; b < nb; ++b, ++g) {
                const int s = g % NSTAGE, sb = g % NSB;
                float x[32];
                // P^T buffer free (PV of block g-2 done), then S of this block; both waits serve
                // rescale requests, as neither holds live values
                bad = bad || !sm_wait(tc::smem_u32(&sm.p_empty[sb]), ((g / NSB) & 1) ^ 1) ||
                      !sm_wait(tc::smem_u32(&sm.s_full[sb]), (g / NSB) & 1);
                if (bad) break;
                tc::fence_after();
                {
                    // lane l < 16 holds the K-half-0 row, lane l+16 the K-half-1 row of the
                    // same head; swap halves so that each keeps 32 slots of the sum
                    uint32_t va[32], vb[32];
                    tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sb, va);
                    tc::tmem_ld32(tmem + lane_base + TM_S + 64 * sb + 32, vb);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const uint32_t send = hs ? va[j] : vb[j];
                        const float recv = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
                        x[j] = __uint_as_float(hs ? vb[j] : va[j]) + recv;
                    }
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.s_free[sb]));
                // the block's valid-slot mask (S of the block was computed, so its copies have landed)
                bad = !warp_wait(tc::smem_u32(&sm.kv_full[s]), (g / NSTAGE) & 1, abort_flag);
                if (bad) break;
                const uint32_t mask = (uint32_t)(*reinterpret_cast<volatile uint64_t*>(&sm.mask[s][0]) >> (32 * hs));
                // every slot of the warp's half-blocks valid (all but a row's last block): x stays
                // unscaled, the exceed test runs on the block max (scaling by a positive factor
                // and rounding keep the order) and the scale is fused into the exponent's FMA
                const bool full = __all_sync(0xffffffffu, mask == 0xffffffffu) && scale_log2 > 0.f;
                if (!full) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = ((mask >> j) & 1u) ? x[j] * scale_log2 : -INFINITY;
                }
                float t16[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) t16[j] = fmaxf(x[j], x[j + 16]);
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int j = 0; j < w; ++j) t16[j] = fmaxf(t16[j], t16[j + w]);
                const float lmax = full ? t16[0] * scale_log2 : t16[0];
                // the running max of a head moves only when a slot beats it by more than 2^TAU
                // (-inf until the row's first valid slot); the warp decides alone, and a move of a
                // max that O^T already depends on is passed to the PV issuer as a rescale request
                float alpha = 1.f;
                bool need = false;
                if (__any_sync(0xffffffffu, lmax > m_ref + TAU)) {
                    const float bmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, 16));
                    if (bmax > m_ref + TAU) {
                        if (m_ref != -INFINITY) {          // O^T holds this head's earlier slots
                            alpha = fast_exp2(m_ref - bmax);
                            l *= alpha;
                            need = true;
                        }
                        m_ref = bmax;
                    }
                }
                const bool warp_need = __any_sync(0xffffffffu, need);
                // P^T row h, slots 32*hs .. 32*hs+31: 64 bytes, 16-byte units 4hs .. 4hs+3
                if (warp_need) {
                    if (hs == 0) sm.alpha[sb][h] = alpha;
                    if (lane == 0) sm.resc_flag[sb][wid] = 1;
                }
                {
                    uint32_t pk[16];
                    float2 ps[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    const bool live = m_ref != -INFINITY;
                    if (full) {
                        const float nm = -m_ref;
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float2 p = make_float2(fast_exp2(fmaf(x[j], scale_log2, nm)),
                                                         fast_exp2(fmaf(x[j + 1], scale_log2, nm)));
                            ps[(j >> 1) & 1] = __fadd2_rn(ps[(j >> 1) & 1], p);
                            pk[j >> 1] = pack_bf16(p.x, p.y);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float2 p = make_float2(live ? fast_exp2(x[j] - m_ref) : 0.f,
                                                         live ? fast_exp2(x[j + 1] - m_ref) : 0.f);
                            ps[(j >> 1) & 1] = __fadd2_rn(ps[(j >> 1) & 1], p);
                            pk[j >> 1] = pack_bf16(p.x, p.y);
                        }
                    }
                    l += (ps[0].x + ps[1].x) + (ps[0].y + ps[1].y);
                    uint8_t* prow = smem + OFF_P + sb * P_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(prow + swz(h, 4 * hs + k)) =
                            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    tc::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.p_full[sb]));
                }
            }
            if (wg_or(bad)) { bad = true; break; }
            // ---- epilogue: O^T / l -> bf16 out, lse
            bad = !sm_wait(tc::smem_u32(&sm.o_full), qn & 1);
            const float lt = l + __shfl_xor_sync(0xffffffffu, l, 16);
            if (hs == 0) {
                sm.inv_l[qn & 1][h] = lt > 0.f ? 1.f / lt : 0.f;
                if (h < H)
                    lse[(int64_t)i * H + h] = lt > 0.f ? (m_ref + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
            }
            if (wg_or(bad)) { bad = true; break; }
            tc::fence_after();
            // Thread (subpartition wid, lane l) holds latent row 128t + 32wid + l of O^T
            // tile t for every head.  Lanes l and l^1 swap one value per head pair so
            // that the even lane writes latent pair (l, l+1) of head 2p and the odd
            // lane the same pair of head 2p+1: one 4-byte store each, and every store
            // instruction covers two 64-byte runs of the output rows.
            uint16_t* orow = out + (int64_t)i * H * D_LAT;
            const int odd = lane & 1;
#pragma unroll 1
            for (int t = 0; t < 4; ++t) {
                const int d = t * 128 + wid * 32 + (lane & ~1);
                // both 32-column halves of the tile in flight under one wait
                uint32_t o[2][32];
                if (nb > 0) {
                    tc::tmem_ld32(tmem + lane_base + TM_O + 64 * t, o[0]);
                    tc::tmem_ld32(tmem + lane_base + TM_O + 64 * t + 32, o[1]);
                    tc::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[0][j] = o[1][j] = 0u;
                }
                if (t == 3) {                        // O^T is read: the next query's PV may start
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.o_free));
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int c0 = 32 * hf;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 il = *reinterpret_cast<const float2*>(&sm.inv_l[qn & 1][c0 + j]);
                        const float a = __uint_as_float(o[hf][j]) * il.x;
                        const float b = __uint_as_float(o[hf][j + 1]) * il.y;
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
                        const uint32_t w = odd ? pack_bf16(recv, b) : pack_bf16(a, recv);
                        const int hh = c0 + j + odd;
                        if (hh < H) *reinterpret_cast<uint32_t*>(orow + hh * D_LAT + d) = w;
                    }
                }
            }
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

int launch_sparse_mla(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int n_rows,
                      int T, int n_heads, float scale, uint16_t* out, float* lse, int32_t* status,
                      cudaStream_t stream) {
    if (n_rows <= 0) return KPOOL_OK;
    if (n_heads < 1 || n_heads > HP) return KPOOL_ERR_SHAPE;
    static int n_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    if (n_sm[dev] == 0) {
        if (cudaFuncSetAttribute(sparse_mla_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(sparse_mla_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return KPOOL_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KPOOL_ERR_CUDA;
        n_sm[dev] = sms;
    }
    const int grid = n_rows < n_sm[dev] ? n_rows : n_sm[dev];
    const float scale_log2 = scale * 1.4426950408889634f;
    if (n_rows <= n_sm[dev])                          // one query per CTA
        sparse_mla_tc_kernel<true><<<grid, THREADS, SMEM_BYTES, stream>>>(q_lat, kv_lat, indices, W, n_rows, T,
                                                                          n_heads, scale_log2, out, lse, status);
    else
        sparse_mla_tc_kernel<false><<<grid, THREADS, SMEM_BYTES, stream>>>(q_lat, kv_lat, indices, W, n_rows, T,
                                                                           n_heads, scale_log2, out, lse, status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
