// Sparse latent attention backward (absorbed NoPE MLA over index rows), tcgen05.
//
// NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog and
// section "cuDNN sparse MLA parity and performance": the same latent sparse
// attention runs forward and backward in training (dQ and dKV are the
// gradients that section compares).  The 512-wide latent row is both key and
// value, so its gradient sums a value term and a key term.  Per query i, head
// h, over the valid slots j of the row (lse and delta = dout . out saved from
// the forward):
//   P    = exp(scale * Q Kv^T - lse)           dP = dO Kv^T
//   dZ'  = scale * P * (dP - delta)
//   dQ   = dZ' Kv                               (accumulated over the row)
//   dKv  = P^T dO + dZ'^T Q                     (scattered to kv rows idx_j)
//
// Persistent CTAs walk queries i = blockIdx.x + k*gridDim.x; each query's row
// is cut into blocks of 32 slots, gathered into a two-stage ring, and pairs of
// blocks share one P / dZ' tile.  On the tensor pipe (kind::f16):
//   [S; dP]    per block: M = 128, N = 32 slots, K = 512.  A stacks Q and dO:
//              in every 32-row group w, rows 0-15 are the Q rows and rows 16-31
//              the dO rows of heads 16w .. 16w+15, so TMEM lane l < 16 of
//              subpartition w gets the S row and lane l + 16 the dP row of
//              the same head
//   dQ^T      += Kv^T dZ'^T   per block: M = 128 latent rows (4 tiles),
//              N = 64 heads, K = 32 slots (A = the block read MN-major); the
//              block's ring stage is free after these
//   dKv^T      = dO^T P + Q^T dZ'   per pair: M = 128 latent rows, one tile at
//              a time, N = 64 slots, K = 64 heads (A = the dO / Q rows of the
//              stacked operand read MN-major, B = the pair's P / dZ' tile read
//              MN-major); tiles alternate between two TMEM buffers
// TMEM (512 columns): dQ^T 0-255, dKv^T tile buffers 256-319 / 320-383,
// [S; dP] buffers 384-415 / 416-447.
// Shared memory: the stacked Q / dO operand (128 KB, 128-byte swizzled,
// K-major, also read MN-major), two 32 KB gathered blocks, and two pair
// tiles of P and dZ' [64 heads x 64 slots] (32 KB).
//
// dKv leaves through fp32 reductions (red.global.add.f32, each warp
// instruction 128 contiguous bytes of one kv row) into a [T, 512] fp32 buffer
// that the call zeroes; a 32K-token row set holds 64 MB and stays in L2.
// With the gather (1 KB per slot in) these reductions (2 KB per slot out) make
// the SM's traffic with L2 the bound.
//
// Warp roles (640 threads, per-warpgroup register budgets set with setmaxnreg):
//   warps 0-3   producers: the Q / dO rows of subpartition w, 8 latent rows
//               of every block (cp.async, completion counted on mbarriers)
//   warps 4-7   P / dZ' (one head per lane pair, 16 slots per lane), and the
//               dQ epilogue of each query
//   warps 8-11  dKv scatter of the tiles in TMEM buffer 0 (latent tiles 0, 2)
//   warps 16-19 dKv scatter of the tiles in TMEM buffer 1 (latent tiles 1, 3);
//               one latent row of a tile per thread
//   warp 12     [S; dP] issuer (and TMEM owner)
//   warp 13     dQ^T / dKv^T issuer
//   warp 14     row scanner: block count and range check of each index row,
//               two queries ahead
// Every wait is bounded; on expiry the kernel records KPOOL_ERR_TIMEOUT, the
// roles leave their loops, in-flight MMAs are drained and TMEM is freed.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"
#include "tc_ptx.cuh"

namespace kpool {

namespace {

constexpr int BN = 32;                 // slots per gathered block
constexpr int NSTAGE = 2;              // gathered-block ring
constexpr int HP = 64;                 // head rows
constexpr int THREADS = 640;
constexpr int NPROD = 4;
constexpr int ROWS_PER_PROD = BN / NPROD;
constexpr int QD_CHUNK = 128 * 128;    // 16 KB: 128 stacked rows x 128 B (64 bf16 of the latent)
constexpr int KV_CHUNK = BN * 128;     // 4 KB: 32 slots x 128 B
constexpr int KV_STAGE = 8 * KV_CHUNK; // 32 KB
constexpr int PZ_TILE = 64 * 128;      // 8 KB: 64 heads x 64 slots (a pair of blocks)

constexpr int OFF_QD = 0;
constexpr int OFF_KV = OFF_QD + 8 * QD_CHUNK;
constexpr int OFF_PZ = OFF_KV + NSTAGE * KV_STAGE;     // pair buffer t: P at OFF_PZ + 2t*PZ_TILE, dZ' after it
constexpr int OFF_SMALL = OFF_PZ + 4 * PZ_TILE;

struct BwSmall {
    uint64_t qd_full, qd_empty, dq_full, dq_free, drain;
    uint64_t kv_full[NSTAGE], kv_empty[NSTAGE], sdp_full[2], sdp_free[2];
    uint64_t pzb_full[4], pz_empty[2], dk_full[2], dk_empty[2];
    uint64_t nb_full[2], nb_empty[2];
    int nbq[2];                        // row scanner -> producers
    int nbv[2];                        // producers -> every role, by query parity
    int abort;
    uint32_t tmem;
};
constexpr int SMEM_BYTES = OFF_SMALL + (int)sizeof(BwSmall) + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

constexpr uint32_t TM_DQ = 0;
constexpr uint32_t TM_DK = 256;
constexpr uint32_t TM_SD = 384;

constexpr uint32_t ID_SD = tc::idesc(128, BN, 1, 1, false, false);
constexpr uint32_t ID_DQ = tc::idesc(128, HP, 1, 1, true, false);
constexpr uint32_t ID_DK = tc::idesc(128, 2 * BN, 1, 1, true, true);

constexpr uint32_t COPY_ARRIVALS = NPROD * 32 + NPROD;   // copies + one explicit arrive per warp
constexpr uint32_t QD_RELEASES = 2 + 4 + 8;              // two issuers, four P/dZ warps, eight scatter warps

// Per-warpgroup register budgets (launch: 640 threads x 96): producers 40, P/dZ 120, two
// scatter groups 112 each, issuers and row scanner 88 -- 472 of the 480 per thread-quintet.
template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }

__device__ __forceinline__ uint32_t swz(int row, int unit) { return (uint32_t)(row * 128 + ((unit ^ (row & 7)) << 4)); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(addr, parity, abort) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void fail(BwSmall& sm, int32_t* status) {
    sm.abort = 1;
    set_status(status, KPOOL_ERR_TIMEOUT);
}

__device__ __forceinline__ void red_add(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;\n" ::"l"(p), "f"(v) : "memory");
}

// red.global.add.f32 when `on`, without a branch.
__device__ __forceinline__ void red_add_if(float* p, float v, bool on) {
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q red.global.add.f32 [%0], %1;\n}\n" ::"l"(p), "f"(v),
                 "r"((uint32_t)on)
                 : "memory");
}

// Row of the stacked Q / dO operand that holds head h (dO: the second half of its 32-row group).
__device__ __forceinline__ int qd_row(int h, int is_do) { return 32 * (h >> 4) + 16 * is_do + (h & 15); }

}  // namespace

__global__ void __launch_bounds__(THREADS, 1) sparse_mla_bwd_kernel(
    const uint16_t* __restrict__ q_lat, const uint16_t* __restrict__ kv_lat, const int32_t* __restrict__ indices,
    int W, int n_rows, int T, int H, float scale, const float* __restrict__ lse, const float* __restrict__ delta,
    const uint16_t* __restrict__ dout, uint16_t* __restrict__ dq, float* __restrict__ dkv, int32_t* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    BwSmall& sm = *reinterpret_cast<BwSmall*>(smem + OFF_SMALL);
    const uint32_t s_base = tc::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &sm.abort;

    if (tid == 0) {
        tc::mbar_init(tc::smem_u32(&sm.qd_full), COPY_ARRIVALS);
        tc::mbar_init(tc::smem_u32(&sm.qd_empty), QD_RELEASES);
        tc::mbar_init(tc::smem_u32(&sm.dq_full), 1);
        tc::mbar_init(tc::smem_u32(&sm.dq_free), 4);
        tc::mbar_init(tc::smem_u32(&sm.drain), 2);
        for (int s = 0; s < NSTAGE; ++s) {
            tc::mbar_init(tc::smem_u32(&sm.kv_full[s]), COPY_ARRIVALS);
            tc::mbar_init(tc::smem_u32(&sm.kv_empty[s]), 2);     // [S; dP] issuer, dQ issuer
        }
        for (int b = 0; b < 4; ++b) tc::mbar_init(tc::smem_u32(&sm.pzb_full[b]), 4);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tc::smem_u32(&sm.sdp_full[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.sdp_free[b]), 4);
            tc::mbar_init(tc::smem_u32(&sm.pz_empty[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.dk_full[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.dk_empty[b]), 4);
            tc::mbar_init(tc::smem_u32(&sm.nb_full[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.nb_empty[b]), NPROD);
        }
        sm.abort = 0;
        tc::mbar_init_fence();
    }
    if (warp == 12) tc::tmem_alloc(tc::smem_u32(&sm.tmem), 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem;

    if (warp < NPROD) {
        // ===================================================== producers
        regs_dec<40>();
        uint32_t g = 0, qn = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_rows && ok; i += gridDim.x, ++qn) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int32_t* irow = indices + (int64_t)i * W;
            if (!warp_wait(tc::smem_u32(&sm.nb_full[qn & 1]), (qn >> 1) & 1, abort_flag)) { ok = false; break; }
            const int nb = sm.nbq[qn & 1];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.nb_empty[qn & 1]));
            // Q and dO rows of heads 16w .. 16w+15 (rows past H are zero-filled)
            if (!warp_wait(tc::smem_u32(&sm.qd_empty), (qn & 1) ^ 1, abort_flag)) { ok = false; break; }
            for (int r = 0; r < 16; ++r) {
                const int h = warp * 16 + r;
                const bool v = h < H && nb > 0;
                const int64_t off = ((int64_t)i * H + (h < H ? h : 0)) * D_LAT;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int u = k * 32 + lane;
                    const uint32_t cb = s_base + OFF_QD + (u >> 3) * QD_CHUNK;
                    tc::cp_async16(cb + swz(qd_row(h, 0), u & 7), q_lat + off + (v ? u * 8 : 0), v);
                    tc::cp_async16(cb + swz(qd_row(h, 1), u & 7), dout + off + (v ? u * 8 : 0), v);
                }
            }
            tc::cp_async_arrive_noinc(tc::smem_u32(&sm.qd_full));
            if (lane == 0) {
                if (warp == 0) sm.nbv[qn & 1] = nb;
                tc::mbar_arrive(tc::smem_u32(&sm.qd_full));
            }
            // latent rows 8w .. 8w+7 of every block; lane l < 8 holds the slot of row 8w + l
            for (int b = 0; b < nb; ++b, ++g) {
                const int s = g % NSTAGE;
                const int slot = b * BN + warp * ROWS_PER_PROD + lane;
                int myv = (lane < ROWS_PER_PROD && slot < W) ? __ldg(irow + slot) : -1;
                myv = (myv >= 0 && myv < T) ? myv : -1;
                if (!warp_wait(tc::smem_u32(&sm.kv_empty[s]), ((g / NSTAGE) & 1) ^ 1, abort_flag)) { ok = false; break; }
                const uint32_t stage = s_base + OFF_KV + s * KV_STAGE;
#pragma unroll
                for (int rr = 0; rr < ROWS_PER_PROD; ++rr) {
                    const int row = warp * ROWS_PER_PROD + rr;
                    const int v = __shfl_sync(0xffffffffu, myv, rr);
                    const bool valid = v >= 0;
                    const uint16_t* src = valid ? kv_lat + (int64_t)v * D_LAT : kv_lat;
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int u = k * 32 + lane;
                        tc::cp_async16(stage + (u >> 3) * KV_CHUNK + swz(row, u & 7), src + (valid ? u * 8 : 0), valid);
                    }
                }
                tc::cp_async_arrive_noinc(tc::smem_u32(&sm.kv_full[s]));
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.kv_full[s]));
            }
        }
        tc::cp_async_wait<0>();
        if (!ok) fail(sm, status);
    } else if (warp >= 12 && warp < 16) {
      regs_dec<88>();
      if (warp == 12) {
        // ===================================================== [S; dP] issuer
        if (lane == 0) {
            uint32_t g = 0, qn = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_rows && ok && !*abort_flag; i += gridDim.x, ++qn) {
                if (!tc::mbar_wait(tc::smem_u32(&sm.qd_full), qn & 1, abort_flag)) { ok = false; break; }
                tc::fence_proxy_async();                // Q / dO were written by cp.async
                tc::fence_after();
                const int nb = sm.nbv[qn & 1];
                for (int b = 0; b < nb; ++b, ++g) {
                    const int s = g % NSTAGE, sb = g & 1;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.kv_full[s]), (g / NSTAGE) & 1, abort_flag) ||
                        !tc::mbar_wait(tc::smem_u32(&sm.sdp_free[sb]), ((g >> 1) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::fence_proxy_async();
                    tc::fence_after();
                    const uint32_t stage = s_base + OFF_KV + s * KV_STAGE;
#pragma unroll
                    for (int kl = 0; kl < D_LAT / 16; ++kl)
                        tc::mma_bf16(tmem + TM_SD + BN * sb,
                                     tc::sw128_desc(s_base + OFF_QD + (kl >> 2) * QD_CHUNK + (kl & 3) * 32, 0, 1024),
                                     tc::sw128_desc(stage + (kl >> 2) * KV_CHUNK + (kl & 3) * 32, 0, 1024), ID_SD,
                                     kl > 0 ? 1u : 0u);
                    tc::commit(tc::smem_u32(&sm.sdp_full[sb]));
                    tc::commit(tc::smem_u32(&sm.kv_empty[s]));
                }
                if (!ok) break;
                tc::commit(tc::smem_u32(&sm.qd_empty));
            }
            if (!ok) fail(sm, status);
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else if (warp == 13) {
        // ===================================================== dQ^T / dKv^T issuer
        if (lane == 0) {
            uint32_t g = 0, qn = 0, gp = 0, c = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_rows && ok && !*abort_flag; i += gridDim.x, ++qn) {
                if (!tc::mbar_wait(tc::smem_u32(&sm.qd_full), qn & 1, abort_flag)) { ok = false; break; }
                tc::fence_proxy_async();
                tc::fence_after();
                const int nb = sm.nbv[qn & 1];
                // the previous query's dQ epilogue must be done before dQ^T is overwritten (and
                // dq_full / dq_free strictly alternate, also for an empty row)
                if (!tc::mbar_wait(tc::smem_u32(&sm.dq_free), (qn & 1) ^ 1, abort_flag)) { ok = false; break; }
                for (int b0 = 0; b0 < nb && ok; b0 += 2, ++gp) {
                    const int pt = gp & 1;
                    const uint32_t p_t = s_base + OFF_PZ + 2 * pt * PZ_TILE, dz_t = p_t + PZ_TILE;
                    const int nbp = (nb - b0) < 2 ? (nb - b0) : 2;      // blocks in this pair
                    for (int hb = 0; hb < nbp; ++hb, ++g) {
                        const int s = g % NSTAGE;
                        if (!tc::mbar_wait(tc::smem_u32(&sm.pzb_full[2 * pt + hb]), (gp >> 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc::fence_proxy_async();        // P / dZ' were written by the P/dZ warps
                        tc::fence_after();
                        const uint32_t stage = s_base + OFF_KV + s * KV_STAGE;
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                tc::mma_bf16(tmem + TM_DQ + 64 * t,
                                             tc::sw128_desc(stage + 2 * t * KV_CHUNK + kk * 2048, KV_CHUNK, 1024),
                                             tc::sw128_desc(dz_t + hb * 64 + kk * 32, 0, 1024), ID_DQ,
                                             (b0 == 0 && hb == 0 && kk == 0) ? 0u : 1u);
                        tc::commit(tc::smem_u32(&sm.kv_empty[s]));
                    }
                    if (!ok) break;
                    for (int t = 0; t < 4; ++t, ++c) {
                        const int kb = c & 1;
                        if (!tc::mbar_wait(tc::smem_u32(&sm.dk_empty[kb]), ((c >> 1) & 1) ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
#pragma unroll
                        for (int kh = 0; kh < HP / 16; ++kh) {
                            const uint32_t a = s_base + OFF_QD + 2 * t * QD_CHUNK + 32 * kh * 128;
                            tc::mma_bf16(tmem + TM_DK + 64 * kb, tc::sw128_desc(a + 16 * 128, QD_CHUNK, 1024),
                                         tc::sw128_desc(p_t + kh * 2048, PZ_TILE, 1024), ID_DK, kh > 0 ? 1u : 0u);
                            tc::mma_bf16(tmem + TM_DK + 64 * kb, tc::sw128_desc(a, QD_CHUNK, 1024),
                                         tc::sw128_desc(dz_t + kh * 2048, PZ_TILE, 1024), ID_DK, 1u);
                        }
                        tc::commit(tc::smem_u32(&sm.dk_full[kb]));
                    }
                    if (!ok) break;
                    tc::commit(tc::smem_u32(&sm.pz_empty[pt]));
                }
                if (!ok) break;
                tc::commit(tc::smem_u32(&sm.dq_full));
                tc::commit(tc::smem_u32(&sm.qd_empty));
            }
            if (!ok) fail(sm, status);
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else if (warp == 14) {
        // ===================================================== row scanner
        uint32_t qn = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_rows; i += gridDim.x, ++qn) {
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int r = qn & 1;
            if (!warp_wait(tc::smem_u32(&sm.nb_empty[r]), ((qn >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            const int64_t ahead = (int64_t)i + 2 * (int64_t)gridDim.x;
            if (lane == 0 && ahead < n_rows && (W & 3) == 0 && ((reinterpret_cast<uintptr_t>(indices) & 15u) == 0))
                tc::prefetch_l2(indices + ahead * W, (uint32_t)W * 4u);
            const int32_t* irow = indices + (int64_t)i * W;
            int last = -1;
            bool out_of_range = false;
#pragma unroll 4
            for (int j = lane; j < W; j += 32) {
                const int v = __ldg(irow + j);
                const bool valid = v >= 0 && v < T;
                last = valid ? j : last;
                out_of_range |= !valid && v != -1;
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
        // ===================================================== P / dZ' and the dQ epilogue
        regs_inc<120>();
        // Lane pair (l, l+16) owns head h = 16*sp + l; lane half hs owns slots 16hs .. 16hs+15 of a block.
        const int sp = warp - 4;
        const int hs = lane >> 4;
        const int h = sp * 16 + (lane & 15);
        const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
        const float c_log2 = scale * 1.4426950408889634f;
        uint32_t g = 0, qn = 0, gp = 0;
        bool bad = false;
        for (int i = blockIdx.x; i < n_rows && !bad; i += gridDim.x, ++qn) {
            if (!warp_wait(tc::smem_u32(&sm.qd_full), qn & 1, abort_flag)) { bad = true; break; }
            const int nb = sm.nbv[qn & 1];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.qd_empty));
            // padded heads (h >= H) get P = 0 and dZ' = 0
            const float lse2 = h < H ? lse[(int64_t)i * H + h] * 1.4426950408889634f : INFINITY;
            const float dl = h < H ? delta[(int64_t)i * H + h] : 0.f;
            const int32_t* irow = indices + (int64_t)i * W;
            for (int b = 0; b < nb; ++b, ++g) {
                const int pt = gp & 1, hb = b & 1;
                // validity of the block's 32 slots (one ballot)
                const int sl = b * BN + lane;
                const int v = sl < W ? __ldg(irow + sl) : -1;
                const uint32_t mask = __ballot_sync(0xffffffffu, v >= 0 && v < T) >> (16 * hs);
                const int sb = g & 1;
                if (!warp_wait(tc::smem_u32(&sm.sdp_full[sb]), (g >> 1) & 1, abort_flag)) { bad = true; break; }
                tc::fence_after();
                // lane l < 16 reads the S row of head h, lane l + 16 its dP row; after the swap lane l
                // has slots 0-15 and lane l + 16 slots 16-31 of both
                uint32_t a[32];
                tc::tmem_ld32(tmem + lane_base + TM_SD + BN * sb, a);
                tc::tmem_wait_ld();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.sdp_free[sb]));
                uint32_t pk[8], zk[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, hs ? a[j] : a[16 + j], 16);
                    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, hs ? a[j + 1] : a[17 + j], 16);
                    const float s0 = __uint_as_float(hs ? r0 : a[j]), s1 = __uint_as_float(hs ? r1 : a[j + 1]);
                    const float d0 = __uint_as_float(hs ? a[16 + j] : r0), d1 = __uint_as_float(hs ? a[17 + j] : r1);
                    const float p0 = ((mask >> j) & 1u) ? fast_exp2(s0 * c_log2 - lse2) : 0.f;
                    const float p1 = ((mask >> (j + 1)) & 1u) ? fast_exp2(s1 * c_log2 - lse2) : 0.f;
                    pk[j >> 1] = pack2(p0, p1);
                    zk[j >> 1] = pack2(scale * p0 * (d0 - dl), scale * p1 * (d1 - dl));
                }
                if (hb == 0 &&
                    !warp_wait(tc::smem_u32(&sm.pz_empty[pt]), ((gp >> 1) & 1) ^ 1, abort_flag)) {
                    bad = true;
                    break;
                }
                uint8_t* prow = smem + OFF_PZ + 2 * pt * PZ_TILE;
                uint8_t* zrow = prow + PZ_TILE;
                const int u0 = 4 * hb + 2 * hs;      // 16-byte units of slots 32hb + 16hs .. +15
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    *reinterpret_cast<uint4*>(prow + swz(h, u0 + k)) =
                        make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                    *reinterpret_cast<uint4*>(zrow + swz(h, u0 + k)) =
                        make_uint4(zk[4 * k], zk[4 * k + 1], zk[4 * k + 2], zk[4 * k + 3]);
                }
                tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(tc::smem_u32(&sm.pzb_full[2 * pt + hb]));
                    // a pair cut short by the end of the row still completes its second half's phase
                    if (hb == 0 && b == nb - 1) tc::mbar_arrive(tc::smem_u32(&sm.pzb_full[2 * pt + 1]));
                }
                if (hb == 1 || b == nb - 1) ++gp;
            }
            if (bad) break;
            // ---- dQ epilogue: thread (subpartition sp, lane l) holds latent row 128t + 32sp + l of
            // dQ^T tile t for every head; lanes l and l^1 swap one value per head pair so that each
            // 4-byte store writes a latent pair of one head.
            if (!warp_wait(tc::smem_u32(&sm.dq_full), qn & 1, abort_flag)) { bad = true; break; }
            tc::fence_after();
            uint16_t* orow = dq + (int64_t)i * H * D_LAT;
            const int odd = lane & 1;
            for (int t = 0; t < 4; ++t) {
                const int d = t * 128 + sp * 32 + (lane & ~1);
#pragma unroll 1
                for (int c0 = 0; c0 < HP; c0 += 32) {
                    uint32_t o[32];
                    if (nb > 0) {
                        tc::tmem_ld32(tmem + lane_base + TM_DQ + 64 * t + c0, o);
                        tc::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float x0 = __uint_as_float(o[j]), x1 = __uint_as_float(o[j + 1]);
                        const float recv = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
                        const uint32_t w = odd ? pack2(recv, x1) : pack2(x0, recv);
                        const int hh = c0 + j + odd;
                        if (hh < H) *reinterpret_cast<uint32_t*>(orow + hh * D_LAT + d) = w;
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.dq_free));
        }
        if (bad) fail(sm, status);
    } else {
        // ===================================================== dKv scatter (warps 8-11: tiles 0, 2; 16-19: tiles 1, 3)
        regs_inc<112>();
        // Thread (subpartition sp, lane l) holds latent row d = 128t + 32sp + l of the dKv^T tile
        // t for the pair's 64 slots; a warp's reduction covers 128 contiguous bytes of one kv row.
        const int sp = warp & 3;
        const int grp = warp >= 16 ? 1 : 0;           // TMEM buffer (and tile parity) of this group
        const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
        uint32_t qn = 0, c = 0;
        bool bad = false;
        for (int i = blockIdx.x; i < n_rows && !bad; i += gridDim.x, ++qn) {
            if (!warp_wait(tc::smem_u32(&sm.qd_full), qn & 1, abort_flag)) { bad = true; break; }
            const int nb = sm.nbv[qn & 1];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.qd_empty));
            const int32_t* irow = indices + (int64_t)i * W;
            for (int b0 = 0; b0 < nb && !bad; b0 += 2) {
                // rows of the pair's slots: lane l holds slot l of each block (-1: invalid or absent)
                const int s0 = b0 * BN + lane, s1 = s0 + BN;
                int r0 = s0 < W ? __ldg(irow + s0) : -1;
                int r1 = (b0 + 1 < nb && s1 < W) ? __ldg(irow + s1) : -1;
                r0 = (r0 >= 0 && r0 < T) ? r0 : -1;
                r1 = (r1 >= 0 && r1 < T) ? r1 : -1;
                for (int t = 0; t < 4; ++t, ++c) {
                    const int kb = c & 1;
                    if (kb != grp) continue;
                    if (!warp_wait(tc::smem_u32(&sm.dk_full[kb]), (c >> 1) & 1, abort_flag)) { bad = true; break; }
                    tc::fence_after();
                    uint32_t v0[32], v1[32];
                    tc::tmem_ld32(tmem + lane_base + TM_DK + 64 * kb, v0);
                    tc::tmem_ld32(tmem + lane_base + TM_DK + 64 * kb + 32, v1);
                    tc::tmem_wait_ld();
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.dk_empty[kb]));
                    float* col = dkv + t * 128 + sp * 32 + lane;
                    // all row indices first (independent shuffles), then branch-free predicated reductions
                    int rw[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) rw[j] = __shfl_sync(0xffffffffu, r0, j);
#pragma unroll
                    for (int j = 0; j < 32; ++j) red_add_if(col + (int64_t)rw[j] * D_LAT, __uint_as_float(v0[j]), rw[j] >= 0);
#pragma unroll
                    for (int j = 0; j < 32; ++j) rw[j] = __shfl_sync(0xffffffffu, r1, j);
#pragma unroll
                    for (int j = 0; j < 32; ++j) red_add_if(col + (int64_t)rw[j] * D_LAT, __uint_as_float(v1[j]), rw[j] >= 0);
                }
            }
        }
        if (bad) fail(sm, status);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 12) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// delta[r] = sum_d out[r, d] * dout[r, d] over n_vec rows of 512 bf16 (fp32 sums); one warp per row.
__global__ void __launch_bounds__(256) mla_bwd_delta_kernel(const uint16_t* __restrict__ out,
                                                            const uint16_t* __restrict__ dout, int64_t n_vec,
                                                            float* __restrict__ delta) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_vec; r += warps) {
        const uint4* a = reinterpret_cast<const uint4*>(out + r * D_LAT);
        const uint4* b = reinterpret_cast<const uint4*>(dout + r * D_LAT);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint4 x = __ldg(a + lane + 32 * k), y = __ldg(b + lane + 32 * k);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s += __uint_as_float(xs[e] << 16) * __uint_as_float(ys[e] << 16);
                s += __uint_as_float(xs[e] & 0xffff0000u) * __uint_as_float(ys[e] & 0xffff0000u);
            }
        }
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) delta[r] = s;
    }
}

int launch_sparse_mla_bwd(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int n_rows,
                          int T, int n_heads, float scale, const uint16_t* out, const float* lse,
                          const uint16_t* dout, uint16_t* dq, float* dkv, float* delta, int32_t* status,
                          cudaStream_t stream) {
    if (n_heads < 1 || n_heads > HP) return KPOOL_ERR_SHAPE;
    if (T > 0 && cudaMemsetAsync(dkv, 0, (size_t)T * D_LAT * sizeof(float), stream) != cudaSuccess)
        return KPOOL_ERR_CUDA;
    if (n_rows <= 0) return KPOOL_OK;
    static int n_sm[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    if (n_sm[dev] == 0) {
        if (cudaFuncSetAttribute(sparse_mla_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
            cudaSuccess)
            return KPOOL_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KPOOL_ERR_CUDA;
        n_sm[dev] = sms;
    }
    const int64_t n_vec = (int64_t)n_rows * n_heads;
    const int dgrid = (int)((n_vec + 7) / 8 < 4 * n_sm[dev] ? (n_vec + 7) / 8 : 4 * n_sm[dev]);
    mla_bwd_delta_kernel<<<dgrid, 256, 0, stream>>>(out, dout, n_vec, delta);
    const int grid = n_rows < n_sm[dev] ? n_rows : n_sm[dev];
    sparse_mla_bwd_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(q_lat, kv_lat, indices, W, n_rows, T, n_heads,
                                                                 scale, lse, delta, dout, dq, dkv, status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool

namespace kpool {

// Adds 1.0f to every element of the 512-float rows buf[row_ids[k]] with
// red.global.add.f32, each warp instruction covering 128 contiguous bytes of a
// row: the access pattern of the dKv scatter above, without its compute.
__global__ void __launch_bounds__(512) l2_reduce_kernel(float* __restrict__ buf, int rows,
                                                        const int32_t* __restrict__ row_ids, int n_ids) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t k = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); k < n_ids; k += warps) {
        const int r = __ldg(row_ids + k);
        if (r < 0 || r >= rows) continue;
        float* p = buf + (int64_t)r * D_LAT + lane;
#pragma unroll
        for (int c = 0; c < D_LAT / 32; ++c) red_add(p + 32 * c, 1.0f);
    }
}

int launch_l2_reduce(float* buf, int rows, const int32_t* row_ids, int n_ids, cudaStream_t stream) {
    if (n_ids <= 0) return KPOOL_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KPOOL_ERR_CUDA;
    l2_reduce_kernel<<<2 * sms, 512, 0, stream>>>(buf, rows, row_ids, n_ids);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
