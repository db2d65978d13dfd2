// Absorbed-MLA projections on tcgen05: the query absorption before the sparse
// latent attention and the V projection after it.
//
// NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog: the K
// projection is absorbed into the query, attention runs over the shared
// 512-wide latent, and the model-owned V projection is applied afterwards.
// miles "GLM-5.3-Flash" recipe, section 6 "LoRA RL": both use the kv_b_proj
// weight [H*(d_nope+d_v), 512] directly; head h owns d_nope key rows, then
// d_v value rows.
//
//   absorb:  q_lat[t,h,:] = q_nope[t,h,:] . W_UK[h]      M = tokens, N = 512, K = d_nope
//   v_proj:  o_v[t,h,:]   = W_UV[h] . o_lat[t,h,:]        M = tokens, N = d_v, K = 512
//
// Both are per-head GEMMs whose weight slice (d x 512 bf16, at most 128 KB)
// stays in shared memory.  Work is the flat sequence of (head, 128-token tile)
// pairs, cut into one contiguous range per persistent CTA, so a CTA loads a
// weight slice once, or twice when its range crosses a head.  Activations
// come in by TMA through 3-D tensor maps [T][H][width] that pick one head's
// rows; MMAs (M = 128) accumulate in TMEM; the epilogue converts 64-column
// chunks to bf16 in a 128-byte-swizzled staging tile that a TMA store writes
// out.  Each op moves its activations once through HBM (in and out) and reads
// the weights from L2, so HBM bounds it, not the tensor pipe.
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 4-7 epilogue (TMEM subpartition w-4 = tile rows 32(w-4)..).
// Waits are bounded (KPOOL_ERR_TIMEOUT), as in the other tcgen05 kernels.
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"
#include "tc_ptx.cuh"
#include "tmap_host.h"

namespace kpool {

namespace {

constexpr int PJ_THREADS = 256;
constexpr int BM = 128;                // tokens per tile
constexpr int CHUNK = BM * 128;        // 16 KB: 128 rows x 64 bf16, 128-byte swizzle
constexpr int NSTG = 2;                // output staging tiles
constexpr int MAX_STAGES = 8;
constexpr int PJ_SMEM_LIMIT = 227 * 1024;

struct PjSmall {
    uint64_t a_full[MAX_STAGES], a_empty[MAX_STAGES];
    uint64_t b_full, b_empty, acc_full[2], acc_empty[2], drain;
    int abort;
    uint32_t tmem;
};

// Bytes of the staged weight slice, of one activation stage, and the whole layout.
struct PjGeom {
    int b_bytes, stage_bytes, n_stages, off_a, off_stg, off_small, smem;
};

__host__ __device__ inline PjGeom pj_geom(bool absorb, int dn, int dv) {
    PjGeom g;
    g.b_bytes = (absorb ? dn : dv) * 1024;            // 8 chunks of 64 columns x rows x 2 B
    g.stage_bytes = absorb ? (dn / 64) * CHUNK : CHUNK;
    const int fixed = g.b_bytes + NSTG * CHUNK + (int)sizeof(PjSmall) + 1024;
    int n = (PJ_SMEM_LIMIT - fixed) / g.stage_bytes;
    g.n_stages = n < 1 ? 1 : (n > MAX_STAGES ? MAX_STAGES : n);
    g.off_a = g.b_bytes;
    g.off_stg = g.off_a + g.n_stages * g.stage_bytes;
    g.off_small = g.off_stg + NSTG * CHUNK;
    g.smem = g.off_small + (int)sizeof(PjSmall) + 1024;
    return g;
}

__device__ __forceinline__ bool pj_warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(addr, parity, abort) ? 1u : 0u;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Named barrier 1 over the 128 epilogue threads, ORing a predicate.
__device__ __forceinline__ bool epi_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t*>(&v);
}

// 64 accumulator columns of this thread's tile row -> bf16 -> its row of a
// swizzled staging tile (the layout the TMA store reads).
__device__ __forceinline__ void stage_row(uint32_t taddr, uint8_t* stg, int row) {
    uint32_t a[32], b[32];
    tc::tmem_ld32(taddr, a);
    tc::tmem_ld32(taddr + 32, b);
    tc::tmem_wait_ld();
    uint8_t* dst = stg + row * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t* s = u < 4 ? a + 8 * u : b + 8 * (u - 4);
        const uint4 v = make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                                   pack_bf16x2(s[6], s[7]));
        *reinterpret_cast<uint4*>(dst + ((u ^ (row & 7)) << 4)) = v;
    }
}

}  // namespace

template <bool ABSORB>
__global__ void __launch_bounds__(PJ_THREADS, 1) mla_proj_kernel(const __grid_constant__ CUtensorMap map_a,
                                                                 const __grid_constant__ CUtensorMap map_w,
                                                                 const __grid_constant__ CUtensorMap map_c, int T,
                                                                 int H, int dn, int dv, uint32_t a_box_bytes,
                                                                 int32_t* status) {
    const PjGeom geo = pj_geom(ABSORB, dn, dv);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    PjSmall& sm = *reinterpret_cast<PjSmall*>(smem + geo.off_small);
    const uint32_t s_base = tc::smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &sm.abort;
    const int n_tt = (T + BM - 1) / BM;
    const int64_t U = (int64_t)H * n_tt;
    const int u0 = (int)(U * blockIdx.x / gridDim.x), u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
    const int ns = geo.n_stages;
    const int wrows = ABSORB ? dn : dv;               // weight rows per 64-column box

    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            tc::mbar_init(tc::smem_u32(&sm.a_full[s]), 1);
            tc::mbar_init(tc::smem_u32(&sm.a_empty[s]), 1);
        }
        tc::mbar_init(tc::smem_u32(&sm.b_full), 1);
        tc::mbar_init(tc::smem_u32(&sm.b_empty), 1);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(tc::smem_u32(&sm.acc_full[b]), 1);
            tc::mbar_init(tc::smem_u32(&sm.acc_empty[b]), 4);
        }
        tc::mbar_init(tc::smem_u32(&sm.drain), 1);
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
            uint32_t na = 0, nb = 0;
            int cur_h = -1;
            bool ok = true;
            for (int u = u0; u < u1 && ok; ++u) {
                const int h = u / n_tt, t0 = (u % n_tt) * BM;
                if (h != cur_h) {
                    if (!tc::mbar_wait(tc::smem_u32(&sm.b_empty), (nb & 1) ^ 1, abort_flag)) { ok = false; break; }
                    tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.b_full), (uint32_t)geo.b_bytes);
                    const int wrow = h * (dn + dv) + (ABSORB ? 0 : dn);
                    for (int n = 0; n < 8; ++n)
                        tc::tma_load_2d(s_base + n * wrows * 128, &map_w, 64 * n, wrow, tc::smem_u32(&sm.b_full));
                    cur_h = h;
                    ++nb;
                }
                const int per_tile = ABSORB ? 1 : 8;
                for (int c = 0; c < per_tile; ++c, ++na) {
                    const int s = na % ns;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.a_empty[s]), ((na / ns) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = s_base + geo.off_a + s * geo.stage_bytes;
                    if (ABSORB) {
                        tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.a_full[s]), a_box_bytes * (dn / 64));
                        for (int k = 0; k < dn / 64; ++k)
                            tc::tma_load_3d(dst + k * CHUNK, &map_a, 64 * k, h, t0, tc::smem_u32(&sm.a_full[s]));
                    } else {
                        tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.a_full[s]), a_box_bytes);
                        tc::tma_load_3d(dst, &map_a, 64 * c, h, t0, tc::smem_u32(&sm.a_full[s]));
                    }
                }
            }
            if (!ok) {
                sm.abort = 1;
                set_status(status, KPOOL_ERR_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        if (lane == 0) {
            uint32_t na = 0, nb = 0, nt = 0;
            int cur_h = -1;
            bool ok = true;
            const uint32_t id = ABSORB ? tc::idesc(128, 256, 1, 1, false, true) : tc::idesc(128, dv, 1, 1, false, false);
            for (int u = u0; u < u1 && ok && !*abort_flag; ++u, ++nt) {
                const int h = u / n_tt;
                if (h != cur_h) {
                    if (cur_h >= 0) tc::commit(tc::smem_u32(&sm.b_empty));   // the old slice is free once its MMAs end
                    if (!tc::mbar_wait(tc::smem_u32(&sm.b_full), nb & 1, abort_flag)) { ok = false; break; }
                    cur_h = h;
                    ++nb;
                }
                if (ABSORB) {
                    const int s = na % ns;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.a_full[s]), (na / ns) & 1, abort_flag)) { ok = false; break; }
                    const uint32_t a_base = s_base + geo.off_a + s * geo.stage_bytes;
                    for (int j = 0; j < 2 && ok; ++j) {       // output columns 256j .. 256j+255
                        if (!tc::mbar_wait(tc::smem_u32(&sm.acc_empty[j]), (nt & 1) ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        // W_UK slice as an MN-major operand: 64-column chunk n at n * dn * 128,
                        // K rows of 128 B, 8-row atoms of 1024 B
                        const uint32_t b_base = s_base + 4 * j * dn * 128;
                        for (int k = 0; k < dn / 16; ++k)
                            tc::mma_bf16(tmem + 256 * j,
                                         tc::sw128_desc(a_base + (k >> 2) * CHUNK + (k & 3) * 32, 0, 1024),
                                         tc::sw128_desc(b_base + k * 2048, dn * 128, 1024), id, k > 0 ? 1u : 0u);
                        tc::commit(tc::smem_u32(&sm.acc_full[j]));
                    }
                    if (!ok) break;
                    tc::commit(tc::smem_u32(&sm.a_empty[s]));
                    ++na;
                } else {
                    const int ab = nt & 1;
                    if (!tc::mbar_wait(tc::smem_u32(&sm.acc_empty[ab]), ((nt >> 1) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    for (int kc = 0; kc < 8; ++kc, ++na) {    // latent columns 64kc .. 64kc+63
                        const int s = na % ns;
                        if (!tc::mbar_wait(tc::smem_u32(&sm.a_full[s]), (na / ns) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                        const uint32_t a_base = s_base + geo.off_a + s * CHUNK;
                        const uint32_t b_base = s_base + kc * dv * 128;   // W_UV rows, K-major
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_bf16(tmem + dv * ab, tc::sw128_desc(a_base + kk * 32, 0, 1024),
                                         tc::sw128_desc(b_base + kk * 32, 0, 1024), id, (kc | kk) ? 1u : 0u);
                        tc::commit(tc::smem_u32(&sm.a_empty[s]));
                    }
                    if (!ok) break;
                    tc::commit(tc::smem_u32(&sm.acc_full[ab]));
                }
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
        const int sp = warp & 3;
        const int row = sp * 32 + lane;                // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
        uint8_t* stg0 = smem + geo.off_stg;
        uint32_t nt = 0, nch = 0;
        bool bad = false;
        const int n_acc = ABSORB ? 2 : 1;               // accumulators per tile
        const int n_q = ABSORB ? 4 : dv / 64;           // 64-column chunks per accumulator
        for (int u = u0; u < u1 && !bad; ++u, ++nt) {
            const int h = u / n_tt, t0 = (u % n_tt) * BM;
            for (int j = 0; j < n_acc && !bad; ++j) {
                const int ab = ABSORB ? j : (int)(nt & 1);
                const uint32_t par = ABSORB ? (nt & 1) : ((nt >> 1) & 1);
                bad = !pj_warp_wait(tc::smem_u32(&sm.acc_full[ab]), par, abort_flag);
                const uint32_t col0 = ABSORB ? 256u * j : (uint32_t)(dv * ab);
                for (int q = 0; q < n_q; ++q, ++nch) {
                    const int buf = nch % NSTG;
                    if (tid == 128 && nch >= NSTG) tc::bulk_wait_read<NSTG - 1>();   // staging tile free
                    if (epi_or(bad)) { bad = true; break; }
                    tc::fence_after();
                    stage_row(tmem + lane_base + col0 + 64 * q, stg0 + buf * CHUNK, row);
                    if (q == n_q - 1) {                 // accumulator read out
                        tc::fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.acc_empty[ab]));
                    }
                    tc::fence_proxy_async();
                    epi_or(false);
                    if (tid == 128) {
                        const int x = ABSORB ? 256 * j + 64 * q : 64 * q;
                        tc::tma_store_3d(&map_c, x, h, t0, tc::smem_u32(stg0 + buf * CHUNK));
                        tc::bulk_commit();
                    }
                }
            }
        }
        if (tid == 128) tc::bulk_wait<0>();
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

namespace {

// 3-D bf16 tensor [T][H][width] (width contiguous), box {64, 1, box_t}, 128-byte swizzle.
bool make_map3(CUtensorMap* m, const void* base, int width, int H, int T, int box_t) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * H};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_t};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// kv_b_proj weight [rows][512] bf16, box {64, box_rows}, 128-byte swizzle.
bool make_map_w(CUtensorMap* m, const void* base, int rows, int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D_LAT, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D_LAT * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mla_proj_shape_ok(int n_heads, int d_nope, int d_v) {
    return n_heads >= 1 && n_heads <= 1024 && (d_nope == 64 || d_nope == 128) && (d_v == 64 || d_v == 128);
}

int launch_mla_proj(bool absorb, const void* act, const void* w_kv_b, int T, int n_heads, int d_nope, int d_v,
                    void* out, int32_t* status, cudaStream_t stream) {
    if (T <= 0) return KPOOL_OK;
    if (!mla_proj_shape_ok(n_heads, d_nope, d_v)) return KPOOL_ERR_SHAPE;
    static int n_sm[64] = {0};
    static bool attr_set[2][64] = {{false}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    const PjGeom geo = pj_geom(absorb, d_nope, d_v);
    if (!attr_set[absorb ? 1 : 0][dev]) {
        const cudaError_t e = absorb ? cudaFuncSetAttribute(mla_proj_kernel<true>,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, PJ_SMEM_LIMIT)
                                     : cudaFuncSetAttribute(mla_proj_kernel<false>,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, PJ_SMEM_LIMIT);
        if (e != cudaSuccess) return KPOOL_ERR_CUDA;
        attr_set[absorb ? 1 : 0][dev] = true;
    }
    if (n_sm[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KPOOL_ERR_CUDA;
        n_sm[dev] = sms;
    }
    const int box_t = T < BM ? T : BM;
    const int in_w = absorb ? d_nope : D_LAT, out_w = absorb ? D_LAT : d_v;
    CUtensorMap ma, mw, mc;
    if (!make_map3(&ma, act, in_w, n_heads, T, box_t) ||
        !make_map_w(&mw, w_kv_b, n_heads * (d_nope + d_v), absorb ? d_nope : d_v) ||
        !make_map3(&mc, out, out_w, n_heads, T, box_t))
        return KPOOL_ERR_CUDA;
    const int64_t units = (int64_t)n_heads * ((T + BM - 1) / BM);
    const int grid = units < n_sm[dev] ? (int)units : n_sm[dev];
    const uint32_t a_box_bytes = (uint32_t)box_t * 128u;
    if (absorb)
        mla_proj_kernel<true><<<grid, PJ_THREADS, geo.smem, stream>>>(ma, mw, mc, T, n_heads, d_nope, d_v,
                                                                      a_box_bytes, status);
    else
        mla_proj_kernel<false><<<grid, PJ_THREADS, geo.smem, stream>>>(ma, mw, mc, T, n_heads, d_nope, d_v,
                                                                       a_box_bytes, status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
