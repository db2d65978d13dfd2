// Sparse latent attention forward (absorbed NoPE MLA over index rows).
//
// NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog: the K
// projection is absorbed into the query and attention runs over the shared
// 512-wide latent, which is both key and value; the V projection is applied
// afterwards by the caller.  miles "GLM-5.3-Flash" recipe, section 1: NoPE
// MLA with 64 heads.
//
// One CTA per query token, all heads at once (heads are the MMA M dimension).
// The index row is walked in blocks of 64 slots; each block's latent rows are
// gathered with cp.async into a double-buffered, XOR-swizzled shared tile
// while the previous block computes.  S = Q K^T and O += P V run on bf16
// tensor-core MMAs (m16n8k16, fp32 accumulate); the online softmax keeps the
// running max and sum per head in shared memory and uses base-2 exponentials
// on logits pre-multiplied by scale*log2(e).
#include <cstdint>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

namespace {

constexpr int MLA_THREADS = 256;
constexpr int BN = 64;                       // slots per block
constexpr int HP = 64;                       // padded head rows
constexpr int ROW_BYTES = D_LAT * 2;         // 1024
constexpr int S_STRIDE = BN + 4;             // fp32 row stride of the score tile

struct MlaSmem {
    uint8_t q[HP * ROW_BYTES];               // 64 KB, swizzled
    uint8_t kv[2][BN * ROW_BYTES];           // 2 x 64 KB, swizzled
    float s[HP * S_STRIDE];                  // 17 KB
    uint8_t p[HP * BN * 2];                  // 8 KB bf16, swizzled
    int32_t idx[2][BN];
    int32_t any_valid[2];
    float m[HP], l[HP], alpha[HP];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 1024-byte rows of 64 16-byte chunks; chunk c of row r lives at c ^ (r & 7).
__device__ __forceinline__ uint32_t swz1k(int row, int chunk) {
    return (uint32_t)(row * ROW_BYTES + ((chunk ^ (row & 7)) << 4));
}
// 128-byte rows of 8 chunks.
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace

template <int MT>
__global__ void __launch_bounds__(MLA_THREADS, 1) sparse_mla_kernel(const uint16_t* __restrict__ q_lat,
                                                                   const uint16_t* __restrict__ kv_lat,
                                                                   const int32_t* __restrict__ indices, int W, int T,
                                                                   int H, float scale_log2, uint16_t* __restrict__ out,
                                                                   float* __restrict__ lse, int32_t* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    MlaSmem& sm = *reinterpret_cast<MlaSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tig = lane & 3;
    const int i = blockIdx.x;
    const int32_t* irow = indices + (int64_t)i * W;
    const int nblk = (W + BN - 1) / BN;
    const uint32_t q_base = smem_u32(sm.q);
    const uint32_t kv_base[2] = {smem_u32(sm.kv[0]), smem_u32(sm.kv[1])};
    const uint32_t p_base = smem_u32(sm.p);

    // ---- Q tile (rows >= H are zero) and running statistics
    {
        const uint16_t* qsrc = q_lat + (int64_t)i * H * D_LAT;
        for (int c = tid; c < HP * 64; c += MLA_THREADS) {
            const int row = c >> 6, ch = c & 63;
            const bool v = row < H;
            cp_async16(q_base + swz1k(row, ch), v ? qsrc + row * D_LAT + ch * 8 : q_lat, v);
        }
    }
    if (tid < HP) {
        sm.m[tid] = -INFINITY;
        sm.l[tid] = 0.f;
    }

    auto load_idx = [&](int blk, int buf) {
        int valid = 0;
        if (tid < BN) {
            const int slot = blk * BN + tid;
            int v = slot < W ? irow[slot] : -1;
            if (v < -1 || v >= T) {
                set_status(status, KPOOL_ERR_INDEX_RANGE);
                v = -1;
            }
            sm.idx[buf][tid] = v;
            valid = v >= 0;
        }
        valid = __syncthreads_or(valid);
        if (tid == 0) sm.any_valid[buf] = valid;
    };
    auto load_kv = [&](int buf) {
        const int ch = tid & 63;
        for (int row = tid >> 6; row < BN; row += MLA_THREADS / 64) {
            const int v = sm.idx[buf][row];
            cp_async16(kv_base[buf] + swz1k(row, ch), v >= 0 ? kv_lat + (int64_t)v * D_LAT + ch * 8 : kv_lat,
                       v >= 0);
        }
    };

    load_idx(0, 0);
    load_kv(0);
    cp_async_commit();

    float o[32][4];
#pragma unroll
    for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    const int mt = warp & 3, half = warp >> 2;

    for (int blk = 0; blk < nblk; ++blk) {
        const int buf = blk & 1;
        if (blk + 1 < nblk) {
            load_idx(blk + 1, buf ^ 1);
            load_kv(buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (!sm.any_valid[buf]) continue;          // uniform across the block

        // ---- S = Q K^T for 16 heads x 32 slots per warp
        if (mt < MT) {
            float acc[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll 4
            for (int kk = 0; kk < D_LAT / 16; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(q_base + swz1k(mt * 16 + (lane & 15), kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    const int nrow = half * 32 + pr * 16 + (lane & 7) + ((lane >> 4) << 3);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kv_base[buf] + swz1k(nrow, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
                    mma_bf16_16816(acc[pr * 2], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(acc[pr * 2 + 1], a0, a1, a2, a3, b2, b3);
                }
            }
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int col = half * 32 + n * 8 + tig * 2;
                const bool v0 = sm.idx[buf][col] >= 0, v1 = sm.idx[buf][col + 1] >= 0;
                const int r0 = mt * 16 + g;
                sm.s[r0 * S_STRIDE + col] = v0 ? acc[n][0] * scale_log2 : -INFINITY;
                sm.s[r0 * S_STRIDE + col + 1] = v1 ? acc[n][1] * scale_log2 : -INFINITY;
                sm.s[(r0 + 8) * S_STRIDE + col] = v0 ? acc[n][2] * scale_log2 : -INFINITY;
                sm.s[(r0 + 8) * S_STRIDE + col + 1] = v1 ? acc[n][3] * scale_log2 : -INFINITY;
            }
        }
        __syncthreads();

        // ---- online softmax: 4 threads per head row, 16 slots each
        {
            const int row = tid >> 2, qtr = tid & 3;
            if (row < MT * 16) {
                float v[16];
                float bmax = -INFINITY;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    v[j] = sm.s[row * S_STRIDE + qtr * 16 + j];
                    bmax = fmaxf(bmax, v[j]);
                }
                bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
                bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 2));
                const float m_old = sm.m[row];
                const float m_new = fmaxf(m_old, bmax);
                float alpha = 1.f, psum = 0.f;
                uint32_t pk[8];
                if (m_new == -INFINITY) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) pk[j] = 0u;
                } else {
                    alpha = exp2f(m_old - m_new);
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float p0 = exp2f(v[j] - m_new), p1 = exp2f(v[j + 1] - m_new);
                        psum += p0 + p1;
                        pk[j >> 1] = pack_bf16(p0, p1);
                    }
                }
                psum += __shfl_xor_sync(0xffffffffu, psum, 1);
                psum += __shfl_xor_sync(0xffffffffu, psum, 2);
                *reinterpret_cast<uint4*>(sm.p + swz128(row, qtr * 2)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(sm.p + swz128(row, qtr * 2 + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                if (qtr == 0) {
                    sm.m[row] = m_new;
                    sm.l[row] = sm.l[row] * alpha + psum;
                    sm.alpha[row] = alpha;
                }
            }
        }
        __syncthreads();

        // ---- O = alpha * O + P V for 16 heads x 256 latent columns per warp
        if (mt < MT) {
            const float al0 = sm.alpha[mt * 16 + g], al1 = sm.alpha[mt * 16 + g + 8];
#pragma unroll
            for (int n = 0; n < 32; ++n) {
                o[n][0] *= al0; o[n][1] *= al0;
                o[n][2] *= al1; o[n][3] *= al1;
            }
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(p_base + swz128(mt * 16 + (lane & 15), kk * 2 + (lane >> 4)), a0, a1, a2, a3);
                const int krow = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int np = 0; np < 16; ++np) {
                    const int chunk = (half * 256 + np * 16) / 8 + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(kv_base[buf] + swz1k(krow, chunk), b0, b1, b2, b3);
                    mma_bf16_16816(o[np * 2], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(o[np * 2 + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        __syncthreads();
    }

    // ---- epilogue: normalise, round to bf16, write out and lse
    if (mt < MT) {
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        const float l0 = sm.l[r0], l1 = sm.l[r1];
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int n = 0; n < 32; ++n) {
            const int col = half * 256 + n * 8 + tig * 2;
            if (r0 < H)
                *reinterpret_cast<uint32_t*>(out + ((int64_t)i * H + r0) * D_LAT + col) =
                    pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
            if (r1 < H)
                *reinterpret_cast<uint32_t*>(out + ((int64_t)i * H + r1) * D_LAT + col) =
                    pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
        }
    }
    if (tid < H) {
        const float l = sm.l[tid];
        lse[(int64_t)i * H + tid] = l > 0.f ? (sm.m[tid] + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
}

template <int MT>
static int launch_mla_t(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int T, int H,
                        float scale, uint16_t* out, float* lse, int32_t* status, cudaStream_t stream) {
    const int smem = (int)sizeof(MlaSmem);
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(sparse_mla_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return KPOOL_ERR_CUDA;
        attr_done[dev] = true;
    }
    const float scale_log2 = scale * 1.4426950408889634f;
    sparse_mla_kernel<MT><<<T, MLA_THREADS, smem, stream>>>(q_lat, kv_lat, indices, W, T, H, scale_log2, out, lse,
                                                            status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

int launch_sparse_mla(const uint16_t* q_lat, const uint16_t* kv_lat, const int32_t* indices, int W, int T,
                      int n_heads, float scale, uint16_t* out, float* lse, int32_t* status, cudaStream_t stream) {
    if (T <= 0) return KPOOL_OK;
    switch ((n_heads + 15) / 16) {
        case 1: return launch_mla_t<1>(q_lat, kv_lat, indices, W, T, n_heads, scale, out, lse, status, stream);
        case 2: return launch_mla_t<2>(q_lat, kv_lat, indices, W, T, n_heads, scale, out, lse, status, stream);
        case 3: return launch_mla_t<3>(q_lat, kv_lat, indices, W, T, n_heads, scale, out, lse, status, stream);
        case 4: return launch_mla_t<4>(q_lat, kv_lat, indices, W, T, n_heads, scale, out, lse, status, stream);
        default: return KPOOL_ERR_SHAPE;
    }
}

}  // namespace kpool
