// Decode side of the k-pool indexer: paged pooled-key cache and paged FP8 scoring.
//
// prime-rl PR "GLM-5.3-Flash text model", section "Patches and workarounds":
// serving aligns hybrid KV blocks to index_kpool x 32 = 128 tokens, and the
// paged indexer kernel takes pages of 32 pools on SM100; so the latent cache and
// the pooled keys live in 128-token pages and a decode query scores its
// sequence's pages.  The same PR, Summary: pooled keys are the per-channel
// softmax(gate + ape)-weighted mean of 4 tokens, Hadamard-rotated in an fp32
// butterfly and quantised to FP8; a query scores the complete pools that end
// at or before it.
//
// Cache layout (one page id indexes all three):
//   k8_cache  e4m3 [n_pages][32][d_i]   codes of the page's 32 pooled keys
//   sk_cache  fp32 [n_pages][32]        their scales
//   kv_cache  bf16 [n_pages][128][512]  the page's 128 latent rows (attention side)
// block_table[b][j] is the page holding tokens 128j .. 128j+127 of sequence b.
#include <cstdint>
#include <cuda_fp8.h>

#include "kpool_common.cuh"
#include "kpool_launch.h"
#include "tc_ptx.cuh"
#include "tmap_host.h"

namespace kpool {

constexpr int PAGE_POOLS = 32;
constexpr int PAGE_TOKENS = PAGE_POOLS * KPOOL;   // 128

// ---------------------------------------------------------------- paged append
// One 128-thread block per pooled key.  Thread c pools channel c of the 4 token
// rows starting at row pool_tok[v] of k / gate (fp64 softmax(gate + ape)
// weights, rounded once to fp32: the prefill pooling's arithmetic, spread over
// 128 threads because fp64 is slow on this part).  Warp 0 then applies the
// prefill's key quantisation (lane l holds elements 4l .. 4l+3: butterfly,
// scale, E4M3 cast) and writes codes and scale to slot pool_idx[v] % 32 of page
// block_table[pool_seq[v]][pool_idx[v] / 32].  d_i = 128.
__global__ void __launch_bounds__(128) paged_append_kernel(
    const uint16_t* __restrict__ k, const float* __restrict__ gate, const float* __restrict__ ape,
    const int32_t* __restrict__ pool_tok, const int32_t* __restrict__ pool_seq, const int32_t* __restrict__ pool_idx,
    int n_items, const int32_t* __restrict__ block_table, int max_pages, int n_pages, uint8_t* __restrict__ k8_cache,
    float* __restrict__ sk_cache, int32_t* status) {
    constexpr int D = 128, E = 4;
    __shared__ __align__(16) float pooled[D];
    const int tid = threadIdx.x, lane = tid & 31;
    const float c = 0.08838834764831845f;          // fp32(1/sqrt(128))
    for (int64_t v = blockIdx.x; v < n_items; v += gridDim.x) {
        const int pidx = pool_idx[v];
        const int pj = pidx / PAGE_POOLS;
        const int page = (pidx >= 0 && pj < max_pages) ? block_table[(int64_t)pool_seq[v] * max_pages + pj] : -1;
        if (page < 0 || page >= n_pages) {         // uniform over the block
            if (tid == 0) set_status(status, KPOOL_ERR_INDEX_RANGE);
            continue;
        }
        const int64_t t0 = pool_tok[v];
        {
            double lg[KPOOL], kv[KPOOL];
#pragma unroll
            for (int j = 0; j < KPOOL; ++j) {
                lg[j] = __dadd_rn((double)gate[(t0 + j) * D + tid], (double)ape[j * D + tid]);
                kv[j] = (double)bf16_bits_to_float(k[(t0 + j) * D + tid]);
            }
            double m = lg[0];
#pragma unroll
            for (int j = 1; j < KPOOL; ++j) m = fmax(m, lg[j]);
            double w[KPOOL], s = 0.0;
#pragma unroll
            for (int j = 0; j < KPOOL; ++j) {
                w[j] = exp(__dsub_rn(lg[j], m));
                s = __dadd_rn(s, w[j]);
            }
            double acc = 0.0;
#pragma unroll
            for (int j = 0; j < KPOOL; ++j) acc = __dadd_rn(acc, __dmul_rn(__ddiv_rn(w[j], s), kv[j]));
            pooled[tid] = (float)acc;
        }
        __syncthreads();
        if (tid < 32) {
            const float4 x = *reinterpret_cast<const float4*>(pooled + lane * E);
            float e[E] = {x.x, x.y, x.z, x.w};
            // butterfly: strides 1, 2 inside the thread, then 4 .. 64 across lanes
#pragma unroll
            for (int h = 1; h < E; h <<= 1)
#pragma unroll
                for (int j = 0; j < E; ++j)
                    if ((j & h) == 0) {
                        const float a = e[j], b = e[j + h];
                        e[j] = __fadd_rn(a, b);
                        e[j + h] = __fsub_rn(a, b);
                    }
#pragma unroll
            for (int lb = 1; lb < 32; lb <<= 1) {
                const bool high = (lane & lb) != 0;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const float other = __shfl_xor_sync(0xffffffffu, e[j], lb);
                    e[j] = high ? __fsub_rn(other, e[j]) : __fadd_rn(e[j], other);
                }
            }
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                e[j] = __fmul_rn(e[j], c);
                amax = fmaxf(amax, fabsf(e[j]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            uint32_t packed = 0;
            float sc = 0.f;
            if (amax > 0.f) {
                const float inv = __fdiv_rn(448.f, amax);
                sc = __fdiv_rn(amax, 448.f);
                const uint16_t lo = cvt_e4m3x2(__fmul_rn(e[0], inv), __fmul_rn(e[1], inv));
                const uint16_t hi = cvt_e4m3x2(__fmul_rn(e[2], inv), __fmul_rn(e[3], inv));
                packed = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            const int64_t slot = (int64_t)page * PAGE_POOLS + (pidx % PAGE_POOLS);
            *reinterpret_cast<uint32_t*>(k8_cache + slot * D + lane * E) = packed;
            if (lane == 0) sk_cache[slot] = sc;
        }
        __syncthreads();                             // `pooled` is rewritten for the next item
    }
}

// ---------------------------------------------------------------- paged scoring
// One CTA per (group of DS_TILES 128-pool tiles, sequence).  All the group's
// pages of codes (TMA, 4 KB each; a tile's 4 pages are the M = 128 operand) and
// the query's H_i rows of codes (the N = H_i operand) are requested at once,
// one barrier per tile; warp 4 issues each tile's 4 tcgen05 kind::f8f6f4 MMAs
// (K = 32 each) into that tile's own TMEM accumulator as soon as its pages
// land, so the loads of later tiles, the MMAs and the epilogue of earlier ones
// overlap.  Epilogue: thread t of warps 0-3 owns pool 128*tile + t: ReLU, the
// head weights ws, the pool scale.  Scores of row b go to scores[b * stride + p].
namespace {

constexpr int DS_TILES = 4;                        // 128-pool tiles per CTA
constexpr int DS_THREADS = 160;                    // warps 0-3 epilogue, warp 4 TMA + MMA
constexpr int DS_A_BYTES = 128 * 128;

struct DsSmall {
    uint64_t q_full, full[DS_TILES], done[DS_TILES], drain;
    uint32_t tmem;
    int abort;
};
template <int HI>
constexpr int ds_smem() { return DS_TILES * DS_A_BYTES + HI * 128 + (int)sizeof(DsSmall) + 1024; }

template <int HI>
__global__ void __launch_bounds__(DS_THREADS) decode_score_kernel(const __grid_constant__ CUtensorMap map_q,
                                                                  const __grid_constant__ CUtensorMap map_k,
                                                                  const float* __restrict__ ws,
                                                                  const float* __restrict__ sk_cache,
                                                                  const int32_t* __restrict__ block_table,
                                                                  int max_pages, int n_pages,
                                                                  const int32_t* __restrict__ seq_lens,
                                                                  float* __restrict__ scores, int64_t stride,
                                                                  int32_t* status) {
    extern __shared__ __align__(1024) uint8_t ds_raw[];
    uint8_t* smem = ds_raw + ((1024u - (tc::smem_u32(ds_raw) & 1023u)) & 1023u);
    uint8_t* a_tiles = smem;
    uint8_t* b_tile = smem + DS_TILES * DS_A_BYTES;
    DsSmall& sm = *reinterpret_cast<DsSmall*>(b_tile + HI * 128);
    __shared__ __align__(16) float wsh[HI];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y, tile0 = blockIdx.x * DS_TILES;
    const int L = seq_lens[b];
    if (L > max_pages * PAGE_TOKENS) {                // the block table cannot hold the sequence
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, KPOOL_ERR_SHAPE);
        return;
    }
    const int n = L / KPOOL;                          // complete pools of the sequence
    if (tile0 * 128 >= n) return;
    const int nt = min(DS_TILES, (n - tile0 * 128 + 127) / 128);   // tiles of this CTA
    if (tid < HI) wsh[tid] = ws[(int64_t)b * HI + tid];
    if (tid == 128) {
        tc::mbar_init(tc::smem_u32(&sm.q_full), 1);
        for (int j = 0; j < DS_TILES; ++j) {
            tc::mbar_init(tc::smem_u32(&sm.full[j]), 1);
            tc::mbar_init(tc::smem_u32(&sm.done[j]), 1);
        }
        tc::mbar_init(tc::smem_u32(&sm.drain), 1);
        sm.abort = 0;
        tc::mbar_init_fence();
    }
    if (warp == 4) tc::tmem_alloc(tc::smem_u32(&sm.tmem), 128);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = sm.tmem;
    volatile int* abort_flag = &sm.abort;

    if (warp == 4) {
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.q_full), (uint32_t)(HI * 128));
            tc::tma_load_2d(tc::smem_u32(b_tile), &map_q, 0, b * HI, tc::smem_u32(&sm.q_full));
            for (int j = 0; j < nt; ++j) {
                const int tile = tile0 + j;
                const int npg = min(4, (n - tile * 128 + PAGE_POOLS - 1) / PAGE_POOLS);   // pages of this tile
                tc::mbar_arrive_expect_tx(tc::smem_u32(&sm.full[j]), (uint32_t)(npg * PAGE_POOLS * 128));
                for (int g = 0; g < npg; ++g) {
                    const int page = block_table[(int64_t)b * max_pages + tile * 4 + g];
                    // an out-of-range page id reads TMA's zero fill; the epilogue flags it
                    tc::tma_load_2d(tc::smem_u32(a_tiles + j * DS_A_BYTES + g * PAGE_POOLS * 128), &map_k, 0,
                                    page * PAGE_POOLS, tc::smem_u32(&sm.full[j]));
                }
            }
            bool ok = tc::mbar_wait(tc::smem_u32(&sm.q_full), 0, abort_flag);
            const uint64_t bd = tc::sw128_desc(tc::smem_u32(b_tile), 0, 1024);
            constexpr uint32_t id = tc::idesc(128, HI, 0, 0, false, false);
            for (int j = 0; ok && j < nt; ++j) {
                ok = tc::mbar_wait(tc::smem_u32(&sm.full[j]), 0, abort_flag);
                if (!ok) break;
                tc::fence_after();
                const uint64_t ad = tc::sw128_desc(tc::smem_u32(a_tiles + j * DS_A_BYTES), 0, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_e4m3(tmem + 32 * j, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), id,
                                 kk > 0 ? 1u : 0u);
                tc::commit(tc::smem_u32(&sm.done[j]));
            }
            if (!ok) {
                sm.abort = 1;                          // the epilogue stops waiting
                set_status(status, KPOOL_ERR_TIMEOUT);
            }
            // every MMA issued has completed before TMEM is released
            tc::commit(tc::smem_u32(&sm.drain));
            const uint64_t t0 = tc::globaltimer_ns();
            while (!tc::mbar_try(tc::smem_u32(&sm.drain), 0) && tc::globaltimer_ns() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
        __syncwarp();
    } else {
        // thread t: TMEM lane t = pool 128*tile + t; columns 32j .. 32j + HI - 1 = heads of tile j
        for (int j = 0; j < nt; ++j) {
            const int p = (tile0 + j) * 128 + tid;
            const int page = p < n ? block_table[(int64_t)b * max_pages + (p / PAGE_POOLS)] : -1;
            const bool page_ok = page >= 0 && page < n_pages;
            const float sk = page_ok ? sk_cache[(int64_t)page * PAGE_POOLS + (p % PAGE_POOLS)] : 0.f;
            uint32_t ok = 0;
            if (lane == 0) ok = tc::mbar_wait(tc::smem_u32(&sm.done[j]), 0, abort_flag) ? 1u : 0u;
            if (__shfl_sync(0xffffffffu, ok, 0) == 0) break;
            tc::fence_after();
            uint32_t acc[32];
            tc::tmem_ld32(tmem + 32 * j + ((uint32_t)(warp * 32) << 16), acc);
            tc::tmem_wait_ld32(acc);
            float2 part[4];
#pragma unroll
            for (int h = 0; h < HI; h += 2) {
                const float2 x = make_float2(fmaxf(__uint_as_float(acc[h]), 0.f),
                                             fmaxf(__uint_as_float(acc[h + 1]), 0.f));
                const float2 w2 = make_float2(wsh[h], wsh[h + 1]);
                if (h < 8) part[h / 2] = __fmul2_rn(x, w2);
                else part[(h / 2) & 3] = __ffma2_rn(x, w2, part[(h / 2) & 3]);
            }
            part[0] = __fadd2_rn(__fadd2_rn(part[0], part[1]), __fadd2_rn(part[2], part[3]));
            const float s = part[0].x + part[0].y;
            if (p < n) {
                if (page_ok) {
                    scores[(int64_t)b * stride + p] = s * sk;
                } else {
                    scores[(int64_t)b * stride + p] = -INFINITY;
                    set_status(status, KPOOL_ERR_INDEX_RANGE);
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 4) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 128);
    }
}

bool make_u8_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
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
int launch_ds(const uint8_t* q8, const float* ws, const uint8_t* k8_cache, const float* sk_cache, int n_pages,
              const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B, float* scores,
              int64_t stride, int32_t* status, cudaStream_t stream) {
    CUtensorMap mq, mk;
    if (!make_u8_map(&mq, q8, (uint64_t)B * HI, HI) ||
        !make_u8_map(&mk, k8_cache, (uint64_t)n_pages * PAGE_POOLS, PAGE_POOLS))
        return KPOOL_ERR_CUDA;
    static bool attr[64] = {false};                   // per device: the shared-memory opt-in is set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KPOOL_ERR_CUDA;
    if (!attr[dev]) {
        if (cudaFuncSetAttribute(decode_score_kernel<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 ds_smem<HI>()) != cudaSuccess)
            return KPOOL_ERR_CUDA;
        attr[dev] = true;
    }
    const dim3 grid((unsigned)((max_pages + 4 * DS_TILES - 1) / (4 * DS_TILES)), (unsigned)B);
    decode_score_kernel<HI><<<grid, DS_THREADS, ds_smem<HI>(), stream>>>(mq, mk, ws, sk_cache, block_table, max_pages,
                                                                       n_pages, seq_lens, scores, stride, status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace

int launch_paged_append(const void* k, const float* gate, const float* ape, const int32_t* pool_tok,
                        const int32_t* pool_seq, const int32_t* pool_idx, int n_items, const int32_t* block_table,
                        int max_pages, int n_pages, uint8_t* k8_cache, float* sk_cache, int32_t* status,
                        cudaStream_t stream) {
    if (n_items <= 0) return KPOOL_OK;
    const int64_t blocks = n_items < 152 * 64 ? n_items : 152 * 64;
    paged_append_kernel<<<(unsigned)blocks, 128, 0, stream>>>(
        static_cast<const uint16_t*>(k), gate, ape, pool_tok, pool_seq, pool_idx, n_items, block_table, max_pages,
        n_pages, k8_cache, sk_cache, status);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

int launch_decode_score(const uint8_t* q8, const float* ws, const uint8_t* k8_cache, const float* sk_cache,
                        int n_pages, const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                        int n_idx_heads, float* scores, int64_t stride, int32_t* status, cudaStream_t stream) {
    if (B <= 0 || max_pages <= 0) return KPOOL_OK;
    switch (n_idx_heads) {
        case 16: return launch_ds<16>(q8, ws, k8_cache, sk_cache, n_pages, block_table, max_pages, seq_lens, B, scores, stride, status, stream);
        case 32: return launch_ds<32>(q8, ws, k8_cache, sk_cache, n_pages, block_table, max_pages, seq_lens, B, scores, stride, status, stream);
        default: return KPOOL_ERR_SHAPE;
    }
}

}  // namespace kpool
