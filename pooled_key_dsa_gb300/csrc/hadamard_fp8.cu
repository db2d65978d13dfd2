// Fused Hadamard rotation + per-vector FP8 (E4M3) quantisation.
//
// prime-rl PR "GLM-5.3-Flash text model", Summary: queries and pooled keys are
// Hadamard-rotated in an fp32 butterfly before FP8 scoring.  One warp owns one
// vector of width D (64 or 128): lane l holds elements [E*l, E*l+E) with
// E = D/32.  Stages with stride h < E run inside the thread, wider ones
// exchange with lane l ^ (h/E).  Every stage is the same fp32 add/subtract of
// the pair (x[j], x[j+h]) -> (x[j] + x[j+h], x[j] - x[j+h]), applied in
// ascending stride order, then one multiply by fp32(1/sqrt(D)).  The scale is
// amax/448 and the codes are E4M3(x * (448/amax)) with IEEE division and
// round-to-nearest-even, saturating.  A warp takes 4 consecutive vectors per
// step, their loads issued together, and each cross-lane butterfly step is one
// FMA by +-1 (the sum or difference rounded once, as before).
#include <cstdint>
#include <cuda_fp8.h>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

template <int D, bool IN_BF16>
__device__ __forceinline__ void load_vec(const void* __restrict__ x, int64_t v, bool valid, int lane, float (&e)[D / 32]) {
    constexpr int E = D / 32;
    if (!valid) {
#pragma unroll
        for (int j = 0; j < E; ++j) e[j] = 0.f;
    } else if (IN_BF16) {
        const uint16_t* src = static_cast<const uint16_t*>(x) + v * D + lane * E;
        if (E == 4) {
            const uint2 b = *reinterpret_cast<const uint2*>(src);
            e[0] = __uint_as_float(b.x << 16);
            e[1] = __uint_as_float(b.x & 0xffff0000u);
            e[2 % E] = __uint_as_float(b.y << 16);
            e[3 % E] = __uint_as_float(b.y & 0xffff0000u);
        } else {
            const uint32_t b = *reinterpret_cast<const uint32_t*>(src);
            e[0] = __uint_as_float(b << 16);
            e[1] = __uint_as_float(b & 0xffff0000u);
        }
    } else {
        const float* src = static_cast<const float*>(x) + v * D + lane * E;
        if (E == 4) {
            const float4 f = *reinterpret_cast<const float4*>(src);
            e[0] = f.x; e[1] = f.y; e[2 % E] = f.z; e[3 % E] = f.w;
        } else {
            const float2 f = *reinterpret_cast<const float2*>(src);
            e[0] = f.x; e[1] = f.y;
        }
    }
}

// Each warp takes VPW consecutive vectors per step: their loads are issued together, so a warp
// has VPW * 32 * E elements in flight instead of one vector's (the kernel is bound by memory-level
// parallelism, not arithmetic); each vector's arithmetic is unchanged.
template <int D, bool IN_BF16, int VPW>
__global__ void __launch_bounds__(256) hadamard_fp8_kernel(const void* __restrict__ x, int64_t n_vec,
                                                           const int32_t* __restrict__ n_valid_dev,
                                                           const float* __restrict__ w,
                                                           uint8_t* __restrict__ codes, float* __restrict__ scales,
                                                           float* __restrict__ ws_out, float c) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t n_valid = n_valid_dev ? (int64_t)max(*n_valid_dev, 0) : n_vec;
    for (int64_t v0 = warp0 * VPW; v0 < n_vec; v0 += nwarps * VPW) {
        float e[VPW][E];
#pragma unroll
        for (int u = 0; u < VPW; ++u) load_vec<D, IN_BF16>(x, v0 + u, v0 + u < n_valid && v0 + u < n_vec, lane, e[u]);
        // in-thread stages
#pragma unroll
        for (int h = 1; h < E; h <<= 1) {
#pragma unroll
            for (int u = 0; u < VPW; ++u)
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    if ((j & h) == 0) {
                        const float a = e[u][j], b = e[u][j + h];
                        e[u][j] = __fadd_rn(a, b);
                        e[u][j + h] = __fsub_rn(a, b);
                    }
                }
        }
        // cross-lane stages: the lane with the partner bit clear holds x[j].  The pair's sum or
        // difference is one FMA with a +-1 multiplier: fma(e, -1, other) rounds other - e once,
        // exactly as the subtraction does (and fma(e, 1, other) rounds e + other).
#pragma unroll
        for (int lb = 1; lb < 32; lb <<= 1) {
            const float sgn = (lane & lb) != 0 ? -1.f : 1.f;
#pragma unroll
            for (int u = 0; u < VPW; ++u)
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const float other = __shfl_xor_sync(0xffffffffu, e[u][j], lb);
                    e[u][j] = __fmaf_rn(e[u][j], sgn, other);
                }
        }
        float amax[VPW];
#pragma unroll
        for (int u = 0; u < VPW; ++u) {
            amax[u] = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                e[u][j] = __fmul_rn(e[u][j], c);
                amax[u] = fmaxf(amax[u], fabsf(e[u][j]));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < VPW; ++u) amax[u] = fmaxf(amax[u], __shfl_xor_sync(0xffffffffu, amax[u], o));
#pragma unroll
        for (int u = 0; u < VPW; ++u) {
            const int64_t v = v0 + u;
            if (v >= n_vec) break;                      // warp-uniform
            uint8_t q[E];
            float s = 0.f;
            if (amax[u] > 0.f) {
                const float inv = __fdiv_rn(448.f, amax[u]);
                s = __fdiv_rn(amax[u], 448.f);
#pragma unroll
                for (int j = 0; j < E; j += 2) {
                    const uint16_t pr = cvt_e4m3x2(__fmul_rn(e[u][j], inv), __fmul_rn(e[u][j + 1], inv));
                    q[j] = (uint8_t)(pr & 0xff);
                    q[j + 1] = (uint8_t)(pr >> 8);
                }
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) q[j] = 0;
            }
            uint8_t* dst = codes + v * D + lane * E;
            if (E == 4) {
                *reinterpret_cast<uint32_t*>(dst) =
                    (uint32_t)q[0] | ((uint32_t)q[1] << 8) | ((uint32_t)q[2 % E] << 16) | ((uint32_t)q[3 % E] << 24);
            } else {
                *reinterpret_cast<uint16_t*>(dst) = (uint16_t)((uint32_t)q[0] | ((uint32_t)q[1] << 8));
            }
            if (lane == 0) {
                if (scales) scales[v] = s;
                if (ws_out) ws_out[v] = w ? __fmul_rn(w[v], s) : s;
            }
        }
    }
}

// E4M3 codes of n fp32 values with the quantisers' conversion (a test and
// diagnostic entry: the oracle's encoder is checked against it value by value).
__global__ void __launch_bounds__(256) cast_e4m3_kernel(const float* __restrict__ x, int64_t n,
                                                        uint8_t* __restrict__ codes) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 2;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2; i < n; i += stride) {
        if (i + 1 < n) {
            const uint16_t c = cvt_e4m3x2(x[i], x[i + 1]);
            codes[i] = (uint8_t)(c & 0xff);
            codes[i + 1] = (uint8_t)(c >> 8);
        } else {
            codes[i] = (uint8_t)(cvt_e4m3x2(x[i], 0.f) & 0xff);
        }
    }
}

int launch_cast_e4m3(const float* x, int64_t n, uint8_t* codes, cudaStream_t stream) {
    if (n <= 0) return KPOOL_OK;
    const int64_t want = (n + 511) / 512;
    const unsigned blocks = (unsigned)(want < 152 * 32 ? want : 152 * 32);
    cast_e4m3_kernel<<<blocks, 256, 0, stream>>>(x, n, codes);
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

int launch_hadamard_fp8(const void* x, bool in_bf16, int64_t n_vec, int d, const int32_t* n_valid_dev,
                        const float* w, uint8_t* codes, float* scales, float* ws_out, cudaStream_t stream) {
    if (n_vec <= 0) return KPOOL_OK;
    const float c = (float)(1.0 / sqrt((double)d));
    constexpr int VPW = 4;
    const int64_t want_blocks = (n_vec + 8 * VPW - 1) / (8 * VPW);
    const unsigned blocks = (unsigned)(want_blocks < 152 * 64 ? want_blocks : 152 * 64);
    if (d == 128) {
        if (in_bf16)
            hadamard_fp8_kernel<128, true, VPW><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
        else
            hadamard_fp8_kernel<128, false, VPW><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
    } else if (d == 64) {
        if (in_bf16)
            hadamard_fp8_kernel<64, true, VPW><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
        else
            hadamard_fp8_kernel<64, false, VPW><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
    } else {
        return KPOOL_ERR_SHAPE;
    }
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
