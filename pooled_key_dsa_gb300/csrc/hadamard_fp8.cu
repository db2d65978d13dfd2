// Fused Hadamard rotation + per-vector FP8 (E4M3) quantisation.
//
// prime-rl PR "GLM-5.3-Flash text model", Summary: queries and pooled keys are
// Hadamard-rotated in an fp32 butterfly before FP8 scoring.  A group of 8
// lanes owns one vector of width D (64 or 128), so a warp takes 4 vectors at
// once: lane l' of a group holds elements [EL*l', EL*l'+EL) with EL = D/8.
// Stages with stride h < EL run inside the thread, wider ones exchange with
// lane l' ^ (h/EL) of the group.  Every stage is the same fp32 add/subtract of
// the pair (x[j], x[j+h]) -> (x[j] + x[j+h], x[j] - x[j+h]), applied in
// ascending stride order (a cross-lane step is one FMA by +-1, which rounds the
// sum or difference once, as the add/subtract does), then one multiply by
// fp32(1/sqrt(D)).  The scale is amax/448 and the codes are
// E4M3(x * (448/amax)) with IEEE division and round-to-nearest-even,
// saturating; the two divisions serve the 4 vectors of a warp at once.
#include <cstdint>
#include <cuda_fp8.h>

#include "kpool_common.cuh"
#include "kpool_launch.h"

namespace kpool {

// A vector of width D is held by a group of 8 lanes (lane g*8 + l' holds elements [EL*l', EL*l'+EL),
// EL = D/8), so a warp holds 4 vectors at once.  Stages with stride h < EL run inside the thread, the
// wider ones (h = EL, 2EL, 4EL) exchange with lane l' ^ (h/EL) of the group.
template <int D, bool IN_BF16>
__device__ __forceinline__ void load_vec8(const void* __restrict__ x, int64_t v, bool valid, int lg, bool a16,
                                          float (&e)[D / 8]) {
    constexpr int EL = D / 8;
    if (!valid) {
#pragma unroll
        for (int j = 0; j < EL; ++j) e[j] = 0.f;
    } else if (IN_BF16) {
        const uint16_t* src16 = static_cast<const uint16_t*>(x) + v * D + lg * EL;
#pragma unroll
        for (int q = 0; q < EL / 8; ++q) {                  // 8 bf16 per 16-byte unit
            uint4 b;
            if (a16) {
                b = reinterpret_cast<const uint4*>(src16)[q];
            } else {                                        // the input is only 8-byte aligned
                const uint2 lo = reinterpret_cast<const uint2*>(src16)[2 * q];
                const uint2 hi = reinterpret_cast<const uint2*>(src16)[2 * q + 1];
                b = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
            const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                e[8 * q + 2 * k] = __uint_as_float(w[k] << 16);
                e[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
            }
        }
    } else {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + v * D + lg * EL);
#pragma unroll
        for (int q = 0; q < EL / 4; ++q) {
            const float4 f = src[q];
            e[4 * q] = f.x; e[4 * q + 1] = f.y; e[4 * q + 2] = f.z; e[4 * q + 3] = f.w;
        }
    }
}

template <int D, bool IN_BF16>
__global__ void __launch_bounds__(256) hadamard_fp8_kernel(const void* __restrict__ x, int64_t n_vec,
                                                           const int32_t* __restrict__ n_valid_dev,
                                                           const float* __restrict__ w,
                                                           uint8_t* __restrict__ codes, float* __restrict__ scales,
                                                           float* __restrict__ ws_out, float c) {
    constexpr int EL = D / 8;
    const int lane = threadIdx.x & 31;
    const int grp = lane >> 3, lg = lane & 7;               // vector of the warp step, lane in its group
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t n_valid = n_valid_dev ? (int64_t)max(*n_valid_dev, 0) : n_vec;
    const bool a16 = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    for (int64_t v0 = warp0 * 4; v0 < n_vec; v0 += nwarps * 4) {
        const int64_t v = v0 + grp;
        float e[EL];
        load_vec8<D, IN_BF16>(x, v, v < n_valid && v < n_vec, lg, a16, e);
        // in-thread stages
#pragma unroll
        for (int h = 1; h < EL; h <<= 1)
#pragma unroll
            for (int j = 0; j < EL; ++j)
                if ((j & h) == 0) {
                    const float a = e[j], b = e[j + h];
                    e[j] = __fadd_rn(a, b);
                    e[j + h] = __fsub_rn(a, b);
                }
        // cross-lane stages within the group: the lane with the partner bit clear holds x[j].  The pair's sum
        // or difference is one FMA with a +-1 multiplier: fma(e, -1, other) rounds other - e once, exactly as
        // the subtraction does (and fma(e, 1, other) rounds e + other).
#pragma unroll
        for (int lb = 1; lb < 8; lb <<= 1) {
            const float sgn = (lg & lb) != 0 ? -1.f : 1.f;
#pragma unroll
            for (int j = 0; j < EL; ++j) {
                const float other = __shfl_xor_sync(0xffffffffu, e[j], lb);
                e[j] = __fmaf_rn(e[j], sgn, other);
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < EL; ++j) {
            e[j] = __fmul_rn(e[j], c);
            amax = fmaxf(amax, fabsf(e[j]));
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (v >= n_vec) continue;                          // a whole 8-lane group
        uint8_t q[EL];
        float sc = 0.f;
        if (amax > 0.f) {
            const float inv = __fdiv_rn(448.f, amax);
            sc = __fdiv_rn(amax, 448.f);
#pragma unroll
            for (int j = 0; j < EL; j += 2) {
                const uint16_t pr = cvt_e4m3x2(__fmul_rn(e[j], inv), __fmul_rn(e[j + 1], inv));
                q[j] = (uint8_t)(pr & 0xff);
                q[j + 1] = (uint8_t)(pr >> 8);
            }
        } else {
#pragma unroll
            for (int j = 0; j < EL; ++j) q[j] = 0;
        }
        uint32_t pw[EL / 4];
#pragma unroll
        for (int k = 0; k < EL / 4; ++k)
            pw[k] = (uint32_t)q[4 * k] | ((uint32_t)q[4 * k + 1] << 8) | ((uint32_t)q[4 * k + 2] << 16) |
                    ((uint32_t)q[4 * k + 3] << 24);
        uint8_t* dst = codes + v * D + lg * EL;
        if (EL == 16) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(pw[0], pw[1 % (EL / 4)], pw[2 % (EL / 4)], pw[3 % (EL / 4)]);
        } else {
            *reinterpret_cast<uint2*>(dst) = make_uint2(pw[0], pw[1 % (EL / 4)]);
        }
        if (lg == 0) {
            if (scales) scales[v] = sc;
            if (ws_out) ws_out[v] = w ? __fmul_rn(w[v], sc) : sc;
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
    const int64_t want_blocks = (n_vec + 31) / 32;          // 8 warps x 4 vectors
    const unsigned blocks = (unsigned)(want_blocks < 152 * 64 ? want_blocks : 152 * 64);
    if (d == 128) {
        if (in_bf16)
            hadamard_fp8_kernel<128, true><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
        else
            hadamard_fp8_kernel<128, false><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
    } else if (d == 64) {
        if (in_bf16)
            hadamard_fp8_kernel<64, true><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
        else
            hadamard_fp8_kernel<64, false><<<blocks, 256, 0, stream>>>(x, n_vec, n_valid_dev, w, codes, scales, ws_out, c);
    } else {
        return KPOOL_ERR_SHAPE;
    }
    return cudaGetLastError() == cudaSuccess ? KPOOL_OK : KPOOL_ERR_CUDA;
}

}  // namespace kpool
