// Shared device helpers of the KPool-DSA kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "kpooldsa.h"

namespace kpool {

constexpr int KPOOL = 4;
constexpr int D_LAT = 512;

// First error wins: a kernel that meets bad data records it here and goes on
// with a safe value.
__device__ __forceinline__ void set_status(int32_t* status, int code) {
    if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// Internal bounds checks.  In the KPOOL_CHECKED build a failed check records
// KPOOL_ERR_CHECK in the call's status word and the caller skips the access;
// in the default build the check is compiled out (every checked index holds by
// construction there, and the checked build's tests show it).
#ifdef KPOOL_CHECKED
__device__ __forceinline__ bool in_bounds(bool ok, int32_t* status) {
    if (!ok) set_status(status, KPOOL_ERR_CHECK);
    return ok;
}
#else
__device__ __forceinline__ bool in_bounds(bool, int32_t*) { return true; }
#endif

// Number of (query, candidate pool) score slots before in-document position r:
// sum over r' < r of floor((r'+1)/4) = sum_{m=1..r} floor(m/4).
// With r = 4a + b: 4 * (0 + 1 + ... + (a-1)) + a * (b + 1).
__host__ __device__ __forceinline__ int64_t pairs_before(int64_t r) {
    const int64_t a = r >> 2, b = r & 3;
    return 2 * a * (a - 1) + a * (b + 1);
}

// Order-preserving map of an fp32 score to uint32: larger score, larger key.
// -0 is folded onto +0 first; NaN (never produced from finite inputs) maps
// below every number.
__device__ __forceinline__ uint32_t score_key(float s) {
    if (s != s) return 0u;
    uint32_t u = __float_as_uint(s + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// E4M3 codes of two fp32 values (round to nearest, ties to even; magnitudes
// above 448 saturate to 448), low byte from `lo`: the one conversion every
// FP8 quantiser of the library uses (and kpool_cast_e4m3 exposes for tests).
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace kpool
