// Device helpers shared by the kernels: exact float32 arithmetic that matches a
// plain IEEE evaluation (no contraction), e4m3 packing, and small PTX wrappers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace kvring_impl {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// RoPE on one interleaved pair, every product and sum rounded on its own:
//   y0 = x0*c - x1*s,  y1 = x0*s + x1*c
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0, float& y1) {
    y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    y1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
}

// Pair norm fl(sqrt(fl(x0*x0 + x1*x1))).
__device__ __forceinline__ float pair_norm(float x0, float x1) {
    return __fsqrt_rn(__fadd_rn(__fmul_rn(x0, x0), __fmul_rn(x1, x1)));
}

// e4m3 codes of (a, b), round to nearest even, saturating at +-448; a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Two e4m3 codes (low byte first) -> two exact floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
    __half2 hh = *reinterpret_cast<__half2*>(&h);
    return __half22float2(hh);
}

// (scale, inv) from a chunk amax: amax/448 and 448/amax, both IEEE divisions; amax 0 -> (1, 1).
__device__ __forceinline__ float scale_of(float amax) { return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f); }
__device__ __forceinline__ float inv_of(float amax) { return amax == 0.f ? 1.f : __fdiv_rn(448.f, amax); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace kvring_impl
