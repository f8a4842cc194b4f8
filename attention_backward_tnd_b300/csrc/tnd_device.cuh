// Device helpers shared by the kernels of the TND attention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tnd_internal.h"

namespace tnd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x with the SFU instruction (inputs far below -126 flush to 0).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float load(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void store(__half *p, float x) { *p = __float2half_rn(x); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

// Record the first device-side error of a call (later ones keep the first).
__device__ __forceinline__ void set_status(uint32_t *status, uint32_t code, uint32_t detail)
{
    if (atomicCAS(status + kStatusWord, 0u, code) == 0u) {
        atomicExch(status + kStatusDetail, detail);
    }
}

// Dropout multiplier z of (b, h, i, j): keep-bit / keepProb.
__device__ __forceinline__ float drop_z(const uint8_t *mask, int64_t base, int32_t h, int64_t i,
                                        int64_t j, int64_t sq, int64_t skv, float inv_keep)
{
    const int64_t idx = base + ((int64_t)h * sq + i) * skv + j;
    return ((mask[idx >> 3] >> (idx & 7)) & 1) ? inv_keep : 0.0f;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace tnd
