// Small device helpers shared by the SIMT kernels of libbsp.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "bsp_internal.h"

namespace bsp {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// 16-byte vector of T (4 fp32 or 8 bf16/fp16) converted to / from fp32
template <typename T>
struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    __device__ __forceinline__ static void load(const T* p, float (&out)[N]) {
        uint4 raw = *reinterpret_cast<const uint4*>(p);
        const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int k = 0; k < N; ++k) out[k] = to_f32(e[k]);
    }
    __device__ __forceinline__ static void store(T* p, const float (&in)[N]) {
        uint4 raw;
        T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
        for (int k = 0; k < N; ++k) e[k] = from_f32<T>(in[k]);
        *reinterpret_cast<uint4*>(p) = raw;
    }
};

__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace bsp
