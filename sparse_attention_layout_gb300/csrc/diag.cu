// Diagnostics: device routines that the kernels use internally, evaluated on
// caller data so that tests can hold them to their stated error bounds.
#include <cuda_runtime.h>

#include "tc_common.cuh"

namespace {

__global__ void exp2_poly_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;
    if (i + 1 < n) {
        const float2 r = bsp::tc::exp2_poly2(make_float2(x[i], x[i + 1]));
        y[i] = r.x;
        y[i + 1] = r.y;
    } else if (i < n) {
        y[i] = bsp::tc::exp2_poly2(make_float2(x[i], 0.f)).x;
    }
}

}  // namespace

extern "C" int bsp_diag_exp2(const float* x, float* y, int64_t n, void* stream) {
    if (n < 0 || (n > 0 && (!x || !y))) return BSP_ERR_INVALID_ARG;
    if (n == 0) return BSP_OK;
    const int64_t pairs = (n + 1) / 2;
    const int threads = 256;
    const int64_t blocks = (pairs + threads - 1) / threads;
    if (blocks > 0x7fffffff) return BSP_ERR_INVALID_ARG;
    exp2_poly_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(x, y, n);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}
