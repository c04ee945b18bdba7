// Diagnostics: device routines that the kernels use internally, evaluated on
// caller data so that tests can hold them to their stated error bounds.
#include <cuda_runtime.h>

#include "bsp_internal.h"
#include "geometry.cuh"
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

extern "C" int bsp_diag_geometry_steps(bsp_layout_t L, int32_t* step_col, int32_t* step_blk) {
    using namespace bsp;
    if (!L || !step_col || !step_blk) return BSP_ERR_INVALID_ARG;
    if (!L->host_tables || L->geo_rec.empty()) return BSP_ERR_UNSUPPORTED;
    const int G = L->G, nb = L->nb;
    for (int tile = 0; tile < L->n_tiles; ++tile) {
        const int h = tile / L->ngroups, gq = tile % L->ngroups;
        const GeoHead gh = geo_load(&L->geo_rec[(size_t)h * kGeoRec]);
        const GeoTile gt = geo_tile(gh, gq * G, geo_min(gq * G + G, nb) - 1, nb);
        const int s0 = L->tile_step_ptr[(size_t)tile], ns = L->tile_step_ptr[(size_t)tile + 1] - s0;
        for (int n = 0; n < ns; ++n)
            for (int b = 0; b < G; ++b) {
                const int c = geo_col(gh, gt, n * G + b);
                step_col[(size_t)(s0 + n) * G + b] = c;
                for (int a = 0; a < G; ++a) {
                    const int rb = gq * G + a;
                    step_blk[((size_t)(s0 + n) * G + a) * G + b] = (c >= 0 && rb < nb && geo_has(gh, rb, c)) ? 1 : 0;
                }
            }
    }
    return BSP_OK;
}
