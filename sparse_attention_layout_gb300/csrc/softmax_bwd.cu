// Backward of the block-sparse row softmax: with Y = softmax(scale X) over the
// kept entries of each row ("question on blocksparse", openai/triton issue
// 117: the softmax of the SDD output across the row's blocks) and dY the
// gradient of Y, the gradient of X is
//     dX = scale * Y .* (dY - rowsum(Y .* dY)),
// which is 0 wherever Y is 0 (masked entries, rows with nothing kept).
//
// One warp per query row.  A row is nnz_i segments of B contiguous elements
// (row a of each of its block-row's blocks; the blocks of a block-row are
// consecutive in storage), read with 16-byte loads.  Rows of up to 160 chunks
// stay in registers (one pass: load, reduce the dot product, write dX); longer
// rows take two passes, the second re-reading the row.  A lane touches the
// same chunks for reading and writing, so dX may alias dY.  HBM-bound: 2
// reads and 1 write of Z * nnz * B^2 elements.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace bsp {
namespace {

constexpr int kBwdThreads = 256;
// 16-byte chunks per lane kept in registers (rows up to 160 chunks, e.g. 9 blocks
// of 128 bf16); few enough registers for 3 blocks of 256 threads per SM, which
// a memory-bound kernel needs (8 chunks and 1 block per SM ran at 3.8 TB/s)
constexpr int kRegChunks = 5;

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& v, float (&f)[16 / sizeof(T)]) {
    const T* p = reinterpret_cast<const T*>(&v);
#pragma unroll
    for (int k = 0; k < (int)(16 / sizeof(T)); ++k) f[k] = to_f32(p[k]);
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&f)[16 / sizeof(T)]) {
    uint4 v;
    T* p = reinterpret_cast<T*>(&v);
#pragma unroll
    for (int k = 0; k < (int)(16 / sizeof(T)); ++k) p[k] = from_f32<T>(f[k]);
    return v;
}

template <typename T, int BLK>
__global__ void __launch_bounds__(kBwdThreads, 3)
softmax_bwd_kernel(LayoutView L, const T* __restrict__ Y, const T* dY, T* dX, int Z, float scale) {
    constexpr int E = 16 / sizeof(T);           // elements per 16-byte chunk
    constexpr int CH = BLK * (int)sizeof(T) / 16;  // chunks per row segment
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)Z * L.H * L.nb * BLK;
    const int64_t nwarps = (int64_t)gridDim.x * (kBwdThreads / 32);
    for (int64_t row = ((int64_t)blockIdx.x * kBwdThreads + threadIdx.x) / 32; row < rows; row += nwarps) {
        const int a = (int)(row % BLK);
        const int64_t rest = row / BLK;
        const int key = (int)(rest % ((int64_t)L.H * L.nb));
        const int64_t z = rest / ((int64_t)L.H * L.nb);
        const int h = key / L.nb, i = key % L.nb;
        const int p0 = L.row_ptr[h * (L.nb + 1) + i];
        const int nq = L.row_ptr[h * (L.nb + 1) + i + 1] - p0;
        if (nq == 0) continue;
        const int64_t base = (((int64_t)z * L.nnz + p0) * BLK + a) * BLK;  // element offset of segment 0
        auto off = [&](int c) { return base + (int64_t)(c / CH) * BLK * BLK + (int64_t)(c % CH) * E; };
        const int nch = nq * CH;
        if (nch <= 32 * kRegChunks) {
            // the row fits in registers: one pass, all loads in flight together
            uint4 yv[kRegChunks], gv[kRegChunks];
            float dot = 0.f;
#pragma unroll
            for (int t = 0; t < kRegChunks; ++t) {
                const int c = lane + 32 * t;
                if (c < nch) {
                    yv[t] = *reinterpret_cast<const uint4*>(Y + off(c));
                    gv[t] = *reinterpret_cast<const uint4*>(dY + off(c));
                }
            }
#pragma unroll
            for (int t = 0; t < kRegChunks; ++t) {
                if (lane + 32 * t < nch) {
                    float y[E], g[E];
                    unpack16<T>(yv[t], y);
                    unpack16<T>(gv[t], g);
#pragma unroll
                    for (int k = 0; k < E; ++k) dot = fmaf(y[k], g[k], dot);
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
#pragma unroll
            for (int t = 0; t < kRegChunks; ++t) {
                const int c = lane + 32 * t;
                if (c < nch) {
                    float y[E], g[E], x[E];
                    unpack16<T>(yv[t], y);
                    unpack16<T>(gv[t], g);
#pragma unroll
                    for (int k = 0; k < E; ++k) x[k] = scale * y[k] * (g[k] - dot);
                    *reinterpret_cast<uint4*>(dX + off(c)) = pack16<T>(x);
                }
            }
            continue;
        }
        // long rows: two passes (the second read mostly from L2)
        float dot = 0.f;
        for (int c = lane; c < nq * CH; c += 32) {
            float y[E], g[E];
            unpack16<T>(*reinterpret_cast<const uint4*>(Y + off(c)), y);
            unpack16<T>(*reinterpret_cast<const uint4*>(dY + off(c)), g);
#pragma unroll
            for (int k = 0; k < E; ++k) dot = fmaf(y[k], g[k], dot);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        for (int c = lane; c < nq * CH; c += 32) {
            float y[E], g[E], x[E];
            unpack16<T>(*reinterpret_cast<const uint4*>(Y + off(c)), y);
            unpack16<T>(*reinterpret_cast<const uint4*>(dY + off(c)), g);
#pragma unroll
            for (int k = 0; k < E; ++k) x[k] = scale * y[k] * (g[k] - dot);
            *reinterpret_cast<uint4*>(dX + off(c)) = pack16<T>(x);
        }
    }
}

template <typename T, int BLK>
int bwd_launch(const bsp_layout_s* L, const void* Y, const void* dY, void* dX, int Z, float scale,
               cudaStream_t s) {
    const int64_t rows = (int64_t)Z * L->H * L->nb * BLK;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 16);
    softmax_bwd_kernel<T, BLK><<<(unsigned)std::max<int64_t>(blocks, 1), kBwdThreads, 0, s>>>(
        L->view, (const T*)Y, (const T*)dY, (T*)dX, Z, scale);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int bwd_t(const bsp_layout_s* L, const void* Y, const void* dY, void* dX, int Z, float scale, cudaStream_t s) {
    switch (L->B) {
        case 16: return bwd_launch<T, 16>(L, Y, dY, dX, Z, scale, s);
        case 32: return bwd_launch<T, 32>(L, Y, dY, dX, Z, scale, s);
        case 64: return bwd_launch<T, 64>(L, Y, dY, dX, Z, scale, s);
        case 128: return bwd_launch<T, 128>(L, Y, dY, dX, Z, scale, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

// out[r] = sum_d A[r][d] B[r][d] in fp32 (the rowsum(dO .* O) of the attention
// backward): LPR lanes per row (the row's 16-byte chunks, at most 32), 32 / LPR
// rows per warp, grid-stride over groups of rows.
template <typename T, int LPR>
__global__ void __launch_bounds__(256) row_dot_kernel(const T* __restrict__ A, const T* __restrict__ B,
                                                      float* __restrict__ out, int64_t rows, int D) {
    constexpr int E = 16 / sizeof(T);  // elements per 16-byte load
    constexpr int RPW = 32 / LPR;      // rows per warp
    const int lane = threadIdx.x & 31, sub = lane % LPR;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW; r0 < rows;
         r0 += warps * RPW) {
        const int64_t r = r0 + lane / LPR;
        float acc = 0.f;
        if (r < rows) {
            const T* a = A + r * D;
            const T* b = B + r * D;
            for (int d = sub * E; d < D; d += LPR * E) {
                float fa[E], fb[E];
                Vec16<T>::load(a + d, fa);
                Vec16<T>::load(b + d, fb);
#pragma unroll
                for (int k = 0; k < E; ++k) acc = fmaf(fa[k], fb[k], acc);
            }
        }
        // every lane of the warp reaches the shuffles (r0 is warp-uniform)
#pragma unroll
        for (int o = LPR / 2; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (r < rows && sub == 0) out[r] = acc;
    }
}

template <typename T, int LPR>
int row_dot_launch(const void* A, const void* B, float* out, int64_t rows, int D, cudaStream_t s) {
    constexpr int RPB = 256 / LPR;  // rows per block
    const int64_t blocks = std::min<int64_t>((rows + RPB - 1) / RPB, (int64_t)sm_count() * 16);
    row_dot_kernel<T, LPR><<<(unsigned)blocks, 256, 0, s>>>((const T*)A, (const T*)B, out, rows, D);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int row_dot_t(const void* A, const void* B, float* out, int64_t rows, int D, cudaStream_t s) {
    if (rows == 0) return BSP_OK;
    const int chunks = D / (int)(16 / sizeof(T));  // 16-byte chunks per row
    if (chunks <= 2) return row_dot_launch<T, 2>(A, B, out, rows, D, s);
    if (chunks <= 4) return row_dot_launch<T, 4>(A, B, out, rows, D, s);
    if (chunks <= 8) return row_dot_launch<T, 8>(A, B, out, rows, D, s);
    if (chunks <= 16) return row_dot_launch<T, 16>(A, B, out, rows, D, s);
    return row_dot_launch<T, 32>(A, B, out, rows, D, s);
}

}  // namespace

int launch_row_dot(int dtype, const void* A, const void* B, float* out, int64_t rows, int D, cudaStream_t s) {
    if (D % 8 != 0) return BSP_ERR_UNSUPPORTED;  // whole 16-byte loads
    switch (dtype) {
        case BSP_F32: return row_dot_t<float>(A, B, out, rows, D, s);
        case BSP_BF16: return row_dot_t<__nv_bfloat16>(A, B, out, rows, D, s);
        case BSP_F16: return row_dot_t<__half>(A, B, out, rows, D, s);
        default: return BSP_ERR_INVALID_ARG;
    }
}

int launch_softmax_backward(const bsp_layout_s* L, int dtype, const void* Y, const void* dY, void* dX, int Z,
                            float scale, cudaStream_t s) {
    switch (dtype) {
        case BSP_F32: return bwd_t<float>(L, Y, dY, dX, Z, scale, s);
        case BSP_BF16: return bwd_t<__nv_bfloat16>(L, Y, dY, dX, Z, scale, s);
        case BSP_F16: return bwd_t<__half>(L, Y, dY, dX, Z, scale, s);
        default: return BSP_ERR_INVALID_ARG;
    }
}

}  // namespace bsp
