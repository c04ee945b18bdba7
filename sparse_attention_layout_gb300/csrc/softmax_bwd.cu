// Backward of the block-sparse row softmax: with Y = softmax(scale X) over the
// kept entries of each row ("question on blocksparse", openai/triton issue
// 117: the softmax of the SDD output across the row's blocks) and dY the
// gradient of Y, the gradient of X is
//     dX = scale * Y .* (dY - rowsum(Y .* dY)),
// which is 0 wherever Y is 0 (masked entries, rows with nothing kept).
//
// HBM-bound: 2 reads and 1 write of Z * nnz * B^2 elements.  Two kernels,
// chosen by the layout's longest row:
//
// softmax_bwd_kernel (every row within 160 vectors of 16 bytes, and layouts
// whose chunks would not fit twice in shared memory): one warp per query row,
// a row's nnz_i segments of B contiguous elements (row a of each of its
// block-row's blocks, which are consecutive in storage) read with 16-byte
// loads from global memory.  Rows of up to 160 vectors stay in registers (one
// pass); longer rows take two passes, the second re-reading the row.  A lane
// touches the same vectors for reading and writing, so dX may alias dY.
//
// softmax_bwd_chunk_kernel (layouts with longer rows) takes the forward's
// chunk list: a CTA moves R consecutive rows of one block-row of Y and of dY
// into shared memory with one bulk copy per present block and array, reduces
// each row's dot product there (8, 16 or 32 lanes a row with the row in
// registers; rows too long for registers shared by several warps), writes dX
// over dY's copy and sends it back with one bulk store per block.  Every byte
// crosses HBM once, in transfers of R * B elements.  A CTA reads its whole
// chunk before it writes any of it, so dX may alias dY.
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

namespace bsp {
namespace {

constexpr int kBwdThreads = 256;
// 16-byte chunks per lane kept in registers (rows up to 160 chunks, e.g. 9 blocks
// of 128 bf16); few enough registers for 3 or 4 blocks of 256 threads per SM,
// which a memory-bound kernel needs (8 chunks and 1 block per SM ran at 3.8 TB/s)
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

// MINB blocks of 256 threads per SM: 3 (79 registers) for layouts whose rows
// average more than 4 vectors per lane and for fp32, 4 (64 registers) for
// 16-bit layouts of shorter rows, which need the extra warps to keep as many
// bytes in flight
template <typename T, int BLK, int MINB>
__global__ void __launch_bounds__(kBwdThreads, MINB)
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

// ---------------------------------------------------------------- chunks ----
constexpr int kBwdChunkThreads = 128;
constexpr int kBwdChunkWarps = kBwdChunkThreads / 32;
constexpr int kBwdRegElems = 40;                 // row elements per lane and array held in registers
constexpr int kBwdChunkMaxBytes = 48 * 1024;     // largest chunk per array: two CTAs per SM at least

// Offset of dY's copy in shared memory (Y's copy starts at 0).
__host__ __device__ inline size_t bwd_chunk_second(int max_bytes) { return ((size_t)max_bytes + 127) & ~(size_t)127; }

template <typename T, int BLK>
__global__ void __launch_bounds__(kBwdChunkThreads, 4)
softmax_bwd_chunk_kernel(LayoutView L, const T* Y, const T* dY, T* dX, float scale) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int VPB = BLK / VEC;  // 16-byte vectors per row slice of one block
    constexpr int E = sizeof(T) == 4 ? 1 : 0;
    constexpr int KR = kBwdRegElems / VEC;  // vectors per lane and array kept in registers
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    __shared__ float part[kBwdChunkWarps];  // long rows: each warp's part of the dot product
    const int n_items = L.sm_n_items[E];
    const int64_t z = blockIdx.x / n_items;
    const int it = (int)(blockIdx.x % n_items);
    // the chunk: rows r0 .. r0+R-1 of the block-row whose blocks are the
    // consecutive ids p0 .. p0+nq-1
    const int4 item = reinterpret_cast<const int4*>(L.sm_items[E])[it];
    const int p0 = item.y, nq = item.z;
    const int r0 = item.w & 0xffff, R = item.w >> 16;
    const uint32_t slice = (uint32_t)R * BLK * sizeof(T);  // bytes of one block's part of the chunk
    uint8_t* gbuf_raw = smem_raw + bwd_chunk_second(L.sm_max_bytes[E]);
    const T* ys = reinterpret_cast<const T*>(smem_raw);
    T* gs = reinterpret_cast<T*>(gbuf_raw);
    const size_t first = ((z * L.nnz + p0) * BLK + r0) * BLK;  // element offset of the chunk's first slice
    tc::Abort ab{&abort_flag, L.status, L.wait_ns};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
        tc::mbar_arrive_expect_tx(&bar, 2 * slice * nq);
        for (int q = 0; q < nq; ++q) {
            const size_t o = first + (size_t)q * BLK * BLK;
            tc::bulk_load(tc::smem_u32(smem_raw + (size_t)q * slice), Y + o, slice, &bar);
            tc::bulk_load(tc::smem_u32(gbuf_raw + (size_t)q * slice), dY + o, slice, &bar);
        }
    }
    __syncthreads();
    const bool ok = tc::mbar_wait(&bar, 0, ab);
    if (__syncthreads_and(ok)) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int nvec = nq * VPB;
        // element index of vector v of row rr inside either copy
        auto at = [&](int rr, int v) { return ((size_t)(v / VPB) * R + rr) * BLK + (v % VPB) * VEC; };
        auto dot16 = [](const uint4& a, const uint4& b, float acc) {
            float x[VEC], y[VEC];
            unpack16<T>(a, x);
            unpack16<T>(b, y);
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc = fmaf(x[k], y[k], acc);
            return acc;
        };
        // dX = scale * y * (g - dot), written over g's place in dY's copy
        auto write16 = [&](size_t e, const uint4& a, const uint4& b, float dot) {
            float y[VEC], g[VEC];
            unpack16<T>(a, y);
            unpack16<T>(b, g);
#pragma unroll
            for (int k = 0; k < VEC; ++k) y[k] = scale * y[k] * (g[k] - dot);
            *reinterpret_cast<uint4*>(gs + e) = pack16<T>(y);
        };
        if (nvec <= 32 * KR) {
            // rows in registers: GS lanes a row (the fewest of 8, 16, 32 that
            // hold it), 32 / GS rows a warp, the dot product reduced within
            // the lane group.  All rows of a chunk have nvec vectors.
            auto rows_in_registers = [&](auto gs_tag) {
                constexpr int GS = decltype(gs_tag)::value;
                constexpr int RPW = 32 / GS;
                const int sub = lane / GS, gl = lane % GS;
                for (int base = warp * RPW; base < R; base += kBwdChunkWarps * RPW) {
                    const int rr = base + sub;
                    const int nv = rr < R ? nvec : 0;  // lanes of rows past the chunk hold nothing
                    uint4 yv[KR], gv[KR];
                    float dot = 0.f;
#pragma unroll
                    for (int k = 0; k < KR; ++k) {
                        const int v = gl + GS * k;
                        if (v < nv) {
                            yv[k] = *reinterpret_cast<const uint4*>(ys + at(rr, v));
                            gv[k] = *reinterpret_cast<const uint4*>(gs + at(rr, v));
                            dot = dot16(yv[k], gv[k], dot);
                        }
                    }
#pragma unroll
                    for (int o = GS >> 1; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
#pragma unroll
                    for (int k = 0; k < KR; ++k) {
                        const int v = gl + GS * k;
                        if (v < nv) write16(at(rr, v), yv[k], gv[k], dot);
                    }
                }
            };
            if (nvec <= 8 * KR) rows_in_registers(std::integral_constant<int, 8>{});
            else if (nvec <= 16 * KR) rows_in_registers(std::integral_constant<int, 16>{});
            else rows_in_registers(std::integral_constant<int, 32>{});
        } else {
            // long rows: wpr warps a row when the chunk has fewer rows than
            // warps (R is a power of two), each taking every wpr-th 32-vector
            // slice; a pass for the dot product and one that writes dX
            const int wpr = R >= kBwdChunkWarps ? 1 : kBwdChunkWarps / R;
            const int wr = warp % wpr;
            for (int rr = warp / wpr; rr < R; rr += kBwdChunkWarps / wpr) {
                float dot = 0.f;
                for (int v = lane + 32 * wr; v < nvec; v += 32 * wpr)
                    dot = dot16(*reinterpret_cast<const uint4*>(ys + at(rr, v)),
                                *reinterpret_cast<const uint4*>(gs + at(rr, v)), dot);
#pragma unroll
                for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if (wpr > 1) {
                    // every warp runs exactly one row here (R < warps), so the
                    // barrier is reached by all of them
                    if (lane == 0) part[warp] = dot;
                    __syncthreads();
                    const int w0 = (warp / wpr) * wpr;
                    dot = 0.f;
                    for (int k = 0; k < wpr; ++k) dot += part[w0 + k];
                }
                for (int v = lane + 32 * wr; v < nvec; v += 32 * wpr) {
                    const size_t e = at(rr, v);
                    write16(e, *reinterpret_cast<const uint4*>(ys + e), *reinterpret_cast<const uint4*>(gs + e), dot);
                }
            }
        }
        tc::fence_proxy_async_smem();  // generic-proxy writes -> visible to the bulk copy engine
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int q = 0; q < nq; ++q)
                tc::bulk_store(dX + first + (size_t)q * BLK * BLK, tc::smem_u32(gbuf_raw + (size_t)q * slice), slice);
            tc::bulk_commit();
            tc::bulk_wait_read_all();  // shared memory must outlive the reads of the stores
        }
    } else if (threadIdx.x == 0) {
        tc::mbar_drain(&bar, 0, ab);  // the wait ran out: the copies in land before the CTA exits
    }
}

// BSP_ERR_UNSUPPORTED: the layout's chunks are missing or too large for this
// kernel (the caller then takes softmax_bwd_kernel)
template <typename T, int BLK>
int bwd_chunk_launch(const bsp_layout_s* Lh, const void* Y, const void* dY, void* dX, int Z, float scale,
                     cudaStream_t s) {
    constexpr int E = sizeof(T) == 4 ? 1 : 0;
    const LayoutView& V = Lh->view;
    if (!V.sm_fits[E] || V.sm_max_bytes[E] > kBwdChunkMaxBytes) return BSP_ERR_UNSUPPORTED;
    const int64_t grid = (int64_t)Z * V.sm_n_items[E];
    if (grid == 0) return BSP_OK;
    if (grid > INT32_MAX) return BSP_ERR_UNSUPPORTED;
    const size_t smem = bwd_chunk_second(V.sm_max_bytes[E]) + (size_t)V.sm_max_bytes[E];
    auto kern = softmax_bwd_chunk_kernel<T, BLK>;
    // the opt-in counts the kernel's static shared memory as well
    if (smem + 1024 > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    kern<<<(unsigned)grid, kBwdChunkThreads, smem, s>>>(V, (const T*)Y, (const T*)dY, (T*)dX, scale);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T, int BLK>
int bwd_launch(const bsp_layout_s* L, const void* Y, const void* dY, void* dX, int Z, float scale,
               cudaStream_t s) {
    // the chunk kernel when a row is too long for this kernel's registers
    // (which would take the two-pass loop over global memory); with every row
    // in registers this kernel keeps more loads in flight than a chunk's
    // copy-compute-store sequence
    if ((int64_t)L->max_row_nnz * BLK * (int64_t)sizeof(T) / 16 > 32 * kRegChunks) {
        const int rc = bwd_chunk_launch<T, BLK>(L, Y, dY, dX, Z, scale, s);
        if (rc != BSP_ERR_UNSUPPORTED) return rc;
    }
    const int64_t rows = (int64_t)Z * L->H * L->nb * BLK;
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 16);
    // mean 16-byte vectors per row over the layout's block-rows
    const int64_t per_row = L->nnz * BLK * (int64_t)sizeof(T) / 16 / std::max<int64_t>((int64_t)L->H * L->nb, 1);
    const unsigned g = (unsigned)std::max<int64_t>(blocks, 1);
    bool four = false;
    if constexpr (sizeof(T) == 2) four = per_row <= 4 * 32;  // fp32 spills at 64 registers
    if (four) {
        if constexpr (sizeof(T) == 2)
            softmax_bwd_kernel<T, BLK, 4><<<g, kBwdThreads, 0, s>>>(L->view, (const T*)Y, (const T*)dY, (T*)dX, Z,
                                                                     scale);
    } else {
        softmax_bwd_kernel<T, BLK, 3><<<g, kBwdThreads, 0, s>>>(L->view, (const T*)Y, (const T*)dY, (T*)dX, Z, scale);
    }
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
