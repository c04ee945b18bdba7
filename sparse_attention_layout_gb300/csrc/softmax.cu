// Block-sparse row softmax on the block-compressed SDD output.
//
// "question on blocksparse" (openai/triton issue 117): the softmax reduces
// each row of the SDD output across the row's present blocks and equals the
// dense softmax restricted to those entries; dense masks remove entries inside
// blocks.  Row reduction follows the Triton-Puzzles blog, Puzzle 8 "Long
// Softmax": subtract the row max, exponentiate in base 2 with a log2(e)
// prescale, divide by the sum; rows too long for registers merge per-lane
// (max, sum) pairs with the online update sum' = sum * exp(m1 - m2) + ...
//
// Design: one warp per row, 16-byte vector loads.  A row of block-row i spans
// nnz_i separate B-element slices (one per present block), each a contiguous
// run inside its block.  Rows that fit in registers (<= 32*MAXV vectors) are
// read once and written once: exactly the algorithmic bytes.  Longer rows take
// an online (max, sum) pass and a normalising pass.
#include <cfloat>

#include "common.cuh"

namespace bsp {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxVec = 8;  // 16-byte vectors per lane held in registers

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
struct RowCtx {
    static constexpr int VEC = 16 / sizeof(T);
    const LayoutView& L;
    int64_t z;
    int r, i, a, p0, vpb;
    float c2;  // scale * log2(e)
    int kind;
    const uint8_t* mask;

    __device__ __forceinline__ int64_t offset(int v, int& col) const {
        const int q = v / vpb, e = (v - q * vpb) * VEC;
        const int64_t n = L.blk_id[p0 + q];
        col = L.col_idx[p0 + q] * L.B + e;
        return ((z * L.nnz + n) * L.B + a) * (int64_t)L.B + e;
    }
    // load one vector, scale into the log2 domain, masked entries -> -inf
    __device__ __forceinline__ void load(const T* X, int v, float (&x)[VEC], int64_t& off) const {
        int col;
        off = offset(v, col);
        Vec16<T>::load(X + off, x);
#pragma unroll
        for (int k = 0; k < VEC; ++k) x[k] *= c2;
        if (kind == BSP_MASK_DIAG_CAUSAL) {
            if (col / L.B == i) {
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    if (col + k > r) x[k] = -INFINITY;
            }
        } else if (kind == BSP_MASK_DENSE) {
            const uint8_t* mp = mask + (int64_t)r * L.S + col;
            uint8_t mb[VEC];
            if constexpr (VEC == 8) {
                *reinterpret_cast<uint2*>(mb) = *reinterpret_cast<const uint2*>(mp);
            } else {
                *reinterpret_cast<uint32_t*>(mb) = *reinterpret_cast<const uint32_t*>(mp);
            }
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                if (!mb[k]) x[k] = -INFINITY;
        }
    }
};

template <typename T>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
softmax_rows_kernel(LayoutView L, const T* X, T* Y, int64_t rows_total, float c2, int kind,
                    const uint8_t* __restrict__ mask) {
    using V = Vec16<T>;
    constexpr int VEC = V::N;
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (w >= rows_total) return;
    const int S = L.S, B = L.B;
    const int r = (int)(w % S);
    const int64_t zh = w / S;
    const int h = (int)(zh % L.H);
    const int i = r / B;
    const int p0 = L.row_ptr[h * (L.nb + 1) + i];
    const int p1 = L.row_ptr[h * (L.nb + 1) + i + 1];
    RowCtx<T> ctx{L, zh / L.H, r, i, r - i * B, p0, B / VEC, c2, kind, mask};
    const int nvec = (p1 - p0) * ctx.vpb;
    if (nvec == 0) return;

    if (nvec <= 32 * kMaxVec) {
        // whole row in registers: one read, one write
        float x[kMaxVec][VEC];
        int64_t off[kMaxVec];
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxVec; ++k) {
            const int v = lane + 32 * k;
            if (v < nvec) {
                ctx.load(X, v, x[k], off[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, x[k][e]);
            }
        }
        m = warp_max(m);
        float l = 0.f;
        if (m != -INFINITY) {
#pragma unroll
            for (int k = 0; k < kMaxVec; ++k) {
                if (lane + 32 * k < nvec) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        x[k][e] = exp2f(x[k][e] - m);
                        l += x[k][e];
                    }
                }
            }
            l = warp_sum(l);
        }
        const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
        for (int k = 0; k < kMaxVec; ++k) {
            if (lane + 32 * k < nvec) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) x[k][e] = (m != -INFINITY) ? x[k][e] * inv : 0.f;
                V::store(Y + off[k], x[k]);
            }
        }
        return;
    }

    // long row: online (max, sum) per lane, merged across the warp, then a
    // normalising pass that re-reads the row
    float m = -INFINITY, l = 0.f;
    for (int v = lane; v < nvec; v += 32) {
        float x[VEC];
        int64_t off;
        ctx.load(X, v, x, off);
        float vm = -INFINITY;
#pragma unroll
        for (int e = 0; e < VEC; ++e) vm = fmaxf(vm, x[e]);
        if (vm > m) {
            l = (m == -INFINITY) ? 0.f : l * exp2f(m - vm);
            m = vm;
        }
        if (m != -INFINITY) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) l += exp2f(x[e] - m);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        const float mn = fmaxf(m, m2);
        const float a1 = (m == -INFINITY) ? 0.f : l * exp2f(m - mn);
        const float a2 = (m2 == -INFINITY) ? 0.f : l2 * exp2f(m2 - mn);
        l = a1 + a2;
        m = mn;
    }
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    for (int v = lane; v < nvec; v += 32) {
        float x[VEC];
        int64_t off;
        ctx.load(X, v, x, off);
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[e] = (m != -INFINITY) ? exp2f(x[e] - m) * inv : 0.f;
        V::store(Y + off, x);
    }
}

template <typename T>
int launch_t(const bsp_layout_s* Lh, const void* X, void* Y, int Z, float scale, int kind,
             const uint8_t* mask, cudaStream_t s) {
    const int64_t rows = (int64_t)Z * Lh->H * Lh->S;
    if (rows == 0) return BSP_OK;
    const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > INT32_MAX) return BSP_ERR_UNSUPPORTED;
    softmax_rows_kernel<T><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, s>>>(
        Lh->view, (const T*)X, (T*)Y, rows, scale * kLog2e, kind, mask);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

}  // namespace

int launch_softmax(const bsp_layout_s* L, int dtype, const void* X, void* Y, int Z, float scale,
                   int kind, const uint8_t* mask, cudaStream_t s) {
    switch (dtype) {
        case BSP_F32: return launch_t<float>(L, X, Y, Z, scale, kind, mask, s);
        case BSP_BF16: return launch_t<__nv_bfloat16>(L, X, Y, Z, scale, kind, mask, s);
        case BSP_F16: return launch_t<__half>(L, X, Y, Z, scale, kind, mask, s);
        default: return BSP_ERR_INVALID_ARG;
    }
}

}  // namespace bsp
