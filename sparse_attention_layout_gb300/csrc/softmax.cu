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
// Design.  A row of block-row i spans nnz_i separate B-element slices (one per
// present block); R consecutive rows of one block are contiguous.  The main
// kernel (softmax_chunk_kernel) moves an R-row chunk of a block-row with one
// bulk copy per block into shared memory and back, so every byte crosses HBM
// once in large transfers.  Rows too long for a 64 KB chunk fall back to
// softmax_rows_kernel: one warp per row with 16-byte loads straight from
// global memory (register-resident when the row fits, else an online pass and
// a normalising pass).
#include <cfloat>
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

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

// ---------------------------------------------------------------- chunks ----
// One CTA per (z, h, block-row i, chunk of R consecutive rows).  Rows r0..r0+R-1
// of one block are R*B contiguous elements, so the chunk arrives as nnz_i bulk
// copies (one per present block) into shared memory and leaves the same way:
// every HBM byte moves once, in large contiguous transfers.  Warps then own
// rows: an online (max, sum) pass and a normalising pass over shared memory.
// Several CTAs per SM overlap one CTA's transfers with another's arithmetic.
// 4 warps: with 64 registers a thread, 8 CTAs share an SM, so that with
// chunks of about 24 KB eight chunks are in flight per SM, each CTA in its own
// phase (copy in, arithmetic, copy out)
constexpr int kChunkThreads = 128;
constexpr int kChunkRegElems = 40;  // row elements per lane held in registers

// Chunks come from the layout's list for this element size: each block-row is
// cut into chunks of the largest power-of-two row count that fits the budget.
template <typename T, int BLK>
__global__ void __launch_bounds__(kChunkThreads, 8)
softmax_chunk_kernel(LayoutView L, const T* X, T* Y, float c2, int kind, const uint8_t* __restrict__ mask) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int VPB = BLK / VEC;  // 16-byte vectors per row slice of one block
    constexpr int E = sizeof(T) == 4 ? 1 : 0;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    __shared__ float2 part[kChunkThreads / 32];  // long rows: each warp's (max, sum) of its part
    const int n_items = L.sm_n_items[E];
    const int64_t z = blockIdx.x / n_items;
    const int it = (int)(blockIdx.x % n_items);
    // one 16-byte load describes the chunk; the blocks of block-row i are the
    // consecutive ids p0 .. p0+nq-1 (ids are CSR positions)
    const int4 item = reinterpret_cast<const int4*>(L.sm_items[E])[it];
    const int key = item.x, p0 = item.y, nq = item.z;
    const int r0 = item.w & 0xffff, R = item.w >> 16;
    const int i = key % L.nb;  // block-row (the chunk's head is key / nb)
    const uint32_t slice = (uint32_t)R * BLK * sizeof(T);  // bytes of one block's part of the chunk
    T* buf = reinterpret_cast<T*>(smem_raw);
    int* scol = reinterpret_cast<int*>(smem_raw + L.sm_max_bytes[E]);
    tc::Abort ab{&abort_flag, L.status, L.wait_ns};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
        tc::mbar_arrive_expect_tx(&bar, slice * nq);
        const T* src = X + ((z * L.nnz + p0) * BLK + r0) * BLK;
        for (int q = 0; q < nq; ++q)
            tc::bulk_load(tc::smem_u32(smem_raw + (size_t)q * slice), src + (size_t)q * BLK * BLK, slice, &bar);
    }
    if (kind != BSP_MASK_NONE)
        for (int q = threadIdx.x; q < nq; q += kChunkThreads) scol[q] = L.col_idx[p0 + q];
    __syncthreads();
    const bool ok = tc::mbar_wait(&bar, 0, ab);
    if (__syncthreads_and(ok)) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int nvec = nq * VPB;
        // raw values of vector v of row rr (the scale is folded into the
        // exponent), masked -> -inf
        auto load = [&](int rr, int v, float (&x)[VEC], T*& p) {
            const int r = r0 + rr;           // row inside the block-row
            const int rseq = i * BLK + r;    // row inside the sequence
            const int q = v / VPB, e = v % VPB;
            p = buf + ((size_t)q * R + rr) * BLK + e * VEC;
            Vec16<T>::load(p, x);
            const int col = scol[q] * BLK + e * VEC;
            if (kind == BSP_MASK_DIAG_CAUSAL) {
                if (scol[q] == i) {
#pragma unroll
                    for (int k = 0; k < VEC; ++k)
                        if (e * VEC + k > r) x[k] = -INFINITY;
                }
            } else if (kind == BSP_MASK_DENSE) {
                const uint8_t* mp = mask + (int64_t)rseq * L.S + col;
#pragma unroll
                for (int k = 0; k < VEC; ++k)
                    if (!mp[k]) x[k] = -INFINITY;
            }
        };
        constexpr int kRegVec = kChunkRegElems / VEC;  // vectors per lane kept in registers
        if (nvec <= 32 * kRegVec) {
            // rows in registers: GS lanes per row (the fewest of 8, 16, 32 that
            // hold the row), 32 / GS rows per warp, reductions within the lane
            // group; max, then 2^(x c2 - m c2) (one FFMA + one MUFU per entry),
            // sum, normalise, store -- one pass over shared memory.  A chunk's
            // rows all have nvec vectors (one block-row), so GS is uniform.
            auto rows_in_registers = [&](auto gs_tag) {
                constexpr int GS = decltype(gs_tag)::value;
                constexpr int RPW = 32 / GS;
                const int sub = lane / GS, gl = lane % GS;
                for (int base = warp * RPW; base < R; base += (kChunkThreads / 32) * RPW) {
                    const int rr = base + sub;
                    const int nv = rr < R ? nvec : 0;  // lanes of rows past the chunk hold nothing
                    float x[kRegVec][VEC];
                    float m = -INFINITY;
#pragma unroll
                    for (int k = 0; k < kRegVec; ++k) {
                        if (gl + GS * k < nv) {
                            T* p;
                            load(rr, gl + GS * k, x[k], p);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) m = fmaxf(m, x[k][e]);
                        }
                    }
#pragma unroll
                    for (int o = GS >> 1; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    const float ms = (m == -INFINITY) ? 0.f : m * c2;
                    float l = 0.f;
#pragma unroll
                    for (int k = 0; k < kRegVec; ++k) {
                        if (gl + GS * k < nv) {
#pragma unroll
                            for (int e = 0; e < VEC; ++e) {
                                x[k][e] = tc::ex2_approx(fmaf(x[k][e], c2, -ms));
                                l += x[k][e];
                            }
                        }
                    }
#pragma unroll
                    for (int o = GS >> 1; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                    const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
                    for (int k = 0; k < kRegVec; ++k) {
                        const int v = gl + GS * k;
                        if (v < nv) {
#pragma unroll
                            for (int e = 0; e < VEC; ++e) x[k][e] *= inv;
                            Vec16<T>::store(buf + ((size_t)(v / VPB) * R + rr) * BLK + (v % VPB) * VEC, x[k]);
                        }
                    }
                }
            };
            if (nvec <= 8 * kRegVec) rows_in_registers(std::integral_constant<int, 8>{});
            else if (nvec <= 16 * kRegVec) rows_in_registers(std::integral_constant<int, 16>{});
            else rows_in_registers(std::integral_constant<int, 32>{});
        } else {
            // long rows: wpr warps per row when the chunk has fewer rows than
            // warps (R is a power of two), each taking every wpr-th 32-vector
            // slice of it; R >= warps: one warp per row
            constexpr int NW = kChunkThreads / 32;
            const int wpr = R >= NW ? 1 : NW / R;
            const int wr = warp % wpr;
            for (int rr = warp / wpr; rr < R; rr += NW / wpr) {
                // online (max, sum) per lane in the scaled log2 domain, merged
                // across the warp (and across the row's warps through shared
                // memory), then a normalising pass
                float m = -INFINITY, l = 0.f;
                for (int v = lane + 32 * wr; v < nvec; v += 32 * wpr) {
                    float x[VEC];
                    T* p;
                    load(rr, v, x, p);
                    float vm = -INFINITY;
    #pragma unroll
                    for (int k = 0; k < VEC; ++k) vm = fmaxf(vm, x[k]);
                    vm *= c2;
                    if (vm > m) {
                        l = (m == -INFINITY) ? 0.f : l * tc::ex2_approx(m - vm);
                        m = vm;
                    }
                    if (m != -INFINITY) {
    #pragma unroll
                        for (int k = 0; k < VEC; ++k) l += tc::ex2_approx(fmaf(x[k], c2, -m));
                    }
                }
    #pragma unroll
                for (int o = 16; o; o >>= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
                    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
                    const float mn = fmaxf(m, m2);
                    l = ((m == -INFINITY) ? 0.f : l * tc::ex2_approx(m - mn)) +
                        ((m2 == -INFINITY) ? 0.f : l2 * tc::ex2_approx(m2 - mn));
                    m = mn;
                }
                if (wpr > 1) {
                    // every warp runs exactly one row here (R < NW), so the
                    // barriers are reached by all of them
                    if (lane == 0) part[warp] = make_float2(m, l);
                    __syncthreads();
                    const int w0 = (warp / wpr) * wpr;
                    float mr = -INFINITY;
                    for (int k = 0; k < wpr; ++k) mr = fmaxf(mr, part[w0 + k].x);
                    float lr = 0.f;
                    if (mr != -INFINITY)
                        for (int k = 0; k < wpr; ++k) {
                            const float2 pk = part[w0 + k];
                            if (pk.x != -INFINITY) lr += pk.y * tc::ex2_approx(pk.x - mr);
                        }
                    m = mr;
                    l = lr;
                }
                const float inv = l > 0.f ? 1.0f / l : 0.f;
                const float ms = (m == -INFINITY) ? 0.f : m;
                for (int v = lane + 32 * wr; v < nvec; v += 32 * wpr) {
                    float x[VEC];
                    T* p;
                    load(rr, v, x, p);
    #pragma unroll
                    for (int k = 0; k < VEC; ++k) x[k] = tc::ex2_approx(fmaf(x[k], c2, -ms)) * inv;
                    Vec16<T>::store(p, x);
                }
            }
        }
        tc::fence_proxy_async_smem();  // generic-proxy writes -> visible to the bulk copy engine
        __syncthreads();
        if (threadIdx.x == 0) {
            T* dst = Y + ((z * L.nnz + p0) * BLK + r0) * BLK;
            for (int q = 0; q < nq; ++q)
                tc::bulk_store(dst + (size_t)q * BLK * BLK, tc::smem_u32(smem_raw + (size_t)q * slice), slice);
            tc::bulk_commit();
            tc::bulk_wait_read_all();  // shared memory must outlive the reads of the stores
        }
    } else if (threadIdx.x == 0) {
        tc::mbar_drain(&bar, 0, ab);  // the wait ran out: the copies in land before the CTA exits
    }
}

template <typename T, int BLK>
int launch_chunk(const bsp_layout_s* Lh, const void* X, void* Y, int Z, float scale, int kind,
                 const uint8_t* mask, cudaStream_t s) {
    constexpr int E = sizeof(T) == 4 ? 1 : 0;
    const LayoutView& V = Lh->view;
    if (!V.sm_fits[E]) return BSP_ERR_UNSUPPORTED;  // some row longer than one chunk
    if (V.sm_n_items[E] == 0) return BSP_OK;
    const size_t smem = (size_t)V.sm_max_bytes[E] + (size_t)Lh->max_row_nnz * sizeof(int);
    const int64_t grid = (int64_t)Z * V.sm_n_items[E];
    if (grid > INT32_MAX) return BSP_ERR_UNSUPPORTED;
    auto kern = softmax_chunk_kernel<T, BLK>;
    // the opt-in counts the kernel's static shared memory as well
    if (smem + 1024 > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    kern<<<(unsigned)grid, kChunkThreads, smem, s>>>(V, (const T*)X, (T*)Y, scale * kLog2e, kind, mask);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int launch_t(const bsp_layout_s* Lh, const void* X, void* Y, int Z, float scale, int kind,
             const uint8_t* mask, cudaStream_t s) {
    int rc = BSP_ERR_UNSUPPORTED;
    switch (Lh->B) {
        case 16: rc = launch_chunk<T, 16>(Lh, X, Y, Z, scale, kind, mask, s); break;
        case 32: rc = launch_chunk<T, 32>(Lh, X, Y, Z, scale, kind, mask, s); break;
        case 64: rc = launch_chunk<T, 64>(Lh, X, Y, Z, scale, kind, mask, s); break;
        case 128: rc = launch_chunk<T, 128>(Lh, X, Y, Z, scale, kind, mask, s); break;
    }
    if (rc != BSP_ERR_UNSUPPORTED) return rc;
    // rows too long for one chunk: one warp per row, streaming from global memory
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
