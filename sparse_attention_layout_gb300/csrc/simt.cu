// CUDA-core (FFMA) kernels for every op and dtype: the fp32 path, and the
// path for shapes the tensor-core kernels do not cover.  fp32 accumulation.
//
// Operations ("question on blocksparse", openai/triton issue 117):
//   SDD  C_blk(h,i,j) = op(A)[iB.., :] . op(B)[:, jB..]   on present blocks
//   DSD  C = op(A_sp) . op(B)      (lhs block-sparse)
//   DDS  C = op(A) . op(B_sp)      (rhs block-sparse)
// and the fused SDD -> softmax -> DSD attention chain, with the online-softmax
// recurrence of the Triton-Puzzles blog, Puzzle 9 "Simple FlashAttention":
//   m2 = max(m1, rowmax(s)),  l2 = l1 exp(m1 - m2) + sum exp(s - m2),
//   o2 = o1 exp(m1 - m2) + sum exp(s - m2) v       (divided by l at the end).
#include <type_traits>

#include "common.cuh"

namespace bsp {
namespace {

constexpr int kThreads = 256;  // 16 x 16 thread grid in every kernel here

// asynchronous 16-byte global -> shared copies (both addresses 16-byte aligned)
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
constexpr int KC = 16;         // contraction chunk staged in shared memory

// ---------------------------------------------------------------- SDD ----
// One CTA per (z, block n).  Thread (ty, tx) owns rows ty + 16u, columns
// tx + 16v of the BS x BS block (u, v < BS/16).
template <typename T, int BS>
__global__ void __launch_bounds__(kThreads)
sdd_simt_kernel(LayoutView L, const T* __restrict__ A, const T* __restrict__ Bm, T* __restrict__ C,
                int Z, int K, int ta, int tb) {
    constexpr int R = BS / 16;
    __shared__ float As[KC][BS + 1];
    __shared__ float Bs[KC][BS + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int64_t total = (int64_t)Z * L.nnz;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t z = w / L.nnz, n = w % L.nnz;
        const int key = L.blk_key[n];
        const int h = key / L.nb, i = key % L.nb;
        // block-column of n: position n in CSR order holds it (ids are CSR ranks)
        const int j = L.col_idx[n];
        const int64_t zh = z * L.H + h;
        const int64_t S = L.S;
        float acc[R][R];
#pragma unroll
        for (int u = 0; u < R; ++u)
#pragma unroll
            for (int v = 0; v < R; ++v) acc[u][v] = 0.f;
        for (int k0 = 0; k0 < K; k0 += KC) {
            for (int e = threadIdx.x; e < KC * BS; e += kThreads) {
                int kk, a;
                if (ta) { kk = e / BS; a = e % BS; } else { a = e / KC; kk = e % KC; }
                const int k = k0 + kk;
                float va = 0.f, vb = 0.f;
                if (k < K) {
                    const int64_t row = (int64_t)i * BS + a, col = (int64_t)j * BS + a;
                    va = to_f32(ta ? A[(zh * K + k) * S + row] : A[(zh * S + row) * K + k]);
                    vb = to_f32(tb ? Bm[(zh * S + col) * K + k] : Bm[(zh * K + k) * S + col]);
                }
                As[kk][a] = va;
                Bs[kk][a] = vb;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < KC; ++kk) {
                float ra[R], rb[R];
#pragma unroll
                for (int u = 0; u < R; ++u) ra[u] = As[kk][ty + 16 * u];
#pragma unroll
                for (int v = 0; v < R; ++v) rb[v] = Bs[kk][tx + 16 * v];
#pragma unroll
                for (int u = 0; u < R; ++u)
#pragma unroll
                    for (int v = 0; v < R; ++v) acc[u][v] = fmaf(ra[u], rb[v], acc[u][v]);
            }
            __syncthreads();
        }
        T* out = C + w * BS * BS;
#pragma unroll
        for (int u = 0; u < R; ++u)
#pragma unroll
            for (int v = 0; v < R; ++v) out[(ty + 16 * u) * BS + tx + 16 * v] = from_f32<T>(acc[u][v]);
    }
}

// ---------------------------------------------------------------- DSD ----
// One CTA per (z, h, block-row i of op(A_sp), 64-column tile of C).
// op(A_sp) row i: CSR row i (trans_a = 0) or CSC column i (trans_a = 1).
template <typename T, int BS>
__global__ void __launch_bounds__(kThreads)
dsd_simt_kernel(LayoutView L, const T* __restrict__ Asp, const T* __restrict__ Bd,
                T* __restrict__ C, int Z, int N, int ta, int tb) {
    constexpr int R = BS / 16;  // rows per thread
    constexpr int NT = 64;      // C columns per CTA, 4 per thread
    __shared__ float As[KC][BS + 1];
    __shared__ float Bs[KC][NT + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int ntiles = (N + NT - 1) / NT;
    const int64_t units = (int64_t)L.H * L.nb;
    const int64_t total = units * Z * ntiles;
    const int64_t S = L.S;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t rank = w / ((int64_t)Z * ntiles);
        const int rem = (int)(w % ((int64_t)Z * ntiles));
        const int64_t z = rem / ntiles;
        const int n0 = (rem % ntiles) * NT;
        const int key = L.row_order[rank];  // same ordering used for both trans (nnz-balanced)
        const int h = key / L.nb, i = key % L.nb;
        const int64_t zh = z * L.H + h;
        const int32_t* ptr = ta ? L.col_ptr : L.row_ptr;
        const int32_t* idx = ta ? L.row_idx : L.col_idx;
        const int32_t* bid = ta ? L.blk_id_csc : L.blk_id;
        const int q0 = ptr[h * (L.nb + 1) + i], q1 = ptr[h * (L.nb + 1) + i + 1];
        float acc[R][4];
#pragma unroll
        for (int u = 0; u < R; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
        for (int q = q0; q < q1; ++q) {
            const int j = idx[q];
            const T* blk = Asp + ((int64_t)z * L.nnz + bid[q]) * BS * BS;
            for (int c0 = 0; c0 < BS; c0 += KC) {
                for (int e = threadIdx.x; e < KC * BS; e += kThreads) {
                    const int a = e / KC, cc = e % KC;  // op(A)[a][c0+cc]
                    As[cc][a] = to_f32(ta ? blk[(c0 + cc) * BS + a] : blk[a * BS + c0 + cc]);
                }
                for (int e = threadIdx.x; e < KC * NT; e += kThreads) {
                    int cc, nn;
                    if (tb) { nn = e / KC; cc = e % KC; } else { cc = e / NT; nn = e % NT; }
                    const int64_t krow = (int64_t)j * BS + c0 + cc;
                    const int n = n0 + nn;
                    float v = 0.f;
                    if (n < N) v = to_f32(tb ? Bd[(zh * N + n) * S + krow] : Bd[(zh * S + krow) * N + n]);
                    Bs[cc][nn] = v;
                }
                __syncthreads();
#pragma unroll
                for (int cc = 0; cc < KC; ++cc) {
                    float ra[R], rb[4];
#pragma unroll
                    for (int u = 0; u < R; ++u) ra[u] = As[cc][ty + 16 * u];
#pragma unroll
                    for (int v = 0; v < 4; ++v) rb[v] = Bs[cc][tx + 16 * v];
#pragma unroll
                    for (int u = 0; u < R; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(ra[u], rb[v], acc[u][v]);
                }
                __syncthreads();
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int64_t row = (int64_t)i * BS + ty + 16 * u;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int n = n0 + tx + 16 * v;
                if (n < N) C[(zh * S + row) * N + n] = from_f32<T>(acc[u][v]);
            }
        }
    }
}

// ---------------------------------------------------------------- DDS ----
// One CTA per (z, h, block-column j of op(B_sp), 64-row tile of C).
// op(B_sp) column j: CSC column j (trans_b = 0) or CSR row j (trans_b = 1).
template <typename T, int BS>
__global__ void __launch_bounds__(kThreads)
dds_simt_kernel(LayoutView L, const T* __restrict__ Ad, const T* __restrict__ Bsp,
                T* __restrict__ C, int Z, int M, int ta, int tb) {
    constexpr int R = BS / 16;  // columns per thread
    constexpr int MT = 64;      // C rows per CTA, 4 per thread
    __shared__ float As[KC][MT + 1];
    __shared__ float Bs[KC][BS + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int mtiles = (M + MT - 1) / MT;
    const int64_t units = (int64_t)L.H * L.nb;
    const int64_t total = units * Z * mtiles;
    const int64_t S = L.S;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t rank = w / ((int64_t)Z * mtiles);
        const int rem = (int)(w % ((int64_t)Z * mtiles));
        const int64_t z = rem / mtiles;
        const int m0 = (rem % mtiles) * MT;
        const int key = tb ? L.row_order[rank] : L.col_order[rank];
        const int h = key / L.nb, j = key % L.nb;
        const int64_t zh = z * L.H + h;
        const int32_t* ptr = tb ? L.row_ptr : L.col_ptr;
        const int32_t* idx = tb ? L.col_idx : L.row_idx;
        const int32_t* bid = tb ? L.blk_id : L.blk_id_csc;
        const int q0 = ptr[h * (L.nb + 1) + j], q1 = ptr[h * (L.nb + 1) + j + 1];
        float acc[4][R];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < R; ++v) acc[u][v] = 0.f;
        for (int q = q0; q < q1; ++q) {
            const int i = idx[q];  // block-row of op(B_sp) = contraction block
            const T* blk = Bsp + ((int64_t)z * L.nnz + bid[q]) * BS * BS;
            for (int k0 = 0; k0 < BS; k0 += KC) {
                for (int e = threadIdx.x; e < KC * MT; e += kThreads) {
                    int kk, mm;
                    if (ta) { kk = e / MT; mm = e % MT; } else { mm = e / KC; kk = e % KC; }
                    const int64_t kcol = (int64_t)i * BS + k0 + kk;
                    const int m = m0 + mm;
                    float v = 0.f;
                    if (m < M) v = to_f32(ta ? Ad[(zh * S + kcol) * M + m] : Ad[(zh * M + m) * S + kcol]);
                    As[kk][mm] = v;
                }
                for (int e = threadIdx.x; e < KC * BS; e += kThreads) {
                    const int kk = e / BS, b = e % BS;  // op(B)[k0+kk][b]
                    Bs[kk][b] = to_f32(tb ? blk[b * BS + k0 + kk] : blk[(k0 + kk) * BS + b]);
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < KC; ++kk) {
                    float ra[4], rb[R];
#pragma unroll
                    for (int u = 0; u < 4; ++u) ra[u] = As[kk][ty + 16 * u];
#pragma unroll
                    for (int v = 0; v < R; ++v) rb[v] = Bs[kk][tx + 16 * v];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int v = 0; v < R; ++v) acc[u][v] = fmaf(ra[u], rb[v], acc[u][v]);
                }
                __syncthreads();
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int m = m0 + ty + 16 * u;
            if (m >= M) continue;
#pragma unroll
            for (int v = 0; v < R; ++v)
                C[(zh * M + m) * S + (int64_t)j * BS + tx + 16 * v] = from_f32<T>(acc[u][v]);
        }
    }
}

// ---------------------------------------------------------- attention ----
// One CTA per (z, h, block-row i, chunk of TR = min(B, 64) rows).  Keys are
// visited block by block along the row's CSR list, TR keys at a time.  Thread
// (ty, tx) owns score rows ty + 16u and keys tx + 16v of a chunk, and output
// rows ty + 16u, columns tx + 16d.  Each 16-thread half-warp owns whole rows,
// so row max / sum are half-warp shuffles.
template <typename T, int TR>
__global__ void __launch_bounds__(kThreads)
attention_simt_kernel(LayoutView L, const T* __restrict__ Q, const T* __restrict__ K,
                      const T* __restrict__ V, T* __restrict__ O, float* __restrict__ lse, int Z, int D, float c2,
                      int kind, const uint8_t* __restrict__ mask) {
    constexpr int R = TR / 16;
    constexpr int DMAX = 128;
    constexpr int DR = DMAX / 16;  // output columns per thread (upper bound)
    extern __shared__ float smem[];
    const int DP = D + 1;
    float* Qs = smem;              // [TR][DP]
    float* Ks = Qs + TR * DP;      // [TR][DP]
    float* Vs = Ks + TR * DP;      // [TR][DP]
    float* Ps = Vs + TR * DP;      // [TR][TR + 1]
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int B = L.B, S = L.S;
    const int nsub = B / TR;
    const int64_t total = (int64_t)L.H * L.nb * Z * nsub;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t rank = w / ((int64_t)Z * nsub);
        const int rem = (int)(w % ((int64_t)Z * nsub));
        const int64_t z = rem / nsub;
        const int sub = rem % nsub;
        const int key = L.row_order[rank];
        const int h = key / L.nb, i = key % L.nb;
        const int64_t zh = z * L.H + h;
        const int r0 = i * B + sub * TR;  // first query row of this CTA
        for (int e = threadIdx.x; e < TR * D; e += kThreads) {
            const int rr = e / D, d = e % D;
            Qs[rr * DP + d] = to_f32(Q[(zh * S + r0 + rr) * D + d]) * c2;
        }
        float m[R], l[R], acc[R][DR];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            m[u] = -INFINITY;
            l[u] = 0.f;
#pragma unroll
            for (int d = 0; d < DR; ++d) acc[u][d] = 0.f;
        }
        const int q0 = L.row_ptr[h * (L.nb + 1) + i], q1 = L.row_ptr[h * (L.nb + 1) + i + 1];
        for (int q = q0; q < q1; ++q) {
            const int j = L.col_idx[q];
            for (int kc = 0; kc < B; kc += TR) {
                const int c0 = j * B + kc;  // first key row of the chunk
                __syncthreads();  // previous chunk fully consumed (and Qs written)
                for (int e = threadIdx.x; e < TR * D; e += kThreads) {
                    const int cc = e / D, d = e % D;
                    Ks[cc * DP + d] = to_f32(K[(zh * S + c0 + cc) * D + d]);
                    Vs[cc * DP + d] = to_f32(V[(zh * S + c0 + cc) * D + d]);
                }
                __syncthreads();
                float s[R][R];
#pragma unroll
                for (int u = 0; u < R; ++u)
#pragma unroll
                    for (int v = 0; v < R; ++v) s[u][v] = 0.f;
                for (int d = 0; d < D; ++d) {
                    float qa[R], kb[R];
#pragma unroll
                    for (int u = 0; u < R; ++u) qa[u] = Qs[(ty + 16 * u) * DP + d];
#pragma unroll
                    for (int v = 0; v < R; ++v) kb[v] = Ks[(tx + 16 * v) * DP + d];
#pragma unroll
                    for (int u = 0; u < R; ++u)
#pragma unroll
                        for (int v = 0; v < R; ++v) s[u][v] = fmaf(qa[u], kb[v], s[u][v]);
                }
                // intra-block mask
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    const int r = r0 + ty + 16 * u;
#pragma unroll
                    for (int v = 0; v < R; ++v) {
                        const int c = c0 + tx + 16 * v;
                        bool keep = true;
                        if (kind == BSP_MASK_DIAG_CAUSAL) keep = (j != i) || (c <= r);
                        else if (kind == BSP_MASK_DENSE) keep = mask[(int64_t)r * S + c] != 0;
                        if (!keep) s[u][v] = -INFINITY;
                    }
                }
                // online softmax update per row
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    float cm = -INFINITY;
#pragma unroll
                    for (int v = 0; v < R; ++v) cm = fmaxf(cm, s[u][v]);
#pragma unroll
                    for (int o = 8; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
                    const float mn = fmaxf(m[u], cm);
                    float alpha = 1.f, rs = 0.f;
                    if (mn != -INFINITY) {
                        alpha = (m[u] == -INFINITY) ? 0.f : exp2f(m[u] - mn);
#pragma unroll
                        for (int v = 0; v < R; ++v) {
                            s[u][v] = exp2f(s[u][v] - mn);
                            rs += s[u][v];
                        }
                    } else {
#pragma unroll
                        for (int v = 0; v < R; ++v) s[u][v] = 0.f;
                    }
#pragma unroll
                    for (int o = 8; o; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
                    l[u] = l[u] * alpha + rs;
                    m[u] = mn;
#pragma unroll
                    for (int d = 0; d < DR; ++d) acc[u][d] *= alpha;
#pragma unroll
                    for (int v = 0; v < R; ++v) Ps[(ty + 16 * u) * (TR + 1) + tx + 16 * v] = s[u][v];
                }
                __syncthreads();
                for (int cc = 0; cc < TR; ++cc) {
                    float pa[R];
#pragma unroll
                    for (int u = 0; u < R; ++u) pa[u] = Ps[(ty + 16 * u) * (TR + 1) + cc];
#pragma unroll
                    for (int d = 0; d < DR; ++d) {
                        const int dd = tx + 16 * d;
                        if (dd < D) {
                            const float vv = Vs[cc * DP + dd];
#pragma unroll
                            for (int u = 0; u < R; ++u) acc[u][d] = fmaf(pa[u], vv, acc[u][d]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const float inv = l[u] > 0.f ? 1.0f / l[u] : 0.f;
            const int64_t r = r0 + ty + 16 * u;
            // the row's log-sum-exp of the scaled scores (natural log; -inf when
            // nothing is kept): m is in scaled log2 units
            if (lse && tx == 0) lse[zh * S + r] = l[u] > 0.f ? (m[u] + log2f(l[u])) * kLn2 : -INFINITY;
#pragma unroll
            for (int d = 0; d < DR; ++d) {
                const int dd = tx + 16 * d;
                if (dd < D) O[(zh * S + r) * D + dd] = from_f32<T>(acc[u][d] * inv);
            }
        }
        __syncthreads();  // Qs reused by the next work item
    }
}

int grid_for(int64_t total) {
    const int64_t cap = (int64_t)sm_count() * 16;
    return (int)(total < cap ? (total > 0 ? total : 1) : cap);
}

template <typename T>
int sdd_t(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int K, int ta,
          int tb, cudaStream_t s) {
    const int64_t total = (int64_t)Z * L->nnz;
    if (total == 0) return BSP_OK;
    const int g = grid_for(total);
    const T *a = (const T*)A, *b = (const T*)B;
    T* c = (T*)C;
    switch (L->B) {
        case 16: sdd_simt_kernel<T, 16><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, K, ta, tb); break;
        case 32: sdd_simt_kernel<T, 32><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, K, ta, tb); break;
        case 64: sdd_simt_kernel<T, 64><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, K, ta, tb); break;
        case 128: sdd_simt_kernel<T, 128><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, K, ta, tb); break;
        default: return BSP_ERR_INVALID_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int dsd_t(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int N, int ta,
          int tb, cudaStream_t s) {
    const int64_t total = (int64_t)L->H * L->nb * Z * ((N + 63) / 64);
    if (total == 0) return BSP_OK;
    const int g = grid_for(total);
    const T *a = (const T*)A, *b = (const T*)B;
    T* c = (T*)C;
    switch (L->B) {
        case 16: dsd_simt_kernel<T, 16><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, N, ta, tb); break;
        case 32: dsd_simt_kernel<T, 32><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, N, ta, tb); break;
        case 64: dsd_simt_kernel<T, 64><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, N, ta, tb); break;
        case 128: dsd_simt_kernel<T, 128><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, N, ta, tb); break;
        default: return BSP_ERR_INVALID_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int dds_t(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int M, int ta,
          int tb, cudaStream_t s) {
    const int64_t total = (int64_t)L->H * L->nb * Z * ((M + 63) / 64);
    if (total == 0) return BSP_OK;
    const int g = grid_for(total);
    const T *a = (const T*)A, *b = (const T*)B;
    T* c = (T*)C;
    switch (L->B) {
        case 16: dds_simt_kernel<T, 16><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, M, ta, tb); break;
        case 32: dds_simt_kernel<T, 32><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, M, ta, tb); break;
        case 64: dds_simt_kernel<T, 64><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, M, ta, tb); break;
        case 128: dds_simt_kernel<T, 128><<<g, kThreads, 0, s>>>(L->view, a, b, c, Z, M, ta, tb); break;
        default: return BSP_ERR_INVALID_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

// Register-tiled variant for B >= 64 and D = 64 or 128 (the fp32 workloads'
// head sizes).  Same work split, online recurrence and masks as above, but the
// shared-memory traffic is vectorised: rows are padded to D + 4 floats (an odd
// number of 16-byte units, so the strided row reads below hit distinct banks),
// Q K^T reads float4 along D (8 vector loads per 64 FMAs instead of one scalar
// load per 2 FMAs), and each thread owns 4 contiguous output columns per 64 so
// that P V reads V and P as float4 too.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2)
attention_simt_v4_kernel(LayoutView L, const T* __restrict__ Q, const T* __restrict__ K,
                         const T* __restrict__ V, T* __restrict__ O, float* __restrict__ lse, int Z, float c2,
                         int kind,
                         const uint8_t* __restrict__ mask) {
    constexpr int TR = 64, R = 4, DP = D + 4, PP = TR + 4, NG = D / 64, D4 = D / 4;
    // fp32 inputs: K and V chunks arrive by asynchronous 16-byte copies into two
    // buffers, the next chunk's while the current one is computed; 16-bit
    // inputs are converted on the way in (one buffer)
    constexpr bool ASYNC = std::is_same<T, float>::value;
    constexpr int NBUF = ASYNC ? 2 : 1;
    extern __shared__ float4 smem_v4[];
    float* Qs = reinterpret_cast<float*>(smem_v4);  // [TR][DP], pre-scaled by c2
    float* Ks = Qs + TR * DP;                        // [NBUF][TR][DP]
    float* Vs = Ks + NBUF * TR * DP;                 // [NBUF][TR][DP]
    float* Ps = Vs + NBUF * TR * DP;                 // [TR][PP]
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int B = L.B, S = L.S;
    const int nsub = B / TR;
    const int64_t total = (int64_t)L.H * L.nb * Z * nsub;
    auto load_tile = [&](float* dst, const T* src, float mul) {
        for (int e = threadIdx.x; e < TR * D4; e += kThreads) {
            const int rr = e / D4, c4 = e % D4;
            const T* p = src + (int64_t)rr * D + 4 * c4;
            *reinterpret_cast<float4*>(dst + rr * DP + 4 * c4) =
                make_float4(to_f32(p[0]) * mul, to_f32(p[1]) * mul, to_f32(p[2]) * mul, to_f32(p[3]) * mul);
        }
    };
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t rank = w / ((int64_t)Z * nsub);
        const int rem = (int)(w % ((int64_t)Z * nsub));
        const int64_t z = rem / nsub;
        const int sub = rem % nsub;
        const int key = L.row_order[rank];
        const int h = key / L.nb, i = key % L.nb;
        const int64_t zh = z * L.H + h;
        const int r0 = i * B + sub * TR;  // first query row of this CTA
        load_tile(Qs, Q + (zh * S + r0) * D, c2);
        float m[R], l[R];
        float2 acc[R][NG][2];  // output columns 4 tx + 64 g + {0, 1}, {2, 3}
#pragma unroll
        for (int u = 0; u < R; ++u) {
            m[u] = -INFINITY;
            l[u] = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
                for (int c = 0; c < 2; ++c) acc[u][g][c] = make_float2(0.f, 0.f);
        }
        const int q0 = L.row_ptr[h * (L.nb + 1) + i], q1 = L.row_ptr[h * (L.nb + 1) + i + 1];
        // chunks of TR key rows: nsub per present block, in CSR order
        const int nch = (q1 - q0) * nsub;
        auto chunk_row = [&](int t) { return L.col_idx[q0 + t / nsub] * B + (t % nsub) * TR; };
        auto issue = [&](int t, int buf) {
            const int c = chunk_row(t);
            const float* ks = reinterpret_cast<const float*>(K) + (zh * S + c) * D;
            const float* vs = reinterpret_cast<const float*>(V) + (zh * S + c) * D;
            for (int e = threadIdx.x; e < TR * D4; e += kThreads) {
                const int rr = e / D4, c4 = e % D4;
                cp_async16(Ks + (buf * TR + rr) * DP + 4 * c4, ks + (int64_t)rr * D + 4 * c4);
                cp_async16(Vs + (buf * TR + rr) * DP + 4 * c4, vs + (int64_t)rr * D + 4 * c4);
            }
            cp_async_commit();
        };
        if constexpr (ASYNC) {
            if (nch > 0) issue(0, 0);
        }
        {
            for (int t = 0; t < nch; ++t) {
                const int j = L.col_idx[q0 + t / nsub];
                const int c0 = chunk_row(t);  // first key row of the chunk
                const int buf = ASYNC ? (t & 1) : 0;
                const float* Kb = Ks + buf * TR * DP;
                const float* Vb = Vs + buf * TR * DP;
                __syncthreads();  // previous chunk fully consumed (and Qs written)
                if constexpr (ASYNC) {
                    if (t + 1 < nch) {
                        issue(t + 1, buf ^ 1);
                        cp_async_wait<1>();  // this chunk's copies have landed
                    } else {
                        cp_async_wait<0>();
                    }
                } else {
                    load_tile(Ks, K + (zh * S + c0) * D, 1.f);
                    load_tile(Vs, V + (zh * S + c0) * D, 1.f);
                }
                __syncthreads();
                // scores with paired FMAs (even and odd d in the two halves of a
                // float2, added at the end): half the FMA instructions
                float s[R][R];
                float2 s2[R][R];
#pragma unroll
                for (int u = 0; u < R; ++u)
#pragma unroll
                    for (int v = 0; v < R; ++v) s2[u][v] = make_float2(0.f, 0.f);
#pragma unroll 4
                for (int d4 = 0; d4 < D4; ++d4) {
                    float4 qa[R], kb[R];
#pragma unroll
                    for (int u = 0; u < R; ++u) qa[u] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * u) * DP + 4 * d4);
#pragma unroll
                    for (int v = 0; v < R; ++v) kb[v] = *reinterpret_cast<const float4*>(Kb + (tx + 16 * v) * DP + 4 * d4);
#pragma unroll
                    for (int u = 0; u < R; ++u)
#pragma unroll
                        for (int v = 0; v < R; ++v) {
                            s2[u][v] = __ffma2_rn(make_float2(qa[u].x, qa[u].y), make_float2(kb[v].x, kb[v].y), s2[u][v]);
                            s2[u][v] = __ffma2_rn(make_float2(qa[u].z, qa[u].w), make_float2(kb[v].z, kb[v].w), s2[u][v]);
                        }
                }
#pragma unroll
                for (int u = 0; u < R; ++u)
#pragma unroll
                    for (int v = 0; v < R; ++v) s[u][v] = s2[u][v].x + s2[u][v].y;
                // intra-block mask
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    const int r = r0 + ty + 16 * u;
#pragma unroll
                    for (int v = 0; v < R; ++v) {
                        const int c = c0 + tx + 16 * v;
                        bool keep = true;
                        if (kind == BSP_MASK_DIAG_CAUSAL) keep = (j != i) || (c <= r);
                        else if (kind == BSP_MASK_DENSE) keep = mask[(int64_t)r * S + c] != 0;
                        if (!keep) s[u][v] = -INFINITY;
                    }
                }
                // online softmax update per row (a row's 16 threads form a half-warp)
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    float cm = -INFINITY;
#pragma unroll
                    for (int v = 0; v < R; ++v) cm = fmaxf(cm, s[u][v]);
#pragma unroll
                    for (int o = 8; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
                    const float mn = fmaxf(m[u], cm);
                    float alpha = 1.f, rs = 0.f;
                    if (mn != -INFINITY) {
                        alpha = (m[u] == -INFINITY) ? 0.f : exp2f(m[u] - mn);
#pragma unroll
                        for (int v = 0; v < R; ++v) {
                            s[u][v] = exp2f(s[u][v] - mn);
                            rs += s[u][v];
                        }
                    } else {
#pragma unroll
                        for (int v = 0; v < R; ++v) s[u][v] = 0.f;
                    }
#pragma unroll
                    for (int o = 8; o; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
                    l[u] = l[u] * alpha + rs;
                    m[u] = mn;
#pragma unroll
                    for (int g = 0; g < NG; ++g)
#pragma unroll
                        for (int c = 0; c < 2; ++c) acc[u][g][c] = __fmul2_rn(acc[u][g][c], make_float2(alpha, alpha));
#pragma unroll
                    for (int v = 0; v < R; ++v) Ps[(ty + 16 * u) * PP + tx + 16 * v] = s[u][v];
                }
                __syncthreads();
#pragma unroll 2
                for (int cc4 = 0; cc4 < TR / 4; ++cc4) {
                    float4 pa[R];
#pragma unroll
                    for (int u = 0; u < R; ++u) pa[u] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * u) * PP + 4 * cc4);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        float4 vv[NG];
#pragma unroll
                        for (int g = 0; g < NG; ++g)
                            vv[g] = *reinterpret_cast<const float4*>(Vb + (4 * cc4 + k4) * DP + 64 * g + 4 * tx);
#pragma unroll
                        for (int u = 0; u < R; ++u) {
                            const float p = k4 == 0 ? pa[u].x : k4 == 1 ? pa[u].y : k4 == 2 ? pa[u].z : pa[u].w;
                            const float2 pp = make_float2(p, p);
#pragma unroll
                            for (int g = 0; g < NG; ++g) {
                                acc[u][g][0] = __ffma2_rn(pp, make_float2(vv[g].x, vv[g].y), acc[u][g][0]);
                                acc[u][g][1] = __ffma2_rn(pp, make_float2(vv[g].z, vv[g].w), acc[u][g][1]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const float inv = l[u] > 0.f ? 1.0f / l[u] : 0.f;
            const int64_t r = r0 + ty + 16 * u;
            if (lse && tx == 0) lse[zh * S + r] = l[u] > 0.f ? (m[u] + log2f(l[u])) * kLn2 : -INFINITY;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                T* dst = O + (zh * S + r) * D + 64 * g + 4 * tx;
                dst[0] = from_f32<T>(acc[u][g][0].x * inv);
                dst[1] = from_f32<T>(acc[u][g][0].y * inv);
                dst[2] = from_f32<T>(acc[u][g][1].x * inv);
                dst[3] = from_f32<T>(acc[u][g][1].y * inv);
            }
        }
        __syncthreads();  // Qs reused by the next work item
    }
}

template <typename T, int D>
int attn_v4(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, float scale,
            int kind, const uint8_t* mask, cudaStream_t s) {
    const int64_t total = (int64_t)L->H * L->nb * Z * (L->B / 64);
    if (total == 0) return BSP_OK;
    constexpr int nbuf = std::is_same<T, float>::value ? 2 : 1;  // K / V buffers (see the kernel)
    const size_t smem = sizeof(float) * ((size_t)(1 + 2 * nbuf) * 64 * (D + 4) + (size_t)64 * (64 + 4));
    auto kern = attention_simt_v4_kernel<T, D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    kern<<<grid_for(total), kThreads, smem, s>>>(L->view, (const T*)Q, (const T*)K, (const T*)V, (T*)O, lse, Z,
                                                  scale * kLog2e, kind, mask);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T, int TR>
int attn_tr(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z,
            int D, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    const int64_t total = (int64_t)L->H * L->nb * Z * (L->B / TR);
    if (total == 0) return BSP_OK;
    const size_t smem = sizeof(float) * ((size_t)3 * TR * (D + 1) + (size_t)TR * (TR + 1));
    auto kern = attention_simt_kernel<T, TR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    kern<<<grid_for(total), kThreads, smem, s>>>(L->view, (const T*)Q, (const T*)K, (const T*)V,
                                                  (T*)O, lse, Z, D, scale * kLog2e, kind, mask);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int attn_t(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, int D,
           float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if (L->B >= 64 && D == 64) return attn_v4<T, 64>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
    if (L->B >= 64 && D == 128) return attn_v4<T, 128>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
    switch (L->B) {
        case 16: return attn_tr<T, 16>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        case 32: return attn_tr<T, 32>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        default: return attn_tr<T, 64>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
    }
}

}  // namespace

#define BSP_DISPATCH(fn, ...)                                                  \
    switch (dtype) {                                                           \
        case BSP_F32: return fn<float>(__VA_ARGS__);                           \
        case BSP_BF16: return fn<__nv_bfloat16>(__VA_ARGS__);                  \
        case BSP_F16: return fn<__half>(__VA_ARGS__);                          \
        default: return BSP_ERR_INVALID_ARG;                                   \
    }

int launch_sdd_simt(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                    int K, int ta, int tb, cudaStream_t s) {
    BSP_DISPATCH(sdd_t, L, A, B, C, Z, K, ta, tb, s)
}
int launch_dsd_simt(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                    int N, int ta, int tb, cudaStream_t s) {
    BSP_DISPATCH(dsd_t, L, A, B, C, Z, N, ta, tb, s)
}
int launch_dds_simt(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                    int M, int ta, int tb, cudaStream_t s) {
    BSP_DISPATCH(dds_t, L, A, B, C, Z, M, ta, tb, s)
}
int launch_attention_simt(const bsp_layout_s* L, int dtype, const void* Q, const void* K,
                          const void* V, void* O, float* lse, int Z, int D, float scale, int kind,
                          const uint8_t* mask, cudaStream_t s) {
    BSP_DISPATCH(attn_t, L, Q, K, V, O, lse, Z, D, scale, kind, mask, s)
}

}  // namespace bsp
