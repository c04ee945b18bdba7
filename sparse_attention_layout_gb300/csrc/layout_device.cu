// Layout compiler on the device: the tables of layout.cpp built by kernels
// from a layout that already lives in device memory (a layout that changes
// every step never has to visit the host).  Same definitions as the host
// compiler: blocks numbered by rank in row-major (h, i, j) order (the SDD
// output order of "question on blocksparse", openai/triton issue 117), CSR and
// CSC tables, row tiles of G = 128/B block-rows cut into steps of G slots,
// line groups in both orientations, softmax chunk items, and longest-first
// orders (stable, ties by key).  Every table equals the host compiler's.
//
// Phases: (1) per-row / per-column / per-group sizes and a validity flag,
// prefix sums by one-CTA scans; (2) one small read-back of the totals (the
// table sizes), then one allocation; (3) fill kernels; (4) stable counting
// sorts, one warp per order, ranks among equal weights from __match_any_sync.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>

#include "bsp_internal.h"

namespace bsp {
namespace {

struct Totals {
    int err;                // some layout value is not 0 or 1
    int nnz, n_steps, slots[2], items[2];
    int sm_max_bytes[2];
    int sm_unfit[2];        // some single row exceeds the chunk budget
    int max_tile_steps;
    int max_row_nnz, max_col_nnz;  // the softmax sizes its shared column-index array by the first
};

constexpr int kScanThreads = 1024;

// exclusive prefix sum of in[0..n) into out[0..n), the total into *total
__global__ void __launch_bounds__(kScanThreads) k_scan(const int* __restrict__ in, int* __restrict__ out, int n,
                                                       int* total) {
    __shared__ int part[kScanThreads];
    const int t = threadIdx.x;
    const int per = (n + kScanThreads - 1) / kScanThreads;
    const int lo = min(n, t * per), hi = min(n, lo + per);
    int s = 0;
    for (int e = lo; e < hi; ++e) s += in[e];
    part[t] = s;
    __syncthreads();
    for (int d = 1; d < kScanThreads; d <<= 1) {  // inclusive Hillis-Steele scan of the partial sums
        const int v = t >= d ? part[t - d] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int run = part[t] - s;  // exclusive start of this thread's chunk
    for (int e = lo; e < hi; ++e) {
        const int v = in[e];
        out[e] = run;
        run += v;
    }
    if (t == kScanThreads - 1) *total = part[t];
}

// per block-row: block count, validity
__global__ void k_rows(const uint8_t* __restrict__ lay, int rows, int nb, int* row_len, Totals* tot) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const uint8_t* p = lay + (int64_t)r * nb;
    int c = 0, bad = 0;
    for (int j = 0; j < nb; ++j) {
        const uint8_t v = p[j];
        bad |= v > 1;
        c += v != 0;
    }
    if (bad) atomicOr(&tot->err, 1);
    row_len[r] = c;
    atomicMax(&tot->max_row_nnz, c);
}

// per block-row: softmax chunk counts (both element sizes), once the longest
// row, which sets the chunk budget, is known
__global__ void k_row_items(int rows, int B, const int* row_len, int* items0, int* items1, Totals* tot) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const int c = row_len[r];
    for (int e = 0; e < 2; ++e) {
        const int64_t per_row = (int64_t)c * B * (e ? 4 : 2);
        const int64_t budget = softmax_chunk_budget((int64_t)tot->max_row_nnz * B * (e ? 4 : 2));
        int items = 0;
        if (per_row > 0) {
            int R = B;
            while (R > 1 && R * per_row > budget) R >>= 1;
            if (R * per_row > budget) atomicOr(&tot->sm_unfit[e], 1);
            atomicMax(&tot->sm_max_bytes[e], (int)(R * per_row < INT32_MAX ? R * per_row : INT32_MAX));
            items = B / R;
        }
        (e ? items1 : items0)[r] = items;
    }
}

// per block-column: block count
__global__ void k_cols(const uint8_t* __restrict__ lay, int H, int nb, int* col_len, Totals* tot) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= H * nb) return;
    const int h = c / nb, j = c % nb;
    int n = 0;
    for (int i = 0; i < nb; ++i) n += lay[((int64_t)h * nb + i) * nb + j] != 0;
    col_len[c] = n;
    atomicMax(&tot->max_col_nnz, n);
}

__device__ __forceinline__ bool present(const uint8_t* lay, int nb, int h, int i, int j) {
    return lay[((int64_t)h * nb + i) * nb + j] != 0;
}

// block-wide exclusive scan of one flag per thread; returns the exclusive rank,
// *count receives the total (blockDim.x a multiple of 32, at most 1024)
__device__ int block_rank(int flag, int* warp_sums, int* count) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_sums[wid] = __popc(bal);
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int w = 0; w < nw; ++w) {
            const int v = warp_sums[w];
            warp_sums[w] = s;
            s += v;
        }
        *count = s;
    }
    __syncthreads();
    const int r = warp_sums[wid] + in_warp;
    __syncthreads();
    return r;
}

// union size of each group (o = 0: G block-rows, o = 1: G block-columns)
__global__ void k_group_sizes(const uint8_t* __restrict__ lay, int H, int nb, int G, int ngroups, int* steps,
                              int* size0, int* size1, Totals* tot) {
    __shared__ int ws[32], cnt;
    const int o = blockIdx.y, t = blockIdx.x;
    const int h = t / ngroups, g = t % ngroups;
    int total = 0;
    for (int u0 = 0; u0 < nb; u0 += blockDim.x) {
        const int u = u0 + threadIdx.x;
        int f = 0;
        if (u < nb)
            for (int a = 0; a < G && g * G + a < nb; ++a)
                f |= o ? present(lay, nb, h, u, g * G + a) : present(lay, nb, h, g * G + a, u);
        block_rank(f, ws, &cnt);
        total += cnt;
    }
    if (threadIdx.x == 0) {
        if (o == 0) {
            size0[t] = total;
            steps[t] = (total + G - 1) / G;
            atomicMax(&tot->max_tile_steps, (total + G - 1) / G);
        } else {
            size1[t] = total;
        }
    }
}

struct Tables {
    int32_t *row_ptr, *col_idx, *blk_id, *col_ptr, *row_idx, *blk_id_csc, *blk_key, *row_order, *col_order;
    int32_t *tile_step_ptr, *tile_order, *tile_run, *step_col, *step_blk, *sm_items[2];
    int32_t *gl_ptr[2], *gl_order[2], *gl_idx[2], *gl_blk[2];
};

// CSR, block ids, row keys and the dense id map
__global__ void k_fill_rows(const uint8_t* __restrict__ lay, int H, int nb, const int* row_start, Tables T,
                            int32_t* ids) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= H * nb) return;
    const int h = r / nb, i = r % nb;
    int p = row_start[r];
    T.row_ptr[h * (nb + 1) + i] = p;
    for (int j = 0; j < nb; ++j) {
        if (present(lay, nb, h, i, j)) {
            T.col_idx[p] = j;
            T.blk_id[p] = p;
            T.blk_key[p] = r;
            ids[(int64_t)r * nb + j] = p++;
        } else {
            ids[(int64_t)r * nb + j] = -1;
        }
    }
    if (i == nb - 1) T.row_ptr[h * (nb + 1) + nb] = p;
}

__global__ void k_fill_cols(int H, int nb, const int* col_start, const int32_t* __restrict__ ids, Tables T) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= H * nb) return;
    const int h = c / nb, j = c % nb;
    int q = col_start[c];
    T.col_ptr[h * (nb + 1) + j] = q;
    for (int i = 0; i < nb; ++i) {
        const int id = ids[((int64_t)h * nb + i) * nb + j];
        if (id >= 0) {
            T.row_idx[q] = i;
            T.blk_id_csc[q++] = id;
        }
    }
    if (j == nb - 1) T.col_ptr[h * (nb + 1) + nb] = q;
}

// tile lists (o = 0 only) and line-group lists, one CTA per (group, orientation)
__global__ void k_fill_groups(const int32_t* __restrict__ ids, int H, int nb, int G, int ngroups,
                              const int* tile_start, const int* gl_start0, const int* gl_start1, Tables T) {
    __shared__ int ws[32], cnt;
    const int o = blockIdx.y, t = blockIdx.x;
    const int h = t / ngroups, g = t % ngroups;
    const int base = o ? gl_start1[t] : gl_start0[t];
    int k0 = 0;
    for (int u0 = 0; u0 < nb; u0 += blockDim.x) {
        const int u = u0 + threadIdx.x;
        int blk[8];  // G <= 8
        int f = 0;
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            blk[a] = -1;
            if (a < G && u < nb && g * G + a < nb)
                blk[a] = o ? ids[((int64_t)h * nb + u) * nb + g * G + a] : ids[((int64_t)h * nb + g * G + a) * nb + u];
            f |= blk[a] >= 0;
        }
        const int k = k0 + block_rank(f, ws, &cnt);
        if (f) {
            T.gl_idx[o][base + k] = u;
            for (int a = 0; a < G; ++a) T.gl_blk[o][(int64_t)(base + k) * G + a] = blk[a];
            if (o == 0) {
                const int s = tile_start[t] + k / G, b = k % G;
                T.step_col[(int64_t)s * G + b] = u;
                for (int a = 0; a < G; ++a) T.step_blk[((int64_t)s * G + a) * G + b] = blk[a];
            }
        }
        k0 += cnt;
    }
    if (o == 0) {  // padding slots of the last step
        const int steps = (k0 + G - 1) / G;
        for (int k = k0 + threadIdx.x; k < steps * G; k += blockDim.x) {
            const int s = tile_start[t] + k / G, b = k % G;
            T.step_col[(int64_t)s * G + b] = -1;
            for (int a = 0; a < G; ++a) T.step_blk[((int64_t)s * G + a) * G + b] = -1;
        }
    }
}

__global__ void k_fill_items(int rows, int B, int max_row_nnz, const int* row_len, const int* row_start,
                             const int* item_start0, const int* item_start1, Tables T) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows || row_len[r] == 0) return;
    for (int e = 0; e < 2; ++e) {
        const int64_t per_row = (int64_t)row_len[r] * B * (e ? 4 : 2);
        const int64_t budget = softmax_chunk_budget((int64_t)max_row_nnz * B * (e ? 4 : 2));
        int R = B;
        while (R > 1 && R * per_row > budget) R >>= 1;
        int32_t* it = T.sm_items[e] + 4 * (int64_t)(e ? item_start1[r] : item_start0[r]);
        for (int r0 = 0; r0 < B; r0 += R, it += 4) {
            it[0] = r;
            it[1] = row_start[r];
            it[2] = row_len[r];
            it[3] = r0 | (R << 16);
        }
    }
}

// Stable order of 0..n-1 by descending weight (ties by index), weights in
// [0, wmax]: counting sort by one warp; the rank among equal weights inside a
// batch of 32 comes from __match_any_sync.  One CTA (32 threads) per list.
struct OrderJob {
    const int* w;
    int32_t* out;
    int n;
};
// tile_run[r] = (tile, first step, step count, 0) of the r-th tile of tile_order
__global__ void k_tile_run(Tables T, int ntiles) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= ntiles) return;
    const int t = T.tile_order[r];
    const int s0 = T.tile_step_ptr[t];
    reinterpret_cast<int4*>(T.tile_run)[r] = make_int4(t, s0, T.tile_step_ptr[t + 1] - s0, 0);
}

__global__ void k_orders(const OrderJob* jobs, int wmax) {
    extern __shared__ int sh[];
    int* start = sh;              // [wmax + 1]
    int* used = sh + wmax + 1;    // [wmax + 1]
    const OrderJob J = jobs[blockIdx.x];
    const int lane = threadIdx.x;
    for (int v = lane; v <= wmax; v += 32) used[v] = 0;
    __syncwarp();
    for (int e = lane; e < J.n; e += 32) atomicAdd(&used[J.w[e]], 1);
    __syncwarp();
    if (lane == 0) {  // bucket starts, largest weight first
        int s = 0;
        for (int v = wmax; v >= 0; --v) {
            start[v] = s;
            s += used[v];
            used[v] = 0;
        }
    }
    __syncwarp();
    for (int b0 = 0; b0 < J.n; b0 += 32) {
        const int e = b0 + lane;
        const unsigned act = __ballot_sync(0xffffffffu, e < J.n);
        if (e < J.n) {
            const int w = J.w[e];
            const unsigned peers = __match_any_sync(act, w);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            J.out[start[w] + used[w] + rank] = e;
            __syncwarp(act);
            if (rank == 0) used[w] += __popc(peers);
        }
        __syncwarp();
    }
}

// [H][nb][nb] 0/1 layout of per-head affine records (8 ints per head: band
// on, beta, kappa; column on, beta, sigma, kappa, causal)
__global__ void k_expand_affine(const int32_t* __restrict__ rec, int H, int nb, uint8_t* __restrict__ out) {
    const int64_t total = (int64_t)H * nb * nb;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(e % nb);
        const int64_t hi = e / nb;
        const int i = (int)(hi % nb), h = (int)(hi / nb);
        const int32_t* r = rec + (size_t)h * kGeoRec;
        bool v = r[0] && j - i >= r[1] && j - i < r[1] + r[2];
        if (r[3] && !v && j >= r[4] && (!r[7] || j <= i)) {
            const int d = j - r[4];
            v = d % r[5] == 0 && d / r[5] < r[6];
        }
        out[e] = v ? 1 : 0;
    }
}

template <typename T>
size_t padded(size_t n) {
    return ((n * sizeof(T) + 255) / 256) * 256;
}

bool valid_block(int B) { return B == 16 || B == 32 || B == 64 || B == 128; }

}  // namespace
}  // namespace bsp

extern "C" int bsp_layout_compile_device(const uint8_t* layout, int H, int nb, int block, void* stream,
                                         bsp_layout_t* out) {
    using namespace bsp;
    if (!out) return BSP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!layout || H < 1 || nb < 1 || !valid_block(block)) return BSP_ERR_INVALID_ARG;
    // counting sorts keep a weight histogram of nb + 1 entries in shared memory
    if (nb > 4096 || (int64_t)nb * block > (1 << 24) || (int64_t)H * nb * nb > ((int64_t)1 << 30))
        return BSP_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    const int G = 128 / block, ngroups = (nb + G - 1) / G, ntiles = H * ngroups, rows = H * nb;

    // scratch: sizes, starts, the dense id map, totals
    enum { ROW_LEN, COL_LEN, ROW_START, COL_START, ITEMS0, ITEMS1, ITEM_START0, ITEM_START1, NPER_ROW };
    enum { STEPS, SIZE0, SIZE1, TILE_START, GL_START0, GL_START1, NPER_TILE };
    const size_t scratch_bytes = padded<int>((size_t)NPER_ROW * rows) + padded<int>((size_t)NPER_TILE * ntiles) +
                                 padded<int32_t>((size_t)rows * nb) + padded<Totals>(1) + padded<OrderJob>(5);
    char* scratch = nullptr;
    if (cudaMalloc((void**)&scratch, scratch_bytes) != cudaSuccess) {
        cudaGetLastError();
        return BSP_ERR_OOM;
    }
    int* pr = (int*)scratch;
    int* pt = (int*)(scratch + padded<int>((size_t)NPER_ROW * rows));
    int32_t* ids = (int32_t*)((char*)pt + padded<int>((size_t)NPER_TILE * ntiles));
    Totals* dtot = (Totals*)((char*)ids + padded<int32_t>((size_t)rows * nb));
    OrderJob* djobs = (OrderJob*)((char*)dtot + padded<Totals>(1));
    auto R = [&](int k) { return pr + (size_t)k * rows; };
    auto Tt = [&](int k) { return pt + (size_t)k * ntiles; };

    bsp_layout_s* L = new (std::nothrow) bsp_layout_s();
    if (!L) {
        cudaFree(scratch);
        return BSP_ERR_OOM;
    }
    auto fail = [&](int rc) {
        cudaGetLastError();
        cudaStreamSynchronize(s);
        cudaFree(scratch);
        if (L->dmem) cudaFree(L->dmem);
        delete L;
        return rc;
    };
    L->H = H;
    L->nb = nb;
    L->B = block;
    L->S = nb * block;
    L->G = G;
    L->ngroups = ngroups;
    L->n_tiles = ntiles;
    L->host_tables = false;
    if (cudaGetDevice(&L->device) != cudaSuccess) return fail(BSP_ERR_CUDA);

    // (1) sizes and starts
    const int tb = 256;
    bool ok = cudaMemsetAsync(dtot, 0, sizeof(Totals), s) == cudaSuccess;
    k_rows<<<(rows + tb - 1) / tb, tb, 0, s>>>(layout, rows, nb, R(ROW_LEN), dtot);
    k_row_items<<<(rows + tb - 1) / tb, tb, 0, s>>>(rows, block, R(ROW_LEN), R(ITEMS0), R(ITEMS1), dtot);
    k_cols<<<(rows + tb - 1) / tb, tb, 0, s>>>(layout, H, nb, R(COL_LEN), dtot);
    k_group_sizes<<<dim3(ntiles, 2), tb, 0, s>>>(layout, H, nb, G, ngroups, Tt(STEPS), Tt(SIZE0), Tt(SIZE1), dtot);
    k_scan<<<1, kScanThreads, 0, s>>>(R(ROW_LEN), R(ROW_START), rows, &dtot->nnz);
    k_scan<<<1, kScanThreads, 0, s>>>(R(COL_LEN), R(COL_START), rows, &dtot->nnz);  // same total
    k_scan<<<1, kScanThreads, 0, s>>>(R(ITEMS0), R(ITEM_START0), rows, &dtot->items[0]);
    k_scan<<<1, kScanThreads, 0, s>>>(R(ITEMS1), R(ITEM_START1), rows, &dtot->items[1]);
    k_scan<<<1, kScanThreads, 0, s>>>(Tt(STEPS), Tt(TILE_START), ntiles, &dtot->n_steps);
    k_scan<<<1, kScanThreads, 0, s>>>(Tt(SIZE0), Tt(GL_START0), ntiles, &dtot->slots[0]);
    k_scan<<<1, kScanThreads, 0, s>>>(Tt(SIZE1), Tt(GL_START1), ntiles, &dtot->slots[1]);
    // (2) the table sizes
    Totals tot;
    ok = ok && cudaGetLastError() == cudaSuccess &&
         cudaMemcpyAsync(&tot, dtot, sizeof(Totals), cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaStreamSynchronize(s) == cudaSuccess;
    if (!ok) return fail(BSP_ERR_CUDA);
    if (tot.err) return fail(BSP_ERR_INVALID_ARG);
    L->nnz = tot.nnz;
    L->n_steps = tot.n_steps;
    L->max_tile_steps = tot.max_tile_steps;
    L->max_row_nnz = tot.max_row_nnz;
    L->max_col_nnz = tot.max_col_nnz;
    for (int e = 0; e < 2; ++e) {
        L->gl_slots[e] = tot.slots[e];
        L->sm_n_items_dev[e] = tot.items[e];
        L->sm_max_bytes[e] = tot.sm_max_bytes[e];
        L->sm_fits[e] = !tot.sm_unfit[e];
    }
    const size_t nnz = (size_t)tot.nnz, nst = (size_t)tot.n_steps;
    const size_t sizes[] = {(size_t)H * (nb + 1), nnz, nnz, (size_t)H * (nb + 1), nnz, nnz, nnz, (size_t)rows,
                            (size_t)rows, (size_t)ntiles + 1, (size_t)ntiles, 4 * (size_t)ntiles, nst * G,
                            nst * G * G,
                            4 * (size_t)tot.items[0], 4 * (size_t)tot.items[1],
                            (size_t)ntiles + 1, (size_t)ntiles, (size_t)tot.slots[0], (size_t)tot.slots[0] * G,
                            (size_t)ntiles + 1, (size_t)ntiles, (size_t)tot.slots[1], (size_t)tot.slots[1] * G};
    LayoutView& V = L->view;
    const int32_t** dst[] = {&V.row_ptr, &V.col_idx, &V.blk_id, &V.col_ptr, &V.row_idx, &V.blk_id_csc, &V.blk_key,
                             &V.row_order, &V.col_order, &V.tile_step_ptr, &V.tile_order, &V.tile_run,
                             &V.step_col, &V.step_blk, &V.sm_items[0], &V.sm_items[1], &V.gl_ptr[0], &V.gl_order[0],
                             &V.gl_idx[0], &V.gl_blk[0], &V.gl_ptr[1], &V.gl_order[1], &V.gl_idx[1],
                             &V.gl_blk[1]};
    constexpr int nparts = sizeof(sizes) / sizeof(sizes[0]);
    size_t total = padded<int>(4);
    for (int k = 0; k < nparts; ++k) total += padded<int32_t>(sizes[k] + 1);
    char* base = nullptr;
    if (cudaMalloc((void**)&base, total) != cudaSuccess) return fail(BSP_ERR_OOM);
    L->dmem = base;
    V.status = (int*)base;
    V.wait_ns = kDefaultWaitNs;
    V.inject = 0;
    size_t off = padded<int>(4);
    for (int k = 0; k < nparts; ++k) {
        *dst[k] = (const int32_t*)(base + off);
        off += padded<int32_t>(sizes[k] + 1);
    }
    Tables T;
    int32_t** tptr[] = {&T.row_ptr, &T.col_idx, &T.blk_id, &T.col_ptr, &T.row_idx, &T.blk_id_csc, &T.blk_key,
                        &T.row_order, &T.col_order, &T.tile_step_ptr, &T.tile_order, &T.tile_run, &T.step_col,
                        &T.step_blk,
                        &T.sm_items[0], &T.sm_items[1], &T.gl_ptr[0], &T.gl_order[0], &T.gl_idx[0], &T.gl_blk[0],
                        &T.gl_ptr[1], &T.gl_order[1], &T.gl_idx[1], &T.gl_blk[1]};
    for (int k = 0; k < nparts; ++k) *tptr[k] = const_cast<int32_t*>(*dst[k]);

    // (3) fill: starts of the tile / group lists are their scans, plus the end entries
    ok = cudaMemsetAsync(base, 0, padded<int>(4), s) == cudaSuccess &&
         cudaMemcpyAsync(T.tile_step_ptr, Tt(TILE_START), ntiles * sizeof(int), cudaMemcpyDeviceToDevice, s) ==
             cudaSuccess &&
         cudaMemcpyAsync(T.tile_step_ptr + ntiles, &dtot->n_steps, sizeof(int), cudaMemcpyDeviceToDevice, s) ==
             cudaSuccess &&
         cudaMemcpyAsync(T.gl_ptr[0], Tt(GL_START0), ntiles * sizeof(int), cudaMemcpyDeviceToDevice, s) ==
             cudaSuccess &&
         cudaMemcpyAsync(T.gl_ptr[0] + ntiles, &dtot->slots[0], sizeof(int), cudaMemcpyDeviceToDevice, s) ==
             cudaSuccess &&
         cudaMemcpyAsync(T.gl_ptr[1], Tt(GL_START1), ntiles * sizeof(int), cudaMemcpyDeviceToDevice, s) ==
             cudaSuccess &&
         cudaMemcpyAsync(T.gl_ptr[1] + ntiles, &dtot->slots[1], sizeof(int), cudaMemcpyDeviceToDevice, s) ==
             cudaSuccess;
    k_fill_rows<<<(rows + tb - 1) / tb, tb, 0, s>>>(layout, H, nb, R(ROW_START), T, ids);
    k_fill_cols<<<(rows + tb - 1) / tb, tb, 0, s>>>(H, nb, R(COL_START), ids, T);
    k_fill_groups<<<dim3(ntiles, 2), tb, 0, s>>>(ids, H, nb, G, ngroups, Tt(TILE_START), Tt(GL_START0),
                                                 Tt(GL_START1), T);
    k_fill_items<<<(rows + tb - 1) / tb, tb, 0, s>>>(rows, block, tot.max_row_nnz, R(ROW_LEN), R(ROW_START),
                                                     R(ITEM_START0), R(ITEM_START1), T);
    // (4) longest-first orders
    const OrderJob jobs[5] = {{R(ROW_LEN), T.row_order, rows}, {R(COL_LEN), T.col_order, rows},
                              {Tt(STEPS), T.tile_order, ntiles}, {Tt(SIZE0), T.gl_order[0], ntiles},
                              {Tt(SIZE1), T.gl_order[1], ntiles}};
    ok = ok && cudaMemcpyAsync(djobs, jobs, sizeof(jobs), cudaMemcpyHostToDevice, s) == cudaSuccess;
    k_orders<<<5, 32, 2 * (nb + 1) * sizeof(int), s>>>(djobs, nb);
    if (ntiles > 0) k_tile_run<<<(ntiles + tb - 1) / tb, tb, 0, s>>>(T, ntiles);
    ok = ok && cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess;
    if (!ok) return fail(BSP_ERR_CUDA);
    cudaFree(scratch);
    V.H = H;
    V.nb = nb;
    V.B = block;
    V.S = L->S;
    V.G = G;
    V.ngroups = ngroups;
    V.n_tiles = ntiles;
    V.nnz = L->nnz;
    for (int e = 0; e < 2; ++e) {
        V.sm_n_items[e] = tot.items[e];
        V.sm_max_bytes[e] = tot.sm_max_bytes[e];
        V.sm_fits[e] = tot.sm_unfit[e] ? 0 : 1;
    }
    L->on_device = true;
    *out = L;
    return BSP_OK;
}

extern "C" int bsp_layout_compile_affine(const int32_t* n_terms, const bsp_affine_term_t* terms, int H, int nb,
                                         int block, void* stream, bsp_layout_t* out) {
    using namespace bsp;
    if (!out) return BSP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!n_terms || !terms || H < 1 || nb < 1 || !valid_block(block)) return BSP_ERR_INVALID_ARG;
    if (nb > 4096 || (int64_t)nb * block > (1 << 24) || (int64_t)H * nb * nb > ((int64_t)1 << 30))
        return BSP_ERR_UNSUPPORTED;
    // the description, checked and turned into the kernels' records
    bsp_layout_s desc;
    desc.H = H;
    desc.nb = nb;
    desc.geo_n.assign(n_terms, n_terms + H);
    desc.geo_terms.assign((size_t)H * BSP_MAX_AFFINE_TERMS, bsp_affine_term_t{0, 0, 0, 0, 0});
    for (int h = 0; h < H; ++h) {
        const int rc = affine_validate(nb, n_terms[h], terms + (size_t)h * BSP_MAX_AFFINE_TERMS);
        if (rc != BSP_OK) return rc;
        std::copy_n(terms + (size_t)h * BSP_MAX_AFFINE_TERMS, n_terms[h],
                    &desc.geo_terms[(size_t)h * BSP_MAX_AFFINE_TERMS]);
    }
    affine_records(&desc);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t rec_bytes = desc.geo_rec.size() * sizeof(int32_t);
    int32_t* rec = nullptr;
    uint8_t* lay = nullptr;
    if (cudaMalloc((void**)&rec, rec_bytes) != cudaSuccess) {
        cudaGetLastError();
        return BSP_ERR_OOM;
    }
    if (cudaMalloc((void**)&lay, (size_t)H * nb * nb) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(rec);
        return BSP_ERR_OOM;
    }
    int rc = BSP_OK;
    if (cudaMemcpyAsync(rec, desc.geo_rec.data(), rec_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) rc = BSP_ERR_CUDA;
    if (rc == BSP_OK) {
        const int64_t blocks = std::min<int64_t>(((int64_t)H * nb * nb + 255) / 256, (int64_t)sm_count() * 8);
        k_expand_affine<<<(unsigned)blocks, 256, 0, s>>>(rec, H, nb, lay);
        if (cudaGetLastError() != cudaSuccess) rc = BSP_ERR_CUDA;
    }
    // compiles the expanded layout and synchronises the stream, after which
    // the layout buffer is no longer read
    if (rc == BSP_OK) rc = bsp_layout_compile_device(lay, H, nb, block, stream, out);
    if (rc != BSP_OK) cudaStreamSynchronize(s);
    cudaFree(lay);
    if (rc != BSP_OK) {
        cudaGetLastError();
        cudaFree(rec);
        return rc;
    }
    bsp_layout_s* L = *out;
    L->geo_n = std::move(desc.geo_n);
    L->geo_terms = std::move(desc.geo_terms);
    L->geo_rec = std::move(desc.geo_rec);
    L->geo_dmem = rec;
    L->view.geo = rec;
    return BSP_OK;
}
