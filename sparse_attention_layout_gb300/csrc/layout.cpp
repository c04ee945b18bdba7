// Layout compiler: validates a 0/1 block layout and builds the lookup tables
// and work lists the kernels read.
//
// The layout is the tensor of 0s and 1s of "question on blocksparse"
// (openai/triton issue 117, answer on how a block is defined): one entry per
// non-overlapping square block of 16, 32, 64 or 128 elements.  Blocks are
// numbered by their rank in row-major (h, i, j) order, the order in which the
// block-sparse SDD output stores them.
#include <algorithm>
#include <cstring>
#include <new>
#include <numeric>

#include "bsp_internal.h"

namespace {

bool valid_block(int B) { return B == 16 || B == 32 || B == 64 || B == 128; }

// Stable order of keys 0..n-1 by descending weight (longest-processing-time
// first), ties by key.
std::vector<int32_t> order_by_weight_desc(const std::vector<int32_t>& weight) {
    std::vector<int32_t> ord(weight.size());
    std::iota(ord.begin(), ord.end(), 0);
    std::stable_sort(ord.begin(), ord.end(),
                     [&](int32_t a, int32_t b) { return weight[a] > weight[b]; });
    return ord;
}

int build_tables(bsp_layout_s* L, const uint8_t* lay) {
    const int H = L->H, nb = L->nb;
    const int64_t cells = (int64_t)H * nb * nb;
    std::vector<int64_t> ids(cells, -1);
    int64_t next = 0;
    for (int64_t e = 0; e < cells; ++e) {
        if (lay[e] > 1) return BSP_ERR_INVALID_ARG;
        if (lay[e]) ids[e] = next++;
    }
    if (next > INT32_MAX / 2) return BSP_ERR_UNSUPPORTED;
    L->nnz = next;
    const int nnz = (int)next;
    auto id_at = [&](int h, int i, int j) { return ids[((int64_t)h * nb + i) * nb + j]; };

    // CSR (row) tables
    L->row_ptr.assign((size_t)H * (nb + 1), 0);
    L->col_idx.resize(nnz);
    L->blk_id.resize(nnz);
    L->blk_key.resize(nnz);
    std::vector<int32_t> row_len((size_t)H * nb, 0), col_len((size_t)H * nb, 0);
    int32_t p = 0;
    for (int h = 0; h < H; ++h) {
        for (int i = 0; i < nb; ++i) {
            L->row_ptr[(size_t)h * (nb + 1) + i] = p;
            for (int j = 0; j < nb; ++j) {
                int64_t id = id_at(h, i, j);
                if (id < 0) continue;
                L->col_idx[p] = j;
                L->blk_id[p] = (int32_t)id;
                L->blk_key[id] = h * nb + i;
                ++p;
            }
            row_len[(size_t)h * nb + i] = p - L->row_ptr[(size_t)h * (nb + 1) + i];
        }
        L->row_ptr[(size_t)h * (nb + 1) + nb] = p;
    }
    // CSC (column) tables
    L->col_ptr.assign((size_t)H * (nb + 1), 0);
    L->row_idx.resize(nnz);
    L->blk_id_csc.resize(nnz);
    int32_t q = 0;
    for (int h = 0; h < H; ++h) {
        for (int j = 0; j < nb; ++j) {
            L->col_ptr[(size_t)h * (nb + 1) + j] = q;
            for (int i = 0; i < nb; ++i) {
                int64_t id = id_at(h, i, j);
                if (id < 0) continue;
                L->row_idx[q] = i;
                L->blk_id_csc[q] = (int32_t)id;
                ++q;
            }
            col_len[(size_t)h * nb + j] = q - L->col_ptr[(size_t)h * (nb + 1) + j];
        }
        L->col_ptr[(size_t)h * (nb + 1) + nb] = q;
    }
    L->row_order = order_by_weight_desc(row_len);
    L->col_order = order_by_weight_desc(col_len);
    L->max_row_nnz = row_len.empty() ? 0 : *std::max_element(row_len.begin(), row_len.end());
    L->max_col_nnz = col_len.empty() ? 0 : *std::max_element(col_len.begin(), col_len.end());

    // Row tiles for the tensor-core kernels: G = 128/B consecutive block-rows
    // of one head form a 128-row tile.  Its block-columns are the union of the
    // rows' columns, cut into steps of G slots (128 key rows per step).
    const int G = 128 / L->B;
    L->G = G;
    L->ngroups = (nb + G - 1) / G;
    L->n_tiles = H * L->ngroups;
    L->tile_step_ptr.assign((size_t)L->n_tiles + 1, 0);
    L->step_col.clear();
    L->step_blk.clear();
    std::vector<int32_t> tile_steps((size_t)L->n_tiles, 0);
    std::vector<uint8_t> in_union((size_t)nb);
    int64_t steps = 0;
    for (int h = 0; h < H; ++h) {
        for (int g = 0; g < L->ngroups; ++g) {
            const int t = h * L->ngroups + g;
            std::fill(in_union.begin(), in_union.end(), 0);
            for (int a = 0; a < G; ++a) {
                const int i = g * G + a;
                if (i >= nb) break;
                for (int pp = L->row_ptr[(size_t)h * (nb + 1) + i];
                     pp < L->row_ptr[(size_t)h * (nb + 1) + i + 1]; ++pp)
                    in_union[L->col_idx[pp]] = 1;
            }
            std::vector<int32_t> cols;
            for (int j = 0; j < nb; ++j)
                if (in_union[j]) cols.push_back(j);
            const int ns = (int)((cols.size() + G - 1) / G);
            L->tile_step_ptr[t] = (int32_t)steps;
            tile_steps[t] = ns;
            for (int s = 0; s < ns; ++s) {
                for (int b = 0; b < G; ++b) {
                    const size_t k = (size_t)s * G + b;
                    L->step_col.push_back(k < cols.size() ? cols[k] : -1);
                }
                for (int a = 0; a < G; ++a) {
                    const int i = g * G + a;
                    for (int b = 0; b < G; ++b) {
                        const size_t k = (size_t)s * G + b;
                        int32_t id = -1;
                        if (i < nb && k < cols.size()) id = (int32_t)id_at(h, i, cols[k]);
                        L->step_blk.push_back(id);
                    }
                }
            }
            steps += ns;
        }
    }
    L->tile_step_ptr[L->n_tiles] = (int32_t)steps;
    L->n_steps = steps;
    L->tile_order = order_by_weight_desc(tile_steps);
    L->tile_run.resize((size_t)4 * L->n_tiles);
    for (int r = 0; r < L->n_tiles; ++r) {
        const int t = L->tile_order[r];
        L->tile_run[4 * r + 0] = t;
        L->tile_run[4 * r + 1] = L->tile_step_ptr[t];
        L->tile_run[4 * r + 2] = L->tile_step_ptr[t + 1] - L->tile_step_ptr[t];
        L->tile_run[4 * r + 3] = 0;
    }

    // Line groups for the block-sparse matmuls: G consecutive block-rows (o = 0,
    // CSR) or block-columns (o = 1, CSC) of one head, one slot per block index
    // of the union of their blocks.
    for (int o = 0; o < 2; ++o) {
        const std::vector<int32_t>& lp = o ? L->col_ptr : L->row_ptr;
        const std::vector<int32_t>& li = o ? L->row_idx : L->col_idx;
        L->gl_ptr[o].assign((size_t)L->n_tiles + 1, 0);
        L->gl_idx[o].clear();
        L->gl_blk[o].clear();
        std::vector<int32_t> sizes((size_t)L->n_tiles, 0);
        int64_t slots = 0;
        for (int h = 0; h < H; ++h) {
            for (int g = 0; g < L->ngroups; ++g) {
                const int t = h * L->ngroups + g;
                std::fill(in_union.begin(), in_union.end(), 0);
                for (int a = 0; a < G && g * G + a < nb; ++a) {
                    const int line = g * G + a;
                    for (int pp = lp[(size_t)h * (nb + 1) + line]; pp < lp[(size_t)h * (nb + 1) + line + 1]; ++pp)
                        in_union[li[pp]] = 1;
                }
                L->gl_ptr[o][t] = (int32_t)slots;
                for (int u = 0; u < nb; ++u) {
                    if (!in_union[u]) continue;
                    L->gl_idx[o].push_back(u);
                    for (int a = 0; a < G; ++a) {
                        const int line = g * G + a;
                        int32_t id = -1;
                        if (line < nb) id = (int32_t)(o ? id_at(h, u, line) : id_at(h, line, u));
                        L->gl_blk[o].push_back(id);
                    }
                    ++slots;
                    ++sizes[t];
                }
            }
        }
        L->gl_ptr[o][L->n_tiles] = (int32_t)slots;
        L->gl_order[o] = order_by_weight_desc(sizes);
    }

    // softmax chunk lists (element sizes 2 and 4 bytes)
    for (int e = 0; e < 2; ++e) {
        const int64_t elt = e ? 4 : 2;
        const int64_t budget = softmax_chunk_budget((int64_t)L->max_row_nnz * L->B * elt);
        L->sm_items[e].clear();
        L->sm_max_bytes[e] = 0;
        L->sm_fits[e] = true;
        for (int key = 0; key < H * nb; ++key) {
            const int64_t per_row = (int64_t)row_len[key] * L->B * elt;
            if (per_row == 0) continue;
            int R = L->B;
            while (R > 1 && R * per_row > budget) R >>= 1;
            if (R * per_row > budget) L->sm_fits[e] = false;
            L->sm_max_bytes[e] = std::max<int>(L->sm_max_bytes[e], (int)std::min<int64_t>(R * per_row, INT32_MAX));
            const int h = key / nb, i = key % nb;
            for (int r0 = 0; r0 < L->B; r0 += R) {
                L->sm_items[e].push_back(key);
                L->sm_items[e].push_back(L->row_ptr[(size_t)h * (nb + 1) + i]);  // = first block id
                L->sm_items[e].push_back(row_len[key]);
                L->sm_items[e].push_back(r0 | (R << 16));
            }
        }
    }
    L->max_tile_steps = tile_steps.empty() ? 0 : *std::max_element(tile_steps.begin(), tile_steps.end());
    return BSP_OK;
}

template <typename T>
size_t padded(size_t n) {
    return ((n * sizeof(T) + 255) / 256) * 256;
}

}  // namespace

namespace bsp {

// bsp_layout_plan with the affine-geometry analysis optional (callers that
// only need the tables skip it)
int layout_plan(const uint8_t* layout, int H, int nb, int block, bool analyse, bsp_layout_t* out) {
    if (!out) return BSP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!layout || H < 1 || nb < 1 || !valid_block(block)) return BSP_ERR_INVALID_ARG;
    if ((int64_t)nb * block > (1 << 24) || (int64_t)H * nb * nb > ((int64_t)1 << 31))
        return BSP_ERR_UNSUPPORTED;
    bsp_layout_s* L = new (std::nothrow) bsp_layout_s();
    if (!L) return BSP_ERR_OOM;
    L->H = H;
    L->nb = nb;
    L->B = block;
    L->S = nb * block;
    int rc;
    try {
        rc = build_tables(L, layout);
        if (rc == BSP_OK && analyse) affine_analyse(L, layout);
    } catch (const std::bad_alloc&) {
        rc = BSP_ERR_OOM;
    }
    if (rc != BSP_OK) {
        delete L;
        return rc;
    }
    *out = L;
    return BSP_OK;
}

}  // namespace bsp

extern "C" int bsp_layout_plan(const uint8_t* layout, int H, int nb, int block, bsp_layout_t* out) {
    return bsp::layout_plan(layout, H, nb, block, true, out);
}

extern "C" int bsp_layout_compile(const uint8_t* layout, int H, int nb, int block, void* stream,
                                  bsp_layout_t* out) {
    int rc = bsp_layout_plan(layout, H, nb, block, out);
    if (rc != BSP_OK) return rc;
    bsp_layout_s* L = *out;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaGetDevice(&L->device) != cudaSuccess) {
        delete L;
        *out = nullptr;
        return BSP_ERR_CUDA;
    }
    struct Part { const std::vector<int32_t>* v; const int32_t** dst; };
    LayoutView& V = L->view;
    Part parts[] = {
        {&L->row_ptr, &V.row_ptr},       {&L->col_idx, &V.col_idx},
        {&L->blk_id, &V.blk_id},         {&L->col_ptr, &V.col_ptr},
        {&L->row_idx, &V.row_idx},       {&L->blk_id_csc, &V.blk_id_csc},
        {&L->blk_key, &V.blk_key},       {&L->row_order, &V.row_order},
        {&L->col_order, &V.col_order},   {&L->tile_step_ptr, &V.tile_step_ptr},
        {&L->tile_order, &V.tile_order}, {&L->tile_run, &V.tile_run}, {&L->step_col, &V.step_col},
        {&L->step_blk, &V.step_blk},      {&L->sm_items[0], &V.sm_items[0]},
        {&L->sm_items[1], &V.sm_items[1]},
        {&L->gl_ptr[0], &V.gl_ptr[0]},   {&L->gl_order[0], &V.gl_order[0]},
        {&L->gl_idx[0], &V.gl_idx[0]},   {&L->gl_blk[0], &V.gl_blk[0]},
        {&L->gl_ptr[1], &V.gl_ptr[1]},   {&L->gl_order[1], &V.gl_order[1]},
        {&L->gl_idx[1], &V.gl_idx[1]},   {&L->gl_blk[1], &V.gl_blk[1]},
        {&L->geo_rec, &V.geo},
    };
    size_t total = padded<int>(4);  // status word first
    for (const Part& pt : parts) total += padded<int32_t>(pt.v->size() + 1);
    char* base = nullptr;
    if (cudaMalloc((void**)&base, total) != cudaSuccess) {
        cudaGetLastError();
        delete L;
        *out = nullptr;
        return BSP_ERR_OOM;
    }
    L->dmem = base;
    V.status = (int*)base;
    V.wait_ns = kDefaultWaitNs;
    V.inject = 0;
    size_t off = padded<int>(4);
    bool ok = cudaMemsetAsync(base, 0, padded<int>(4), s) == cudaSuccess;
    for (const Part& pt : parts) {
        int32_t* dst = (int32_t*)(base + off);
        *pt.dst = dst;
        if (!pt.v->empty())
            ok = ok && cudaMemcpyAsync(dst, pt.v->data(), pt.v->size() * sizeof(int32_t),
                                       cudaMemcpyHostToDevice, s) == cudaSuccess;
        off += padded<int32_t>(pt.v->size() + 1);
    }
    if (L->geo_rec.empty()) V.geo = nullptr;  // some head has no affine description
    V.H = L->H;
    V.nb = L->nb;
    V.B = L->B;
    V.S = L->S;
    V.G = L->G;
    V.ngroups = L->ngroups;
    V.n_tiles = L->n_tiles;
    V.nnz = L->nnz;
    for (int e = 0; e < 2; ++e) {
        V.sm_n_items[e] = (int)(L->sm_items[e].size() / 4);
        V.sm_max_bytes[e] = L->sm_max_bytes[e];
        V.sm_fits[e] = L->sm_fits[e] ? 1 : 0;
    }
    if (!ok) {
        cudaGetLastError();
        cudaStreamSynchronize(s);
        cudaFree(base);
        delete L;
        *out = nullptr;
        return BSP_ERR_CUDA;
    }
    L->on_device = true;
    return BSP_OK;
}

extern "C" int bsp_layout_destroy(bsp_layout_t L) {
    if (!L) return BSP_OK;
    int rc = BSP_OK;
    if (L->dmem) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != L->device) cudaSetDevice(L->device);
        if (cudaDeviceSynchronize() != cudaSuccess) rc = BSP_ERR_CUDA;
        bsp::host_pipe_destroy(L);
        bsp::schedules_destroy(L);
        if (cudaFree(L->dmem) != cudaSuccess) rc = BSP_ERR_CUDA;
        if (L->geo_dmem && cudaFree(L->geo_dmem) != cudaSuccess) rc = BSP_ERR_CUDA;
        if (cur >= 0 && cur != L->device) cudaSetDevice(cur);
    }
    delete L;
    return rc;
}

extern "C" int bsp_layout_info(bsp_layout_t L, int* H, int* nb, int* block, int64_t* nnz) {
    if (!L) return BSP_ERR_INVALID_ARG;
    if (H) *H = L->H;
    if (nb) *nb = L->nb;
    if (block) *block = L->B;
    if (nnz) *nnz = L->nnz;
    return BSP_OK;
}

extern "C" int bsp_layout_get_luts(bsp_layout_t L, int32_t* row_ptr, int32_t* col_idx,
                                   int32_t* blk_id, int32_t* col_ptr, int32_t* row_idx,
                                   int32_t* blk_id_csc) {
    if (!L) return BSP_ERR_INVALID_ARG;
    struct Out { int32_t* dst; const std::vector<int32_t>* host; const int32_t* dev; };
    Out outs[] = {{row_ptr, &L->row_ptr, L->view.row_ptr},
                  {col_idx, &L->col_idx, L->view.col_idx},
                  {blk_id, &L->blk_id, L->view.blk_id},
                  {col_ptr, &L->col_ptr, L->view.col_ptr},
                  {row_idx, &L->row_idx, L->view.row_idx},
                  {blk_id_csc, &L->blk_id_csc, L->view.blk_id_csc}};
    if (L->on_device) {
        if (cudaDeviceSynchronize() != cudaSuccess) return BSP_ERR_CUDA;
    }
    const size_t ptr_len = (size_t)L->H * (L->nb + 1), nnz = (size_t)L->nnz;
    const size_t lens[] = {ptr_len, nnz, nnz, ptr_len, nnz, nnz};
    int k = 0;
    for (const Out& o : outs) {
        const size_t len = L->host_tables ? o.host->size() : lens[k];
        ++k;
        if (!o.dst || len == 0) continue;
        const size_t bytes = len * sizeof(int32_t);
        if (L->on_device) {
            if (cudaMemcpy(o.dst, o.dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
                return BSP_ERR_CUDA;
        } else {
            std::memcpy(o.dst, o.host->data(), bytes);
        }
    }
    return BSP_OK;
}

extern "C" int bsp_layout_groups(bsp_layout_t L, int orient, int* G, int* n_groups, int64_t* n_slots,
                                 int32_t* grp_ptr, int32_t* grp_order, int32_t* slot_idx, int32_t* slot_blk) {
    if (!L || (orient != 0 && orient != 1)) return BSP_ERR_INVALID_ARG;
    if (G) *G = L->G;
    if (n_groups) *n_groups = L->n_tiles;
    if (!L->host_tables) {
        const size_t g = (size_t)L->G, nt = (size_t)L->n_tiles, sl = (size_t)L->gl_slots[orient];
        if (n_slots) *n_slots = (int64_t)sl;
        if (cudaDeviceSynchronize() != cudaSuccess) return BSP_ERR_CUDA;
        struct D { int32_t* dst; const int32_t* src; size_t n; };
        const D ds[] = {{grp_ptr, L->view.gl_ptr[orient], nt + 1}, {grp_order, L->view.gl_order[orient], nt},
                        {slot_idx, L->view.gl_idx[orient], sl}, {slot_blk, L->view.gl_blk[orient], sl * g}};
        for (const D& d : ds)
            if (d.dst && d.n && cudaMemcpy(d.dst, d.src, d.n * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
                return BSP_ERR_CUDA;
        return BSP_OK;
    }
    if (n_slots) *n_slots = (int64_t)L->gl_idx[orient].size();
    auto put = [](int32_t* dst, const std::vector<int32_t>& v) {
        if (dst && !v.empty()) std::copy(v.begin(), v.end(), dst);
    };
    put(grp_ptr, L->gl_ptr[orient]);
    put(grp_order, L->gl_order[orient]);
    put(slot_idx, L->gl_idx[orient]);
    put(slot_blk, L->gl_blk[orient]);
    return BSP_OK;
}

extern "C" int bsp_layout_softmax_chunks(bsp_layout_t L, int elt_bytes, int64_t* n_chunks, int* max_bytes,
                                         int* fits, int32_t* items) {
    if (!L || (elt_bytes != 2 && elt_bytes != 4)) return BSP_ERR_INVALID_ARG;
    const int e = elt_bytes == 4 ? 1 : 0;
    if (max_bytes) *max_bytes = L->sm_max_bytes[e];
    if (fits) *fits = L->sm_fits[e] ? 1 : 0;
    if (!L->host_tables) {
        const int64_t n = L->sm_n_items_dev[e];
        if (n_chunks) *n_chunks = n;
        if (items && n > 0) {
            if (cudaDeviceSynchronize() != cudaSuccess) return BSP_ERR_CUDA;
            if (cudaMemcpy(items, L->view.sm_items[e], (size_t)n * 4 * sizeof(int32_t), cudaMemcpyDeviceToHost) !=
                cudaSuccess)
                return BSP_ERR_CUDA;
        }
        return BSP_OK;
    }
    if (n_chunks) *n_chunks = (int64_t)(L->sm_items[e].size() / 4);
    if (items && !L->sm_items[e].empty()) std::copy(L->sm_items[e].begin(), L->sm_items[e].end(), items);
    return BSP_OK;
}

extern "C" int bsp_layout_tiles(bsp_layout_t L, int* G, int* n_tiles, int64_t* n_steps,
                                int32_t* tile_step_ptr, int32_t* tile_order, int32_t* step_col,
                                int32_t* step_blk) {
    if (!L) return BSP_ERR_INVALID_ARG;
    if (G) *G = L->G;
    if (n_tiles) *n_tiles = L->n_tiles;
    if (n_steps) *n_steps = L->n_steps;
    if (!L->host_tables) {
        const size_t G = (size_t)L->G, ns = (size_t)L->n_steps, nt = (size_t)L->n_tiles;
        if (cudaDeviceSynchronize() != cudaSuccess) return BSP_ERR_CUDA;
        struct D { int32_t* dst; const int32_t* src; size_t n; };
        const D ds[] = {{tile_step_ptr, L->view.tile_step_ptr, nt + 1}, {tile_order, L->view.tile_order, nt},
                        {step_col, L->view.step_col, ns * G}, {step_blk, L->view.step_blk, ns * G * G}};
        for (const D& d : ds)
            if (d.dst && d.n && cudaMemcpy(d.dst, d.src, d.n * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
                return BSP_ERR_CUDA;
        return BSP_OK;
    }
    auto put = [](int32_t* dst, const std::vector<int32_t>& v) {
        if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int32_t));
    };
    put(tile_step_ptr, L->tile_step_ptr);
    put(tile_order, L->tile_order);
    put(step_col, L->step_col);
    put(step_blk, L->step_blk);
    return BSP_OK;
}
