// Static schedules of the persistent attention kernels: which (tile, batch
// entry) work items each CTA runs, by longest-processing-time-first greedy
// assignment (every item, longest first, to the CTA with the least work so
// far).  A plain round-robin over the longest-first order gives one CTA every
// grid-th item, so a layout with a few very long tiles (BigBird's global rows:
// 64 blocks against ~6) leaves most CTAs idle while a few finish their long
// tiles plus a full share of short ones; the greedy assignment gives the CTAs
// that hold a long tile correspondingly fewer short ones.
//
// A schedule depends on the batch size Z and the grid, so it is built on the
// first launch with that pair and kept by the handle (one allocation each,
// read-only afterwards, so concurrent launches may share it).
#include <algorithm>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include "bsp_internal.h"

struct Schedules {
    std::mutex mu;
    struct Entry {
        int Z, grid;
        void* dmem;
    };
    std::vector<Entry> entries;
};

namespace bsp {

void schedules_destroy(bsp_layout_s* L) {
    if (!L->schedules) return;
    for (auto& e : L->schedules->entries) cudaFree(e.dmem);
    delete L->schedules;
    L->schedules = nullptr;
}

namespace {

// Items of all CTAs for the tiles' (tile, first step, step count) rows `run`
// (longest-first order, 4 ints each): offs [grid + 1], items [4 * Z * nt].
void build_schedule(const int32_t* run, int nt, int Z, int grid, std::vector<int32_t>& offs,
                    std::vector<int32_t>& items) {
    // work item w = rank * Z + z, weights non-increasing in w; each to the CTA
    // with the least work (ties: the lowest CTA index)
    const int64_t total = (int64_t)Z * nt;
    std::vector<int32_t> owner((size_t)total);
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < grid; ++c) heap.push({0, c});
    std::vector<int32_t> count((size_t)grid, 0);
    for (int64_t w = 0; w < total; ++w) {
        const int r = (int)(w / Z);
        const int64_t weight = std::max<int32_t>(run[4 * r + 2], 0) + 1;  // steps (+1: a tile's fixed cost)
        Load top = heap.top();
        heap.pop();
        owner[w] = top.second;
        ++count[top.second];
        heap.push({top.first + weight, top.second});
    }
    offs.assign((size_t)grid + 1, 0);
    for (int c = 0; c < grid; ++c) offs[c + 1] = offs[c] + count[c];
    items.assign((size_t)4 * total, 0);
    std::vector<int32_t> fill(offs.begin(), offs.end() - 1);
    for (int64_t w = 0; w < total; ++w) {  // each CTA's items in longest-first order
        const int r = (int)(w / Z), c = owner[w];
        int32_t* it = &items[(size_t)4 * fill[c]++];
        it[0] = run[4 * r + 0];
        it[1] = run[4 * r + 1];
        it[2] = run[4 * r + 2];
        it[3] = (int32_t)(w % Z);
    }
}

}  // namespace

int tile_schedule(bsp_layout_s* L, int Z, int grid, const int32_t** ptr, const int4** items) {
    if (!L->schedules) {
        static std::mutex create_mu;
        std::lock_guard<std::mutex> g(create_mu);
        if (!L->schedules) L->schedules = new (std::nothrow) Schedules();
        if (!L->schedules) return BSP_ERR_OOM;
    }
    Schedules* S = L->schedules;
    std::lock_guard<std::mutex> lock(S->mu);
    const size_t off_bytes = ((size_t)(grid + 1) * sizeof(int32_t) + 15) & ~(size_t)15;
    for (const auto& e : S->entries)
        if (e.Z == Z && e.grid == grid) {
            *ptr = (const int32_t*)e.dmem;
            *items = (const int4*)((char*)e.dmem + off_bytes);
            return BSP_OK;
        }
    // the tiles with their step counts in longest-first order (the host tables,
    // or the device tables read back for a handle compiled on the device)
    const int nt = L->n_tiles;
    std::vector<int32_t> run((size_t)4 * nt);
    if (nt > 0) {
        if (L->host_tables) {
            run = L->tile_run;
        } else if (cudaMemcpy(run.data(), L->view.tile_run, run.size() * sizeof(int32_t), cudaMemcpyDeviceToHost) !=
                   cudaSuccess) {
            cudaGetLastError();
            return BSP_ERR_CUDA;
        }
    }
    std::vector<int32_t> offs, items_h;
    build_schedule(run.data(), nt, Z, grid, offs, items_h);
    void* d = nullptr;
    const size_t bytes = off_bytes + items_h.size() * sizeof(int32_t);
    if (cudaMalloc(&d, bytes) != cudaSuccess) {
        cudaGetLastError();
        return BSP_ERR_OOM;
    }
    if (cudaMemcpy(d, offs.data(), offs.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
        (!items_h.empty() && cudaMemcpy((char*)d + off_bytes, items_h.data(), items_h.size() * sizeof(int32_t),
                                        cudaMemcpyHostToDevice) != cudaSuccess)) {
        cudaGetLastError();
        cudaFree(d);
        return BSP_ERR_CUDA;
    }
    S->entries.push_back({Z, grid, d});
    *ptr = (const int32_t*)d;
    *items = (const int4*)((char*)d + off_bytes);
    return BSP_OK;
}

}  // namespace bsp

extern "C" int bsp_diag_attention_schedule(bsp_layout_t L, int Z, int grid, int32_t* ptr, int32_t* items) {
    if (!L || !L->host_tables || Z < 1 || grid < 1 || !ptr || (!items && L->n_tiles > 0))
        return BSP_ERR_INVALID_ARG;
    std::vector<int32_t> offs, it;
    bsp::build_schedule(L->tile_run.data(), L->n_tiles, Z, grid, offs, it);
    std::copy(offs.begin(), offs.end(), ptr);
    std::copy(it.begin(), it.end(), items);
    return BSP_OK;
}
