// Static schedules of the persistent attention kernels: which work items each
// CTA runs, by longest-processing-time-first greedy assignment (every item,
// longest first, to the CTA with the least work so far).  A plain round-robin
// over the longest-first order gives one CTA every grid-th item, so a layout
// with a few very long tiles (BigBird's global rows: 64 blocks against ~6)
// leaves most CTAs idle while a few finish their long tiles plus a full share
// of short ones; the greedy assignment gives the CTAs that hold a long tile
// correspondingly fewer short ones.
//
// When one tile alone outweighs a CTA's fair share (a global row of a long
// sequence), no assignment of whole tiles balances the CTAs: such tiles are
// cut into pieces of consecutive steps.  Each piece writes its partial result
// -- the rows' unnormalised output with their running max and sum, the state
// of the online-softmax recurrence of the Triton-Puzzles blog, Puzzle 9
// "Simple FlashAttention" -- into a workspace slot, and a combine kernel
// merges the pieces of each tile by the same recurrence in piece order, so
// the result does not depend on which piece finished first.
//
// A schedule depends on the batch size Z, the number of SMs and the split
// setting; it is built on the first launch with that triple and kept by the
// handle (read-only afterwards; the workspace of a schedule with split tiles
// is ordered between streams by an event).
#include <algorithm>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include "bsp_internal.h"

struct Schedules {
    std::mutex mu;
    struct Entry {
        int Z, sms, split, force_cap;
        bsp::AttnSchedule sc;
        void* dmem;
    };
    std::vector<Entry> entries;
};

namespace bsp {

namespace {

struct Item {
    int32_t tile, s0, ns, z;
    int32_t part;  // workspace slot of a piece of a split tile, else -1
};

struct Built {
    int grid = 0;
    std::vector<int32_t> offs, items, part, combine;
    int n_slots = 0;
};

int64_t weight_of(const Item& it) { return (int64_t)std::max<int32_t>(it.ns, 0) + 1; }  // steps + a fixed cost

// Greedy assignment of `items` (non-increasing weight) to `grid` CTAs (ties:
// the lowest CTA index); returns the makespan, fills owner[i].
int64_t lpt(const std::vector<Item>& items, int grid, std::vector<int32_t>& owner) {
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < grid; ++c) heap.push({0, c});
    owner.assign(items.size(), 0);
    int64_t span = 0;
    for (size_t i = 0; i < items.size(); ++i) {
        Load top = heap.top();
        heap.pop();
        owner[i] = top.second;
        top.first += weight_of(items[i]);
        span = std::max(span, top.first);
        heap.push(top);
    }
    return span;
}

// Cut every item of more than `cap` steps into ceil(ns / cap) pieces of
// consecutive steps (sizes differing by at most one); the pieces of a tile get
// consecutive workspace slots, and `combine` one (tile, batch entry, first
// slot, pieces) record per cut tile.  The result is re-sorted longest-first
// (stable).
std::vector<Item> split_items(const std::vector<Item>& whole, int cap, std::vector<int32_t>& combine, int& n_slots) {
    std::vector<Item> out;
    combine.clear();
    n_slots = 0;
    for (const Item& it : whole) {
        if (it.ns <= cap) {
            out.push_back(it);
            continue;
        }
        const int np = (it.ns + cap - 1) / cap, base = it.ns / np, rem = it.ns % np;
        combine.insert(combine.end(), {it.tile, it.z, n_slots, np});
        int s = it.s0;
        for (int k = 0; k < np; ++k) {
            const int n = base + (k < rem ? 1 : 0);
            out.push_back({it.tile, s, n, it.z, n_slots + k});
            s += n;
        }
        n_slots += np;
    }
    std::stable_sort(out.begin(), out.end(), [](const Item& a, const Item& b) { return a.ns > b.ns; });
    return out;
}

// run: the tiles' (tile, first step, step count, 0) rows in longest-first
// order.  split: 0 = automatic, > 0 = cut every tile of more than `split`
// steps, < 0 = never cut for balance.  force_cap > 0: every tile of more
// than force_cap steps is cut whatever `split` says.
Built build_schedule(const int32_t* run, int nt, int Z, int sms, int split, int force_cap) {
    std::vector<Item> whole;
    whole.reserve((size_t)Z * nt);
    for (int r = 0; r < nt; ++r)
        for (int z = 0; z < Z; ++z) whole.push_back({run[4 * r], run[4 * r + 1], run[4 * r + 2], z, -1});
    int max_ns = 0;
    int64_t total = 0;
    for (const Item& it : whole) {
        max_ns = std::max(max_ns, it.ns);
        total += weight_of(it);
    }
    // items cut at `cap` steps (cap <= 0 or no longer tile: whole tiles)
    struct Plan {
        std::vector<Item> items;
        std::vector<int32_t> combine, owner;
        int n_slots = 0, grid = 0;
        int64_t span = 0;
    };
    auto plan = [&](int cap) {
        Plan p;
        if (cap > 0 && max_ns > cap) p.items = split_items(whole, cap, p.combine, p.n_slots);
        else p.items = whole;
        p.grid = (int)std::min<int64_t>((int64_t)p.items.size(), sms);
        p.span = p.grid > 0 ? lpt(p.items, p.grid, p.owner) : 0;
        return p;
    };
    auto cap_min = [](int a, int b) { return a <= 0 ? b : (b <= 0 ? a : std::min(a, b)); };
    Plan best;
    if (split > 0) {
        best = plan(cap_min(split, force_cap));
    } else if (split < 0) {
        best = plan(force_cap);
    } else {
        // automatic: pieces of about half a CTA's fair share, kept when they
        // shorten the greedy makespan by a tenth and by at least 24 steps of
        // 128 keys (measured: the pieces' partial writes and the combine pass
        // cost more than a predicted saving of 11 steps on a 33-step span)
        best = plan(force_cap);
        const int cap = cap_min((int)std::max<int64_t>(4, (total + 2 * (int64_t)sms - 1) / (2 * (int64_t)sms)),
                                force_cap);
        if (max_ns > cap && cap != force_cap) {
            Plan cut = plan(cap);
            if (best.span - cut.span >= 24 && 10 * cut.span < 9 * best.span) best = std::move(cut);
        }
    }
    Built b;
    b.grid = best.grid;
    b.n_slots = best.n_slots;
    b.combine = best.combine;
    const std::vector<Item>& items = best.items;
    std::vector<int32_t> count((size_t)b.grid, 0);
    for (size_t i = 0; i < items.size(); ++i) ++count[best.owner[i]];
    b.offs.assign((size_t)b.grid + 1, 0);
    for (int c = 0; c < b.grid; ++c) b.offs[c + 1] = b.offs[c] + count[c];
    b.items.assign((size_t)4 * items.size(), 0);
    b.part.assign(items.size(), -1);
    std::vector<int32_t> fill(b.offs.begin(), b.offs.begin() + b.grid);
    for (size_t i = 0; i < items.size(); ++i) {  // each CTA's items in longest-first order
        const int32_t k = fill[best.owner[i]]++;
        b.items[4 * k + 0] = items[i].tile;
        b.items[4 * k + 1] = items[i].s0;
        b.items[4 * k + 2] = items[i].ns;
        b.items[4 * k + 3] = items[i].z;
        b.part[k] = items[i].part;
    }
    return b;
}

size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

}  // namespace

void schedules_destroy(bsp_layout_s* L) {
    if (!L->schedules) return;
    for (auto& e : L->schedules->entries) {
        cudaFree(e.dmem);
        if (e.sc.ws) cudaFree(e.sc.ws);
        if (e.sc.done) cudaEventDestroy(e.sc.done);
        delete e.sc.mu;
    }
    delete L->schedules;
    L->schedules = nullptr;
}

int tile_schedule(bsp_layout_s* L, int Z, int sms, int force_cap, AttnSchedule* out) {
    if (!L->schedules) {
        static std::mutex create_mu;
        std::lock_guard<std::mutex> g(create_mu);
        if (!L->schedules) L->schedules = new (std::nothrow) Schedules();
        if (!L->schedules) return BSP_ERR_OOM;
    }
    Schedules* S = L->schedules;
    std::lock_guard<std::mutex> lock(S->mu);
    const int split = L->attn_split;
    for (const auto& e : S->entries)
        if (e.Z == Z && e.sms == sms && e.split == split && e.force_cap == force_cap) {
            *out = e.sc;
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
    const Built b = build_schedule(run.data(), nt, Z, sms, split, force_cap);
    const size_t o_items = align16(b.offs.size() * sizeof(int32_t));
    const size_t o_part = o_items + b.items.size() * sizeof(int32_t);
    const size_t o_comb = o_part + align16(b.part.size() * sizeof(int32_t));
    const size_t bytes = o_comb + b.combine.size() * sizeof(int32_t);
    AttnSchedule sc{};
    sc.grid = b.grid;
    sc.n_split = (int)(b.combine.size() / 4);
    void* d = nullptr;
    if (cudaMalloc(&d, bytes) != cudaSuccess) {
        cudaGetLastError();
        return BSP_ERR_OOM;
    }
    auto up = [&](size_t off, const std::vector<int32_t>& v) {
        return v.empty() ||
               cudaMemcpy((char*)d + off, v.data(), v.size() * sizeof(int32_t), cudaMemcpyHostToDevice) == cudaSuccess;
    };
    bool ok = up(0, b.offs) && up(o_items, b.items) && up(o_part, b.part) && up(o_comb, b.combine);
    if (ok && sc.n_split > 0) {
        // partial results: per slot 128 rows of O (head size up to 128) and
        // each row's running max and sum
        void* ws = nullptr;
        ok = cudaMalloc(&ws, (size_t)b.n_slots * kPartFloats * sizeof(float)) == cudaSuccess;
        sc.ws = (float*)ws;
        ok = ok && cudaEventCreateWithFlags(&sc.done, cudaEventDisableTiming) == cudaSuccess;
        sc.mu = ok ? new (std::nothrow) std::mutex() : nullptr;
        ok = ok && sc.mu != nullptr;
    }
    if (!ok) {
        cudaGetLastError();
        cudaFree(d);
        if (sc.ws) cudaFree(sc.ws);
        if (sc.done) cudaEventDestroy(sc.done);
        return BSP_ERR_OOM;
    }
    sc.ptr = (const int32_t*)d;
    sc.items = (const int4*)((char*)d + o_items);
    sc.part = (const int32_t*)((char*)d + o_part);
    sc.combine = (const int4*)((char*)d + o_comb);
    S->entries.push_back({Z, sms, split, force_cap, sc, d});
    *out = sc;
    return BSP_OK;
}

}  // namespace bsp

extern "C" int bsp_diag_attention_schedule(bsp_layout_t L, int dtype, int Z, int n_sm, int* grid, int* n_items,
                                           int* n_split, int32_t* ptr, int32_t* items, int32_t* part,
                                           int32_t* combine) {
    if (!L || !L->host_tables || Z < 1 || n_sm < 1 || !grid || !n_items || !n_split) return BSP_ERR_INVALID_ARG;
    if (dtype != BSP_F32 && dtype != BSP_BF16 && dtype != BSP_F16) return BSP_ERR_INVALID_ARG;
    const bsp::Built b = bsp::build_schedule(L->tile_run.data(), L->n_tiles, Z, n_sm, L->attn_split,
                                             bsp::attn_force_cap(dtype));
    *grid = b.grid;
    *n_items = (int)b.part.size();
    *n_split = (int)(b.combine.size() / 4);
    if (ptr) std::copy(b.offs.begin(), b.offs.end(), ptr);
    if (items) std::copy(b.items.begin(), b.items.end(), items);
    if (part) std::copy(b.part.begin(), b.part.end(), part);
    if (combine) std::copy(b.combine.begin(), b.combine.end(), combine);
    return BSP_OK;
}

extern "C" int bsp_diag_attention_split(bsp_layout_t L, int max_steps) {
    if (!L) return BSP_ERR_INVALID_ARG;
    L->attn_split = max_steps;
    return BSP_OK;
}
