// Fused block-sparse attention on tcgen05 tensor cores (bf16 / fp16 in,
// fp32 accumulate): the SDD -> softmax -> DSD chain of "question on
// blocksparse" (openai/triton issue 117) in one pass that never writes the
// scores, with the online-softmax recurrence of the Triton-Puzzles blog,
// Puzzle 9 "Simple FlashAttention" (running max m, running sum l, output
// rescaled by exp(m_old - m_new), divided by l at the end).
//
// Work: one row tile = 128 query rows (G = 128/B consecutive block-rows of one
// head) x one batch entry.  Its key blocks are the union of the block-rows'
// columns, visited 128 key rows (G blocks) per step; a (row block, key block)
// pair that is not in the layout is masked to -inf, as are entries the intra-
// block mask removes.  Persistent CTAs walk the tiles longest-first.
//
// Roles (512 threads, one CTA per SM):
//   warps 0, 3  TMA producers: warp 0 the Q tile (2 stages) and K tiles, warp 3
//               the V tiles (2 stages each), so that K never waits behind V
//   warp 1      TMEM owner; one thread issues S[g%3] = Q K^T (M=128, N=128, K=D)
//   warp 2      one thread issues O += P V (M=128, N=D, K=128; P from TMEM, V
//               MN-major).  Two issuing threads halve each one's per-step
//               barrier waits and commits, which cost about as much as the MMAs.
//   warps 4..7  epilogue: as soon as the last P V of a tile has completed they
//               read O out of TMEM (thread = row), hand the accumulator back to
//               the next tile, scale by 1 / l and write the tile through a
//               128-byte-swizzled shared-memory panel with TMA stores.  The
//               next tile's softmax runs meanwhile, so the tensor core does not
//               wait for the output write.
//   warps 8..15 softmax, both warpgroups on every step, one half row each:
//               thread = one query row = one TMEM lane, warpgroup wg the scores
//               of keys [64 wg, 64 wg + 64).  Reads its half of S from TMEM,
//               masks, takes the half-row max and swaps it with the other
//               thread of the row through shared memory, writes its P
//               (bf16/fp16) into the step's buffer, rescales its half of O in
//               TMEM only when the running max grew by more than 2^8 (the final
//               O / l is exact either way), and hands its half-row sums to the
//               epilogue, which adds them.
// TMEM columns: S0 [0,128), S1 [128,256), S2 [256,384), O [384, 384+D).  Step g
// uses S buffer g % 3; its P (two 16-bit values per column) overwrites the
// first 64 columns of the same buffer once the scores are in registers (keys
// [0, 64) into columns [0, 32) by warpgroup 0, keys [64, 128) into columns
// [32, 64) by warpgroup 1 after warpgroup 0 has announced its maximum, i.e.
// loaded those columns), and P V takes its A operand from there.  With three
// buffers Q K^T of step g waits only for P V of step g - 3, so the next scores
// are ready when the softmax finishes a step.
// GEO (opt-in): every head of the layout has an affine description (band
// and / or column term); the TMA producers compute each step's key blocks
// from it instead of reading the step tables.  The softmax keeps reading the tables:
// its loads are issued a step ahead, so they cost nothing on its critical
// path, while computing columns and presence there (integer divisions for
// the column term, 13 more live registers) slowed the banded workload by 10 %
// and the strided one by 31 %.
#pragma once

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "geometry.cuh"
#include "tc_common.cuh"

namespace bsp {
namespace attn {

using namespace tc;

constexpr int kThreads = 512;
// Registers per thread after the split at kernel start (launched with 128):
// warps 0-3 (producers, issuers) give some to the two softmax warpgroups, the
// epilogue keeps its share.  128 threads x (80 + 128 + 152 + 152) = 65536 =
// 512 threads x 128, the block's allocation at launch.
constexpr uint32_t kRegsLaunch = 128, kRegsCtl = 80, kRegsEpi = 128, kRegsSoftmax = 152;
static_assert(kRegsCtl + kRegsEpi + 2 * kRegsSoftmax <= 4 * kRegsLaunch, "register split exceeds the launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max grows by > 256x
// Of every 8 column pairs of a score row, this many take 2^x from the FMA-pipe
// polynomial and the rest from the special-function unit: with one thread per
// row, the special-function unit alone would need as long per step as both
// matrix products.
#ifndef BSP_ATTN_POLY_PAIRS
#define BSP_ATTN_POLY_PAIRS 0
#endif
constexpr int kPolyPairs = BSP_ATTN_POLY_PAIRS;

template <int D>
struct AttnSmem {
    static constexpr int KP = D / 64;                 // 64-column panels per 128-row tile
    static constexpr int kTile = 128 * D * 2;         // bytes of one 128 x D tile
    static constexpr int QST = 2;                     // Q tile stages
    static constexpr int KVST = 2;                    // K and V step-tile stages each
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + QST * kTile;
    static constexpr int kV = kK + KVST * kTile;
    static constexpr int kEpi = kV + KVST * kTile;    // epilogue staging: one 32 x 64 panel per warp
    static constexpr int kBytes = kEpi + 4 * 4096;
    static constexpr int kAlloc = kBytes + 1024;      // slack for 1024-byte alignment
};

struct AttnArgs {
    LayoutView L;
    void* O;
    const uint8_t* mask;
    // the CTA's work items: sched_items[sched_ptr[c] .. sched_ptr[c + 1]) =
    // (tile, first step, step count, batch entry), longest-first greedy
    const int32_t* sched_ptr;
    const int4* sched_items;
    // per item: the partial-result slot of a piece of a cut tile, else -1;
    // a piece leaves its rows' raw O, running max and sum in part_ws
    const int32_t* sched_part;
    float* part_ws;
    float* lse;  // the rows' log-sum-exp of the scaled scores [Z][H][S] (natural log), or null
    int Z;
    int kind;
    float c2;  // scale * log2(e)
};

template <typename T, int BLK, int D, int KIND, bool GEO>
__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnArgs args) {
    using SM = AttnSmem<D>;
    constexpr int G = 128 / BLK;
    constexpr int KP = SM::KP;
    constexpr uint32_t kTileBytes = SM::kTile;
    constexpr uint32_t kIdescQK = idesc_f16(128, 128, std::is_same<T, __nv_bfloat16>::value, 0, 0);
    constexpr uint32_t kIdescPV = idesc_f16(128, D, std::is_same<T, __nv_bfloat16>::value, 0, 1);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int QST = SM::QST;
    // K and V tiles of step g sit in stage g % 2; S buffer g % 3 has s_full
    // (Q K^T done, which also frees the K stage of that step), p_full (P
    // written) and pv_done (P V done, which frees the buffer and the V stage).
    __shared__ uint64_t q_full[QST], q_empty[QST], k_full[2], v_full[2];
    __shared__ uint64_t s_full[3], p_full[3], pv_done[3];
    // O accumulator: o_full = last P V of the tile completed, o_empty = the
    // epilogue has read it.  Row sums: lsum[tile parity][warpgroup][row], with
    // l_full (softmax wrote them) and l_empty (the epilogue read them).
    __shared__ uint64_t o_full, o_empty, l_full[2], l_empty[2];
    __shared__ float lsum[2][2][128], lref[2][2][128];  // each warpgroup's sum and its reference max
    // half-row maxima of step g, one per warpgroup: xm[g % 2][wg][row], both
    // halves of quadrant q announced by x_full[g % 2][q] (the 2 warps of the
    // quadrant, so each pair of warps proceeds at its own pace)
    __shared__ float xm[2][2][128];
    __shared__ uint64_t x_full[2][4];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    // what each issuing thread had issued when it stopped: K steps, Q tiles
    // (bit 31: the first was skipped by the test injection), V steps, Q K^T
    // steps, P V steps -- drained after the roles stop if the kernel aborted
    __shared__ uint32_t issued[5];

    const LayoutView& L = args.L;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Abort ab{&abort_flag, L.status, L.wait_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 5; ++i) issued[i] = 0;
        for (int i = 0; i < QST; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&pv_done[i], 1);
            // the 8 softmax warps (each writes the P of its half rows)
            mbar_init(&p_full[i], 8);
        }
        mbar_init(&o_full, 1);
        mbar_init(&o_empty, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&l_full[i], 8);
            mbar_init(&l_empty[i], 4);
            for (int q = 0; q < 4; ++q) mbar_init(&x_full[i][q], 2);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;        // S buffers at columns 0, 128 and 256
    const uint32_t tO = tmem_base + 384;  // O at column 384

    const int S = L.S;

    // Each warpgroup changes its register share first thing in its own branch
    // (so the new limit holds for all of the role's code), before any role can
    // leave early.
    if (warp < 4) {
    regs_dec<kRegsCtl>();
    if (warp == 0 || warp == 3) {
        // ----------------------------------------------- TMA producers ----
        // warp 0 loads Q and K, warp 3 loads V: the K tile of a step waits only
        // for Q K^T two steps back, never behind a V tile whose P V is late.
        if (lane == 0) {
            const bool is_v = warp == 3;
            const CUtensorMap* tm = is_v ? &tmV : &tmK;
            if (!is_v) tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(tm);
            uint32_t q_it = 0, g = 0;
            bool q_skipped = false;  // test injection: the first Q tile was never loaded
            for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
                const int4 run = args.sched_items[it];
            const int tile = run.x;
                const int z = run.w;
                const int h = tile / L.ngroups, gq = tile % L.ngroups;
                const int s0 = run.y, ns = run.z;
                if (ns == 0) continue;
                const int64_t zh = (int64_t)z * L.H + h;
                GeoHead gh{};
                GeoTile gt{};
                if constexpr (GEO) {
                    gh = geo_load(L.geo + h * kGeoRec);
                    gt = geo_tile(gh, gq * G, min(gq * G + G, L.nb) - 1, L.nb);
                }
                if (!is_v) {
                    const uint32_t qs = q_it % QST;
                    if (!mbar_wait(&q_empty[qs], ((q_it / QST) & 1) ^ 1, ab)) break;
                    if (q_it == 0 && (L.inject & kInjectSkipFirstQ)) {
                        q_skipped = true;  // neither the copy nor the arrival: Q K^T waits in vain
                    } else {
                        mbar_arrive_expect_tx(&q_full[qs], kTileBytes);
                        for (int p = 0; p < KP; ++p)
                            tma_load_2d(smem_u32(smem + SM::kQ + qs * kTileBytes + p * 16384), &tmQ, p * 64,
                                        (int32_t)(zh * S + gq * 128), &q_full[qs]);
                    }
                    ++q_it;
                }
                for (int n = 0; n < ns; ++n, ++g) {
                    const int s = s0 + n;
                    const uint32_t st = g & 1;
                    int cols[G];
#pragma unroll
                    for (int b = 0; b < G; ++b) {
                        if constexpr (GEO) {
                            const int c = geo_col(gh, gt, n * G + b);
                            cols[b] = c >= 0 ? c : geo_col(gh, gt, n * G);  // padding slot: any valid block
                        } else {
                            const int c = L.step_col[s * G + b];
                            cols[b] = c >= 0 ? c : L.step_col[s * G];  // padding slot: any valid block
                        }
                    }
                    if (!is_v && g == 0 && (L.inject & kInjectBadColumn)) cols[0] = L.nb;
                    // bounds check of the block-columns that become TMA coordinates:
                    // a bad table entry stops the kernel with BSP_ERR_DEVICE_CHECK
                    bool cols_ok = true;
#pragma unroll
                    for (int b = 0; b < G; ++b) cols_ok &= (unsigned)cols[b] < (unsigned)L.nb;
                    if (!cols_ok) {
                        ab.fail(BSP_ERR_DEVICE_CHECK);
                        goto producer_done;
                    }
                    // stage g % 2 is free once step g - 2 has used it: Q K^T for a K
                    // tile, P V for a V tile
                    uint64_t* full = is_v ? &v_full[st] : &k_full[st];
                    if (g >= 2) {
                        const uint32_t gp = g - 2;
                        uint64_t* freed = is_v ? &pv_done[gp % 3] : &s_full[gp % 3];
                        if (!mbar_wait(freed, (gp / 3) & 1, ab)) goto producer_done;
                    }
                    mbar_arrive_expect_tx(full, kTileBytes);
                    const uint32_t base = smem_u32(smem + (is_v ? SM::kV : SM::kK) + st * kTileBytes);
#pragma unroll
                    for (int b = 0; b < G; ++b)
                        for (int p = 0; p < KP; ++p)
                            tma_load_2d(base + p * 16384 + b * BLK * 128, tm, p * 64,
                                        (int32_t)(zh * S + (int64_t)cols[b] * BLK), full);
                }
            }
        producer_done:
            if (is_v) {
                issued[2] = g;
            } else {
                issued[0] = g;
                issued[1] = q_it | (q_skipped ? 0x80000000u : 0u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------- Q K^T issuer (one thread) ----
        if (lane == 0) {
            // descriptors of the first stage; stage / K-step offsets are added to the
            // start-address field (addresses stay below 2^18, so no carry leaves it)
            const uint64_t dq = smem_desc(smem_u32(smem + SM::kQ), 16, 1024, kSw128);
            const uint64_t dk = smem_desc(smem_u32(smem + SM::kK), 16, 1024, kSw128);
            uint32_t q_it = 0, g = 0;
            for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
                const int ns = args.sched_items[it].z;
                if (ns == 0) continue;
                const uint32_t qs = q_it % QST;
                if (!mbar_wait(&q_full[qs], (q_it / QST) & 1, ab)) goto qk_done;
                for (int n = 0; n < ns; ++n, ++g) {
                    const uint32_t st = g & 1, sb = g % 3;
                    // S buffer g % 3 is free once P V of step g - 3 has read its P
                    if (g >= 3 && !mbar_wait(&pv_done[sb], ((g - 3) / 3) & 1, ab)) goto qk_done;
                    if (!mbar_wait(&k_full[st], (g >> 1) & 1, ab)) goto qk_done;
                    tc_fence_after();
                    const uint64_t aq = dq + ((qs * kTileBytes) >> 4), bk = dk + ((st * kTileBytes) >> 4);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t off = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                        mma_f16(tS + sb * 128, aq + off, bk + off, kIdescQK, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&s_full[sb]);
                    if (n == ns - 1) mma_commit(&q_empty[qs]);
                }
                ++q_it;
            }
        qk_done:
            issued[3] = g;
        }
    } else if (warp == 2) {
        // --------------------------------------------- P V issuer (one thread) ----
        if (lane == 0) {
            const uint64_t dv = smem_desc(smem_u32(smem + SM::kV), 128 * 128, 1024, kSw128);
            uint32_t g = 0, tc = 0;  // tc: tiles with at least one step so far
            for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
                const int ns = args.sched_items[it].z;
                if (ns == 0) continue;
                // the previous tile's O must have been read by the epilogue
                if (tc > 0 && !mbar_wait(&o_empty, (tc - 1) & 1, ab)) goto pv_done_label;
                for (int n = 0; n < ns; ++n, ++g) {
                    const uint32_t st = g & 1, sb = g % 3;
                    // P of step g written (and O rescaled) by its warpgroup; V landed
                    if (!mbar_wait(&p_full[sb], (g / 3) & 1, ab)) goto pv_done_label;
                    if (!mbar_wait(&v_full[st], (g >> 1) & 1, ab)) goto pv_done_label;
                    tc_fence_after();
                    const uint64_t bv = dv + ((st * kTileBytes) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)  // P (A operand) from TMEM: 8 columns per 16 keys
                        mma_f16_tmem_a(tO, tS + sb * 128 + ks * 8, bv + ((ks * 2048) >> 4), kIdescPV,
                                       (ks > 0 || n > 0) ? 1u : 0u);
                    mma_commit(&pv_done[sb]);
                }
                mma_commit(&o_full);
                ++tc;
            }
        pv_done_label:
            issued[4] = g;
        }
    }
    } else if (warp < 8) {
        if constexpr (kRegsEpi < kRegsLaunch) regs_dec<kRegsEpi>();
        else if constexpr (kRegsEpi > kRegsLaunch) regs_inc<kRegsEpi>();
        // ---------------------------------------------------- epilogue ----
        // Warp q owns rows [32 q, 32 q + 32) of the tile (TMEM lanes of its
        // quadrant).  O / l leaves through a 32 x 64 staging panel per warp in
        // the 128-byte-swizzled layout (16-byte chunk j of row r at chunk
        // j ^ (r % 8), so the row-per-thread writes hit distinct banks) and
        // one TMA store per panel; rows past the sequence end are clipped by
        // the tensor map.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint8_t* stage = smem + SM::kEpi + quad * 4096;
        const uint32_t stage_s = smem_u32(stage);
        uint32_t tc = 0;
        for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
            const int4 run = args.sched_items[it];
            const int tile = run.x;
            const int z = run.w;
            const int h = tile / L.ngroups, gq = tile % L.ngroups;
            const int ns = run.z;
            const int y0 = gq * 128 + quad * 32;  // first sequence row of this warp
            const int32_t zh = (int32_t)((int64_t)z * L.H + h);
            const bool live = ns > 0;
            const int part = args.sched_part[it];
            const uint32_t lb = tc & 1;
            float inv = 0.f;  // rows with nothing kept are 0
            float mf = -INFINITY, lt = 0.f;
            if (live) {
                bool ok = mbar_wait(&l_full[lb], (tc >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto epilogue_done;
                // O is scaled by the tile's final running max, the larger reference;
                // a warpgroup without a kept entry has reference -inf and sum 0
                const float m0 = lref[lb][0][row], m1 = lref[lb][1][row];
                const float l0 = lsum[lb][0][row], l1 = lsum[lb][1][row];
                __syncwarp();
                if (lane == 0) mbar_arrive(&l_empty[lb]);
                mf = fmaxf(m0, m1);
                lt = mf == -INFINITY ? 0.f : l0 * ex2_approx(m0 - mf) + l1 * ex2_approx(m1 - mf);
                inv = lt > 0.f ? 1.0f / lt : 0.f;
                ok = mbar_wait(&o_full, tc & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto epilogue_done;
                tc_fence_after();
            }
            if (args.lse && part < 0 && y0 + lane < S)  // cut tiles: the combine pass writes it
                args.lse[(int64_t)zh * S + y0 + lane] = lt > 0.f ? (mf + log2f(lt)) * kLn2 : -INFINITY;
            if (part >= 0) {
                // a piece of a cut tile: the row's O as accumulated (relative
                // to its reference max mf), mf and the sum, for the combine
                // pass; every piece has steps, so live holds
                float* pw = args.part_ws + (size_t)part * kPartFloats;
                float* orow = pw + (size_t)row * D;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32_sync(tO + lane_base + c * 32, r);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint4*>(orow + c * 32 + 4 * k) =
                            make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_empty);
                pw[kPartRows * kPartMaxD + row] = mf;
                pw[kPartRows * kPartMaxD + kPartRows + row] = lt;
                ++tc;
                continue;
            }
            // O leaves through the warp's 32 x 64 staging panel, one TMA store per
            // 64 columns.  Every column of O is read out of TMEM before the
            // accumulator is handed back to the next tile's P V, and before any
            // wait on a store of this tile: the first panel goes to the staging
            // panel as it is read (the panel's previous store, issued a tile
            // ago, has long finished reading it), the second is held in
            // registers until the first panel's store has read the staging.
            {
                const bool out = y0 < S;
                uint8_t* rp = stage + lane * 128;
                auto put = [&](const uint32_t (&pk)[32]) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(rp + ((j ^ (lane & 7)) << 4)) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                };
                auto store = [&](int p) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmO, stage_s, p * 64, y0, zh);
                        bulk_commit();
                    }
                };
                auto read_panel = [&](int p, uint32_t (&pk)[32]) {
                    uint32_t r[64];  // 64 columns, two loads and one wait
                    tmem_ld64_sync(tO + lane_base + p * 64, tO + lane_base + p * 64 + 32, r);
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        pk[k] = Pack2<T>::pack(__uint_as_float(r[2 * k]) * inv, __uint_as_float(r[2 * k + 1]) * inv);
                };
                if (out) {
                    if (lane == 0) bulk_wait_read_all();  // the staging panel is free
                    __syncwarp();
                }
                uint32_t pk[32];
                if (live) {
                    read_panel(0, pk);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) pk[k] = 0u;
                }
                if (out) put(pk);
                if constexpr (KP == 2) {
                    if (live) {
                        read_panel(1, pk);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) pk[k] = 0u;
                    }
                }
                if (live) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&o_empty);
                }
                if (out) {
                    store(0);
                    if constexpr (KP == 2) {
                        if (lane == 0) bulk_wait_read_all();  // the first panel's store has read the staging
                        __syncwarp();
                        put(pk);
                        store(1);
                    }
                }
            }
            if (live) ++tc;
        }
    epilogue_done:
        if (lane == 0) bulk_wait_all();
    } else {
        regs_inc<kRegsSoftmax>();
        // ---------------------------------------------------- softmax ----
        // Both warpgroups work on every step, each on one half of the row's
        // 128 scores: warpgroup wg takes keys [64 wg, 64 wg + 64) of the rows
        // of its warp's TMEM lane quadrant (thread = query row = TMEM lane).
        // The two threads of a row (warp 8 + q and warp 12 + q, quadrant q)
        // swap their half-row maxima through shared memory (x_full barriers),
        // so both reach the same running max m and the same decisions; each
        // writes the P of its keys (keys [0, 64) into columns [0, 32), keys
        // [64, 128) into columns [32, 64) -- the latter over scores of the other
        // half, which its owner has loaded before it announced its maximum),
        // rescales its half of O when m moved, and keeps its half-row sum
        // against m; the epilogue adds the two halves.  A step's critical path
        // is half a row of work plus the exchange.
        constexpr int W = BLK < 64 ? BLK : 64;  // columns of one slot inside a half row
        constexpr int LS = 64 / W;              // slots (or slot parts) per half row
        const int sw = warp - 8, wg = sw >> 2, hf = wg;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // query row inside the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int r_in = row % BLK, a = row / BLK;
        uint32_t g = 0, tc = 0;
        // metadata of one half row: block id at (row block a, slot) and block-column, per slot part
        struct Half {
            int blk[LS], cb[LS];
        };
        auto fetch = [&](int s, Half& o) {
#pragma unroll
            for (int ls = 0; ls < LS; ++ls) {
                const int b = (hf * 64 + ls * W) / BLK;
                o.blk[ls] = L.step_blk[(s * G + a) * G + b];
                o.cb[ls] = L.step_col[s * G + b];
            }
        };
        // mask this thread's half (64 columns) of the row in place
        auto mask_half = [&](float (&v)[64], const Half& md, int rb, int rseq) {
#pragma unroll
            for (int ls = 0; ls < LS; ++ls) {
                const int kbase = (hf * 64 + ls * W) % BLK;  // in-block column of v[ls * W]
                if (KIND == BSP_MASK_DIAG_CAUSAL) {
                    // keep columns j <= lim: none if the block is absent, j <= r_in - kbase
                    // inside the diagonal block, all otherwise.  Only a diagonal or an
                    // absent block removes anything, so the selects run only when some
                    // lane of the warp has one (for blocks of 32 and more a warp's rows
                    // are in one block-row, so the test is usually uniform).
                    const int lim = md.blk[ls] < 0 ? -1 : (md.cb[ls] == rb ? r_in - kbase : W);
                    if (__any_sync(0xffffffffu, lim < W - 1)) {
#pragma unroll
                        for (int j = 0; j < W; ++j) v[ls * W + j] = j > lim ? -INFINITY : v[ls * W + j];
                    }
                } else if (md.blk[ls] < 0) {
#pragma unroll
                    for (int j = 0; j < W; ++j) v[ls * W + j] = -INFINITY;
                } else if (KIND == BSP_MASK_DENSE) {
                    const uint8_t* mp = args.mask + (int64_t)rseq * S + (int64_t)md.cb[ls] * BLK + kbase;
#pragma unroll
                    for (int q = 0; q < W / 16; ++q) {
                        uint4 mv = *reinterpret_cast<const uint4*>(mp + q * 16);
                        const uint8_t* mb = reinterpret_cast<const uint8_t*>(&mv);
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (!mb[k]) v[ls * W + q * 16 + k] = -INFINITY;
                    }
                }
            }
        };
        auto max64 = [](const float (&v)[64]) {
            // 8 independent chains of three-input maxima
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = fmax3(v[k], v[k + 8], v[k + 16]);
#pragma unroll
            for (int c = 24; c < 64; c += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = fmax3(m8[k], v[c + k], c + 8 + k < 64 ? v[c + 8 + k] : v[c + k]);
            return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        };
        // p = 2^(s * c2 - msub) for 64 entries -> 32 packed pairs; returns their sum
        auto exp64 = [&](const float (&v)[64], float msub, uint32_t (&pk)[32]) {
            const float2 c2v = make_float2(args.c2, args.c2), nm = make_float2(-msub, -msub);
            float2 rs4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) rs4[k] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 y = __ffma2_rn(make_float2(v[2 * c], v[2 * c + 1]), c2v, nm);
                const float2 p = (c & 7) < kPolyPairs ? exp2_poly2(y) : make_float2(ex2_approx(y.x), ex2_approx(y.y));
                rs4[c & 3] = __fadd2_rn(rs4[c & 3], p);
                pk[c] = Pack2<T>::pack(p.x, p.y);
            }
            const float2 r2 = __fadd2_rn(__fadd2_rn(rs4[0], rs4[1]), __fadd2_rn(rs4[2], rs4[3]));
            return r2.x + r2.y;
        };
        // the CTA's work items (tile id, first step, step count, batch entry);
        // ns = -1 past the end
        const int it_end = args.sched_ptr[blockIdx.x + 1];
        auto tile_info = [&](int it, int& tile, int& s0, int& ns) {
            if (it >= it_end) {
                tile = 0;
                s0 = 0;
                ns = -1;
                return;
            }
            const int4 run = args.sched_items[it];
            tile = run.x;
            s0 = run.y;
            ns = run.z;
        };
        int it = args.sched_ptr[blockIdx.x];
        int tile, s0, ns;
        tile_info(it, tile, s0, ns);
        while (ns == 0) {  // the epilogue writes the zero rows of empty tiles
            ++it;
            tile_info(it, tile, s0, ns);
        }
        Half hnext;
        if (ns > 0) fetch(s0, hnext);
        while (ns > 0) {
            // the next tile's place in the tables: loaded now, first used at this
            // tile's last step, so the loads overlap the steps
            int itn = it + 1;
            int tn, s0n, nsn;
            tile_info(itn, tn, s0n, nsn);
            const int gq = tile % L.ngroups;
            const int rb = gq * G + a;        // block-row of this thread's query row
            const int rseq = gq * 128 + row;  // query position inside the sequence
            float l = 0.f, m = -INFINITY;     // this half row's sum and the running max it is relative to
            for (int n = 0; n < ns; ++n, ++g) {
                const Half c = hnext;
                if (n + 1 < ns) {
                    fetch(s0 + n + 1, hnext);  // latency hidden behind this step
                } else if (nsn > 0) {
                    fetch(s0n, hnext);         // the next tile's first step
                }
                const uint32_t sb = g % 3, xb = g & 1;
                bool ok = mbar_wait(&s_full[sb], (g / 3) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                tc_fence_after();
                const uint32_t srow = tS + sb * 128 + lane_base;
                // a half row whose every slot is absent for all of the warp's rows
                // (the union's blocks of the other block-row, padding) has nothing
                // to load or exponentiate: its P is 0.  With one block-row per tile
                // (blocks of 128) every step's block is present.
                bool skip = false;
                if constexpr (G > 1) {
                    bool absent = true;
#pragma unroll
                    for (int ls = 0; ls < LS; ++ls) absent &= c.blk[ls] < 0;
                    skip = __all_sync(0xffffffffu, absent);
                }
                float x[64];
                float mx = -INFINITY;
                if (!skip) {
                    tmem_ld64_sync(srow + hf * 64, srow + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[64]>(x));
                    mask_half(x, c, rb, rseq);
                    mx = max64(x);
                }
                // swap half-row maxima with the other thread of the row; the arrival
                // also tells it that this half's scores are in registers, so it may
                // write its P over them
                xm[xb][wg][row] = mx;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_full[xb][quad]);
                ok = mbar_wait(&x_full[xb][quad], (g >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                tc_fence_after();
                const float mrow = fmaxf(mx, xm[xb][wg ^ 1][row]);
                // m in the scaled log2 domain (scale > 0 commutes with max); it moves
                // only when the row max grew by more than the threshold
                const float m_new = fmaxf(m, mrow * args.c2);
                const bool need = m_new > m + kRescaleThreshold;  // also true for the first finite max
                const float mnext = need ? m_new : m;
                const float msub = (mnext == -INFINITY) ? 0.f : mnext;
                uint32_t pk[32];
                float rs = 0.f;
                if (!skip) {
                    rs = exp64(x, msub, pk);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) pk[k] = 0u;
                }
                tmem_st32_sync(srow + hf * 32, pk);
                if (n > 0 && __any_sync(0xffffffffu, need)) {
                    // this half of O (scaled by m) is rescaled after P V of step g - 1
                    ok = mbar_wait(&pv_done[(g - 1) % 3], ((g - 1) / 3) & 1, ab);
                    if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                    tc_fence_after();
                    const float alpha = need ? (m == -INFINITY ? 0.f : ex2_approx(m - mnext)) : 1.f;
#pragma unroll
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t r[32];
                        const uint32_t ta = tO + lane_base + hf * (D / 2) + cc * 32;
                        tmem_ld32_sync(ta, r);
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            const float2 v = __fmul2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                                        make_float2(alpha, alpha));
                            r[k] = __float_as_uint(v.x);
                            r[k + 1] = __float_as_uint(v.y);
                        }
                        tmem_st32_sync(ta, r);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
                // this half row's sum, rebased from the previous reference to mnext
                l = (m == -INFINITY ? 0.f : l * ex2_approx(m - msub)) + rs;
                m = mnext;
            }
            // this half row's sum and its reference max -> epilogue (buffer tc % 2,
            // free once the epilogue has read the values of tile tc - 2)
            {
                const uint32_t lb = tc & 1;
                if (tc >= 2) {
                    bool ok = mbar_wait(&l_empty[lb], ((tc - 2) >> 1) & 1, ab);
                    if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                }
                lsum[lb][wg][row] = m == -INFINITY ? 0.f : l;
                lref[lb][wg][row] = m;
                __syncwarp();
                if (lane == 0) mbar_arrive(&l_full[lb]);
                ++tc;
            }
            while (nsn == 0) {  // empty tiles: nothing to compute
                ++itn;
                tile_info(itn, tn, s0n, nsn);
                if (nsn > 0) fetch(s0n, hnext);
            }
            it = itn;
            tile = tn;
            s0 = s0n;
            ns = nsn;
        }
    softmax_done:;
    }

    tc_fence_before();
    __syncthreads();
    if (abort_flag) {
        // stopped early: the copies and products issued before the stop land
        // before the CTA lets go of its shared memory and TMEM (a normal run's
        // consumers have waited for all of them already)
        if (threadIdx.x == 0) {
            mbar_drain_ring(k_full, 2, issued[0], ab);
            const uint32_t qi = issued[1] & 0x7fffffffu;
            if (!((issued[1] >> 31) && qi == 1)) mbar_drain_ring(q_full, QST, qi, ab);
            mbar_drain_ring(v_full, 2, issued[2], ab);
            if (issued[3]) mbar_drain(&s_full[(issued[3] - 1) % 3], ((issued[3] - 1) / 3) & 1, ab);
            if (issued[4]) mbar_drain(&pv_done[(issued[4] - 1) % 3], ((issued[4] - 1) / 3) & 1, ab);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <typename T, int BLK, int D, int KIND, bool GEO>
int launch_attn(const bsp_layout_s* Lh, const void* Q, const void* K, const void* V, void* O, float* lse, int Z,
                float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    const int is_bf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint64_t rows = (uint64_t)Z * Lh->H * Lh->S;
    CUtensorMap mq, mk, mv;
    int rc = make_tmap_2d(&mq, Q, is_bf16, rows, D, 128, 64, 128);
    if (!rc) rc = make_tmap_2d(&mk, K, is_bf16, rows, D, BLK, 64, 128);
    if (!rc) rc = make_tmap_2d(&mv, V, is_bf16, rows, D, BLK, 64, 128);
    CUtensorMap mo;
    if (!rc) rc = make_tmap_3d(&mo, O, is_bf16, D, Lh->S, (uint64_t)Z * Lh->H, 64, 32);
    if (rc) return rc;
    auto kern = attention_tc_kernel<T, BLK, D, KIND, GEO>;
    constexpr int smem = AttnSmem<D>::kAlloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    // the register split at kernel start needs the full launch allocation
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return BSP_ERR_CUDA;
    if ((uint32_t)fa.numRegs != kRegsLaunch) return BSP_ERR_UNSUPPORTED;
    AttnSchedule sc;
    if ((rc = attn_schedule_begin(const_cast<bsp_layout_s*>(Lh), is_bf16 ? BSP_BF16 : BSP_F16, Z, s, &sc))) return rc;
    AttnArgs args{Lh->view, O, mask, sc.ptr, sc.items, sc.part, sc.ws, lse, Z, kind, scale * kLog2e};
    if (sc.grid > 0) {
        kern<<<sc.grid, kThreads, smem, s>>>(mq, mk, mv, mo, args);
        rc = cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
    }
    return attn_schedule_end(Lh, is_bf16 ? BSP_BF16 : BSP_F16, sc, O, lse, D, s, rc);
}

template <typename T, int BLK, int KIND, bool GEO>
int by_d(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, int D, float scale,
         int kind, const uint8_t* mask, cudaStream_t s) {
    if (D == 128) return launch_attn<T, BLK, 128, KIND, GEO>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
    if (D == 64) return launch_attn<T, BLK, 64, KIND, GEO>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
    return BSP_ERR_UNSUPPORTED;
}

template <typename T, int BLK, bool GEO>
int by_kind(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, int D,
            float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    switch (kind) {
        case BSP_MASK_NONE: return by_d<T, BLK, BSP_MASK_NONE, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        case BSP_MASK_DENSE: return by_d<T, BLK, BSP_MASK_DENSE, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        case BSP_MASK_DIAG_CAUSAL:
            return by_d<T, BLK, BSP_MASK_DIAG_CAUSAL, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        default: return BSP_ERR_INVALID_ARG;
    }
}

template <typename T, bool GEO>
int by_block(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, int D,
             float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    switch (L->B) {
        case 128: return by_kind<T, 128, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        case 64: return by_kind<T, 64, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        case 32: return by_kind<T, 32, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        case 16: return by_kind<T, 16, GEO>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

}  // namespace attn
}  // namespace bsp
