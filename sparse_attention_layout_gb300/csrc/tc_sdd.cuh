// Tensor-core (tcgen05) SDD for bf16 / fp16 with fp32 accumulation: the
// sampled dense x dense product of "question on blocksparse" (openai/triton
// issue 117), evaluated on the layout's blocks only.
//
// Row tiles of 128 query rows (the attention work list); each step computes
// the 128 x 128 score tile against G = 128/B key blocks into one of four TMEM
// accumulators; eight epilogue warps write the present blocks while the MMA
// works ahead.  The kernel template and its launch helpers live here; the
// plain and softmax modes are instantiated in tc_sdd.cu, the fused softmax
// backward in tc_sdd_bwd.cu and the attention backward's one-pass mode in
// tc_sdd_attn_bwd.cu (separate translation units compile in parallel).
//
// Operand orientation: op(A) rows and op(B) columns are what the tiles hold.
// trans_a = 0 / trans_b = 1 store them as rows ([S][K]: K-major tiles, 64-column
// panels); trans_a = 1 / trans_b = 0 store them as columns ([K][S]): the tile is
// then loaded as it lies, MN-major (panels of 64 rows, or of one key block of
// 16 / 32 columns with a 32 / 64-byte swizzle), and only the shared-memory
// descriptor and the instruction's major-ness bits change.  No transpose
// happens in memory.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner and
// single-thread MMA issuer, warps 2..9 epilogue (thread = TMEM lane; warps
// 2..5 take columns 0..63 of the 128-column score tile, warps 6..9 columns
// 64..127).  The epilogue stages each present piece's rows in shared memory
// and writes them with asynchronous bulk copies, so its warps never wait on
// the global writes.  Halving each thread's columns (against four warps on
// whole rows) is what the fused modes' epilogue-bound passes need.
//
// SMX (fused SDD + row softmax): the whole key stream of a row tile is one
// CTA's, and an epilogue thread owns one query row, so the row softmax fits
// in the epilogue: every tile's steps run twice, the first pass keeping each
// row's running max and sum of 2^(scale log2(e) s - max) (masked entries
// excluded), the second recomputing the scores and writing
// P = 2^(scale log2(e) s - max) / sum instead of S.  The scores never reach
// HBM; the second pass repeats the matrix products, which cost less than the
// round trip of S they replace.
//
// SMB (fused SDD + softmax backward, for the attention backward): the product
// is dP = dO V^T, and with the softmax output P of the same layout the
// epilogue writes the gradient of the scaled scores,
//     dX = scale P .* (dP - rowsum(P .* dP)),
// the softmax backward of the chain rule.  The row sum needs the whole row,
// so the tile's steps again run twice: the first pass accumulates
// rowsum(P .* dP) (reading the thread's row of every present P block), the
// second recomputes dP and writes dX.  dP never reaches memory and stays in
// fp32; masked entries have P = 0 and so dX = 0.
//
// DUO (MODE 3, the attention backward given what the forward already knows):
// every step runs two products, S = Q K^T and dP = dO V^T, into a pair of
// TMEM accumulators (two pairs, 4 x 128 columns), and the epilogue writes
// both P = exp(scale S - lse), from the rows' log-sum-exp of the forward (no
// statistics pass), and dX = scale P .* (dP - dO_row . O_row), with
// rowsum(P .* dP) = dO_row . O_row (O = P V) taken from a vector computed
// beforehand (no accumulation pass).  P goes out from registers and is never
// read back.  The query-side tiles (Q, dO) share one stage and the key-side
// tiles (K, V) two.
#pragma once

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

namespace bsp {
namespace sddk {

using namespace tc;

constexpr int kThreads = 320;  // producer, MMA issuer, 8 epilogue warps

// ------------------------------------------------------------------ SDD ----

struct SddArgs {
    LayoutView L;
    void* C;
    int Z;
    int kd;      // contraction length K
    int ta, tb;  // trans flags (ta = 1: A tile MN-major; tb = 0: B tile MN-major)
    // fused softmax only: scale * log2(e), mask kind, dense keep-mask [S][S]
    float c2;
    int kind;
    const uint8_t* mask;
    // fused softmax backward only: the softmax output [Z][nnz][B][B] and the scale
    const void* P;
    float scale;
    // DUO: the rows' log-sum-exp [Z][H][S] (natural log) of the forward and
    // their rowsum(dO .* O) [Z][H][S]; P, written beside dX (which goes to C)
    const float* lse;
    const float* dvec;
    void* C2;
};

__host__ __device__ constexpr uint32_t swz_of(int row_bytes) {
    return row_bytes == 128 ? kSw128 : (row_bytes == 64 ? kSw64 : kSw32);
}

// MODE 2 (fused softmax backward): a key-tile stage also holds the step's P
// tile (128 query rows x 128 keys, two 128-byte-swizzled panels of 64 keys,
// copied by the producer with the V tile), and one query-tile stage and two
// key-tile stages make room for it: the product is light there, the
// epilogue is what a step waits for.
template <int KP, int BLK, int MODE>
struct SddCfg {
    static constexpr bool SMB = MODE == 2;
    static constexpr bool DUO = MODE == 3 || MODE == 4;  // two products per step
    static constexpr int kTile = 128 * 64 * KP * 2;  // 128 rows x K (KP panels of 64)
    static constexpr int AST = (SMB || DUO) ? 1 : 2;  // query-tile stages
    // key-tile stages: three, except in the backward modes (two stages of V
    // and P, or of K and V); at K = 128 the fused softmax makes room for the
    // third with one staging buffer per epilogue warp (its per-tile exchange
    // arrays take the rest)
    // MODE 4: three stages of K (held until the step's dQ product) and one of
    // V (released by dP) in the room of two (K, V) stages
    static constexpr bool DQF = MODE == 4;
    static constexpr int BST = DQF ? 3 : ((SMB || DUO) ? 2 : 3);
    static constexpr int kPT = SMB ? 32768 : 0;  // P tile of a key-tile stage
    static constexpr int kAStage = DUO ? 2 * kTile : kTile;  // Q (and dO)
    static constexpr int kBStage = (DUO && !DQF) ? 2 * kTile : kTile + kPT;  // K (and V, or P)
    static constexpr int kA = 0;
    static constexpr int kB = AST * kAStage;
    static constexpr int kV = kB + BST * kBStage;  // MODE 4: the V stage
    static constexpr int kStg = kV + (DQF ? kTile : 0);  // staging: NBUF buffers per epilogue warp
    static constexpr int NBUF = (SMB || (MODE == 1 && KP == 2) || (DUO && KP == 2)) ? 1 : 2;
    // TMEM accumulators: four of 128 columns, two pairs (S, dP), or one pair
    // plus dQ (columns 256 .. 384) and two buffers of dX as 16-bit pairs
    // (columns 384 .. 448 .. 512)
    static constexpr int NACC = MODE == 4 ? 1 : (DUO ? 2 : 4);
    static constexpr int kBuf = 32 * (BLK < 64 ? BLK : 64) * 2;  // a warp's 32 rows of one piece
    static constexpr int kAlloc = kStg + 8 * NBUF * kBuf + 1024;
};

// MODE: 0 plain SDD; 1 fused softmax (SMX, two passes); 2 fused softmax
// backward (SMB, two passes); 3 attention backward from the forward's
// statistics (DUO, one pass: A = Q, A2 = dO, B = K, B2 = V; C = dX, C2 = P);
// 4 mode 3 that also accumulates dQ = dX K (DQF; tmD: dQ, [Z H][S][D])
template <typename T, int BLK, int KP, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
sdd_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
              const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
              const __grid_constant__ CUtensorMap tmD, const SddArgs args) {
    using C = SddCfg<KP, BLK, MODE>;
    constexpr int G = 128 / BLK;
    constexpr int AST = C::AST, BST = C::BST;
    constexpr bool DUO = C::DUO;
    constexpr int NACC = C::NACC;
    constexpr bool DQF = C::DQF;
    static_assert(!DQF || (KP == 2 && BLK >= 64), "dQ fusion: D = 128, blocks of 64 and 128");
    constexpr uint32_t kAccCols = DUO ? 256 : 128;  // TMEM columns per accumulator (pair)
    constexpr uint32_t kTileBytes = C::kTile;
    // MN-major key tiles: panels of W keys (RB bytes per K row), KPB per block
    constexpr int W = BLK < 64 ? BLK : 64, RB = 2 * W, KPB = BLK / W;
    const int kd = args.kd;
    const bool a_mn = args.ta != 0, b_mn = args.tb == 0;
    // bytes one stage's copies deliver: K-major boxes are 64 * KP columns wide
    // (zero-filled past K), MN-major ones exactly K rows
    // DQF: the query-side stage's Q and dO have barriers of their own (a_*
    // for Q, do_* for dO), so that the next tile's Q loads as soon as this
    // tile's last S has read Q, not after its last dP
    const uint32_t a_bytes = (a_mn ? 256u * kd : kTileBytes) * ((DUO && !DQF) ? 2u : 1u);
    const uint32_t b_bytes = (b_mn ? 256u * kd : kTileBytes) * ((DUO && !DQF) ? 2u : 1u);
    constexpr bool SMX = MODE == 1 || DUO, SMB = MODE == 2;
    constexpr bool XCH = MODE == 1 || MODE == 2;  // two passes, row statistics exchanged between them
    constexpr int NPASS = XCH ? 2 : 1;            // passes over a tile's steps

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t a_full[AST], a_empty[AST], b_full[BST], b_empty[BST], s_full[NACC], s_empty[NACC];
    // fused modes: the two halves of every row exchange their statistics once
    // per tile (the two warps of lane quadrant q: xq[q]; values in xs)
    __shared__ uint64_t xq[4];
    __shared__ float2 xs[XCH ? 2 : 1][2][XCH ? 128 : 1];
    __shared__ uint32_t tmem_base;
    // DQF: dP of the step computed (dp_full) and read (dp_empty) -- S and dP
    // have barriers of their own, so the next step's S starts as soon as this
    // step's S is in registers; the step's dX in TMEM buffer g % 2 written by
    // the eight epilogue warps (ds_full) and read by the dQ product
    // (ds_free); the tile's dQ accumulated (dq_full) and read out (dq_empty)
    __shared__ uint64_t dp_full, dp_empty, ds_full[2], ds_free[2], dq_full, dq_empty;
    __shared__ uint64_t v_full, v_empty;  // DQF: the V stage loaded, read by dP
    __shared__ uint64_t do_full, do_empty;  // DQF: the tile's dO loaded, read by its last dP
    // after an abort: the MMA issuer's last commit, which lands once every
    // product it issued has completed
    __shared__ uint64_t mma_fin;
    __shared__ int abort_flag;
    // what the issuing threads had issued when they stopped (A tiles, B
    // steps, MMA steps, dQ steps, V tiles, dO tiles), drained after the roles
    // stop if the kernel aborted
    __shared__ uint32_t issued[6];

    const LayoutView& L = args.L;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Abort ab{&abort_flag, L.status, L.wait_ns};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 6; ++i) issued[i] = 0;
        for (int i = 0; i < AST; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < BST; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], SMB ? 9 : 1);  // SMB: the eight epilogue warps also read the stage's P
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 8);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&xq[i], 2);
        mbar_init(&dp_full, 1);
        mbar_init(&dp_empty, 8);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ds_full[i], 8);
            mbar_init(&ds_free[i], 1);
        }
        mbar_init(&dq_full, 1);
        mbar_init(&dq_empty, 8);
        mbar_init(&mma_fin, 1);
        mbar_init(&v_full, 1);
        mbar_init(&v_empty, 1);
        mbar_init(&do_full, 1);
        mbar_init(&do_empty, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;

    const int64_t total = (int64_t)args.Z * L.n_tiles;
    const int S = L.S;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if constexpr (DUO) {
                tma_prefetch_desc(&tmA2);
                tma_prefetch_desc(&tmB2);
            }
            uint32_t a_it = 0, g = 0, nv = 0, d_it = 0;  // nv, d_it: V and dO tiles issued (DQF)
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                const int4 run = tile_run_at(L, w, args.Z);
            const int tile = run.x;
                const int z = (int)((uint32_t)w % (uint32_t)args.Z);
                const int h = tile / L.ngroups, gq = tile % L.ngroups;
                const int s0 = run.y, ns = run.z;
                if (ns == 0) continue;
                const int64_t zh = (int64_t)z * L.H + h;
                const uint32_t as = a_it % AST;
                if (!mbar_wait(&a_empty[as], ((a_it / AST) & 1) ^ 1, ab)) goto producer_done;
                mbar_arrive_expect_tx(&a_full[as], a_bytes);
                if (a_mn) {
                    // [K rows][128 query columns]: two panels of 64 columns
                    for (int p = 0; p < 2; ++p)
                        tma_load_2d(smem_u32(smem + C::kA + as * C::kAStage + p * (kd * 128)), &tmA,
                                    gq * 128 + 64 * p, (int32_t)(zh * kd), &a_full[as]);
                } else {
                    for (int p = 0; p < KP; ++p) {
                        tma_load_2d(smem_u32(smem + C::kA + as * C::kAStage + p * 16384), &tmA, p * 64,
                                    (int32_t)(zh * S + gq * 128), &a_full[as]);
                        if constexpr (DUO && !DQF)  // dO beside Q
                            tma_load_2d(smem_u32(smem + C::kA + as * C::kAStage + kTileBytes + p * 16384), &tmA2,
                                        p * 64, (int32_t)(zh * S + gq * 128), &a_full[as]);
                    }
                }
                ++a_it;
                for (int it = 0; it < NPASS * ns; ++it, ++g) {
                    const int s = s0 + it % ns;
                    const uint32_t st = g % BST;
                    if (!mbar_wait(&b_empty[st], ((g / BST) & 1) ^ 1, ab)) goto producer_done;
                    uint32_t p_bytes = 0;  // SMB: the step's present P blocks
                    if constexpr (SMB) {
#pragma unroll
                        for (int ra = 0; ra < G; ++ra)
#pragma unroll
                            for (int b = 0; b < G; ++b)
                                if (L.step_blk[(s * G + ra) * G + b] >= 0) p_bytes += BLK * BLK * 2;
                    }
                    mbar_arrive_expect_tx(&b_full[st], b_bytes + p_bytes);
#pragma unroll
                    for (int b = 0; b < G; ++b) {
                        int c = L.step_col[s * G + b];
                        if (c < 0) c = L.step_col[s * G];
                        if (b_mn) {
                            // [K rows][B key columns]: KPB panels of W columns
                            for (int p = 0; p < KPB; ++p)
                                tma_load_2d(smem_u32(smem + C::kB + st * C::kBStage + (b * KPB + p) * (kd * RB)),
                                            &tmB, c * BLK + W * p, (int32_t)(zh * kd), &b_full[st]);
                        } else {
                            for (int p = 0; p < KP; ++p) {
                                tma_load_2d(smem_u32(smem + C::kB + st * C::kBStage + p * 16384 + b * BLK * 128),
                                            &tmB, p * 64, (int32_t)(zh * S + (int64_t)c * BLK), &b_full[st]);
                                if constexpr (DUO && !DQF)  // V beside K
                                    tma_load_2d(smem_u32(smem + C::kB + st * C::kBStage + kTileBytes + p * 16384 +
                                                         b * BLK * 128),
                                                &tmB2, p * 64, (int32_t)(zh * S + (int64_t)c * BLK), &b_full[st]);
                            }
                        }
                    }
                    if constexpr (DQF) {
                        if (it == 0) {
                            // the tile's dO beside Q, once the previous tile's last dP has read it
                            if (!mbar_wait(&do_empty, (d_it & 1) ^ 1, ab)) goto producer_done;
                            mbar_arrive_expect_tx(&do_full, kTileBytes);
                            for (int p = 0; p < KP; ++p)
                                tma_load_2d(smem_u32(smem + C::kA + as * C::kAStage + kTileBytes + p * 16384), &tmA2,
                                            p * 64, (int32_t)(zh * S + gq * 128), &do_full);
                            ++d_it;
                        }
                        // V into its single stage once dP of the previous step has read it
                        if (!mbar_wait(&v_empty, (g & 1) ^ 1, ab)) goto producer_done;
                        mbar_arrive_expect_tx(&v_full, kTileBytes);
                        ++nv;
#pragma unroll
                        for (int b = 0; b < G; ++b) {
                            int c = L.step_col[s * G + b];
                            if (c < 0) c = L.step_col[s * G];
                            for (int p = 0; p < KP; ++p)
                                tma_load_2d(smem_u32(smem + C::kV + p * 16384 + b * BLK * 128), &tmB2, p * 64,
                                            (int32_t)(zh * S + (int64_t)c * BLK), &v_full);
                        }
                    }
                    if constexpr (SMB) {
                        // P block (row block ra, slot b) -> rows [ra B, ra B + B) of the
                        // panel(s) of keys [b B, b B + B)
                        const uint32_t pt = smem_u32(smem + C::kB + st * C::kBStage + C::kTile);
#pragma unroll
                        for (int ra = 0; ra < G; ++ra)
#pragma unroll
                            for (int b = 0; b < G; ++b) {
                                const int blk = L.step_blk[(s * G + ra) * G + b];
                                if (blk < 0) continue;
                                const int32_t prow = (int32_t)(((int64_t)z * L.nnz + blk) * BLK);
#pragma unroll
                                for (int p = 0; p < BLK / 64; ++p)
                                    tma_load_2d(pt + (b * (BLK / 64) + p) * 16384 + ra * BLK * 128, &tmP, p * 64, prow,
                                                &b_full[st]);
                            }
                    }
                }
            }
        producer_done:
            issued[0] = a_it;
            issued[1] = g;
            issued[4] = nv;
            issued[5] = d_it;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, 128, std::is_same<T, __nv_bfloat16>::value, a_mn ? 1 : 0, b_mn ? 1 : 0);
            // 16-deep contraction steps: every K-major panel of 64 (zeros past K)
            // when both tiles are K-major, else exactly K / 16
            const int nks = (a_mn || b_mn) ? kd / 16 : KP * 4;
            uint32_t a_it = 0, g = 0;
            // DQF: dQ += dX K of step g - 1 is issued after the products of
            // step g, once the epilogue has written that step's dX into TMEM
            // buffer (g - 1) % 2 (the A operand: 8 columns of 16-bit pairs per
            // 16 keys) -- the K tile (the B operand, MN-major) still sits in
            // its stage, which the dQ product releases
            constexpr uint32_t kIdescDQ = idesc_f16(128, 128, std::is_same<T, __nv_bfloat16>::value, 0, 1);
            uint32_t nq = 0, tq = 0;  // dQ steps issued, tiles whose dQ has started
            int pend = 0;             // a dQ step pending: 0 none, else 1 | 2 (first of its tile) | 4 (last)
            uint32_t pend_st = 0;
            auto issue_dq = [&]() -> bool {
                const uint32_t db = nq & 1;  // dX buffer
                if (!mbar_wait(&ds_full[db], (nq >> 1) & 1, ab)) return false;
                if ((pend & 2) && tq > 0 && !mbar_wait(&dq_empty, (tq - 1) & 1, ab)) return false;
                tc_fence_after();
                const uint32_t dk0 = smem_u32(smem + C::kB + pend_st * C::kBStage);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {  // 16 keys per product
                    const uint64_t dk = smem_desc(dk0 + ks * 2048, 16384, 1024, kSw128);
                    mma_f16_tmem_a(tS + 256, tS + 384 + db * 64 + ks * 8, dk, kIdescDQ,
                                   ((pend & 2) && ks == 0) ? 0u : 1u);
                }
                mma_commit(&ds_free[db]);
                mma_commit(&b_empty[pend_st]);
                if (pend & 4) {
                    mma_commit(&dq_full);
                    ++tq;
                }
                ++nq;
                pend = 0;
                return true;
            };
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                const int ns = tile_run_at(L, w, args.Z).z;
                if (ns == 0) continue;
                if constexpr (DQF) {
                    // the previous tile's last dQ product before waiting for
                    // this tile's operands, so that its dQ leaves without that wait
                    if (pend && !issue_dq()) goto mma_done;
                }
                const uint32_t as = a_it % AST;
                if (!mbar_wait(&a_full[as], (a_it / AST) & 1, ab)) goto mma_done;
                for (int it = 0; it < NPASS * ns; ++it, ++g) {
                    const uint32_t sb = g % NACC, st = g % BST;  // TMEM accumulator, key-tile stage
                    if (!mbar_wait(&s_empty[sb], ((g / NACC) & 1) ^ 1, ab)) goto mma_done;
                    if (!mbar_wait(&b_full[st], (g / BST) & 1, ab)) goto mma_done;
                    tc_fence_after();
                    const uint32_t abase = smem_u32(smem + C::kA + as * C::kAStage);
                    const uint32_t bbase = smem_u32(smem + C::kB + st * C::kBStage);
                    // DUO: S = Q K^T into the pair's first 128 columns, then
                    // dP = dO V^T (the stages' second tiles) into the next 128;
                    // DQF: dP once the previous step's dP has been read
#pragma unroll
                    for (int pr = 0; pr < (DUO ? 2 : 1); ++pr) {
                        uint32_t bb0 = bbase + pr * kTileBytes;
                        if (DQF && pr == 1) {
                            mma_commit(&s_full[sb]);
                            if (it == ns - 1) mma_commit(&a_empty[as]);  // Q read by the tile's last S
                            if (it == 0 && !mbar_wait(&do_full, a_it & 1, ab)) goto mma_done;
                            if (!mbar_wait(&dp_empty, (g & 1) ^ 1, ab)) goto mma_done;
                            if (!mbar_wait(&v_full, g & 1, ab)) goto mma_done;
                            tc_fence_after();
                            bb0 = smem_u32(smem + C::kV);
                        }
                        const uint32_t ab0 = abase + pr * kTileBytes;
                        for (int ks = 0; ks < nks; ++ks) {
                            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;  // K-major step
                            const uint64_t da = a_mn ? smem_desc(ab0 + ks * 2048, kd * 128, 1024, kSw128)
                                                     : smem_desc(ab0 + off, 16, 1024, kSw128);
                            const uint64_t db = b_mn ? smem_desc(bb0 + ks * 16 * RB, kd * RB, 8 * RB, swz_of(RB))
                                                     : smem_desc(bb0 + off, 16, 1024, kSw128);
                            mma_f16(tS + sb * kAccCols + pr * 128, da, db, idesc, ks > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(DQF ? &dp_full : &s_full[sb]);
                    if constexpr (DQF) {
                        mma_commit(&v_empty);
                        if (it == ns - 1) mma_commit(&do_empty);  // dO read by the tile's last dP
                    } else {
                        if (it == NPASS * ns - 1) mma_commit(&a_empty[as]);
                    }
                    if constexpr (DQF) {
                        if (pend && !issue_dq()) goto mma_done;
                        pend = 1 | (it == 0 ? 2 : 0) | (it == ns - 1 ? 4 : 0);
                        pend_st = st;
                    } else {
                        mma_commit(&b_empty[st]);
                    }
                }
                ++a_it;
            }
            if constexpr (DQF) {
                if (pend && !issue_dq()) goto mma_done;
            }
        mma_done:
            issued[2] = g;
            issued[3] = nq;
            if (*ab.flag) {  // stopped early: every product issued lands before the roles stop
                mma_commit(&mma_fin);
                mbar_drain(&mma_fin, 0, ab);
            }
        }
    } else {
        // Epilogue: eight warps; warp w owns 32 rows of the tile (TMEM lanes of
        // quadrant q = w % 4) and one half of the 128 columns (hf = (w - 2) / 4:
        // keys [64 hf, 64 hf + 64)).  A half holds NPH pieces of CW columns:
        // whole blocks when B <= 64, one 64-column half of a block when B = 128.
        // Per present piece the warp stages its rows as the output rows they
        // become and lane 0 issues the copies: a 128-byte-swizzled tensor store
        // (32 rows x 64 columns) for blocks of 64 and 128, one contiguous bulk
        // copy of RS rows otherwise.  The fused modes keep per-half row
        // statistics through their first pass and combine the two halves of
        // every row once per tile (xq barriers, values in xs).
        constexpr int RS = BLK < 32 ? BLK : 32;
        constexpr int CW = BLK < 64 ? BLK : 64;  // columns of one piece
        constexpr int NPH = 64 / CW;             // pieces per half row
        constexpr int RBY = CW * 2;              // bytes per staged row of a piece
        constexpr int C16 = CW * 2 / 16;         // 16-byte chunks per staged row
        constexpr int kSeg = RS * CW * 2;        // one copy unit
        constexpr int NBUF = C::NBUF;
        const int quad = warp & 3, hf = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int a = row / BLK;
        const int seg = lane / RS, rin = lane % RS;
        uint8_t* stg = smem + C::kStg + (warp - 2) * NBUF * C::kBuf;
        T* Cp = reinterpret_cast<T*>(args.C);
        if (lane == 0) {
            tma_prefetch_desc(&tmC);
            if constexpr (DUO) tma_prefetch_desc(&tmP);
        }
        uint32_t g = 0, uses = 0, xc = 0;  // xc: row-statistics exchanges so far
        uint32_t tqe = 0;                  // DQF: tiles whose dQ was read out of TMEM
        for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
            const int4 run = tile_run_at(L, w, args.Z);
            const int tile = run.x;
            const int z = (int)((uint32_t)w % (uint32_t)args.Z);
            const int s0 = run.y, ns = run.z;
            // fused softmax: this half row's running max (scaled log2 domain) and
            // sum, then the row's; fused softmax backward: rowsum(P .* dP)
            const int gq = tile % L.ngroups, rb = gq * G + a, r_in = row % BLK;
            float m = -INFINITY, l = 0.f, msub = 0.f, inv = 0.f;
            float dsum = 0.f;
            if constexpr (DUO) {
                // this row's place in [Z][H][S]; rows past the sequence end are
                // never written.  P = 2^(c s - lse / ln 2): a row with nothing
                // kept (lse = -inf) has every score masked and gets 0;
                // rowsum(P .* dP) = dO_row . O_row, computed beforehand
                const int rseq = gq * 128 + row;
                const int64_t rg = ((int64_t)z * L.H + tile / L.ngroups) * S + rseq;
                const float lse2 = rseq < S ? args.lse[rg] * kLog2e : -INFINITY;
                msub = lse2 == -INFINITY ? 0.f : lse2;
                inv = lse2 == -INFINITY ? 0.f : 1.f;
                dsum = rseq < S ? args.dvec[rg] : 0.f;
            }
            // the pieces of a step (block id of (row block a, slot), the slot's
            // block-column), loaded a step ahead so that their latency passes
            // under the wait for the accumulator
            int nblk[NPH], ncol[NPH];
            auto fetch = [&](int s) {
#pragma unroll
                for (int p = 0; p < NPH; ++p) {
                    const int b = (64 * hf + p * CW) / BLK;
                    nblk[p] = L.step_blk[(s * G + a) * G + b];
                    if constexpr (SMX) ncol[p] = L.step_col[s * G + b];
                    else ncol[p] = 0;
                }
            };
            if (ns > 0) fetch(s0);
            // DQF: this warp's 32 rows x 64 columns of the tile's dQ (zeros for
            // a tile without steps) out through its staging buffer
            const int64_t zh = (int64_t)z * L.H + tile / L.ngroups;
            auto dq_out = [&](bool acc) -> bool {
                uint32_t q[32];
                if (acc) {
                    const bool ok = mbar_wait(&dq_full, tqe & 1, ab);
                    if (!__all_sync(0xffffffffu, ok)) return false;
                    tc_fence_after();
                    uint32_t r[64];
                    tmem_ld64_sync(tS + 256 + lane_base + 64 * hf, tS + 256 + lane_base + 64 * hf + 32, r);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dq_empty);
                    ++tqe;
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        q[k] = Pack2<T>::pack(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) q[k] = 0u;
                }
                const int y0 = gq * 128 + quad * 32;
                if (y0 >= S) return true;  // rows past the sequence end
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                uint8_t* rp = stg + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(rp + ((j ^ (lane & 7)) << 4)) =
                        make_uint4(q[4 * j], q[4 * j + 1], q[4 * j + 2], q[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&tmD, smem_u32(stg), 64 * hf, y0, (int32_t)zh);
                    bulk_commit();
                }
                ++uses;
                return true;
            };
            if constexpr (DQF) {
                if (ns == 0) {
                    if (!dq_out(false)) goto epi_done;
                    continue;
                }
            }
            for (int it = 0; it < NPASS * ns; ++it, ++g) {
                const bool write = !XCH || it >= ns;  // the pass that writes
                int pblk[NPH], pcol[NPH];
#pragma unroll
                for (int p = 0; p < NPH; ++p) {
                    pblk[p] = nblk[p];
                    pcol[p] = ncol[p];
                }
                if (it + 1 < NPASS * ns) fetch(s0 + (it + 1) % ns);
                const uint32_t sb = g % NACC;
                bool ok = mbar_wait(&s_full[sb], (g / NACC) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                tc_fence_after();
                const uint32_t tacc = tS + sb * kAccCols + lane_base + 64 * hf;
                uint32_t x[64];
                tmem_ld32_sync(tacc, *reinterpret_cast<uint32_t(*)[32]>(x));
                tmem_ld32_sync(tacc + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
                if constexpr (!DUO || DQF) {
                    // the accumulator is free once both halves are in registers
                    // (DUO: once dP is in registers too, below; DQF: S has a
                    // barrier of its own)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_empty[sb]);
                }
                float* xf = reinterpret_cast<float*>(x);
                if constexpr (SMB) {
                    // this half row of the stage's P tile (panel hf; the copies
                    // landed: wait on the stage's full barrier), zeros for absent
                    // pieces; then the stage is released by this warp
                    const uint32_t st = g % BST;
                    ok = mbar_wait(&b_full[st], (g / BST) & 1, ab);
                    if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                    uint32_t pv[32];
                    const uint8_t* pb = smem + C::kB + st * C::kBStage + C::kTile + hf * 16384 + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const bool present = pblk[(c * 8) / CW] >= 0;
                        const uint4 v = present ? *reinterpret_cast<const uint4*>(pb + ((c ^ (row & 7)) << 4))
                                                : make_uint4(0u, 0u, 0u, 0u);
                        pv[4 * c + 0] = v.x;
                        pv[4 * c + 1] = v.y;
                        pv[4 * c + 2] = v.z;
                        pv[4 * c + 3] = v.w;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&b_empty[st]);
                    if (!write) {
                        // first pass: this half's rowsum(P .* dP); at the tile's last
                        // step the two halves of the row are added
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float2 pf = Unpack2<T>::unpack(pv[j]);
                            dsum = fmaf(pf.x, xf[2 * j], dsum);
                            dsum = fmaf(pf.y, xf[2 * j + 1], dsum);
                        }
                        if (it == ns - 1) {
                            xs[xc & 1][hf][row] = make_float2(dsum, 0.f);
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&xq[quad]);
                            ok = mbar_wait(&xq[quad], xc & 1, ab);
                            if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                            dsum += xs[xc & 1][hf ^ 1][row].x;
                            ++xc;
                        }
                        continue;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float2 pf = Unpack2<T>::unpack(pv[j]);
                        xf[2 * j] = args.scale * pf.x * (xf[2 * j] - dsum);
                        xf[2 * j + 1] = args.scale * pf.y * (xf[2 * j + 1] - dsum);
                    }
                }
                if constexpr (SMX) {
                    // masked entries -> -inf: absent pieces, columns past the
                    // diagonal inside diagonal blocks, dense-mask zeros
#pragma unroll
                    for (int p = 0; p < NPH; ++p) {
                        const int co = (64 * hf + p * CW) % BLK;
                        const int blk = pblk[p];
                        const int col = pcol[p];
                        // in-piece column j is kept iff j <= lim
                        const int lim =
                            blk < 0 ? -1 : ((args.kind == BSP_MASK_DIAG_CAUSAL && col == rb) ? r_in - co : CW);
                        if (__any_sync(0xffffffffu, lim < CW - 1)) {
#pragma unroll
                            for (int j = 0; j < CW; ++j) xf[p * CW + j] = j > lim ? -INFINITY : xf[p * CW + j];
                        }
                        if (args.kind == BSP_MASK_DENSE && blk >= 0) {
                            const uint8_t* mp = args.mask + (int64_t)(gq * 128 + row) * S + (int64_t)col * BLK + co;
#pragma unroll
                            for (int q = 0; q < CW / 16; ++q) {
                                const uint4 mv = *reinterpret_cast<const uint4*>(mp + q * 16);
                                const uint8_t* mb = reinterpret_cast<const uint8_t*>(&mv);
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    if (!mb[k]) xf[p * CW + q * 16 + k] = -INFINITY;
                            }
                        }
                    }
                    if (!write) {
                        // first pass: this half row's running max and sum; at the
                        // tile's last step the halves of the row are combined
                        float mx = -INFINITY;
#pragma unroll
                        for (int j = 0; j < 64; ++j) mx = fmaxf(mx, xf[j]);
                        const float mn = fmaxf(m, mx * args.c2);
                        if (mn != -INFINITY) {
                            float acc = 0.f;
#pragma unroll
                            for (int j = 0; j < 64; ++j) acc += ex2_approx(fmaf(xf[j], args.c2, -mn));
                            l = (m == -INFINITY ? 0.f : l * ex2_approx(m - mn)) + acc;
                            m = mn;
                        }
                        if (it == ns - 1) {
                            xs[xc & 1][hf][row] = make_float2(m, l);
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&xq[quad]);
                            ok = mbar_wait(&xq[quad], xc & 1, ab);
                            if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                            const float2 o = xs[xc & 1][hf ^ 1][row];
                            const float mr = fmaxf(m, o.x);
                            const float lr = mr == -INFINITY ? 0.f
                                                             : (m == -INFINITY ? 0.f : l * ex2_approx(m - mr)) +
                                                                   (o.x == -INFINITY ? 0.f : o.y * ex2_approx(o.x - mr));
                            msub = mr == -INFINITY ? 0.f : mr;
                            inv = lr > 0.f ? 1.0f / lr : 0.f;
                            ++xc;
                        }
                        continue;
                    }
#pragma unroll
                    for (int j = 0; j < 64; ++j) xf[j] = ex2_approx(fmaf(xf[j], args.c2, -msub)) * inv;
                }

                // stage this warp's rows of every present piece of v (pairs of
                // 16-bit values) and copy them to the output rows of map (base:
                // the same rows, for the contiguous copies of blocks under 64)
                auto store = [&](const uint32_t (&v)[32], const CUtensorMap* map, T* base) {
#pragma unroll
                    for (int p = 0; p < NPH; ++p) {
                        const int blk = pblk[p];
                        if (__all_sync(0xffffffffu, blk < 0)) continue;
                        int sblk[32 / RS];
#pragma unroll
                        for (int sg = 0; sg < 32 / RS; ++sg) sblk[sg] = __shfl_sync(0xffffffffu, blk, sg * RS);
                        uint8_t* buf = stg + (uses % NBUF) * C::kBuf;
                        if (lane == 0) {  // the copy that last read this buffer has read it
                            if constexpr (NBUF == 2) bulk_wait_read<1>();
                            else bulk_wait_read<0>();
                        }
                        __syncwarp();
                        if (blk >= 0) {
                            uint8_t* rbase = buf + seg * kSeg + rin * RBY;
#pragma unroll
                            for (int j = 0; j < C16; ++j) {
                                const int o = (p * CW + 8 * j) / 2;
                                const int pos = CW == 64 ? (j ^ (rin & 7)) : j;
                                *reinterpret_cast<uint4*>(rbase + pos * 16) =
                                    make_uint4(v[o], v[o + 1], v[o + 2], v[o + 3]);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
#pragma unroll
                            for (int sg = 0; sg < 32 / RS; ++sg) {
                                if (sblk[sg] < 0) continue;
                                const int r_in0 = (quad * 32 + sg * RS) % BLK;
                                const int64_t orow = ((int64_t)z * L.nnz + sblk[sg]) * BLK + r_in0;
                                if (BLK >= 64)
                                    tma_store_3d(map, smem_u32(buf + sg * kSeg), (64 * hf + p * CW) % BLK,
                                                 (int32_t)orow, 0);
                                else
                                    bulk_store(base + orow * BLK, smem_u32(buf + sg * kSeg), kSeg);
                            }
                            bulk_commit();
                        }
                        ++uses;
                    }
                };
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) pk[j] = Pack2<T>::pack(xf[2 * j], xf[2 * j + 1]);
                if constexpr (DUO) {
                    // P out first; then this half row of dP, which frees the
                    // accumulator pair, and dX = scale P .* (dP - dO_row . O_row)
                    // from the rounded P (0 where masked)
                    store(pk, &tmP, reinterpret_cast<T*>(args.C2));
                    if constexpr (DQF) {
                        ok = mbar_wait(&dp_full, g & 1, ab);
                        if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                        tc_fence_after();
                    }
                    uint32_t y[64];
                    tmem_ld32_sync(tacc + 128, *reinterpret_cast<uint32_t(*)[32]>(y));
                    tmem_ld32_sync(tacc + 160, *reinterpret_cast<uint32_t(*)[32]>(y + 32));
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(DQF ? &dp_empty : &s_empty[sb]);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float2 pf = Unpack2<T>::unpack(pk[j]);
                        pk[j] = Pack2<T>::pack(args.scale * pf.x * (__uint_as_float(y[2 * j]) - dsum),
                                               args.scale * pf.y * (__uint_as_float(y[2 * j + 1]) - dsum));
                    }
                    if constexpr (DQF) {
                        // this half row of dX into TMEM buffer g % 2 (keys 64 hf ..
                        // 64 hf + 63 as 32 columns of pairs), once the dQ product
                        // of step g - 2 has read the buffer
                        const uint32_t db = g & 1;
                        ok = mbar_wait(&ds_free[db], ((g >> 1) & 1) ^ 1, ab);
                        if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                        tc_fence_after();
                        tmem_st32_sync(tS + 384 + db * 64 + lane_base + 32 * hf, pk);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ds_full[db]);
                    }
                }
                store(pk, &tmC, Cp);
                if constexpr (DQF) {
                    if (it == ns - 1 && !dq_out(true)) goto epi_done;
                }
            }
        }
    epi_done:
        if (lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag) {
        // stopped early: the copies and products issued before the stop land
        // before the CTA lets go of its shared memory and TMEM
        if (threadIdx.x == 0) {
            mbar_drain_ring(a_full, AST, issued[0], ab);
            mbar_drain_ring(b_full, BST, issued[1], ab);
            if (issued[4]) mbar_drain(&v_full, (issued[4] - 1) & 1, ab);
            if (issued[5]) mbar_drain(&do_full, (issued[5] - 1) & 1, ab);
            if (issued[2]) mbar_drain(&s_full[(issued[2] - 1) % NACC], ((issued[2] - 1) / NACC) & 1, ab);
            if (issued[3]) mbar_drain(&ds_free[(issued[3] - 1) & 1], ((issued[3] - 1) >> 1) & 1, ab);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// --------------------------------------------------------------- launch ----

// what the fused modes read besides the two operands
struct SddExtra {
    float c2 = 0.f;                 // scale * log2(e) (softmax modes)
    int kind = 0;                   // mask kind (softmax modes)
    const uint8_t* mask = nullptr;  // dense keep-mask (softmax modes)
    const void* P = nullptr;        // softmax output (backward modes)
    float scale = 0.f;              // softmax scale (backward modes)
    const float* lse = nullptr;     // DUO: the forward's log-sum-exp
    const float* dvec = nullptr;    // DUO: rowsum(dO .* O)
    const void* A2 = nullptr;       // DUO: dO (A is Q)
    const void* B2 = nullptr;       // DUO: V (B is K)
    void* C2 = nullptr;             // DUO: P (C is dX)
    void* D2 = nullptr;             // MODE 4: dQ [Z][H][S][K]
};

template <typename T, int BLK, int KP, int MODE>
int sdd_launch(const bsp_layout_s* Lh, const void* A, const void* B, void* Cout, int Z, int K, int ta, int tb,
               const SddExtra& e, cudaStream_t s) {
    const int bf = std::is_same<T, __nv_bfloat16>::value;
    const uint64_t ZH = (uint64_t)Z * Lh->H, rows = ZH * Lh->S;
    constexpr bool DUO = SddCfg<KP, BLK, MODE>::DUO;
    constexpr int W = BLK < 64 ? BLK : 64;
    CUtensorMap ma, mb, mc, mp, ma2, mb2, md;
    // [S][K] operands: boxes of 128 (A) or B (B) rows x 64 columns; [K][S]
    // operands: boxes of K rows x 64 (A) or W (B) columns
    int rc = ta ? make_tmap_2d(&ma, A, bf, ZH * K, Lh->S, K, 64, 128) : make_tmap_2d(&ma, A, bf, rows, K, 128, 64, 128);
    if (!rc)
        rc = tb ? make_tmap_2d(&mb, B, bf, rows, K, BLK, 64, 128) : make_tmap_2d(&mb, B, bf, ZH * K, Lh->S, K, W, 2 * W);
    // output rows: [Z * nnz * B][B], boxes of min(32, B) rows x W columns
    // (128-byte swizzle for W = 64)
    if (!rc)
        rc = make_tmap_3d(&mc, Cout, bf, BLK, (uint64_t)Z * Lh->nnz * BLK, 1, W, BLK < 32 ? BLK : 32,
                          BLK >= 64 ? 128 : 0);
    // fused softmax backward: P rows [Z * nnz * B][B], boxes of B rows x 64
    // columns, 128-byte swizzle (the other modes never read this map)
    if (!rc) {
        if constexpr (MODE == 2)
            rc = make_tmap_2d(&mp, e.P, bf, (uint64_t)Z * Lh->nnz * BLK, BLK, BLK, 64, 128);
        else if constexpr (DUO)  // P is written like C
            rc = make_tmap_3d(&mp, e.C2, bf, BLK, (uint64_t)Z * Lh->nnz * BLK, 1, W, BLK < 32 ? BLK : 32,
                              BLK >= 64 ? 128 : 0);
        else mp = mc;
    }
    // DUO: dO and V, [S][K] like Q and K
    if (!rc) {
        if constexpr (DUO) {
            rc = make_tmap_2d(&ma2, e.A2, bf, rows, K, 128, 64, 128);
            if (!rc) rc = make_tmap_2d(&mb2, e.B2, bf, rows, K, BLK, 64, 128);
        } else {
            ma2 = ma;
            mb2 = mb;
        }
    }
    // MODE 4: dQ rows [Z * H][S][K], boxes of 32 rows x 64 columns (rows past
    // the sequence end clipped)
    if (!rc) {
        if constexpr (MODE == 4) rc = make_tmap_3d(&md, e.D2, bf, K, Lh->S, ZH, 64, 32);
        else md = mc;
    }
    if (rc) return rc;
    SddArgs a{Lh->view, Cout, Z, K, ta, tb, e.c2, e.kind, e.mask, e.P, e.scale, e.lse, e.dvec, e.C2};
    auto kern = sdd_tc_kernel<T, BLK, KP, MODE>;
    constexpr int smem = SddCfg<KP, BLK, MODE>::kAlloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    const int64_t total = (int64_t)Z * Lh->n_tiles;
    const int grid = (int)std::min<int64_t>(total, sm_count());
    kern<<<grid, kThreads, smem, s>>>(ma, mb, mc, mp, ma2, mb2, md, a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T, int BLK, int MODE>
int sdd_by_k(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int K, int ta, int tb,
             const SddExtra& e, cudaStream_t s) {
    if constexpr (MODE == 4) {  // dQ fused: one 128-column accumulator and D = 128 panels
        if (K != 128) return BSP_ERR_UNSUPPORTED;
    } else {
        if (K <= 64) return sdd_launch<T, BLK, 1, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
    }
    return sdd_launch<T, BLK, 2, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
}

// the fused softmax backward reads P in 64-key panels, and the dQ-fused mode
// stages dX in them: blocks of 64 and 128 only
template <typename T, int MODE>
int sdd_by_block(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int K, int ta, int tb,
                 const SddExtra& e, cudaStream_t s) {
    constexpr bool small_ok = MODE != 2 && MODE != 4;
    switch (L->B) {
        case 16:
            if constexpr (small_ok) return sdd_by_k<T, 16, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
            return BSP_ERR_UNSUPPORTED;
        case 32:
            if constexpr (small_ok) return sdd_by_k<T, 32, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
            return BSP_ERR_UNSUPPORTED;
        case 64: return sdd_by_k<T, 64, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
        case 128: return sdd_by_k<T, 128, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

template <int MODE>
int sdd_by_dtype(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int K, int ta,
                 int tb, const SddExtra& e, cudaStream_t s) {
    if (dtype == BSP_BF16) return sdd_by_block<__nv_bfloat16, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
    if (dtype == BSP_F16) return sdd_by_block<__half, MODE>(L, A, B, C, Z, K, ta, tb, e, s);
    return BSP_ERR_UNSUPPORTED;
}

// shapes the tensor-core SDD covers: K at most 128 (one shared-memory tile);
// both operands [S][K]: K a multiple of 8 (the row pitch of a TMA map is a
// multiple of 16 bytes); an operand stored [K][S]: K a multiple of 16 (its
// tile has exactly K rows)
inline bool sdd_tc_shape(const bsp_layout_s* L, int Z, int K, int ta, int tb) {
    if (K > 128 || K % 8 != 0 || ((ta || !tb) && K % 16 != 0)) return false;
    return (uint64_t)Z * L->H * std::max(L->S, K) < (1ull << 31);
}

}  // namespace sddk
}  // namespace bsp
