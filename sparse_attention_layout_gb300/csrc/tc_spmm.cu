// Tensor-core (tcgen05) SDD, DSD and DDS for bf16 / fp16 with fp32
// accumulation.  Operations of "question on blocksparse" (openai/triton issue
// 117): SDD samples a dense x dense product on the layout's blocks; DSD is
// sparse (lhs) x dense; DDS is dense x sparse (rhs).
//
// DSD / DDS kernel: one work item = one block-row (DSD) or block-column (DDS)
// of the sparse operand x one 128-wide tile of the dense operand's free
// dimension x one batch entry.  Each step contracts one present B x B block:
//     acc[128 x B] += Dense[128 x B] * Block^T[B x B]
// with the dense tile as the MMA's M = 128 operand and the block as N = B, so
// small blocks cost no padding.  TMEM lane = dense index (n for DSD, m for
// DDS), TMEM column = index inside the block.  Operand majorness follows the
// trans flags (a K-major or MN-major shared-memory descriptor; no transposes
// in memory).  Rows of the sparse operand with no block write zeros.
//
// SDD kernel: row tiles of 128 query rows (the attention work list); each
// step computes the 128 x 128 score tile against G key blocks into one of four
// TMEM accumulators; four epilogue warps write the present blocks while the
// MMA works ahead.
//
// Roles in both kernels (192 threads): warp 0 TMA producer, warp 1 TMEM owner
// and single-thread MMA issuer, warps 2..5 epilogue (thread = TMEM lane).
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

namespace bsp {
namespace {

using namespace tc;

constexpr int kThreads = 192;

__host__ __device__ constexpr int swz_code(int row_bytes) {
    return row_bytes == 128 ? kSw128 : (row_bytes == 64 ? kSw64 : kSw32);
}

// ------------------------------------------------------------ DSD / DDS ----

struct SpmmArgs {
    LayoutView L;
    void* C;
    const int32_t* ptr;    // CSR or CSC starts of the sparse operand's lines
    const int32_t* idx;    // contraction block index of each entry
    const int32_t* bid;    // block id of each entry
    const int32_t* order;  // line keys h*nb+u, longest first
    int Z;
    int is_dds;
    int ext;               // free dimension of the dense operand: N (DSD) or M (DDS)
    int ntiles;            // ceil(ext / 128)
    int dense_mn;          // dense tile is MN-major (else K-major)
    int sparse_mn;         // block is MN-major (else K-major)
};

template <int BLK>
struct SpmmCfg {
    static constexpr int W = BLK < 64 ? BLK : 64;       // elements per smem row of a K-major panel
    static constexpr int RB = W * 2;                    // bytes per such row (= swizzle span)
    static constexpr int kDense = 128 * BLK * 2;        // dense tile bytes
    static constexpr int kSparse = BLK * BLK * 2;       // block bytes
    static constexpr int kSlot = ((kDense + kSparse + 1023) / 1024) * 1024;  // one block's operands
    // blocks per pipeline stage: one barrier wait and one commit per stage, so
    // small blocks are batched (the per-step overhead dwarfs a 32-wide MMA)
    static constexpr int KB = (81920 / kSlot) < 1 ? 1 : ((81920 / kSlot) > 8 ? 8 : (81920 / kSlot));
    static constexpr int kStage = KB * kSlot;
    static constexpr int ST = (196608 / kStage) > 4 ? 4 : (196608 / kStage);
    static constexpr int kAlloc = ST * kStage + 1024;
};

template <typename T, int BLK>
__global__ void __launch_bounds__(kThreads, 1)
spmm_tc_kernel(const __grid_constant__ CUtensorMap tmDense, const __grid_constant__ CUtensorMap tmSparse,
               const SpmmArgs args) {
    using C = SpmmCfg<BLK>;
    constexpr int ST = C::ST;
    constexpr int W = C::W, RB = C::RB;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[ST], empty[ST], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const LayoutView& L = args.L;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Abort ab{&abort_flag, L.status};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < ST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tacc = tmem_base;

    const int64_t per_line = (int64_t)args.Z * args.ntiles;
    const int64_t total = (int64_t)L.H * L.nb * per_line;
    const int S = L.S, nb = L.nb;

    auto item = [&](int64_t w, int& h, int& u, int& z, int& t, int& q0, int& q1) {
        const int key = args.order[w / per_line];
        const int rem = (int)(w % per_line);
        z = rem / args.ntiles;
        t = rem % args.ntiles;
        h = key / nb;
        u = key % nb;
        q0 = args.ptr[h * (nb + 1) + u];
        q1 = args.ptr[h * (nb + 1) + u + 1];
    };

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmDense);
            tma_prefetch_desc(&tmSparse);
            uint32_t it = 0;  // stage uses
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                int h, u, z, t, q0, q1;
                item(w, h, u, z, t, q0, q1);
                const int64_t zh = (int64_t)z * L.H + h;
                const int e0 = t * 128;
                for (int c0 = q0; c0 < q1; c0 += C::KB, ++it) {
                    const int nblk = min(C::KB, q1 - c0);
                    const int st = it % ST;
                    if (!mbar_wait(&empty[st], ((it / ST) & 1) ^ 1, ab)) goto producer_done;
                    mbar_arrive_expect_tx(&full[st], nblk * (C::kDense + C::kSparse));
                    for (int sl = 0; sl < nblk; ++sl) {
                        const int q = c0 + sl;
                        uint8_t* dd = smem + st * C::kStage + sl * C::kSlot;
                        uint8_t* sp = dd + C::kDense;
                        const int kb = args.idx[q] * BLK;  // first contraction index of this block
                        if (args.dense_mn) {
                            // rows = contraction index, columns = dense free index
                            for (int p = 0; p < 2; ++p)
                                tma_load_2d(smem_u32(dd + p * (BLK * 128)), &tmDense, e0 + 64 * p,
                                            (int32_t)(zh * S + kb), &full[st]);
                        } else {
                            // rows = dense free index, columns = contraction index
                            for (int p = 0; p < BLK / W; ++p)
                                tma_load_2d(smem_u32(dd + p * (128 * RB)), &tmDense, kb + W * p,
                                            (int32_t)(zh * args.ext + e0), &full[st]);
                        }
                        const int64_t yb = ((int64_t)z * L.nnz + args.bid[q]) * BLK;
                        for (int p = 0; p < BLK / W; ++p)
                            tma_load_2d(smem_u32(sp + p * (BLK * RB)), &tmSparse, W * p, (int32_t)yb, &full[st]);
                    }
                }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, BLK, kBf16, args.dense_mn, args.sparse_mn);
            // descriptors of stage 0, slot 0; per K-step / slot / stage offsets are added
            // to the start-address field (shared addresses stay below 2^18: no carry)
            const uint32_t s0 = smem_u32(smem);
            const uint64_t dA = args.dense_mn ? smem_desc(s0, BLK * 128, 1024, kSw128)
                                              : smem_desc(s0, 16, 8 * RB, swz_code(RB));
            const uint64_t dB = args.sparse_mn ? smem_desc(s0 + C::kDense, BLK * RB, 8 * RB, swz_code(RB))
                                               : smem_desc(s0 + C::kDense, 16, 8 * RB, swz_code(RB));
            uint32_t offA[BLK / 16], offB[BLK / 16];
#pragma unroll
            for (int ks = 0; ks < BLK / 16; ++ks) {
                offA[ks] = (args.dense_mn ? ks * 16 * 128 : (16 * ks / W) * (128 * RB) + (16 * ks % W) * 2) >> 4;
                offB[ks] = (args.sparse_mn ? ks * 16 * RB : (16 * ks / W) * (BLK * RB) + (16 * ks % W) * 2) >> 4;
            }
            uint32_t it = 0, k = 0;
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                int h, u, z, t, q0, q1;
                item(w, h, u, z, t, q0, q1);
                if (q1 == q0) continue;
                const uint32_t buf = k & 1;
                if (!mbar_wait(&acc_empty[buf], ((k >> 1) & 1) ^ 1, ab)) goto mma_done;
                tc_fence_after();
                for (int c0 = q0; c0 < q1; c0 += C::KB, ++it) {
                    const int nblk = min(C::KB, q1 - c0);
                    const int st = it % ST;
                    if (!mbar_wait(&full[st], (it / ST) & 1, ab)) goto mma_done;
                    tc_fence_after();
                    for (int sl = 0; sl < nblk; ++sl) {
                        const uint32_t so = (uint32_t)(st * C::kStage + sl * C::kSlot) >> 4;
#pragma unroll
                        for (int ks = 0; ks < BLK / 16; ++ks)
                            mma_f16(tacc + buf * 128, dA + so + offA[ks], dB + so + offB[ks], idesc,
                                    (c0 > q0 || sl > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[st]);
                }
                mma_commit(&acc_full[buf]);
                ++k;
            }
        mma_done:;
        }
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint32_t k = 0;
        T* Cp = reinterpret_cast<T*>(args.C);
        for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
            int h, u, z, t, q0, q1;
            item(w, h, u, z, t, q0, q1);
            const int64_t zh = (int64_t)z * L.H + h;
            const int e = t * 128 + row;  // dense free index of this lane
            float v[BLK];
            const bool has = q1 > q0;
            const uint32_t buf = k & 1;
            if (has) {
                bool ok = mbar_wait(&acc_full[buf], (k >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                tc_fence_after();
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < (BLK + 31) / 32; ++c) {
                    tmem_ld32_sync(tacc + buf * 128 + lane_base + c * 32, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c * 32 + j < BLK) v[c * 32 + j] = __uint_as_float(r[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
                ++k;
            } else {
#pragma unroll
                for (int j = 0; j < BLK; ++j) v[j] = 0.f;
            }
            if (e < args.ext) {
                if (!args.is_dds) {
                    // C[zh][u*BLK + j][e]: lanes write consecutive e
                    T* dst = Cp + (zh * S + (int64_t)u * BLK) * args.ext + e;
#pragma unroll
                    for (int j = 0; j < BLK; ++j) dst[(int64_t)j * args.ext] = from_f32<T>(v[j]);
                } else {
                    // C[zh][e][u*BLK + j]: contiguous in j
                    T* dst = Cp + (zh * args.ext + e) * (int64_t)S + (int64_t)u * BLK;
#pragma unroll
                    for (int j = 0; j < BLK; j += 8) {
                        uint4 pk;
                        pk.x = Pack2<T>::pack(v[j], v[j + 1]);
                        pk.y = Pack2<T>::pack(v[j + 2], v[j + 3]);
                        pk.z = Pack2<T>::pack(v[j + 4], v[j + 5]);
                        pk.w = Pack2<T>::pack(v[j + 6], v[j + 7]);
                        *reinterpret_cast<uint4*>(dst + j) = pk;
                    }
                }
            }
        }
    epi_done:;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 256);
    }
}

// ------------------------------------------------------------------ SDD ----

struct SddArgs {
    LayoutView L;
    void* C;
    int Z;
};

template <int KP, int BLK>
struct SddCfg {
    static constexpr int kTile = 128 * 64 * KP * 2;  // 128 rows x K (KP panels of 64)
    static constexpr int BST = 3;                    // key-tile stages
    static constexpr int kA = 0;                     // 2 query-tile stages
    static constexpr int kB = 2 * kTile;
    static constexpr int kPitch = BLK * 2 + 16;      // staging row pitch (padded: no bank conflicts)
    static constexpr int kStg = kB + BST * kTile;    // per-warp staging, 32 rows
    static constexpr int kAlloc = kStg + 4 * 32 * kPitch + 1024;
};

template <typename T, int BLK, int KP>
__global__ void __launch_bounds__(kThreads, 1)
sdd_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const SddArgs args) {
    using C = SddCfg<KP, BLK>;
    constexpr int G = 128 / BLK;
    constexpr int BST = C::BST;
    constexpr uint32_t kTileBytes = C::kTile;
    constexpr uint32_t kIdesc = idesc_f16(128, 128, std::is_same<T, __nv_bfloat16>::value, 0, 0);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t a_full[2], a_empty[2], b_full[BST], b_empty[BST], s_full[4], s_empty[4];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const LayoutView& L = args.L;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Abort ab{&abort_flag, L.status};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < BST; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
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
    const uint32_t tS = tmem_base;

    const int64_t total = (int64_t)args.Z * L.n_tiles;
    const int S = L.S;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            uint32_t a_it = 0, g = 0;
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                const int tile = L.tile_order[w / args.Z];
                const int z = (int)(w % args.Z);
                const int h = tile / L.ngroups, gq = tile % L.ngroups;
                const int s0 = L.tile_step_ptr[tile], ns = L.tile_step_ptr[tile + 1] - s0;
                if (ns == 0) continue;
                const int64_t zh = (int64_t)z * L.H + h;
                const uint32_t as = a_it & 1;
                if (!mbar_wait(&a_empty[as], ((a_it >> 1) & 1) ^ 1, ab)) goto producer_done;
                mbar_arrive_expect_tx(&a_full[as], kTileBytes);
                for (int p = 0; p < KP; ++p)
                    tma_load_2d(smem_u32(smem + C::kA + as * kTileBytes + p * 16384), &tmA, p * 64,
                                (int32_t)(zh * S + gq * 128), &a_full[as]);
                ++a_it;
                for (int n = 0; n < ns; ++n, ++g) {
                    const int s = s0 + n;
                    const uint32_t st = g % BST;
                    if (!mbar_wait(&b_empty[st], ((g / BST) & 1) ^ 1, ab)) goto producer_done;
                    mbar_arrive_expect_tx(&b_full[st], kTileBytes);
#pragma unroll
                    for (int b = 0; b < G; ++b) {
                        int c = L.step_col[s * G + b];
                        if (c < 0) c = L.step_col[s * G];
                        for (int p = 0; p < KP; ++p)
                            tma_load_2d(smem_u32(smem + C::kB + st * kTileBytes + p * 16384 + b * BLK * 128), &tmB,
                                        p * 64, (int32_t)(zh * S + (int64_t)c * BLK), &b_full[st]);
                    }
                }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t a_it = 0, g = 0;
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                const int tile = L.tile_order[w / args.Z];
                const int ns = L.tile_step_ptr[tile + 1] - L.tile_step_ptr[tile];
                if (ns == 0) continue;
                const uint32_t as = a_it & 1;
                if (!mbar_wait(&a_full[as], (a_it >> 1) & 1, ab)) goto mma_done;
                for (int n = 0; n < ns; ++n, ++g) {
                    const uint32_t sb = g & 3, st = g % BST;  // TMEM accumulator, key-tile stage
                    if (!mbar_wait(&s_empty[sb], ((g >> 2) & 1) ^ 1, ab)) goto mma_done;
                    if (!mbar_wait(&b_full[st], (g / BST) & 1, ab)) goto mma_done;
                    tc_fence_after();
                    const uint32_t abase = smem_u32(smem + C::kA + as * kTileBytes);
                    const uint32_t bbase = smem_u32(smem + C::kB + st * kTileBytes);
#pragma unroll
                    for (int ks = 0; ks < KP * 4; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_f16(tS + sb * 128, smem_desc(abase + off, 16, 1024, kSw128),
                                smem_desc(bbase + off, 16, 1024, kSw128), kIdesc, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&s_full[sb]);
                    mma_commit(&b_empty[st]);
                    if (n == ns - 1) mma_commit(&a_empty[as]);
                }
                ++a_it;
            }
        mma_done:;
        }
    } else {
        // Epilogue: each warp owns 32 rows of the tile (TMEM lanes 32q..32q+31).
        // Per present block it stages its rows in shared memory, then copies
        // them out together: the warp's rows of one block are RS = min(32, B)
        // consecutive rows, i.e. one contiguous RS*B run of the output.
        constexpr int RS = BLK < 32 ? BLK : 32;
        constexpr int C16 = BLK * 2 / 16;  // 16-byte chunks per block row
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int a = row / BLK;
        uint8_t* stg = smem + C::kStg + quad * 32 * C::kPitch;
        T* Cp = reinterpret_cast<T*>(args.C);
        uint32_t g = 0;
        for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
            const int tile = L.tile_order[w / args.Z];
            const int z = (int)(w % args.Z);
            const int s0 = L.tile_step_ptr[tile], ns = L.tile_step_ptr[tile + 1] - s0;
            for (int n = 0; n < ns; ++n, ++g) {
                const int s = s0 + n;
                const uint32_t sb = g & 3;
                bool ok = mbar_wait(&s_full[sb], (g >> 2) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                tc_fence_after();
                uint32_t x[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_ld32_sync(tS + sb * 128 + lane_base + c * 32,
                                   *reinterpret_cast<uint32_t(*)[32]>(x + 32 * c));
                // the accumulator is free as soon as it is in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
#pragma unroll
                for (int b = 0; b < G; ++b) {
                    const int blk = L.step_blk[(s * G + a) * G + b];
                    if (__all_sync(0xffffffffu, blk < 0)) continue;
                    if (blk >= 0) {
                        uint4* srow = reinterpret_cast<uint4*>(stg + lane * C::kPitch);
#pragma unroll
                        for (int j = 0; j < C16; ++j) {
                            const int o = b * BLK + 8 * j;
                            srow[j] = make_uint4(
                                Pack2<T>::pack(__uint_as_float(x[o]), __uint_as_float(x[o + 1])),
                                Pack2<T>::pack(__uint_as_float(x[o + 2]), __uint_as_float(x[o + 3])),
                                Pack2<T>::pack(__uint_as_float(x[o + 4]), __uint_as_float(x[o + 5])),
                                Pack2<T>::pack(__uint_as_float(x[o + 6]), __uint_as_float(x[o + 7])));
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int seg = 0; seg < 32 / RS; ++seg) {
                        const int sblk = __shfl_sync(0xffffffffu, blk, seg * RS);
                        if (sblk < 0) continue;
                        const int r_in0 = (quad * 32 + seg * RS) % BLK;
                        uint4* dst = reinterpret_cast<uint4*>(Cp + (((int64_t)z * L.nnz + sblk) * BLK + r_in0) * BLK);
                        for (int k = lane; k < RS * C16; k += 32)
                            dst[k] = *reinterpret_cast<const uint4*>(stg + (seg * RS + k / C16) * C::kPitch +
                                                                     (k % C16) * 16);
                    }
                    __syncwarp();
                }
            }
        }
    epi_done:;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// --------------------------------------------------------------- launch ----

template <typename T, int BLK>
int spmm_launch(const bsp_layout_s* Lh, int is_dds, const void* dense, const void* sparse, void* Cout, int Z,
                int ext, int dense_mn, int sparse_mn, int use_csc, cudaStream_t s) {
    using Cfg = SpmmCfg<BLK>;
    const int bf = std::is_same<T, __nv_bfloat16>::value;
    const uint64_t S = Lh->S;
    CUtensorMap md, ms;
    int rc;
    if (dense_mn)  // [Z*H*S rows][ext cols], box BLK x 64
        rc = make_tmap_2d(&md, dense, bf, (uint64_t)Z * Lh->H * S, (uint64_t)ext, BLK, 64, 128);
    else           // [Z*H*ext rows][S cols], box 128 x W
        rc = make_tmap_2d(&md, dense, bf, (uint64_t)Z * Lh->H * ext, S, 128, Cfg::W, Cfg::RB);
    if (!rc)
        rc = make_tmap_2d(&ms, sparse, bf, (uint64_t)Z * Lh->nnz * BLK, BLK, BLK, Cfg::W, Cfg::RB);
    if (rc) return rc;
    const LayoutView& V = Lh->view;
    SpmmArgs a{V, Cout,
               use_csc ? V.col_ptr : V.row_ptr, use_csc ? V.row_idx : V.col_idx,
               use_csc ? V.blk_id_csc : V.blk_id, use_csc ? V.col_order : V.row_order,
               Z, is_dds, ext, (ext + 127) / 128, dense_mn, sparse_mn};
    auto kern = spmm_tc_kernel<T, BLK>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kAlloc) != cudaSuccess)
        return BSP_ERR_CUDA;
    const int64_t total = (int64_t)Lh->H * Lh->nb * Z * a.ntiles;
    const int grid = (int)std::min<int64_t>(total, sm_count());
    kern<<<grid, kThreads, Cfg::kAlloc, s>>>(md, ms, a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T>
int spmm_by_block(const bsp_layout_s* L, int is_dds, const void* dense, const void* sparse, void* C, int Z, int ext,
                  int dense_mn, int sparse_mn, int use_csc, cudaStream_t s) {
    switch (L->B) {
        case 16: return spmm_launch<T, 16>(L, is_dds, dense, sparse, C, Z, ext, dense_mn, sparse_mn, use_csc, s);
        case 32: return spmm_launch<T, 32>(L, is_dds, dense, sparse, C, Z, ext, dense_mn, sparse_mn, use_csc, s);
        case 64: return spmm_launch<T, 64>(L, is_dds, dense, sparse, C, Z, ext, dense_mn, sparse_mn, use_csc, s);
        case 128: return spmm_launch<T, 128>(L, is_dds, dense, sparse, C, Z, ext, dense_mn, sparse_mn, use_csc, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

int spmm_dispatch(const bsp_layout_s* L, int dtype, int is_dds, const void* dense, const void* sparse, void* C,
                  int Z, int ext, int dense_mn, int sparse_mn, int use_csc, cudaStream_t s) {
    // TMA: row strides must be multiples of 16 bytes, coordinates fit int32
    if (ext % 8 != 0) return BSP_ERR_UNSUPPORTED;
    if ((uint64_t)Z * L->H * std::max<int64_t>(L->S, ext) >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;
    if ((uint64_t)Z * L->nnz * L->B >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;
    if (dtype == BSP_BF16)
        return spmm_by_block<__nv_bfloat16>(L, is_dds, dense, sparse, C, Z, ext, dense_mn, sparse_mn, use_csc, s);
    if (dtype == BSP_F16)
        return spmm_by_block<__half>(L, is_dds, dense, sparse, C, Z, ext, dense_mn, sparse_mn, use_csc, s);
    return BSP_ERR_UNSUPPORTED;
}

template <typename T, int BLK, int KP>
int sdd_launch(const bsp_layout_s* Lh, const void* A, const void* B, void* Cout, int Z, int K, cudaStream_t s) {
    const int bf = std::is_same<T, __nv_bfloat16>::value;
    const uint64_t rows = (uint64_t)Z * Lh->H * Lh->S;
    CUtensorMap ma, mb;
    int rc = make_tmap_2d(&ma, A, bf, rows, K, 128, 64, 128);
    if (!rc) rc = make_tmap_2d(&mb, B, bf, rows, K, BLK, 64, 128);
    if (rc) return rc;
    SddArgs a{Lh->view, Cout, Z};
    auto kern = sdd_tc_kernel<T, BLK, KP>;
    constexpr int smem = SddCfg<KP, BLK>::kAlloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    const int64_t total = (int64_t)Z * Lh->n_tiles;
    const int grid = (int)std::min<int64_t>(total, sm_count());
    kern<<<grid, kThreads, smem, s>>>(ma, mb, a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T, int BLK>
int sdd_by_k(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int K, cudaStream_t s) {
    if (K <= 64) return sdd_launch<T, BLK, 1>(L, A, B, C, Z, K, s);
    return sdd_launch<T, BLK, 2>(L, A, B, C, Z, K, s);
}

template <typename T>
int sdd_by_block(const bsp_layout_s* L, const void* A, const void* B, void* C, int Z, int K, cudaStream_t s) {
    switch (L->B) {
        case 16: return sdd_by_k<T, 16>(L, A, B, C, Z, K, s);
        case 32: return sdd_by_k<T, 32>(L, A, B, C, Z, K, s);
        case 64: return sdd_by_k<T, 64>(L, A, B, C, Z, K, s);
        case 128: return sdd_by_k<T, 128>(L, A, B, C, Z, K, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_sdd_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int K, int ta,
                  int tb, cudaStream_t s) {
    // scores Q K^T: both operands [S][K] (K-major); K a multiple of 8, at most 128
    if (ta != 0 || tb != 1 || K % 8 != 0 || K > 128) return BSP_ERR_UNSUPPORTED;
    if ((uint64_t)Z * L->H * L->S >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;
    if (dtype == BSP_BF16) return sdd_by_block<__nv_bfloat16>(L, A, B, C, Z, K, s);
    if (dtype == BSP_F16) return sdd_by_block<__half>(L, A, B, C, Z, K, s);
    return BSP_ERR_UNSUPPORTED;
}

int launch_dsd_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int N, int ta,
                  int tb, cudaStream_t s) {
    // dense operand B: [S][N] (trans_b = 0) is MN-major for the n x k tile, [N][S] is K-major;
    // block of op(A_sp) row i: CSR (trans_a = 0, block[r][c] K-major) or CSC (trans_a = 1, MN-major)
    return spmm_dispatch(L, dtype, 0, B, A, C, Z, N, tb ? 0 : 1, ta ? 1 : 0, ta ? 1 : 0, s);
}

int launch_dds_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int M, int ta,
                  int tb, cudaStream_t s) {
    // dense operand A: [M][S] (trans_a = 0) is K-major, [S][M] MN-major;
    // block of op(B_sp) column j: CSC (trans_b = 0, block[k][c] MN-major) or CSR (trans_b = 1, K-major)
    return spmm_dispatch(L, dtype, 1, A, B, C, Z, M, ta ? 1 : 0, tb ? 0 : 1, tb ? 0 : 1, s);
}

}  // namespace bsp
