// Tensor-core (tcgen05) DSD and DDS on line groups, bf16 / fp16 in, fp32
// accumulate.  Operations of "question on blocksparse" (openai/triton issue
// 117): DSD is sparse (lhs) x dense, DDS is dense x sparse (rhs).
//
// Both are written as  Out[128 x NT] = sum over slots  Sp[128 x B] * Dn[B x NT]:
//  - a group is G = 128/B consecutive lines of the sparse operand (block-rows
//    of op(A_sp) for DSD; block-columns of op(B_sp) for DDS, which is computed
//    transposed: C^T = op(B_sp)^T op(A)^T), so the sparse slab fills the
//    MMA's M = 128 rows;
//  - its slots are the union of the lines' block indices along the
//    contraction; a slot's slab stacks the G lines' blocks at that index
//    (TMA loads), absent blocks written as zeros by the producer warp;
//  - the dense tile is the B rows of the dense operand at that index times
//    NT = 256 of its free columns (128 when the free extent is at most 128),
//    so one dense tile serves G lines and every MMA is 128 x NT x 16.
// Zero blocks inside a slab cost MMA time (the union is denser than any one
// line) but no memory traffic; with 32-wide blocks the old one-line-per-tile
// kernel was bound by re-reading the dense operand once per block line.
//
// Operand majorness follows the trans flags through the shared-memory
// descriptors, never through copies.  The accumulator is double-buffered in
// TMEM (2 x NT columns); four epilogue warps (thread = slab row = TMEM lane)
// write through 4 KB staging panels with TMA stores, so rows or columns past
// the end of C are clipped by the tensor map.
//
// Roles (288 threads): warps 0, 6, 7, 8 TMA producers, each filling every
// fourth pipeline stage (one issuing thread moves only ~24 bytes per clock of
// these tiles), warp 1 TMEM owner and single-thread MMA issuer, warps 2..5
// epilogue.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

namespace bsp {
namespace {

using namespace tc;

constexpr int kProducers = 4;                  // warps 0, 6, 7, 8
constexpr int kGThreads = (6 + kProducers - 1) * 32;

struct GroupArgs {
    LayoutView L;
    int Z;
    int orient;  // 0: groups of block-rows (CSR), 1: groups of block-columns (CSC)
    int ext;     // free extent of the dense operand: N (DSD) or M (DDS)
    int ntiles;  // ceil(ext / NT)
    int sp_mn;   // sparse slab MN-major (block stored [k][line index]) else K-major
    int dn_mn;   // dense tile MN-major (stored [k][free]) else K-major ([free][k])
    int dn_one;  // MN-major dense tile as one box of NT/64 panels (free extent a multiple of 64)
};

__host__ __device__ constexpr int gswz(int row_bytes) {
    return row_bytes == 128 ? kSw128 : (row_bytes == 64 ? kSw64 : kSw32);
}

// NT: dense free columns per tile = MMA N (256, or 128 when the free extent
// is at most 128)
template <int BLK, int NT>
struct GroupCfg {
    static constexpr int W = BLK < 64 ? BLK : 64;  // elements per 16-bit smem row of a block panel
    static constexpr int RB = W * 2;               // bytes per such row (= swizzle span)
    static constexpr int KPp = BLK / W;            // panels across a block
    static constexpr int kSp = 128 * BLK * 2;      // sparse slab of one slot
    static constexpr int kDn = BLK * NT * 2;       // dense tile of one slot
    static constexpr int kSlot = kSp + kDn;        // multiple of 1024 for every BLK
    static constexpr int KB = (49152 / kSlot) < 1 ? 1 : (49152 / kSlot);  // slots per pipeline stage
    static constexpr int kStage = KB * kSlot;
    static constexpr int ST = (196608 / kStage) > 4 ? 4 : (196608 / kStage);
    static constexpr int kEpi = ST * kStage;       // 4 warps x 4 KB staging
    static constexpr int kAlloc = kEpi + 4 * 4096 + 1024;
};

// OUT_T = 0: slab rows are rows of C (DSD): C[zh][line row][free];
// OUT_T = 1: slab rows are columns of C (DDS): C[zh][free][line column].
template <typename T, int BLK, int NT, int OUT_T>
__global__ void __launch_bounds__(kGThreads, 1)
spmm_group_kernel(const __grid_constant__ CUtensorMap tmSp, const __grid_constant__ CUtensorMap tmDn,
                  const __grid_constant__ CUtensorMap tmC, const GroupArgs args) {
    using C = GroupCfg<BLK, NT>;
    constexpr int kNT = NT;
    constexpr int G = 128 / BLK;
    constexpr int ST = C::ST, KB = C::KB, W = C::W, RB = C::RB, KPp = C::KPp;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[ST], empty[ST], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    // stages begun by each producer and by the MMA issuer when they stopped,
    // drained after the roles stop if the kernel aborted
    __shared__ uint32_t issued[kProducers + 1];

    const LayoutView& L = args.L;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Abort ab{&abort_flag, L.status, L.wait_ns};
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i <= kProducers; ++i) issued[i] = 0;
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
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tacc = tmem_base;

    const int o = args.orient;
    const int32_t* gptr = L.gl_ptr[o];
    const int32_t* gidx = L.gl_idx[o];
    const int32_t* gblk = L.gl_blk[o];
    const int64_t total = (int64_t)L.n_tiles * args.Z * args.ntiles;
    const int S = L.S;

    // Items run dense-tile-major (all groups and batch entries of one 256-wide
    // stripe of the dense operand, largest groups first, then the next
    // stripe): the CTAs working at any moment share a few MB of the dense
    // operand, which then stays in L2.
    const int64_t per_stripe = (int64_t)L.n_tiles * args.Z;
    auto item = [&](int64_t w, int& t, int& z, int& nt) {
        nt = (int)(w / per_stripe);
        const int64_t rem = w % per_stripe;
        t = L.gl_order[o][rem / args.Z];
        z = (int)(rem % args.Z);
    };

    if (warp == 0 || warp >= 6) {
        // --------------------------------------------------- TMA producers ----
        // The whole warp walks the slots: every 32 slots each lane loads one
        // slot's index and block ids (one round trip instead of one per slot),
        // lane 0 issues the TMA loads (the dense tile and the present blocks),
        // and the warp zeroes the absent blocks' rows of the slab with shared
        // stores, made visible to the tensor core before the stage's arrival.
        // A stage's barrier gets one arrival (after its last slot) and one
        // expected-bytes increase per slot.  Producer pid fills the stages
        // with it % NP == pid; all walk every slot to keep the count.  NP is at
        // most the number of stages: a producer's parity wait on its next
        // stage (NP uses later) is only sound if its previous wait already
        // ensured that the stage's use before last was consumed, i.e. NP <= ST.
        constexpr uint32_t NP = kProducers < ST ? kProducers : ST;
        const uint32_t pid = warp == 0 ? 0u : (uint32_t)(warp - 5);
        if (lane == 0) {
            tma_prefetch_desc(&tmSp);
            tma_prefetch_desc(&tmDn);
        }
        uint32_t it = 0;  // stages begun
        for (int64_t w = pid < NP ? blockIdx.x : total; w < total; w += gridDim.x) {
            int t, z, nt;
            item(w, t, z, nt);
            const int h = t / L.ngroups;
            const int64_t zh = (int64_t)z * L.H + h;
            const int n0 = nt * kNT;
            const int q0 = gptr[t], q1 = gptr[t + 1];
            for (int base = q0; base < q1; base += 32) {
                const int nq = min(32, q1 - base);
                int my_idx = 0, my_blk[G];
                if (lane < nq) {
                    my_idx = gidx[base + lane];
#pragma unroll
                    for (int a = 0; a < G; ++a) my_blk[a] = gblk[(int64_t)(base + lane) * G + a];
                }
                for (int j = 0; j < nq; ++j) {
                    const int q = base + j, rel = q - q0, sl = rel % KB;
                    const int kb = __shfl_sync(0xffffffffu, my_idx, j) * BLK;  // first contraction index
                    int bid[G];
#pragma unroll
                    for (int a = 0; a < G; ++a) bid[a] = __shfl_sync(0xffffffffu, my_blk[a], j);
                    const int st = it % ST;
                    const bool mine = it % NP == pid;
                    if (sl == 0 && mine) {
                        bool ok = true;
                        if (lane == 0) ok = mbar_wait(&empty[st], ((it / ST) & 1) ^ 1, ab);
                        if (!__shfl_sync(0xffffffffu, ok, 0)) goto producer_done;
                        __syncwarp();  // the stage's previous MMAs are done before any lane writes it
                    }
                    uint8_t* sp = smem + st * C::kStage + sl * C::kSlot;
                    uint8_t* dn = sp + C::kSp;
                    if (!mine) {
                        if (sl == KB - 1 || q == q1 - 1) ++it;
                        continue;
                    }
                    int present = 0;
#pragma unroll
                    for (int a = 0; a < G; ++a) present += bid[a] >= 0;
                    if (lane == 0) {
                        mbar_expect_tx(&full[st], C::kDn + present * (BLK * BLK * 2));
                        if (args.dn_one) {
                            // [k rows][free cols]: NT/64 panels of 64 free columns, B rows each,
                            // in one box (each TMA instruction costs the issuing thread ~60
                            // cycles on top of its bytes, so fewer, larger boxes)
                            tma_load_3d(smem_u32(dn), &tmDn, 0, (int32_t)(zh * S + kb), n0 / 64, &full[st]);
                        } else if (args.dn_mn) {
#pragma unroll
                            for (int p = 0; p < kNT / 64; ++p)
                                tma_load_2d(smem_u32(dn + p * (BLK * 128)), &tmDn, n0 + 64 * p,
                                            (int32_t)(zh * S + kb), &full[st]);
                        } else {
                            // [free rows][k cols]: panels of W contraction columns, NT rows each
#pragma unroll
                            for (int p = 0; p < KPp; ++p)
                                tma_load_2d(smem_u32(dn + p * (kNT * RB)), &tmDn, kb + W * p,
                                            (int32_t)(zh * args.ext + n0), &full[st]);
                        }
                    }
#pragma unroll
                    for (int a = 0; a < G; ++a) {
#pragma unroll
                        for (int p = 0; p < KPp; ++p) {
                            // K-major: panel p of the slab, rows a*B..; MN-major: M-panel a*KPp + p.
                            // Either way BLK * RB contiguous bytes.
                            const int off = args.sp_mn ? (a * KPp + p) * (BLK * RB) : p * (128 * RB) + a * (BLK * RB);
                            if (bid[a] >= 0) {
                                if (lane == 0)
                                    tma_load_2d(smem_u32(sp + off), &tmSp, W * p,
                                                (int32_t)(((int64_t)z * L.nnz + bid[a]) * BLK), &full[st]);
                            } else {
#pragma unroll
                                for (int i = lane * 16; i < BLK * RB; i += 32 * 16)
                                    *reinterpret_cast<uint4*>(sp + off + i) = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                    if (sl == KB - 1 || q == q1 - 1) {
                        // stage complete: zeroes visible to the tensor core, then one arrival
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&full[st]);
                        ++it;
                    }
                }
            }
        }
    producer_done:
        if (lane == 0) issued[pid] = it;
    } else if (warp == 1) {
        // ---------------------------------------------- MMA issuer (one thread) ----
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, kNT, kBf16, args.sp_mn, args.dn_mn);
            const uint32_t s0 = smem_u32(smem);
            const uint64_t dA = args.sp_mn ? smem_desc(s0, BLK * RB, 8 * RB, gswz(RB))
                                           : smem_desc(s0, 16, 8 * RB, gswz(RB));
            const uint64_t dB = args.dn_mn ? smem_desc(s0 + C::kSp, BLK * 128, 1024, kSw128)
                                           : smem_desc(s0 + C::kSp, 16, 8 * RB, gswz(RB));
            uint32_t offA[BLK / 16], offB[BLK / 16];
#pragma unroll
            for (int ks = 0; ks < BLK / 16; ++ks) {
                const int pan = 16 * ks / W, in = 16 * ks % W;
                offA[ks] = (args.sp_mn ? 16 * ks * RB : pan * (128 * RB) + in * 2) >> 4;
                offB[ks] = (args.dn_mn ? 16 * ks * 128 : pan * (kNT * RB) + in * 2) >> 4;
            }
            uint32_t it = 0, k = 0;
            for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
                int t, z, nt;
                item(w, t, z, nt);
                const int q0 = gptr[t], q1 = gptr[t + 1];
                if (q1 == q0) continue;
                const uint32_t buf = k & 1;
                if (!mbar_wait(&acc_empty[buf], ((k >> 1) & 1) ^ 1, ab)) goto mma_done;
                tc_fence_after();
                for (int c0 = q0; c0 < q1; c0 += KB, ++it) {
                    const int ns = min(KB, q1 - c0);
                    const int st = it % ST;
                    if (!mbar_wait(&full[st], (it / ST) & 1, ab)) goto mma_done;
                    tc_fence_after();
                    for (int sl = 0; sl < ns; ++sl) {
                        const uint32_t so = (uint32_t)(st * C::kStage + sl * C::kSlot) >> 4;
#pragma unroll
                        for (int ks = 0; ks < BLK / 16; ++ks)
                            mma_f16(tacc + buf * kNT, dA + so + offA[ks], dB + so + offB[ks], idesc,
                                    (c0 > q0 || sl > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[st]);
                }
                mma_commit(&acc_full[buf]);
                ++k;
            }
        mma_done:
            issued[kProducers] = it;
        }
    } else {
        // -------------------------------------------------------- epilogue ----
        const int quad = warp & 3;  // slab rows 32 quad + lane = TMEM lanes
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint8_t* stage = smem + C::kEpi + quad * 4096;
        const uint32_t stage_s = smem_u32(stage);
        uint32_t k = 0;
        for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
            int t, z, nt;
            item(w, t, z, nt);
            const int g = t % L.ngroups, h = t / L.ngroups;
            const int32_t zh = (int32_t)((int64_t)z * L.H + h);
            const int n0 = nt * kNT;
            const int line0 = g * 128 + quad * 32;  // first C row (DSD) / column (DDS) of this warp
            const bool has = gptr[t + 1] > gptr[t];
            const uint32_t buf = k & 1;
            if (has) {
                bool ok = mbar_wait(&acc_full[buf], (k >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                tc_fence_after();
            }
            // panels of 64 free columns: TMEM -> registers -> staging -> TMA store
#pragma unroll 1
            for (int p = 0; p < kNT / 64; ++p) {
                uint32_t pk[32];
                if (has) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t r[32];
                        tmem_ld32_sync(tacc + buf * kNT + lane_base + p * 64 + hh * 32, r);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[hh * 16 + j] = Pack2<T>::pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                    }
                    if (p == kNT / 64 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&acc_empty[buf]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) pk[j] = 0u;
                }
                if (line0 >= S || n0 + 64 * p >= args.ext) continue;  // wholly past the end of C
                if (lane == 0) bulk_wait_read_all();                   // the panel's previous store has read it
                __syncwarp();
                if (OUT_T == 0) {
                    // [32 rows][64 free] in the 128-byte-swizzled layout
                    uint8_t* rp = stage + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(rp + ((j ^ (lane & 7)) << 4)) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                } else {
                    // [64 free][32 columns]: this lane is one column of C
                    uint16_t* cp = reinterpret_cast<uint16_t*>(stage) + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        cp[(2 * j) * 32] = (uint16_t)(pk[j] & 0xffffu);
                        cp[(2 * j + 1) * 32] = (uint16_t)(pk[j] >> 16);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (OUT_T == 0) tma_store_3d(&tmC, stage_s, n0 + 64 * p, line0, zh);
                    else tma_store_3d(&tmC, stage_s, line0, n0 + 64 * p, zh);
                    bulk_commit();
                }
            }
            if (has) ++k;
        }
    epi_done:
        if (lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag) {
        // stopped early: the copies and products issued before the stop land
        // before the CTA lets go of its shared memory and TMEM -- for each
        // producer the last stage it began on each ring slot, for the MMA
        // issuer its last commit
        if (threadIdx.x == 0) {
            constexpr uint32_t NP = kProducers < ST ? kProducers : ST;
            for (uint32_t pid = 0; pid < NP; ++pid) {
                const uint32_t it = issued[pid];
                for (uint32_t st = 0; st < (uint32_t)ST; ++st) {
                    for (uint32_t j = it; j-- > 0 && j + (uint32_t)(ST * NP) >= it;) {
                        if (j % NP == pid && j % ST == st) {
                            mbar_drain(&full[st], (j / ST) & 1, ab);
                            break;
                        }
                    }
                }
            }
            const uint32_t it = issued[kProducers];
            if (it) mbar_drain(&empty[(it - 1) % ST], ((it - 1) / ST) & 1, ab);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <typename T, int BLK, int NT, int OUT_T>
int group_launch(const bsp_layout_s* Lh, const void* dense, const void* sparse, void* Cout, int Z, int ext,
                 int orient, int sp_mn, int dn_mn, cudaStream_t s) {
    using Cfg = GroupCfg<BLK, NT>;
    constexpr int kNT = NT;
    const int bf = std::is_same<T, __nv_bfloat16>::value;
    const uint64_t ZH = (uint64_t)Z * Lh->H;
    CUtensorMap msp, mdn, mc;
    int rc = make_tmap_2d(&msp, sparse, bf, (uint64_t)Z * Lh->nnz * BLK, BLK, BLK, Cfg::W, Cfg::RB);
    const int dn_one = dn_mn && ext % 64 == 0;
    if (!rc) {
        if (dn_one) rc = make_tmap_panels(&mdn, dense, bf, ZH * Lh->S, ext, BLK, kNT / 64);
        else if (dn_mn) rc = make_tmap_2d(&mdn, dense, bf, ZH * Lh->S, ext, BLK, 64, 128);
        else rc = make_tmap_2d(&mdn, dense, bf, ZH * ext, Lh->S, kNT, Cfg::W, Cfg::RB);
    }
    if (!rc) {
        if (OUT_T == 0) rc = make_tmap_3d(&mc, Cout, bf, ext, Lh->S, ZH, 64, 32, 128);
        else rc = make_tmap_3d(&mc, Cout, bf, Lh->S, ext, ZH, 32, 64, 0);
    }
    if (rc) return rc;
    GroupArgs a{Lh->view, Z, orient, ext, (ext + kNT - 1) / kNT, sp_mn, dn_mn, dn_one};
    auto kern = spmm_group_kernel<T, BLK, NT, OUT_T>;
    constexpr int smem = Cfg::kAlloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    const int64_t total = (int64_t)Lh->n_tiles * Z * a.ntiles;
    const int grid = (int)std::min<int64_t>(total, sm_count());
    kern<<<grid, kGThreads, smem, s>>>(msp, mdn, mc, a);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

template <typename T, int NT, int OUT_T>
int group_by_block(const bsp_layout_s* L, const void* dense, const void* sparse, void* C, int Z, int ext, int orient,
                   int sp_mn, int dn_mn, cudaStream_t s) {
    switch (L->B) {
        case 16: return group_launch<T, 16, NT, OUT_T>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
        case 32: return group_launch<T, 32, NT, OUT_T>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
        case 64: return group_launch<T, 64, NT, OUT_T>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
        case 128: return group_launch<T, 128, NT, OUT_T>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

template <typename T>
int group_by_shape(const bsp_layout_s* L, int out_t, const void* dense, const void* sparse, void* C, int Z, int ext,
                   int orient, int sp_mn, int dn_mn, cudaStream_t s) {
    if (ext <= 128)
        return out_t ? group_by_block<T, 128, 1>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s)
                     : group_by_block<T, 128, 0>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
    return out_t ? group_by_block<T, 256, 1>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s)
                 : group_by_block<T, 256, 0>(L, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
}

int group_dispatch(const bsp_layout_s* L, int dtype, int out_t, const void* dense, const void* sparse, void* C,
                   int Z, int ext, int orient, int sp_mn, int dn_mn, cudaStream_t s) {
    // TMA: row strides multiples of 16 bytes; coordinates (the zero-fill row past
    // the block storage included) fit int32
    if (ext % 8 != 0) return BSP_ERR_UNSUPPORTED;
    if ((uint64_t)Z * L->H * std::max<int64_t>(L->S, ext) >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;
    if ((uint64_t)Z * L->nnz * L->B >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;
    if (dtype == BSP_BF16) return group_by_shape<__nv_bfloat16>(L, out_t, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
    if (dtype == BSP_F16) return group_by_shape<__half>(L, out_t, dense, sparse, C, Z, ext, orient, sp_mn, dn_mn, s);
    return BSP_ERR_UNSUPPORTED;
}

}  // namespace

int launch_dsd_group_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int N,
                        int ta, int tb, cudaStream_t s) {
    // lines: block-rows of op(A_sp) = rows of A (CSR, blocks K-major) or, for
    // trans_a, columns of A (CSC, blocks [k][line]: MN-major); the dense operand
    // B is [S][N] (MN-major tile) or, for trans_b, [N][S] (K-major)
    return group_dispatch(L, dtype, 0, B, A, C, Z, N, ta ? 1 : 0, ta ? 1 : 0, tb ? 0 : 1, s);
}

int launch_dds_group_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int M,
                        int ta, int tb, cudaStream_t s) {
    // C^T = op(B_sp)^T op(A)^T: lines are the block-columns of op(B_sp) =
    // columns of B (CSC, blocks [k][line]: MN-major) or, for trans_b, rows of B
    // (CSR, K-major); the dense operand A is [M][S] (K-major) or, for trans_a,
    // [S][M] (MN-major)
    return group_dispatch(L, dtype, 1, A, B, C, Z, M, tb ? 0 : 1, tb ? 0 : 1, ta ? 1 : 0, s);
}

}  // namespace bsp
