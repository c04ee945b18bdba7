// Fused block-sparse attention for fp32 inputs on tcgen05 tensor cores
// (kind::tf32) with the three-term split that keeps fp32 accuracy: every fp32
// operand x is cut into hi = x rounded to tf32 (10 mantissa bits) and
// lo = x - hi (exact), and a product a b is taken as
// a_hi b_hi + a_hi b_lo + a_lo b_hi (the dropped a_lo b_lo is ~2^-22 of |a b|;
// the tensor core reads only the tf32 bits of lo as well, another ~2^-21).
// The method is the one of "question on blocksparse" (openai/triton issue
// 117: SDD -> softmax -> DSD on the layout's blocks, never writing the scores)
// with the online-softmax recurrence of the Triton-Puzzles blog, Puzzle 9
// "Simple FlashAttention" (running max and sum, output rescaled, divided by
// the sum at the end), like the 16-bit kernel; only the arithmetic of the two
// products changes.  Head size 64.
//
// Work: one row tile = 128 query rows (G = 128/B block-rows of one head) x one
// batch entry, persistent CTAs walking the tiles longest-first.  A step of the
// layout's tables (G slots, 128 keys) is taken as two half-steps of 64 keys:
// one S buffer of 64 fp32 columns per half-step, P (hi and lo) 64 + 64 columns.
//
// Roles (512 threads, one CTA per SM):
//   warp 0      TMA producer of the Q tile and of the K half-tiles (raw fp32)
//   warp 1      TMEM owner; one thread issues S = Q K^T (three products, M=128,
//               N=64, K=64) into S buffer g % 3
//   warp 2      one thread issues O += P V (three products, M=128, N=64, K=64
//               keys, P from TMEM)
//   warps 4..7  converters: split Q and K in place (hi over the raw values, lo
//               into a buffer of its own); V they read from global memory
//               themselves, one half-step ahead, and write transposed into hi
//               and lo buffers (the tensor core reads tf32 operands K-major)
//   warps 8..15 softmax and epilogue: both warpgroups on every half-step, 32
//               keys each (thread = query row = TMEM lane), half-row maxima
//               swapped through shared memory per lane quadrant; P written as
//               hi over the thread's own scores and lo beside them; at a
//               tile's end they add the two half-row sums, read O, scale and
//               store it (fp32, row by row) and hand the accumulator back.
// TMEM columns: S/P_hi buffer b at 128 b, P_lo at 128 b + 64 (b < 3), O at 384.
#include <algorithm>

#include "common.cuh"
#include "tc_common.cuh"

namespace bsp {
namespace attn32 {

using namespace tc;

constexpr int kThreads = 512;
constexpr int D = 64;
// registers after the split at kernel start (launched with 128): control
// warps 72, converters 96, softmax / epilogue 168:
// 128 x (72 + 96) + 256 x 168 = 64512 <= 65536
constexpr uint32_t kRegsLaunch = 128, kRegsCtl = 72, kRegsConv = 96, kRegsSoftmax = 168;
static_assert(kRegsCtl + kRegsConv + 2 * kRegsSoftmax <= 4 * kRegsLaunch, "register split exceeds the launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// shared memory (bytes): every tile in 128-byte-swizzled K-major panels of 32
// fp32 (128-byte rows, 8-row atoms of 1024 bytes)
struct Smem32 {
    static constexpr int kQ = 0;                   // Q: 2 panels x 128 rows (hi, in place)
    static constexpr int kQlo = kQ + 32768;        // Q lo
    static constexpr int kK = kQlo + 32768;        // K: 2 stages x 2 panels x 64 rows (hi, in place)
    static constexpr int kKlo = kK + 2 * 16384;    // K lo, 2 stages
    static constexpr int kVt = kKlo + 2 * 16384;   // V^T hi and lo, 2 stages: 2 panels (32 keys) x 64 dims each
    static constexpr int kBytes = kVt + 2 * 2 * 16384;
    static constexpr int kAlloc = kBytes + 1024;
};

struct Attn32Args {
    LayoutView L;
    const float* V;
    float* O;
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
    float c2;  // scale * log2(e)
};

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// component j (0..3, known at compile time after unrolling) of a float4
__device__ __forceinline__ float comp(const float4& v, int j) {
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// byte offset of element (row r, 16-byte chunk j) in a 128-byte-swizzled panel
__device__ __forceinline__ uint32_t swz(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// Instruction descriptor for kind::tf32, fp32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <int BLK, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
attention_tf32_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const Attn32Args args) {
    using SM = Smem32;
    constexpr int G = 128 / BLK;
    constexpr int R = BLK < 64 ? BLK : 64;  // key rows of one copy of a half-step (one box)
    constexpr int NBOX = 64 / R;            // copies (boxes) per half-step and panel
    constexpr uint32_t kIdescQK = idesc_tf32(128, 64);
    constexpr uint32_t kIdescPV = idesc_tf32(128, D);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t q_full, q_conv, q_empty, k_full[2], k_conv[2], k_empty[2];
    __shared__ uint64_t v_conv[2], v_empty[2];
    __shared__ uint64_t s_full[3], p_full[3], pv_done[3], o_full, o_empty;
    __shared__ uint64_t x_full[2][4], lx_full[4];
    __shared__ float xm[2][2][128], lx[2][128];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    // what each issuing thread had issued when it stopped (Q tiles, K
    // half-steps, -, Q K^T half-steps, P V half-steps), drained after the
    // roles stop if the kernel aborted
    __shared__ uint32_t issued[5];

    const LayoutView& L = args.L;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Abort ab{&abort_flag, L.status, L.wait_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 5; ++i) issued[i] = 0;
        mbar_init(&q_full, 1);
        mbar_init(&q_conv, 4);
        mbar_init(&q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_conv[i], 4);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_conv[i], 4);
            mbar_init(&v_empty[i], 1);
            for (int q = 0; q < 4; ++q) mbar_init(&x_full[i][q], 2);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 8);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(&o_full, 1);
        mbar_init(&o_empty, 8);
        for (int q = 0; q < 4; ++q) mbar_init(&lx_full[q], 2);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base;        // S / P_hi at 128 b, P_lo at 128 b + 64
    const uint32_t tO = tmem_base + 384;  // O

    const int S = L.S;

    if (warp < 4) {
        regs_dec<kRegsCtl>();
        if (warp == 0 && lane == 0) {
            // --------------------------------------------------- TMA producer ----
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            uint32_t q_it = 0, g = 0;
            for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
                const int4 run = args.sched_items[it];
                const int tile = run.x, s0 = run.y, ns = run.z;
                if (ns == 0) continue;
                const int z = run.w;
                const int h = tile / L.ngroups, gq = tile % L.ngroups;
                const int64_t zh = (int64_t)z * L.H + h;
                // Q of this tile once the previous tile's last Q K^T has read it
                if (q_it > 0 && !mbar_wait(&q_empty, (q_it - 1) & 1, ab)) goto producer_done;
                mbar_arrive_expect_tx(&q_full, 32768);
                for (int p = 0; p < 2; ++p)
                    tma_load_2d(smem_u32(smem + SM::kQ + p * 16384), &tmQ, p * 32, (int32_t)(zh * S + gq * 128),
                                &q_full);
                ++q_it;
                for (int n = 0; n < 2 * ns; ++n, ++g) {
                    const int s = s0 + (n >> 1), hh = n & 1;
                    int rows[NBOX];  // first key row of each box
                    bool ok_rows = true;
#pragma unroll
                    for (int j = 0; j < NBOX; ++j) {
                        const int k0 = 64 * hh + j * R;  // key offset inside the step
                        const int b = k0 / BLK;
                        int c = L.step_col[s * G + b];
                        if (c < 0) c = L.step_col[s * G];  // padding slot: any valid block
                        ok_rows &= (unsigned)c < (unsigned)L.nb;
                        rows[j] = c * BLK + k0 % BLK;
                    }
                    if (!ok_rows) {
                        ab.fail(BSP_ERR_DEVICE_CHECK);
                        goto producer_done;
                    }
                    const uint32_t st = g & 1;
                    if (g >= 2 && !mbar_wait(&k_empty[st], ((g - 2) >> 1) & 1, ab)) goto producer_done;
                    mbar_arrive_expect_tx(&k_full[st], 16384);
#pragma unroll
                    for (int j = 0; j < NBOX; ++j)
                        for (int p = 0; p < 2; ++p)
                            tma_load_2d(smem_u32(smem + SM::kK + st * 16384 + p * 8192 + j * R * 128), &tmK, p * 32,
                                        (int32_t)(zh * S + rows[j]), &k_full[st]);
                }
            }
        producer_done:
            issued[0] = q_it;
            issued[1] = g;
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------ Q K^T issuer (one thread) ----
            const uint64_t dq = smem_desc(smem_u32(smem + SM::kQ), 16, 1024, kSw128);
            const uint64_t dql = smem_desc(smem_u32(smem + SM::kQlo), 16, 1024, kSw128);
            const uint64_t dk = smem_desc(smem_u32(smem + SM::kK), 16, 1024, kSw128);
            const uint64_t dkl = smem_desc(smem_u32(smem + SM::kKlo), 16, 1024, kSw128);
            uint32_t q_it = 0, g = 0;
            for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
                const int ns = args.sched_items[it].z;
                if (ns == 0) continue;
                if (!mbar_wait(&q_conv, q_it & 1, ab)) goto qk_done;
                for (int n = 0; n < 2 * ns; ++n, ++g) {
                    const uint32_t st = g & 1, sb = g % 3;
                    if (g >= 3 && !mbar_wait(&pv_done[sb], ((g - 3) / 3) & 1, ab)) goto qk_done;
                    if (!mbar_wait(&k_conv[st], (g >> 1) & 1, ab)) goto qk_done;
                    tc_fence_after();
                    const uint32_t ko = (st * 16384) >> 4;
                    // hi hi, hi lo, lo hi; K-step of 8 fp32 = 32 bytes inside a panel
#pragma unroll
                    for (int term = 0; term < 3; ++term) {
                        const uint64_t a = term == 2 ? dql : dq;
                        const uint64_t b = (term == 1 ? dkl : dk) + ko;
#pragma unroll
                        for (int ks = 0; ks < D / 8; ++ks) {
                            const uint32_t qo = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                            const uint32_t kof = ((ks >> 2) * 8192 + (ks & 3) * 32) >> 4;
                            mma_tf32(tS + sb * 128, a + qo, b + kof, kIdescQK, (term > 0 || ks > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(&s_full[sb]);
                    mma_commit(&k_empty[st]);
                    if (n == 2 * ns - 1) mma_commit(&q_empty);
                }
                ++q_it;
            }
        qk_done:
            issued[3] = g;
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------- P V issuer (one thread) ----
            const uint64_t dv = smem_desc(smem_u32(smem + SM::kVt), 16, 1024, kSw128);
            uint32_t g = 0, tc = 0;
            for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
                const int ns = args.sched_items[it].z;
                if (ns == 0) continue;
                if (tc > 0 && !mbar_wait(&o_empty, (tc - 1) & 1, ab)) goto pv_done_label;
                for (int n = 0; n < 2 * ns; ++n, ++g) {
                    const uint32_t st = g & 1, sb = g % 3;
                    if (!mbar_wait(&p_full[sb], (g / 3) & 1, ab)) goto pv_done_label;
                    if (!mbar_wait(&v_conv[st], (g >> 1) & 1, ab)) goto pv_done_label;
                    tc_fence_after();
                    // V^T stage st: hi at +0, lo at +16384; panel (32 keys) at +8192
                    const uint32_t vo = (st * 32768) >> 4;
#pragma unroll
                    for (int term = 0; term < 3; ++term) {
                        const uint32_t pa = tS + sb * 128 + (term == 2 ? 64 : 0);  // P hi, P hi, P lo
                        const uint64_t b = dv + vo + (term == 1 ? (16384 >> 4) : 0);  // V hi, V lo, V hi
#pragma unroll
                        for (int ks = 0; ks < 64 / 8; ++ks) {
                            const uint32_t bo = ((ks >> 2) * 8192 + (ks & 3) * 32) >> 4;
                            mma_tf32_tmem_a(tO, pa + ks * 8, b + bo, kIdescPV, (n > 0 || term > 0 || ks > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(&pv_done[sb]);
                    mma_commit(&v_empty[st]);
                }
                mma_commit(&o_full);
                ++tc;
            }
        pv_done_label:
            issued[4] = g;
        }
    } else if (warp < 8) {
        regs_dec<kRegsConv>();
        // ------------------------------------------------------- converters ----
        // 128 threads.  Q: 2 panels x 128 rows x 8 chunks of 4 fp32; K: 2 x 64 x 8;
        // V: 64 keys x 64 dims read as 4 x 4 blocks and written transposed.
        const int ct = threadIdx.x - 128;
        uint32_t q_it = 0, g = 0;
        // this thread's part of a V half-tile: 2 blocks of 4 keys x 4 dims, one
        // 16-byte load per key (16 threads cover a 256-byte key row)
        float4 vreg[8];
        auto load_v = [&](int64_t zh, int s, int hh) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int blkv = ct + 128 * i;
                const int kb = (blkv >> 4) * 4, db = (blkv & 15) * 4;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int k0 = 64 * hh + kb + r;  // key offset inside the step
                    const int b = k0 / BLK;
                    int c = L.step_col[s * G + b];
                    if (c < 0) c = L.step_col[s * G];  // padding slot: any valid block
                    c = min(max(c, 0), L.nb - 1);      // the producer's bounds check reports bad columns
                    const int64_t key = zh * S + (int64_t)c * BLK + k0 % BLK;
                    vreg[4 * i + r] = __ldg(reinterpret_cast<const float4*>(args.V + key * D + db));
                }
            }
        };
        auto split_chunk = [](uint8_t* hi, uint8_t* lo) {
            float4 v = *reinterpret_cast<float4*>(hi);
            float4 h, l;
            h.x = __uint_as_float(tf32_rna(v.x));
            h.y = __uint_as_float(tf32_rna(v.y));
            h.z = __uint_as_float(tf32_rna(v.z));
            h.w = __uint_as_float(tf32_rna(v.w));
            l.x = v.x - h.x;
            l.y = v.y - h.y;
            l.z = v.z - h.z;
            l.w = v.w - h.w;
            *reinterpret_cast<float4*>(hi) = h;
            *reinterpret_cast<float4*>(lo) = l;
        };
        for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
            const int4 run = args.sched_items[it];
            const int tile = run.x, s0 = run.y, ns = run.z;
            if (ns == 0) continue;
            const int64_t zh = (int64_t)run.w * L.H + tile / L.ngroups;
            load_v(zh, s0, 0);  // V of the tile's first half-step
            {
                bool ok = mbar_wait(&q_full, q_it & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto conv_done;
                // 2048 chunks of 16 bytes, same offsets in the hi and lo buffers
                for (int c = ct; c < 2048; c += 128)
                    split_chunk(smem + SM::kQ + c * 16, smem + SM::kQlo + c * 16);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_conv);
                ++q_it;
            }
            for (int n = 0; n < 2 * ns; ++n, ++g) {
                const uint32_t st = g & 1;
                bool ok = mbar_wait(&k_full[st], (g >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto conv_done;
                for (int c = ct; c < 1024; c += 128)
                    split_chunk(smem + SM::kK + st * 16384 + c * 16, smem + SM::kKlo + st * 16384 + c * 16);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&k_conv[st]);
                // V(g), read from global memory a half-step ago, -> V^T hi / lo
                // [dim][key] (panel = 32 keys, rows = dims) in stage st, once P V of
                // half-step g - 2 has read the stage; then the loads of V(g + 1)
                if (g >= 2) ok = mbar_wait(&v_empty[st], ((g - 2) >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto conv_done;
                uint8_t* vt = smem + SM::kVt + st * 32768;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int blkv = ct + 128 * i;
                    const int kb = (blkv >> 4) * 4, db = (blkv & 15) * 4;  // 4 keys x 4 dims
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int dim = db + j;
                        const float a0 = comp(vreg[4 * i + 0], j), a1 = comp(vreg[4 * i + 1], j);
                        const float a2 = comp(vreg[4 * i + 2], j), a3 = comp(vreg[4 * i + 3], j);
                        float4 hv, lv;
                        hv.x = __uint_as_float(tf32_rna(a0));
                        hv.y = __uint_as_float(tf32_rna(a1));
                        hv.z = __uint_as_float(tf32_rna(a2));
                        hv.w = __uint_as_float(tf32_rna(a3));
                        lv.x = a0 - hv.x;
                        lv.y = a1 - hv.y;
                        lv.z = a2 - hv.z;
                        lv.w = a3 - hv.w;
                        const uint32_t o = (kb >> 5) * 8192 + swz(dim, (kb & 31) >> 2);
                        *reinterpret_cast<float4*>(vt + o) = hv;
                        *reinterpret_cast<float4*>(vt + 16384 + o) = lv;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&v_conv[st]);
                if (n + 1 < 2 * ns) load_v(zh, s0 + ((n + 1) >> 1), (n + 1) & 1);
            }
        }
    conv_done:;
    } else {
        regs_inc<kRegsSoftmax>();
        // ------------------------------------------------ softmax, epilogue ----
        constexpr int W = BLK < 32 ? BLK : 32;  // columns of one slot inside a quarter row
        constexpr int LS = 32 / W;              // slots (or slot parts) per 32 keys
        const int wg = (warp - 8) >> 2, hf = wg;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // query row inside the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const int r_in = row % BLK, a = row / BLK;
        uint32_t g = 0, tc = 0;
        for (int it = args.sched_ptr[blockIdx.x], it_end = args.sched_ptr[blockIdx.x + 1]; it < it_end; ++it) {
            const int4 run = args.sched_items[it];
            const int tile = run.x, s0 = run.y, ns = run.z;
            const int z = run.w;
            const int h = tile / L.ngroups, gq = tile % L.ngroups;
            const int rb = gq * G + a;        // block-row of this thread's query row
            const int rseq = gq * 128 + row;  // query position inside the sequence
            float* orow = args.O + (((int64_t)z * L.H + h) * S + rseq) * D + 32 * hf;
            if (ns == 0) {  // nothing kept anywhere in the tile: rows of zeros
                if (args.lse && hf == 0 && rseq < S) args.lse[((int64_t)z * L.H + h) * S + rseq] = -INFINITY;
                if (rseq < S)
#pragma unroll
                    for (int k = 0; k < 8; ++k) reinterpret_cast<float4*>(orow)[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                continue;
            }
            float l = 0.f, m = -INFINITY;
            for (int n = 0; n < 2 * ns; ++n, ++g) {
                const int s = s0 + (n >> 1), hh = n & 1;
                // this thread's 32 keys of the half-step: slots and in-block columns
                int blk[LS], cb[LS];
#pragma unroll
                for (int ls = 0; ls < LS; ++ls) {
                    const int k0 = 64 * hh + 32 * hf + ls * W;
                    const int b = k0 / BLK;
                    blk[ls] = L.step_blk[(s * G + a) * G + b];
                    cb[ls] = L.step_col[s * G + b];
                }
                const uint32_t sb = g % 3, xb = g & 1;
                bool ok = mbar_wait(&s_full[sb], (g / 3) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                tc_fence_after();
                const uint32_t srow = tS + sb * 128 + lane_base;
                uint32_t xr[32];
                tmem_ld32_sync(srow + 32 * hf, xr);
                float* x = reinterpret_cast<float*>(xr);
#pragma unroll
                for (int ls = 0; ls < LS; ++ls) {
                    const int kbase = (64 * hh + 32 * hf + ls * W) % BLK;  // in-block column of x[ls * W]
                    if (KIND == BSP_MASK_DIAG_CAUSAL) {
                        const int lim = blk[ls] < 0 ? -1 : (cb[ls] == rb ? r_in - kbase : W);
#pragma unroll
                        for (int j = 0; j < W; ++j) x[ls * W + j] = j > lim ? -INFINITY : x[ls * W + j];
                    } else if (blk[ls] < 0) {
#pragma unroll
                        for (int j = 0; j < W; ++j) x[ls * W + j] = -INFINITY;
                    } else if (KIND == BSP_MASK_DENSE) {
                        const uint8_t* mp = args.mask + (int64_t)rseq * S + (int64_t)cb[ls] * BLK + kbase;
#pragma unroll
                        for (int q = 0; q < W / 16; ++q) {
                            const uint4 mv = *reinterpret_cast<const uint4*>(mp + q * 16);
                            const uint8_t* mb = reinterpret_cast<const uint8_t*>(&mv);
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                if (!mb[k]) x[ls * W + q * 16 + k] = -INFINITY;
                        }
                    }
                }
                float mx = -INFINITY;
#pragma unroll
                for (int k = 0; k < 32; ++k) mx = fmaxf(mx, x[k]);
                // swap quarter-row maxima with the other thread of the row (the
                // arrival also says this thread's scores are in registers)
                xm[xb][wg][row] = mx;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_full[xb][quad]);
                ok = mbar_wait(&x_full[xb][quad], (g >> 1) & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                tc_fence_after();
                const float m_new = fmaxf(m, fmaxf(mx, xm[xb][wg ^ 1][row]) * args.c2);
                const bool need = m_new > m + kRescaleThreshold;
                const float mnext = need ? m_new : m;
                const float msub = (mnext == -INFINITY) ? 0.f : mnext;
                float rs = 0.f;
                uint32_t hi[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float p = ex2_approx(fmaf(x[k], args.c2, -msub));
                    rs += p;
                    hi[k] = tf32_rna(p);
                    xr[k] = __float_as_uint(p - __uint_as_float(hi[k]));  // lo
                }
                tmem_st32_sync(srow + 32 * hf, hi);       // P hi over this thread's own scores
                tmem_st32_sync(srow + 64 + 32 * hf, xr);  // P lo
                if (n > 0 && __any_sync(0xffffffffu, need)) {
                    ok = mbar_wait(&pv_done[(g - 1) % 3], ((g - 1) / 3) & 1, ab);
                    if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                    tc_fence_after();
                    const float alpha = need ? (m == -INFINITY ? 0.f : ex2_approx(m - mnext)) : 1.f;
                    uint32_t r[32];
                    const uint32_t ta = tO + lane_base + 32 * hf;
                    tmem_ld32_sync(ta, r);
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                    tmem_st32_sync(ta, r);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
                l = (need ? (m == -INFINITY ? 0.f : l * ex2_approx(m - msub)) : l) + rs;
                m = mnext;
            }
            // tile end: the row's sum is the two threads' sums (same reference m);
            // O (after the last P V) scaled by 1 / sum, stored, and handed back
            {
                lx[wg][row] = m == -INFINITY ? 0.f : l;
                __syncwarp();
                if (lane == 0) mbar_arrive(&lx_full[quad]);
                bool ok = mbar_wait(&lx_full[quad], tc & 1, ab);
                if (ok) ok = mbar_wait(&o_full, tc & 1, ab);
                if (!__all_sync(0xffffffffu, ok)) goto softmax_done;
                tc_fence_after();
                const float lt = lx[0][row] + lx[1][row];
                const float inv = lt > 0.f ? 1.0f / lt : 0.f;
                uint32_t r[32];
                tmem_ld32_sync(tO + lane_base + 32 * hf, r);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_empty);
                const int part = args.sched_part[it];
                if (args.lse && part < 0 && hf == 0 && rseq < S)  // cut tiles: the combine pass writes it
                    args.lse[((int64_t)z * L.H + h) * S + rseq] = lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
                if (part >= 0) {
                    // a piece of a cut tile: O as accumulated (relative to the
                    // common reference m), m and the sum, for the combine pass
                    float* pw = args.part_ws + (size_t)part * kPartFloats;
                    float* prow = pw + (size_t)row * D + 32 * hf;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        reinterpret_cast<uint4*>(prow)[k] = make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                    if (hf == 0) {
                        pw[kPartRows * kPartMaxD + row] = m;
                        pw[kPartRows * kPartMaxD + kPartRows + row] = lt;
                    }
                } else if (rseq < S) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        reinterpret_cast<float4*>(orow)[k] =
                            make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                        __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
                }
                ++tc;
            }
        }
    softmax_done:;
    }

    tc_fence_before();
    __syncthreads();
    if (abort_flag) {
        // stopped early: the copies and products issued before the stop land
        // before the CTA lets go of its shared memory and TMEM
        if (threadIdx.x == 0) {
            if (issued[0]) mbar_drain(&q_full, (issued[0] - 1) & 1, ab);
            mbar_drain_ring(k_full, 2, issued[1], ab);
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

template <int BLK, int KIND>
int launch32(const bsp_layout_s* Lh, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, float scale,
             const uint8_t* mask, cudaStream_t s) {
    const uint64_t rows = (uint64_t)Z * Lh->H * Lh->S;
    constexpr uint32_t R = BLK < 64 ? BLK : 64;
    CUtensorMap mq, mk;
    int rc = make_tmap_2d_f32(&mq, Q, rows, D, 128, 32);
    if (!rc) rc = make_tmap_2d_f32(&mk, K, rows, D, R, 32);
    if (rc) return rc;
    auto kern = attention_tf32_kernel<BLK, KIND>;
    constexpr int smem = Smem32::kAlloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BSP_ERR_CUDA;
    // the register split at kernel start needs the full launch allocation
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return BSP_ERR_CUDA;
    if ((uint32_t)fa.numRegs != kRegsLaunch) return BSP_ERR_UNSUPPORTED;
    AttnSchedule sc;
    if ((rc = attn_schedule_begin(const_cast<bsp_layout_s*>(Lh), BSP_F32, Z, s, &sc))) return rc;
    Attn32Args args{Lh->view, (const float*)V, (float*)O, mask, sc.ptr, sc.items, sc.part, sc.ws, lse, Z,
                    scale * kLog2e};
    if (sc.grid > 0) {
        kern<<<sc.grid, kThreads, smem, s>>>(mq, mk, args);
        rc = cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
    }
    return attn_schedule_end(Lh, BSP_F32, sc, O, lse, D, s, rc);
}

template <int BLK>
int by_kind32(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, float scale,
              int kind, const uint8_t* mask, cudaStream_t s) {
    switch (kind) {
        case BSP_MASK_NONE: return launch32<BLK, BSP_MASK_NONE>(L, Q, K, V, O, lse, Z, scale, mask, s);
        case BSP_MASK_DENSE: return launch32<BLK, BSP_MASK_DENSE>(L, Q, K, V, O, lse, Z, scale, mask, s);
        case BSP_MASK_DIAG_CAUSAL: return launch32<BLK, BSP_MASK_DIAG_CAUSAL>(L, Q, K, V, O, lse, Z, scale, mask, s);
        default: return BSP_ERR_INVALID_ARG;
    }
}

}  // namespace attn32

int launch_attention_tc_tf32(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z,
                             int D, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if (D != attn32::D) return BSP_ERR_UNSUPPORTED;
    switch (L->B) {
        case 128: return attn32::by_kind32<128>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
        case 64: return attn32::by_kind32<64>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
        case 32: return attn32::by_kind32<32>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
        case 16: return attn32::by_kind32<16>(L, Q, K, V, O, lse, Z, scale, kind, mask, s);
        default: return BSP_ERR_UNSUPPORTED;
    }
}

}  // namespace bsp
