// sm_103a building blocks for the tensor-core kernels: mbarriers with
// bounded waits, TMA tile loads, tcgen05 (TMEM allocation, MMA, commit,
// TMEM <-> register moves) and the shared-memory / instruction descriptors.
//
// Operand tiles live in shared memory in the 128-byte-swizzled canonical
// layouts that TMA writes: rows of 128 bytes (64 16-bit elements), 8-row
// atoms of 1024 bytes, the 16-byte chunk index XOR-ed with (row % 8).
//  - K-major operand (contraction dim contiguous): a [rows x 64] panel per 64
//    contraction elements; descriptor SBO = 1024 (next 8 rows); an MMA K-step
//    of 16 elements starts 32 bytes further inside the panel.
//  - MN-major operand (row/column dim contiguous): rows of the panel are
//    contraction indices; SBO = 1024 (next 8 contraction indices), LBO = the
//    byte distance between consecutive 64-element panels along M/N.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "bsp_internal.h"

namespace bsp {
namespace tc {

// ------------------------------------------------------------- basics ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool elect_one() {
    return (threadIdx.x & 31) == 0;
}

// -------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// raise the phase's expected transaction bytes without arriving
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Shared abort flag: set by the first wait that runs out (or the first
// failed bounds check); every other wait gives up as soon as it sees it.
// limit_ns: the wait limit (0 = kDefaultWaitNs).
struct Abort {
    volatile int* flag;
    int* status;
    uint64_t limit_ns;
    __device__ __forceinline__ uint64_t limit() const { return limit_ns ? limit_ns : kDefaultWaitNs; }
    // record `code` in the status word (the first code wins) and stop every role
    __device__ __forceinline__ void fail(int code) const {
        *flag = 1;
        if (status) atomicCAS(status, 0, code);
    }
};

// Wait for the phase with the given parity to complete.  Bounded: after the
// limit (or once another role has aborted) it records BSP_ERR_TIMEOUT and
// returns false; the caller then leaves its loop.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Abort& ab) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 63) == 0) {
            if (*ab.flag) return false;
            if (globaltimer_ns() - t0 > ab.limit()) {
                ab.fail(BSP_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// After an abort: wait, bounded by the limit but regardless of the abort
// flag, for the phase of `bar` with the given parity, i.e. until the copies
// or matrix products that signal it have landed.  A role calls it for every
// asynchronous operation it issued before it returns, so that no copy writes
// shared memory and no product writes TMEM after the CTA has released them.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, const Abort& ab) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > ab.limit()) return;
}

// Drain a ring of nst stages whose phases were begun in order 0, 1, ...,
// next - 1 (stage = index % nst, phase = index / nst): waits for the last
// phase begun on each stage.
__device__ __forceinline__ void mbar_drain_ring(uint64_t* bars, uint32_t nst, uint32_t next, const Abort& ab) {
    for (uint32_t s = 0; s < nst; ++s) {
        if (next <= s) continue;
        const uint32_t last = s + ((next - 1 - s) / nst) * nst;  // largest index < next on stage s
        mbar_drain(&bars[s], (last / nst) & 1, ab);
    }
}

// The w-th work item of a persistent tile loop (w = rank * Z + z): the tile of
// rank w / Z in longest-first order as (tile id, first step, step count, 0) --
// one 16-byte load, not a chain of dependent ones.  Callers keep w < 2^31.
__device__ __forceinline__ int4 tile_run_at(const LayoutView& L, int64_t w, int Z) {
    return reinterpret_cast<const int4*>(L.tile_run)[(uint32_t)w / (uint32_t)Z];
}

// ------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Non-tensor bulk copies (contiguous bytes; 16-byte aligned addresses, size a
// multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until every committed bulk store has finished READING shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... all but the N most recently committed groups
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Tiled 3-D store shared -> global (bulk group; coordinates innermost first).
// Rows past the tensor's extent in any dimension are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y,
                                             int32_t z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}
// wait until every committed bulk store has completed (its writes included)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------- tcgen05 --

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Change the registers a warp owns (all warps of a warpgroup execute the same
// one).  inc waits until other warpgroups of the block have released enough
// with dec, so the shares of all warpgroups must add up to no more than the
// block was launched with; the launcher checks that before the first launch.
template <uint32_t N> __device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N> __device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 / fp16 in, fp32 accumulate)
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16.  A (M = 128 rows) sits in
// TMEM: row i in lane i, 16-bit elements packed two per 32-bit column (the
// lower K index in the low half), K = 16 per instruction = 8 columns.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every previously issued tcgen05.mma of this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

#define BSP_TMEM_REGS32(r)                                                                                    \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),           \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),            \
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),            \
        "=r"(r[30]), "=r"(r[31])
#define BSP_TMEM_IN32(r)                                                                                       \
    "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),         \
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),         \
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),        \
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// tcgen05.st reads its source registers asynchronously (until
// tcgen05.wait::st), so the store and its wait also form one asm statement:
// the compiler may reuse the registers as soon as the statement ends.
__device__ __forceinline__ void tmem_st32_sync(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        ::"r"(taddr), BSP_TMEM_IN32(r)
        : "memory");
}
// tcgen05.ld is asynchronous: its destination registers hold the data only
// after tcgen05.wait::ld.  The compiler cannot know that, so a load and its
// wait must sit in ONE asm statement, otherwise a register spill between the
// two would copy undefined values.  These helpers do exactly that.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : BSP_TMEM_REGS32(r)
        : "r"(taddr)
        : "memory");
}
#define BSP_TMEM_REGS32_AT(r, o)                                                                                \
    "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]),             \
        "=r"(r[o + 6]), "=r"(r[o + 7]), "=r"(r[o + 8]), "=r"(r[o + 9]), "=r"(r[o + 10]), "=r"(r[o + 11]),       \
        "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), "=r"(r[o + 15]), "=r"(r[o + 16]), "=r"(r[o + 17]),   \
        "=r"(r[o + 18]), "=r"(r[o + 19]), "=r"(r[o + 20]), "=r"(r[o + 21]), "=r"(r[o + 22]), "=r"(r[o + 23]),   \
        "=r"(r[o + 24]), "=r"(r[o + 25]), "=r"(r[o + 26]), "=r"(r[o + 27]), "=r"(r[o + 28]), "=r"(r[o + 29]),   \
        "=r"(r[o + 30]), "=r"(r[o + 31])
// 64 columns (two x32 loads at ta0 and ta1) and one wait, in one statement.
__device__ __forceinline__ void tmem_ld64_sync(uint32_t ta0, uint32_t ta1, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, "
        "%44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, "
        "[%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : BSP_TMEM_REGS32_AT(r, 0), BSP_TMEM_REGS32_AT(r, 32)
        : "r"(ta0), "r"(ta1)
        : "memory");
}

// ----------------------------------------------------------- descriptors --

enum Swizzle : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), version 1, swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= (uint64_t)(swz & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
// ab_bf16: operand type (1 = bf16, 0 = fp16); a_mn / b_mn: 1 = MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int ab_bf16, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)ab_bf16 << 7) | ((uint32_t)ab_bf16 << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 2^x on the special-function unit (PTX ex2.approx; -inf -> +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^y for two values on the FMA pipe instead of the special-function unit
// (the attention softmax evaluates part of its exponentials here so that the
// two units share the work).  Method: Cody-Waite style range reduction
// y = j + f with j = round-to-nearest(y), found by adding and subtracting
// 1.5 * 2^23 (which leaves j in the low mantissa bits of the sum), and
// f in [-1/2, 1/2]; 2^f by the cubic 1 + f (c1 + f (c2 + f c3)), its
// coefficients fitted by iteratively reweighted least squares for the
// smallest maximum relative error over [-1/2, 1/2] with p(0) = 1 held (so
// integer y give exact powers of two; fit_exp2_poly.py in the package
// prints them); 2^j is added to the exponent field.  Maximum relative error
// 1.01e-4, far below the 2^-9 of the 16-bit P it feeds.  y is clamped to >= -125 (the exponent field stays normal), so -inf
// and very negative inputs give a value <= 2^-124.5 instead of 0: callers
// must not rely on exact zeros from masked entries.
__device__ __forceinline__ float2 exp2_poly2(float2 y) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    constexpr float c1 = 0.693282902f, c2 = 0.242210373f, c3 = 0.0550085828f;
    y.x = fmaxf(y.x, -125.0f);
    y.y = fmaxf(y.y, -125.0f);
    const float2 t = __fadd2_rn(y, make_float2(kMagic, kMagic));
    const float2 j = __fadd2_rn(t, make_float2(-kMagic, -kMagic));
    const float2 f = __fadd2_rn(y, make_float2(-j.x, -j.y));
    float2 p = __ffma2_rn(f, make_float2(c3, c3), make_float2(c2, c2));
    p = __ffma2_rn(p, f, make_float2(c1, c1));
    p = __ffma2_rn(p, f, make_float2(1.0f, 1.0f));
    return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                       __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------- conversions --

template <typename T> struct Pack2;
template <> struct Pack2<__nv_bfloat16> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};
template <> struct Pack2<__half> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

// two packed 16-bit values (element 0 in the low half) as floats
template <typename T> struct Unpack2;
template <> struct Unpack2<__nv_bfloat16> {
    __device__ __forceinline__ static float2 unpack(uint32_t u) {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
};
template <> struct Unpack2<__half> {
    __device__ __forceinline__ static float2 unpack(uint32_t u) {
        __half2 v = *reinterpret_cast<__half2*>(&u);
        return __half22float2(v);
    }
};

}  // namespace tc

// host: encode a 2-D tiled tensor map (row-major [rows][cols] of 2-byte
// elements, box [box_rows][box_cols], 128-byte swizzle unless given)
int make_tmap_2d(CUtensorMap* map, const void* base, int is_bf16, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, uint32_t box_cols, int swizzle_bytes);
// host: 2-D tiled tensor map of fp32 [rows][cols], box [box_rows][box_cols]
// (box_cols * 4 <= 128), 128-byte swizzle
int make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     uint32_t box_cols);
// host: 3-D tiled tensor map of 2-byte elements [d2][d1][d0] (d0 contiguous),
// box [1][box1][box0], swizzle 128 / 64 / 32 bytes or 0 (none)
int make_tmap_3d(CUtensorMap* map, const void* base, int is_bf16, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint32_t box0, uint32_t box1, int swizzle_bytes = 128);
// host: a row-major [rows][cols] matrix of 2-byte elements (cols a multiple of
// 64) seen as [cols/64 panels][rows][64]: one box of box_panels panels x
// box_rows rows lands panel after panel, 128-byte swizzled (else
// BSP_ERR_UNSUPPORTED)
int make_tmap_panels(CUtensorMap* map, const void* base, int is_bf16, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_panels);

}  // namespace bsp
