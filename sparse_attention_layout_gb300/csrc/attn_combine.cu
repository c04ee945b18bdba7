// Merging the pieces of cut attention tiles (schedule.cpp): every piece left,
// per query row, the output accumulated over its steps, O_p = sum_j
// 2^(s_j - m_p) v_j, its reference max m_p and its sum l_p = sum_j
// 2^(s_j - m_p) (scores s in log2 units).  The row's result is the online
// softmax recurrence of the Triton-Puzzles blog, Puzzle 9 "Simple
// FlashAttention", applied across the pieces in piece order:
//     M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  O = sum_p O_p 2^(m_p - M) / L,
// with pieces that kept nothing (m_p = -inf, l_p = 0) weighing 0 and rows with
// nothing kept anywhere written as 0.  One CTA per cut tile, a thread per
// (row, 4 columns); the loads of a row's pieces are coalesced across its
// threads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "bsp_internal.h"
#include "common.cuh"

namespace bsp {
namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ void store4(float* o, float4 v) { *reinterpret_cast<float4*>(o) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* o, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(o) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}
__device__ __forceinline__ void store4(__half* o, float4 v) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(o) = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

template <typename T>
__global__ void __launch_bounds__(kCombineThreads)
attn_combine_kernel(const int4* __restrict__ comb, const float* __restrict__ ws, T* __restrict__ O,
                    float* __restrict__ lse, int H, int S, int D, int ngroups) {
    const int4 c = comb[blockIdx.x];  // tile, batch entry, first slot, pieces
    const int tile = c.x, z = c.y, slot0 = c.z, np = c.w;
    const int h = tile / ngroups, gq = tile % ngroups;
    const int tpr = D / 4;  // threads per row
    const int d0 = (threadIdx.x % tpr) * 4;
    for (int r = threadIdx.x / tpr; r < kPartRows; r += kCombineThreads / tpr) {
        const int rseq = gq * kPartRows + r;
        if (rseq >= S) break;
        float M = -INFINITY;
        for (int p = 0; p < np; ++p) M = fmaxf(M, ws[(size_t)(slot0 + p) * kPartFloats + kPartRows * kPartMaxD + r]);
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int p = 0; p < np; ++p) {
                const float* pw = ws + (size_t)(slot0 + p) * kPartFloats;
                const float mp = pw[kPartRows * kPartMaxD + r];
                if (mp == -INFINITY) continue;  // the piece kept nothing of this row
                const float w = exp2f(mp - M);
                Ls += pw[kPartRows * kPartMaxD + kPartRows + r] * w;
                const float4 o = *reinterpret_cast<const float4*>(pw + (size_t)r * D + d0);
                acc.x += o.x * w;
                acc.y += o.y * w;
                acc.z += o.z * w;
                acc.w += o.w * w;
            }
        }
        const float inv = Ls > 0.f ? 1.0f / Ls : 0.f;
        // the row's log-sum-exp (natural log) from the merged statistics
        if (lse && d0 == 0) lse[((int64_t)z * H + h) * S + rseq] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        store4(O + (((int64_t)z * H + h) * S + rseq) * D + d0, acc);
    }
}

// whether work enqueued on s now goes into a graph being captured (then the
// workspace's cross-stream event is left alone: the graph orders its own work)
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return st != cudaStreamCaptureStatusNone;
}

}  // namespace

int launch_attention_combine(const bsp_layout_s* L, int dtype, const AttnSchedule& sc, void* O, float* lse, int D,
                             cudaStream_t s) {
    if (sc.n_split == 0) return BSP_OK;
    if (D % 4 != 0 || D > kPartMaxD || kCombineThreads % (D / 4) != 0) return BSP_ERR_UNSUPPORTED;
    const dim3 grid(sc.n_split), block(kCombineThreads);
    if (dtype == BSP_BF16)
        attn_combine_kernel<<<grid, block, 0, s>>>(sc.combine, sc.ws, (__nv_bfloat16*)O, lse, L->H, L->S, D, L->ngroups);
    else if (dtype == BSP_F16)
        attn_combine_kernel<<<grid, block, 0, s>>>(sc.combine, sc.ws, (__half*)O, lse, L->H, L->S, D, L->ngroups);
    else
        attn_combine_kernel<<<grid, block, 0, s>>>(sc.combine, sc.ws, (float*)O, lse, L->H, L->S, D, L->ngroups);
    return cudaGetLastError() == cudaSuccess ? BSP_OK : BSP_ERR_CUDA;
}

int attn_schedule_begin(bsp_layout_s* L, int dtype, int Z, cudaStream_t s, AttnSchedule* sc) {
    const int rc = tile_schedule(L, Z, sm_count(), attn_force_cap(dtype), sc);
    if (rc || sc->n_split == 0) return rc;
    // the workspace of cut tiles: one launch (kernel + combine) at a time,
    // enqueued under the schedule's lock, each after the previous one's
    // combine on whatever stream that ran
    sc->mu->lock();
    if (!capturing(s) && cudaStreamWaitEvent(s, sc->done, 0) != cudaSuccess) {
        cudaGetLastError();
        sc->mu->unlock();
        return BSP_ERR_CUDA;
    }
    return BSP_OK;
}

int attn_schedule_end(const bsp_layout_s* L, int dtype, const AttnSchedule& sc, void* O, float* lse, int D,
                      cudaStream_t s, int rc) {
    if (sc.n_split == 0) return rc;
    if (rc == BSP_OK) rc = launch_attention_combine(L, dtype, sc, O, lse, D, s);
    if (rc == BSP_OK && !capturing(s) && cudaEventRecord(sc.done, s) != cudaSuccess) {
        cudaGetLastError();
        rc = BSP_ERR_CUDA;
    }
    sc.mu->unlock();
    return rc;
}

}  // namespace bsp
