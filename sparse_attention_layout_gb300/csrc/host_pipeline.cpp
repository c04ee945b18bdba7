// Attention on host tensors with the transfers overlapped: the batch is cut
// into slices of whole batch entries, and each slice's host-to-device copies,
// kernel and device-to-host copy run on three streams of their own, through
// two device slots of a caller-owned workspace, so that the input copy of
// slice k + 1 and the output copy of slice k - 1 proceed while slice k is
// computed.  Independence of the (batch, head) pairs (every block-row's
// softmax and output touch one (batch, head) pair only) is what makes the
// slicing exact.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "bsp_internal.h"

struct HostPipe {
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    const void* last_ws = nullptr;  // workspace of the previous call
    size_t last_slot_bytes = 0;     // and the size of each of its two slots
    cudaEvent_t start = nullptr, done = nullptr, in[2] = {nullptr, nullptr}, out[2] = {nullptr, nullptr},
                freed[2] = {nullptr, nullptr};
};

namespace bsp {

void host_pipe_destroy(bsp_layout_s* L) {
    HostPipe* p = L->pipe;
    if (!p) return;
    for (cudaStream_t s : {p->h2d, p->comp, p->d2h})
        if (s) cudaStreamDestroy(s);
    for (cudaEvent_t e : {p->start, p->done, p->in[0], p->in[1], p->out[0], p->out[1], p->freed[0], p->freed[1]})
        if (e) cudaEventDestroy(e);
    delete p;
    L->pipe = nullptr;
}

namespace {

int pipe_of(bsp_layout_s* L, HostPipe** out) {
    if (!L->pipe) {
        HostPipe* p = new (std::nothrow) HostPipe();
        if (!p) return BSP_ERR_OOM;
        L->pipe = p;
        bool ok = true;
        for (cudaStream_t* s : {&p->h2d, &p->comp, &p->d2h})
            ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
        for (cudaEvent_t* e : {&p->start, &p->done, &p->in[0], &p->in[1], &p->out[0], &p->out[1], &p->freed[0],
                               &p->freed[1]})
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            host_pipe_destroy(L);
            return BSP_ERR_CUDA;
        }
    }
    *out = L->pipe;
    return BSP_OK;
}

size_t elt_size(int dtype) { return dtype == BSP_F32 ? 4 : 2; }

}  // namespace
}  // namespace bsp

extern "C" size_t bsp_attention_host_workspace(bsp_layout_t L, int dtype, int D, int z_slice) {
    if (!L || z_slice < 1 || D < 1) return 0;
    // two slots, each Q, K, V and O of z_slice batch entries
    return (size_t)2 * 4 * z_slice * L->H * (size_t)L->S * D * bsp::elt_size(dtype);
}

extern "C" int bsp_attention_host(bsp_layout_t L, int dtype, const void* Qh, const void* Kh, const void* Vh,
                                  void* Oh, int Z, int D, float scale, int mask_kind, const uint8_t* mask,
                                  void* workspace, size_t workspace_bytes, int flags, void* stream) {
    using namespace bsp;
    if (!L || !L->on_device || Z < 0 || D < 1 || (flags & ~BSP_HOST_RESERVED_WORKSPACE)) return BSP_ERR_INVALID_ARG;
    if (Z == 0) return BSP_OK;
    if (!Qh || !Kh || !Vh || !Oh || !workspace) return BSP_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255u) != 0) return BSP_ERR_ALIGNMENT;
    const size_t per_z = (size_t)L->H * L->S * D * elt_size(dtype);  // one tensor, one batch entry
    const size_t zs_fit = workspace_bytes / (2 * 4 * per_z);
    if (zs_fit < 1) return BSP_ERR_INVALID_ARG;
    // at least two slices when the batch allows it, so that copies overlap kernels
    const int zs = (int)std::min<size_t>(zs_fit, (size_t)std::max(1, Z / 2));
    HostPipe* p = nullptr;
    int rc = pipe_of(L, &p);
    if (rc) return rc;
    cudaStream_t caller = (cudaStream_t)stream;
    const size_t slot_bytes = 4 * (size_t)zs * per_z;
    char* ws = static_cast<char*>(workspace);
    auto fail = [&]() { cudaGetLastError(); return BSP_ERR_CUDA; };
    // kernels and output copies after the work already queued on the caller's
    // stream; input copies too, unless the workspace is reserved for this
    // handle and was the previous call's, cut into slots of the same size:
    // then slot k covers exactly the bytes of the previous call's slot k, so
    // the input copies only wait (below) for that slot to be free and may
    // overlap the previous call's tail.  Slots of another size (another batch
    // slicing, head size or dtype) could overlap the previous call's other
    // slot, so such a call waits for everything queued before it.
    const bool early = (flags & BSP_HOST_RESERVED_WORKSPACE) && p->last_ws == workspace &&
                       p->last_slot_bytes == slot_bytes;
    if (cudaEventRecord(p->start, caller) != cudaSuccess) return fail();
    for (cudaStream_t s : {p->h2d, p->comp, p->d2h}) {
        if (early && s == p->h2d) continue;
        if (cudaStreamWaitEvent(s, p->start, 0) != cudaSuccess) return fail();
    }
    p->last_ws = workspace;
    p->last_slot_bytes = slot_bytes;
    const int nsl = (Z + zs - 1) / zs;
    for (int k = 0; k < nsl; ++k) {
        const int z0 = k * zs, nz = std::min(zs, Z - z0), slot = k & 1;
        const size_t off = (size_t)z0 * per_z, bytes = (size_t)nz * per_z;
        char* q = ws + slot * slot_bytes;
        char* kk = q + (size_t)zs * per_z;
        char* v = kk + (size_t)zs * per_z;
        char* o = v + (size_t)zs * per_z;
        // inputs, once the slot's previous output has been copied out (the
        // previous call's, for the first two slices of an early start)
        if ((k >= 2 || early) && cudaStreamWaitEvent(p->h2d, p->freed[slot], 0) != cudaSuccess) return fail();
        if (cudaMemcpyAsync(q, (const char*)Qh + off, bytes, cudaMemcpyHostToDevice, p->h2d) != cudaSuccess ||
            cudaMemcpyAsync(kk, (const char*)Kh + off, bytes, cudaMemcpyHostToDevice, p->h2d) != cudaSuccess ||
            cudaMemcpyAsync(v, (const char*)Vh + off, bytes, cudaMemcpyHostToDevice, p->h2d) != cudaSuccess ||
            cudaEventRecord(p->in[slot], p->h2d) != cudaSuccess)
            return fail();
        // the kernel on this slice
        if (cudaStreamWaitEvent(p->comp, p->in[slot], 0) != cudaSuccess) return fail();
        rc = bsp_attention(L, dtype, q, kk, v, o, nz, D, scale, mask_kind, mask, p->comp);
        if (rc != BSP_OK) {
            cudaGetLastError();
            return rc;
        }
        if (cudaEventRecord(p->out[slot], p->comp) != cudaSuccess) return fail();
        // the output
        if (cudaStreamWaitEvent(p->d2h, p->out[slot], 0) != cudaSuccess ||
            cudaMemcpyAsync((char*)Oh + off, o, bytes, cudaMemcpyDeviceToHost, p->d2h) != cudaSuccess ||
            cudaEventRecord(p->freed[slot], p->d2h) != cudaSuccess)
            return fail();
    }
    // the last output copy follows every kernel and copy of the call
    if (cudaEventRecord(p->done, p->d2h) != cudaSuccess || cudaStreamWaitEvent(caller, p->done, 0) != cudaSuccess)
        return fail();
    return BSP_OK;
}
