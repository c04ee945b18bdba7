// C ABI entry points of libbsp: argument validation, dispatch between the
// tensor-core and CUDA-core kernels, status reporting.
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "bsp_internal.h"

namespace bsp {

int sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

}  // namespace bsp

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool valid_dtype(int d) { return d == BSP_F32 || d == BSP_BF16 || d == BSP_F16; }
bool valid_kind(int k) { return k == BSP_MASK_NONE || k == BSP_MASK_DENSE || k == BSP_MASK_DIAG_CAUSAL; }

// Common checks for a compute call: a device handle, the right device, a
// valid dtype, non-NULL 16-byte-aligned tensors (any pointer may be NULL when
// the batch is empty, Z == 0).
int check_common(bsp_layout_t L, int dtype, int Z, std::initializer_list<const void*> ptrs) {
    if (!L || !L->on_device) return BSP_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || Z < 0) return BSP_ERR_INVALID_ARG;
    if (Z == 0) return BSP_OK;
    for (const void* p : ptrs)
        if (!p) return BSP_ERR_INVALID_ARG;
    for (const void* p : ptrs)
        if (!aligned16(p)) return BSP_ERR_ALIGNMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSP_ERR_CUDA;
    if (dev != L->device) return BSP_ERR_INVALID_ARG;
    return BSP_OK;
}

// Environment switch (read at every call) that forces the CUDA-core kernels;
// the tests use it to cover both paths in one process.
bool force_simt() {
    const char* e = std::getenv("BSP_FORCE_SIMT");
    return e && e[0] == '1';
}

}  // namespace

extern "C" int bsp_sdd(bsp_layout_t L, int dtype, const void* A, const void* B, void* C, int Z,
                       int K, int trans_a, int trans_b, void* stream) {
    int rc = check_common(L, dtype, Z, {A, B, C});
    if (rc) return rc;
    if (Z < 0 || K < 1 || (trans_a & ~1) || (trans_b & ~1)) return BSP_ERR_INVALID_ARG;
    if (Z == 0 || L->nnz == 0) return BSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (!force_simt()) {
        rc = bsp::launch_sdd_tc(L, dtype, A, B, C, Z, K, trans_a, trans_b, s);
        if (rc != BSP_ERR_UNSUPPORTED) return rc;
    }
    return bsp::launch_sdd_simt(L, dtype, A, B, C, Z, K, trans_a, trans_b, s);
}

extern "C" int bsp_sdd_softmax(bsp_layout_t L, int dtype, const void* A, const void* B, void* P, int Z, int K,
                               int trans_a, int trans_b, float scale, int mask_kind, const uint8_t* mask,
                               void* stream) {
    int rc = check_common(L, dtype, Z, {A, B, P});
    if (rc) return rc;
    if (Z < 0 || K < 1 || (trans_a & ~1) || (trans_b & ~1) || !valid_kind(mask_kind) || !(scale > 0.f) ||
        scale > 3.0e38f)
        return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && !mask) return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && ((uintptr_t)mask & 15u)) return BSP_ERR_ALIGNMENT;
    if (Z == 0 || L->nnz == 0) return BSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const uint8_t* m = mask_kind == BSP_MASK_DENSE ? mask : nullptr;
    if (!force_simt()) {
        rc = bsp::launch_sdd_softmax_tc(L, dtype, A, B, P, Z, K, trans_a, trans_b, scale, mask_kind, m, s);
        if (rc != BSP_ERR_UNSUPPORTED) return rc;
    }
    // the two steps one after the other (scores through HBM, softmax in place)
    rc = bsp_sdd(L, dtype, A, B, P, Z, K, trans_a, trans_b, stream);
    if (rc) return rc;
    return bsp::launch_softmax(L, dtype, P, P, Z, scale, mask_kind, m, s);
}

extern "C" int bsp_dsd(bsp_layout_t L, int dtype, const void* A_sp, const void* B, void* C, int Z,
                       int N, int trans_a, int trans_b, void* stream) {
    int rc = check_common(L, dtype, Z, {A_sp, B, C});
    if (rc) return rc;
    if (Z < 0 || N < 1 || (trans_a & ~1) || (trans_b & ~1)) return BSP_ERR_INVALID_ARG;
    if (Z == 0) return BSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (!force_simt()) {
        rc = bsp::launch_dsd_group_tc(L, dtype, A_sp, B, C, Z, N, trans_a, trans_b, s);
        if (rc != BSP_ERR_UNSUPPORTED) return rc;
    }
    return bsp::launch_dsd_simt(L, dtype, A_sp, B, C, Z, N, trans_a, trans_b, s);
}

extern "C" int bsp_dds(bsp_layout_t L, int dtype, const void* A, const void* B_sp, void* C, int Z,
                       int M, int trans_a, int trans_b, void* stream) {
    int rc = check_common(L, dtype, Z, {A, B_sp, C});
    if (rc) return rc;
    if (Z < 0 || M < 1 || (trans_a & ~1) || (trans_b & ~1)) return BSP_ERR_INVALID_ARG;
    if (Z == 0) return BSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (!force_simt()) {
        rc = bsp::launch_dds_group_tc(L, dtype, A, B_sp, C, Z, M, trans_a, trans_b, s);
        if (rc != BSP_ERR_UNSUPPORTED) return rc;
    }
    return bsp::launch_dds_simt(L, dtype, A, B_sp, C, Z, M, trans_a, trans_b, s);
}

extern "C" int bsp_softmax(bsp_layout_t L, int dtype, const void* X, void* Y, int Z, float scale,
                           int mask_kind, const uint8_t* mask, void* stream) {
    int rc = check_common(L, dtype, Z, {X, Y});
    if (rc) return rc;
    if (Z < 0 || !valid_kind(mask_kind) || !(scale > 0.f) || scale > 3.0e38f) return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && !mask) return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && ((uintptr_t)mask & 15u)) return BSP_ERR_ALIGNMENT;
    if (Z == 0 || L->nnz == 0) return BSP_OK;
    return bsp::launch_softmax(L, dtype, X, Y, Z, scale, mask_kind,
                               mask_kind == BSP_MASK_DENSE ? mask : nullptr, (cudaStream_t)stream);
}

namespace {
int attention_impl(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V, void* O, float* lse,
                   int Z, int D, float scale, int mask_kind, const uint8_t* mask, void* stream) {
    int rc = check_common(L, dtype, Z, {Q, K, V, O});
    if (rc) return rc;
    if (Z < 0 || D < 16 || D > 128 || D % 16 || !valid_kind(mask_kind) || !(scale > 0.f) ||
        scale > 3.0e38f)
        return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && !mask) return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && ((uintptr_t)mask & 15u)) return BSP_ERR_ALIGNMENT;
    if (Z == 0) return BSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const uint8_t* m = mask_kind == BSP_MASK_DENSE ? mask : nullptr;
    if (!force_simt()) {
        rc = bsp::launch_attention_tc(L, dtype, Q, K, V, O, lse, Z, D, scale, mask_kind, m, s);
        if (rc != BSP_ERR_UNSUPPORTED) return rc;
    }
    return bsp::launch_attention_simt(L, dtype, Q, K, V, O, lse, Z, D, scale, mask_kind, m, s);
}
}  // namespace

extern "C" int bsp_attention(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V,
                             void* O, int Z, int D, float scale, int mask_kind, const uint8_t* mask,
                             void* stream) {
    return attention_impl(L, dtype, Q, K, V, O, nullptr, Z, D, scale, mask_kind, mask, stream);
}

extern "C" int bsp_attention_lse(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V, void* O,
                                 float* lse, int Z, int D, float scale, int mask_kind, const uint8_t* mask,
                                 void* stream) {
    if (Z > 0 && !lse) return BSP_ERR_INVALID_ARG;
    if (!aligned16(lse)) return BSP_ERR_ALIGNMENT;
    return attention_impl(L, dtype, Q, K, V, O, lse, Z, D, scale, mask_kind, mask, stream);
}

extern "C" int bsp_status_check(bsp_layout_t L, void* stream) {
    if (!L || !L->on_device) return BSP_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BSP_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, L->view.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BSP_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(L->view.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return BSP_ERR_CUDA;
    }
    return word;
}

extern "C" int bsp_diag_wait_limit(bsp_layout_t L, uint64_t wait_ns, int inject) {
    if (!L || !L->on_device) return BSP_ERR_INVALID_ARG;
    if (inject & ~(kInjectSkipFirstQ | kInjectBadColumn)) return BSP_ERR_INVALID_ARG;
    L->view.wait_ns = wait_ns ? wait_ns : kDefaultWaitNs;
    L->view.inject = inject;
    return BSP_OK;
}

extern "C" const char* bsp_status_string(int status) {
    switch (status) {
        case BSP_OK: return "ok";
        case BSP_ERR_INVALID_ARG: return "invalid argument";
        case BSP_ERR_UNSUPPORTED: return "unsupported combination";
        case BSP_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
        case BSP_ERR_OOM: return "out of memory";
        case BSP_ERR_CUDA: return "CUDA runtime error";
        case BSP_ERR_TIMEOUT: return "device wait timed out";
        case BSP_ERR_DEVICE_CHECK: return "device bounds check failed";
        default: return "unknown status";
    }
}

extern "C" const char* bsp_version(void) { return "libbsp 0.1 (sm_103a)"; }

extern "C" int bsp_softmax_backward(bsp_layout_t L, int dtype, const void* Y, const void* dY, void* dX, int Z,
                                    float scale, void* stream) {
    int rc = check_common(L, dtype, Z, {Y, dY, dX});
    if (rc) return rc;
    if (!(scale > 0.f) || scale > 3.0e38f) return BSP_ERR_INVALID_ARG;
    if (Z == 0 || L->nnz == 0) return BSP_OK;
    return bsp::launch_softmax_backward(L, dtype, Y, dY, dX, Z, scale, (cudaStream_t)stream);
}

namespace {

// The recomputing chain: P = softmax(scale Q K^T) on the layout, as the forward
// computes it (one fused pass: the scores never reach memory), dV = P^T dO,
// dX = scale P .* (dP - rowsum(P .* dP)) with dP = dO V^T, dQ = dX K,
// dK = dX^T Q; P and dX in the workspaces.
int backward_chain(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V, const void* dO, void* dQ,
                   void* dK, void* dV, int Z, int D, float scale, int mask_kind, const uint8_t* mask, void* P_ws,
                   void* dP_ws, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    int rc = bsp_sdd_softmax(L, dtype, Q, K, P_ws, Z, D, 0, 1, scale, mask_kind, mask, stream);
    if (rc) return rc;
    if ((rc = bsp_dsd(L, dtype, P_ws, dO, dV, Z, D, 1, 0, stream))) return rc;
    // dX: one fused pass on the tensor cores (dP stays on chip), else dP
    // through memory and the softmax backward in place
    rc = force_simt() ? BSP_ERR_UNSUPPORTED
                      : bsp::launch_sdd_softmax_bwd_tc(L, dtype, dO, V, P_ws, dP_ws, Z, D, scale, s);
    if (rc == BSP_ERR_UNSUPPORTED) {
        if ((rc = bsp_sdd(L, dtype, dO, V, dP_ws, Z, D, 0, 1, stream))) return rc;
        rc = bsp_softmax_backward(L, dtype, P_ws, dP_ws, dP_ws, Z, scale, stream);
    }
    if (rc) return rc;
    if ((rc = bsp_dsd(L, dtype, dP_ws, K, dQ, Z, D, 0, 0, stream))) return rc;
    return bsp_dsd(L, dtype, dP_ws, Q, dK, Z, D, 1, 0, stream);
}

// The backward from the forward's O and rows' log-sum-exp (16-bit types,
// arguments checked, Z > 0, a layout with blocks): shapes the one-pass
// kernels do not cover take the recomputing chain.  O may live in dV's
// memory and lse in dK's beyond its first Z H S floats: O is read only by
// the row dot, lse only by the one-pass kernel, both before dV and dK are
// written.
int backward_from_stats(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* lse, void* dQ, void* dK, void* dV, int Z, int D, float scale,
                        int mask_kind, const uint8_t* mask, void* P_ws, void* dP_ws, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    const uint8_t* m = mask_kind == BSP_MASK_DENSE ? mask : nullptr;
    // the rows' dO . O (= rowsum(P .* dP), as O = P V) go to dK's memory first
    // (fp32 [Z][H][S] fits in any [Z][H][S][D] tensor of D >= 2); dK receives
    // its own values last
    float* dvec = static_cast<float*>(dK);
    int rc = bsp::launch_row_dot(dtype, dO, O, dvec, (int64_t)Z * L->H * L->S, D, s);
    if (rc) return rc;
    // P = exp(scale Q K^T - lse) and dX = scale P .* (dO V^T - dvec) on the
    // layout, and dQ = dX K accumulated over each row tile's steps: one pass
    // (head size 128, blocks of 64 and 128); else P and dX in one pass and dQ
    // by a DSD
    rc = bsp::launch_sdd_attention_bwd_dq_tc(L, dtype, Q, K, dO, V, lse, dvec, P_ws, dP_ws, dQ, Z, D, scale,
                                             mask_kind, m, s);
    const bool dq_done = rc == BSP_OK;
    if (rc == BSP_ERR_UNSUPPORTED)
        rc = bsp::launch_sdd_attention_bwd_tc(L, dtype, Q, K, dO, V, lse, dvec, P_ws, dP_ws, Z, D, scale, mask_kind,
                                              m, s);
    if (rc == BSP_ERR_UNSUPPORTED)
        return backward_chain(L, dtype, Q, K, V, dO, dQ, dK, dV, Z, D, scale, mask_kind, mask, P_ws, dP_ws, stream);
    if (rc) return rc;
    // dV = P^T dO,  dQ = dX K,  dK = dX^T Q
    if ((rc = bsp_dsd(L, dtype, P_ws, dO, dV, Z, D, 1, 0, stream))) return rc;
    if (!dq_done && (rc = bsp_dsd(L, dtype, dP_ws, K, dQ, Z, D, 0, 0, stream))) return rc;
    return bsp_dsd(L, dtype, dP_ws, Q, dK, Z, D, 1, 0, stream);
}

}  // namespace

extern "C" int bsp_attention_backward(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V,
                                      const void* dO, void* dQ, void* dK, void* dV, int Z, int D, float scale,
                                      int mask_kind, const uint8_t* mask, void* P_ws, void* dP_ws,
                                      void* stream) {
    int rc = check_common(L, dtype, Z, {Q, K, V, dO, dQ, dK, dV});
    if (rc) return rc;
    if (D < 16 || D > 128 || D % 16 || !valid_kind(mask_kind) || !(scale > 0.f) || scale > 3.0e38f)
        return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && !mask) return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && ((uintptr_t)mask & 15u)) return BSP_ERR_ALIGNMENT;
    if (Z == 0) return BSP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (L->nnz == 0) {  // nothing attends to anything: every gradient is 0
        const size_t bytes = (size_t)Z * L->H * L->S * D * (dtype == BSP_F32 ? 4 : 2);
        for (void* p : {dQ, dK, dV})
            if (cudaMemsetAsync(p, 0, bytes, s) != cudaSuccess) return BSP_ERR_CUDA;
        return BSP_OK;
    }
    if (!P_ws || !dP_ws) return BSP_ERR_INVALID_ARG;
    if (!aligned16(P_ws) || !aligned16(dP_ws)) return BSP_ERR_ALIGNMENT;
    if (dtype != BSP_F32 && !force_simt() && (D == 64 || D == 128)) {
        // 16-bit types, head sizes of the fused tensor-core forward: it
        // recomputes O (into dV's memory) and the rows' log-sum-exp (into
        // dK's, after the Z H S floats the row dot takes), and the backward
        // from those statistics follows
        float* lse = reinterpret_cast<float*>(static_cast<char*>(dK) + (size_t)Z * L->H * L->S * sizeof(float));
        if ((rc = attention_impl(L, dtype, Q, K, V, dV, lse, Z, D, scale, mask_kind, mask, stream))) return rc;
        return backward_from_stats(L, dtype, Q, K, V, dV, dO, lse, dQ, dK, dV, Z, D, scale, mask_kind, mask, P_ws,
                                   dP_ws, stream);
    }
    return backward_chain(L, dtype, Q, K, V, dO, dQ, dK, dV, Z, D, scale, mask_kind, mask, P_ws, dP_ws, stream);
}

extern "C" int bsp_attention_backward_lse(bsp_layout_t L, int dtype, const void* Q, const void* K, const void* V,
                                          const void* O, const void* dO, const float* lse, void* dQ, void* dK,
                                          void* dV, int Z, int D, float scale, int mask_kind, const uint8_t* mask,
                                          void* P_ws, void* dP_ws, void* stream) {
    int rc = check_common(L, dtype, Z, {Q, K, V, O, dO, dQ, dK, dV});
    if (rc) return rc;
    if (D < 16 || D > 128 || D % 16 || !valid_kind(mask_kind) || !(scale > 0.f) || scale > 3.0e38f)
        return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && !mask) return BSP_ERR_INVALID_ARG;
    if (mask_kind == BSP_MASK_DENSE && ((uintptr_t)mask & 15u)) return BSP_ERR_ALIGNMENT;
    if (Z > 0 && (!lse || !O)) return BSP_ERR_INVALID_ARG;
    if (!aligned16(lse)) return BSP_ERR_ALIGNMENT;
    if (Z == 0 || L->nnz == 0 || dtype == BSP_F32 || force_simt())  // the chain recomputes what it needs
        return bsp_attention_backward(L, dtype, Q, K, V, dO, dQ, dK, dV, Z, D, scale, mask_kind, mask, P_ws, dP_ws,
                                      stream);
    if (!P_ws || !dP_ws) return BSP_ERR_INVALID_ARG;
    if (!aligned16(P_ws) || !aligned16(dP_ws)) return BSP_ERR_ALIGNMENT;
    return backward_from_stats(L, dtype, Q, K, V, O, dO, lse, dQ, dK, dV, Z, D, scale, mask_kind, mask, P_ws, dP_ws,
                               stream);
}
