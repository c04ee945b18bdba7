// Launcher of the tensor-core SDD in its one-pass attention-backward mode (the
// kernel: tc_sdd.cuh, MODE 3): on the layout, with S = Q K^T and dP = dO V^T,
//     P  = exp(scale S - lse)                          (the forward's softmax)
//     dX = scale P .* (dP - rowsum(dO .* O))           (its backward)
// written together from one pass over the row tiles.  rowsum(dO .* O) equals
// rowsum(P .* dP) because O = P V, and the forward's log-sum-exp makes the
// softmax a single exponential per entry.  The second launcher (MODE 4) also
// accumulates dQ = dX K over each row tile's steps (head size 128, blocks of 64
// and 128).
#include "tc_sdd.cuh"

namespace bsp {

using sddk::SddExtra;
using sddk::sdd_by_dtype;
using sddk::sdd_tc_shape;

int launch_sdd_attention_bwd_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K, const void* dO,
                                const void* V, const float* lse, const float* dvec, void* P, void* dX, int Z, int D,
                                float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if (!sdd_tc_shape(L, Z, D, 0, 1)) return BSP_ERR_UNSUPPORTED;
    SddExtra e;
    e.c2 = scale * kLog2e;
    e.kind = kind;
    e.mask = mask;
    e.scale = scale;
    e.lse = lse;
    e.dvec = dvec;
    e.A2 = dO;
    e.B2 = V;
    e.C2 = P;
    return sdd_by_dtype<3>(L, dtype, Q, K, dX, Z, D, 0, 1, e, s);
}

int launch_sdd_attention_bwd_dq_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K, const void* dO,
                                   const void* V, const float* lse, const float* dvec, void* P, void* dX, void* dQ,
                                   int Z, int D, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if (!sdd_tc_shape(L, Z, D, 0, 1) || D != 128 || L->B < 64) return BSP_ERR_UNSUPPORTED;
    SddExtra e;
    e.c2 = scale * kLog2e;
    e.kind = kind;
    e.mask = mask;
    e.scale = scale;
    e.lse = lse;
    e.dvec = dvec;
    e.A2 = dO;
    e.B2 = V;
    e.C2 = P;
    e.D2 = dQ;
    return sdd_by_dtype<4>(L, dtype, Q, K, dX, Z, D, 0, 1, e, s);
}

}  // namespace bsp
