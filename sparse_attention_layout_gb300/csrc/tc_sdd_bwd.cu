// Launcher of the tensor-core SDD in its fused softmax-backward mode (the
// kernel: tc_sdd.cuh, MODE 2): dX = scale P .* (dP - rowsum(P .* dP)) with
// dP = dO V^T on the layout, for blocks of 64 and 128.
#include "tc_sdd.cuh"

namespace bsp {

using sddk::SddExtra;
using sddk::sdd_by_dtype;
using sddk::sdd_tc_shape;

int launch_sdd_softmax_bwd_tc(const bsp_layout_s* L, int dtype, const void* dO, const void* V, const void* P,
                              void* dX, int Z, int D, float scale, cudaStream_t s) {
    if (!sdd_tc_shape(L, Z, D, 0, 1) || L->B < 64) return BSP_ERR_UNSUPPORTED;
    SddExtra e;
    e.P = P;
    e.scale = scale;
    return sdd_by_dtype<2>(L, dtype, dO, V, dX, Z, D, 0, 1, e, s);
}

}  // namespace bsp
