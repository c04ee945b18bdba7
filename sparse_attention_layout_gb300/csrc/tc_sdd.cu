// Launchers of the tensor-core SDD in its plain and softmax modes (the kernel:
// tc_sdd.cuh).
#include "tc_sdd.cuh"

namespace bsp {

using sddk::SddExtra;
using sddk::sdd_by_dtype;
using sddk::sdd_tc_shape;

int launch_sdd_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z, int K, int ta,
                  int tb, cudaStream_t s) {
    if (!sdd_tc_shape(L, Z, K, ta, tb)) return BSP_ERR_UNSUPPORTED;
    return sdd_by_dtype<0>(L, dtype, A, B, C, Z, K, ta, tb, SddExtra{}, s);
}

int launch_sdd_softmax_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* P, int Z, int K,
                          int ta, int tb, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if (!sdd_tc_shape(L, Z, K, ta, tb)) return BSP_ERR_UNSUPPORTED;
    SddExtra e;
    e.c2 = scale * kLog2e;
    e.kind = kind;
    e.mask = mask;
    return sdd_by_dtype<1>(L, dtype, A, B, P, Z, K, ta, tb, e, s);
}

}  // namespace bsp
