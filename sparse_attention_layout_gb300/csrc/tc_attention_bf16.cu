// bf16 instantiations of the fused tensor-core attention kernel.
#include "tc_attention.cuh"

namespace bsp {

int launch_attention_tc_bf16(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse,
                              int Z, int D, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    return attn::by_block<__nv_bfloat16, false>(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
}

}  // namespace bsp
