// Dispatch of the fused tensor-core attention kernel by dtype.
#include "bsp_internal.h"

namespace bsp {

int launch_attention_tc_bf16(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, int Z,
                             int D, float scale, int kind, const uint8_t* mask, cudaStream_t s);
int launch_attention_tc_f16(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, int Z,
                            int D, float scale, int kind, const uint8_t* mask, cudaStream_t s);

int launch_attention_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K, const void* V, void* O,
                        int Z, int D, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if ((uint64_t)Z * L->H * L->S >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;  // TMA coordinates are int32
    if (dtype == BSP_BF16) return launch_attention_tc_bf16(L, Q, K, V, O, Z, D, scale, kind, mask, s);
    if (dtype == BSP_F16) return launch_attention_tc_f16(L, Q, K, V, O, Z, D, scale, kind, mask, s);
    return BSP_ERR_UNSUPPORTED;
}

}  // namespace bsp
