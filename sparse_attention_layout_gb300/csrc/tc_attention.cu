// Dispatch of the fused tensor-core attention kernel by dtype, and by whether
// the layout's key blocks come from its affine description or its tables.
#include <cstdlib>

#include "bsp_internal.h"

namespace bsp {

#define BSP_ATTN_LAUNCHER(name)                                                                                   \
    int name(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z, int D, float scale, \
             int kind, const uint8_t* mask, cudaStream_t s);
BSP_ATTN_LAUNCHER(launch_attention_tc_bf16)
BSP_ATTN_LAUNCHER(launch_attention_tc_f16)
BSP_ATTN_LAUNCHER(launch_attention_tc_bf16_geo)
BSP_ATTN_LAUNCHER(launch_attention_tc_f16_geo)
#undef BSP_ATTN_LAUNCHER
int launch_attention_tc_tf32(const bsp_layout_s* L, const void* Q, const void* K, const void* V, void* O, float* lse, int Z,
                             int D, float scale, int kind, const uint8_t* mask, cudaStream_t s);

namespace {
// BSP_GEOMETRY=1: layouts whose every head has an affine description take
// their key blocks from it.  Off by default: the table loads it replaces are
// issued ahead of their use, and the variant measured slower (banded
// workload 1218 vs 1238 TFLOP/s, strided 850 vs 958).
bool geometry_on() {
    const char* e = std::getenv("BSP_GEOMETRY");
    return e && e[0] == '1';
}
}  // namespace

int launch_attention_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K, const void* V, void* O,
                        float* lse, int Z, int D, float scale, int kind, const uint8_t* mask, cudaStream_t s) {
    if ((uint64_t)Z * L->H * L->S >= (1ull << 31)) return BSP_ERR_UNSUPPORTED;  // TMA coordinates are int32
    const bool geo = L->view.geo != nullptr && geometry_on();
    if (dtype == BSP_BF16)
        return (geo ? launch_attention_tc_bf16_geo : launch_attention_tc_bf16)(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
    if (dtype == BSP_F16)
        return (geo ? launch_attention_tc_f16_geo : launch_attention_tc_f16)(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
    // fp32: the three-term tf32 split on the tensor cores (head size 64)
    if (dtype == BSP_F32) return launch_attention_tc_tf32(L, Q, K, V, O, lse, Z, D, scale, kind, mask, s);
    return BSP_ERR_UNSUPPORTED;
}

}  // namespace bsp
