// Placeholder tensor-core launchers (replaced as the tcgen05 kernels land).
#include "bsp_internal.h"

namespace bsp {
int launch_sdd_tc(const bsp_layout_s*, int, const void*, const void*, void*, int, int, int, int,
                  cudaStream_t) { return BSP_ERR_UNSUPPORTED; }
int launch_dsd_tc(const bsp_layout_s*, int, const void*, const void*, void*, int, int, int, int,
                  cudaStream_t) { return BSP_ERR_UNSUPPORTED; }
int launch_dds_tc(const bsp_layout_s*, int, const void*, const void*, void*, int, int, int, int,
                  cudaStream_t) { return BSP_ERR_UNSUPPORTED; }
}  // namespace bsp
