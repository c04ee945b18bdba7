// bsp_softmax_noalloc: the block-sparse row softmax for callers that cannot
// allocate device memory.
//
// Some hosts own every byte of device memory themselves (a serving runtime
// that reserves the GPU for its own pool at start-up, a plugin interface that
// hands over only the input and output buffers, a real-time loop where an
// allocation and its implicit synchronisation are not acceptable).  Those
// callers cannot create a compiled layout handle, because bsp_layout_compile
// allocates the device copy of the layout's tables.  This entry point builds
// the tables on the host for every call and places them in a fixed array of
// device memory that the library declares at file scope, so no call allocates.
//
// Costs and limits: every GPU that loads the library holds kScratchBytes of
// device memory until the process exits; the tables of one call must fit in
// it; the tables are rebuilt and uploaded on every call; all calls share the
// array, so calls that overlap on the GPU (for example on two streams) race.
#include <mutex>

#include "bsp_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

// In host code `g_scratch` only names a host-side stand-in for the array; the
// device address comes from cudaGetSymbolAddress (once per device, below).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  The first call on a
// device performs the lookup with that device current; the address is kept
// for the life of the process (a reset of the device's context, after which
// the module is loaded again elsewhere, is not supported).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return BSP_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return BSP_OK;
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

extern "C" int bsp_softmax_noalloc(const uint8_t* layout, int H, int nb, int block, int dtype, const void* X,
                                   void* Y, int Z, float scale, int mask_kind, const uint8_t* mask,
                                   void* stream) {
    if (dtype != BSP_F32 && dtype != BSP_BF16 && dtype != BSP_F16) return BSP_ERR_INVALID_ARG;
    if (Z < 0 || !(scale > 0.f) || scale > 3.0e38f) return BSP_ERR_INVALID_ARG;
    if (mask_kind != BSP_MASK_NONE && mask_kind != BSP_MASK_DENSE && mask_kind != BSP_MASK_DIAG_CAUSAL)
        return BSP_ERR_INVALID_ARG;
    if (Z == 0) return BSP_OK;
    if (!X || !Y || (mask_kind == BSP_MASK_DENSE && !mask)) return BSP_ERR_INVALID_ARG;
    if (((uintptr_t)X & 15u) || ((uintptr_t)Y & 15u) || (mask_kind == BSP_MASK_DENSE && ((uintptr_t)mask & 15u)))
        return BSP_ERR_ALIGNMENT;

    bsp_layout_t L = nullptr;
    int rc = bsp::layout_plan(layout, H, nb, block, false, &L);  // host tables only, no geometry analysis
    if (rc != BSP_OK) return rc;
    const int E = dtype == BSP_F32 ? 1 : 0;
    // what the softmax kernels read: status word, CSR tables, this dtype's chunk list
    struct Part { const std::vector<int32_t>* v; const int32_t** dst; };
    LayoutView& V = L->view;
    Part parts[] = {{&L->row_ptr, &V.row_ptr}, {&L->col_idx, &V.col_idx}, {&L->blk_id, &V.blk_id},
                    {&L->sm_items[E], &V.sm_items[E]}};
    size_t need = align256(sizeof(int));
    for (const Part& p : parts) need += align256(p.v->size() * sizeof(int32_t));
    if (need > kScratchBytes) {
        bsp_layout_destroy(L);
        return BSP_ERR_OOM;  // the layout's tables exceed the fixed scratch
    }
    char* base = nullptr;
    rc = scratch_address((void**)&base);
    if (rc != BSP_OK) {
        bsp_layout_destroy(L);
        return rc;
    }
    cudaStream_t s = (cudaStream_t)stream;
    V.status = (int*)base;
    V.wait_ns = kDefaultWaitNs;
    V.inject = 0;
    bool ok = cudaMemsetAsync(base, 0, sizeof(int), s) == cudaSuccess;  // the status word starts at zero
    size_t off = align256(sizeof(int));
    for (const Part& p : parts) {
        *p.dst = (const int32_t*)(base + off);
        // pageable source: the call returns once the bytes are staged, so the
        // host tables may be freed right after
        if (!p.v->empty())
            ok = ok && cudaMemcpyAsync(base + off, p.v->data(), p.v->size() * sizeof(int32_t),
                                       cudaMemcpyHostToDevice, s) == cudaSuccess;
        off += align256(p.v->size() * sizeof(int32_t));
    }
    V.H = L->H;
    V.nb = L->nb;
    V.B = L->B;
    V.S = L->S;
    V.G = L->G;
    V.ngroups = L->ngroups;
    V.n_tiles = L->n_tiles;
    V.nnz = L->nnz;
    V.sm_n_items[E] = (int)(L->sm_items[E].size() / 4);
    V.sm_max_bytes[E] = L->sm_max_bytes[E];
    V.sm_fits[E] = L->sm_fits[E] ? 1 : 0;
    if (!ok) {
        cudaGetLastError();
        bsp_layout_destroy(L);
        return BSP_ERR_CUDA;
    }
    rc = L->nnz == 0 ? BSP_OK
                     : bsp::launch_softmax(L, dtype, X, Y, Z, scale, mask_kind,
                                           mask_kind == BSP_MASK_DENSE ? mask : nullptr, s);
    bsp_layout_destroy(L);  // host memory only
    return rc;
}
