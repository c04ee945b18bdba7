// Internal definitions shared by the host code and the kernels of libbsp.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/bsp.h"

// Device-side view of a compiled layout: plain pointers into the handle's
// single device allocation plus the sizes.  Passed to kernels by value.
struct LayoutView {
    const int32_t* row_ptr;       // [H*(nb+1)] CSR row starts (global positions)
    const int32_t* col_idx;       // [nnz] block-column of each CSR entry
    const int32_t* blk_id;        // [nnz] block id of each CSR entry
    const int32_t* col_ptr;       // [H*(nb+1)] CSC column starts
    const int32_t* row_idx;       // [nnz] block-row of each CSC entry
    const int32_t* blk_id_csc;    // [nnz] block id of each CSC entry
    const int32_t* blk_key;       // [nnz] h*nb + i of block id n (its row key)
    const int32_t* row_order;     // [H*nb] row keys h*nb+i, longest rows first
    const int32_t* col_order;     // [H*nb] column keys h*nb+j, longest columns first
    // row tiles of G = 128/B consecutive block-rows (same head) with the union
    // of their block-columns cut into steps of G slots
    const int32_t* tile_step_ptr; // [n_tiles+1]
    const int32_t* tile_order;    // [n_tiles] tile ids, most steps first
    // [n_tiles][4] the same tiles in that order as (tile id, first step, step
    // count, 0): one 16-byte load tells a role its next tile
    const int32_t* tile_run;
    const int32_t* step_col;      // [n_steps*G] block-column of each slot, -1 = padding
    const int32_t* step_blk;      // [n_steps*G*G] block id at (row a, slot b), -1 = absent
    // line groups for the block-sparse matmuls, o = 0: G consecutive block-rows,
    // o = 1: G consecutive block-columns (same head).  One slot per block index
    // of the union of the lines' blocks (ascending, no padding).
    const int32_t* gl_ptr[2];     // [n_tiles+1] first slot of each group
    const int32_t* gl_order[2];   // [n_tiles] groups, most slots first
    const int32_t* gl_idx[2];     // [slots] block index along the contraction
    const int32_t* gl_blk[2];     // [slots*G] block id of line a at slot s ([s*G + a]), -1 = absent
    // softmax chunks for 2- and 4-byte elements: int4 (h*nb+i, p0, nnz_i,
    // r0 | R << 16): R rows of block-row i from row r0, whose blocks have ids
    // p0 .. p0+nnz_i-1 (ids are CSR positions), R the largest power of two with
    // R * nnz_i * B * elt <= softmax_chunk_budget(longest row's bytes)
    // (block-rows in memory order)
    const int32_t* sm_items[2];
    int sm_n_items[2];
    int sm_max_bytes[2];          // largest chunk of the list, in bytes
    int sm_fits[2];               // 0: some single row exceeds the budget
    // affine geometry when every head has one, else nullptr: per head 8 ints
    // (band on, band beta, band kappa, column on, column beta, sigma, kappa,
    // causal); see bsp_affine_term_t
    const int32_t* geo;
    int* status;                  // device status word (0 = OK, else a BSP_ERR_* code)
    int H, nb, B, S, G, ngroups, n_tiles;
    int64_t nnz;
    // limit of every bounded wait of the tensor-core kernels, in ns (0: the
    // default kDefaultWaitNs), and test injections (kInject* bits, 0 in use)
    uint64_t wait_ns;
    int inject;
};

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s: far beyond any legal wait
// bsp_diag_wait_limit injections, read by the fused attention kernel only
constexpr int kInjectSkipFirstQ = 1;   // the producer skips the first Q tile's load and its arrival
constexpr int kInjectBadColumn = 2;    // the K producer sees block-column nb for the first step

struct bsp_layout_s {
    int H = 0, nb = 0, B = 0, S = 0;
    int64_t nnz = 0;
    int device = -1;
    bool on_device = false;

    std::vector<int32_t> row_ptr, col_idx, blk_id, col_ptr, row_idx, blk_id_csc, blk_key;
    std::vector<int32_t> row_order, col_order;
    int max_row_nnz = 0, max_col_nnz = 0;

    int G = 1, ngroups = 0, n_tiles = 0;
    int64_t n_steps = 0;
    int max_tile_steps = 0;
    std::vector<int32_t> tile_step_ptr, tile_order, tile_run, step_col, step_blk;
    std::vector<int32_t> gl_ptr[2], gl_order[2], gl_idx[2], gl_blk[2];
    std::vector<int32_t> sm_items[2];
    int sm_max_bytes[2] = {0, 0};
    bool sm_fits[2] = {true, true};

    void* dmem = nullptr;  // one device allocation holding every table
    LayoutView view{};
    // false for a handle compiled on the device: the host vectors above stay
    // empty and the inspection getters read the device tables (sizes below)
    bool host_tables = true;
    int64_t gl_slots[2] = {0, 0};
    int sm_n_items_dev[2] = {0, 0};
    // affine description per head (n = -1: none), the kernels' 8-int records
    // when every head has one (uploaded into dmem, or geo_dmem for a handle
    // compiled from terms)
    std::vector<int32_t> geo_n;
    std::vector<bsp_affine_term_t> geo_terms;  // [H * BSP_MAX_AFFINE_TERMS]
    std::vector<int32_t> geo_rec;              // [H * kGeoRec] or empty
    void* geo_dmem = nullptr;
    // streams and events of bsp_attention_host (created on first use)
    struct HostPipe* pipe = nullptr;
    // work schedules of the persistent attention kernels per (batch size,
    // SM count, split setting), built on first use (schedule.cpp)
    struct Schedules* schedules = nullptr;
    // cutting of long tiles: 0 automatic, > 0 every tile of more steps than
    // this, < 0 never (bsp_diag_attention_split)
    int attn_split = 0;
};

constexpr int kGeoRec = 8;  // ints per head in LayoutView::geo

// Shared-memory bytes of one softmax chunk for a layout whose longest row
// holds max_row_bytes: twice the longest row, at least 24 KB, at most 64 KB.
// Small chunks let eight 4-warp chunk CTAs share an SM (band of 9-block rows
// of 128 bf16: 0.98 of HBM, against 0.77 with 64 KB chunks and 8 warps); the
// longest rows still come two to a chunk (BigBird's 16 KB global rows in fp32:
// 32 KB chunks, 0.76 of HBM, against 0.69 with one row per chunk).
constexpr int kSoftmaxChunkBudget = 64 * 1024;  // the largest chunk
constexpr int kSoftmaxChunkSmall = 24 * 1024;   // the smallest budget
__host__ __device__ inline int64_t softmax_chunk_budget(int64_t max_row_bytes) {
    const int64_t b = 2 * max_row_bytes;
    return b < kSoftmaxChunkSmall ? kSoftmaxChunkSmall : (b > kSoftmaxChunkBudget ? kSoftmaxChunkBudget : b);
}

namespace bsp {

// kernel launchers (return BSP_OK or an error code; they only enqueue work)
int launch_softmax(const bsp_layout_s* L, int dtype, const void* X, void* Y, int Z, float scale,
                   int kind, const uint8_t* mask, cudaStream_t s);

int launch_sdd_simt(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                    int K, int ta, int tb, cudaStream_t s);
int launch_dsd_simt(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                    int N, int ta, int tb, cudaStream_t s);
int launch_dds_simt(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                    int M, int ta, int tb, cudaStream_t s);
int launch_attention_simt(const bsp_layout_s* L, int dtype, const void* Q, const void* K,
                          const void* V, void* O, float* lse, int Z, int D, float scale, int kind,
                          const uint8_t* mask, cudaStream_t s);

// tensor-core (tcgen05) paths; return BSP_ERR_UNSUPPORTED when the shape is
// not covered so that the caller can take the SIMT path instead
int launch_attention_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K,
                        const void* V, void* O, float* lse, int Z, int D, float scale, int kind,
                        const uint8_t* mask, cudaStream_t s);
int launch_sdd_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                  int K, int ta, int tb, cudaStream_t s);
// fused SDD + row softmax (P = softmax(scale * SDD) on the layout's blocks)
int launch_sdd_softmax_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* P, int Z, int K,
                          int ta, int tb, float scale, int kind, const uint8_t* mask, cudaStream_t s);
// dX = scale P .* (dP - rowsum(P .* dP)) with dP = dO V^T on the layout
// (fused SDD + softmax backward; 16-bit types, tensor-core shapes only)
int launch_sdd_softmax_bwd_tc(const bsp_layout_s* L, int dtype, const void* dO, const void* V, const void* P,
                              void* dX, int Z, int D, float scale, cudaStream_t s);
// P = exp(scale Q K^T - lse) and dX = scale P .* (dO V^T - dvec) on the layout,
// one pass (tensor cores; BSP_ERR_UNSUPPORTED outside their shapes)
int launch_sdd_attention_bwd_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K, const void* dO,
                                const void* V, const float* lse, const float* dvec, void* P, void* dX, int Z, int D,
                                float scale, int kind, const uint8_t* mask, cudaStream_t s);
// the same, also writing dQ = dX K [Z][H][S][D] (D = 128, blocks of 64 and 128)
int launch_sdd_attention_bwd_dq_tc(const bsp_layout_s* L, int dtype, const void* Q, const void* K, const void* dO,
                                   const void* V, const float* lse, const float* dvec, void* P, void* dX, void* dQ,
                                   int Z, int D, float scale, int kind, const uint8_t* mask, cudaStream_t s);
// out[r] = sum_d A[r][d] B[r][d] (fp32) for rows of D elements (D a multiple of 8)
int launch_row_dot(int dtype, const void* A, const void* B, float* out, int64_t rows, int D, cudaStream_t s);
int launch_dsd_group_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                        int N, int ta, int tb, cudaStream_t s);
int launch_dds_group_tc(const bsp_layout_s* L, int dtype, const void* A, const void* B, void* C, int Z,
                        int M, int ta, int tb, cudaStream_t s);

// backward of the block-sparse softmax (CUDA cores; HBM-bound)
int launch_softmax_backward(const bsp_layout_s* L, int dtype, const void* Y, const void* dY, void* dX, int Z,
                            float scale, cudaStream_t s);

int sm_count();  // multiprocessors of the current device (cached per device)

// bsp_layout_plan, the affine-geometry analysis optional (layout.cpp)
int layout_plan(const uint8_t* layout, int H, int nb, int block, bool analyse, bsp_layout_t* out);

// streams and events of bsp_attention_host (host_pipeline.cpp)
void host_pipe_destroy(bsp_layout_s* L);

// Floats of one partial-result slot of a cut tile: 128 rows of O (head size
// up to 128), then the rows' running maxima (log2 units) and sums.
constexpr int kPartRows = 128, kPartMaxD = 128;
constexpr size_t kPartFloats = (size_t)kPartRows * (kPartMaxD + 2);

// The work schedule of a persistent attention launch with batch Z on a GPU
// with `sms` SMs (schedule.cpp): CTA c of `grid` runs items ptr[c] ..
// ptr[c + 1] - 1, each (tile, first step, step count, batch entry) with
// part[i] = its partial-result slot when the item is a piece of a cut tile,
// else -1; combine [n_split] = (tile, batch entry, first slot, pieces) of the
// cut tiles, merged after the kernel by launch_attention_combine; ws: the
// slots (n_split > 0 only), ordered between streams by the event `done`.
struct AttnSchedule {
    int grid;
    int n_split;
    const int32_t* ptr;
    const int4* items;
    const int32_t* part;
    const int4* combine;
    float* ws;
    cudaEvent_t done;
    std::mutex* mu;  // held from attn_schedule_begin to attn_schedule_end when n_split > 0
};
// Tiles of more steps than this are always cut for the given input type:
// fp32 results keep their 1e-5 accuracy while one accumulation of O in
// tensor memory spans at most 32 steps (4096 keys; measured: one accumulation
// over 16384 keys gave a normwise error of 1.5e-5); the pieces are merged in
// fp32 on the CUDA cores.  0: no forced cut.
constexpr int kF32MaxSteps = 32;
inline int attn_force_cap(int dtype) { return dtype == BSP_F32 ? kF32MaxSteps : 0; }
// Built and uploaded (synchronously) on the first launch with (Z, sms, the
// handle's split setting, force_cap), kept by the handle.
int tile_schedule(bsp_layout_s* L, int Z, int sms, int force_cap, AttnSchedule* out);
void schedules_destroy(bsp_layout_s* L);
// O rows of the cut tiles from their pieces' partial results (attn_combine.cu)
int launch_attention_combine(const bsp_layout_s* L, int dtype, const AttnSchedule& sc, void* O, float* lse, int D,
                             cudaStream_t s);
// Around one persistent attention launch on stream s: begin fetches the
// schedule and, when it cuts tiles, takes the workspace (lock, and a wait for
// the workspace's previous launch); end (called whenever begin succeeded, with
// the launch's status rc) merges the cut tiles and releases the workspace.
int attn_schedule_begin(bsp_layout_s* L, int dtype, int Z, cudaStream_t s, AttnSchedule* sc);
int attn_schedule_end(const bsp_layout_s* L, int dtype, const AttnSchedule& sc, void* O, float* lse, int D,
                      cudaStream_t s, int rc);

// affine geometry (geometry.cpp)
int affine_validate(int nb, int n, const bsp_affine_term_t* t);
int affine_detect(const uint8_t* head, int nb, bsp_affine_term_t* t);
// per-head descriptions of a [H][nb][nb] host layout into L->geo_n / geo_terms / geo_rec
void affine_analyse(bsp_layout_s* L, const uint8_t* lay);
// L->geo_rec from L->geo_n / geo_terms (left empty unless every head is described)
void affine_records(bsp_layout_s* L);

}  // namespace bsp
