/*
 * bsp.h — C ABI of libbsp: block-sparse matrix multiply (SDD, DSD, DDS),
 * block-sparse row softmax and block-sparse attention on one GB300 GPU.
 *
 * Source of the operations: "question on blocksparse" (openai/triton issue
 * 117).  The sparsity layout is a tensor of 0s and 1s in which each entry
 * stands for one square block of 16, 32, 64 or 128 elements; blocks never
 * overlap.  There are three matmul modes: SDD (a sampled dense x dense
 * product whose output is block-sparse), DSD (dense = sparse x dense) and DDS
 * (dense = dense x sparse).  The SDD output is the input of the block-sparse
 * softmax, which reduces each row across the row's blocks and equals the dense
 * softmax of the present entries; dense masks may be passed for the entries
 * inside blocks (the diagonal blocks of a block-causal layout are full).
 * Chained, SDD -> softmax -> DSD is block-sparse attention.
 *
 * Conventions for every call:
 *  - Layout: host array uint8 [H][nb][nb] with values 0/1, S = nb * block.
 *    The layout is shared by all Z batch entries.
 *  - Block-sparse tensors are [Z][nnz][block][block], row-major inside a
 *    block; block n is the n-th present block in row-major (h, i, j) order
 *    (nnz counts all heads).
 *  - Dense tensors are contiguous row-major [Z][H][rows][cols].
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, 16-byte
 *    aligned (else BSP_ERR_ALIGNMENT); the library never frees it.  With an
 *    empty batch (Z == 0) a call does nothing and its pointers may be NULL.
 *  - dtype (bsp_dtype_t) is the type of every floating-point input and output
 *    of the call; accumulation is always fp32.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every compute
 *    call only enqueues work on it and returns; results are ready when the
 *    stream is.
 *  - Argument errors are detected before anything is launched; nothing aborts,
 *    throws or traps.  Kernels that detect an impossible state (a bounded wait
 *    of the tensor-core kernels that ran out, or a block-column read from the
 *    tables that lies outside the layout in the fused attention kernel) skip
 *    the access, record a code in the handle's device status word, wait for
 *    their own copies and products in flight and return; bsp_status_check
 *    reads it (bsp_diag_wait_limit provokes both on purpose).
 *  - The handle is immutable after compilation and may be used concurrently
 *    from several streams of the device it was compiled on.
 */
#ifndef BSP_H
#define BSP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bsp_layout_s* bsp_layout_t;

typedef enum { BSP_F32 = 0, BSP_BF16 = 1, BSP_F16 = 2 } bsp_dtype_t;

/* Mask applied inside present blocks by the softmax and attention.
 * NONE: keep everything.  DENSE: keep (r, c) iff mask[r * S + c] != 0, mask a
 * DEVICE uint8 [S][S] shared by all heads and batch entries.  DIAG_CAUSAL:
 * inside the diagonal blocks (block-row == block-column) keep c <= r only. */
typedef enum {
    BSP_MASK_NONE = 0,
    BSP_MASK_DENSE = 1,
    BSP_MASK_DIAG_CAUSAL = 2
} bsp_mask_kind_t;

enum {
    BSP_OK = 0,
    BSP_ERR_INVALID_ARG = -1,  /* bad value, size, handle or NULL pointer   */
    BSP_ERR_UNSUPPORTED = -2,  /* valid but not implemented combination      */
    BSP_ERR_ALIGNMENT = -3,    /* a tensor pointer is not 16-byte aligned    */
    BSP_ERR_OOM = -4,          /* device or host allocation failed           */
    BSP_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed       */
    BSP_ERR_TIMEOUT = -6,      /* a kernel's bounded wait ran out            */
    BSP_ERR_DEVICE_CHECK = -7  /* a kernel's bounds check failed             */
};

/* ---- layout ------------------------------------------------------------ */

/* Validate a 0/1 layout and build its lookup tables on the host only.
 * Produces per-row (CSR) and per-column (CSC) block tables and the work lists
 * the kernels consume.  The handle owns host memory only; compute calls reject
 * it with BSP_ERR_INVALID_ARG.  Used to inspect the tables without a GPU.
 * layout: host uint8 [H][nb][nb], each value 0 or 1 (else INVALID_ARG).
 * block: 16, 32, 64 or 128 (else INVALID_ARG).  H, nb >= 1.
 * On success *out receives a new handle (free with bsp_layout_destroy). */
int bsp_layout_plan(const uint8_t* layout, int H, int nb, int block, bsp_layout_t* out);

/* bsp_layout_plan followed by an upload of every table to the current device,
 * enqueued on `stream` (the host copies stay owned by the handle, so the
 * upload may still be in flight when the call returns).  The handle owns its
 * device memory (one allocation) and its device status word. */
int bsp_layout_compile(const uint8_t* layout, int H, int nb, int block, void* stream,
                       bsp_layout_t* out);

/* bsp_layout_compile for a layout that is already in DEVICE memory (uint8
 * [H][nb][nb], values 0/1), e.g. one that changes every step: every table is
 * built by kernels on `stream` (no host copy of the layout, no host loop over
 * it).  The call reads back the table sizes once, so it synchronises `stream`,
 * and makes one allocation of scratch and one for the tables.  The tables
 * equal bsp_layout_compile's for the same layout, so every compute call
 * behaves the same; the inspection getters read them from the device.
 * Values other than 0/1: BSP_ERR_INVALID_ARG.  nb > 4096 or H * nb^2 > 2^30:
 * BSP_ERR_UNSUPPORTED.  The pages build layouts on the host; this entry point
 * is an implementation addition for dynamic layouts. */
int bsp_layout_compile_device(const uint8_t* layout, int H, int nb, int block, void* stream,
                              bsp_layout_t* out);

/* ---- affine geometry ----------------------------------------------------
 * The SPLAT / ACSR abstract (NSF PAR record, "affine-compressed-sparse-row"):
 * regular attention layouts (banded, strided) have block-rows whose columns
 * follow a formula in the row index, so a kernel can compute them instead of
 * reading per-block tables.  Reading used here (the abstract gives no
 * format): a head is the union of at most BSP_MAX_AFFINE_TERMS terms, one of
 * each kind, where a term (alpha, beta, sigma, kappa, causal) holds block
 * (i, j) when j = alpha*i + beta + sigma*k for some 0 <= k < kappa, with
 * 0 <= j < nb and (causal == 0 or j <= i):
 *   band term   alpha = 1, sigma = 1, causal = 0, kappa >= 1,
 *               -(nb-1) <= beta <= nb-1, beta + kappa - 1 <= nb - 1
 *               (offsets beta .. beta+kappa-1 from the diagonal);
 *   column term alpha = 0, sigma >= 1 (sigma = 1 when kappa = 1), kappa >= 1,
 *               0 <= beta, beta + sigma*(kappa-1) <= nb - 1, causal 0 or 1
 *               (the same columns in every row, or in the rows at or below
 *               each column when causal).
 * A head's band term, when it has one, comes first. */
#define BSP_MAX_AFFINE_TERMS 2
typedef struct {
    int32_t alpha, beta, sigma, kappa, causal;
} bsp_affine_term_t;

/* Build a compiled handle from per-head affine terms (HOST arrays): n_terms
 * [H] (0 .. 2; 0 = an empty head) and terms [H][BSP_MAX_AFFINE_TERMS] (the
 * first n_terms[h] of head h are used).  The layout is expanded on the
 * device and compiled as by bsp_layout_compile_device (same tables, same
 * limits, synchronises `stream`); the handle records the terms, so the
 * attention kernel computes its key blocks from them.  Terms that break the
 * rules above: BSP_ERR_INVALID_ARG. */
int bsp_layout_compile_affine(const int32_t* n_terms, const bsp_affine_term_t* terms, int H, int nb,
                              int block, void* stream, bsp_layout_t* out);

/* The handle's affine description, into HOST arrays n_terms [H] and terms
 * [H][BSP_MAX_AFFINE_TERMS] (unused entries zeroed).  n_terms[h] = -1: head h
 * has no description of this form.  bsp_layout_plan / bsp_layout_compile
 * analyse every head (exact: the terms reproduce the head's layout; complete
 * for nb <= 256, i.e. a head is reported -1 only when no band / column pair
 * describes it; for larger nb the eight longest candidate bands are tried);
 * bsp_layout_compile_affine records the terms it was given;
 * bsp_layout_compile_device does not analyse (every head -1).  With the
 * environment variable BSP_GEOMETRY=1, and every head described, the fused
 * attention kernel's TMA producers compute each step's key blocks from the
 * terms instead of reading the step tables (same results; off by default
 * because it measured slower: the table loads are issued ahead of use). */
int bsp_layout_geometry(bsp_layout_t layout, int32_t* n_terms, bsp_affine_term_t* terms);

/* Free a handle (synchronises the device first if it owns device memory).
 * NULL is accepted and ignored. */
int bsp_layout_destroy(bsp_layout_t layout);

/* Sizes of a handle; any output pointer may be NULL. */
int bsp_layout_info(bsp_layout_t layout, int* H, int* nb, int* block, int64_t* nnz);

/* Copy the lookup tables into caller-owned HOST arrays (any may be NULL).
 * For a compiled handle they are read back from the device copies the
 * kernels use.  Sizes: row_ptr, col_ptr [H*(nb+1)]; the others [nnz].
 * row_ptr[h*(nb+1)+i] is the position (global over heads) of the first block
 * of block-row i of head h in col_idx / blk_id, columns ascending; col_ptr,
 * row_idx, blk_id_csc describe the same blocks column by column, rows
 * ascending.  blk_id and blk_id_csc hold block ids (row-major rank). */
int bsp_layout_get_luts(bsp_layout_t layout, int32_t* row_ptr, int32_t* col_idx,
                        int32_t* blk_id, int32_t* col_ptr, int32_t* row_idx,
                        int32_t* blk_id_csc);

/* Row-tile work list used by the tensor-core SDD and attention kernels (host
 * copies, for inspection; any pointer may be NULL, call first with NULL
 * arrays to get the sizes).  A tile is G = 128/block consecutive block-rows of
 * one head (tile t = h * ceil(nb/G) + g); the union of their block-columns is
 * cut into steps of G slots.  tile_step_ptr [n_tiles+1]: first step of each
 * tile; tile_order [n_tiles]: tiles with the most steps first; step_col
 * [n_steps*G]: block-column of each slot (-1 = padding); step_blk
 * [n_steps*G*G]: block id at (row a of the tile, slot b), -1 when absent. */
int bsp_layout_tiles(bsp_layout_t layout, int* G, int* n_tiles, int64_t* n_steps,
                     int32_t* tile_step_ptr, int32_t* tile_order, int32_t* step_col,
                     int32_t* step_blk);

/* Line groups used by the tensor-core DSD / DDS kernels (host copies, for
 * inspection; any pointer may be NULL, call first with NULL arrays to get the
 * sizes).  orient 0: a group is G = 128/block consecutive block-rows of one
 * head (group t = h * ceil(nb/G) + g); orient 1: G consecutive block-columns.
 * Each group has one slot per block index of the union of its lines' blocks,
 * ascending.  grp_ptr [n_groups+1]: first slot of each group; grp_order
 * [n_groups]: groups with the most slots first; slot_idx [n_slots]: the block
 * index along the contraction (block-column for orient 0, block-row for 1);
 * slot_blk [n_slots*G]: block id of line a of the group at slot s, at
 * [s*G + a], -1 when absent.  orient not 0 or 1: BSP_ERR_INVALID_ARG. */
int bsp_layout_groups(bsp_layout_t layout, int orient, int* G, int* n_groups, int64_t* n_slots,
                      int32_t* grp_ptr, int32_t* grp_order, int32_t* slot_idx, int32_t* slot_blk);

/* Chunks of the block-sparse row softmax ("question on blocksparse", openai/
 * triton issue 117: the softmax reduces each row of the SDD output across the
 * row's present blocks) for elements of elt_bytes (2 or 4) bytes: host copy,
 * for inspection; any pointer may be NULL (call first with items = NULL to
 * get n_chunks).  A chunk is R consecutive rows of one block-row, moved through
 * shared memory by one CTA: items [n_chunks*4] int32 = (h*nb + i, first block
 * id of the block-row p0, its block count nnz_i, r0 | R << 16), block-rows in
 * memory order and rows r0 .. r0+R-1.  R is the largest power of two (at most
 * block) with R * nnz_i * block * elt_bytes <= the layout's chunk budget:
 * twice the bytes of its longest row, at least 24 KB, at most 64 KB.
 * max_bytes: the largest chunk.  fits: 0 when a single row exceeds the
 * budget, in which case the softmax takes one warp per row instead of this
 * list.  elt_bytes not 2 or 4: BSP_ERR_INVALID_ARG. */
int bsp_layout_softmax_chunks(bsp_layout_t layout, int elt_bytes, int64_t* n_chunks, int* max_bytes, int* fits,
                              int32_t* items);

/* ---- matmul modes ------------------------------------------------------ */

/* SDD: C = op(A) . op(B) evaluated on the present blocks only.
 * A: [Z][H][S][K] (trans_a = 0) or [Z][H][K][S] (trans_a = 1).
 * B: [Z][H][K][S] (trans_b = 0) or [Z][H][S][K] (trans_b = 1).
 * C: [Z][nnz][block][block] (output).  Attention scores use trans_b = 1
 * (C = Q K^T with Q, K both [S][K]).  K >= 1. */
int bsp_sdd(bsp_layout_t layout, int dtype, const void* A, const void* B, void* C,
            int Z, int K, int trans_a, int trans_b, void* stream);

/* Fused SDD + row softmax: P = softmax(scale * SDD(op(A), op(B))) on the
 * layout's blocks, with the mask kinds and masked-entry rules of
 * bsp_softmax, in one pass whose scores never reach memory (tensor cores for
 * bf16 / fp16 and the shapes bsp_sdd runs there; otherwise bsp_sdd followed by
 * bsp_softmax in place).  Arguments as bsp_sdd (P is its C: [Z][nnz][B][B]),
 * plus scale > 0, mask_kind and mask as bsp_softmax.  This is the first two
 * steps of the unfused attention chain of "question on blocksparse" (issue
 * 117) fused; the result equals bsp_softmax(bsp_sdd(...)) up to rounding. */
int bsp_sdd_softmax(bsp_layout_t layout, int dtype, const void* A, const void* B, void* P, int Z, int K,
                    int trans_a, int trans_b, float scale, int mask_kind, const uint8_t* mask, void* stream);

/* DSD: C = op(A_sp) . op(B), A_sp the S x S block-sparse matrix.
 * A_sp: [Z][nnz][block][block]; trans_a = 1 uses its transpose.
 * B: [Z][H][S][N] (trans_b = 0) or [Z][H][N][S] (trans_b = 1).
 * C: [Z][H][S][N] (output); rows of empty block-rows are written as 0. */
int bsp_dsd(bsp_layout_t layout, int dtype, const void* A_sp, const void* B, void* C,
            int Z, int N, int trans_a, int trans_b, void* stream);

/* DDS: C = op(A) . op(B_sp), B_sp the S x S block-sparse matrix.
 * A: [Z][H][M][S] (trans_a = 0) or [Z][H][S][M] (trans_a = 1).
 * B_sp: [Z][nnz][block][block]; trans_b = 1 uses its transpose.
 * C: [Z][H][M][S] (output); columns of empty block-columns are written as 0. */
int bsp_dds(bsp_layout_t layout, int dtype, const void* A, const void* B_sp, void* C,
            int Z, int M, int trans_a, int trans_b, void* stream);

/* ---- softmax ----------------------------------------------------------- */

/* Row softmax of scale * X over the kept entries of each row, on SDD output.
 * X, Y: [Z][nnz][block][block]; Y may equal X (in place).  Entries of
 * present blocks that the mask removes are written as 0, and so is every
 * entry of a row with nothing kept.  scale > 0 and finite.
 * mask: DEVICE uint8 [S][S] for BSP_MASK_DENSE, ignored otherwise. */
int bsp_softmax(bsp_layout_t layout, int dtype, const void* X, void* Y, int Z, float scale,
                int mask_kind, const uint8_t* mask, void* stream);

/* Allocation-free variant of bsp_softmax (the pages have no counterpart: this
 * entry point exists for deployment, not for the method).  Some callers cannot
 * allocate device memory -- a serving runtime that reserves the whole GPU for
 * its own memory pool, a plugin that is handed only its input and output
 * buffers -- and so cannot create a compiled layout handle, whose tables live
 * in memory bsp_layout_compile allocates.  This call takes the HOST layout
 * (uint8 [H][nb][nb], as for bsp_layout_compile), builds the tables on the
 * host on every call and uploads them into a fixed array of device memory
 * that the library declares itself (4 MiB, held by every GPU that loads the
 * library until the process exits).  It calls no cudaMalloc / cudaFree and no
 * allocating library routine; the caller still passes X and Y (device,
 * [Z][nnz][block][block], Y may equal X) and, for BSP_MASK_DENSE, the mask.
 * Results equal bsp_softmax's.
 *  - Layouts whose tables (row pointers, block columns, block ids and the
 *    softmax chunk list) exceed the array return BSP_ERR_OOM and launch
 *    nothing.
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.  The
 *    address is kept for the life of the process, so calls after a reset of
 *    that device's context (cudaDeviceReset) are not supported.
 *  - Every call shares the array and it keeps the last call's tables; calls
 *    that overlap on the GPU (e.g. on two streams) race.  Calls ordered on one
 *    stream are safe.
 *  - Device-side timeouts are recorded in the array's status word, which this
 *    entry point clears at the start of each call but does not report. */
int bsp_softmax_noalloc(const uint8_t* layout, int H, int nb, int block, int dtype, const void* X,
                        void* Y, int Z, float scale, int mask_kind, const uint8_t* mask,
                        void* stream);

/* ---- attention --------------------------------------------------------- */

/* Fused block-sparse attention: O = softmax(scale Q K^T restricted to the
 * layout and mask) V, the SDD -> softmax -> DSD chain in one pass that never
 * writes the scores.  Q, K, V, O: [Z][H][S][D]; rows with nothing kept are 0.
 * D: 16..128, a multiple of 16.  mask as for bsp_softmax.
 * The tensor-core kernels (16-bit types with D 64 or 128; fp32 with D 64, as
 * three TF32 products per fp32 product) run as one persistent CTA per SM over
 * a work schedule that the first call with a given Z builds on the host and
 * uploads synchronously into device memory kept by the handle (see
 * bsp_diag_attention_schedule); make that first call outside any stream
 * capture.  A schedule that cuts long tiles adds a combine pass and a
 * workspace of the handle: calls on different streams then run one after
 * the other (an event orders them; inside a stream capture the graph's own
 * order holds, and two graphs replaying such calls of one handle must not run
 * concurrently).  Other shapes run on the FFMA kernel. */
int bsp_attention(bsp_layout_t layout, int dtype, const void* Q, const void* K, const void* V,
                  void* O, int Z, int D, float scale, int mask_kind, const uint8_t* mask,
                  void* stream);

/* bsp_attention that also writes each query row's log-sum-exp of its kept
 * scaled scores, lse[z][h][r] = ln sum_{c kept} exp(scale q_r . k_c) (the
 * softmax's normaliser; -inf for rows with nothing kept), for
 * bsp_attention_backward_lse.  lse: DEVICE float [Z][H][S], 16-byte aligned
 * (else BSP_ERR_ALIGNMENT), NULL only when Z == 0 (else BSP_ERR_INVALID_ARG).
 * Every other argument and the output O as for bsp_attention.  The pages
 * define no such output; it is the forward half of the backward below. */
int bsp_attention_lse(bsp_layout_t layout, int dtype, const void* Q, const void* K, const void* V, void* O,
                      float* lse, int Z, int D, float scale, int mask_kind, const uint8_t* mask, void* stream);

/* ---- backward ---------------------------------------------------------- */

/* Backward of bsp_softmax.  Y: the forward's output (0 at masked entries),
 * dY: the gradient of Y; writes the gradient of X,
 *     dX = scale * Y .* (dY - rowsum(Y .* dY))   (row sums over the row's blocks),
 * which is 0 wherever Y is 0.  Y, dY, dX: DEVICE [Z][nnz][block][block];
 * dX may equal dY (in place).  scale > 0 and finite, as in the forward.  The
 * pages state no backward; this is the chain rule applied to the softmax
 * they define. */
int bsp_softmax_backward(bsp_layout_t layout, int dtype, const void* Y, const void* dY, void* dX, int Z,
                         float scale, void* stream);

/* Gradients of bsp_attention for the output gradient dO, as the chain
 *     P = softmax(scale Q K^T on the layout and mask)   (recomputed)
 *     dV = P^T dO,  dP = dO V^T (on the layout),  dX = bsp_softmax_backward(P, dP),
 *     dQ = dX K,  dK = dX^T Q
 * enqueued on `stream`.  For 16-bit types with head size 64 or 128 the fused
 * forward first recomputes O and the rows' log-sum-exp (O in dV's memory, lse
 * in dK's), and the backward from them (bsp_attention_backward_lse) follows;
 * otherwise the chain runs as this library's fused SDD + softmax, DSD, SDD and
 * softmax backward calls (bsp_sdd_softmax, bsp_dsd, bsp_sdd,
 * bsp_softmax_backward), with dP and dX from one fused pass on the tensor-core
 * shapes (dP = dO V^T kept in fp32 on chip, dX written), else dP written and
 * the softmax backward run in place.  Q, K, V, dO, dQ, dK, dV:
 * DEVICE [Z][H][S][D], D and the mask as for bsp_attention.  P_ws, dP_ws:
 * caller-owned DEVICE workspace of Z * nnz * block * block elements each (P
 * and dX live there afterwards); they may be NULL when the layout has no
 * block, in which case dQ, dK, dV are zeroed.
 * The pages state no backward (the chain rule on their definitions). */
int bsp_attention_backward(bsp_layout_t layout, int dtype, const void* Q, const void* K, const void* V,
                           const void* dO, void* dQ, void* dK, void* dV, int Z, int D, float scale,
                           int mask_kind, const uint8_t* mask, void* P_ws, void* dP_ws, void* stream);

/* Gradients of bsp_attention as bsp_attention_backward, given also the
 * forward's output O and its rows' log-sum-exp lse (bsp_attention_lse, same
 * inputs).  With the statistics known, P = exp(scale Q K^T - lse) needs no
 * statistics pass, and rowsum(P .* dP) = rowsum(dO .* O) per row (O = P V),
 * so one tensor-core pass over the row tiles computes both products of a
 * step, S = Q K^T and dP = dO V^T, and writes P and
 * dX = scale P .* (dP - rowsum(dO .* O)) together (P is not read back); for
 * head size 128 and blocks of 64 and 128 the same pass accumulates
 * dQ = dX K per row tile on the tensor cores.  Then dV = P^T dO, dK = dX^T Q
 * (and dQ = dX K where the pass did not).  O, dO: DEVICE [Z][H][S][D]; lse:
 * DEVICE float [Z][H][S], 16-byte aligned; the rest as for
 * bsp_attention_backward; dK's memory holds the rows' dO . O (fp32) until it
 * receives dK.  fp32, and shapes the one-pass kernel does not cover, take
 * bsp_attention_backward's recomputing chain (O and lse unused).  Not from
 * the pages: the chain rule with the forward's statistics kept. */
int bsp_attention_backward_lse(bsp_layout_t layout, int dtype, const void* Q, const void* K, const void* V,
                               const void* O, const void* dO, const float* lse, void* dQ, void* dK, void* dV,
                               int Z, int D, float scale, int mask_kind, const uint8_t* mask, void* P_ws,
                               void* dP_ws, void* stream);

/* Attention on HOST tensors (Q, K, V, O as in bsp_attention, in host memory;
 * pinned memory lets the copies overlap the kernels, pageable memory works
 * but serialises them).  The batch is processed in slices of whole batch
 * entries (at least two slices when Z >= 2, as many entries per slice as the
 * workspace holds) through a caller-owned DEVICE workspace (256-byte aligned,
 * bsp_attention_host_workspace(layout, dtype, D, z_slice) bytes for slices of
 * z_slice entries); each slice's host-to-device copies, kernel and
 * device-to-host copy run on three streams owned by the handle, so copies of
 * neighbouring slices overlap each kernel.  Asynchronous like the other
 * calls: it starts after the work queued on `stream` and `stream` waits for
 * its end; the host buffers and the workspace must stay valid until then.
 * mask: DEVICE [S][S] as in bsp_attention.  flags: 0, or
 * BSP_HOST_RESERVED_WORKSPACE — the caller promises that nothing but this
 * handle's calls touches the workspace between them; a call given the same
 * workspace as the handle's previous call, sliced into slots of the same size
 * (same batch slicing, D and dtype), then starts its input copies as soon as
 * the slots they fill are free (overlapping the previous call's last kernel
 * and output copy) instead of after all the work on `stream`; a call whose
 * slots differ in size waits for all the work on `stream` first.  Calls
 * that share a handle must not run concurrently from several host threads.
 * Workspace smaller than one slice or unknown flags: BSP_ERR_INVALID_ARG.
 * (Not from the pages: the end-to-end path through host memory.) */
#define BSP_HOST_RESERVED_WORKSPACE 1
int bsp_attention_host(bsp_layout_t layout, int dtype, const void* Q, const void* K, const void* V, void* O,
                       int Z, int D, float scale, int mask_kind, const uint8_t* mask, void* workspace,
                       size_t workspace_bytes, int flags, void* stream);
size_t bsp_attention_host_workspace(bsp_layout_t layout, int dtype, int D, int z_slice);

/* ---- diagnostics ------------------------------------------------------- */

/* Evaluate, on n DEVICE floats x, the software 2^x that the attention softmax
 * computes on the FMA pipe for part of its score columns (range reduction to
 * x = j + f, |f| <= 1/2, a cubic for 2^f, j added to the exponent; maximum
 * relative error 1.02e-4 for x >= -125; inputs below -125, -inf included,
 * give a value in (0, 2^-124.5]).  y: DEVICE float [n] (output).  Enqueued on
 * `stream`.  The method is the implementation's, not the pages'. */
int bsp_diag_exp2(const float* x, float* y, int64_t n, void* stream);

/* For a host-planned or compiled handle whose every head has an affine
 * description: evaluate ON THE HOST the routines with which the geometry
 * variant of the attention kernel computes each step's key blocks and their
 * presence, into HOST arrays shaped like bsp_layout_tiles' step_col [n_steps*G]
 * (block-column of each slot, -1 = padding) and step_blk [n_steps*G*G] (1 when
 * (row a, slot b) is in the layout, else 0), so that tests can compare them
 * with the step tables without a GPU.  Other handles: BSP_ERR_UNSUPPORTED. */
int bsp_diag_geometry_steps(bsp_layout_t layout, int32_t* step_col, int32_t* step_blk);

/* The work schedule of the fused attention kernel for a batch of Z entries of
 * type dtype on a GPU with n_sm SMs, computed ON THE HOST (a handle with host
 * tables: bsp_layout_plan or bsp_layout_compile; the setting of
 * bsp_diag_attention_split applies).  The work items are the (tile, batch
 * entry) pairs (n_tiles as bsp_layout_tiles reports), or pieces of them: a
 * tile may be cut into pieces of consecutive steps, each of which leaves a
 * partial result (the rows' unnormalised output, running max and sum) that a
 * combine pass merges by the running-max / running-sum recurrence of the
 * Triton-Puzzles blog, Puzzle 9 "Simple FlashAttention".  For fp32 every
 * tile of more than 32 steps of 128 keys is cut, whatever the split setting:
 * the output keeps its 1e-5 accuracy while one accumulation in tensor memory
 * spans at most 4096 keys (the pieces are merged in fp32 on the CUDA cores);
 * 16-bit types are cut only for balance.  The items are
 * taken longest-first and each given to the CTA with the least work so far
 * (work of an item = its step count + 1; ties: the lowest CTA index).
 * Outputs: *grid CTAs, *n_items items, *n_split cut tiles; with non-NULL
 * arrays also ptr [grid + 1] (CTA c runs items ptr[c] .. ptr[c + 1] - 1 in
 * that order), items [4 * n_items] (tile, first step, step count, batch
 * entry), part [n_items] (the partial-result slot of a piece, else -1) and
 * combine [4 * n_split] (tile, batch entry, first slot, pieces), all HOST
 * int32.  The kernel builds the same schedule on its first launch with a
 * given Z, dtype and split setting, keeps it in device memory of the handle
 * and reuses it afterwards.  Z < 1, n_sm < 1, an unknown dtype, NULL counts
 * or a handle compiled on the device: BSP_ERR_INVALID_ARG.  Not from the pages: the load balance of
 * this implementation. */
int bsp_diag_attention_schedule(bsp_layout_t layout, int dtype, int Z, int n_sm, int* grid, int* n_items,
                                int* n_split, int32_t* ptr, int32_t* items, int32_t* part, int32_t* combine);

/* How the fused attention kernels of this handle cut long tiles from now on:
 * max_steps 0 (the default) cuts only when the greedy makespan of whole
 * tiles is at least a tenth and 24 steps longer than with pieces of about
 * half a CTA's fair share; max_steps > 0 cuts every tile of more than
 * max_steps steps of 128 keys into pieces of at most max_steps steps;
 * max_steps < 0 never cuts (fp32 launches still cut every tile of more than
 * 32 steps, see bsp_diag_attention_schedule).  A launch with cut tiles adds
 * the combine pass and
 * uses a device workspace of the handle (128 x 130 floats per piece) that
 * launches on different streams take in turn.  NULL handle:
 * BSP_ERR_INVALID_ARG.  Not from the pages: the load balance of this
 * implementation. */
int bsp_diag_attention_split(bsp_layout_t layout, int max_steps);

/* Set the limit of every bounded wait in the tensor-core kernels launched
 * with this handle from now on (wait_ns; 0 restores the default of 2 s) and
 * test injections that make one of those waits, or one of the kernels' bounds
 * checks, fail on purpose without touching memory out of bounds:
 *   inject & 1  the fused attention kernel never loads the first Q tile of
 *               each CTA and never signals it, so the Q K^T issuer's wait
 *               runs out: the call records BSP_ERR_TIMEOUT;
 *   inject & 2  the fused attention kernel's K producer sees block-column nb
 *               (out of range) for its first step; its bounds check of the
 *               columns that become copy coordinates records
 *               BSP_ERR_DEVICE_CHECK.
 * Either way every role of the kernel stops, waits for the copies and matrix
 * products it had already issued, frees its tensor memory and returns; the
 * output is then undefined and bsp_status_check reports the code.  inject 0
 * restores normal operation.  Other inject bits: BSP_ERR_INVALID_ARG.  Not
 * from the pages: the robustness checks of this implementation. */
int bsp_diag_wait_limit(bsp_layout_t layout, uint64_t wait_ns, int inject);

/* ---- status ------------------------------------------------------------ */

/* Synchronise `stream`, then return and clear the handle's device status
 * word: BSP_OK, BSP_ERR_TIMEOUT or BSP_ERR_DEVICE_CHECK (or BSP_ERR_CUDA if
 * the synchronisation itself failed). */
int bsp_status_check(bsp_layout_t layout, void* stream);

/* Static text for a status code. */
const char* bsp_status_string(int status);

/* Library build identification (static text). */
const char* bsp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSP_H */
