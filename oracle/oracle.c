/*
 * fp64 CPU oracle for block-sparse SDD / DSD / DDS, the block-sparse row
 * softmax and block-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Everything here is the plain definition written out: the 0/1 block layout
 * is expanded to an element mask and the masked products and the softmax are
 * evaluated entry by entry, in double precision.  Inputs are float32 arrays
 * holding the (already dtype-rounded) values; all arithmetic is double.
 *
 * Sources (web pages this follows):
 *  [T117]  "question on blocksparse", openai/triton issue 117: the layout is
 *          a tensor of 0s and 1s, one entry per 16/32/64/128-square block,
 *          blocks never overlap; the three modes SDD (sparse = dense x dense,
 *          sampled), DSD (dense = sparse x dense) and DDS (dense = dense x
 *          sparse); the SDD output is block-sparse and is what the softmax
 *          reduces row by row; the softmax is the same as the dense one; dense
 *          masks may be passed because the diagonal blocks of a block-causal
 *          layout are full.
 *  [PUZ8]  Triton-Puzzles blog post ("Triton", tag "kernel"), Puzzle 8
 *          "Long Softmax": numerically stable softmax, max subtracted first,
 *          computed as max pass, sum pass, normalise pass.
 *  [PUZ9]  same post, Puzzle 9 "Simple FlashAttention": the attention output
 *          row is the softmax-weighted sum of the value rows.
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *  - blocks are numbered by their rank in row-major (h, i, j) order;
 *  - a mask is a keep-mask (1 = keep) applied after scaling; masked entries of
 *    present blocks and whole rows with nothing kept produce 0;
 *  - mask kind 2 ("diagonal causal") masks c > r inside diagonal blocks only.
 *
 * Parity pins: every function here is pinned by tests that do not reuse this
 * file's arithmetic (library routines on special cases, closed forms and
 * invariants; see the tests directory).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MASK_NONE 0
#define MASK_DENSE 1
#define MASK_DIAG_CAUSAL 2

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* layout bookkeeping                                                      */
/* ---------------------------------------------------------------------- */

int64_t oracle_count_nnz(const uint8_t* layout, int H, int nb) {
    int64_t n = 0;
    for (int64_t e = 0; e < (int64_t)H * nb * nb; ++e) n += layout[e] != 0;
    return n;
}

/* Block id of (h, i, j): its rank among the present blocks in row-major
 * (h, i, j) order, or -1 when absent.  ids is [H][nb][nb]. */
static int64_t* block_ids(const uint8_t* layout, int H, int nb) {
    int64_t* ids = (int64_t*)malloc(sizeof(int64_t) * (size_t)H * nb * nb);
    int64_t next = 0;
    for (int64_t e = 0; e < (int64_t)H * nb * nb; ++e)
        ids[e] = layout[e] ? next++ : -1;
    return ids;
}

/* CSR and CSC descriptions of the layout.
 * row_ptr[h*(nb+1) + i] : position of the first block of block-row i of head h
 *                         in the CSR arrays (global over heads);
 * col_idx[p], blk_id[p] : block-column and block id of CSR entry p, columns
 *                         ascending within a row;
 * col_ptr[h*(nb+1) + j] : same for block-column j in the CSC arrays;
 * row_idx[q], blk_id_csc[q] : block-row and block id of CSC entry q, rows
 *                         ascending within a column. */
void oracle_luts(const uint8_t* layout, int H, int nb,
                 int32_t* row_ptr, int32_t* col_idx, int32_t* blk_id,
                 int32_t* col_ptr, int32_t* row_idx, int32_t* blk_id_csc) {
    int64_t* ids = block_ids(layout, H, nb);
    int32_t p = 0;
    for (int h = 0; h < H; ++h) {
        for (int i = 0; i < nb; ++i) {
            row_ptr[h * (nb + 1) + i] = p;
            for (int j = 0; j < nb; ++j) {
                int64_t id = ids[((int64_t)h * nb + i) * nb + j];
                if (id >= 0) { col_idx[p] = j; blk_id[p] = (int32_t)id; ++p; }
            }
        }
        row_ptr[h * (nb + 1) + nb] = p;
    }
    int32_t q = 0;
    for (int h = 0; h < H; ++h) {
        for (int j = 0; j < nb; ++j) {
            col_ptr[h * (nb + 1) + j] = q;
            for (int i = 0; i < nb; ++i) {
                int64_t id = ids[((int64_t)h * nb + i) * nb + j];
                if (id >= 0) { row_idx[q] = i; blk_id_csc[q] = (int32_t)id; ++q; }
            }
        }
        col_ptr[h * (nb + 1) + nb] = q;
    }
    free(ids);
}

/* Element keep-mask inside a present block: the dense intra-block mask. */
static int keep(int kind, const uint8_t* mask, int64_t S, int B, int64_t r, int64_t c) {
    if (kind == MASK_DENSE) return mask[r * S + c] != 0;
    if (kind == MASK_DIAG_CAUSAL) return (r / B != c / B) || (c <= r);
    return 1;
}

/* ---------------------------------------------------------------------- */
/* SDD  [T117: "SDD: sparse = dense x dense, sampled dense-dense matmul"] */
/* ---------------------------------------------------------------------- */
/* C = op(A) . op(B) evaluated only on the present blocks.
 * A : [Z][H][S][K] (trans_a = 0) or [Z][H][K][S] (trans_a = 1)
 * B : [Z][H][K][S] (trans_b = 0) or [Z][H][S][K] (trans_b = 1)
 * out : [nsel][B][B]; unit u = z*nnz + n selects block n of batch z
 *       (sel == NULL: all Z*nnz blocks in order). */
void oracle_sdd(const uint8_t* layout, int H, int nb, int B, int Z, int K,
                int trans_a, int trans_b, const float* A, const float* Bm,
                int64_t nsel, const int64_t* sel, double* out) {
    const int64_t S = (int64_t)nb * B;
    const int64_t nnz = oracle_count_nnz(layout, H, nb);
    /* coordinates of block id n */
    int32_t* bh = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int32_t* bi = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int32_t* bj = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nnz ? nnz : 1));
    int64_t n = 0;
    for (int h = 0; h < H; ++h)
        for (int i = 0; i < nb; ++i)
            for (int j = 0; j < nb; ++j)
                if (layout[((int64_t)h * nb + i) * nb + j]) { bh[n] = h; bi[n] = i; bj[n] = j; ++n; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < nsel; ++s) {
        int64_t u = sel ? sel[s] : s;
        int64_t z = u / nnz, id = u % nnz;
        int h = bh[id];
        const float* Ab = A + ((int64_t)z * H + h) * S * K;
        const float* Bb = Bm + ((int64_t)z * H + h) * S * K;
        double* o = out + s * (int64_t)B * B;
        for (int a = 0; a < B; ++a) {
            int64_t r = (int64_t)bi[id] * B + a;
            for (int b = 0; b < B; ++b) {
                int64_t c = (int64_t)bj[id] * B + b;
                double acc = 0.0;
                for (int k = 0; k < K; ++k) {
                    double x = trans_a ? Ab[(int64_t)k * S + r] : Ab[r * K + k];
                    double y = trans_b ? Bb[c * K + k] : Bb[(int64_t)k * S + c];
                    acc += x * y;
                }
                o[a * B + b] = acc;
            }
        }
    }
    free(bh); free(bi); free(bj);
}

/* ---------------------------------------------------------------------- */
/* softmax  [T117 softmax answers; PUZ8 max / sum / normalise]            */
/* ---------------------------------------------------------------------- */
/* One row: global row r of head h, batch z.  X is the block-compressed input
 * [Z][nnz][B][B].  Writes y_c for every column c of the dense row into
 * row_out[0..S) (0 outside the kept set R). */
static void softmax_row(const uint8_t* layout, const int64_t* ids, int H, int nb, int B,
                        int64_t nnz, int64_t z, int h, int64_t r, const float* X,
                        double scale, int kind, const uint8_t* mask, double* row_out) {
    const int64_t S = (int64_t)nb * B;
    const int64_t i = r / B, a = r % B;
    for (int64_t c = 0; c < S; ++c) row_out[c] = 0.0;
    /* pass 1: max over the kept entries */
    double m = -INFINITY;
    int64_t count = 0;
    for (int j = 0; j < nb; ++j) {
        int64_t id = ids[((int64_t)h * nb + i) * nb + j];
        if (id < 0) continue;
        const float* blk = X + ((int64_t)z * nnz + id) * B * B + a * B;
        for (int b = 0; b < B; ++b) {
            int64_t c = (int64_t)j * B + b;
            if (!keep(kind, mask, S, B, r, c)) continue;
            double v = scale * (double)blk[b];
            if (v > m) m = v;
            ++count;
        }
    }
    if (count == 0) return; /* nothing kept: the row is all zeros */
    /* pass 2: sum of exp(v - m) */
    double sum = 0.0;
    for (int j = 0; j < nb; ++j) {
        int64_t id = ids[((int64_t)h * nb + i) * nb + j];
        if (id < 0) continue;
        const float* blk = X + ((int64_t)z * nnz + id) * B * B + a * B;
        for (int b = 0; b < B; ++b) {
            int64_t c = (int64_t)j * B + b;
            if (!keep(kind, mask, S, B, r, c)) continue;
            sum += exp(scale * (double)blk[b] - m);
        }
    }
    /* pass 3: normalise */
    for (int j = 0; j < nb; ++j) {
        int64_t id = ids[((int64_t)h * nb + i) * nb + j];
        if (id < 0) continue;
        const float* blk = X + ((int64_t)z * nnz + id) * B * B + a * B;
        for (int b = 0; b < B; ++b) {
            int64_t c = (int64_t)j * B + b;
            if (!keep(kind, mask, S, B, r, c)) continue;
            row_out[c] = exp(scale * (double)blk[b] - m) / sum;
        }
    }
}

/* Selected rows as dense rows.  unit u = (z*H + h)*S + r; out [nsel][S]. */
void oracle_softmax_rows(const uint8_t* layout, int H, int nb, int B, int Z,
                         const float* X, double scale, int kind, const uint8_t* mask,
                         int64_t nsel, const int64_t* sel, double* out) {
    const int64_t S = (int64_t)nb * B;
    const int64_t nnz = oracle_count_nnz(layout, H, nb);
    int64_t* ids = block_ids(layout, H, nb);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t s = 0; s < nsel; ++s) {
        int64_t u = sel ? sel[s] : s;
        int64_t r = u % S, zh = u / S;
        softmax_row(layout, ids, H, nb, B, nnz, zh / H, (int)(zh % H), r, X, scale, kind, mask,
                    out + s * S);
    }
    free(ids);
    (void)Z;
}

/* Full softmax in the block-compressed format: Y [Z][nnz][B][B]. */
void oracle_softmax(const uint8_t* layout, int H, int nb, int B, int Z,
                    const float* X, double scale, int kind, const uint8_t* mask, double* Y) {
    const int64_t S = (int64_t)nb * B;
    const int64_t nnz = oracle_count_nnz(layout, H, nb);
    int64_t* ids = block_ids(layout, H, nb);
    #pragma omp parallel
    {
        double* row = (double*)malloc(sizeof(double) * (size_t)S);
        #pragma omp for schedule(dynamic, 4)
        for (int64_t u = 0; u < (int64_t)Z * H * S; ++u) {
            int64_t r = u % S, zh = u / S, z = zh / H;
            int h = (int)(zh % H);
            softmax_row(layout, ids, H, nb, B, nnz, z, h, r, X, scale, kind, mask, row);
            int64_t i = r / B, a = r % B;
            for (int j = 0; j < nb; ++j) {
                int64_t id = ids[((int64_t)h * nb + i) * nb + j];
                if (id < 0) continue;
                double* yb = Y + ((int64_t)z * nnz + id) * B * B + a * B;
                for (int b = 0; b < B; ++b) yb[b] = row[(int64_t)j * B + b];
            }
        }
        free(row);
    }
    free(ids);
}

/* ---------------------------------------------------------------------- */
/* DSD  [T117: "DSD: dense = sparse x dense, the lhs is sparse"]           */
/* ---------------------------------------------------------------------- */
/* Value of the sparse S x S operand of head h, batch z at element (r, c):
 * 0 outside the present blocks. */
static double sparse_at(const int64_t* ids, int nb, int B, int64_t nnz, const float* Xs,
                        int64_t z, int h, int64_t r, int64_t c) {
    int64_t id = ids[((int64_t)h * nb + r / B) * nb + c / B];
    if (id < 0) return 0.0;
    return (double)Xs[((z * nnz + id) * B + r % B) * B + c % B];
}

/* C[z,h] = op(A_sp) . op(Bd).
 * A_sp: [Z][nnz][B][B] blocks of an S x S matrix (trans_a: use its transpose)
 * Bd  : [Z][H][S][N] (trans_b = 0) or [Z][H][N][S] (trans_b = 1)
 * out : [nsel][N]; unit u = (z*H + h)*S + r. */
void oracle_dsd(const uint8_t* layout, int H, int nb, int B, int Z, int N,
                int trans_a, int trans_b, const float* Asp, const float* Bd,
                int64_t nsel, const int64_t* sel, double* out) {
    const int64_t S = (int64_t)nb * B;
    const int64_t nnz = oracle_count_nnz(layout, H, nb);
    int64_t* ids = block_ids(layout, H, nb);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t s = 0; s < nsel; ++s) {
        int64_t u = sel ? sel[s] : s;
        int64_t r = u % S, zh = u / S, z = zh / H;
        int h = (int)(zh % H);
        const float* Bb = Bd + zh * S * N;
        double* o = out + s * N;
        for (int n = 0; n < N; ++n) o[n] = 0.0;
        for (int64_t c = 0; c < S; ++c) {
            /* element (r, c) of op(A_sp); skip entries outside the layout */
            int64_t rr = trans_a ? c : r, cc = trans_a ? r : c;
            if (ids[((int64_t)h * nb + rr / B) * nb + cc / B] < 0) continue;
            double x = sparse_at(ids, nb, B, nnz, Asp, z, h, rr, cc);
            for (int n = 0; n < N; ++n) {
                double y = trans_b ? Bb[(int64_t)n * S + c] : Bb[c * N + n];
                o[n] += x * y;
            }
        }
    }
    free(ids);
    (void)Z;
}

/* ---------------------------------------------------------------------- */
/* DDS  [T117: "DDS: dense = dense x sparse, the rhs is sparse"]           */
/* ---------------------------------------------------------------------- */
/* C[z,h] = op(Ad) . op(B_sp).
 * Ad  : [Z][H][M][S] (trans_a = 0) or [Z][H][S][M] (trans_a = 1)
 * B_sp: [Z][nnz][B][B] blocks of an S x S matrix (trans_b: its transpose)
 * out : [nsel][S]; unit u = (z*H + h)*M + m. */
void oracle_dds(const uint8_t* layout, int H, int nb, int B, int Z, int M,
                int trans_a, int trans_b, const float* Ad, const float* Bsp,
                int64_t nsel, const int64_t* sel, double* out) {
    const int64_t S = (int64_t)nb * B;
    const int64_t nnz = oracle_count_nnz(layout, H, nb);
    int64_t* ids = block_ids(layout, H, nb);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t s = 0; s < nsel; ++s) {
        int64_t u = sel ? sel[s] : s;
        int64_t m = u % M, zh = u / M, z = zh / H;
        int h = (int)(zh % H);
        const float* Ab = Ad + zh * (int64_t)M * S;
        double* o = out + s * S;
        for (int64_t c = 0; c < S; ++c) {
            double acc = 0.0;
            for (int64_t k = 0; k < S; ++k) {
                /* element (k, c) of op(B_sp) */
                int64_t rr = trans_b ? c : k, cc = trans_b ? k : c;
                if (ids[((int64_t)h * nb + rr / B) * nb + cc / B] < 0) continue;
                double x = trans_a ? Ab[k * M + m] : Ab[m * S + k];
                acc += x * sparse_at(ids, nb, B, nnz, Bsp, z, h, rr, cc);
            }
            o[c] = acc;
        }
    }
    free(ids);
    (void)Z;
}

/* ---------------------------------------------------------------------- */
/* attention  [T117: SDD -> softmax -> DSD chain; PUZ9 weighted sum]      */
/* ---------------------------------------------------------------------- */
/* O[z,h,r,:] = sum_{c in R} softmax_R(scale * q_r . k_c) v_c, with
 * R = {c : layout[h][r/B][c/B] = 1 and keep(r, c)}; O row = 0 when R is empty.
 * Q, K, V: [Z][H][S][D]; out [nsel][D]; unit u = (z*H + h)*S + r. */
void oracle_attention(const uint8_t* layout, int H, int nb, int B, int Z, int D,
                      const float* Q, const float* K, const float* V,
                      double scale, int kind, const uint8_t* mask,
                      int64_t nsel, const int64_t* sel, double* out) {
    const int64_t S = (int64_t)nb * B;
    #pragma omp parallel
    {
        double* sc = (double*)malloc(sizeof(double) * (size_t)S);
        uint8_t* inR = (uint8_t*)malloc((size_t)S);
        #pragma omp for schedule(dynamic, 4)
        for (int64_t s = 0; s < nsel; ++s) {
            int64_t u = sel ? sel[s] : s;
            int64_t r = u % S, zh = u / S;
            int h = (int)(zh % H);
            const float* q = Q + (zh * S + r) * D;
            const float* Kb = K + zh * S * D;
            const float* Vb = V + zh * S * D;
            double* o = out + s * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            double m = -INFINITY;
            int64_t count = 0;
            for (int64_t c = 0; c < S; ++c) {
                inR[c] = layout[((int64_t)h * nb + r / B) * nb + c / B] &&
                         keep(kind, mask, S, B, r, c);
                if (!inR[c]) continue;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += (double)q[d] * (double)Kb[c * D + d];
                sc[c] = scale * dot;
                if (sc[c] > m) m = sc[c];
                ++count;
            }
            if (count == 0) continue;
            double sum = 0.0;
            for (int64_t c = 0; c < S; ++c)
                if (inR[c]) sum += exp(sc[c] - m);
            for (int64_t c = 0; c < S; ++c) {
                if (!inR[c]) continue;
                double p = exp(sc[c] - m) / sum;
                for (int d = 0; d < D; ++d) o[d] += p * (double)Vb[c * D + d];
            }
        }
        free(sc);
        free(inR);
    }
    (void)Z;
}

/* Log-sum-exp of a row's kept scores, the normaliser of the softmax above
 * (not in the pages; what a backward needs to rebuild P = exp(x - lse)):
 *     lse[z,h,r] = log sum_{c in R} exp(scale * q_r . k_c),
 * -inf when R is empty.  Q, K: [Z][H][S][D]; out [nsel]; unit u as above. */
void oracle_attention_lse(const uint8_t* layout, int H, int nb, int B, int Z, int D,
                          const float* Q, const float* K, double scale, int kind,
                          const uint8_t* mask, int64_t nsel, const int64_t* sel, double* out) {
    const int64_t S = (int64_t)nb * B;
    #pragma omp parallel
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)S);
        #pragma omp for schedule(dynamic, 4)
        for (int64_t s = 0; s < nsel; ++s) {
            const int64_t u = sel ? sel[s] : s;
            const int64_t row = u % S, zh = u / S;
            const int hh = (int)(zh % H);
            const float* qr = Q + (zh * S + row) * D;
            double top = -INFINITY;
            for (int64_t c = 0; c < S; ++c) {
                const int present = layout[((int64_t)hh * nb + row / B) * nb + c / B];
                if (!present || !keep(kind, mask, S, B, row, c)) {
                    t[c] = -INFINITY;  /* not in R */
                    continue;
                }
                const float* kc = K + (zh * S + c) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += (double)qr[d] * (double)kc[d];
                t[c] = acc * scale;
                top = t[c] > top ? t[c] : top;
            }
            if (top == -INFINITY) {  /* R empty */
                out[s] = -INFINITY;
                continue;
            }
            double total = 0.0;
            for (int64_t c = 0; c < S; ++c) total += exp(t[c] - top);  /* exp(-inf) = 0 outside R */
            out[s] = top + log(total);
        }
        free(t);
    }
    (void)Z;
}

/* ---------------------------------------------------------------------- */
/* backward  [next row: dV = P^T dO, dP = dO V^T, softmax backward,        */
/*            dQ / dK from dS]; the chain rule applied to the definitions  */
/*            above, written out without reuse of the forward code paths   */
/* ---------------------------------------------------------------------- */
/* Softmax backward in the block format.  Y = softmax rows (the forward's
 * output, 0 at masked entries and outside the layout), dY its gradient; for
 * y = softmax(scale * x) over the kept set R of a row,
 *     dx_c = scale * y_c * (dy_c - sum_{c' in R} y_c' dy_c').
 * Entries with y_c = 0 (masked) get dx_c = 0. */
void oracle_softmax_backward(const uint8_t* layout, int H, int nb, int B, int Z,
                             const float* Y, const float* dY, double scale, double* dX) {
    const int64_t S = (int64_t)nb * B;
    const int64_t nnz = oracle_count_nnz(layout, H, nb);
    int64_t* ids = block_ids(layout, H, nb);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t u = 0; u < (int64_t)Z * H * S; ++u) {
        int64_t r = u % S, zh = u / S, z = zh / H;
        int h = (int)(zh % H);
        int64_t i = r / B, a = r % B;
        double dot = 0.0;
        for (int j = 0; j < nb; ++j) {
            int64_t id = ids[((int64_t)h * nb + i) * nb + j];
            if (id < 0) continue;
            const int64_t off = ((int64_t)z * nnz + id) * B * B + a * B;
            for (int b = 0; b < B; ++b) dot += (double)Y[off + b] * (double)dY[off + b];
        }
        for (int j = 0; j < nb; ++j) {
            int64_t id = ids[((int64_t)h * nb + i) * nb + j];
            if (id < 0) continue;
            const int64_t off = ((int64_t)z * nnz + id) * B * B + a * B;
            for (int b = 0; b < B; ++b)
                dX[off + b] = scale * (double)Y[off + b] * ((double)dY[off + b] - dot);
        }
    }
    free(ids);
}

/* Attention backward from the dense-mask definition.  Given dO = dL/dO for
 * O = softmax_R(scale Q K^T) V (rows of R empty -> O row 0), returns
 *     dV = P^T dO,  dP = dO V^T,  dS = P .* (dP - rowsum(P .* dP)),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 * Q, K, V, dO: [Z][H][S][D]; dQ, dK, dV: [Z][H][S][D] (double).  One (z, h)
 * slice per thread (dK and dV sum over rows); P and dS are dense S x S. */
void oracle_attention_backward(const uint8_t* layout, int H, int nb, int B, int Z, int D,
                               const float* Q, const float* K, const float* V, const float* dO,
                               double scale, int kind, const uint8_t* mask,
                               double* dQ, double* dK, double* dV) {
    const int64_t S = (int64_t)nb * B;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t zh = 0; zh < (int64_t)Z * H; ++zh) {
        const int h = (int)(zh % H);
        const float* q = Q + zh * S * D;
        const float* k = K + zh * S * D;
        const float* v = V + zh * S * D;
        const float* go = dO + zh * S * D;
        double* gq = dQ + zh * S * D;
        double* gk = dK + zh * S * D;
        double* gv = dV + zh * S * D;
        for (int64_t e = 0; e < S * D; ++e) gq[e] = gk[e] = gv[e] = 0.0;
        double* P = (double*)calloc((size_t)(S * S), sizeof(double));
        uint8_t* inR = (uint8_t*)malloc((size_t)S);
        for (int64_t r = 0; r < S; ++r) {
            double m = -INFINITY;
            int64_t count = 0;
            for (int64_t c = 0; c < S; ++c) {
                const uint8_t present = layout[((int64_t)h * nb + r / B) * nb + c / B];
                inR[c] = present && keep(kind, mask, S, B, r, c);
                if (!inR[c]) continue;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += (double)q[r * D + d] * (double)k[c * D + d];
                P[r * S + c] = scale * dot;
                if (P[r * S + c] > m) m = P[r * S + c];
                ++count;
            }
            if (count == 0) continue;
            double sum = 0.0;
            for (int64_t c = 0; c < S; ++c)
                if (inR[c]) sum += exp(P[r * S + c] - m);
            for (int64_t c = 0; c < S; ++c)
                P[r * S + c] = inR[c] ? exp(P[r * S + c] - m) / sum : 0.0;
        }
        for (int64_t r = 0; r < S; ++r) {
            /* dP_rc = dO_r . V_c over the support of P's row; delta_r */
            double delta = 0.0;
            for (int64_t c = 0; c < S; ++c) {
                const double p = P[r * S + c];
                if (p == 0.0) continue;
                double dp = 0.0;
                for (int d = 0; d < D; ++d) dp += (double)go[r * D + d] * (double)v[c * D + d];
                delta += p * dp;
            }
            for (int64_t c = 0; c < S; ++c) {
                const double p = P[r * S + c];
                if (p == 0.0) continue;
                double dp = 0.0;
                for (int d = 0; d < D; ++d) dp += (double)go[r * D + d] * (double)v[c * D + d];
                const double ds = p * (dp - delta);
                for (int d = 0; d < D; ++d) {
                    gv[c * D + d] += p * (double)go[r * D + d];
                    gq[r * D + d] += scale * ds * (double)k[c * D + d];
                    gk[c * D + d] += scale * ds * (double)q[r * D + d];
                }
            }
        }
        free(P);
        free(inR);
    }
}

/* ----------------------------------------------------------------------
 * Affine block-row geometry.  [SPLAT] (the SPLAT / ACSR abstract, NSF PAR
 * record): the regular sparse-attention patterns (banded, strided, ...) have
 * rows whose column sets follow a formula in the row index, which a format can
 * store instead of per-block indices.  The abstract gives no format; the
 * reading used here: a head is described by at most two terms, each a column
 * progression whose start moves with the row,
 *     term (alpha, beta, sigma, kappa, causal) puts block (i, j) in the layout
 *     when j = alpha * i + beta + sigma * k for some 0 <= k < kappa, j inside
 *     [0, nb), and (causal == 0 or j <= i),
 * a "band" term (alpha = 1, sigma = 1, causal = 0: offsets beta .. beta+kappa-1
 * from the diagonal) and a "column" term (alpha = 0: the same progression of
 * columns in every row, or in every row at or below it when causal).  A head's
 * layout is the union of its terms.
 * ---------------------------------------------------------------------- */

static int term_has(const int32_t* t, int64_t i, int64_t j) {
    const int64_t alpha = t[0], beta = t[1], sigma = t[2], kappa = t[3], causal = t[4];
    if (causal && j > i) return 0;
    const int64_t d = j - alpha * i - beta;
    if (d < 0 || sigma <= 0 || d % sigma != 0) return 0;
    return d / sigma < kappa;
}

/* terms: int32 [H][2][5]; n_terms[h] terms of head h are used (0..2).
 * out: uint8 [H][nb][nb]. */
void oracle_affine_expand(const int32_t* n_terms, const int32_t* terms, int H, int nb, uint8_t* out) {
    for (int h = 0; h < H; ++h)
        for (int64_t i = 0; i < nb; ++i)
            for (int64_t j = 0; j < nb; ++j) {
                uint8_t v = 0;
                for (int t = 0; t < n_terms[h]; ++t)
                    if (term_has(terms + ((int64_t)h * 2 + t) * 5, i, j)) v = 1;
                out[((int64_t)h * nb + i) * nb + j] = v;
            }
}

static int head_equals(const uint8_t* head, int nb, const int32_t* band, const int32_t* col) {
    for (int64_t i = 0; i < nb; ++i)
        for (int64_t j = 0; j < nb; ++j) {
            const int v = (band && term_has(band, i, j)) || (col && term_has(col, i, j));
            if (v != (head[i * nb + j] != 0)) return 0;
        }
    return 1;
}

/* 1 if some band term and / or column term (each optional) reproduces the
 * head's [nb][nb] layout exactly, found by trying every parameter set: for
 * small nb only (about nb^6 candidates). */
int oracle_affine_describable(const uint8_t* head, int nb) {
    for (int with_band = 0; with_band <= 1; ++with_band)
        for (int bb = -(nb - 1); bb <= (with_band ? nb - 1 : -(nb - 1)); ++bb)
            for (int bk = 1; bk <= (with_band ? 2 * nb - 1 : 1); ++bk) {
                const int32_t band[5] = {1, bb, 1, bk, 0};
                const int32_t* pb = with_band ? band : NULL;
                if (head_equals(head, nb, pb, NULL)) return 1;
                for (int cb = 0; cb < nb; ++cb)
                    for (int cs = 1; cs <= nb; ++cs)
                        for (int ck = 1; ck <= nb; ++ck)
                            for (int cc = 0; cc <= 1; ++cc) {
                                const int32_t col[5] = {0, cb, cs, ck, cc};
                                if (head_equals(head, nb, pb, col)) return 1;
                            }
            }
    return 0;
}
