// Device side of the affine block-row geometry (the SPLAT / ACSR abstract,
// NSF PAR record: columns of a regular layout's block-rows follow a formula
// in the row index).  A head's record holds at most a band term (offsets
// beta .. beta+kappa-1 from the diagonal) and a column term (columns
// beta + sigma*k, k < kappa, causal: only in rows at or below the column);
// from it the attention kernel's TMA producers compute the key blocks of a
// row tile instead of reading the step tables (geo_col), and the host-side
// check of that arithmetic also evaluates each block's presence (geo_has).
// The helpers compile for the host too, so that check needs no GPU.
#pragma once

#include <cstdint>

namespace bsp {

#define BSP_HD __host__ __device__ __forceinline__
BSP_HD int geo_min(int a, int b) { return a < b ? a : b; }
BSP_HD int geo_max(int a, int b) { return a > b ? a : b; }

struct GeoHead {
    int b_on, b_beta, b_kappa, c_on, c_beta, c_sigma, c_kappa, c_causal;
};

// rec: 8 ints, 16-byte aligned (two vector loads on the device)
BSP_HD GeoHead geo_load(const int32_t* rec) {
#ifdef __CUDA_ARCH__
    const int4 a = *reinterpret_cast<const int4*>(rec), b = *reinterpret_cast<const int4*>(rec + 4);
    return GeoHead{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#else
    return GeoHead{rec[0], rec[1], rec[2], rec[3], rec[4], rec[5], rec[6], rec[7]};
#endif
}

// The union of the columns of block-rows [i0, i1] of one head, ascending:
// the column term's columns below the band's range [lo, hi) (indices
// 0 .. n_low-1), the range, then the column term's columns from index hi_idx
// up to np (np = those kept by some row of the tile).
struct GeoTile {
    int lo, hi, n_low, hi_idx, np;
};

BSP_HD GeoTile geo_tile(const GeoHead& g, int i0, int i1, int nb) {
    GeoTile u{0, 0, 0, 0, 0};
    if (g.b_on) {
        // rows whose band is not clipped away entirely: i + beta + kappa > 0, i + beta < nb
        const int first = geo_max(i0, 1 - g.b_beta - g.b_kappa), last = geo_min(i1, nb - 1 - g.b_beta);
        if (first <= last) {
            u.lo = geo_max(0, first + g.b_beta);
            u.hi = geo_min(nb, last + g.b_beta + g.b_kappa);
        }
    }
    if (g.c_on)
        u.np = !g.c_causal ? g.c_kappa : (i1 < g.c_beta ? 0 : geo_min(g.c_kappa, (i1 - g.c_beta) / g.c_sigma + 1));
    // column-term columns below x (np = 0 without a column term, whose sigma is 0)
    auto n_lt = [&](int x) {
        return (u.np == 0 || x <= g.c_beta) ? 0 : geo_min(u.np, (x - g.c_beta + g.c_sigma - 1) / g.c_sigma);
    };
    u.n_low = n_lt(u.lo);
    u.hi_idx = n_lt(u.hi);
    return u;
}

// k-th key block of the tile, -1 past the end of the union
BSP_HD int geo_col(const GeoHead& g, const GeoTile& u, int k) {
    if (k < u.n_low) return g.c_beta + g.c_sigma * k;
    k -= u.n_low;
    if (k < u.hi - u.lo) return u.lo + k;
    k += u.hi_idx - (u.hi - u.lo);
    return k < u.np ? g.c_beta + g.c_sigma * k : -1;
}

// whether block (i, j) is in the head's layout (0 <= i, j < nb)
BSP_HD bool geo_has(const GeoHead& g, int i, int j) {
    if (g.b_on && j - i >= g.b_beta && j - i < g.b_beta + g.b_kappa) return true;
    if (!g.c_on || j < g.c_beta || (g.c_causal && j > i)) return false;
    const int d = j - g.c_beta;
    return d % g.c_sigma == 0 && d / g.c_sigma < g.c_kappa;
}

#undef BSP_HD

}  // namespace bsp
