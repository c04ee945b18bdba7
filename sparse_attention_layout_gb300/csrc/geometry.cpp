// Affine block-row geometry of a layout: the idea of the SPLAT / ACSR abstract
// (NSF PAR record, "affine-compressed-sparse-row") that regular attention
// layouts (banded, strided) have rows whose columns follow a formula in the
// row index.  A head is described by at most a band term (offsets beta ..
// beta+kappa-1 from the diagonal) and a column term (columns beta + sigma*k,
// k < kappa, in every row, or only in rows at or below the column when
// causal); bsp_affine_term_t states the rules.
//
// Detection per head, exact (the terms found are expanded and compared with
// the head):
//  1. a band can only hold full diagonals (every block on offset o present),
//     so the candidates are the maximal runs of full diagonals, plus no band;
//  2. what the band leaves must lie on columns of the column term; the
//     smallest progression through those columns (first one, gcd of the gaps)
//     is tried non-causal, then causal.
// A longer band explains a superset and a smaller progression adds a subset,
// so trying every run finds a description whenever one exists; heads with
// more than kMaxRuns runs try the kMaxRuns longest only.
#include <algorithm>
#include <cstdlib>
#include <numeric>

#include "bsp_internal.h"

namespace bsp {
namespace {

constexpr int kMaxRuns = 32;

bool term_has(const bsp_affine_term_t& t, int i, int j) {
    if (t.causal && j > i) return false;
    const int d = j - t.alpha * i - t.beta;
    return d >= 0 && d % t.sigma == 0 && d / t.sigma < t.kappa;
}

bool matches(const uint8_t* lay, int nb, int n, const bsp_affine_term_t* t) {
    for (int i = 0; i < nb; ++i)
        for (int j = 0; j < nb; ++j) {
            bool v = false;
            for (int k = 0; k < n && !v; ++k) v = term_has(t[k], i, j);
            if (v != (lay[(size_t)i * nb + j] != 0)) return false;
        }
    return true;
}

}  // namespace

int affine_validate(int nb, int n, const bsp_affine_term_t* t) {
    if (n < 0 || n > BSP_MAX_AFFINE_TERMS) return BSP_ERR_INVALID_ARG;
    int bands = 0, cols = 0;
    for (int k = 0; k < n; ++k) {
        const bsp_affine_term_t& x = t[k];
        if (x.kappa < 1) return BSP_ERR_INVALID_ARG;
        if (x.alpha == 1) {
            if (++bands > 1 || k != 0 || x.sigma != 1 || x.causal != 0) return BSP_ERR_INVALID_ARG;
            if (x.beta < -(nb - 1) || x.beta > nb - 1 || (int64_t)x.beta + x.kappa - 1 > nb - 1)
                return BSP_ERR_INVALID_ARG;
        } else if (x.alpha == 0) {
            if (++cols > 1 || x.sigma < 1 || (x.kappa == 1 && x.sigma != 1)) return BSP_ERR_INVALID_ARG;
            if (x.causal != 0 && x.causal != 1) return BSP_ERR_INVALID_ARG;
            if (x.beta < 0 || (int64_t)x.beta + (int64_t)x.sigma * (x.kappa - 1) > nb - 1) return BSP_ERR_INVALID_ARG;
        } else {
            return BSP_ERR_INVALID_ARG;
        }
    }
    return BSP_OK;
}

int affine_detect(const uint8_t* lay, int nb, bsp_affine_term_t* out) {
    // blocks per diagonal offset o = j - i (index o + nb - 1)
    std::vector<int> cnt(2 * (size_t)nb - 1, 0);
    bool any = false;
    for (int i = 0; i < nb; ++i)
        for (int j = 0; j < nb; ++j)
            if (lay[(size_t)i * nb + j]) {
                ++cnt[(size_t)(j - i + nb - 1)];
                any = true;
            }
    if (!any) return 0;
    // maximal runs of full diagonals: (first offset, length)
    std::vector<std::pair<int, int>> runs;
    for (int o = -(nb - 1); o <= nb - 1; ++o) {
        if (cnt[(size_t)(o + nb - 1)] != nb - std::abs(o)) continue;
        if (!runs.empty() && runs.back().first + runs.back().second == o)
            ++runs.back().second;
        else
            runs.push_back({o, 1});
    }
    std::stable_sort(runs.begin(), runs.end(),
                     [](const std::pair<int, int>& a, const std::pair<int, int>& b) { return a.second > b.second; });
    if ((int)runs.size() > kMaxRuns) runs.resize(kMaxRuns);
    runs.push_back({0, 0});  // no band
    std::vector<char> col(nb);
    for (const auto& r : runs) {
        bsp_affine_term_t t[BSP_MAX_AFFINE_TERMS];
        int n = 0;
        if (r.second > 0) t[n++] = {1, r.first, 1, r.second, 0};
        // columns of the blocks the band leaves
        std::fill(col.begin(), col.end(), 0);
        bool rest = false;
        for (int i = 0; i < nb; ++i)
            for (int j = 0; j < nb; ++j)
                if (lay[(size_t)i * nb + j] && (r.second == 0 || j - i < r.first || j - i >= r.first + r.second)) {
                    col[(size_t)j] = 1;
                    rest = true;
                }
        if (!rest) {
            for (int k = 0; k < n; ++k) out[k] = t[k];
            return n;
        }
        int first = -1, last = -1, g = 0;
        for (int j = 0; j < nb; ++j) {
            if (!col[(size_t)j]) continue;
            if (first < 0) first = j;
            else g = std::gcd(g, j - last);
            last = j;
        }
        const int sigma = g > 0 ? g : 1;
        for (int causal = 0; causal <= 1; ++causal) {
            t[n] = {0, first, sigma, (last - first) / sigma + 1, causal};
            if (matches(lay, nb, n + 1, t)) {
                for (int k = 0; k <= n; ++k) out[k] = t[k];
                return n + 1;
            }
        }
    }
    return -1;
}

void affine_records(bsp_layout_s* L) {
    L->geo_rec.clear();
    for (int h = 0; h < L->H; ++h)
        if (L->geo_n[(size_t)h] < 0) return;
    L->geo_rec.assign((size_t)L->H * kGeoRec, 0);
    for (int h = 0; h < L->H; ++h) {
        int32_t* r = &L->geo_rec[(size_t)h * kGeoRec];
        for (int k = 0; k < L->geo_n[(size_t)h]; ++k) {
            const bsp_affine_term_t& t = L->geo_terms[(size_t)h * BSP_MAX_AFFINE_TERMS + k];
            if (t.alpha == 1) {
                r[0] = 1;
                r[1] = t.beta;
                r[2] = t.kappa;
            } else {
                r[3] = 1;
                r[4] = t.beta;
                r[5] = t.sigma;
                r[6] = t.kappa;
                r[7] = t.causal;
            }
        }
    }
}

void affine_analyse(bsp_layout_s* L, const uint8_t* lay) {
    L->geo_n.assign((size_t)L->H, -1);
    L->geo_terms.assign((size_t)L->H * BSP_MAX_AFFINE_TERMS, bsp_affine_term_t{0, 0, 0, 0, 0});
    const size_t hsz = (size_t)L->nb * L->nb;
    for (int h = 0; h < L->H; ++h) {
        // heads equal to the previous one (a layout shared by all heads) reuse its answer
        if (h > 0 && std::equal(lay + (size_t)h * hsz, lay + (size_t)(h + 1) * hsz, lay + (size_t)(h - 1) * hsz)) {
            L->geo_n[(size_t)h] = L->geo_n[(size_t)h - 1];
            std::copy_n(&L->geo_terms[(size_t)(h - 1) * BSP_MAX_AFFINE_TERMS], BSP_MAX_AFFINE_TERMS,
                        &L->geo_terms[(size_t)h * BSP_MAX_AFFINE_TERMS]);
            continue;
        }
        L->geo_n[(size_t)h] = affine_detect(lay + (size_t)h * hsz, L->nb, &L->geo_terms[(size_t)h * BSP_MAX_AFFINE_TERMS]);
    }
    affine_records(L);
}

}  // namespace bsp

extern "C" int bsp_layout_geometry(bsp_layout_t L, int32_t* n_terms, bsp_affine_term_t* terms) {
    if (!L) return BSP_ERR_INVALID_ARG;
    for (int h = 0; h < L->H; ++h) {
        const bool known = (size_t)h < L->geo_n.size();
        if (n_terms) n_terms[h] = known ? L->geo_n[(size_t)h] : -1;
        for (int k = 0; k < BSP_MAX_AFFINE_TERMS && terms; ++k)
            terms[(size_t)h * BSP_MAX_AFFINE_TERMS + k] =
                known ? L->geo_terms[(size_t)h * BSP_MAX_AFFINE_TERMS + k] : bsp_affine_term_t{0, 0, 0, 0, 0};
    }
    return BSP_OK;
}
