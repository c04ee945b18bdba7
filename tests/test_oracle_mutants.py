"""The pins must catch plausible mistakes in the oracle.

Each case copies oracle.c to a temporary directory, plants one mistake (a
transposed operand, a wrong index, a dropped term, a wrong sign, an off-by-one
mask), builds it with gcc and runs the pin suite against it: at least one pin
has to fail.  The real oracle is never modified.
"""

import inspect
import os

import numpy as np
import pytest

import oracle as oracle_pkg
import test_oracle_pins as pins
from oracle import Oracle

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "oracle.c")

MUTANTS = {
    "sdd_transposed_b": ("double y = trans_b ? Bb[c * K + k] : Bb[(int64_t)k * S + c];",
                         "double y = trans_b ? Bb[(int64_t)k * S + c] : Bb[c * K + k];"),
    "softmax_no_max_in_sum": ("sum += exp(scale * (double)blk[b] - m);",
                              "sum += exp(scale * (double)blk[b]);"),
    "softmax_wrong_sign": ("double v = scale * (double)blk[b];",
                           "double v = -scale * (double)blk[b];"),
    "softmax_bad_normaliser": ("row_out[c] = exp(scale * (double)blk[b] - m) / sum;",
                               "row_out[c] = exp(scale * (double)blk[b] - m) / (sum + 1.0);"),
    "diag_causal_strict": ("return (r / B != c / B) || (c <= r);",
                           "return (r / B != c / B) || (c < r);"),
    "dsd_ignores_trans_a": ("int64_t rr = trans_a ? c : r, cc = trans_a ? r : c;\n"
                            "            if (ids[((int64_t)h * nb + rr / B) * nb + cc / B] < 0) continue;\n"
                            "            double x = sparse_at",
                            "int64_t rr = r, cc = c;\n"
                            "            if (ids[((int64_t)h * nb + rr / B) * nb + cc / B] < 0) continue;\n"
                            "            double x = sparse_at"),
    "dds_transposed_a": ("double x = trans_a ? Ab[k * M + m] : Ab[m * S + k];",
                         "double x = trans_a ? Ab[m * S + k] : Ab[k * M + m];"),
    "attention_wrong_value_row": ("o[d] += p * (double)Vb[c * D + d];",
                                  "o[d] += p * (double)Vb[r * D + d];"),
    "attention_transposed_layout": ("inR[c] = layout[((int64_t)h * nb + r / B) * nb + c / B] &&",
                                    "inR[c] = layout[((int64_t)h * nb + c / B) * nb + r / B] &&"),
    "attention_dropped_scale": ("sc[c] = scale * dot;", "sc[c] = dot;"),
    "csc_wrong_row": ("if (id >= 0) { row_idx[q] = i;", "if (id >= 0) { row_idx[q] = j;"),
    "sdd_wrong_block_row": ("int64_t r = (int64_t)bi[id] * B + a;", "int64_t r = (int64_t)bj[id] * B + a;"),
    "softmax_bwd_no_delta": ("dX[off + b] = scale * (double)Y[off + b] * ((double)dY[off + b] - dot);",
                             "dX[off + b] = scale * (double)Y[off + b] * ((double)dY[off + b]);"),
    "softmax_bwd_no_scale": ("dX[off + b] = scale * (double)Y[off + b] * ((double)dY[off + b] - dot);",
                             "dX[off + b] = (double)Y[off + b] * ((double)dY[off + b] - dot);"),
    "attention_bwd_dk_wrong_operand": ("gk[c * D + d] += scale * ds * (double)q[r * D + d];",
                                       "gk[c * D + d] += scale * ds * (double)k[c * D + d];"),
    "attention_bwd_dv_uses_ds": ("gv[c * D + d] += p * (double)go[r * D + d];",
                                 "gv[c * D + d] += ds * (double)go[r * D + d];"),
    "attention_bwd_unweighted_delta": ("delta += p * dp;", "delta += dp;"),
    "attention_bwd_transposed_layout": ("const uint8_t present = layout[((int64_t)h * nb + r / B) * nb + c / B];",
                                        "const uint8_t present = layout[((int64_t)h * nb + c / B) * nb + r / B];"),
    "affine_causal_ignored": ("if (causal && j > i) return 0;", "(void)causal;"),
    "affine_kappa_off_by_one": ("return d / sigma < kappa;", "return d / sigma <= kappa;"),
    "affine_row_slope_dropped": ("const int64_t d = j - alpha * i - beta;", "const int64_t d = j - beta;"),
    "lse_ignores_intra_block_mask": ("if (!present || !keep(kind, mask, S, B, row, c)) {", "if (!present) {"),
    "lse_drops_max": ("out[s] = top + log(total);", "out[s] = log(total);"),
    "lse_log2": ("out[s] = top + log(total);", "out[s] = top + log2(total);"),
}


def _pin_cases():
    """(name, callable(oracle)) for every pin, parametrised cases expanded."""
    cases = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if not params:
            cases.append((name, lambda o, fn=fn: fn(o)))
            continue
        argnames = [a.strip() for a in params[0].args[0].split(",")]
        for values in params[0].args[1]:
            values = values if isinstance(values, (tuple, list)) else (values,)
            kw = dict(zip(argnames, values))
            cases.append((f"{name}{list(values)}", lambda o, fn=fn, kw=kw: fn(o, **kw)))
    return cases


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, mutant):
    old, new = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {mutant} not unique"
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    lib = oracle_pkg.load(oracle_pkg.build(force=True, src=str(path), out=str(tmp_path / "libmut.so")))
    mut = Oracle(lib=lib)
    caught = []
    with np.errstate(all="ignore"):
        for name, run in _pin_cases():
            try:
                run(mut)
            except AssertionError:
                caught.append(name)
    assert caught, f"no pin caught mutant {mutant}"
