"""fp64 CPU oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The CUDA library never loads it, and it
loads nothing from the CUDA library: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
output rows); this module compiles it with gcc on first use and marshals numpy
arrays.  Inputs are passed as float32 arrays holding the dtype-rounded values
(exact for bf16, fp16 and fp32); every result is float64.

Pins: each function is checked in ``tests/test_oracle_pins.py`` against
library routines on special cases, closed forms and invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE = 0
MASK_DENSE = 1
MASK_DIAG_CAUSAL = 2


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_num_threads.restype = i32
    lib.oracle_count_nnz.restype = i64
    lib.oracle_count_nnz.argtypes = [P, i32, i32]
    lib.oracle_luts.argtypes = [P, i32, i32, P, P, P, P, P, P]
    lib.oracle_sdd.argtypes = [P, i32, i32, i32, i32, i32, i32, i32, P, P, i64, P, P]
    lib.oracle_softmax_rows.argtypes = [P, i32, i32, i32, i32, P, dbl, i32, P, i64, P, P]
    lib.oracle_softmax.argtypes = [P, i32, i32, i32, i32, P, dbl, i32, P, P]
    lib.oracle_dsd.argtypes = [P, i32, i32, i32, i32, i32, i32, i32, P, P, i64, P, P]
    lib.oracle_dds.argtypes = [P, i32, i32, i32, i32, i32, i32, i32, P, P, i64, P, P]
    lib.oracle_attention.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, dbl, i32, P, i64, P, P]
    lib.oracle_attention_lse.argtypes = [P, i32, i32, i32, i32, i32, P, P, dbl, i32, P, i64, P, P]
    lib.oracle_softmax_backward.argtypes = [P, i32, i32, i32, i32, P, P, dbl, P]
    lib.oracle_attention_backward.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, dbl, i32, P, P, P, P]
    lib.oracle_affine_expand.argtypes = [P, P, i32, i32, P]
    lib.oracle_affine_describable.restype = i32
    lib.oracle_affine_describable.argtypes = [P, i32]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  A path may be given to
    load another build of oracle.c (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (any float dtype) -> exact float32
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _u8(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.uint8)


def _ptr(a) -> ctypes.c_void_p:
    return ctypes.c_void_p(0) if a is None else ctypes.c_void_p(a.ctypes.data)


def _sel(sel, total):
    if sel is None:
        return None, total
    s = np.ascontiguousarray(sel, dtype=np.int64)
    if s.size and (s.min() < 0 or s.max() >= total):
        raise IndexError("selection out of range")
    return s, s.size


class Oracle:
    """Thin numpy front end over oracle.c.  `lib` defaults to the real build."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def nnz(self, layout) -> int:
        lay = _u8(layout)
        return int(self.lib.oracle_count_nnz(_ptr(lay), lay.shape[0], lay.shape[1]))

    def luts(self, layout):
        lay = _u8(layout)
        H, nb = lay.shape[0], lay.shape[1]
        nnz = self.nnz(lay)
        out = {k: np.zeros(H * (nb + 1) if k.endswith("ptr") else max(nnz, 1), dtype=np.int32)
               for k in ("row_ptr", "col_idx", "blk_id", "col_ptr", "row_idx", "blk_id_csc")}
        self.lib.oracle_luts(_ptr(lay), H, nb, *[_ptr(out[k]) for k in
                             ("row_ptr", "col_idx", "blk_id", "col_ptr", "row_idx", "blk_id_csc")])
        for k in ("col_idx", "blk_id", "row_idx", "blk_id_csc"):
            out[k] = out[k][:nnz]
        return out

    def sdd(self, layout, B, A, Bm, trans_a=0, trans_b=1, sel=None):
        """Blocks of op(A) op(B) on the layout.  A, Bm: [Z, H, ., .].
        Returns [Z, nnz, B, B] (sel None) or [len(sel), B, B]."""
        lay, A, Bm = _u8(layout), _f32(A), _f32(Bm)
        H, nb = lay.shape[0], lay.shape[1]
        Z = A.shape[0]
        K = A.shape[2] if trans_a else A.shape[3]
        nnz = self.nnz(lay)
        s, ns = _sel(sel, Z * nnz)
        out = np.zeros((ns, B, B), dtype=np.float64)
        self.lib.oracle_sdd(_ptr(lay), H, nb, B, Z, K, int(trans_a), int(trans_b),
                            _ptr(A), _ptr(Bm), ns, _ptr(s), _ptr(out))
        return out.reshape(Z, nnz, B, B) if sel is None else out

    def softmax(self, layout, B, X, scale, kind=MASK_NONE, mask=None):
        """Full block-format softmax: X [Z, nnz, B, B] -> [Z, nnz, B, B]."""
        lay, X = _u8(layout), _f32(X)
        m = None if mask is None else _u8(mask)
        H, nb = lay.shape[0], lay.shape[1]
        Z = X.shape[0]
        out = np.zeros(X.shape, dtype=np.float64)
        self.lib.oracle_softmax(_ptr(lay), H, nb, B, Z, _ptr(X), float(scale), int(kind),
                                _ptr(m), _ptr(out))
        return out

    def softmax_rows(self, layout, B, X, scale, kind=MASK_NONE, mask=None, sel=None):
        """Selected rows u = (z*H + h)*S + r as dense rows [len(sel), S]."""
        lay, X = _u8(layout), _f32(X)
        m = None if mask is None else _u8(mask)
        H, nb = lay.shape[0], lay.shape[1]
        Z, S = X.shape[0], nb * B
        s, ns = _sel(sel, Z * H * S)
        out = np.zeros((ns, S), dtype=np.float64)
        self.lib.oracle_softmax_rows(_ptr(lay), H, nb, B, Z, _ptr(X), float(scale), int(kind),
                                     _ptr(m), ns, _ptr(s), _ptr(out))
        return out

    def dsd(self, layout, B, Asp, Bd, trans_a=0, trans_b=0, sel=None):
        """op(A_sp) op(Bd).  Asp [Z, nnz, B, B]; Bd [Z, H, S, N] or [Z, H, N, S].
        Returns [Z, H, S, N] (sel None) or [len(sel), N]."""
        lay, Asp, Bd = _u8(layout), _f32(Asp), _f32(Bd)
        H, nb = lay.shape[0], lay.shape[1]
        Z, S = Bd.shape[0], nb * B
        N = Bd.shape[2] if trans_b else Bd.shape[3]
        s, ns = _sel(sel, Z * H * S)
        out = np.zeros((ns, N), dtype=np.float64)
        self.lib.oracle_dsd(_ptr(lay), H, nb, B, Z, N, int(trans_a), int(trans_b),
                            _ptr(Asp), _ptr(Bd), ns, _ptr(s), _ptr(out))
        return out.reshape(Z, H, S, N) if sel is None else out

    def dds(self, layout, B, Ad, Bsp, trans_a=0, trans_b=0, sel=None):
        """op(Ad) op(B_sp).  Ad [Z, H, M, S] or [Z, H, S, M]; Bsp [Z, nnz, B, B].
        Returns [Z, H, M, S] (sel None) or [len(sel), S]."""
        lay, Ad, Bsp = _u8(layout), _f32(Ad), _f32(Bsp)
        H, nb = lay.shape[0], lay.shape[1]
        Z, S = Ad.shape[0], nb * B
        M = Ad.shape[3] if trans_a else Ad.shape[2]
        s, ns = _sel(sel, Z * H * M)
        out = np.zeros((ns, S), dtype=np.float64)
        self.lib.oracle_dds(_ptr(lay), H, nb, B, Z, M, int(trans_a), int(trans_b),
                            _ptr(Ad), _ptr(Bsp), ns, _ptr(s), _ptr(out))
        return out.reshape(Z, H, M, S) if sel is None else out

    def attention(self, layout, B, Q, K, V, scale, kind=MASK_NONE, mask=None, sel=None):
        """Block-sparse attention.  Q, K, V [Z, H, S, D].
        Returns [Z, H, S, D] (sel None) or [len(sel), D]."""
        lay, Q, K, V = _u8(layout), _f32(Q), _f32(K), _f32(V)
        m = None if mask is None else _u8(mask)
        H, nb = lay.shape[0], lay.shape[1]
        Z, S, D = Q.shape[0], Q.shape[2], Q.shape[3]
        s, ns = _sel(sel, Z * H * S)
        out = np.zeros((ns, D), dtype=np.float64)
        self.lib.oracle_attention(_ptr(lay), H, nb, B, Z, D, _ptr(Q), _ptr(K), _ptr(V),
                                  float(scale), int(kind), _ptr(m), ns, _ptr(s), _ptr(out))
        return out.reshape(Z, H, S, D) if sel is None else out

    def attention_lse(self, layout, B, Q, K, scale, kind=MASK_NONE, mask=None, sel=None):
        """Log-sum-exp of every row's kept scaled scores (-inf for rows with
        nothing kept).  Q, K [Z, H, S, D].  Returns [Z, H, S] or [len(sel)]."""
        lay, Q, K = _u8(layout), _f32(Q), _f32(K)
        m = None if mask is None else _u8(mask)
        H, nb = lay.shape[0], lay.shape[1]
        Z, S, D = Q.shape[0], Q.shape[2], Q.shape[3]
        s, ns = _sel(sel, Z * H * S)
        out = np.zeros(ns, dtype=np.float64)
        self.lib.oracle_attention_lse(_ptr(lay), H, nb, B, Z, D, _ptr(Q), _ptr(K), float(scale), int(kind), _ptr(m),
                                      ns, _ptr(s), _ptr(out))
        return out.reshape(Z, H, S) if sel is None else out

    def softmax_backward(self, layout, B, Y, dY, scale):
        """Softmax backward in the block format: Y (the forward's output) and
        dY [Z, nnz, B, B] -> dX [Z, nnz, B, B]."""
        lay, Y, dY = _u8(layout), _f32(Y), _f32(dY)
        H, nb = lay.shape[0], lay.shape[1]
        out = np.zeros(Y.shape, dtype=np.float64)
        self.lib.oracle_softmax_backward(_ptr(lay), H, nb, B, Y.shape[0], _ptr(Y), _ptr(dY), float(scale),
                                         _ptr(out))
        return out

    def attention_backward(self, layout, B, Q, K, V, dO, scale, kind=MASK_NONE, mask=None):
        """Gradients (dQ, dK, dV) [Z, H, S, D] of block-sparse attention for
        the output gradient dO.  Dense S x S work per (z, h): small sizes."""
        lay, Q, K, V, dO = _u8(layout), _f32(Q), _f32(K), _f32(V), _f32(dO)
        m = None if mask is None else _u8(mask)
        H, nb = lay.shape[0], lay.shape[1]
        Z, D = Q.shape[0], Q.shape[3]
        outs = [np.zeros(Q.shape, dtype=np.float64) for _ in range(3)]
        self.lib.oracle_attention_backward(_ptr(lay), H, nb, B, Z, D, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO),
                                           float(scale), int(kind), _ptr(m), *[_ptr(o) for o in outs])
        return tuple(outs)

    def affine_expand(self, n_terms, terms, nb):
        """0/1 layout [H, nb, nb] of per-head affine terms: n_terms [H] (0..2),
        terms [H, 2, 5] rows (alpha, beta, sigma, kappa, causal)."""
        n = np.ascontiguousarray(n_terms, dtype=np.int32)
        t = np.ascontiguousarray(terms, dtype=np.int32).reshape(n.size, 2, 5)
        out = np.zeros((n.size, nb, nb), dtype=np.uint8)
        self.lib.oracle_affine_expand(_ptr(n), _ptr(t), n.size, nb, _ptr(out))
        return out

    def affine_describable(self, head) -> bool:
        """Whether a band term and / or a column term reproduce one head's
        [nb, nb] layout exactly (exhaustive search: nb up to about 10)."""
        lay = _u8(head)
        return bool(self.lib.oracle_affine_describable(_ptr(lay), lay.shape[0]))
