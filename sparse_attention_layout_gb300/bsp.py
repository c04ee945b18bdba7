"""Thin ctypes binding of libbsp (the C ABI declared in include/bsp.h).

Argument marshalling only: every step of every operation runs in the CUDA
library.  PyTorch supplies device memory (output allocation) and the current
stream.  If the library is missing the first call raises: there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

MASK_NONE, MASK_DENSE, MASK_DIAG_CAUSAL = 0, 1, 2
F32, BF16, F16 = 0, 1, 2
_DTYPES = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}

STATUS = {0: "BSP_OK", -1: "BSP_ERR_INVALID_ARG", -2: "BSP_ERR_UNSUPPORTED",
          -3: "BSP_ERR_ALIGNMENT", -4: "BSP_ERR_OOM", -5: "BSP_ERR_CUDA",
          -6: "BSP_ERR_TIMEOUT", -7: "BSP_ERR_DEVICE_CHECK"}

_lib = None


class BspError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({lib().bsp_status_string(code).decode()})")


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded libbsp (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libbsp.so not found at {path}; build it with "
                               "sparse_attention_layout_gb300.build.build()")
        L = ctypes.CDLL(path)
        P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.bsp_layout_plan.argtypes = [P, i32, i32, i32, ctypes.POINTER(P)]
        L.bsp_layout_compile.argtypes = [P, i32, i32, i32, P, ctypes.POINTER(P)]
        L.bsp_layout_compile_device.argtypes = [P, i32, i32, i32, P, ctypes.POINTER(P)]
        L.bsp_layout_destroy.argtypes = [P]
        L.bsp_layout_info.argtypes = [P, P, P, P, P]
        L.bsp_layout_get_luts.argtypes = [P] * 7
        L.bsp_layout_tiles.argtypes = [P] * 8
        L.bsp_sdd.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, P]
        L.bsp_sdd_softmax.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, f32, i32, P, P]
        L.bsp_dsd.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, P]
        L.bsp_dds.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, P]
        L.bsp_softmax.argtypes = [P, i32, P, P, i32, f32, i32, P, P]
        L.bsp_attention.argtypes = [P, i32, P, P, P, P, i32, i32, f32, i32, P, P]
        L.bsp_softmax_backward.argtypes = [P, i32, P, P, P, i32, f32, P]
        L.bsp_attention_backward.argtypes = [P, i32, P, P, P, P, P, P, P, i32, i32, f32, i32, P, P, P, P]
        L.bsp_attention_lse.argtypes = [P, i32, P, P, P, P, P, i32, i32, f32, i32, P, P]
        L.bsp_attention_backward_lse.argtypes = [P, i32, P, P, P, P, P, P, P, P, P, i32, i32, f32, i32, P, P, P,
                                                 P]
        L.bsp_layout_groups.argtypes = [P, i32, P, P, P, P, P, P, P]
        L.bsp_layout_softmax_chunks.argtypes = [P, i32, P, P, P, P]
        L.bsp_layout_geometry.argtypes = [P, P, P]
        L.bsp_layout_compile_affine.argtypes = [P, P, i32, i32, i32, P, ctypes.POINTER(P)]
        L.bsp_attention_host.argtypes = [P, i32, P, P, P, P, i32, i32, f32, i32, P, P, ctypes.c_size_t, i32, P]
        L.bsp_diag_attention_schedule.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P]
        L.bsp_diag_attention_split.argtypes = [P, i32]
        L.bsp_attention_host_workspace.argtypes = [P, i32, i32, i32]
        L.bsp_attention_host_workspace.restype = ctypes.c_size_t
        L.bsp_status_check.argtypes = [P, P]
        L.bsp_diag_wait_limit.argtypes = [P, ctypes.c_uint64, i32]
        L.bsp_diag_wait_limit.restype = i32
        L.bsp_status_string.restype = ctypes.c_char_p
        L.bsp_status_string.argtypes = [i32]
        L.bsp_version.restype = ctypes.c_char_p
        for name in ("bsp_layout_plan", "bsp_layout_compile", "bsp_layout_compile_device", "bsp_layout_destroy",
                     "bsp_layout_info",
                     "bsp_layout_get_luts", "bsp_layout_tiles", "bsp_sdd", "bsp_dsd", "bsp_dds", "bsp_softmax",
                     "bsp_attention", "bsp_softmax_backward", "bsp_attention_backward", "bsp_layout_groups",
                     "bsp_layout_softmax_chunks",
                     "bsp_status_check", "bsp_layout_geometry", "bsp_layout_compile_affine", "bsp_attention_host", "bsp_sdd_softmax",
                     "bsp_attention_lse", "bsp_attention_backward_lse"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        raise BspError(rc, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dtype(*ts):
    d = ts[0].dtype
    for t in ts:
        if t.dtype != d:
            raise TypeError("all tensors of a call must share one dtype")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if d not in _DTYPES:
        raise TypeError(f"unsupported dtype {d}")
    return _DTYPES[d]


class Layout:
    """Owning wrapper of a bsp_layout_t handle."""

    def __init__(self, handle: ctypes.c_void_p, layout: np.ndarray, block: int):
        self.handle = handle
        self.layout = layout
        self.block = block
        H, nb, B, nnz = (ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int64())
        _check(lib().bsp_layout_info(handle, ctypes.byref(H), ctypes.byref(nb), ctypes.byref(B),
                                     ctypes.byref(nnz)), "bsp_layout_info")
        self.H, self.nb, self.B, self.nnz = H.value, nb.value, B.value, nnz.value
        self.S = self.nb * self.B

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.bsp_layout_destroy(self.handle)
            self.handle = None

    def luts(self) -> dict:
        H, nb, nnz = self.H, self.nb, self.nnz
        out = {k: np.zeros(H * (nb + 1) if k.endswith("ptr") else max(nnz, 1), np.int32)
               for k in ("row_ptr", "col_idx", "blk_id", "col_ptr", "row_idx", "blk_id_csc")}
        _check(lib().bsp_layout_get_luts(self.handle, *[ctypes.c_void_p(out[k].ctypes.data) for k in
                                                        ("row_ptr", "col_idx", "blk_id", "col_ptr",
                                                         "row_idx", "blk_id_csc")]),
               "bsp_layout_get_luts")
        for k in ("col_idx", "blk_id", "row_idx", "blk_id_csc"):
            out[k] = out[k][:nnz]
        return out

    def tiles(self) -> dict:
        G, nt, ns = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
        f = lib().bsp_layout_tiles
        _check(f(self.handle, ctypes.byref(G), ctypes.byref(nt), ctypes.byref(ns), None, None, None, None),
               "bsp_layout_tiles")
        G, nt, ns = G.value, nt.value, ns.value
        out = {"tile_step_ptr": np.zeros(nt + 1, np.int32), "tile_order": np.zeros(max(nt, 1), np.int32),
               "step_col": np.zeros(max(ns * G, 1), np.int32), "step_blk": np.zeros(max(ns * G * G, 1), np.int32)}
        _check(f(self.handle, None, None, None, *[ctypes.c_void_p(out[k].ctypes.data) for k in
                                                  ("tile_step_ptr", "tile_order", "step_col", "step_blk")]),
               "bsp_layout_tiles")
        out["step_col"] = out["step_col"][:ns * G].reshape(ns, G)
        out["step_blk"] = out["step_blk"][:ns * G * G].reshape(ns, G, G)
        out["tile_order"] = out["tile_order"][:nt]
        out.update(G=G, n_tiles=nt, n_steps=ns)
        return out


    def groups(self, orient: int) -> dict:
        """Line groups of the tensor-core DSD / DDS kernels (orient 0: block-rows,
        1: block-columns)."""
        G, ng, ns = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
        f = lib().bsp_layout_groups
        _check(f(self.handle, int(orient), ctypes.byref(G), ctypes.byref(ng), ctypes.byref(ns), None, None,
                 None, None), "bsp_layout_groups")
        G, ng, ns = G.value, ng.value, ns.value
        out = {"grp_ptr": np.zeros(ng + 1, np.int32), "grp_order": np.zeros(max(ng, 1), np.int32),
               "slot_idx": np.zeros(max(ns, 1), np.int32), "slot_blk": np.zeros(max(ns * G, 1), np.int32)}
        _check(f(self.handle, int(orient), None, None, None,
                 *[ctypes.c_void_p(out[k].ctypes.data) for k in ("grp_ptr", "grp_order", "slot_idx", "slot_blk")]),
               "bsp_layout_groups")
        out["grp_order"] = out["grp_order"][:ng]
        out["slot_idx"] = out["slot_idx"][:ns]
        out["slot_blk"] = out["slot_blk"][:ns * G].reshape(ns, G)
        out.update(G=G, n_groups=ng, n_slots=ns)
        return out

    def softmax_chunks(self, elt_bytes: int) -> dict:
        """Chunks of the softmax for 2- or 4-byte elements: items [n, 4] int32
        (h*nb + i, first block id, blocks in the row, r0 | R << 16), the largest
        chunk's bytes and whether every row fits one chunk."""
        n, mb, fits = ctypes.c_int64(), ctypes.c_int(), ctypes.c_int()
        f = lib().bsp_layout_softmax_chunks
        _check(f(self.handle, int(elt_bytes), ctypes.byref(n), ctypes.byref(mb), ctypes.byref(fits), None),
               "bsp_layout_softmax_chunks")
        items = np.zeros((max(n.value, 1), 4), np.int32)
        _check(f(self.handle, int(elt_bytes), None, None, None, ctypes.c_void_p(items.ctypes.data)),
               "bsp_layout_softmax_chunks")
        return {"items": items[:n.value], "max_bytes": mb.value, "fits": bool(fits.value)}

    def geometry(self):
        """Affine description per head: (n_terms [H] int32, -1 = none;
        terms [H, 2, 5] int32 rows (alpha, beta, sigma, kappa, causal))."""
        n = np.zeros(self.H, np.int32)
        t = np.zeros((self.H, MAX_AFFINE_TERMS, 5), np.int32)
        _check(lib().bsp_layout_geometry(self.handle, ctypes.c_void_p(n.ctypes.data), ctypes.c_void_p(t.ctypes.data)),
               "bsp_layout_geometry")
        return n, t


def _layout_args(layout, block):
    lay = np.ascontiguousarray(layout, dtype=np.uint8)
    if lay.ndim != 3 or lay.shape[1] != lay.shape[2]:
        raise ValueError("layout must be [H, nb, nb]")
    return lay, lay.shape[0], lay.shape[1], int(block)


def bsp_layout_plan(layout, block: int) -> Layout:
    lay, H, nb, B = _layout_args(layout, block)
    h = ctypes.c_void_p()
    _check(lib().bsp_layout_plan(ctypes.c_void_p(lay.ctypes.data), H, nb, B, ctypes.byref(h)),
           "bsp_layout_plan")
    return Layout(h, lay, B)


def bsp_layout_compile(layout, block: int, stream=None) -> Layout:
    lay, H, nb, B = _layout_args(layout, block)
    h = ctypes.c_void_p()
    _check(lib().bsp_layout_compile(ctypes.c_void_p(lay.ctypes.data), H, nb, B, _stream(stream),
                                    ctypes.byref(h)), "bsp_layout_compile")
    return Layout(h, lay, B)


def bsp_layout_compile_device(layout, block: int, stream=None) -> Layout:
    """Compile a layout held in device memory (torch uint8 CUDA tensor
    [H, nb, nb]) on the device."""
    if not (isinstance(layout, torch.Tensor) and layout.is_cuda and layout.dtype == torch.uint8):
        raise TypeError("layout must be a CUDA uint8 tensor")
    lay = layout.contiguous()
    if lay.dim() != 3 or lay.shape[1] != lay.shape[2]:
        raise ValueError("layout must be [H, nb, nb]")
    h = ctypes.c_void_p()
    _check(lib().bsp_layout_compile_device(ctypes.c_void_p(lay.data_ptr()), lay.shape[0], lay.shape[1], int(block),
                                           _stream(stream), ctypes.byref(h)), "bsp_layout_compile_device")
    return Layout(h, None, int(block))


MAX_AFFINE_TERMS = 2


def bsp_layout_compile_affine(n_terms, terms, nb: int, block: int, stream=None) -> Layout:
    """Compile a layout given by per-head affine terms (n_terms [H], terms
    [H, 2, 5] rows (alpha, beta, sigma, kappa, causal)) on the device."""
    n = np.ascontiguousarray(n_terms, dtype=np.int32)
    t = np.ascontiguousarray(terms, dtype=np.int32).reshape(n.size, MAX_AFFINE_TERMS, 5)
    h = ctypes.c_void_p()
    _check(lib().bsp_layout_compile_affine(ctypes.c_void_p(n.ctypes.data), ctypes.c_void_p(t.ctypes.data), n.size,
                                           int(nb), int(block), _stream(stream), ctypes.byref(h)),
           "bsp_layout_compile_affine")
    return Layout(h, None, int(block))


def bsp_sdd(L: Layout, A, B, C=None, trans_a: int = 0, trans_b: int = 1, stream=None):
    """C[z, n] = block n of op(A) op(B).  A, B: [Z, H, ., .] device tensors."""
    Z = A.shape[0]
    K = A.shape[2] if trans_a else A.shape[3]
    if C is None:
        C = torch.empty((Z, L.nnz, L.B, L.B), dtype=A.dtype, device=A.device)
    dt = _dtype(A, B, C)
    _check(lib().bsp_sdd(L.handle, dt, _ptr(A), _ptr(B), _ptr(C), Z, K, int(trans_a), int(trans_b),
                         _stream(stream)), "bsp_sdd")
    return C


def bsp_sdd_softmax(L: Layout, A, B, P=None, scale: float = 1.0, mask_kind: int = MASK_NONE, mask=None,
                    trans_a: int = 0, trans_b: int = 1, stream=None):
    """P = softmax(scale * SDD(op(A), op(B))) in one fused pass."""
    Z = A.shape[0]
    K = A.shape[2] if trans_a else A.shape[3]
    if P is None:
        P = torch.empty((Z, L.nnz, L.B, L.B), dtype=A.dtype, device=A.device)
    dt = _dtype(A, B, P)
    _check(lib().bsp_sdd_softmax(L.handle, dt, _ptr(A), _ptr(B), _ptr(P), Z, K, int(trans_a), int(trans_b),
                                 float(scale), int(mask_kind), _ptr(mask), _stream(stream)), "bsp_sdd_softmax")
    return P


def bsp_dsd(L: Layout, A_sp, B, C=None, trans_a: int = 0, trans_b: int = 0, stream=None):
    """C = op(A_sp) op(B).  A_sp [Z, nnz, B, B]; B [Z, H, S, N] or [Z, H, N, S]."""
    Z = B.shape[0]
    N = B.shape[2] if trans_b else B.shape[3]
    if C is None:
        C = torch.empty((Z, L.H, L.S, N), dtype=B.dtype, device=B.device)
    dt = _dtype(A_sp, B, C)
    _check(lib().bsp_dsd(L.handle, dt, _ptr(A_sp), _ptr(B), _ptr(C), Z, N, int(trans_a), int(trans_b),
                         _stream(stream)), "bsp_dsd")
    return C


def bsp_dds(L: Layout, A, B_sp, C=None, trans_a: int = 0, trans_b: int = 0, stream=None):
    """C = op(A) op(B_sp).  A [Z, H, M, S] or [Z, H, S, M]; B_sp [Z, nnz, B, B]."""
    Z = A.shape[0]
    M = A.shape[3] if trans_a else A.shape[2]
    if C is None:
        C = torch.empty((Z, L.H, M, L.S), dtype=A.dtype, device=A.device)
    dt = _dtype(A, B_sp, C)
    _check(lib().bsp_dds(L.handle, dt, _ptr(A), _ptr(B_sp), _ptr(C), Z, M, int(trans_a), int(trans_b),
                         _stream(stream)), "bsp_dds")
    return C


def bsp_softmax(L: Layout, X, Y=None, scale: float = 1.0, mask_kind: int = MASK_NONE, mask=None,
                stream=None):
    """Row softmax of scale * X on the layout.  Y = X for in place."""
    if Y is None:
        Y = torch.empty_like(X)
    dt = _dtype(X, Y)
    _check(lib().bsp_softmax(L.handle, dt, _ptr(X), _ptr(Y), X.shape[0], float(scale), int(mask_kind),
                             _ptr(mask), _stream(stream)), "bsp_softmax")
    return Y


def bsp_attention(L: Layout, Q, K, V, O=None, scale: float = 1.0, mask_kind: int = MASK_NONE,
                  mask=None, stream=None):
    """Fused block-sparse attention.  Q, K, V, O: [Z, H, S, D]."""
    if O is None:
        O = torch.empty_like(Q)
    dt = _dtype(Q, K, V, O)
    _check(lib().bsp_attention(L.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), Q.shape[0], Q.shape[3],
                               float(scale), int(mask_kind), _ptr(mask), _stream(stream)),
           "bsp_attention")
    return O


def bsp_attention_host_workspace(L: Layout, dtype, D: int, z_slice: int) -> int:
    """Device workspace bytes of bsp_attention_host for slices of z_slice batch entries."""
    return int(lib().bsp_attention_host_workspace(L.handle, _DTYPES[dtype], int(D), int(z_slice)))


HOST_RESERVED_WORKSPACE = 1


def bsp_attention_host(L: Layout, Q, K, V, O=None, scale: float = 1.0, mask_kind: int = MASK_NONE,
                       mask=None, workspace=None, reserved_workspace: bool = False, stream=None):
    """Fused attention on HOST tensors Q, K, V (O allocated pinned when None);
    the library copies slices of the batch in and out on its own streams,
    overlapped with the kernels.  workspace: device uint8 tensor (allocated for
    slices of one batch entry when None).  reserved_workspace: the workspace is
    used by nothing but this handle's calls in between, so a call may start its
    input copies during the previous call's tail."""
    if O is None:
        O = torch.empty(Q.shape, dtype=Q.dtype, pin_memory=True)
    if any(t.is_cuda for t in (Q, K, V, O)):
        raise ValueError("bsp_attention_host takes host tensors")
    dt = _dtype(Q, K, V, O)
    if workspace is None:
        nbytes = bsp_attention_host_workspace(L, Q.dtype, Q.shape[3], 1)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    _check(lib().bsp_attention_host(L.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), Q.shape[0], Q.shape[3],
                                    float(scale), int(mask_kind), _ptr(mask), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    HOST_RESERVED_WORKSPACE if reserved_workspace else 0, _stream(stream)),
           "bsp_attention_host")
    return O


def bsp_status_check(L: Layout, stream=None) -> int:
    return int(lib().bsp_status_check(L.handle, _stream(stream)))


INJECT_SKIP_FIRST_Q, INJECT_BAD_COLUMN = 1, 2


def bsp_diag_wait_limit(L: Layout, wait_ns: int = 0, inject: int = 0):
    """Wait limit of the handle's tensor-core kernels (0 = the 2 s default)
    and test injections (INJECT_* bits; 0 = none)."""
    _check(lib().bsp_diag_wait_limit(L.handle, int(wait_ns), int(inject)), "bsp_diag_wait_limit")


def bsp_diag_attention_schedule(L: Layout, Z: int, n_sm: int, dtype=torch.bfloat16):
    """The fused attention kernel's work schedule, computed on the host:
    dict(grid, ptr [grid + 1], items [n, 4] (tile, first step, step count,
    batch entry), part [n] (partial-result slot of a piece of a cut tile, else
    -1), combine [n_split, 4] (tile, batch entry, first slot, pieces)); CTA c
    runs items[ptr[c]:ptr[c + 1]]."""
    f = lib().bsp_diag_attention_schedule
    dt = _DTYPES[dtype]
    g, n, ns = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(f(L.handle, dt, int(Z), int(n_sm), ctypes.byref(g), ctypes.byref(n), ctypes.byref(ns), None, None, None, None),
           "bsp_diag_attention_schedule")
    out = {"ptr": np.zeros(g.value + 1, np.int32), "items": np.zeros((max(n.value, 1), 4), np.int32),
           "part": np.zeros(max(n.value, 1), np.int32), "combine": np.zeros((max(ns.value, 1), 4), np.int32)}
    _check(f(L.handle, dt, int(Z), int(n_sm), ctypes.byref(g), ctypes.byref(n), ctypes.byref(ns),
             *[ctypes.c_void_p(out[k].ctypes.data) for k in ("ptr", "items", "part", "combine")]),
           "bsp_diag_attention_schedule")
    out["items"], out["part"], out["combine"] = out["items"][:n.value], out["part"][:n.value], out["combine"][:ns.value]
    out["grid"] = g.value
    return out


def bsp_diag_attention_split(L: Layout, max_steps: int):
    """Cutting of long tiles by the handle's fused attention kernels: 0
    automatic (default), > 0 every tile of more than max_steps steps, < 0
    never."""
    _check(lib().bsp_diag_attention_split(L.handle, int(max_steps)), "bsp_diag_attention_split")


def attention_unfused(L: Layout, Q, K, V, scale: float, mask_kind: int = MASK_NONE, mask=None,
                      stream=None):
    """The SDD -> softmax -> DSD chain: scores and probabilities go through HBM."""
    P = bsp_sdd(L, Q, K, trans_a=0, trans_b=1, stream=stream)
    bsp_softmax(L, P, P, scale, mask_kind, mask, stream=stream)
    return bsp_dsd(L, P, V, stream=stream)


# --------------------------------------------------------------- backward --

def bsp_softmax_backward(L: Layout, Y, dY, dX=None, scale: float = 1.0, stream=None):
    """Gradient of the softmax input: scale * Y * (dY - rowsum(Y * dY)).
    dX = dY for in place."""
    if dX is None:
        dX = torch.empty_like(dY)
    dt = _dtype(Y, dY, dX)
    _check(lib().bsp_softmax_backward(L.handle, dt, _ptr(Y), _ptr(dY), _ptr(dX), Y.shape[0], float(scale),
                                      _stream(stream)), "bsp_softmax_backward")
    return dX


def attention_backward(L: Layout, Q, K, V, dO, scale: float, mask_kind: int = MASK_NONE, mask=None,
                       stream=None):
    """(dQ, dK, dV) of block-sparse attention for the output gradient dO.
    Allocates the two [Z, nnz, B, B] workspaces the C call takes."""
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    ws = (Q.shape[0], max(L.nnz, 1), L.B, L.B)
    P_ws = torch.empty(ws, dtype=Q.dtype, device=Q.device) if L.nnz else None
    dP_ws = torch.empty(ws, dtype=Q.dtype, device=Q.device) if L.nnz else None
    dt = _dtype(Q, K, V, dO, dQ, dK, dV)
    _check(lib().bsp_attention_backward(L.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), _ptr(dK),
                                        _ptr(dV), Q.shape[0], Q.shape[3], float(scale), int(mask_kind),
                                        _ptr(mask), _ptr(P_ws), _ptr(dP_ws), _stream(stream)),
           "bsp_attention_backward")
    return dQ, dK, dV


def bsp_attention_lse(L: Layout, Q, K, V, O=None, lse=None, scale: float = 1.0, mask_kind: int = MASK_NONE,
                      mask=None, stream=None):
    """Fused attention that also returns each row's log-sum-exp of its kept
    scaled scores: (O [Z, H, S, D], lse fp32 [Z, H, S])."""
    if O is None:
        O = torch.empty_like(Q)
    if lse is None:
        lse = torch.empty(Q.shape[:3], dtype=torch.float32, device=Q.device)
    dt = _dtype(Q, K, V, O)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor")
    _check(lib().bsp_attention_lse(L.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), Q.shape[0],
                                   Q.shape[3], float(scale), int(mask_kind), _ptr(mask), _stream(stream)),
           "bsp_attention_lse")
    return O, lse


def attention_backward_lse(L: Layout, Q, K, V, O, dO, lse, scale: float, mask_kind: int = MASK_NONE, mask=None,
                           stream=None):
    """(dQ, dK, dV) given the forward's output O and lse (bsp_attention_lse).
    Allocates the two [Z, nnz, B, B] workspaces the C call takes."""
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    ws = (Q.shape[0], max(L.nnz, 1), L.B, L.B)
    P_ws = torch.empty(ws, dtype=Q.dtype, device=Q.device) if L.nnz else None
    dP_ws = torch.empty(ws, dtype=Q.dtype, device=Q.device) if L.nnz else None
    dt = _dtype(Q, K, V, O, dO, dQ, dK, dV)
    _check(lib().bsp_attention_backward_lse(L.handle, dt, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse),
                                            _ptr(dQ), _ptr(dK), _ptr(dV), Q.shape[0], Q.shape[3], float(scale),
                                            int(mask_kind), _ptr(mask), _ptr(P_ws), _ptr(dP_ws), _stream(stream)),
           "bsp_attention_backward_lse")
    return dQ, dK, dV


class _BlockSparseAttention(torch.autograd.Function):
    """Fused forward keeping the rows' log-sum-exp (bsp_attention_lse);
    backward through bsp_attention_backward_lse."""

    @staticmethod
    def forward(ctx, Q, K, V, L, scale, mask_kind, mask):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        O, lse = bsp_attention_lse(L, Q, K, V, None, None, scale, mask_kind, mask)
        ctx.save_for_backward(Q, K, V, O, lse)
        ctx.L, ctx.scale, ctx.mask_kind, ctx.mask = L, scale, mask_kind, mask
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, lse = ctx.saved_tensors
        dQ, dK, dV = attention_backward_lse(ctx.L, Q, K, V, O, dO.contiguous(), lse, ctx.scale, ctx.mask_kind,
                                            ctx.mask)
        return dQ, dK, dV, None, None, None, None


def block_sparse_attention(L: Layout, Q, K, V, scale: float, mask_kind: int = MASK_NONE, mask=None):
    """Differentiable block-sparse attention (torch autograd) on a compiled layout."""
    return _BlockSparseAttention.apply(Q, K, V, L, float(scale), int(mask_kind), mask)
