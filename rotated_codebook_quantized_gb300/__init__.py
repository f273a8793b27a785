"""Python binding of libtq.so, the CUDA library of rotated-codebook quantization.

Argument marshalling only: every function here checks shapes, allocates the
output tensors with torch (device memory), and calls the C entry point of the
same name on torch's current CUDA stream.  All arithmetic runs in the library's
kernels.  There is no CPU fallback: if the library cannot be loaded, ``load()``
raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq.so")

TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2
TQ_OK, TQ_ERR_INVALID, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_TIMEOUT, TQ_ERR_DEVICE = range(6)
TQ_DEVERR_BAD_ID, TQ_DEVERR_TIMEOUT, TQ_DEVERR_BAD_BOOK = 1, 2, 4

_c_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_sz = ctypes.c_size_t


class tq_codebook_t(ctypes.Structure):
    _fields_ = [("levels", _i32), ("centroids", _c_p), ("thresholds", _c_p)]


class tq_rotation_t(ctypes.Structure):
    _fields_ = [("dim", _i32), ("block", _i32), ("signs", _c_p)]


class tq_qweight_t(ctypes.Structure):
    _fields_ = [("codes", _c_p), ("scales", _c_p), ("experts", _i32), ("rows", _i32), ("cols", _i32),
                ("group", _i32), ("row_stride_words", _i64), ("expert_stride_words", _i64),
                ("expert_stride_scales", _i64), ("cb", tq_codebook_t)]


class tq_layer_desc_t(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 64), ("experts", _i32), ("rows", _i32), ("cols", _i32), ("group", _i32),
                ("row_stride_words", _i64), ("levels", _i32), ("rot_dim", _i32), ("rot_block", _i32),
                ("rot_seed", ctypes.c_uint64), ("centroids", _c_p), ("codes", _c_p), ("scales", _c_p)]


class tq_tier_policy_t(ctypes.Structure):
    _fields_ = [(n, _i32) for n in ("down_levels", "down_group", "expert_levels", "expert_group", "mlp_levels",
                                    "mlp_group", "attn_levels", "attn_group", "other_levels", "other_group")]


_P = ctypes.POINTER
# name -> (restype, argtypes), exactly the declarations of include/tq.h
_SIGS = {
    "tq_status_string": (ctypes.c_char_p, [_i32]),
    "tq_codes_per_word": (_i32, [_i32]),
    "tq_row_words": (_i64, [_i32, _i32]),
    "tq_row_stride_words": (_i64, [_i32, _i32]),
    "tq_codebook": (_i32, [_i32, _P(ctypes.c_double), _P(ctypes.c_double)]),
    "tq_rotation_signs": (_i32, [ctypes.c_uint64, _i32, _P(ctypes.c_int8)]),
    "tq_rotate": (_i32, [_P(tq_rotation_t), _c_p, _i32, _i64, _c_p, _i32, _c_p]),
    "tq_quantize": (_i32, [_c_p, _i32, _i64, _i32, _i32, _P(tq_rotation_t), _P(tq_codebook_t), _c_p, _c_p, _i64,
                           _c_p]),
    "tq_qmv": (_i32, [_P(tq_qweight_t), _c_p, _i32, _c_p, _i32, _c_p]),
    "tq_qmv_tc": (_i32, [_P(tq_qweight_t), _c_p, _i32, _c_p, _c_p, _sz, _c_p, _c_p]),
    "tq_qmv_tc_workspace_bytes": (_sz, [_i32, _i32]),
    "tq_gather_qmv": (_i32, [_P(tq_qweight_t), _c_p, _c_p, _i32, _i32, _c_p, _i32, _c_p, _sz, _c_p, _c_p]),
    "tq_gather_qmv_workspace_bytes": (_sz, [_P(tq_qweight_t), _i32, _i32]),
    "tq_multi_gather_qmv": (_i32, [_P(tq_qweight_t), _c_p, _c_p, _i32, _c_p, _i32, _c_p, _sz, _c_p, _c_p]),
    "tq_multi_gather_qmv_workspace_bytes": (_sz, [_P(tq_qweight_t), _i32]),
    "tq_gather_qmv_rotate": (_i32, [_P(tq_qweight_t), _c_p, _i32, _P(tq_rotation_t), _c_p, _i32, _i32, _c_p, _i32,
                                    _c_p, _c_p]),
    "tq_multi_gather_qmv_swiglu": (_i32, [_P(tq_qweight_t), _c_p, _P(tq_rotation_t), _c_p, _i32, _c_p, _i32, _c_p,
                                          _c_p]),
    "tq_moe_route": (_i32, [_c_p, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _sz, _c_p]),
    "tq_route_workspace_bytes": (_sz, [_i32]),
    "tq_swiglu_rotate": (_i32, [_c_p, _i64, _i32, _P(tq_rotation_t), _c_p, _i32, _c_p]),
    "tq_moe_combine": (_i32, [_c_p, _c_p, _c_p, _i32, _i32, _i32, _c_p, _i32, _c_p]),
    "tq_gather_qmm": (_i32, [_P(tq_qweight_t), _c_p, _i32, _c_p, _c_p, _i32, _i32, _i32, _c_p, _i32, _c_p, _sz,
                             _c_p, _c_p]),
    "tq_gather_qmm_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "tq_dequant_experts": (_i32, [_P(tq_qweight_t), _c_p, _i32, _c_p, _i32, _c_p, _c_p]),
    "tq_kv_quantize": (_i32, [_c_p, _c_p, _i32, _i32, _i32, _i32, _i64, _i64, _P(tq_rotation_t),
                              _P(tq_codebook_t), _P(tq_codebook_t), _i32, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "tq_kv_attend": (_i32, [_c_p, _i32, _i32, _i32, _i32, _i64, _i64, _P(tq_rotation_t), _P(tq_codebook_t),
                            _P(tq_codebook_t), _i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _sz, _c_p]),
    "tq_kv_attend_workspace_bytes": (_sz, [_i32, _i32, _i64]),
    "tq_kv_attend_noalloc": (_i32, [_c_p, _i32, _i32, _i32, _i32, _i64, _i64, _P(tq_rotation_t), _P(tq_codebook_t),
                                    _P(tq_codebook_t), _i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "tq_kv_attend_noalloc_max_scratch_bytes": (_sz, []),
    "tq_moe_decode_layer_workspace_bytes": (_sz, [_P(tq_qweight_t), _P(tq_qweight_t), _i32]),
    "tq_moe_decode_layer": (_i32, [_P(tq_qweight_t), _P(tq_qweight_t), _P(tq_rotation_t), _P(tq_rotation_t), _c_p,
                                   _c_p, _i32, _i32, _c_p, _i32, _c_p, _sz, _c_p, _c_p]),
    "tq_check_error": (_i32, [_c_p, _P(_u32), _c_p]),
    "tq_set_wait_budget": (_i32, [_i64]),
    "tq_rotation_dense": (_i32, [ctypes.c_uint64, _i32, _P(ctypes.c_double)]),
    "tq_rotate_dense": (_i32, [_c_p, _i32, _c_p, _i32, _i64, _c_p, _i32, _c_p]),
    "tq_layer_tier": (_i32, [ctypes.c_char_p, _P(tq_tier_policy_t), _P(_i32), _P(_i32)]),
    "tq_pack_file_write": (_i32, [ctypes.c_char_p, _P(tq_layer_desc_t), _i32]),
    "tq_pack_file_info": (_i32, [ctypes.c_char_p, _P(_i32), _P(tq_layer_desc_t), _i32]),
    "tq_pack_file_read_layer": (_i32, [ctypes.c_char_p, _i32, _c_p, _c_p, _c_p]),
    "tq_expert_cache_create": (_i32, [_P(tq_qweight_t), _i32, _c_p, _c_p, _P(_c_p)]),
    "tq_expert_cache_destroy": (None, [_c_p]),
    "tq_expert_cache_plan": (_i32, [_c_p, _c_p, _i32, _c_p, _c_p]),
    "tq_expert_cache_map": (_i32, [_c_p, _c_p, _i32, _c_p, _c_p]),
    "tq_expert_cache_stats": (_i32, [_c_p, _P(_i64), _P(_i64), _P(_i64)]),
    "tq_selftest_trit_decode": (_i32, [_u32, _u32, _c_p, _c_p]),
}

_lib = None


def load(path: str | None = None):
    """Load libtq.so (raises if it is missing) and declare every entry point."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libtq.so not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class TQError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != TQ_OK:
        raise TQError(f"{what}: {load().tq_status_string(status).decode()} ({status})")


# ---------------------------------------------------------------- torch marshalling

def _torch():
    import torch

    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream():
    return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _dt(t) -> int:
    torch = _torch()
    return {torch.float32: TQ_F32, torch.bfloat16: TQ_BF16, torch.float16: TQ_F16}[t.dtype]


def _torch_dtype(code: int):
    torch = _torch()
    return {TQ_F32: torch.float32, TQ_BF16: torch.bfloat16, TQ_F16: torch.float16}[code]


def _contig(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


# ---------------------------------------------------------------- host helpers

def codes_per_word(levels: int) -> int:
    return int(load().tq_codes_per_word(levels))


def row_words(levels: int, cols: int) -> int:
    return int(load().tq_row_words(levels, cols))


def row_stride_words(levels: int, cols: int) -> int:
    return int(load().tq_row_stride_words(levels, cols))


def codebook(levels: int):
    """Host fp64 Gaussian Lloyd-Max book: (centroids[levels], thresholds[levels-1]) numpy arrays."""
    c = np.zeros(levels, dtype=np.float64)
    t = np.zeros(max(levels - 1, 1), dtype=np.float64)
    _check(load().tq_codebook(levels, c.ctypes.data_as(_P(ctypes.c_double)), t.ctypes.data_as(_P(ctypes.c_double))),
           "tq_codebook")
    return c, t[:levels - 1]


def rotation_signs(seed: int, dim: int) -> np.ndarray:
    s = np.zeros(dim, dtype=np.int8)
    _check(load().tq_rotation_signs(ctypes.c_uint64(seed), dim, s.ctypes.data_as(_P(ctypes.c_int8))),
           "tq_rotation_signs")
    return s


def rotation_dense(seed: int, dim: int) -> np.ndarray:
    """Host fp64 dense rotation [dim, dim] of the QR fallback (see include/tq.h, tq_rotation_dense)."""
    R = np.zeros((dim, dim), dtype=np.float64)
    _check(load().tq_rotation_dense(ctypes.c_uint64(seed), dim, R.ctypes.data_as(_P(ctypes.c_double))),
           "tq_rotation_dense")
    return R


# ---------------------------------------------------------------- device descriptors

class Codebook:
    """A codebook on the device: fp32 centroids and thresholds."""

    def __init__(self, levels: int, device="cuda", centroids=None, thresholds=None):
        torch = _torch()
        if centroids is None:
            centroids, thresholds = codebook(levels)
        self.levels = int(levels)
        self.centroids = torch.tensor(np.asarray(centroids, np.float32), device=device)
        self.thresholds = torch.tensor(np.asarray(thresholds, np.float32).reshape(-1), device=device)
        if self.thresholds.numel() == 0:
            self.thresholds = torch.zeros(1, dtype=torch.float32, device=device)

    def c(self) -> tq_codebook_t:
        return tq_codebook_t(self.levels, self.centroids.data_ptr(), self.thresholds.data_ptr())


class Rotation:
    """R = blockdiag(H_block) diag(signs) / sqrt(block) over vectors of length dim."""

    def __init__(self, dim: int, block: int, seed: int | None = None, signs=None, device="cuda"):
        torch = _torch()
        if signs is None:
            signs = rotation_signs(seed, dim)
        self.dim, self.block = int(dim), int(block)
        self.signs = torch.tensor(np.asarray(signs, np.int8), device=device)

    def c(self) -> tq_rotation_t:
        return tq_rotation_t(self.dim, self.block, self.signs.data_ptr())


class DenseRotation:
    """The QR-fallback rotation of a dimension on the device (fp32 [dim, dim]), from its seed or given."""

    def __init__(self, dim: int, seed: int | None = None, R=None, device="cuda"):
        torch = _torch()
        if R is None:
            R = rotation_dense(seed, dim)
        self.dim = int(dim)
        self.R = torch.tensor(np.asarray(R, np.float32), device=device)

    def identity(self, device="cuda") -> "Rotation":
        """The identity rotation of this dim (block 1, signs +1): what tq_quantize takes after rotate_dense."""
        return Rotation(self.dim, 1, signs=np.ones(self.dim, np.int8), device=device)


class QWeight:
    """A bank of quantized matrices [experts, rows, cols] as written by ``quantize``."""

    def __init__(self, codes, scales, experts: int, rows: int, cols: int, group: int, cb: Codebook,
                 row_stride: int | None = None):
        self.codes, self.scales, self.cb = codes, scales, cb
        self.experts, self.rows, self.cols, self.group = int(experts), int(rows), int(cols), int(group)
        self.row_stride = int(row_stride if row_stride is not None else row_stride_words(cb.levels, cols))

    def c(self) -> tq_qweight_t:
        esw = self.rows * self.row_stride
        ess = self.rows * (self.cols // self.group)
        return tq_qweight_t(self.codes.data_ptr(), self.scales.data_ptr(), self.experts, self.rows, self.cols,
                            self.group, self.row_stride, esw, ess, self.cb.c())


# ---------------------------------------------------------------- device entry points

def rotate(x, rot: Rotation, out_dtype=None):
    torch = _torch()
    _contig(x, "x")
    out = torch.empty(x.shape, dtype=out_dtype or torch.float32, device=x.device)
    r = rot.c()
    _check(load().tq_rotate(ctypes.byref(r), _ptr(x), _dt(x), x.numel() // rot.dim, _ptr(out), _dt(out), _stream()),
           "tq_rotate")
    return out


def rotate_dense(x, rot: DenseRotation, precise: bool = False):
    """R x for every row of x (f32 out); precise accumulates in fp64."""
    torch = _torch()
    _contig(x, "x")
    out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _check(load().tq_rotate_dense(_ptr(rot.R), rot.dim, _ptr(x), _dt(x), x.numel() // rot.dim, _ptr(out),
                                  int(precise), _stream()), "tq_rotate_dense")
    return out


def quantize_dense(W, group: int, rot: DenseRotation, cb: Codebook, row_stride: int | None = None):
    """Encode rows of W with the dense rotation: rotate (fp64 sums), then group RMS, snap and pack."""
    return quantize(rotate_dense(W, rot, precise=True), group, rot.identity(device=W.device), cb, row_stride)


def quantize(W, group: int, rot: Rotation, cb: Codebook, row_stride: int | None = None):
    """Encode rows of W [rows, cols] -> (codes uint32 [rows, stride] as int32 storage, scales fp16 bits)."""
    torch = _torch()
    _contig(W, "W")
    rows, cols = W.shape
    stride = row_stride if row_stride is not None else row_stride_words(cb.levels, cols)
    codes = torch.empty((rows, stride), dtype=torch.int32, device=W.device)
    scales = torch.empty((rows, cols // group), dtype=torch.int16, device=W.device)
    r, b = rot.c(), cb.c()
    _check(load().tq_quantize(_ptr(W), _dt(W), rows, cols, group, ctypes.byref(r), ctypes.byref(b), _ptr(codes),
                              _ptr(scales), stride, _stream()), "tq_quantize")
    return codes, scales


def qmv(w: QWeight, x_rot, out_dtype=None, tensor_cores=True):
    """y = W x_rot for every row of x_rot.  With tensor_cores, an f32 output and two or more
    rows, the tq_qmv_tc form runs where it applies (fp16 operands, fp32 sums; at one row the
    CUDA-core kernel is as fast); elsewhere tq_qmv."""
    torch = _torch()
    _contig(x_rot, "x_rot")
    T = x_rot.shape[0]
    y = torch.empty((T, w.rows), dtype=out_dtype or torch.float32, device=x_rot.device)
    q = w.c()
    if tensor_cores and y.dtype == torch.float32 and T >= 2:
        nb = int(load().tq_qmv_tc_workspace_bytes(T, w.cols))
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=x_rot.device)
        st = load().tq_qmv_tc(ctypes.byref(q), _ptr(x_rot), T, _ptr(y), _ptr(ws), nb, None, _stream())
        if st != TQ_ERR_UNSUPPORTED:
            _check(st, "tq_qmv_tc")
            return y
    _check(load().tq_qmv(ctypes.byref(q), _ptr(x_rot), T, _ptr(y), _dt(y), _stream()), "tq_qmv")
    return y


def qmv_tc(w: QWeight, x_rot, err=None):
    """The tensor-core dense matvec alone (raises TQError where it does not apply)."""
    torch = _torch()
    _contig(x_rot, "x_rot")
    T = x_rot.shape[0]
    y = torch.empty((T, w.rows), dtype=torch.float32, device=x_rot.device)
    nb = int(load().tq_qmv_tc_workspace_bytes(T, w.cols))
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=x_rot.device)
    q = w.c()
    _check(load().tq_qmv_tc(ctypes.byref(q), _ptr(x_rot), T, _ptr(y), _ptr(ws), nb, _ptr(err), _stream()),
           "tq_qmv_tc")
    return y


def _workspace(nbytes: int, device, ws=None):
    """A caller's scratch buffer if it is large enough, else a new one (None when nothing is needed)."""
    if nbytes <= 0:
        return None
    if ws is not None and ws.numel() * ws.element_size() >= nbytes:
        return ws
    return _torch().empty(nbytes, dtype=_torch().uint8, device=device)


def gather_qmv(w: QWeight, x_rot, ids, out_dtype=None, err=None, ws=None, use_ws=True):
    """y[t, j] = W_{ids[t, j]} x_rot[t].  use_ws=False passes no scratch (the single-pass kernel
    then takes rows the table-lookup kernel would split)."""
    torch = _torch()
    _contig(x_rot, "x_rot")
    _contig(ids, "ids")
    T, k = ids.shape
    y = torch.empty((T, k, w.rows), dtype=out_dtype or torch.float32, device=x_rot.device)
    q = w.c()
    nb = int(load().tq_gather_qmv_workspace_bytes(ctypes.byref(q), T, k)) if use_ws else 0
    ws = _workspace(nb, x_rot.device, ws)
    _check(load().tq_gather_qmv(ctypes.byref(q), _ptr(x_rot), _ptr(ids), T, k, _ptr(y), _dt(y), _ptr(ws), nb,
                                _ptr(err), _stream()), "tq_gather_qmv")
    return y


def multi_gather_qmv(w: QWeight, x_rot, ids, out_dtype=None, err=None, ws=None, use_ws=True):
    """y[p] = W_{ids[p]} x_rot[p] (use_ws as for gather_qmv)."""
    torch = _torch()
    _contig(x_rot, "x_rot")
    _contig(ids, "ids")
    P = ids.shape[0]
    y = torch.empty((P, w.rows), dtype=out_dtype or torch.float32, device=x_rot.device)
    q = w.c()
    nb = int(load().tq_multi_gather_qmv_workspace_bytes(ctypes.byref(q), P)) if use_ws else 0
    ws = _workspace(nb, x_rot.device, ws)
    _check(load().tq_multi_gather_qmv(ctypes.byref(q), _ptr(x_rot), _ptr(ids), P, _ptr(y), _dt(y), _ptr(ws), nb,
                                      _ptr(err), _stream()), "tq_multi_gather_qmv")
    return y


def gather_qmv_rotate(w: QWeight, x, rot: Rotation, ids, out_dtype=None, err=None):
    """gather_qmv of R x with the rotation done inside the matvec (x: f32 or bf16 [T, cols])."""
    torch = _torch()
    _contig(x, "x")
    _contig(ids, "ids")
    T, k = ids.shape
    y = torch.empty((T, k, w.rows), dtype=out_dtype or torch.float32, device=x.device)
    q, r = w.c(), rot.c()
    _check(load().tq_gather_qmv_rotate(ctypes.byref(q), _ptr(x), _dt(x), ctypes.byref(r), _ptr(ids), T, k, _ptr(y),
                                       _dt(y), _ptr(err), _stream()), "tq_gather_qmv_rotate")
    return y


def multi_gather_qmv_swiglu(w: QWeight, gate_up, rot: Rotation, ids, out_dtype=None, err=None):
    """multi_gather_qmv of R (silu(gate) * up) per pair, SwiGLU and rotation inside (gate_up: f32 [P, 2*cols])."""
    torch = _torch()
    _contig(gate_up, "gate_up")
    _contig(ids, "ids")
    P = ids.shape[0]
    y = torch.empty((P, w.rows), dtype=out_dtype or torch.float32, device=gate_up.device)
    q, r = w.c(), rot.c()
    _check(load().tq_multi_gather_qmv_swiglu(ctypes.byref(q), _ptr(gate_up), ctypes.byref(r), _ptr(ids), P, _ptr(y),
                                             _dt(y), _ptr(err), _stream()), "tq_multi_gather_qmv_swiglu")
    return y


def moe_route(logits, k: int, sort: bool = True):
    """-> ids [T,k] int32, probs [T,k] f32, perm [T*k], pair_pos [T*k], offsets [E+1].

    With sort=False only ids and probs are computed (the other three are None).
    """
    torch = _torch()
    _contig(logits, "logits")
    T, E = logits.shape
    dev = logits.device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    probs = torch.empty((T, k), dtype=torch.float32, device=dev)
    if not sort:
        _check(load().tq_moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(probs), None, None, None, None, 0,
                                   _stream()), "tq_moe_route")
        return ids, probs, None, None, None
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    nb = int(load().tq_route_workspace_bytes(E))
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    _check(load().tq_moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(probs), _ptr(perm), _ptr(pos), _ptr(off),
                               _ptr(ws), nb, _stream()), "tq_moe_route")
    return ids, probs, perm, pos, off


def swiglu_rotate(gate_up, inter: int, rot: Rotation, out_dtype=None):
    torch = _torch()
    _contig(gate_up, "gate_up")
    P = gate_up.numel() // (2 * inter)
    out = torch.empty((P, inter), dtype=out_dtype or torch.float32, device=gate_up.device)
    r = rot.c()
    _check(load().tq_swiglu_rotate(_ptr(gate_up), P, inter, ctypes.byref(r), _ptr(out), _dt(out), _stream()),
           "tq_swiglu_rotate")
    return out


def moe_combine(y, probs, k: int, pair_pos=None, out_dtype=None):
    torch = _torch()
    _contig(y, "y")
    H = y.shape[-1]
    T = probs.numel() // k
    out = torch.empty((T, H), dtype=out_dtype or torch.float32, device=y.device)
    _check(load().tq_moe_combine(_ptr(y), _ptr(probs), _ptr(pair_pos), T, k, H, _ptr(out), _dt(out), _stream()),
           "tq_moe_combine")
    return out


def gather_qmm(w: QWeight, x, perm, offsets, k: int, per_pair_input: bool = False, out_dtype=None, err=None):
    torch = _torch()
    _contig(x, "x")
    P = int(perm.numel()) if not per_pair_input else int(x.shape[0])
    y = torch.empty((P, w.rows), dtype=out_dtype or torch.float32, device=x.device)
    nb = int(load().tq_gather_qmm_workspace_bytes(P, w.cols, int(per_pair_input)))
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=x.device)
    q = w.c()
    _check(load().tq_gather_qmm(ctypes.byref(q), _ptr(x), _dt(x), _ptr(perm), _ptr(offsets), P, k,
                                int(per_pair_input), _ptr(y), _dt(y), _ptr(ws), nb, _ptr(err), _stream()),
           "tq_gather_qmm")
    return y


def dequant_experts(w: QWeight, ids, out_dtype=None, err=None):
    torch = _torch()
    _contig(ids, "ids")
    n = ids.numel()
    out = torch.empty((n, w.rows, w.cols), dtype=out_dtype or torch.float32, device=ids.device)
    q = w.c()
    _check(load().tq_dequant_experts(ctypes.byref(q), _ptr(ids), n, _ptr(out), _dt(out), _ptr(err), _stream()),
           "tq_dequant_experts")
    return out


class KVCache:
    """Compressed KV cache: codes and fp16 scales per (kv head, position)."""

    def __init__(self, capacity: int, heads: int, dim: int, group: int, kcb: Codebook, vcb: Codebook,
                 rot: Rotation, device="cuda"):
        torch = _torch()
        self.capacity, self.heads, self.dim, self.group = capacity, heads, dim, group
        self.kcb, self.vcb, self.rot = kcb, vcb, rot
        self.kw, self.vw = row_words(kcb.levels, dim), row_words(vcb.levels, dim)
        self.kcodes = torch.zeros((heads, capacity, self.kw), dtype=torch.int32, device=device)
        self.vcodes = torch.zeros((heads, capacity, self.vw), dtype=torch.int32, device=device)
        self.kscales = torch.zeros((heads, capacity, dim // group), dtype=torch.int16, device=device)
        self.vscales = torch.zeros((heads, capacity, dim // group), dtype=torch.int16, device=device)
        self.length = 0


def kv_quantize(cache: KVCache, k, v, pos: int | None = None):
    _contig(k, "k")
    _contig(v, "v")
    T = k.shape[0]
    pos = cache.length if pos is None else pos
    r, kb, vb = cache.rot.c(), cache.kcb.c(), cache.vcb.c()
    _check(load().tq_kv_quantize(_ptr(k), _ptr(v), _dt(k), T, cache.heads, cache.dim, pos, cache.capacity,
                                 ctypes.byref(r), ctypes.byref(kb), ctypes.byref(vb), cache.group, _ptr(cache.kcodes),
                                 _ptr(cache.kscales), _ptr(cache.vcodes), _ptr(cache.vscales), _stream()),
           "tq_kv_quantize")
    cache.length = max(cache.length, pos + T)


def kv_attend(cache: KVCache, q, ctx: int | None = None, ws=None):
    torch = _torch()
    _contig(q, "q")
    Hq = q.shape[0]
    ctx = cache.length if ctx is None else ctx
    o = torch.empty((Hq, cache.dim), dtype=torch.float32, device=q.device)
    nb = int(load().tq_kv_attend_workspace_bytes(Hq, cache.dim, ctx))
    if ws is None:
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=q.device)
    r, kb, vb = cache.rot.c(), cache.kcb.c(), cache.vcb.c()
    _check(load().tq_kv_attend(_ptr(q), _dt(q), Hq, cache.heads, cache.dim, ctx, cache.capacity, ctypes.byref(r),
                               ctypes.byref(kb), ctypes.byref(vb), cache.group, _ptr(cache.kcodes),
                               _ptr(cache.kscales), _ptr(cache.vcodes), _ptr(cache.vscales), _ptr(o), _ptr(ws),
                               ws.numel(), _stream()), "tq_kv_attend")
    return o


def kv_attend_noalloc(cache: KVCache, q, ctx: int | None = None):
    """kv_attend with the library's fixed device scratch instead of a workspace (see include/tq.h)."""
    torch = _torch()
    _contig(q, "q")
    Hq = q.shape[0]
    ctx = cache.length if ctx is None else ctx
    o = torch.empty((Hq, cache.dim), dtype=torch.float32, device=q.device)
    r, kb, vb = cache.rot.c(), cache.kcb.c(), cache.vcb.c()
    _check(load().tq_kv_attend_noalloc(_ptr(q), _dt(q), Hq, cache.heads, cache.dim, ctx, cache.capacity,
                                       ctypes.byref(r), ctypes.byref(kb), ctypes.byref(vb), cache.group,
                                       _ptr(cache.kcodes), _ptr(cache.kscales), _ptr(cache.vcodes),
                                       _ptr(cache.vscales), _ptr(o), _stream()), "tq_kv_attend_noalloc")
    return o


def moe_decode_layer(gate_up: QWeight, down: QWeight, rot_h: Rotation, rot_i: Rotation, logits, x, k: int,
                     out_dtype=None, err=None, ws=None):
    """One token through the MoE layer in one launch: route, rotate, gate||up, SwiGLU + rotate, down,
    combine.  logits: f32 [E] (or [1, E]); x: [H] (or [1, H]) f32/bf16/f16.  Returns out [1, H]."""
    torch = _torch()
    _contig(logits, "logits")
    _contig(x, "x")
    H = gate_up.cols
    out = torch.empty((1, H), dtype=out_dtype or torch.float32, device=x.device)
    g, d, rh, ri = gate_up.c(), down.c(), rot_h.c(), rot_i.c()
    nb = int(load().tq_moe_decode_layer_workspace_bytes(ctypes.byref(g), ctypes.byref(d), k))
    ws = _workspace(nb, x.device, ws)
    _check(load().tq_moe_decode_layer(ctypes.byref(g), ctypes.byref(d), ctypes.byref(rh), ctypes.byref(ri),
                                      _ptr(logits), _ptr(x), _dt(x), k, _ptr(out), _dt(out), _ptr(ws), nb, _ptr(err),
                                      _stream()), "tq_moe_decode_layer")
    return out


def check_error(err) -> int:
    """Synchronises, returns the device error bits and clears them."""
    bits = _u32(0)
    st = load().tq_check_error(_ptr(err), ctypes.byref(bits), _stream())
    if st not in (TQ_OK, TQ_ERR_TIMEOUT, TQ_ERR_DEVICE):
        _check(st, "tq_check_error")
    return int(bits.value)


def set_wait_budget(cycles: int) -> None:
    """Test hook: cycle budget of the tensor-core kernels' bounded waits (-1: the default)."""
    _check(load().tq_set_wait_budget(int(cycles)), "tq_set_wait_budget")


def selftest_trit_decode(first: int = 0, count: int = 3 ** 20) -> int:
    torch = _torch()
    m = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(load().tq_selftest_trit_decode(first, count, _ptr(m), _stream()), "tq_selftest_trit_decode")
    return int(m.item())


# ---------------------------------------------------------------- per-layer tiers and the packed file

# "How it works": ternary experts, 4-bit down projections, 3-bit protected layers; group 16 for
# MLP and expert layers.
DEFAULT_TIERS = {"down": (16, 16), "expert": (3, 16), "mlp": (8, 16), "attn": (8, 64), "other": (8, 64)}


def tier_policy(tiers: dict | None = None) -> tq_tier_policy_t:
    t = dict(DEFAULT_TIERS, **(tiers or {}))
    return tq_tier_policy_t(t["down"][0], t["down"][1], t["expert"][0], t["expert"][1], t["mlp"][0], t["mlp"][1],
                            t["attn"][0], t["attn"][1], t["other"][0], t["other"][1])


def layer_tier(name: str, policy: tq_tier_policy_t | None = None) -> tuple[int, int]:
    """(codebook size, group) of layer `name` under the tier policy."""
    lv, g = _i32(0), _i32(0)
    pol = policy if policy is not None else tier_policy()
    _check(load().tq_layer_tier(name.encode(), ctypes.byref(pol), ctypes.byref(lv), ctypes.byref(g)), "tq_layer_tier")
    return int(lv.value), int(g.value)


class PackedLayer:
    """A layer as stored in a packed file: host numpy arrays and their metadata."""

    def __init__(self, name, codes, scales, centroids, group, rot_block, rot_seed):
        self.name = name
        self.codes = np.ascontiguousarray(codes, dtype=np.uint32)        # [experts, rows, row_stride]
        self.scales = np.ascontiguousarray(scales).view(np.uint16)        # [experts, rows, cols/group]
        self.centroids = np.ascontiguousarray(centroids, dtype=np.float64)
        self.experts, self.rows, self.row_stride = self.codes.shape
        self.group = int(group)
        self.cols = self.scales.shape[-1] * self.group
        self.rot_block, self.rot_seed = int(rot_block), int(rot_seed)

    @property
    def levels(self) -> int:
        return len(self.centroids)

    def qweight(self, device="cuda") -> "QWeight":
        """The layer on the device (its codebook's thresholds are the midpoints of the centroids)."""
        torch = _torch()
        c = self.centroids
        cb = Codebook(self.levels, device=device, centroids=c, thresholds=(c[1:] + c[:-1]) / 2)
        codes = torch.from_numpy(self.codes.view(np.int32)).to(device)
        scales = torch.from_numpy(self.scales.view(np.int16)).to(device)
        return QWeight(codes, scales, self.experts, self.rows, self.cols, self.group, cb, row_stride=self.row_stride)


def save_packed(path: str, layers: list[PackedLayer]) -> None:
    descs = (tq_layer_desc_t * max(len(layers), 1))()
    for d, L in zip(descs, layers):
        d.name = L.name.encode()
        d.experts, d.rows, d.cols, d.group = L.experts, L.rows, L.cols, L.group
        d.row_stride_words, d.levels = L.row_stride, L.levels
        d.rot_dim, d.rot_block, d.rot_seed = L.cols, L.rot_block, L.rot_seed
        d.centroids = L.centroids.ctypes.data
        d.codes = L.codes.ctypes.data
        d.scales = L.scales.ctypes.data
    _check(load().tq_pack_file_write(path.encode(), descs, len(layers)), "tq_pack_file_write")


def load_packed(path: str) -> list[PackedLayer]:
    lib = load()
    n = _i32(0)
    _check(lib.tq_pack_file_info(path.encode(), ctypes.byref(n), None, 0), "tq_pack_file_info")
    infos = (tq_layer_desc_t * max(n.value, 1))()
    _check(lib.tq_pack_file_info(path.encode(), ctypes.byref(n), infos, n.value), "tq_pack_file_info")
    out = []
    for i in range(n.value):
        d = infos[i]
        c = np.zeros(d.levels, np.float64)
        codes = np.zeros((d.experts, d.rows, d.row_stride_words), np.uint32)
        scales = np.zeros((d.experts, d.rows, d.cols // d.group), np.uint16)
        _check(lib.tq_pack_file_read_layer(path.encode(), i, c.ctypes.data, codes.ctypes.data, scales.ctypes.data),
               "tq_pack_file_read_layer")
        out.append(PackedLayer(d.name.decode(), codes, scales, c, d.group, d.rot_block, d.rot_seed))
    return out


# ---------------------------------------------------------------- expert streaming

class ExpertCache:
    """Experts of a bank held in host memory, streamed into ``slots`` device slots (LRU).

    ``codes`` (int32/uint32 [experts, rows, row_stride]) and ``scales`` (16-bit
    [experts, rows, cols/group]) are host arrays: pinned torch CPU tensors for
    ``map`` (the copies are asynchronous), or numpy arrays for ``plan`` alone.
    ``view`` is the slot bank on the device, a QWeight with ``slots`` experts
    that the gather entry points run on with ids remapped to slots.
    """

    def __init__(self, codes, scales, experts: int, rows: int, cols: int, group: int, cb: Codebook, slots: int,
                 row_stride: int | None = None, device="cuda"):
        self.host_codes, self.host_scales = codes, scales
        self.row_stride = int(row_stride if row_stride is not None else row_stride_words(cb.levels, cols))
        self.experts, self.rows, self.cols, self.group, self.slots = experts, rows, cols, group, int(slots)
        self.cb = cb
        cp = codes.data_ptr() if hasattr(codes, "data_ptr") else codes.ctypes.data
        sp = scales.data_ptr() if hasattr(scales, "data_ptr") else scales.ctypes.data
        host = tq_qweight_t(cp, sp, experts, rows, cols, group, self.row_stride, rows * self.row_stride,
                            rows * (cols // group), cb.c())
        self.view = None
        dc = ds = None
        if device is not None:
            torch = _torch()
            dcodes = torch.empty((self.slots, rows, self.row_stride), dtype=torch.int32, device=device)
            dscales = torch.empty((self.slots, rows, cols // group), dtype=torch.int16, device=device)
            self.view = QWeight(dcodes, dscales, self.slots, rows, cols, group, cb, row_stride=self.row_stride)
            dc, ds = dcodes.data_ptr(), dscales.data_ptr()
        h = _c_p()
        _check(load().tq_expert_cache_create(ctypes.byref(host), self.slots, dc, ds, ctypes.byref(h)),
               "tq_expert_cache_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.tq_expert_cache_destroy(h)
            self._h = None

    @staticmethod
    def _ids(ids) -> np.ndarray:
        if hasattr(ids, "detach"):
            ids = ids.detach().to("cpu").numpy()
        return np.ascontiguousarray(np.asarray(ids).reshape(-1), dtype=np.int32)

    def plan(self, ids):
        """LRU bookkeeping only (host): (slot of each id, 1 where the id is a first miss)."""
        a = self._ids(ids)
        slots = np.zeros(a.size, np.int32)
        miss = np.zeros(a.size, np.uint8)
        _check(load().tq_expert_cache_plan(self._h, a.ctypes.data, a.size, slots.ctypes.data, miss.ctypes.data),
               "tq_expert_cache_plan")
        return slots, miss

    def map(self, ids):
        """Brings the experts of ``ids`` into the slots on the current stream; their slots (host int32)."""
        a = self._ids(ids)
        slots = np.zeros(a.size, np.int32)
        _check(load().tq_expert_cache_map(self._h, a.ctypes.data, a.size, slots.ctypes.data, _stream()),
               "tq_expert_cache_map")
        return slots

    def stats(self) -> tuple[int, int, int]:
        """(hits, misses, bytes copied) since creation."""
        h, m, b = _i64(0), _i64(0), _i64(0)
        _check(load().tq_expert_cache_stats(self._h, ctypes.byref(h), ctypes.byref(m), ctypes.byref(b)),
               "tq_expert_cache_stats")
        return int(h.value), int(m.value), int(b.value)

    def gather_qmv(self, x_rot, ids, out_dtype=None, err=None):
        """gather_qmv of the host bank: maps ``ids`` [T, k], then gathers from the slots."""
        torch = _torch()
        shape = tuple(ids.shape)
        slots = torch.from_numpy(self.map(ids)).reshape(shape).pin_memory().to(x_rot.device, non_blocking=True)
        return gather_qmv(self.view, x_rot, slots, out_dtype=out_dtype, err=err)
