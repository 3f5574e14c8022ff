"""Thin Python binding over the C ABI in ``include/samu.h``.

Argument marshalling only: tensors are checked for dtype, device and
contiguity, their ``data_ptr()`` and the current CUDA stream are handed to the
shared library, and every step of the computation runs in its CUDA kernels.
There is no fallback: if ``liblrs_gb300.so`` is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "liblrs_gb300.so"
_lock = threading.Lock()
_lib = None

LRS_GRAD_BF16 = 0
LRS_GRAD_FP32 = 1
LRS_TRANSITION_CHAINED = 0
LRS_TRANSITION_CLOSED_FORM = 1

# names and argument kinds of every exported symbol (checked by the tests)
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZP = ctypes.POINTER(ctypes.c_size_t)
_SIGNATURES = {
    "lrs_status_string": ([_I], ctypes.c_char_p),
    "samu_status_string": ([_I], ctypes.c_char_p),
    "lrs_version": ([], _I),
    "lrs_device_status": ([_P, ctypes.POINTER(_I), _P], _I),
    "lrs_selftest_wait_timeout": ([_P, _P], _I),
    "lrs_profile_begin": ([_I], _I),
    "lrs_profile_end": ([_P, _P, _I, ctypes.POINTER(_I)], _I),
    "samu_set_chunk_transition": ([_I], _I),
    "samu_get_chunk_transition": ([], _I),
    "samu_workspace_bytes": ([_I, _I, _I, _SZP, _SZP], _I),
    "samu_forward": ([_P] * 10 + [_I, _I, _I] + [_P] * 6, _I),
    "samu_backward": ([_P] * 12 + [_I, _I, _I] + [_P, _P, _P, _I] + [_P] * 9, _I),
    "samu_forward_noalloc": ([_P] * 10 + [_I, _I, _I] + [_P] * 4, _I),
    "samu_forward_noalloc_status": ([ctypes.POINTER(_I), _P], _I),
    "samu_decode_params_floats": ([_I, _SZP], _I),
    "samu_decode_prepare": ([_P] * 6 + [_I, _P, _P], _I),
    "samu_decode_step": ([_P] * 6 + [_I, _I, _P, _P, _P], _I),
    "rglru_workspace_bytes": ([_I, _I, _I, _SZP, _SZP], _I),
    "rglru_forward": ([_P] * 6 + [_I, _I, _I] + [_P] * 6, _I),
    "rglru_backward": ([_P] * 8 + [_I, _I, _I] + [_P] * 4 + [_I] + [_P] * 4, _I),
    "rglru_proj_workspace_bytes": ([_I, _I, _I, _SZP, _SZP], _I),
    "rglru_proj_forward": ([_P] * 8 + [_I, _I, _I] + [_P] * 6, _I),
    "rglru_proj_backward": ([_P] * 10 + [_I, _I, _I] + [_P] * 2 + [_I] + [_P] * 8, _I),
    "samu_block_workspace_bytes": ([_I] * 4 + [_SZP, _SZP], _I),
    "samu_block_forward": ([_P] * 4 + [_I] * 4 + [_P] * 5, _I),
    "samu_block_backward": ([_P] * 6 + [_I] * 4 + [_P] * 6, _I),
    "lrs_dense_gemm": ([_I, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "rglru_block_workspace_bytes": ([_I] * 4 + [_SZP, _SZP], _I),
    "rglru_block_forward": ([_P] * 4 + [_I] * 4 + [_P] * 5, _I),
    "rglru_block_backward": ([_P] * 6 + [_I] * 4 + [_P] * 6, _I),
}

# samu_block_params / samu_block_grads (include/samu.h): one pointer per field, in order
BLOCK_PARAMS = ("gamma1", "w_in", "conv_k", "conv_b", "nu", "theta", "w_phi", "w_r", "a_phi", "a_r",
                "w_o", "gamma2", "w_mlp_in", "w_mlp_out")


class _BlockParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in BLOCK_PARAMS]


class _BlockGrads(ctypes.Structure):
    _fields_ = [("d" + n, ctypes.c_void_p) for n in BLOCK_PARAMS]


# rglru_block_params / rglru_block_grads: the block around the RG-LRU mixer
RGLRU_BLOCK_PARAMS = ("gamma1", "w_in", "conv_k", "conv_b", "w_x", "b_x", "w_a", "b_a", "alpha",
                      "w_o", "gamma2", "w_mlp_in", "w_mlp_out")


class _RgBlockParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in RGLRU_BLOCK_PARAMS]


class _RgBlockGrads(ctypes.Structure):
    _fields_ = [("d" + n, ctypes.c_void_p) for n in RGLRU_BLOCK_PARAMS]


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{_LIB_NAME} is not built ({path}); run __graft_entry__.build() first")
            lib = ctypes.CDLL(path)
            for name, (argtypes, restype) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = lib
    return _lib


class LrsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _load().lrs_status_string(status).decode()
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def _check(fn: str, status: int):
    if status != 0:
        raise LrsError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, device, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _opt(t, name, dtype, device, shape=None):
    return None if t is None else _need(t, name, dtype, device, shape)


def _empty(shape, dtype, device, out, key):
    if out is not None and key in out and out[key] is not None:
        return _need(out[key], key, dtype, device, shape)
    return torch.empty(shape, dtype=dtype, device=device)


# ---------------------------------------------------------------------------
# SAMU
# ---------------------------------------------------------------------------
def samu_workspace_bytes(B: int, L: int, D: int):
    lib = _load()
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    _check("samu_workspace_bytes", lib.samu_workspace_bytes(B, L, D, ctypes.byref(s), ctypes.byref(c)))
    return int(s.value), int(c.value)


def samu_forward(x_sel, w, h0, reset, nu, theta, w_phi, w_r, a_phi, a_r, *, want_y32=False,
                 out=None, saved=None, scratch=None):
    """SAMU mixer forward through ``samu_forward``.  Returns dict(y, y32, hT, saved, scratch)."""
    dev = x_sel.device
    B, L, D = x_sel.shape
    M = D // 2
    _need(x_sel, "x_sel", torch.bfloat16, dev)
    _need(w, "w", torch.bfloat16, dev, (B, L, D))
    _opt(h0, "h0", torch.float32, dev, (B, M, 2))
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    _need(nu, "nu", torch.float32, dev, (M,))
    _need(theta, "theta", torch.float32, dev, (M,))
    _need(w_phi, "w_phi", torch.float32, dev, (D + 1,))
    _need(w_r, "w_r", torch.float32, dev, (D + 1,))
    _need(a_phi, "a_phi", torch.float32, dev, (1,))
    _need(a_r, "a_r", torch.float32, dev, (1,))
    nsaved, nscratch = samu_workspace_bytes(B, L, D)
    y = _empty((B, L, D), torch.bfloat16, dev, out, "y")
    y32 = _empty((B, L, D), torch.float32, dev, out, "y32") if want_y32 else None
    hT = _empty((B, M, 2), torch.float32, dev, out, "hT")
    if saved is None:
        saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    if saved.numel() < nsaved or scratch.numel() < nscratch:
        raise ValueError("saved/scratch buffers are too small")
    st = _load().samu_forward(_ptr(x_sel), _ptr(w), _ptr(h0), _ptr(reset), _ptr(nu), _ptr(theta),
                              _ptr(w_phi), _ptr(w_r), _ptr(a_phi), _ptr(a_r), B, L, D,
                              _ptr(y), _ptr(y32), _ptr(hT), _ptr(saved), _ptr(scratch), _stream(dev))
    _check("samu_forward", st)
    return {"y": y, "y32": y32, "hT": hT, "saved": saved, "scratch": scratch}


def samu_backward(dy, dhT, x_sel, w, h0, reset, nu, theta, w_phi, w_r, a_phi, a_r, saved, *,
                  grad_fp32=False, out=None, scratch=None):
    """SAMU mixer backward through ``samu_backward``.

    Returns dict(dx_sel, dw, dh0, dnu, dtheta, dw_phi, dw_r, da_phi, da_r, scratch).
    """
    dev = x_sel.device
    B, L, D = x_sel.shape
    M = D // 2
    _need(dy, "dy", torch.bfloat16, dev, (B, L, D))
    _opt(dhT, "dhT", torch.float32, dev, (B, M, 2))
    _need(x_sel, "x_sel", torch.bfloat16, dev)
    _need(w, "w", torch.bfloat16, dev, (B, L, D))
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    nsaved, nscratch = samu_workspace_bytes(B, L, D)
    if saved is None or saved.numel() < nsaved:
        raise ValueError("saved must be the forward's saved buffer")
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    gdt = torch.float32 if grad_fp32 else torch.bfloat16
    o = {
        "dx_sel": _empty((B, L, D), gdt, dev, out, "dx_sel"),
        "dw": _empty((B, L, D), gdt, dev, out, "dw"),
        "dh0": _empty((B, M, 2), torch.float32, dev, out, "dh0"),
        "dnu": _empty((M,), torch.float32, dev, out, "dnu"),
        "dtheta": _empty((M,), torch.float32, dev, out, "dtheta"),
        "dw_phi": _empty((D + 1,), torch.float32, dev, out, "dw_phi"),
        "dw_r": _empty((D + 1,), torch.float32, dev, out, "dw_r"),
        "da_phi": _empty((1,), torch.float32, dev, out, "da_phi"),
        "da_r": _empty((1,), torch.float32, dev, out, "da_r"),
    }
    st = _load().samu_backward(_ptr(dy), _ptr(dhT), _ptr(x_sel), _ptr(w), _ptr(h0), _ptr(reset), _ptr(nu),
                               _ptr(theta), _ptr(w_phi), _ptr(w_r), _ptr(a_phi), _ptr(a_r), B, L, D,
                               _ptr(saved), _ptr(o["dx_sel"]), _ptr(o["dw"]),
                               LRS_GRAD_FP32 if grad_fp32 else LRS_GRAD_BF16,
                               _ptr(o["dh0"]), _ptr(o["dnu"]), _ptr(o["dtheta"]), _ptr(o["dw_phi"]),
                               _ptr(o["dw_r"]), _ptr(o["da_phi"]), _ptr(o["da_r"]), _ptr(scratch), _stream(dev))
    _check("samu_backward", st)
    o["scratch"] = scratch
    return o


def samu_forward_noalloc(x_sel, w, h0, reset, nu, theta, w_phi, w_r, a_phi, a_r, *, want_y32=False,
                         out=None):
    """SAMU forward through ``samu_forward_noalloc``: for callers that cannot
    allocate device memory for the workspace, the library keeps its
    intermediates in one fixed device array (LRS_NOALLOC_BYTES, shared by all
    calls on a device; calls that overlap on the GPU race).  Outputs are still
    caller-provided (``out``) or allocated here by torch.  Returns dict(y, y32, hT)."""
    dev = x_sel.device
    B, L, D = x_sel.shape
    M = D // 2
    _need(x_sel, "x_sel", torch.bfloat16, dev)
    _need(w, "w", torch.bfloat16, dev, (B, L, D))
    _opt(h0, "h0", torch.float32, dev, (B, M, 2))
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    _need(nu, "nu", torch.float32, dev, (M,))
    _need(theta, "theta", torch.float32, dev, (M,))
    _need(w_phi, "w_phi", torch.float32, dev, (D + 1,))
    _need(w_r, "w_r", torch.float32, dev, (D + 1,))
    _need(a_phi, "a_phi", torch.float32, dev, (1,))
    _need(a_r, "a_r", torch.float32, dev, (1,))
    y = _empty((B, L, D), torch.bfloat16, dev, out, "y")
    y32 = _empty((B, L, D), torch.float32, dev, out, "y32") if want_y32 else None
    hT = _empty((B, M, 2), torch.float32, dev, out, "hT")
    st = _load().samu_forward_noalloc(_ptr(x_sel), _ptr(w), _ptr(h0), _ptr(reset), _ptr(nu), _ptr(theta),
                                      _ptr(w_phi), _ptr(w_r), _ptr(a_phi), _ptr(a_r), B, L, D,
                                      _ptr(y), _ptr(y32), _ptr(hT), _stream(dev))
    _check("samu_forward_noalloc", st)
    return {"y": y, "y32": y32, "hT": hT}


def samu_set_chunk_transition(kind: int) -> None:
    """Process-wide form of the SAMU maps kernels' item transitions
    (LRS_TRANSITION_CHAINED or LRS_TRANSITION_CLOSED_FORM) for later calls."""
    _check("samu_set_chunk_transition", _load().samu_set_chunk_transition(int(kind)))


def samu_get_chunk_transition() -> int:
    return int(_load().samu_get_chunk_transition())


# ---------------------------------------------------------------------------
# SAMU decode step
# ---------------------------------------------------------------------------
def samu_decode_params_floats(D: int) -> int:
    n = ctypes.c_size_t(0)
    _check("samu_decode_params_floats", _load().samu_decode_params_floats(D, ctypes.byref(n)))
    return int(n.value)


def samu_decode_prepare(nu, theta, w_phi, w_r, a_phi, a_r, *, params=None):
    """Per-parameter part of the decode step through ``samu_decode_prepare``.  Returns the parameter block."""
    dev = nu.device
    M = nu.shape[0]
    D = 2 * M
    _need(nu, "nu", torch.float32, dev, (M,))
    _need(theta, "theta", torch.float32, dev, (M,))
    _need(w_phi, "w_phi", torch.float32, dev, (D + 1,))
    _need(w_r, "w_r", torch.float32, dev, (D + 1,))
    _need(a_phi, "a_phi", torch.float32, dev, (1,))
    _need(a_r, "a_r", torch.float32, dev, (1,))
    n = samu_decode_params_floats(D)
    if params is None:
        params = torch.empty(n, dtype=torch.float32, device=dev)
    if params.numel() < n:
        raise ValueError("params block is too small")
    _check("samu_decode_prepare", _load().samu_decode_prepare(_ptr(nu), _ptr(theta), _ptr(w_phi), _ptr(w_r),
                                                             _ptr(a_phi), _ptr(a_r), D, _ptr(params), _stream(dev)))
    return params


def samu_decode_step(x_sel, w, state, params, reset=None, *, state_out=None, want_y32=False, out=None):
    """One token of each of B sequences through ``samu_decode_step``.  x_sel, w: [B,D] BF16; state: [B,M,2] FP32.

    state_out defaults to ``state`` (updated in place).  Returns dict(y, y32, state)."""
    dev = x_sel.device
    B, D = x_sel.shape
    M = D // 2
    _need(x_sel, "x_sel", torch.bfloat16, dev)
    _need(w, "w", torch.bfloat16, dev, (B, D))
    _need(state, "state", torch.float32, dev, (B, M, 2))
    _opt(reset, "reset", torch.uint8, dev, (B,))
    so = state if state_out is None else state_out
    _need(so, "state_out", torch.float32, dev, (B, M, 2))
    y = _empty((B, D), torch.bfloat16, dev, out, "y")
    y32 = _empty((B, D), torch.float32, dev, out, "y32") if want_y32 else None
    _check("samu_decode_step", _load().samu_decode_step(_ptr(x_sel), _ptr(w), _ptr(state), _ptr(so), _ptr(reset),
                                                       _ptr(params), B, D, _ptr(y), _ptr(y32), _stream(dev)))
    return {"y": y, "y32": y32, "state": so}


# ---------------------------------------------------------------------------
# RG-LRU
# ---------------------------------------------------------------------------
def rglru_workspace_bytes(B: int, L: int, D: int):
    lib = _load()
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    _check("rglru_workspace_bytes", lib.rglru_workspace_bytes(B, L, D, ctypes.byref(s), ctypes.byref(c)))
    return int(s.value), int(c.value)


def rglru_forward(x, lx, la, alpha, h0, reset, *, want_y32=False, out=None, saved=None, scratch=None):
    """RG-LRU forward through ``rglru_forward``.  Returns dict(y, y32, hT, saved, scratch)."""
    dev = x.device
    B, L, D = x.shape
    _need(x, "x", torch.bfloat16, dev)
    _need(lx, "lx", torch.bfloat16, dev, (B, L, D))
    _need(la, "la", torch.bfloat16, dev, (B, L, D))
    _need(alpha, "alpha", torch.float32, dev, (D,))
    _opt(h0, "h0", torch.float32, dev, (B, D))
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    nsaved, nscratch = rglru_workspace_bytes(B, L, D)
    y = _empty((B, L, D), torch.bfloat16, dev, out, "y")
    y32 = _empty((B, L, D), torch.float32, dev, out, "y32") if want_y32 else None
    hT = _empty((B, D), torch.float32, dev, out, "hT")
    if saved is None:
        saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    st = _load().rglru_forward(_ptr(x), _ptr(lx), _ptr(la), _ptr(alpha), _ptr(h0), _ptr(reset), B, L, D,
                               _ptr(y), _ptr(y32), _ptr(hT), _ptr(saved), _ptr(scratch), _stream(dev))
    _check("rglru_forward", st)
    return {"y": y, "y32": y32, "hT": hT, "saved": saved, "scratch": scratch}


def rglru_backward(dy, dhT, x, lx, la, alpha, h0, reset, saved, *, grad_fp32=False, out=None, scratch=None):
    """RG-LRU backward through ``rglru_backward``.  Returns dict(dx, dlx, dla, dalpha, dh0, scratch)."""
    dev = x.device
    B, L, D = x.shape
    _need(dy, "dy", torch.bfloat16, dev, (B, L, D))
    _opt(dhT, "dhT", torch.float32, dev, (B, D))
    nsaved, nscratch = rglru_workspace_bytes(B, L, D)
    if saved is None or saved.numel() < nsaved:
        raise ValueError("saved must be the forward's saved buffer")
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    gdt = torch.float32 if grad_fp32 else torch.bfloat16
    o = {
        "dx": _empty((B, L, D), gdt, dev, out, "dx"),
        "dlx": _empty((B, L, D), gdt, dev, out, "dlx"),
        "dla": _empty((B, L, D), gdt, dev, out, "dla"),
        "dalpha": _empty((D,), torch.float32, dev, out, "dalpha"),
        "dh0": _empty((B, D), torch.float32, dev, out, "dh0"),
    }
    st = _load().rglru_backward(_ptr(dy), _ptr(dhT), _ptr(x), _ptr(lx), _ptr(la), _ptr(alpha), _ptr(h0),
                                _ptr(reset), B, L, D, _ptr(saved), _ptr(o["dx"]), _ptr(o["dlx"]), _ptr(o["dla"]),
                                LRS_GRAD_FP32 if grad_fp32 else LRS_GRAD_BF16,
                                _ptr(o["dalpha"]), _ptr(o["dh0"]), _ptr(scratch), _stream(dev))
    _check("rglru_backward", st)
    o["scratch"] = scratch
    return o


# ---------------------------------------------------------------------------
# RG-LRU with its block-diagonal gate projections
# ---------------------------------------------------------------------------
PROJ_BLOCKS = 16


def rglru_proj_workspace_bytes(B: int, L: int, D: int):
    lib = _load()
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    _check("rglru_proj_workspace_bytes", lib.rglru_proj_workspace_bytes(B, L, D, ctypes.byref(s), ctypes.byref(c)))
    return int(s.value), int(c.value)


def _proj_params(x, w_x, b_x, w_a, b_a, alpha):
    dev = x.device
    B, L, D = x.shape
    dk = D // PROJ_BLOCKS
    _need(x, "x", torch.bfloat16, dev)
    for t, n in ((w_x, "w_x"), (w_a, "w_a")):
        _need(t, n, torch.bfloat16, dev, (PROJ_BLOCKS, dk, dk))
    for t, n in ((b_x, "b_x"), (b_a, "b_a"), (alpha, "alpha")):
        _need(t, n, torch.float32, dev, (D,))
    return dev, B, L, D, dk


def rglru_proj_forward(x, w_x, b_x, w_a, b_a, alpha, h0, reset, *, want_y32=False, out=None, saved=None,
                       scratch=None):
    """RG-LRU forward with the block-diagonal gate projections (``rglru_proj_forward``).
    Returns dict(y, y32, hT, saved, scratch)."""
    dev, B, L, D, dk = _proj_params(x, w_x, b_x, w_a, b_a, alpha)
    _opt(h0, "h0", torch.float32, dev, (B, D))
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    nsaved, nscratch = rglru_proj_workspace_bytes(B, L, D)
    y = _empty((B, L, D), torch.bfloat16, dev, out, "y")
    y32 = _empty((B, L, D), torch.float32, dev, out, "y32") if want_y32 else None
    hT = _empty((B, D), torch.float32, dev, out, "hT")
    if saved is None:
        saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    st = _load().rglru_proj_forward(_ptr(x), _ptr(w_x), _ptr(b_x), _ptr(w_a), _ptr(b_a), _ptr(alpha), _ptr(h0),
                                    _ptr(reset), B, L, D, _ptr(y), _ptr(y32), _ptr(hT), _ptr(saved), _ptr(scratch),
                                    _stream(dev))
    _check("rglru_proj_forward", st)
    return {"y": y, "y32": y32, "hT": hT, "saved": saved, "scratch": scratch}


def rglru_proj_backward(dy, dhT, x, w_x, b_x, w_a, b_a, alpha, h0, reset, saved, *, grad_fp32=False, out=None,
                        scratch=None):
    """Backward of rglru_proj_forward (``rglru_proj_backward``).
    Returns dict(dx, dw_x, db_x, dw_a, db_a, dalpha, dh0, scratch)."""
    dev, B, L, D, dk = _proj_params(x, w_x, b_x, w_a, b_a, alpha)
    _need(dy, "dy", torch.bfloat16, dev, (B, L, D))
    _opt(dhT, "dhT", torch.float32, dev, (B, D))
    nsaved, nscratch = rglru_proj_workspace_bytes(B, L, D)
    if saved is None or saved.numel() < nsaved:
        raise ValueError("saved must be the forward's saved buffer")
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    o = {
        "dx": _empty((B, L, D), torch.float32 if grad_fp32 else torch.bfloat16, dev, out, "dx"),
        "dw_x": _empty((PROJ_BLOCKS, dk, dk), torch.float32, dev, out, "dw_x"),
        "db_x": _empty((D,), torch.float32, dev, out, "db_x"),
        "dw_a": _empty((PROJ_BLOCKS, dk, dk), torch.float32, dev, out, "dw_a"),
        "db_a": _empty((D,), torch.float32, dev, out, "db_a"),
        "dalpha": _empty((D,), torch.float32, dev, out, "dalpha"),
        "dh0": _empty((B, D), torch.float32, dev, out, "dh0"),
    }
    st = _load().rglru_proj_backward(_ptr(dy), _ptr(dhT), _ptr(x), _ptr(w_x), _ptr(b_x), _ptr(w_a), _ptr(b_a),
                                     _ptr(alpha), _ptr(h0), _ptr(reset), B, L, D, _ptr(saved), _ptr(o["dx"]),
                                     LRS_GRAD_FP32 if grad_fp32 else LRS_GRAD_BF16, _ptr(o["dw_x"]), _ptr(o["db_x"]),
                                     _ptr(o["dw_a"]), _ptr(o["db_a"]), _ptr(o["dalpha"]), _ptr(o["dh0"]),
                                     _ptr(scratch), _stream(dev))
    _check("rglru_proj_backward", st)
    o["scratch"] = scratch
    return o


# ---------------------------------------------------------------------------
# One RecurrentBlock around the SAMU mixer
# ---------------------------------------------------------------------------
def samu_block_workspace_bytes(B: int, L: int, Dm: int, D: int, mixer: str = "samu"):
    lib = _load()
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    fn = "samu_block_workspace_bytes" if mixer == "samu" else "rglru_block_workspace_bytes"
    _check(fn, getattr(lib, fn)(B, L, Dm, D, ctypes.byref(s), ctypes.byref(c)))
    return int(s.value), int(c.value)


def _block_shapes(Dm: int, D: int) -> dict:
    M, F, dk = D // 2, 3 * Dm, D // PROJ_BLOCKS
    return {"gamma1": (Dm,), "w_in": (2 * D, Dm), "conv_k": (4, D), "conv_b": (D,), "nu": (M,), "theta": (M,),
            "w_phi": (D + 1,), "w_r": (D + 1,), "a_phi": (1,), "a_r": (1,), "w_o": (Dm, D), "gamma2": (Dm,),
            "w_mlp_in": (2 * F, Dm), "w_mlp_out": (Dm, F), "w_x": (PROJ_BLOCKS, dk, dk), "b_x": (D,),
            "w_a": (PROJ_BLOCKS, dk, dk), "b_a": (D,), "alpha": (D,)}


_BLOCK_BF16 = ("w_in", "w_o", "w_mlp_in", "w_mlp_out", "w_x", "w_a")


def _block_kind(params: dict):
    """(mixer, names, params struct, grads struct, D) of a parameter dict."""
    if "nu" in params:
        return "samu", BLOCK_PARAMS, _BlockParams, _BlockGrads, 2 * params["nu"].numel()
    return "rglru", RGLRU_BLOCK_PARAMS, _RgBlockParams, _RgBlockGrads, params["alpha"].numel()


def _block_params(params: dict, Dm: int, dev):
    mixer, names, Struct, _, D = _block_kind(params)
    shapes = _block_shapes(Dm, D)
    st = Struct()
    for n in names:
        dt = torch.bfloat16 if n in _BLOCK_BF16 else torch.float32
        setattr(st, n, _need(params.get(n), n, dt, dev, shapes[n]).data_ptr())
    return st


def _state_shape(mixer, B, D):
    return (B, D // 2, 2) if mixer == "samu" else (B, D)


def samu_block_forward(x, params: dict, h0=None, reset=None, *, out=None, saved=None, scratch=None):
    """One RecurrentBlock forward through ``samu_block_forward`` (params with
    the SAMU mixer's nu, theta, ...) or ``rglru_block_forward`` (params with
    the RG-LRU mixer's w_x, b_x, w_a, b_a, alpha).  x: [B,L,Dm] BF16.
    Returns dict(out, hT, saved, scratch)."""
    dev = x.device
    B, L, Dm = x.shape
    _need(x, "x", torch.bfloat16, dev)
    mixer, _, _, _, D = _block_kind(params)
    sshape = _state_shape(mixer, B, D)
    _opt(h0, "h0", torch.float32, dev, sshape)
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    ps = _block_params(params, Dm, dev)
    nsaved, nscratch = samu_block_workspace_bytes(B, L, Dm, D, mixer)
    y = _empty((B, L, Dm), torch.bfloat16, dev, out, "out")
    hT = _empty(sshape, torch.float32, dev, out, "hT")
    if saved is None:
        saved = torch.empty(nsaved, dtype=torch.uint8, device=dev)
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    if saved.numel() < nsaved or scratch.numel() < nscratch:
        raise ValueError("saved/scratch buffers are too small")
    fn = "samu_block_forward" if mixer == "samu" else "rglru_block_forward"
    st = getattr(_load(), fn)(ctypes.cast(ctypes.pointer(ps), _P), _ptr(x), _ptr(h0), _ptr(reset), B, L, Dm, D,
                              _ptr(y), _ptr(hT), _ptr(saved), _ptr(scratch), _stream(dev))
    _check(fn, st)
    return {"out": y, "hT": hT, "saved": saved, "scratch": scratch}


def samu_block_backward(dout, dhT, x, params: dict, h0, reset, saved, *, out=None, scratch=None):
    """Backward of samu_block_forward (either mixer).  Returns dict(dx, dh0,
    d<param> for every parameter (FP32, the parameter's shape), scratch)."""
    dev = x.device
    B, L, Dm = x.shape
    mixer, names, _, Grads, D = _block_kind(params)
    sshape = _state_shape(mixer, B, D)
    _need(dout, "dout", torch.bfloat16, dev, (B, L, Dm))
    _opt(dhT, "dhT", torch.float32, dev, sshape)
    _opt(reset, "reset", torch.uint8, dev, (B, L))
    ps = _block_params(params, Dm, dev)
    nsaved, nscratch = samu_block_workspace_bytes(B, L, Dm, D, mixer)
    if saved is None or saved.numel() < nsaved:
        raise ValueError("saved must be the forward's saved buffer")
    if scratch is None:
        scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    shapes = _block_shapes(Dm, D)
    o = {"dx": _empty((B, L, Dm), torch.bfloat16, dev, out, "dx"),
         "dh0": _empty(sshape, torch.float32, dev, out, "dh0")}
    gs = Grads()
    for n in names:
        o["d" + n] = _empty(shapes[n], torch.float32, dev, out, "d" + n)
        setattr(gs, "d" + n, o["d" + n].data_ptr())
    fn = "samu_block_backward" if mixer == "samu" else "rglru_block_backward"
    st = getattr(_load(), fn)(ctypes.cast(ctypes.pointer(ps), _P), _ptr(x), _ptr(h0), _ptr(reset), _ptr(dout),
                              _ptr(dhT), B, L, Dm, D, _ptr(saved), _ptr(o["dx"]), _ptr(o["dh0"]),
                              ctypes.cast(ctypes.pointer(gs), _P), _ptr(scratch), _stream(dev))
    _check(fn, st)
    o["scratch"] = scratch
    return o


LRS_GEMM_NT, LRS_GEMM_NN, LRS_GEMM_TN = 0, 1, 2


def dense_gemm(layout: int, A, B, M: int, N: int, K: int, *, out=None, scratch=None):
    """The block's tensor-core contraction on its own (``lrs_dense_gemm``):
    NT: C[M,N] = A[M,K] B[N,K]^T (BF16); NN: C = A[M,K] B[K,N] (BF16);
    TN: C[M,N] = A[K,M]^T B[K,N] (FP32)."""
    dev = A.device
    _need(A, "A", torch.bfloat16, dev, (K, M) if layout == LRS_GEMM_TN else (M, K))
    _need(B, "B", torch.bfloat16, dev, (N, K) if layout == LRS_GEMM_NT else (K, N))
    dt = torch.float32 if layout == LRS_GEMM_TN else torch.bfloat16
    C = out if out is not None else torch.empty((M, N), dtype=dt, device=dev)
    _need(C, "C", dt, dev, (M, N))
    if scratch is None:
        scratch = torch.empty(256, dtype=torch.uint8, device=dev)
    _check("lrs_dense_gemm", _load().lrs_dense_gemm(layout, _ptr(A), _ptr(B), _ptr(C), M, N, K, _ptr(scratch),
                                                    _stream(dev)))
    return C


def block_tensors_from_numpy(inp: dict, device) -> dict:
    """Device tensors of synth.block_inputs: {"x", "dout", "h0", "dhT", "reset", "params": {...}}."""
    params = {}
    for n in (BLOCK_PARAMS if inp.get("mixer", "samu") == "samu" else RGLRU_BLOCK_PARAMS):
        params[n] = _bf16(inp[n], device) if n in _BLOCK_BF16 else _f32(inp[n], device)
    out = {"x": _bf16(inp["x"], device), "dout": _bf16(inp["dout"], device), "h0": _f32(inp["h0"], device),
           "dhT": _f32(inp["dhT"], device), "params": params}
    out["reset"] = None if inp["reset"] is None else torch.from_numpy(inp["reset"]).to(device)
    return out


def selftest_wait_timeout(scratch, device=None) -> None:
    """Launches the library's failure-path self-test on ``scratch`` (see
    lrs_selftest_wait_timeout); with ``scratch=None``, on the status word of the
    no-allocation forward's fixed array (on ``device``)."""
    dev = scratch.device if scratch is not None else device
    _check("lrs_selftest_wait_timeout", _load().lrs_selftest_wait_timeout(_ptr(scratch), _stream(dev)))


def samu_forward_noalloc_status(device) -> int:
    """Status word of the most recent ``samu_forward_noalloc`` on ``device``
    (LRS_OK, or LRS_ERR_TIMEOUT; synchronises the current stream)."""
    v = ctypes.c_int(0)
    _check("samu_forward_noalloc_status",
           _load().samu_forward_noalloc_status(ctypes.byref(v), _stream(device)))
    return int(v.value)


def device_status(scratch, device=None) -> int:
    """Status word of the most recent call that used ``scratch`` (synchronises the stream)."""
    dev = scratch.device if device is None else device
    v = ctypes.c_int(0)
    _check("lrs_device_status", _load().lrs_device_status(_ptr(scratch), ctypes.byref(v), _stream(dev)))
    return int(v.value)


KERNEL_NAMES = {
    2: "samu_ctrl_fwd_kernel", 3: "samu_fwd_replay_kernel",
    4: "samu_bwd_main_kernel", 5: "samu_ctrl_bwd_kernel", 6: "samu_params_kernel",
    7: "rglru_scan_fwd_kernel", 8: "rglru_scan_bwd_kernel", 9: "rglru_alpha_kernels",
    10: "samu_fwd_maps_kernel", 11: "samu_bwd_maps_kernel", 12: "samu_decode_prepare_kernel",
    13: "samu_decode_step_kernel", 14: "proj_gemm_kernel<logits>", 15: "proj_gemm_kernel<dx, dW>",
    16: "proj_pack_kernel", 17: "block_gemm_kernel", 18: "rmsnorm_kernels", 19: "conv_kernels",
    20: "join_fwd_kernel", 21: "sum_parts_kernel",
}


def profile_begin(capacity: int) -> None:
    """Record CUDA events around every library kernel launched until profile_end()."""
    _check("lrs_profile_begin", _load().lrs_profile_begin(int(capacity)))


def profile_end(capacity: int):
    """Returns (list of (kernel name, ms) for the recorded launches, total launches seen)."""
    ids = (ctypes.c_int * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = ctypes.c_int(0)
    _check("lrs_profile_end", _load().lrs_profile_end(ids, ms, capacity, ctypes.byref(n)))
    k = min(n.value, capacity)
    return [(KERNEL_NAMES.get(ids[i], str(ids[i])), float(ms[i])) for i in range(k)], int(n.value)


# ---------------------------------------------------------------------------
# numpy (seeded generator output) -> device tensors
# ---------------------------------------------------------------------------
def _bf16(bits: np.ndarray, device):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def _f32(a, device):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32).reshape(np.shape(a) or (1,))).to(device)


def samu_tensors_from_numpy(inp: dict, device) -> dict:
    out = {k: _bf16(inp[k], device) for k in ("x_sel", "w", "dy")}
    for k in ("nu", "theta", "w_phi", "w_r", "a_phi", "a_r", "h0", "dhT"):
        out[k] = _f32(inp[k], device)
    out["reset"] = None if inp["reset"] is None else torch.from_numpy(inp["reset"]).to(device)
    return out


def rglru_proj_tensors_from_numpy(inp: dict, device) -> dict:
    out = {k: _bf16(inp[k], device) for k in ("x", "w_x", "w_a", "dy")}
    for k in ("b_x", "b_a", "alpha", "h0", "dhT"):
        out[k] = _f32(inp[k], device)
    out["reset"] = None if inp["reset"] is None else torch.from_numpy(inp["reset"]).to(device)
    return out


def rglru_tensors_from_numpy(inp: dict, device) -> dict:
    out = {k: _bf16(inp[k], device) for k in ("x", "lx", "la", "dy")}
    for k in ("alpha", "h0", "dhT"):
        out[k] = _f32(inp[k], device)
    out["reset"] = None if inp["reset"] is None else torch.from_numpy(inp["reset"]).to(device)
    return out
