"""FP64 CPU oracle for the SAMU mixer and the RG-LRU scan (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product path never does.  The C
source ``oracle.c`` is the plain sequential definition of the equations on the
SAMU GPU page (section 05 for SAMU, section 04 for RG-LRU) and shares no code
with the CUDA library.

Every function takes float64 numpy arrays in the layouts documented in
``oracle.c`` and returns float64 results.  Parity status: every function here
is pinned by ``tests/test_oracle_pins.py`` (closed forms, special cases,
invariants, finite differences, the pages' printed parameter counts).
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


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            i = ctypes.c_int
            d = ctypes.c_double
            lib.oracle_samu_forward.argtypes = [i, i, i, dp, dp, dp, u8p, dp, dp, dp, dp, d, d, dp, dp, dp]
            lib.oracle_samu_forward.restype = None
            lib.oracle_samu_backward.argtypes = [i, i, i, dp, dp, dp, u8p, dp, dp, dp, dp, d, d,
                                                 dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_samu_backward.restype = None
            lib.oracle_rglru_forward.argtypes = [i, i, i, dp, dp, dp, dp, dp, u8p, dp, dp]
            lib.oracle_rglru_forward.restype = None
            lib.oracle_rglru_backward.argtypes = [i, i, i, dp, dp, dp, dp, dp, u8p, dp, dp,
                                                  dp, dp, dp, dp, dp]
            lib.oracle_rglru_backward.restype = None
            lib.oracle_bf16_rne_array.argtypes = [dp, ctypes.POINTER(ctypes.c_uint16), ctypes.c_long]
            lib.oracle_bf16_rne_array.restype = None
            _lib = lib
    return _lib


def _dptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _u8(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.uint8)


def _u8ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def bf16_rne(v) -> np.ndarray:
    """Round float64 values to bfloat16 (ties to even) directly; returns uint16 bit patterns."""
    lib = _load()
    v = _f64(v)
    out = np.empty(v.shape, dtype=np.uint16)
    lib.oracle_bf16_rne_array(_dptr(v), out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), v.size)
    return out


def samu_forward(x_sel, w, h0, reset, nu, theta, w_phi, w_r, a_phi, a_r):
    """SAMU mixer forward.  x_sel, w: [B,L,D]; h0: [B,M,2] or None; reset: [B,L] or None.

    Returns dict(y=[B,L,D], hT=[B,M,2], ctrl=[B,L,5] with columns p, r, E, C, S).
    """
    lib = _load()
    x_sel, w = _f64(x_sel), _f64(w)
    B, L, D = x_sel.shape
    M = D // 2
    h0, reset = _f64(h0), _u8(reset)
    nu, theta, w_phi, w_r = _f64(nu), _f64(theta), _f64(w_phi), _f64(w_r)
    y = np.empty((B, L, D))
    hT = np.empty((B, M, 2))
    ctrl = np.empty((B, L, 5))
    lib.oracle_samu_forward(B, L, D, _dptr(x_sel), _dptr(w), _dptr(h0), _u8ptr(reset),
                            _dptr(nu), _dptr(theta), _dptr(w_phi), _dptr(w_r),
                            float(a_phi), float(a_r), _dptr(y), _dptr(hT), _dptr(ctrl))
    return {"y": y, "hT": hT, "ctrl": ctrl}


def samu_decode_step(x_sel, w, state, reset, nu, theta, w_phi, w_r, a_phi, a_r):
    """One token of each of B sequences: the forward definition ([SAMU page]
    section 05) over a single token with the carried state as z_{t-1}.

    x_sel, w: [B,D]; state: [B,M,2]; reset: [B] or None.  Returns dict(y=[B,D],
    state=[B,M,2], ctrl=[B,5]).  Token after token it reproduces samu_forward
    over the sequence (pinned in tests/test_oracle_pins.py)."""
    x_sel, w = _f64(x_sel), _f64(w)
    rs = None if reset is None else np.asarray(reset).reshape(-1, 1)
    f = samu_forward(x_sel[:, None, :], w[:, None, :], state, rs, nu, theta, w_phi, w_r, a_phi, a_r)
    return {"y": f["y"][:, 0, :], "state": f["hT"], "ctrl": f["ctrl"][:, 0, :]}


def samu_chunk_transition(nu, theta, E, d, reset=None):
    """Transition of a chunk of K consecutive tokens, P_m = prod_t lambda_{t,m},
    by the closed form of the SAMU GPU page (section 05, exact chunk closed
    form): P_m = e^{-nu_m G} e^{i (K theta_m + D)} with G = sum_t E_t and
    D = sum_t d_t; zero when a token of the chunk is a reset (lambda = 0 there).

    nu, theta: [M]; E, d: [K] (the chunk's per-token controls); reset: [K] or
    None.  FP64 numpy; returns complex [M]."""
    nu, theta = np.asarray(nu, np.float64), np.asarray(theta, np.float64)
    E, d = np.asarray(E, np.float64), np.asarray(d, np.float64)
    if reset is not None and np.any(np.asarray(reset) != 0):
        return np.zeros(nu.shape, np.complex128)
    K = E.shape[0]
    return np.exp(-nu * E.sum()) * np.exp(1j * (K * theta + d.sum()))


def samu_backward(x_sel, w, h0, reset, nu, theta, w_phi, w_r, a_phi, a_r, dy, dhT):
    """SAMU mixer backward (hand-derived adjoint).  dhT may be None (zero).

    Returns dict(dx_sel, dw, dh0, dnu, dtheta, dw_phi, dw_r, da_phi, da_r).
    """
    lib = _load()
    x_sel, w, dy = _f64(x_sel), _f64(w), _f64(dy)
    B, L, D = x_sel.shape
    M = D // 2
    h0, reset, dhT = _f64(h0), _u8(reset), _f64(dhT)
    nu, theta, w_phi, w_r = _f64(nu), _f64(theta), _f64(w_phi), _f64(w_r)
    out = {
        "dx_sel": np.empty((B, L, D)), "dw": np.empty((B, L, D)), "dh0": np.empty((B, M, 2)),
        "dnu": np.empty(M), "dtheta": np.empty(M), "dw_phi": np.empty(D + 1), "dw_r": np.empty(D + 1),
    }
    da_phi = ctypes.c_double(0.0)
    da_r = ctypes.c_double(0.0)
    lib.oracle_samu_backward(B, L, D, _dptr(x_sel), _dptr(w), _dptr(h0), _u8ptr(reset),
                             _dptr(nu), _dptr(theta), _dptr(w_phi), _dptr(w_r),
                             float(a_phi), float(a_r), _dptr(dy), _dptr(dhT),
                             _dptr(out["dx_sel"]), _dptr(out["dw"]), _dptr(out["dh0"]),
                             _dptr(out["dnu"]), _dptr(out["dtheta"]),
                             _dptr(out["dw_phi"]), _dptr(out["dw_r"]),
                             ctypes.byref(da_phi), ctypes.byref(da_r))
    out["da_phi"] = da_phi.value
    out["da_r"] = da_r.value
    return out


def rglru_forward(x, lx, la, alpha, h0, reset):
    """RG-LRU forward.  x, lx, la: [B,L,D]; alpha: [D]; h0: [B,D] or None.  Returns dict(y, hT)."""
    lib = _load()
    x, lx, la = _f64(x), _f64(lx), _f64(la)
    B, L, D = x.shape
    alpha, h0, reset = _f64(alpha), _f64(h0), _u8(reset)
    y = np.empty((B, L, D))
    hT = np.empty((B, D))
    lib.oracle_rglru_forward(B, L, D, _dptr(x), _dptr(lx), _dptr(la), _dptr(alpha), _dptr(h0),
                             _u8ptr(reset), _dptr(y), _dptr(hT))
    return {"y": y, "hT": hT}


def rglru_backward(x, lx, la, alpha, h0, reset, dy, dhT):
    """RG-LRU backward.  Returns dict(dx, dlx, dla, dalpha, dh0)."""
    lib = _load()
    x, lx, la, dy = _f64(x), _f64(lx), _f64(la), _f64(dy)
    B, L, D = x.shape
    alpha, h0, reset, dhT = _f64(alpha), _f64(h0), _u8(reset), _f64(dhT)
    out = {"dx": np.empty((B, L, D)), "dlx": np.empty((B, L, D)), "dla": np.empty((B, L, D)),
           "dalpha": np.empty(D), "dh0": np.empty((B, D))}
    lib.oracle_rglru_backward(B, L, D, _dptr(x), _dptr(lx), _dptr(la), _dptr(alpha), _dptr(h0),
                              _u8ptr(reset), _dptr(dy), _dptr(dhT),
                              _dptr(out["dx"]), _dptr(out["dlx"]), _dptr(out["dla"]),
                              _dptr(out["dalpha"]), _dptr(out["dh0"]))
    return out


# ---------------------------------------------------------------------------
# RG-LRU mixer with its two block-diagonal gate projections (SAMU GPU page,
# section 04 forward "two canonical block-diagonal projections" and the
# section 06 parameter table; protocol page "RG-LRU 的固定方程": 16-block
# block-diagonal linear layers).  Plain FP64 numpy for the projections and
# their chain rule, the C oracle above for the scan.
# ---------------------------------------------------------------------------
def rglru_gate_projection(x, w, b):
    """l[..., h dk + o] = sum_i x[..., h dk + i] w[h, i, o] + b[h dk + o].

    x: [..., D]; w: [H, dk, dk] with H dk = D; b: [D].  FP64."""
    x, w, b = _f64(x), _f64(w), _f64(b)
    H, dk, _ = w.shape
    xf = x.reshape(-1, H, dk)
    out = np.empty(xf.shape)
    for h in range(H):                       # one matrix product per diagonal block
        out[:, h, :] = xf[:, h, :] @ w[h]
    return out.reshape(x.shape) + b


def rglru_proj_forward(x, w_x, b_x, w_a, b_a, alpha, h0, reset):
    """RG-LRU forward on the projected logits.  Returns dict(y, hT, lx, la)."""
    lx = rglru_gate_projection(x, w_x, b_x)
    la = rglru_gate_projection(x, w_a, b_a)
    out = rglru_forward(x, lx, la, alpha, h0, reset)
    out["lx"], out["la"] = lx, la
    return out


def rglru_proj_backward(x, w_x, b_x, w_a, b_a, alpha, h0, reset, dy, dhT):
    """Backward of rglru_proj_forward: the scan's own gradients (dx through the
    write term, dl^x, dl^a, dalpha, dh0) and the chain rule through the two
    projections: dx += dl W^T per block, dW[h] = sum_{b,t} x_h^T dl_h,
    db = sum_{b,t} dl.  Returns dict(dx, dw_x, db_x, dw_a, db_a, dalpha, dh0)."""
    x = _f64(x)
    lx = rglru_gate_projection(x, w_x, b_x)
    la = rglru_gate_projection(x, w_a, b_a)
    g = rglru_backward(x, lx, la, alpha, h0, reset, dy, dhT)
    w_x, w_a = _f64(w_x), _f64(w_a)
    H, dk, _ = w_x.shape
    xf, gx, ga = x.reshape(-1, H, dk), g["dlx"].reshape(-1, H, dk), g["dla"].reshape(-1, H, dk)
    dxp = np.empty(xf.shape)
    dw_x, dw_a = np.empty(w_x.shape), np.empty(w_a.shape)
    for h in range(H):                       # per diagonal block: dx += dl W^T, dW = x^T dl
        dxp[:, h, :] = gx[:, h, :] @ w_x[h].T + ga[:, h, :] @ w_a[h].T
        dw_x[h] = xf[:, h, :].T @ gx[:, h, :]
        dw_a[h] = xf[:, h, :].T @ ga[:, h, :]
    lead = tuple(range(x.ndim - 1))
    return {"dx": g["dx"] + dxp.reshape(x.shape),
            "dw_x": dw_x, "db_x": g["dlx"].sum(axis=lead),
            "dw_a": dw_a, "db_a": g["dla"].sum(axis=lead),
            "dalpha": g["dalpha"], "dh0": g["dh0"]}
