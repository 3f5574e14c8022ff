"""FP64 oracle of one RecurrentBlock with the SAMU mixer inside (forward and
hand-derived backward).

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): the tests, the smoke
check and the benchmark's CPU legs may import it; the product path never does.

What the block is.  The SAMU GPU page ("SAMU 与 RG-LRU 的 H800 训练性能对比",
section 03, the single-block table; the glossary entries on the mixer and the
complete block) lists its layers: a normalisation, two input projections, a
per-channel (depthwise) convolution, the recurrent mixer, the join with the
other branch and the output projection, a second normalisation and a gated
MLP, with the input and parameter backward.  The SAMU project page (the
mixer's equations) adds that the block's existing wide input branch, split
into its real and imaginary halves, is the mixer's write w, with no extra
projection.  Everything else is left open; the readings taken here (each
listed in the design notes) are:
  - both normalisations are RMSNorm with a learned scale gamma and eps 1e-6:
    h = x / sqrt(mean(x^2) + eps) * gamma;
  - GeLU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)));
  - the two input projections are bias-free: g = h W_g^T (gate branch),
    v = h W_v^T (recurrent branch), W_g, W_v: [D, Dm];
  - the convolution is causal, width 4, per channel, with a bias:
    u[t, c] = kb[c] + sum_{j<4} k[j, c] v[t - j, c], taps before the start of
    t's segment (the last reset at or before t; t = 0 always starts one) are
    zero, so nothing leaks across a packed-sequence boundary;
  - the mixer reads x_sel = w = u (SAMU); the RG-LRU block, the pages'
    comparison, puts the RG-LRU mixer with its two 16-block gate projections
    (oracle.rglru_proj_forward) in the same place, on x = u;
  - the join is j = GeLU(g) * y_mixer, then r1 = x + j W_o^T (W_o: [Dm, D]);
  - the gated MLP has hidden width F = 3 Dm: q = GeLU(h2 W_1^T) * (h2 W_2^T),
    out = r1 + q W_3^T (W_1, W_2: [F, Dm]; W_3: [Dm, F]).

bf16=True rounds (round to nearest even) every tensor the CUDA path stores in
BF16, at the same points and from the same operands; bf16=False is the plain
FP64 function, the one the finite-difference pins differentiate.
"""
from __future__ import annotations

import numpy as np

from . import bf16_rne, rglru_proj_backward, rglru_proj_forward, samu_backward, samu_forward

EPS = 1e-6
GELU_C = np.sqrt(2.0 / np.pi)
GELU_A = 0.044715
CONV_W = 4


def _bf(a, on):
    """BF16 round trip (RNE) of float64 values when `on`, else the values."""
    if not on:
        return np.asarray(a, dtype=np.float64)
    bits = bf16_rne(a).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def gelu(x):
    return 0.5 * x * (1.0 + np.tanh(GELU_C * (x + GELU_A * x ** 3)))


def gelu_grad(x):
    """d GeLU / dx of the tanh form."""
    u = GELU_C * (x + GELU_A * x ** 3)
    th = np.tanh(u)
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * GELU_C * (1.0 + 3.0 * GELU_A * x * x)


def rmsnorm(x, gamma):
    """RMSNorm over the last axis: returns (h, rstd) with rstd = 1/sqrt(mean(x^2) + eps)."""
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)
    return x * rstd * gamma, rstd[..., 0]


def rmsnorm_backward(x, gamma, rstd, dh):
    """Gradients of h = x rstd gamma: (dx, dgamma).  With n = x rstd and
    g = dh gamma: dx = rstd (g - n mean(g n))."""
    r = rstd[..., None]
    n = x * r
    g = dh * gamma
    dx = r * (g - n * np.mean(g * n, axis=-1, keepdims=True))
    lead = tuple(range(x.ndim - 1))
    return dx, np.sum(dh * n, axis=lead)


def segment_starts(reset, B, L):
    """start[b, t] = the last t' <= t with reset[b, t'] set (t' = 0 if none)."""
    start = np.zeros((B, L), dtype=np.int64)
    for b in range(B):
        s = 0
        for t in range(L):
            if t == 0 or (reset is not None and reset[b, t]):
                s = t
            start[b, t] = s
    return start


def conv_forward(v, k, kb, start):
    """u[b, t, c] = kb[c] + sum_j k[j, c] v[b, t - j, c] over the taps that stay in t's segment."""
    B, L, _ = v.shape
    u = np.broadcast_to(kb, v.shape).copy()
    for j in range(CONV_W):
        for t in range(L):
            ok = (t - j >= 0) & (t - j >= start[:, t])          # [B]
            if j <= t:
                u[:, t, :] += np.where(ok[:, None], k[j] * v[:, t - j, :], 0.0)
    return u


def conv_backward(v, k, start, du):
    """Adjoint of conv_forward: dv[t - j] += k[j] du[t] on the kept taps;
    dk[j] = sum du[t] v[t - j]; dkb = sum du."""
    B, L, _ = v.shape
    dv = np.zeros_like(v)
    dk = np.zeros_like(k)
    for j in range(CONV_W):
        for t in range(j, L):
            ok = (t - j >= start[:, t])[:, None]
            dv[:, t - j, :] += np.where(ok, k[j] * du[:, t, :], 0.0)
            dk[j] += np.sum(np.where(ok, du[:, t, :] * v[:, t - j, :], 0.0), axis=0)
    return dv, dk, du.sum(axis=(0, 1))


def _mixer_forward(mixer, u, p, h0, reset):
    if mixer == "samu":
        return samu_forward(u, u, h0, reset, p["nu"], p["theta"], p["w_phi"], p["w_r"], p["a_phi"], p["a_r"])
    return rglru_proj_forward(u, p["w_x"], p["b_x"], p["w_a"], p["b_a"], p["alpha"], h0, reset)


def _mixer_backward(mixer, u, p, h0, reset, dym, dhT, r):
    """The mixer's input gradient (BF16 points as the CUDA path stores them)
    and its parameter gradients."""
    if mixer == "samu":
        gm = samu_backward(u, u, h0, reset, p["nu"], p["theta"], p["w_phi"], p["w_r"], p["a_phi"], p["a_r"],
                           dym, dhT)
        du = r(gm["dx_sel"]) + r(gm["dw"])          # x_sel = w = u: both gradients reach u
        keys = ("dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r", "dh0")
    else:
        gm = rglru_proj_backward(u, p["w_x"], p["b_x"], p["w_a"], p["b_a"], p["alpha"], h0, reset, dym, dhT)
        du = r(gm["dx"])
        keys = ("dw_x", "db_x", "dw_a", "db_a", "dalpha", "dh0")
    return du, {k: gm[k] for k in keys}


def samu_block_forward(x, p, h0=None, reset=None, bf16=True, mixer="samu"):
    """x: [B, L, Dm]; p: dict of parameters (gamma1, w_g, w_v, conv_k, conv_b,
    the mixer's: nu, theta, w_phi, w_r, a_phi, a_r for SAMU, w_x, b_x, w_a,
    b_a, alpha for mixer="rglru"; w_o, gamma2, w_1, w_2, w_3), all float64
    (BF16 values where the CUDA path keeps them in BF16).  Returns a dict with
    out [B, L, Dm], hT (the mixer's final state) and every saved
    intermediate."""
    x = np.asarray(x, dtype=np.float64)
    B, L, _ = x.shape
    r = lambda a: _bf(a, bf16)
    h1, rstd1 = rmsnorm(x, p["gamma1"])
    h1 = r(h1)
    g = r(h1 @ p["w_g"].T)
    v = r(h1 @ p["w_v"].T)
    start = segment_starts(reset, B, L)
    u = r(conv_forward(v, p["conv_k"], p["conv_b"], start))
    mix = _mixer_forward(mixer, u, p, h0, reset)
    ym = r(mix["y"])
    j = r(gelu(g) * ym)
    r1 = r(x + j @ p["w_o"].T)
    h2, rstd2 = rmsnorm(r1, p["gamma2"])
    h2 = r(h2)
    a = r(h2 @ p["w_1"].T)
    b = r(h2 @ p["w_2"].T)
    q = r(gelu(a) * b)
    out = r(r1 + q @ p["w_3"].T)
    return {"out": out, "hT": mix["hT"], "h1": h1, "rstd1": rstd1, "g": g, "v": v, "u": u, "ym": ym,
            "j": j, "r1": r1, "h2": h2, "rstd2": rstd2, "a": a, "b": b, "q": q, "start": start}


def samu_block_backward(x, p, dout, h0=None, reset=None, dhT=None, bf16=True, mixer="samu"):
    """Backward of samu_block_forward for the cotangents dout [B, L, Dm] and
    dhT (the mixer's final state; None: zero).  Returns dx and the gradient of
    every parameter (keys d<name>), plus dh0."""
    x = np.asarray(x, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    f = samu_block_forward(x, p, h0, reset, bf16, mixer)
    r = lambda a: _bf(a, bf16)
    flat = lambda a: a.reshape(-1, a.shape[-1])
    # gated MLP: out = r1 + q W_3^T, q = GeLU(a) b
    dq = dout @ p["w_3"]
    dw_3 = flat(dout).T @ flat(f["q"])
    da = r(dq * f["b"] * gelu_grad(f["a"]))
    db = r(dq * gelu(f["a"]))
    dh2 = r(da @ p["w_1"] + db @ p["w_2"])
    dw_1 = flat(da).T @ flat(f["h2"])
    dw_2 = flat(db).T @ flat(f["h2"])
    dr1n, dgamma2 = rmsnorm_backward(f["r1"], p["gamma2"], f["rstd2"], dh2)
    dr1 = r(dout + dr1n)
    # join: r1 = x + j W_o^T, j = GeLU(g) ym
    dj = dr1 @ p["w_o"]
    dw_o = flat(dr1).T @ flat(f["j"])
    dym = r(dj * gelu(f["g"]))
    dg = r(dj * f["ym"] * gelu_grad(f["g"]))
    # the mixer: the oracle's own adjoint, BF16 outputs as the CUDA path stores them
    du, gm = _mixer_backward(mixer, f["u"], p, h0, reset, dym, dhT, r)
    dv, dconv_k, dconv_b = conv_backward(f["v"], p["conv_k"], f["start"], du)
    dv = r(dv)
    # input projections and the first norm
    dh1 = r(dg @ p["w_g"] + dv @ p["w_v"])
    dw_g = flat(dg).T @ flat(f["h1"])
    dw_v = flat(dv).T @ flat(f["h1"])
    dxn, dgamma1 = rmsnorm_backward(x, p["gamma1"], f["rstd1"], dh1)
    dx = r(dr1 + dxn)
    out = {"dx": dx, "dgamma1": dgamma1, "dw_g": dw_g, "dw_v": dw_v, "dconv_k": dconv_k, "dconv_b": dconv_b,
           "dw_o": dw_o, "dgamma2": dgamma2, "dw_1": dw_1, "dw_2": dw_2, "dw_3": dw_3}
    out.update(gm)
    return out
