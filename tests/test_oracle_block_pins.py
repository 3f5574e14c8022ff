"""Pins of the FP64 RecurrentBlock oracle (oracle/block.py) against facts that
do not come from the oracle itself: central finite differences of the plain
FP64 block for every gradient it returns, numpy's convolution segment by
segment, the odd-part identity of the tanh-form GeLU, RMSNorm's closed form
and the residual identities of the block with its output projections zeroed."""
import numpy as np
import pytest

import oracle
from oracle import block as ob


def _params(rng, Dm, D, F, active=True):
    M = D // 2
    s = lambda *shape: rng.standard_normal(shape)
    return {
        "gamma1": 1.0 + 0.2 * s(Dm), "w_g": 0.4 * s(D, Dm), "w_v": 0.4 * s(D, Dm),
        "conv_k": 0.5 * s(4, D), "conv_b": 0.1 * s(D),
        "nu": rng.uniform(0.05, 0.6, M), "theta": rng.uniform(-np.pi, np.pi, M),
        "w_phi": s(D + 1), "w_r": s(D + 1),
        "a_phi": 0.7 if active else 0.0, "a_r": -0.5 if active else 0.0,
        "w_o": 0.4 * s(Dm, D), "gamma2": 1.0 + 0.2 * s(Dm),
        "w_1": 0.4 * s(F, Dm), "w_2": 0.4 * s(F, Dm), "w_3": 0.3 * s(Dm, F),
    }


def _rglru_params(rng, Dm, D, F):
    """The block's own parameters with the RG-LRU mixer's (16 gate-projection
    blocks of width D/16)."""
    p = _params(rng, Dm, D, F)
    for k in ("nu", "theta", "w_phi", "w_r", "a_phi", "a_r"):
        del p[k]
    dk = D // 16
    p["w_x"] = rng.standard_normal((16, dk, dk)) / np.sqrt(dk)
    p["w_a"] = rng.standard_normal((16, dk, dk)) / np.sqrt(dk)
    p["b_x"] = 0.1 * rng.standard_normal(D)
    p["b_a"] = 0.1 * rng.standard_normal(D)
    p["alpha"] = rng.uniform(-4.0, -1.0, D)
    return p


def _case(seed=3, B=2, L=11, Dm=6, D=8, mixer="samu"):
    rng = np.random.default_rng(seed)
    F = 3 * Dm
    p = _params(rng, Dm, D, F) if mixer == "samu" else _rglru_params(rng, Dm, D, F)
    x = rng.standard_normal((B, L, Dm))
    h0 = 0.3 * rng.standard_normal((B, D // 2, 2) if mixer == "samu" else (B, D))
    reset = np.zeros((B, L), dtype=np.uint8)
    reset[1, 5] = 1
    reset[0, 9] = 1
    return rng, p, x, h0, reset


def _loss(x, p, h0, reset, R, S, mixer="samu"):
    f = ob.samu_block_forward(x, p, h0, reset, bf16=False, mixer=mixer)
    return float(np.sum(f["out"] * R) + np.sum(f["hT"] * S))


GRAD_OF = {"gamma1": "dgamma1", "w_g": "dw_g", "w_v": "dw_v", "conv_k": "dconv_k", "conv_b": "dconv_b",
           "nu": "dnu", "theta": "dtheta", "w_phi": "dw_phi", "w_r": "dw_r", "a_phi": "da_phi", "a_r": "da_r",
           "w_o": "dw_o", "gamma2": "dgamma2", "w_1": "dw_1", "w_2": "dw_2", "w_3": "dw_3"}


def test_block_gradients_match_central_differences():
    rng, p, x, h0, reset = _case()
    R = rng.standard_normal((x.shape[0], x.shape[1], x.shape[2]))
    S = rng.standard_normal(h0.shape)
    g = ob.samu_block_backward(x, p, R, h0, reset, dhT=S, bf16=False)
    eps = 1e-5

    def check(name, grad, perturb):
        d = rng.standard_normal(np.shape(grad))
        lp = _loss(*perturb(+eps * d), R, S)
        lm = _loss(*perturb(-eps * d), R, S)
        fd = (lp - lm) / (2 * eps)
        an = float(np.sum(np.asarray(grad) * d))
        assert abs(fd - an) <= 2e-6 * max(1.0, abs(an)), (name, fd, an)

    for key, gk in GRAD_OF.items():
        def perturb(delta, key=key):
            q = dict(p)
            q[key] = p[key] + (delta if np.ndim(p[key]) else float(delta))
            return x, q, h0, reset
        check(key, g[gk], perturb)
    check("x", g["dx"], lambda delta: (x + delta, p, h0, reset))
    check("h0", g["dh0"], lambda delta: (x, p, h0 + delta, reset))


RGLRU_GRAD_OF = {"gamma1": "dgamma1", "w_g": "dw_g", "w_v": "dw_v", "conv_k": "dconv_k", "conv_b": "dconv_b",
                 "w_x": "dw_x", "b_x": "db_x", "w_a": "dw_a", "b_a": "db_a", "alpha": "dalpha",
                 "w_o": "dw_o", "gamma2": "dgamma2", "w_1": "dw_1", "w_2": "dw_2", "w_3": "dw_3"}


def test_rglru_block_gradients_match_central_differences():
    """The same pins for the block with the RG-LRU mixer (the pages' comparison),
    D = 32 (16 gate-projection blocks of width 2); the gates stay inside the
    square-root clip's unclipped branch on these inputs."""
    rng, p, x, h0, reset = _case(seed=4, D=32, mixer="rglru")
    R = rng.standard_normal(x.shape)
    S = rng.standard_normal(h0.shape)
    g = ob.samu_block_backward(x, p, R, h0, reset, dhT=S, bf16=False, mixer="rglru")
    eps = 1e-5

    def check(name, grad, perturb):
        d = rng.standard_normal(np.shape(grad))
        lp = _loss(*perturb(+eps * d), R, S, mixer="rglru")
        lm = _loss(*perturb(-eps * d), R, S, mixer="rglru")
        fd = (lp - lm) / (2 * eps)
        an = float(np.sum(np.asarray(grad) * d))
        assert abs(fd - an) <= 2e-6 * max(1.0, abs(an)), (name, fd, an)

    for key, gk in RGLRU_GRAD_OF.items():
        def perturb(delta, key=key):
            q = dict(p)
            q[key] = p[key] + delta
            return x, q, h0, reset
        check(key, g[gk], perturb)
    check("x", g["dx"], lambda delta: (x + delta, p, h0, reset))
    check("h0", g["dh0"], lambda delta: (x, p, h0 + delta, reset))


def test_conv_matches_numpy_convolve_per_segment():
    rng = np.random.default_rng(5)
    B, L, D = 2, 13, 5
    v = rng.standard_normal((B, L, D))
    k = rng.standard_normal((4, D))
    kb = rng.standard_normal(D)
    reset = np.zeros((B, L), dtype=np.uint8)
    reset[0, 4] = reset[0, 6] = reset[1, 12] = 1
    start = ob.segment_starts(reset, B, L)
    u = ob.conv_forward(v, k, kb, start)
    for b in range(B):
        bounds = [t for t in range(L) if t == 0 or reset[b, t]] + [L]
        for s0, s1 in zip(bounds[:-1], bounds[1:]):
            for c in range(D):
                ref = np.convolve(v[b, s0:s1, c], k[:, c])[: s1 - s0] + kb[c]
                np.testing.assert_allclose(u[b, s0:s1, c], ref, rtol=1e-13, atol=1e-13)


def test_conv_identity_kernel_passes_input_through():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, 9, 3))
    k = np.zeros((4, 3))
    k[0] = 1.0
    u = ob.conv_forward(v, k, np.zeros(3), ob.segment_starts(None, 1, 9))
    np.testing.assert_array_equal(u, v)


def test_gelu_odd_part_and_derivative():
    x = np.linspace(-6, 6, 241)
    np.testing.assert_allclose(ob.gelu(x) - ob.gelu(-x), x, rtol=0, atol=1e-14)
    assert ob.gelu(np.array([0.0]))[0] == 0.0
    h = 1e-6
    fd = (ob.gelu(x + h) - ob.gelu(x - h)) / (2 * h)
    np.testing.assert_allclose(ob.gelu_grad(x), fd, rtol=1e-7, atol=1e-8)


def test_rmsnorm_closed_form():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4, 10)) * 3.0
    h, rstd = ob.rmsnorm(x, np.ones(10))
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(h * h, axis=-1), ms / (ms + ob.EPS), rtol=1e-13)
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt(ms + ob.EPS), rtol=1e-14)
    c = np.full((1, 8), 2.5)
    hc, _ = ob.rmsnorm(c, np.arange(1.0, 9.0))
    np.testing.assert_allclose(hc[0], np.arange(1.0, 9.0) * 2.5 / np.sqrt(6.25 + ob.EPS), rtol=1e-14)


def test_block_residual_identities():
    rng, p, x, h0, reset = _case(seed=9)
    q = dict(p)
    q["w_o"] = np.zeros_like(p["w_o"])
    q["w_3"] = np.zeros_like(p["w_3"])
    f = ob.samu_block_forward(x, q, h0, reset, bf16=False)
    np.testing.assert_array_equal(f["out"], x)
    # with only the MLP's output projection zeroed, out = x + (GeLU(g) * y_mixer) W_o^T, the mixer
    # called directly on the convolution's output
    q = dict(p)
    q["w_3"] = np.zeros_like(p["w_3"])
    f = ob.samu_block_forward(x, q, h0, reset, bf16=False)
    h1, _ = ob.rmsnorm(x, p["gamma1"])
    v = h1 @ p["w_v"].T
    u = ob.conv_forward(v, p["conv_k"], p["conv_b"], ob.segment_starts(reset, *x.shape[:2]))
    ym = oracle.samu_forward(u, u, h0, reset, p["nu"], p["theta"], p["w_phi"], p["w_r"], p["a_phi"],
                             p["a_r"])["y"]
    ref = x + (ob.gelu(h1 @ p["w_g"].T) * ym) @ p["w_o"].T
    np.testing.assert_allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


def test_block_bf16_points_round_every_stored_tensor():
    rng, p, x, h0, reset = _case(seed=11)
    x = ob._bf(x, True)
    f = ob.samu_block_forward(x, p, h0, reset, bf16=True)
    for k in ("h1", "g", "v", "u", "ym", "j", "r1", "h2", "a", "b", "q", "out"):
        np.testing.assert_array_equal(ob._bf(f[k], True), f[k], err_msg=k)
    plain = ob.samu_block_forward(x, p, h0, reset, bf16=False)
    rel = np.linalg.norm(f["out"] - plain["out"]) / np.linalg.norm(plain["out"])
    assert 1e-5 < rel < 2e-2, rel
