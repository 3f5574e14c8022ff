"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Sources (cited by page title and section):
  SAMU GPU page  = "SAMU 与 RG-LRU 的 H800 训练性能对比", section 05 (SAMU
                   controller / transition / recurrence / composition / adjoint),
                   section 04 (RG-LRU equations and reset rule), section 06
                   (parameter-count table).
  Final report   = "SAMU strengthened-baseline H800 report" (exact RTU
                   degeneration at zero controller amplitude).

Each pin is chosen so that a plausible slip in the oracle (a sign, a swapped
real/imaginary half, a wrong normalisation span, a dropped term of the adjoint)
fails at least one of them:
  * closed forms: geometric series when the transition is constant in time
    (zero amplitudes = RTU degeneration; or all-zero x_sel tokens, where every
    token has the same controls), computed with numpy complex exponentials in
    polar form rather than the pages' expanded cos/sin product;
  * one-hot single-token controller values;
  * reset semantics (z_t = b_t) and non-leakage;
  * the algebra of the affine composition (associativity, chunked and grouped
    prefix compositions equal the step recurrence);
  * central finite differences of the forward for every input and parameter;
  * the pages' printed parameter counts;
  * the chunk closed form (section 05) against the forward's own state
    transition over a chunk with zero writes.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng0 = np.random.default_rng


def _samu_rand(B, L, D, seed, reset_p=0.0, amps=True, h0=True):
    r = rng0(seed)
    M = D // 2
    inp = dict(
        x_sel=r.standard_normal((B, L, D)),
        w=r.standard_normal((B, L, D)),
        h0=0.3 * r.standard_normal((B, M, 2)) if h0 else None,
        reset=(r.random((B, L)) < reset_p).astype(np.uint8) if reset_p > 0 else None,
        nu=-np.log(r.uniform(0.9, 0.999, M)),
        theta=r.uniform(0, 2 * math.pi, M),
        w_phi=r.standard_normal(D + 1),
        w_r=r.standard_normal(D + 1),
        a_phi=float(r.uniform(-1, 1)) if amps else 0.0,
        a_r=float(r.uniform(-1, 1)) if amps else 0.0,
    )
    return inp


def _cplx(y, M):
    """[.., L, D] halves layout -> complex [.., L, M]."""
    return y[..., :M] + 1j * y[..., M:]


# ---------------------------------------------------------------------------
# BF16 rounding helper
# ---------------------------------------------------------------------------

def test_bf16_rne_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    r = rng0(1)
    v = np.concatenate([r.standard_normal(20000) * 10.0 ** r.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40]]).astype(np.float32)
    ours = oracle.bf16_rne(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_rne_ties_and_no_double_rounding():
    # 1 + 2^-8 is half-way between 1 and 1 + 2^-7: ties to even -> 1.0
    assert oracle.bf16_rne(np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    # 1 + 3*2^-8 is half-way between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6
    assert oracle.bf16_rne(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # just above the half-way point: a detour through float would round to the
    # tie and then to even (1.0); the direct rounding must go up
    assert oracle.bf16_rne(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert oracle.bf16_rne(np.array([-(1 + 2.0 ** -8 + 2.0 ** -40)]))[0] == 0xBF81


# ---------------------------------------------------------------------------
# Parameter set: the pages' printed parameter counts (3D + 4)
# ---------------------------------------------------------------------------

def test_parameter_count_matches_pages_table():
    rows = [tuple(int(v) for v in line.split()) for line in open(os.path.join(GOLDEN, "param_counts.txt"))
            if line.strip() and not line.startswith("#")]
    assert rows
    for D, count in rows:
        inp = _samu_rand(1, 2, D, seed=D)
        g = oracle.samu_backward(**inp, dy=np.ones((1, 2, D)), dhT=None)
        n = (g["dnu"].size + g["dtheta"].size + g["dw_phi"].size + g["dw_r"].size
             + np.size(g["da_phi"]) + np.size(g["da_r"]))
        assert n == count, (D, n, count)


# ---------------------------------------------------------------------------
# Forward closed forms
# ---------------------------------------------------------------------------

def _geometric(lam, h0, b, L):
    """z_t = lam^{t+1} h0 + b (1 - lam^{t+1}) / (1 - lam) for constant lam, b (per mode)."""
    t = np.arange(1, L + 1)[:, None]
    lt = lam[None, :] ** t
    return lt * h0[None, :] + b[None, :] * (1 - lt) / (1 - lam[None, :])


def test_rtu_degeneration_closed_form():
    """Zero amplitudes: d = c = 0, lambda_m = e^{-nu_m} e^{i theta_m} for every token."""
    B, L, D = 2, 300, 10
    M = D // 2
    inp = _samu_rand(B, L, D, seed=2, amps=False)
    r = rng0(3)
    bconst = r.standard_normal((B, M)) + 1j * r.standard_normal((B, M))
    w = np.empty((B, L, D))
    w[..., :M] = bconst.real[:, None, :]
    w[..., M:] = bconst.imag[:, None, :]
    inp["w"] = w
    out = oracle.samu_forward(**inp)
    lam = np.exp(-inp["nu"]) * np.exp(1j * inp["theta"])
    for b in range(B):
        h0 = inp["h0"][b, :, 0] + 1j * inp["h0"][b, :, 1]
        z = _geometric(lam, h0, bconst[b], L)
        np.testing.assert_allclose(_cplx(out["y"][b], M), z, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out["hT"][b, :, 0] + 1j * out["hT"][b, :, 1], z[-1], rtol=1e-12)
    # controls at zero amplitude
    np.testing.assert_array_equal(out["ctrl"][..., 2], 1.0)   # E = e^0
    np.testing.assert_array_equal(out["ctrl"][..., 3], 1.0)   # C = cos 0
    np.testing.assert_array_equal(out["ctrl"][..., 4], 0.0)   # S = sin 0


def test_rtu_degeneration_zero_controller_gradients():
    """At zero amplitudes the controller is inert: dx_sel, dw_phi, dw_r vanish exactly."""
    inp = _samu_rand(2, 40, 8, seed=4, amps=False, reset_p=0.1)
    r = rng0(5)
    g = oracle.samu_backward(**inp, dy=r.standard_normal((2, 40, 8)), dhT=r.standard_normal((2, 4, 2)))
    assert np.all(g["dx_sel"] == 0.0)
    assert np.all(g["dw_phi"] == 0.0)
    assert np.all(g["dw_r"] == 0.0)
    assert g["da_phi"] != 0.0 and g["da_r"] != 0.0   # the amplitude gradients do not vanish


def test_constant_tokens_closed_form():
    """x_sel = 0 for every token: s_phi = w_phi[D]/||w_phi|| (norm over all D+1 entries),
    so p, r, d, c and lambda are the same at every position."""
    B, L, D = 1, 257, 12
    M = D // 2
    inp = _samu_rand(B, L, D, seed=6)
    inp["x_sel"] = np.zeros((B, L, D))
    inp["a_phi"], inp["a_r"] = 0.9, -0.8
    r = rng0(7)
    bconst = r.standard_normal(M) + 1j * r.standard_normal(M)
    w = np.empty((B, L, D))
    w[..., :M] = bconst.real
    w[..., M:] = bconst.imag
    inp["w"] = w
    out = oracle.samu_forward(**inp)
    p = np.tanh(inp["w_phi"][D] / np.linalg.norm(inp["w_phi"]))
    rr = np.tanh(inp["w_r"][D] / np.linalg.norm(inp["w_r"]))
    d = np.tanh(0.9) / math.sqrt(M) * p
    c = np.tanh(-0.8) / math.sqrt(M) * rr / (1 + rr * rr)
    lam = np.exp(-inp["nu"] * np.exp(c)) * np.exp(1j * (inp["theta"] + d))
    h0 = inp["h0"][0, :, 0] + 1j * inp["h0"][0, :, 1]
    np.testing.assert_allclose(_cplx(out["y"][0], M), _geometric(lam, h0, bconst, L), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["ctrl"][0, :, 0], p, rtol=1e-14)
    np.testing.assert_allclose(out["ctrl"][0, :, 1], rr, rtol=1e-14)


@pytest.mark.parametrize("j", [0, 3, 7, 11])
def test_one_hot_token_controller(j):
    """A single token x_sel = s e_j: the projection picks w_hat[j] and the bias w_hat[D]."""
    D = 12
    M = D // 2
    inp = _samu_rand(1, 1, D, seed=8 + j)
    inp["x_sel"] = np.zeros((1, 1, D))
    inp["x_sel"][0, 0, j] = 1.7
    inp["a_phi"], inp["a_r"] = -0.6, 0.7
    out = oracle.samu_forward(**inp)
    nphi, nr = np.linalg.norm(inp["w_phi"]), np.linalg.norm(inp["w_r"])
    p = np.tanh((1.7 * inp["w_phi"][j] + inp["w_phi"][D]) / nphi)
    rr = np.tanh((1.7 * inp["w_r"][j] + inp["w_r"][D]) / nr)
    d = np.tanh(-0.6) / math.sqrt(M) * p
    c = np.tanh(0.7) / math.sqrt(M) * rr / (1 + rr ** 2)
    lam = np.exp(-inp["nu"] * np.exp(c) + 1j * (inp["theta"] + d))
    h0 = inp["h0"][0, :, 0] + 1j * inp["h0"][0, :, 1]
    b = inp["w"][0, 0, :M] + 1j * inp["w"][0, 0, M:]
    np.testing.assert_allclose(_cplx(out["y"][0, 0], M), lam * h0 + b, rtol=1e-13, atol=1e-14)


def test_reset_sets_state_to_write_and_does_not_leak():
    B, L, D = 2, 64, 8
    M = D // 2
    inp = _samu_rand(B, L, D, seed=9)
    reset = np.zeros((B, L), np.uint8)
    reset[0, 20] = 1
    reset[1, 0] = 1
    reset[1, 63] = 1
    inp["reset"] = reset
    out = oracle.samu_forward(**inp)
    for b, t in [(0, 20), (1, 0), (1, 63)]:
        np.testing.assert_array_equal(out["y"][b, t], inp["w"][b, t])   # z_t = b_t exactly
    # perturb everything strictly before the reset at (0, 20): outputs from t=20 on are identical
    pert = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    pert["x_sel"][0, :20] += 0.5
    pert["w"][0, :20] -= 0.25
    pert["h0"][0] += 1.0
    out2 = oracle.samu_forward(**pert)
    np.testing.assert_array_equal(out2["y"][0, 20:], out["y"][0, 20:])
    np.testing.assert_array_equal(out2["hT"][0], out["hT"][0])
    # backward mirror: cotangents at t >= 20 do not reach anything before the reset
    r = rng0(10)
    dy = r.standard_normal((B, L, D))
    g1 = oracle.samu_backward(**inp, dy=dy, dhT=None)
    dy2 = dy.copy()
    dy2[0, 20:] += 3.0
    g2 = oracle.samu_backward(**inp, dy=dy2, dhT=r.standard_normal((B, M, 2)) * 0.0)
    np.testing.assert_array_equal(g2["dw"][0, :20], g1["dw"][0, :20])
    np.testing.assert_array_equal(g2["dh0"][0], g1["dh0"][0])


def test_rotation_equivariance_of_writes():
    """With h0 = 0, rotating every write b_t by e^{i phi} rotates every output by e^{i phi}."""
    B, L, D = 1, 50, 8
    M = D // 2
    inp = _samu_rand(B, L, D, seed=11, h0=False, reset_p=0.05)
    out = oracle.samu_forward(**inp)
    phi = 0.7
    bc = _cplx(inp["w"], M) * np.exp(1j * phi)
    inp2 = dict(inp)
    inp2["w"] = np.concatenate([bc.real, bc.imag], axis=-1)
    out2 = oracle.samu_forward(**inp2)
    np.testing.assert_allclose(_cplx(out2["y"], M), _cplx(out["y"], M) * np.exp(1j * phi), rtol=1e-12, atol=1e-12)


def test_theta_periodicity():
    inp = _samu_rand(1, 40, 8, seed=12)
    out = oracle.samu_forward(**inp)
    inp2 = dict(inp)
    inp2["theta"] = inp["theta"] + 2 * math.pi
    np.testing.assert_allclose(oracle.samu_forward(**inp2)["y"], out["y"], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# Affine composition algebra: (l2,b2) o (l1,b1) = (l2 l1, l2 b1 + b2)
# ---------------------------------------------------------------------------

def _compose(s2, s1):
    return (s2[0] * s1[0], s2[0] * s1[1] + s2[1])


def test_composition_is_associative():
    r = rng0(13)
    T = [(r.standard_normal(50) + 1j * r.standard_normal(50), r.standard_normal(50) + 1j * r.standard_normal(50))
         for _ in range(3)]
    a = _compose(T[2], _compose(T[1], T[0]))
    b = _compose(_compose(T[2], T[1]), T[0])
    np.testing.assert_allclose(a[0], b[0], rtol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13, atol=1e-14)
    # and it is not commutative
    c = _compose(T[0], T[1])
    d = _compose(T[1], T[0])
    assert np.max(np.abs(c[1] - d[1])) > 1e-3


def _recover_steps(out, inp, M):
    """Per-step maps (lambda_t, b_t) recovered from the oracle's outputs: lambda_t = (z_t - b_t)/z_{t-1}."""
    z = _cplx(out["y"][0], M)
    b = _cplx(inp["w"][0], M)
    zprev = np.vstack([inp["h0"][0, :, 0] + 1j * inp["h0"][0, :, 1], z[:-1]])
    return (z - b) / zprev, b, zprev[0]


@pytest.mark.parametrize("K,G", [(1, 4), (3, 2), (32, 64), (7, 3)])
def test_chunked_and_grouped_prefix_equal_step_recurrence(K, G):
    """S_c = T_e o ... o T_s per chunk; Q_c = L_c o O_g with groups of G chunks
    (SAMU GPU page, section 05) reproduce the step-by-step states, L % K != 0 included."""
    L, D = 203, 6
    M = D // 2
    inp = _samu_rand(1, L, D, seed=14)
    out = oracle.samu_forward(**inp)
    lam, b, h0 = _recover_steps(out, inp, M)
    C = -(-L // K)
    ident = (np.ones(M, complex), np.zeros(M, complex))
    S = []
    for c in range(C):
        acc = ident
        for t in range(c * K, min(L, (c + 1) * K)):
            acc = _compose((lam[t], b[t]), acc)
        S.append(acc)
    nG = -(-C // G)
    U = []
    for g in range(nG):
        acc = ident
        for c in range(g * G, min(C, (g + 1) * G)):
            acc = _compose(S[c], acc)
        U.append(acc)
    z = _cplx(out["y"][0], M)
    for c in range(C):
        g = c // G
        Lc = ident
        for cc in range(g * G, c):
            Lc = _compose(S[cc], Lc)
        Og = ident
        for gg in range(g):
            Og = _compose(U[gg], Og)
        Q = _compose(Lc, Og)
        entry = Q[0] * h0 + Q[1]
        # replay the chunk from its entry state
        h = entry
        for t in range(c * K, min(L, (c + 1) * K)):
            h = lam[t] * h + b[t]
            np.testing.assert_allclose(h, z[t], rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------------------
# Finite differences for the SAMU adjoint
# ---------------------------------------------------------------------------

def _samu_loss(inp, G, GT):
    out = oracle.samu_forward(**inp)
    return float(np.sum(out["y"] * G) + np.sum(out["hT"] * GT))


FD_KEYS = ["x_sel", "w", "h0", "nu", "theta", "w_phi", "w_r", "a_phi", "a_r"]
GRAD_NAME = {"x_sel": "dx_sel", "w": "dw", "h0": "dh0", "nu": "dnu", "theta": "dtheta",
             "w_phi": "dw_phi", "w_r": "dw_r", "a_phi": "da_phi", "a_r": "da_r"}


@pytest.mark.parametrize("seed,reset_p", [(20, 0.0), (21, 0.15)])
def test_samu_backward_matches_finite_differences(seed, reset_p):
    B, L, D = 2, 23, 6
    M = D // 2
    inp = _samu_rand(B, L, D, seed=seed, reset_p=reset_p)
    inp["a_phi"], inp["a_r"] = 0.8, -0.9      # large amplitudes make the controller matter
    r = rng0(seed + 100)
    G = r.standard_normal((B, L, D))
    GT = r.standard_normal((B, M, 2))
    g = oracle.samu_backward(**inp, dy=G, dhT=GT)
    eps = 1e-6
    for key in FD_KEYS:
        base = inp[key]
        for trial in range(2):
            v = r.standard_normal(np.shape(base))
            plus = dict(inp)
            minus = dict(inp)
            if np.ndim(base) == 0:
                plus[key] = base + eps * float(v)
                minus[key] = base - eps * float(v)
                analytic = g[GRAD_NAME[key]] * float(v)
            else:
                plus[key] = base + eps * v
                minus[key] = base - eps * v
                analytic = float(np.sum(g[GRAD_NAME[key]] * v))
            fd = (_samu_loss(plus, G, GT) - _samu_loss(minus, G, GT)) / (2 * eps)
            assert abs(fd - analytic) <= 1e-6 * max(1.0, abs(fd)), (key, fd, analytic)


def test_samu_backward_per_element_finite_differences():
    """Element-wise check of a few entries of every gradient (catches compensating errors)."""
    B, L, D = 1, 9, 4
    M = D // 2
    inp = _samu_rand(B, L, D, seed=30, reset_p=0.0)
    inp["reset"] = np.zeros((B, L), np.uint8)
    inp["reset"][0, 4] = 1
    inp["a_phi"], inp["a_r"] = -0.7, 0.95
    r = rng0(31)
    G = r.standard_normal((B, L, D))
    GT = r.standard_normal((B, M, 2))
    g = oracle.samu_backward(**inp, dy=G, dhT=GT)
    eps = 1e-6
    for key in ["x_sel", "w", "h0", "nu", "theta", "w_phi", "w_r"]:
        arr = inp[key]
        for flat in r.choice(arr.size, size=min(6, arr.size), replace=False):
            plus = dict(inp)
            minus = dict(inp)
            a1 = arr.copy().ravel()
            a2 = arr.copy().ravel()
            a1[flat] += eps
            a2[flat] -= eps
            plus[key] = a1.reshape(arr.shape)
            minus[key] = a2.reshape(arr.shape)
            fd = (_samu_loss(plus, G, GT) - _samu_loss(minus, G, GT)) / (2 * eps)
            an = g[GRAD_NAME[key]].ravel()[flat]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (key, flat, fd, an)


# ---------------------------------------------------------------------------
# RG-LRU
# ---------------------------------------------------------------------------

def _rg_rand(B, L, D, seed, reset_p=0.0, h0=True):
    r = rng0(seed)
    sp = -np.log(r.uniform(0.9, 0.999, D)) / 8.0
    return dict(
        x=r.standard_normal((B, L, D)), lx=r.standard_normal((B, L, D)), la=r.standard_normal((B, L, D)),
        alpha=np.log(np.expm1(sp)),
        h0=0.3 * r.standard_normal((B, D)) if h0 else None,
        reset=(r.random((B, L)) < reset_p).astype(np.uint8) if reset_p > 0 else None,
    )


def test_rglru_constant_gates_closed_form():
    """Constant x, l^x, l^a per channel: a and b are constant and h is a geometric series."""
    B, L, D = 2, 200, 5
    inp = _rg_rand(B, L, D, seed=40)
    r = rng0(41)
    for k in ("x", "lx", "la"):
        inp[k] = np.broadcast_to(r.standard_normal((B, 1, D)), (B, L, D)).copy()
    out = oracle.rglru_forward(**inp)
    sp = np.logaddexp(0.0, inp["alpha"])                      # library softplus
    for b in range(B):
        a = np.exp(-8.0 * expit(inp["la"][b, 0]) * sp)
        bb = inp["x"][b, 0] * expit(inp["lx"][b, 0]) * np.sqrt(1 - a * a)
        t = np.arange(1, L + 1)[:, None]
        h = a ** t * inp["h0"][b] + bb * (1 - a ** t) / (1 - a)
        np.testing.assert_allclose(out["y"][b], h, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(out["hT"][b], h[-1], rtol=1e-12)


def test_rglru_reset_and_non_leakage():
    B, L, D = 1, 60, 4
    inp = _rg_rand(B, L, D, seed=42)
    reset = np.zeros((B, L), np.uint8)
    reset[0, [0, 25]] = 1
    inp["reset"] = reset
    out = oracle.rglru_forward(**inp)
    for t in (0, 25):   # a = 0 and the normaliser is 1 at a segment start
        np.testing.assert_allclose(out["y"][0, t], inp["x"][0, t] * expit(inp["lx"][0, t]), rtol=1e-15)
    pert = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    pert["x"][0, :25] += 1.0
    pert["la"][0, :25] -= 1.0
    out2 = oracle.rglru_forward(**pert)
    np.testing.assert_array_equal(out2["y"][0, 25:], out["y"][0, 25:])


def _rg_loss(inp, G, GT):
    out = oracle.rglru_forward(**inp)
    return float(np.sum(out["y"] * G) + np.sum(out["hT"] * GT))


@pytest.mark.parametrize("seed,reset_p", [(50, 0.0), (51, 0.2)])
def test_rglru_backward_matches_finite_differences(seed, reset_p):
    B, L, D = 2, 21, 3
    inp = _rg_rand(B, L, D, seed=seed, reset_p=reset_p)
    r = rng0(seed + 100)
    G = r.standard_normal((B, L, D))
    GT = r.standard_normal((B, D))
    g = oracle.rglru_backward(**inp, dy=G, dhT=GT)
    names = {"x": "dx", "lx": "dlx", "la": "dla", "alpha": "dalpha", "h0": "dh0"}
    eps = 1e-6
    for key, gname in names.items():
        for trial in range(2):
            v = r.standard_normal(inp[key].shape)
            plus = dict(inp)
            minus = dict(inp)
            plus[key] = inp[key] + eps * v
            minus[key] = inp[key] - eps * v
            fd = (_rg_loss(plus, G, GT) - _rg_loss(minus, G, GT)) / (2 * eps)
            an = float(np.sum(g[gname] * v))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (key, fd, an)


def test_rglru_sqrt_derivative_is_bounded():
    """Gates near a = 1 (u = 1 - a^2 -> 0): the normaliser derivative is capped, so the
    gate gradient stays finite (the cap value itself is not printed on the pages)."""
    B, L, D = 1, 4, 2
    inp = _rg_rand(B, L, D, seed=60)
    inp["la"][:] = -40.0          # sigmoid ~ 4e-18 -> a ~ 1 - 1e-19 -> u ~ 0
    g = oracle.rglru_backward(**inp, dy=np.ones((B, L, D)), dhT=None)
    assert np.all(np.isfinite(g["dla"])) and np.all(np.isfinite(g["dalpha"]))


# ---------------------------------------------------------------------------
# Decode step (one token of each sequence, carried state)
# ---------------------------------------------------------------------------

def test_decode_step_token_by_token_equals_forward():
    """The decode step applied token after token reproduces the forward over
    the sequence exactly (the same FP64 operations in the same order)."""
    B, L, D = 3, 17, 12
    inp = _samu_rand(B, L, D, seed=21, reset_p=0.1)
    ref = oracle.samu_forward(**inp)
    state = inp["h0"].copy()
    common = {k: inp[k] for k in ("nu", "theta", "w_phi", "w_r", "a_phi", "a_r")}
    for t in range(L):
        out = oracle.samu_decode_step(inp["x_sel"][:, t], inp["w"][:, t], state, inp["reset"][:, t], **common)
        np.testing.assert_array_equal(out["y"], ref["y"][:, t])
        np.testing.assert_array_equal(out["ctrl"], ref["ctrl"][:, t])
        state = out["state"]
    np.testing.assert_array_equal(state, ref["hT"])


def test_decode_step_zero_amplitudes_closed_form():
    """With a_phi = a_r = 0 the controller drops out (d = c = 0, E = 1): one
    step is z <- e^{-nu} e^{i theta} z + b, written out with numpy complex."""
    B, D = 4, 10
    M = D // 2
    inp = _samu_rand(B, 1, D, seed=22, amps=False)
    state = inp["h0"]
    out = oracle.samu_decode_step(inp["x_sel"][:, 0], inp["w"][:, 0], state, None,
                                  **{k: inp[k] for k in ("nu", "theta", "w_phi", "w_r", "a_phi", "a_r")})
    lam = np.exp(-inp["nu"]) * np.exp(1j * inp["theta"])
    z = lam[None, :] * (state[..., 0] + 1j * state[..., 1]) + _cplx(inp["w"][:, 0], M)
    np.testing.assert_allclose(_cplx(out["y"], M), z, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["state"][..., 0] + 1j * out["state"][..., 1], z, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# Closed-form chunk transition (SAMU GPU page, section 05, exact chunk closed form)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K,seed", [(1, 30), (16, 31), (32, 32), (61, 33)])
def test_chunk_closed_form_equals_forward_transition(K, seed):
    """With zero writes and h0 = 1 in every mode, the forward's final state over
    K tokens is the product of the K transitions; the closed form built from
    the controller's own E_t and d_t = tanh(a_phi) p_t / sqrt(M) must equal it."""
    D = 14
    M = D // 2
    inp = _samu_rand(1, K, D, seed=seed)
    inp["w"] = np.zeros_like(inp["w"])
    h0 = np.zeros((1, M, 2))
    h0[..., 0] = 1.0
    inp["h0"] = h0
    ref = oracle.samu_forward(**inp)
    ctrl = ref["ctrl"][0]
    E = ctrl[:, 2]
    d = math.tanh(inp["a_phi"]) / math.sqrt(M) * ctrl[:, 0]
    np.testing.assert_allclose(np.arctan2(ctrl[:, 4], ctrl[:, 3]), d, rtol=0, atol=1e-15)   # S, C are sin d, cos d
    P = oracle.samu_chunk_transition(inp["nu"], inp["theta"], E, d)
    hT = ref["hT"][0, :, 0] + 1j * ref["hT"][0, :, 1]
    np.testing.assert_allclose(P, hT, rtol=1e-12, atol=0)


def test_chunk_closed_form_reset_and_split():
    """A reset anywhere in the chunk zeroes its transition; and the closed form
    of a chunk is the product of the closed forms of its two halves."""
    r = rng0(34)
    M, K = 9, 32
    nu, theta = -np.log(r.uniform(0.9, 0.999, M)), r.uniform(0, 2 * math.pi, M)
    E, d = np.exp(r.uniform(-0.05, 0.05, K)), r.uniform(-0.05, 0.05, K)
    rs = np.zeros(K, np.uint8)
    rs[17] = 1
    assert not np.any(oracle.samu_chunk_transition(nu, theta, E, d, rs))
    whole = oracle.samu_chunk_transition(nu, theta, E, d)
    halves = (oracle.samu_chunk_transition(nu, theta, E[:11], d[:11])
              * oracle.samu_chunk_transition(nu, theta, E[11:], d[11:]))
    np.testing.assert_allclose(whole, halves, rtol=1e-13)


def test_chunk_closed_form_phase_needs_more_than_fp32():
    """Why the closed form is formed with the phase K theta in FP64: rounding
    K theta + D to FP32 (|K theta| up to 2 pi K) already moves the transition by
    more than the pages' 5e-6 output gate at K = 32, while rounding the FP64
    result lbar^K once to FP32 stays near FP32 precision."""
    K = 32
    theta = np.array([6.2831])                   # theta near 2 pi: the largest phase
    nu = np.array([1e-3])
    E, d = np.ones(K), np.full(K, 0.01)
    exact = oracle.samu_chunk_transition(nu, theta, E, d)
    phase32 = np.float32(np.float32(K) * np.float32(theta[0])) + np.float32(d.sum())
    fp32_phase = np.exp(-nu * E.sum()) * np.exp(1j * np.float64(phase32))
    lbarK = np.exp(-K * nu) * np.exp(1j * K * theta)
    once = np.complex64(lbarK) * np.exp(1j * d.sum())
    assert abs(fp32_phase - exact)[0] / abs(exact)[0] > 5e-6
    assert abs(once - exact)[0] / abs(exact)[0] < 2e-7


# ---------------------------------------------------------------------------
# RG-LRU block-diagonal gate projections (SAMU GPU page, sections 04 and 06;
# protocol page "RG-LRU 的固定方程")
# ---------------------------------------------------------------------------

def _proj_rand(B, L, D, seed, reset_p=0.0):
    r = rng0(seed)
    H, dk = 16, D // 16
    return dict(
        x=r.standard_normal((B, L, D)),
        w_x=r.standard_normal((H, dk, dk)) / math.sqrt(dk),
        b_x=0.1 * r.standard_normal(D),
        w_a=r.standard_normal((H, dk, dk)) / math.sqrt(dk),
        b_a=0.1 * r.standard_normal(D),
        alpha=np.log(np.expm1(-np.log(r.uniform(0.9, 0.999, D)) / 8.0)),
        h0=0.1 * r.standard_normal((B, D)),
        reset=(r.random((B, L)) < reset_p).astype(np.uint8) if reset_p > 0 else None,
    )


def test_gate_projection_is_a_dense_block_diagonal_product():
    """The projection equals x times the dense [D, D] matrix assembled by
    scipy's block_diag from the 16 blocks, plus the bias (an independent
    construction: no per-block indexing)."""
    from scipy.linalg import block_diag
    inp = _proj_rand(2, 7, 48, seed=60)
    dense = block_diag(*inp["w_x"])
    want = inp["x"] @ dense + inp["b_x"]
    np.testing.assert_allclose(oracle.rglru_gate_projection(inp["x"], inp["w_x"], inp["b_x"]), want,
                               rtol=1e-13, atol=1e-13)
    # block 0's outputs (channels 0..2) depend on its inputs 0..2 only
    base = oracle.rglru_gate_projection(inp["x"], inp["w_x"], inp["b_x"])
    pert2 = inp["x"].copy()
    pert2[..., 3:] = 0.0
    only0 = oracle.rglru_gate_projection(pert2, inp["w_x"], inp["b_x"])
    np.testing.assert_allclose(only0[..., :3], base[..., :3], rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("D,count", [(1024, 134_144), (2048, 530_432), (2560, 826_880)])
def test_rglru_mixer_parameter_count_matches_pages_table(D, count):
    """Two 16-block diagonal projections, two biases and alpha: the pages'
    RG-LRU mixer parameter counts (SAMU GPU page, section 06 table)."""
    from linear_recurrence_sequence_gb300 import synth
    dk = D // synth.PROJ_BLOCKS
    shapes = {"w_x": (16, dk, dk), "w_a": (16, dk, dk), "b_x": (D,), "b_a": (D,), "alpha": (D,)}
    assert sum(int(np.prod(s)) for s in shapes.values()) == count
    inp = synth.rglru_proj_inputs(1, 2, D, 0)
    for k, s in shapes.items():
        assert inp[k].shape == s, k


def _proj_loss(inp, G, GT):
    out = oracle.rglru_proj_forward(**inp)
    return float(np.sum(out["y"] * G) + np.sum(out["hT"] * GT))


@pytest.mark.parametrize("seed,reset_p", [(61, 0.0), (62, 0.15)])
def test_rglru_proj_backward_matches_finite_differences(seed, reset_p):
    B, L, D = 2, 13, 32
    inp = _proj_rand(B, L, D, seed=seed, reset_p=reset_p)
    r = rng0(seed + 100)
    G = r.standard_normal((B, L, D))
    GT = r.standard_normal((B, D))
    g = oracle.rglru_proj_backward(**inp, dy=G, dhT=GT)
    names = {"x": "dx", "w_x": "dw_x", "b_x": "db_x", "w_a": "dw_a", "b_a": "db_a", "alpha": "dalpha", "h0": "dh0"}
    eps = 1e-6
    for key, gname in names.items():
        for trial in range(2):
            v = r.standard_normal(inp[key].shape)
            plus = dict(inp)
            minus = dict(inp)
            plus[key] = inp[key] + eps * v
            minus[key] = inp[key] - eps * v
            fd = (_proj_loss(plus, G, GT) - _proj_loss(minus, G, GT)) / (2 * eps)
            an = float(np.sum(g[gname] * v))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (key, fd, an)
