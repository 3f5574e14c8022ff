"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the FP64 oracle on the same seeded inputs, and compare.

Tolerances (per element set):
  FP32 pre-cast outputs and final state     rel-L2 <= 1e-5
  BF16 outputs                              within 1 BF16 ulp of RNE(oracle) for every
                                            component >= 2^-6 of its state magnitude
                                            (see BF16_FLOOR_EXP)
  input and state gradients (FP32 run)      rel-L2 <= 1e-4
  parameter gradients                       rel-L2 <= 5e-4 (scalars: relative error)
"""
from __future__ import annotations

import numpy as np

import oracle
from linear_recurrence_sequence_gb300 import synth

TOL_OUT = 1e-5
TOL_GRAD = 1e-4
TOL_PARAM = 5e-4
TOL_BF16_GRAD = 8e-3     # rel-L2 of BF16-rounded gradients (quantisation alone is ~2e-3)


def rel_l2(gpu, ref) -> float:
    g = np.asarray(gpu, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    den = np.linalg.norm(r)
    num = np.linalg.norm(g - r)
    if den == 0.0:
        return float(num)
    return float(num / den)


def _ordered(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp_distance(gpu_bits, ref_f64):
    """Distance in BF16 ulps between the GPU's BF16 output and RNE(oracle)."""
    ref_bits = oracle.bf16_rne(np.asarray(ref_f64, dtype=np.float64))
    return np.abs(_ordered(gpu_bits) - _ordered(ref_bits))


# Components smaller than 2^BF16_FLOOR_EXP of their state magnitude are
# exempt from the per-element ulp check (they stay inside the rel-L2 checks).
# Reason: FP32 state arithmetic leaves an error relative to the typical state
# magnitude |z| of the mode (its RMS over time), amplified by the mode's memory
# 1/(1 - |lambda|) <= ~10^3 steps; simulating the recurrence with exactly
# rounded FP32 transitions gives up to ~3e-5 |z| at nu = 1e-3.  A component of
# magnitude >= |z|/64 has a BF16 ulp >= |z| 2^-14 ~ 6e-5 |z|, so above that
# floor one ulp is a real bound; below it a component can sit several of its
# own ulps away (or change sign).
BF16_FLOOR_EXP = -6


def bf16_ulp_report(gpu_bits, ref_f64, state_scale):
    """Returns (max distance over all elements, number of elements > 1 ulp,
    number of elements > 1 ulp whose oracle magnitude is at or above the floor)."""
    dist = bf16_ulp_distance(gpu_bits, ref_f64)
    ref = np.abs(np.asarray(ref_f64, dtype=np.float64))
    big = ref >= state_scale * 2.0 ** BF16_FLOOR_EXP
    return int(dist.max(initial=0)), int((dist > 1).sum()), int(((dist > 1) & big).sum())


def torch_bits(t):
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
def run_samu_oracle(inp):
    f64 = synth.bf16_bits_to_f64
    x, w, dy = f64(inp["x_sel"]), f64(inp["w"]), f64(inp["dy"])
    args = (x, w, inp["h0"], inp["reset"], inp["nu"], inp["theta"], inp["w_phi"], inp["w_r"],
            float(inp["a_phi"]), float(inp["a_r"]))
    fwd = oracle.samu_forward(*args)
    bwd = oracle.samu_backward(*args, dy, inp["dhT"])
    return fwd, bwd


def run_samu_gpu(inp, device, grad_fp32=True, dhT=True):
    import torch
    from linear_recurrence_sequence_gb300 import api
    t = api.samu_tensors_from_numpy(inp, device)
    fwd = api.samu_forward(t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"],
                           t["w_r"], t["a_phi"], t["a_r"], want_y32=True)
    bwd = api.samu_backward(t["dy"], t["dhT"] if dhT else None, t["x_sel"], t["w"], t["h0"], t["reset"],
                            t["nu"], t["theta"], t["w_phi"], t["w_r"], t["a_phi"], t["a_r"], fwd["saved"],
                            grad_fp32=grad_fp32)
    torch.cuda.synchronize(device)
    assert api.device_status(bwd["scratch"]) == 0
    return fwd, bwd


def samu_state_scale(y_ref, M):
    """RMS over time of |z| per (b, m): the typical state magnitude of the mode
    (the FP32 error scales with it, not with the momentary |z_t|), broadcast
    back onto the halves layout."""
    z2 = y_ref[..., :M] ** 2 + y_ref[..., M:] ** 2
    rms = np.sqrt(np.mean(z2, axis=1, keepdims=True))
    return np.broadcast_to(np.concatenate([rms, rms], axis=-1), y_ref.shape)


def check_samu(inp, fwd, bwd, ref_f, ref_b, grad_fp32=True, label=""):
    """Asserts every SAMU tolerance; returns the measured errors."""
    D = inp["D"]
    M = D // 2
    err = {}
    err["y32"] = rel_l2(fwd["y32"].cpu().numpy(), ref_f["y"])
    err["hT"] = rel_l2(fwd["hT"].cpu().numpy(), ref_f["hT"])
    mx, n_bad, n_bad_big = bf16_ulp_report(torch_bits(fwd["y"]), ref_f["y"], samu_state_scale(ref_f["y"], M))
    err["y_ulp_max"], err["y_ulp_gt1"], err["y_ulp_gt1_above_floor"] = mx, n_bad, n_bad_big
    for k in ("dx_sel", "dw"):
        err[k] = rel_l2(bwd[k].float().cpu().numpy(), ref_b[k])
    err["dh0"] = rel_l2(bwd["dh0"].cpu().numpy(), ref_b["dh0"])
    for k in ("dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r"):
        err[k] = rel_l2(bwd[k].cpu().numpy(), ref_b[k])
    msg = f"{label} errors: " + ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                                          for k, v in err.items())
    print(msg)
    assert err["y32"] <= TOL_OUT, msg
    assert err["hT"] <= TOL_OUT, msg
    assert err["y_ulp_gt1_above_floor"] == 0, msg
    gtol = TOL_GRAD if grad_fp32 else TOL_BF16_GRAD
    assert err["dx_sel"] <= gtol and err["dw"] <= gtol, msg
    assert err["dh0"] <= TOL_GRAD, msg
    for k in ("dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r"):
        assert err[k] <= TOL_PARAM, msg
    return err


# ---------------------------------------------------------------------------
def run_rglru_oracle(inp):
    f64 = synth.bf16_bits_to_f64
    x, lx, la, dy = f64(inp["x"]), f64(inp["lx"]), f64(inp["la"]), f64(inp["dy"])
    fwd = oracle.rglru_forward(x, lx, la, inp["alpha"], inp["h0"], inp["reset"])
    bwd = oracle.rglru_backward(x, lx, la, inp["alpha"], inp["h0"], inp["reset"], dy, inp["dhT"])
    return fwd, bwd


def run_rglru_gpu(inp, device, grad_fp32=True):
    import torch
    from linear_recurrence_sequence_gb300 import api
    t = api.rglru_tensors_from_numpy(inp, device)
    fwd = api.rglru_forward(t["x"], t["lx"], t["la"], t["alpha"], t["h0"], t["reset"], want_y32=True)
    bwd = api.rglru_backward(t["dy"], t["dhT"], t["x"], t["lx"], t["la"], t["alpha"], t["h0"], t["reset"],
                             fwd["saved"], grad_fp32=grad_fp32)
    torch.cuda.synchronize(device)
    assert api.device_status(bwd["scratch"]) == 0
    return fwd, bwd


def check_rglru(inp, fwd, bwd, ref_f, ref_b, grad_fp32=True, label=""):
    err = {}
    err["y32"] = rel_l2(fwd["y32"].cpu().numpy(), ref_f["y"])
    err["hT"] = rel_l2(fwd["hT"].cpu().numpy(), ref_f["hT"])
    # per (batch, channel) RMS over time as the magnitude scale of the state
    scale = np.broadcast_to(np.sqrt(np.mean(ref_f["y"] ** 2, axis=1, keepdims=True)), ref_f["y"].shape)
    mx, n_bad, n_bad_big = bf16_ulp_report(torch_bits(fwd["y"]), ref_f["y"], scale)
    err["y_ulp_max"], err["y_ulp_gt1"], err["y_ulp_gt1_above_floor"] = mx, n_bad, n_bad_big
    for k in ("dx", "dlx", "dla"):
        err[k] = rel_l2(bwd[k].float().cpu().numpy(), ref_b[k])
    err["dh0"] = rel_l2(bwd["dh0"].cpu().numpy(), ref_b["dh0"])
    err["dalpha"] = rel_l2(bwd["dalpha"].cpu().numpy(), ref_b["dalpha"])
    msg = f"{label} errors: " + ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                                          for k, v in err.items())
    print(msg)
    assert err["y32"] <= TOL_OUT, msg
    assert err["hT"] <= TOL_OUT, msg
    assert err["y_ulp_gt1_above_floor"] == 0, msg
    gtol = TOL_GRAD if grad_fp32 else TOL_BF16_GRAD
    for k in ("dx", "dlx", "dla"):
        assert err[k] <= gtol, msg
    assert err["dh0"] <= TOL_GRAD, msg
    assert err["dalpha"] <= TOL_PARAM, msg
    return err


# ---------------------------------------------------------------------------
# RG-LRU with its block-diagonal gate projections
# ---------------------------------------------------------------------------
def run_rglru_proj_oracle(inp):
    f64 = synth.bf16_bits_to_f64
    x, dy, w_x, w_a = f64(inp["x"]), f64(inp["dy"]), f64(inp["w_x"]), f64(inp["w_a"])
    args = (x, w_x, inp["b_x"], w_a, inp["b_a"], inp["alpha"], inp["h0"], inp["reset"])
    return oracle.rglru_proj_forward(*args), oracle.rglru_proj_backward(*args, dy, inp["dhT"])


def run_rglru_proj_gpu(inp, device, grad_fp32=True):
    import torch
    from linear_recurrence_sequence_gb300 import api
    t = api.rglru_proj_tensors_from_numpy(inp, device)
    p = (t["x"], t["w_x"], t["b_x"], t["w_a"], t["b_a"], t["alpha"], t["h0"], t["reset"])
    fwd = api.rglru_proj_forward(*p, want_y32=True)
    bwd = api.rglru_proj_backward(t["dy"], t["dhT"], *p, fwd["saved"], grad_fp32=grad_fp32)
    torch.cuda.synchronize(device)
    assert api.device_status(bwd["scratch"]) == 0
    return fwd, bwd


def check_rglru_proj(inp, fwd, bwd, ref_f, ref_b, grad_fp32=True, label=""):
    err = {}
    err["y32"] = rel_l2(fwd["y32"].cpu().numpy(), ref_f["y"])
    err["hT"] = rel_l2(fwd["hT"].cpu().numpy(), ref_f["hT"])
    scale = np.broadcast_to(np.sqrt(np.mean(ref_f["y"] ** 2, axis=1, keepdims=True)), ref_f["y"].shape)
    mx, n_bad, n_bad_big = bf16_ulp_report(torch_bits(fwd["y"]), ref_f["y"], scale)
    err["y_ulp_max"], err["y_ulp_gt1"], err["y_ulp_gt1_above_floor"] = mx, n_bad, n_bad_big
    err["dx"] = rel_l2(bwd["dx"].float().cpu().numpy(), ref_b["dx"])
    for k in ("dh0",):
        err[k] = rel_l2(bwd[k].cpu().numpy(), ref_b[k])
    for k in ("dw_x", "db_x", "dw_a", "db_a", "dalpha"):
        err[k] = rel_l2(bwd[k].cpu().numpy(), ref_b[k])
    msg = f"{label} errors: " + ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                                          for k, v in err.items())
    print(msg)
    assert err["y32"] <= TOL_OUT, msg
    assert err["hT"] <= TOL_OUT, msg
    assert err["y_ulp_gt1_above_floor"] == 0, msg
    assert err["dx"] <= (TOL_GRAD if grad_fp32 else TOL_BF16_GRAD), msg
    assert err["dh0"] <= TOL_GRAD, msg
    for k in ("dw_x", "db_x", "dw_a", "db_a", "dalpha"):
        assert err[k] <= TOL_PARAM, msg
    return err
