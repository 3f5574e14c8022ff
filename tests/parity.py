"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the FP64 oracle on the same seeded inputs, and compare.

Tolerances (per element set):
  FP32 pre-cast outputs and final state     rel-L2 <= 1e-5
  BF16 outputs                              within 1 BF16 ulp of RNE(oracle) for every
                                            component >= 2^-6 of its state magnitude
                                            (see BF16_FLOOR_EXP); below that floor, within
                                            one BF16 ulp of the floor magnitude (absolute)
  input and state gradients (FP32 run)      rel-L2 <= 1e-4
  BF16 input gradients (dw, dx_sel)         element by element as the BF16 outputs, with
                                            the floor taken from the gradient's own scale
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


# Bound on the share of elements more than one BF16 ulp from RNE(oracle).  All
# of them must lie below the floor (checked separately).  Below the floor, a
# component of magnitude |v| is more than one of its own ulps (~|v| 2^-8) off
# only when |v| < 2^8 e, with e the FP32 error relative to the scale: about
# 1e-6 on these inputs (3e-5 for memories of 10^4 tokens), so for values
# spread like a Gaussian of that scale, a share of about 2^8 e (1e-3 at most)
# is expected.
BF16_GT1_SHARE_MAX = 1e-3


def bf16_ulp_of(mag):
    """One BF16 ulp at magnitude `mag` (float64 array, > 0): 2^(exponent - 7)."""
    mag = np.asarray(mag, dtype=np.float64)
    e = np.floor(np.log2(np.maximum(mag, np.finfo(np.float64).tiny)))
    return np.exp2(e - 7)


def bf16_elementwise(gpu_bits, ref_f64, scale):
    """Element-wise BF16 check against RNE(oracle).

    Every element with |oracle| >= scale 2^BF16_FLOOR_EXP must be within one
    BF16 ulp of RNE(oracle).  An element below that floor must be within one
    BF16 ulp at the floor magnitude of the oracle value (an absolute bound:
    FP32 state arithmetic leaves an error relative to the scale, not to the
    component).  Returns a dict of statistics; 'bad' counts the elements that
    break either rule."""
    ref = np.asarray(ref_f64, dtype=np.float64)
    dist = bf16_ulp_distance(gpu_bits, ref)
    floor = np.asarray(scale, dtype=np.float64) * 2.0 ** BF16_FLOOR_EXP
    below = np.abs(ref) < floor
    gpu = np.asarray(gpu_bits, dtype=np.uint16).astype(np.uint32) << 16
    gpu = gpu.view(np.float32).astype(np.float64)
    abs_ok = np.abs(gpu - ref) <= bf16_ulp_of(floor)
    gt1 = dist > 1
    bad = gt1 & (~below | ~abs_ok)
    n = ref.size
    return {"ulp_max": int(dist.max(initial=0)), "gt1": int(gt1.sum()),
            "gt1_share": float(gt1.sum()) / max(n, 1), "below_floor": int(below.sum()),
            "bad": int(bad.sum()), "n": int(n)}


def assert_bf16_elementwise(stats, what, msg=""):
    assert stats["bad"] == 0, f"{what}: {stats} {msg}"
    assert stats["gt1_share"] <= BF16_GT1_SHARE_MAX, f"{what}: {stats} {msg}"


def row_scale(ref_f64):
    """RMS over all of a batch row's elements (tokens and channels), broadcast
    back: the scale of a gradient whose FP32 error is absolute over the row
    (dx_sel: per-token controller scalars times the unit directions)."""
    r = np.asarray(ref_f64, dtype=np.float64)
    rms = np.sqrt(np.mean(r * r, axis=tuple(range(1, r.ndim)), keepdims=True))
    return np.broadcast_to(rms, r.shape)


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


def run_samu_gpu(inp, device, grad_fp32=True, dhT=True, want_y32=True):
    import torch
    from linear_recurrence_sequence_gb300 import api
    t = api.samu_tensors_from_numpy(inp, device)
    fwd = api.samu_forward(t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"],
                           t["w_r"], t["a_phi"], t["a_r"], want_y32=want_y32)
    bwd = api.samu_backward(t["dy"], t["dhT"] if dhT else None, t["x_sel"], t["w"], t["h0"], t["reset"],
                            t["nu"], t["theta"], t["w_phi"], t["w_r"], t["a_phi"], t["a_r"], fwd["saved"],
                            grad_fp32=grad_fp32)
    torch.cuda.synchronize(device)
    assert api.device_status(bwd["scratch"]) == 0
    return fwd, bwd


def run_samu_gpu_graph(inp, device, replays=2):
    """One forward + backward as the benchmark runs it: BF16 gradients, no
    FP32 pre-cast output, preallocated outputs and workspaces, the two calls
    captured once as a CUDA graph and replayed `replays` times (an L2-sized
    buffer cleared before each replay).  Returns the outputs of the last replay."""
    import torch
    from linear_recurrence_sequence_gb300 import api
    t = api.samu_tensors_from_numpy(inp, device)
    B, L, D = inp["B"], inp["L"], inp["D"]
    M = D // 2
    nsaved, nscratch = api.samu_workspace_bytes(B, L, D)
    saved = torch.empty(nsaved, dtype=torch.uint8, device=device)
    scratch = torch.empty(nscratch, dtype=torch.uint8, device=device)
    bf, f32 = torch.bfloat16, torch.float32
    fo = {"y": torch.empty((B, L, D), dtype=bf, device=device),
          "hT": torch.empty((B, M, 2), dtype=f32, device=device)}
    go = {"dx_sel": torch.empty((B, L, D), dtype=bf, device=device),
          "dw": torch.empty((B, L, D), dtype=bf, device=device),
          "dh0": torch.empty((B, M, 2), dtype=f32, device=device),
          "dnu": torch.empty((M,), dtype=f32, device=device), "dtheta": torch.empty((M,), dtype=f32, device=device),
          "dw_phi": torch.empty((D + 1,), dtype=f32, device=device),
          "dw_r": torch.empty((D + 1,), dtype=f32, device=device),
          "da_phi": torch.empty((1,), dtype=f32, device=device), "da_r": torch.empty((1,), dtype=f32, device=device)}

    def step():
        api.samu_forward(t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
                         t["a_phi"], t["a_r"], out=fo, saved=saved, scratch=scratch)
        api.samu_backward(t["dy"], t["dhT"], t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"],
                          t["w_phi"], t["w_r"], t["a_phi"], t["a_r"], saved, out=go, scratch=scratch)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    step()   # eager first call (per-device set-up happens outside the capture)
    torch.cuda.synchronize(device)
    cs = torch.cuda.Stream(device)
    cs.wait_stream(torch.cuda.current_stream(device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        step()
    for k in go.values():
        k.zero_()
    fo["y"].zero_()
    fo["hT"].zero_()
    for _ in range(replays):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize(device)
    assert api.device_status(scratch) == 0
    return fo, go


def samu_state_scale(y_ref, M):
    """RMS over time of |z| per (b, m): the typical state magnitude of the mode
    (the FP32 error scales with it, not with the momentary |z_t|), broadcast
    back onto the halves layout."""
    z2 = y_ref[..., :M] ** 2 + y_ref[..., M:] ** 2
    rms = np.sqrt(np.mean(z2, axis=1, keepdims=True))
    return np.broadcast_to(np.concatenate([rms, rms], axis=-1), y_ref.shape)


def check_samu_bench_variant(inp, fwd, bwd, ref_f, ref_b, label=""):
    """The benchmark's outputs: BF16 y, dw and dx_sel element by element
    (bf16_elementwise), FP32 dh0 and the parameter gradients by rel-L2."""
    M = inp["D"] // 2
    stats = {
        "y": bf16_elementwise(torch_bits(fwd["y"]), ref_f["y"], samu_state_scale(ref_f["y"], M)),
        "dw": bf16_elementwise(torch_bits(bwd["dw"]), ref_b["dw"], samu_state_scale(ref_b["dw"], M)),
        "dx_sel": bf16_elementwise(torch_bits(bwd["dx_sel"]), ref_b["dx_sel"], row_scale(ref_b["dx_sel"])),
    }
    err = {"hT": rel_l2(fwd["hT"].cpu().numpy(), ref_f["hT"]),
           "dh0": rel_l2(bwd["dh0"].cpu().numpy(), ref_b["dh0"])}
    for k in ("dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r"):
        err[k] = rel_l2(bwd[k].cpu().numpy(), ref_b[k])
    # whole-tensor rel-L2 of the BF16 tensors as well (quantisation ~2e-3)
    for k, v in (("y", fwd["y"]), ("dw", bwd["dw"]), ("dx_sel", bwd["dx_sel"])):
        err[f"{k}_rel_l2"] = rel_l2(v.float().cpu().numpy(), (ref_f if k == "y" else ref_b)[k])
    msg = f"{label}: " + ", ".join(f"{k}={v:.3g}" for k, v in err.items()) + " " + \
        "; ".join(f"{k} ulp_max={v['ulp_max']} gt1={v['gt1']} below_floor={v['below_floor']} of {v['n']}"
                  for k, v in stats.items())
    print(msg)
    for k, v in stats.items():
        assert_bf16_elementwise(v, k, msg)
    assert err["hT"] <= TOL_OUT, msg
    assert err["dh0"] <= TOL_GRAD, msg
    for k in ("dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r"):
        assert err[k] <= TOL_PARAM, msg
    for k in ("y", "dw", "dx_sel"):
        assert err[f"{k}_rel_l2"] <= TOL_BF16_GRAD, msg
    return err, stats


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
