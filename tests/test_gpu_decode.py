"""SAMU single-token decode step: CUDA path (through the C ABI) vs the FP64
oracle on seeded inputs: one step from a random state, many steps carried on
the GPU against the oracle's forward over the whole sequence, resets, ragged
widths, and a width-2048 batch."""
import numpy as np
import pytest

import oracle
from linear_recurrence_sequence_gb300 import synth
from parity import TOL_OUT, bf16_ulp_report, rel_l2, torch_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def _tensors(inp, dev):
    from linear_recurrence_sequence_gb300 import api
    return api.samu_tensors_from_numpy(inp, dev)


def _params(t):
    from linear_recurrence_sequence_gb300 import api
    return api.samu_decode_prepare(t["nu"], t["theta"], t["w_phi"], t["w_r"], t["a_phi"], t["a_r"])


def _common(inp):
    return dict(nu=inp["nu"], theta=inp["theta"], w_phi=inp["w_phi"], w_r=inp["w_r"],
                a_phi=float(inp["a_phi"]), a_r=float(inp["a_r"]))


@pytest.mark.parametrize("B,D,reset_p,seed", [(64, 256, 0.0, 31), (48, 64, 0.25, 32), (5, 400, 0.2, 33),
                                              (3, 16, 0.0, 34), (7, 4096, 0.1, 37)])
def test_decode_single_step(B, D, reset_p, seed, dev):
    import torch
    from linear_recurrence_sequence_gb300 import api
    M = D // 2
    inp = synth.samu_inputs(B, 1, D, seed, h0=True, reset_p=reset_p)
    t = _tensors(inp, dev)
    params = _params(t)
    state = t["h0"].clone()
    reset = None if inp["reset"] is None else t["reset"][:, 0].contiguous()
    out = api.samu_decode_step(t["x_sel"][:, 0].contiguous(), t["w"][:, 0].contiguous(), state, params, reset,
                               want_y32=True)
    torch.cuda.synchronize(dev)
    f64 = synth.bf16_bits_to_f64
    ref = oracle.samu_decode_step(f64(inp["x_sel"])[:, 0], f64(inp["w"])[:, 0], inp["h0"],
                                  None if inp["reset"] is None else inp["reset"][:, 0], **_common(inp))
    e_y = rel_l2(out["y32"].cpu().numpy(), ref["y"])
    e_s = rel_l2(out["state"].cpu().numpy(), ref["state"])
    assert e_y <= TOL_OUT and e_s <= TOL_OUT, (e_y, e_s)
    mx, _, above = bf16_ulp_report(torch_bits(out["y"]), ref["y"], np.abs(ref["y"]).max(axis=0, keepdims=True))
    assert above == 0, mx


def test_decode_steps_carry_state_equal_forward(dev):
    """64 decode steps on the GPU (state updated in place) against the oracle
    forward over the 64-token sequences."""
    import torch
    from linear_recurrence_sequence_gb300 import api
    B, L, D = 8, 64, 512
    M = D // 2
    inp = synth.samu_inputs(B, L, D, 35, h0=True, reset_p=1 / 32)
    t = _tensors(inp, dev)
    params = _params(t)
    state = t["h0"].clone()
    ys = []
    for s in range(L):
        reset = None if inp["reset"] is None else t["reset"][:, s].contiguous()
        o = api.samu_decode_step(t["x_sel"][:, s].contiguous(), t["w"][:, s].contiguous(), state, params, reset,
                                 want_y32=True)
        ys.append(o["y32"])
    y32 = torch.stack(ys, dim=1)
    torch.cuda.synchronize(dev)
    f64 = synth.bf16_bits_to_f64
    ref = oracle.samu_forward(f64(inp["x_sel"]), f64(inp["w"]), inp["h0"], inp["reset"], **_common(inp))
    e_y = rel_l2(y32.cpu().numpy(), ref["y"])
    e_s = rel_l2(state.cpu().numpy(), ref["hT"])
    print(f"decode x{L}: y32 {e_y:.3g}  state {e_s:.3g}")
    assert e_y <= TOL_OUT and e_s <= TOL_OUT, (e_y, e_s)
    # the same sequences through the scan forward: both paths agree within the tolerance too
    fwd = api.samu_forward(t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
                           t["a_phi"], t["a_r"], want_y32=True)
    torch.cuda.synchronize(dev)
    assert rel_l2(y32.cpu().numpy(), fwd["y32"].cpu().numpy()) <= TOL_OUT


def test_decode_width_2048_batch(dev):
    import torch
    from linear_recurrence_sequence_gb300 import api
    B, D = 1024, 2048
    inp = synth.samu_inputs(B, 1, D, 36, h0=True, reset_p=0.01)
    t = _tensors(inp, dev)
    params = _params(t)
    state = t["h0"].clone()
    out_state = torch.empty_like(state)
    o = api.samu_decode_step(t["x_sel"][:, 0].contiguous(), t["w"][:, 0].contiguous(), state, params,
                             t["reset"][:, 0].contiguous(), state_out=out_state, want_y32=True)
    torch.cuda.synchronize(dev)
    f64 = synth.bf16_bits_to_f64
    ref = oracle.samu_decode_step(f64(inp["x_sel"])[:, 0], f64(inp["w"])[:, 0], inp["h0"], inp["reset"][:, 0],
                                  **_common(inp))
    assert rel_l2(o["y32"].cpu().numpy(), ref["y"]) <= TOL_OUT
    assert rel_l2(out_state.cpu().numpy(), ref["state"]) <= TOL_OUT
    # the input state was not touched when a separate output was given
    np.testing.assert_array_equal(state.cpu().numpy(), inp["h0"].astype(np.float32))
