"""RG-LRU real scan: CUDA path (through the C ABI) vs the FP64 oracle."""
import numpy as np
import pytest

from linear_recurrence_sequence_gb300 import synth
from parity import check_rglru, run_rglru_gpu, run_rglru_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


SMALL = {
    "ragged_B2_L50_D8": dict(B=2, L=50, D=8, seed=21, h0=True, resets=0.1),
    "D16_L33": dict(B=3, L=33, D=16, seed=22, h0=True, resets="none"),
    "single_token": dict(B=1, L=1, D=24, seed=23, h0=True, resets="none"),
    "partial_group_B2_L700_D1304": dict(B=2, L=700, D=1304, seed=24, h0=True, resets="segments"),
    "tile_edges_B1_L257_D72": dict(B=1, L=257, D=72, seed=27, h0=True, resets=0.01),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_rglru_small_cases(name, dev):
    kw = SMALL[name]
    inp = synth.rglru_inputs(kw["B"], kw["L"], kw["D"], kw["seed"], h0=kw["h0"], resets=kw["resets"])
    ref_f, ref_b = run_rglru_oracle(inp)
    fwd, bwd = run_rglru_gpu(inp, dev)
    check_rglru(inp, fwd, bwd, ref_f, ref_b, label=name)


def test_rglru_bf16_gradients(dev):
    inp = synth.rglru_inputs(2, 1000, 256, 25, h0=True, resets="segments")
    ref_f, ref_b = run_rglru_oracle(inp)
    fwd, bwd = run_rglru_gpu(inp, dev, grad_fp32=False)
    check_rglru(inp, fwd, bwd, ref_f, ref_b, grad_fp32=False, label="bf16_grads")


def test_rglru_run_to_run_bitwise(dev):
    import torch
    inp = synth.rglru_inputs(2, 3000, 512, 26, h0=True, resets="segments")
    f1, b1 = run_rglru_gpu(inp, dev)
    f2, b2 = run_rglru_gpu(inp, dev)
    for k in ("y", "y32", "hT"):
        assert torch.equal(f1[k], f2[k]), k
    for k in ("dx", "dlx", "dla", "dalpha", "dh0"):
        assert torch.equal(b1[k], b2[k]), k


@pytest.mark.parametrize("name", ["rglru_2k", "rglru_4k", "rglru_8k", "rglru_16k"])
def test_rglru_workloads(name, dev):
    inp = synth.WORKLOADS[name].make()
    ref_f, ref_b = run_rglru_oracle(inp)
    fwd, bwd = run_rglru_gpu(inp, dev)
    check_rglru(inp, fwd, bwd, ref_f, ref_b, label=name)
