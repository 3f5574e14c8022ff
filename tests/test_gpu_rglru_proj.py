"""RG-LRU mixer with its two 16-block block-diagonal gate projections: CUDA
path (tcgen05 contraction kernels + the FP32-logit scan, through the C ABI) vs the
FP64 oracle (numpy projections + the oracle scan), element by element."""
import pytest

from linear_recurrence_sequence_gb300 import synth
from parity import check_rglru_proj, run_rglru_proj_gpu, run_rglru_proj_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


SMALL = {
    "D128_L300_resets": dict(B=2, L=300, D=128, seed=70, h0=True, resets=0.02),
    "D256_L1000_segments": dict(B=2, L=1000, D=256, seed=71, h0=True, resets="segments"),
    "D1024_L129_tile_edge": dict(B=1, L=129, D=1024, seed=72, h0=False, resets="none"),
    "D2048_L200": dict(B=1, L=200, D=2048, seed=73, h0=True, resets="segments"),
    "single_token_D128": dict(B=3, L=1, D=128, seed=74, h0=True, resets="none"),
    "D512_L513_resets": dict(B=2, L=513, D=512, seed=77, h0=True, resets=0.01),
    "D1536_L140_gemm_path": dict(B=1, L=140, D=1536, seed=78, h0=True, resets="none"),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_rglru_proj_small_cases(name, dev):
    kw = SMALL[name]
    inp = synth.rglru_proj_inputs(kw["B"], kw["L"], kw["D"], kw["seed"], h0=kw["h0"], resets=kw["resets"])
    ref_f, ref_b = run_rglru_proj_oracle(inp)
    fwd, bwd = run_rglru_proj_gpu(inp, dev)
    check_rglru_proj(inp, fwd, bwd, ref_f, ref_b, label=name)


def test_rglru_proj_bf16_dx(dev):
    inp = synth.rglru_proj_inputs(2, 700, 256, 75, h0=True, resets="segments")
    ref_f, ref_b = run_rglru_proj_oracle(inp)
    fwd, bwd = run_rglru_proj_gpu(inp, dev, grad_fp32=False)
    check_rglru_proj(inp, fwd, bwd, ref_f, ref_b, grad_fp32=False, label="bf16_dx")


def test_rglru_proj_run_to_run_bitwise(dev):
    import torch
    inp = synth.rglru_proj_inputs(2, 2000, 512, 76, h0=True, resets="segments")
    f1, b1 = run_rglru_proj_gpu(inp, dev)
    f2, b2 = run_rglru_proj_gpu(inp, dev)
    for k in ("y", "y32", "hT"):
        assert torch.equal(f1[k], f2[k]), k
    for k in ("dx", "dw_x", "db_x", "dw_a", "db_a", "dalpha", "dh0"):
        assert torch.equal(b1[k], b2[k]), k


@pytest.mark.parametrize("name", ["rglru_proj_8k"])
def test_rglru_proj_workloads(name, dev):
    inp = synth.WORKLOADS[name].make()
    ref_f, ref_b = run_rglru_proj_oracle(inp)
    fwd, bwd = run_rglru_proj_gpu(inp, dev)
    check_rglru_proj(inp, fwd, bwd, ref_f, ref_b, label=name)
