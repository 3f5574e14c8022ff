"""SAMU mixer: CUDA path (through the C ABI) vs the FP64 oracle, element by element,
on seeded inputs of every measured workload plus ragged and degenerate shapes."""
import numpy as np
import pytest

from linear_recurrence_sequence_gb300 import synth
from parity import (check_samu, check_samu_bench_variant, run_samu_gpu, run_samu_gpu_graph,
                    run_samu_oracle, torch_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def _case(B, L, D, seed, h0=True, reset_p=0.0):
    return synth.samu_inputs(B, L, D, seed, h0=h0, reset_p=reset_p)


SMALL = {
    "tiny_B2_L2048_D256": dict(B=2, L=2048, D=256, seed=0, h0=True, reset_p=1 / 512),
    "ragged_B3_L77_D64": dict(B=3, L=77, D=64, seed=11, h0=True, reset_p=0.05),
    "single_token_B2_L1_D16": dict(B=2, L=1, D=16, seed=12, h0=True),
    "one_subchunk_plus_one_L17_D400": dict(B=1, L=17, D=400, seed=13, h0=True, reset_p=0.1),
    "one_tile_plus_one_L129_D96": dict(B=2, L=129, D=96, seed=20, h0=True, reset_p=0.02),
    "partial_group_B2_L300_D1552": dict(B=2, L=300, D=1552, seed=14, h0=True, reset_p=0.01),
    "many_chunks_B1_L5003_D32": dict(B=1, L=5003, D=32, seed=15, h0=True, reset_p=0.002),
    "widest_B1_L300_D4096": dict(B=1, L=300, D=4096, seed=17, h0=True, reset_p=0.01),
    "many_rows_B64_L40_D128": dict(B=64, L=40, D=128, seed=18, h0=True, reset_p=0.02),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_samu_small_cases(name, dev):
    inp = _case(**SMALL[name])
    ref_f, ref_b = run_samu_oracle(inp)
    fwd, bwd = run_samu_gpu(inp, dev, grad_fp32=True)
    check_samu(inp, fwd, bwd, ref_f, ref_b, grad_fp32=True, label=name)


def test_samu_bf16_gradients(dev):
    inp = _case(**SMALL["tiny_B2_L2048_D256"])
    ref_f, ref_b = run_samu_oracle(inp)
    fwd, bwd = run_samu_gpu(inp, dev, grad_fp32=False)
    check_samu(inp, fwd, bwd, ref_f, ref_b, grad_fp32=False, label="tiny_bf16_grads")


def test_samu_resets_at_ends_and_everywhere(dev):
    inp = _case(B=2, L=64, D=32, seed=16, h0=True)
    reset = np.zeros((2, 64), np.uint8)
    reset[0, 0] = 1
    reset[0, 63] = 1
    reset[1, :] = 1                     # every token starts a segment: y = w, dh0 = 0
    inp["reset"] = reset
    ref_f, ref_b = run_samu_oracle(inp)
    fwd, bwd = run_samu_gpu(inp, dev)
    check_samu(inp, fwd, bwd, ref_f, ref_b, label="resets")
    w32 = synth.bf16_bits_to_f32(inp["w"][1])
    np.testing.assert_array_equal(fwd["y32"][1].cpu().numpy(), w32)
    assert float(bwd["dh0"][1].abs().max()) == 0.0


def test_samu_no_dhT_no_h0(dev):
    inp = _case(B=2, L=333, D=64, seed=17, h0=False, reset_p=0.0)
    inp["dhT"] = None
    ref_f, ref_b = run_samu_oracle(inp)
    fwd, bwd = run_samu_gpu(inp, dev, dhT=False)
    check_samu(inp, fwd, bwd, ref_f, ref_b, label="no_dhT")


def test_samu_rtu_degeneration_exact_zeros(dev):
    """Zero amplitudes: the controller is inert, dx_sel and dw_phi, dw_r are exactly zero."""
    inp = synth.samu_inputs(1, 500, 64, 18, h0=True, reset_p=0.01, zero_amplitudes=True)
    ref_f, ref_b = run_samu_oracle(inp)
    fwd, bwd = run_samu_gpu(inp, dev)
    check_samu(inp, fwd, bwd, ref_f, ref_b, label="rtu")
    assert float(bwd["dx_sel"].abs().max()) == 0.0
    assert float(bwd["dw_phi"].abs().max()) == 0.0
    assert float(bwd["dw_r"].abs().max()) == 0.0


def test_samu_run_to_run_bitwise(dev):
    """Look-back entry states equal the serial chunk chain bit for bit, and every
    reduction has a fixed order, so two runs agree exactly."""
    import torch
    inp = _case(B=2, L=4096, D=512, seed=19, h0=True, reset_p=1 / 1000)
    f1, b1 = run_samu_gpu(inp, dev)
    f2, b2 = run_samu_gpu(inp, dev)
    for k in ("y", "y32", "hT"):
        assert torch.equal(f1[k], f2[k]), k
    for k in ("dx_sel", "dw", "dh0", "dnu", "dtheta", "dw_phi", "dw_r", "da_phi", "da_r"):
        assert torch.equal(b1[k], b2[k]), k


@pytest.fixture
def chained():
    """Item transitions by the running product instead of the closed form."""
    from linear_recurrence_sequence_gb300 import api
    api.samu_set_chunk_transition(api.LRS_TRANSITION_CHAINED)
    yield
    api.samu_set_chunk_transition(api.LRS_TRANSITION_CLOSED_FORM)


@pytest.mark.parametrize("name", ["tiny_B2_L2048_D256", "ragged_B3_L77_D64", "partial_group_B2_L300_D1552",
                                  "many_chunks_B1_L5003_D32"])
def test_samu_chained_item_transitions(name, dev, chained):
    from linear_recurrence_sequence_gb300 import api
    assert api.samu_get_chunk_transition() == api.LRS_TRANSITION_CHAINED
    inp = _case(**SMALL[name])
    ref_f, ref_b = run_samu_oracle(inp)
    fwd, bwd = run_samu_gpu(inp, dev, grad_fp32=True)
    check_samu(inp, fwd, bwd, ref_f, ref_b, grad_fp32=True, label=f"chained/{name}")


@pytest.mark.parametrize("form", ["closed_form", "chained"])
def test_samu_long_memory_modes(form, dev):
    """Modes that remember thousands of tokens (|lbar| up to 1 - 1e-4) and phases
    spread over [0, 2 pi): the item transitions' rounding accumulates over the
    longest chains here, in either form."""
    from linear_recurrence_sequence_gb300 import api
    inp = _case(B=1, L=8192, D=512, seed=23, h0=True)
    r = np.random.default_rng(123)
    M = 256
    inp["nu"] = (-np.log(r.uniform(0.999, 0.9999, M))).astype(np.float32)
    inp["theta"] = r.uniform(0, 2 * np.pi, M).astype(np.float32)
    kind = api.LRS_TRANSITION_CLOSED_FORM if form == "closed_form" else api.LRS_TRANSITION_CHAINED
    api.samu_set_chunk_transition(kind)
    try:
        ref_f, ref_b = run_samu_oracle(inp)
        fwd, bwd = run_samu_gpu(inp, dev, grad_fp32=True)
    finally:
        api.samu_set_chunk_transition(api.LRS_TRANSITION_CLOSED_FORM)
    check_samu(inp, fwd, bwd, ref_f, ref_b, grad_fp32=True, label=f"long_memory/{form}")


WORKLOADS = ["short", "length_8k", "length_32k", "length_64k", "length_128k",
             "width_1024", "width_1536", "width_2048", "width_2560", "medium_8k_2560"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_samu_workloads(name, dev):
    wl = synth.WORKLOADS[name]
    for seed in wl.seeds:
        inp = wl.make(seed)
        ref_f, ref_b = run_samu_oracle(inp)
        fwd, bwd = run_samu_gpu(inp, dev)
        check_samu(inp, fwd, bwd, ref_f, ref_b, label=f"{name}/seed{seed}")
        del ref_f, ref_b, fwd, bwd


# ---------------------------------------------------------------------------
# The kernel variants the benchmark times: the forward without the FP32
# pre-cast output (replay kernel without y32), BF16 gradients (the reverse
# replay writes dw through shared memory by TMA when M is a multiple of 64,
# with plain stores otherwise), the step replayed as a CUDA graph.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["width_2048", "length_128k"])
def test_samu_benchmarked_variants_full_size(name, dev):
    """B1 L32K D2048 is the benchmark's own workload; B1 L128K D1024 the longest
    chain.  BF16 y, dw and dx_sel are checked element by element against RNE
    of the FP64 oracle; y must equal, bit for bit, the y of a run that also
    writes the FP32 pre-cast output."""
    import torch
    wl = synth.WORKLOADS[name]
    inp = wl.make(wl.seeds[0])
    ref_f, ref_b = run_samu_oracle(inp)
    fo, go = run_samu_gpu_graph(inp, dev)
    check_samu_bench_variant(inp, fo, go, ref_f, ref_b, label=f"bench_variant/{name}")
    f32run, _ = run_samu_gpu(inp, dev, grad_fp32=True, want_y32=True)
    assert torch.equal(f32run["y"], fo["y"])
    assert torch.equal(f32run["hT"], fo["hT"])


BF16_PLAIN_STORE = {
    # M % 64 != 0: dw leaves the reverse replay through plain BF16 stores
    "bf16_partial_group_B2_L300_D1552": dict(B=2, L=300, D=1552, seed=14, h0=True, reset_p=0.01),
    "bf16_B1_L8192_D400": dict(B=1, L=8192, D=400, seed=41, h0=True, reset_p=1 / 4096),
    "bf16_ragged_B3_L77_D64": dict(B=3, L=77, D=64, seed=11, h0=True, reset_p=0.05),
    # M % 64 == 0 with a ragged tail and resets: the TMA store path
    "bf16_tma_B2_L1000_D256": dict(B=2, L=1000, D=256, seed=42, h0=True, reset_p=0.01),
}


@pytest.mark.parametrize("name", list(BF16_PLAIN_STORE))
def test_samu_bf16_gradient_variants(name, dev):
    inp = _case(**BF16_PLAIN_STORE[name])
    ref_f, ref_b = run_samu_oracle(inp)
    fo, go = run_samu_gpu_graph(inp, dev)
    check_samu_bench_variant(inp, fo, go, ref_f, ref_b, label=f"bf16_variant/{name}")


def test_samu_forward_without_y32_equals_with_y32(dev):
    """The two replay variants write the same BF16 y and hT bit for bit."""
    import torch
    inp = _case(**SMALL["partial_group_B2_L300_D1552"])
    a, _ = run_samu_gpu(inp, dev, want_y32=True)
    b, _ = run_samu_gpu(inp, dev, want_y32=False)
    assert b["y32"] is None
    assert torch.equal(a["y"], b["y"])
    assert torch.equal(a["hT"], b["hT"])
    np.testing.assert_array_equal(torch_bits(a["y"]), torch_bits(b["y"]))


@pytest.mark.parametrize("B,L,D", [(1, 32768, 2048), (1, 16384, 4096), (3, 5000, 1552)])
def test_samu_forward_bitwise_across_runs_at_streaming_sizes(B, L, D, dev):
    """Shapes whose controller forward refills its staging slots many times
    (several 16-token items per CTA, finalised by different warps): three
    forward calls give the same outputs bit for bit."""
    import torch
    from linear_recurrence_sequence_gb300 import api
    inp = synth.samu_inputs(B, L, D, 51, h0=True, reset_p=1 / 4096)
    t = api.samu_tensors_from_numpy(inp, dev)
    args = (t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"], t["a_phi"], t["a_r"])
    runs = [api.samu_forward(*args, want_y32=True) for _ in range(3)]
    torch.cuda.synchronize()
    for r in runs:
        assert api.device_status(r["scratch"]) == 0
    for r in runs[1:]:   # (the workspaces' alignment padding is never written, so only outputs are compared)
        assert torch.equal(r["y"], runs[0]["y"])
        assert torch.equal(r["y32"], runs[0]["y32"])
        assert torch.equal(r["hT"], runs[0]["hT"])
