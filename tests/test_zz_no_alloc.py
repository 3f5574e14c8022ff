"""samu_forward_noalloc: the SAMU forward for callers that cannot allocate.

Callers such as an application whose device memory belongs to its own pooled
allocator, or a latency-critical loop that must not take cudaMalloc's implicit
synchronisation, cannot hand the library a `saved`/`scratch` buffer.  This
entry point keeps every intermediate in one fixed device array inside the
library instead.  These tests call it through the C ABI and check, on calls in
a row with different inputs, that it reproduces the allocating samu_forward
within the tolerances the parity suite uses (at B=1, L=32768, D=2048 too),
that its status word can be read back (a bounded wait that gives up on the
fixed array is reported, and the next call clears it), and that a problem too
large for the fixed array is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest

from linear_recurrence_sequence_gb300 import synth
from parity import TOL_OUT, bf16_ulp_distance, rel_l2, torch_bits

pytestmark = pytest.mark.gpu

LRS_ERR_TOO_LARGE = 5


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def _forward_both(api, t, noalloc_calls=1):
    args = (t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
            t["a_phi"], t["a_r"])
    ref = api.samu_forward(*args, want_y32=True)
    outs = [api.samu_forward_noalloc(*args, want_y32=True) for _ in range(noalloc_calls)]
    return ref, outs


def _check_close(ref, out):
    import torch
    torch.cuda.synchronize()
    assert rel_l2(out["y32"].cpu().numpy(), ref["y32"].cpu().numpy()) <= TOL_OUT
    assert rel_l2(out["hT"].cpu().numpy(), ref["hT"].cpu().numpy()) <= TOL_OUT
    # BF16 outputs within one BF16 ulp of the allocating path's
    ref_y = ref["y"].float().cpu().numpy().astype(np.float64)
    assert int(bf16_ulp_distance(torch_bits(out["y"]), ref_y).max(initial=0)) <= 1


def test_noalloc_forward_matches_samu_forward_on_calls_in_a_row(dev):
    from linear_recurrence_sequence_gb300 import api
    cases = [
        synth.samu_inputs(2, 2048, 256, 0, h0=True, reset_p=1 / 512),
        synth.samu_inputs(1, 5003, 96, 31, h0=False, reset_p=0.0),
        synth.samu_inputs(1, 8192, 1024, 32, h0=True, reset_p=1 / 4096),
    ]
    for inp in cases:
        t = api.samu_tensors_from_numpy(inp, dev)
        ref, outs = _forward_both(api, t, noalloc_calls=2)
        for out in outs:
            _check_close(ref, out)


def test_noalloc_forward_at_the_benchmark_shape(dev):
    """B=1, L=32768, D=2048 (about 52 MiB of intermediates) fits the array."""
    from linear_recurrence_sequence_gb300 import api
    inp = synth.WORKLOADS["width_2048"].make(0)
    t = api.samu_tensors_from_numpy(inp, dev)
    ref, outs = _forward_both(api, t, noalloc_calls=2)
    for out in outs:
        _check_close(ref, out)
    assert api.samu_forward_noalloc_status(dev) == 0


def test_noalloc_forward_without_y32_matches_bitwise(dev):
    """Without the FP32 pre-cast output both paths run the same replay kernel:
    BF16 y and hT agree bit for bit."""
    import torch
    from linear_recurrence_sequence_gb300 import api
    inp = synth.samu_inputs(1, 4099, 512, 33, h0=True, reset_p=1 / 1024)
    t = api.samu_tensors_from_numpy(inp, dev)
    args = (t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
            t["a_phi"], t["a_r"])
    ref = api.samu_forward(*args, want_y32=False)
    for _ in range(2):
        out = api.samu_forward_noalloc(*args, want_y32=False)
        torch.cuda.synchronize()
        assert out["y32"] is None
        assert torch.equal(out["y"], ref["y"])
        assert torch.equal(out["hT"], ref["hT"])
    assert api.samu_forward_noalloc_status(dev) == 0


def test_noalloc_status_reports_a_wait_that_gave_up(dev):
    """The library's failure-path self-test on the fixed array's status word
    (a bounded wait on a barrier that nothing completes) is reported as
    LRS_ERR_TIMEOUT; the next call clears the word and computes normally."""
    from linear_recurrence_sequence_gb300 import api
    LRS_ERR_TIMEOUT = 4
    inp = synth.samu_inputs(2, 1000, 128, 34, h0=True, reset_p=0.01)
    t = api.samu_tensors_from_numpy(inp, dev)
    ref, outs = _forward_both(api, t)   # sets the array up in this context
    api.selftest_wait_timeout(None, dev)
    assert api.samu_forward_noalloc_status(dev) == LRS_ERR_TIMEOUT
    ref, outs = _forward_both(api, t)
    assert api.samu_forward_noalloc_status(dev) == 0
    _check_close(ref, outs[0])


def test_noalloc_forward_refuses_problems_beyond_its_workspace(dev):
    from linear_recurrence_sequence_gb300 import api
    import torch
    lib = api._load()
    buf = torch.zeros(1024, dtype=torch.float32, device=dev)
    p = ctypes.c_void_p(buf.data_ptr())
    # B=1, L=131072, D=2048 needs ~170 MiB of intermediates: refused before any launch
    st = lib.samu_forward_noalloc(p, p, None, None, p, p, p, p, p, p, 1, 131072, 2048,
                                  p, None, p, ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == LRS_ERR_TOO_LARGE
    assert b"no-allocation" in lib.lrs_status_string(st)
