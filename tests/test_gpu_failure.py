"""Failure detection without a GPU fault: a bounded device-side wait that runs
out (an mbarrier that nothing completes) reports LRS_ERR_TIMEOUT through the
status word, and the context stays usable for the next call."""
import pytest

from linear_recurrence_sequence_gb300 import synth
from parity import TOL_OUT, rel_l2, run_samu_oracle

pytestmark = pytest.mark.gpu

LRS_ERR_TIMEOUT = 4


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    from linear_recurrence_sequence_gb300 import api
    dev = torch.device("cuda:0")
    inp = synth.samu_inputs(1, 64, 32, 90, h0=True)
    t = api.samu_tensors_from_numpy(inp, dev)
    _, nscratch = api.samu_workspace_bytes(1, 64, 32)
    scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    api.selftest_wait_timeout(scratch)
    assert api.device_status(scratch) == LRS_ERR_TIMEOUT
    # the next call clears the word and runs normally on the same context
    fwd = api.samu_forward(t["x_sel"], t["w"], t["h0"], t["reset"], t["nu"], t["theta"], t["w_phi"], t["w_r"],
                           t["a_phi"], t["a_r"], want_y32=True, scratch=scratch)
    torch.cuda.synchronize(dev)
    assert api.device_status(scratch) == 0
    ref_f, _ = run_samu_oracle(inp)
    assert rel_l2(fwd["y32"].cpu().numpy(), ref_f["y"]) <= TOL_OUT
