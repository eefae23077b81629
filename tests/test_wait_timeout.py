"""The error path of the bounded device waits, on a GPU, without a hang or a
fault: a wait on an mbarrier that nothing arrives on gives up after a few
polls, sets the sticky error word, the host reads SSM_ERR_TIMEOUT once, and the
context stays usable for a normal forward afterwards."""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


@pytest.mark.parametrize("polls", [0, 1, 1000])
def test_wait_that_runs_out_is_reported_and_cleared(oracle, polls):
    S.check_device_errors()  # nothing pending before
    S.selftest_wait_timeout(polls)
    with pytest.raises(S.SsmError) as ei:
        S.check_device_errors()
    assert ei.value.status == S.Status.ERR_TIMEOUT
    S.check_device_errors()  # read once, then cleared

    # a normal forward afterwards runs and reports no error
    w = W.WORKLOADS[2].scaled(batch=1, seqlen=300, dim=32)
    inp = W.make_inputs(w)
    t = W.to_torch(inp, "cuda")
    y, _ = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"])
    torch.cuda.synchronize()
    S.check_device_errors()
    y_ref, _ = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                               None, None)
    yg = y.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(yg - y_ref)) / np.max(np.abs(y_ref)) <= 1e-5
