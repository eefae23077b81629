"""The allocation-free end-to-end entry point (``ssm_scan_fwd_host_static``).

It must give the result of ``ssm_scan_fwd_host`` (the same pieces chained by
the carried state, the same kernels) on two calls in a row, within the
parity tolerances, without allocating device memory; and refuse problems
larger than its fixed workspace.  The file is collected last, and passes
alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def _rel(a, b):
    a, b = a.float().numpy().astype(np.float64), b.float().numpy().astype(np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


CASES = {
    "fp32-long-pieces": W.WORKLOADS[2].scaled(batch=2, seqlen=3000, dim=64),
    "bf16-gate-mask-states": W.WORKLOADS[4].scaled(batch=4, seqlen=700, dim=48),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_matches_the_workspace_entry_on_two_calls(name):
    w = CASES[name]
    inp = W.make_inputs(w)
    if inp["valid_len"] is not None:
        inp["valid_len"] = np.array([700, 0, 333, 1], np.int32)
    t = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v)
         for k, v in W.to_torch(inp, "cpu").items()}
    cl = w.chunk_len
    assert S.host_workspace_bytes(w.batch, w.seqlen, w.dim, w.dstate, dtype=w.dtype, gate=w.gate,
                                  mask=w.mask is not None, chunk_len=cl) <= S.static_capacity()
    y_ref, s_ref = S.scan_fwd_host(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                   t["valid_len"], chunk_len=cl)
    torch.cuda.synchronize()
    nch = (w.seqlen + cl - 1) // cl if cl else 0
    y = torch.empty_like(y_ref).pin_memory()
    st = torch.empty((w.batch, nch, w.dim, w.dstate), dtype=torch.float32).pin_memory() if cl else None
    S.scan_fwd_host_static(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["valid_len"], out=y, chunk_len=cl, out_states=st)
    torch.cuda.synchronize()  # the first call has done its set-up
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        y.zero_()
        if st is not None:
            st.zero_()
        S.scan_fwd_host_static(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                               t["valid_len"], out=y, chunk_len=cl, out_states=st)
        torch.cuda.synchronize()
        assert _rel(y, y_ref) <= TOL[w.dtype]
        if st is not None:
            assert _rel(st, s_ref) <= 1e-5
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "the call allocated device memory"


def test_oversize_is_refused():
    cap = S.static_capacity()
    dim = 1024
    L = cap // (2 * dim * 4) + 64  # x alone ([2, L, dim] fp32) exceeds the workspace
    x = torch.zeros((2, L, dim), dtype=torch.float32)
    Bm = torch.zeros((2, L, 16), dtype=torch.float32)
    A = torch.zeros((dim, 16), dtype=torch.float32)
    y = torch.empty_like(x)
    with pytest.raises(S.SsmError) as ei:
        S.scan_fwd_host_static(x, x, A, Bm, Bm, out=y)
    assert ei.value.status == S.Status.ERR_SHAPE
