"""The allocation-free end-to-end entry point (``ssm_scan_fwd_host_static``).

It runs the same pieces, chained by the carried state, with the same kernels
as ``ssm_scan_fwd_host``, so on two calls in a row its outputs must equal that
entry point's bit for bit, and agree with the fp64 oracle within the parity
tolerances; it must not allocate device memory, and must refuse problems
larger than its fixed workspace.  The file is collected last, and passes alone
in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}
TOL_STATES = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def _f64(t):
    return t.float().numpy().astype(np.float64)


def _rel(a, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(a - ref)) / den) if den > 0 else float(np.max(np.abs(a)))


def _largest_seqlen_under_capacity(w):
    """The longest sequence whose workspace still fits the fixed array (the
    last 256-byte-aligned region then ends just below its end)."""
    cap = S.static_capacity()

    def need(L):
        return S.host_workspace_bytes(w.batch, L, w.dim, w.dstate, dtype=w.dtype, has_D=True,
                                      gate=w.gate, mask=w.mask is not None,
                                      chunk_len=w.chunk_len)
    lo, hi = 1, 1 << 22
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if need(mid) <= cap:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _near_capacity():
    w = W.WORKLOADS[2].scaled(batch=2, seqlen=64, dim=512)
    return w.scaled(seqlen=_largest_seqlen_under_capacity(w))


CASES = {
    "fp32-long-pieces": (W.WORKLOADS[2].scaled(batch=2, seqlen=3000, dim=64), True),
    "fp32-no-D": (W.WORKLOADS[2].scaled(batch=3, seqlen=1500, dim=32), False),
    "bf16-gate-mask-states": (W.WORKLOADS[4].scaled(batch=4, seqlen=700, dim=48), True),
    "fp32-workspace-at-capacity": (None, True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_matches_the_workspace_entry_and_the_oracle_on_two_calls(oracle, name):
    w, with_D = CASES[name]
    if w is None:
        w = _near_capacity()
    inp = W.make_inputs(w)
    if not with_D:
        inp["D"] = None
    if inp["valid_len"] is not None:
        inp["valid_len"] = np.array([700, 0, 333, 1], np.int32)
    t = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v)
         for k, v in W.to_torch(inp, "cpu").items()}
    cl = w.chunk_len
    need = S.host_workspace_bytes(w.batch, w.seqlen, w.dim, w.dstate, dtype=w.dtype,
                                  has_D=with_D, gate=w.gate, mask=w.mask is not None,
                                  chunk_len=cl)
    assert need <= S.static_capacity()
    y_ref, s_ref = S.scan_fwd_host(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                   t["valid_len"], chunk_len=cl)
    torch.cuda.synchronize()
    yo, so = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["z"], inp["valid_len"], chunk_len=cl)
    nch = (w.seqlen + cl - 1) // cl if cl else 0
    y = torch.empty_like(y_ref).pin_memory()
    st = torch.empty((w.batch, nch, w.dim, w.dstate), dtype=torch.float32).pin_memory() if cl else None
    S.scan_fwd_host_static(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["valid_len"], out=y, chunk_len=cl, out_states=st)
    torch.cuda.synchronize()  # the first call has done its set-up
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        y.fill_(float("nan"))
        if st is not None:
            st.fill_(float("nan"))
        S.scan_fwd_host_static(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                               t["valid_len"], out=y, chunk_len=cl, out_states=st)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), "differs from ssm_scan_fwd_host"
        assert _rel(_f64(y), yo) <= TOL[w.dtype]
        if st is not None:
            assert torch.equal(st, s_ref), "chunk states differ from ssm_scan_fwd_host"
            assert _rel(_f64(st), so) <= TOL_STATES
        if inp["valid_len"] is not None:
            for b, v in enumerate(inp["valid_len"]):
                assert torch.all(y[b, int(v):] == 0)
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
