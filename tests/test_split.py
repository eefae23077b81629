"""The time split of the forward (``ssm_scan_fwd_split``): aggregate pass,
carry between segments, output pass.  Its outputs must match the fp64 oracle
of the unsplit sequence within the parity tolerances for any segment count,
including masks that end inside, at the edge of, or before a segment, chunk
states that straddle segments, an initial state, and the bf16 gated form."""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_Y = {"f32": 1e-5, "bf16": 1e-2}
TOL_STATES = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def _rel(a, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(a - ref)) / den) if den > 0 else float(np.max(np.abs(a)))


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _case(batch, L, dim, N, dtype="f32", gate=False, mask=None, chunk=0, h0=False, seed=5):
    w = W.Workload(0, "split", batch, L, dim, N, dtype, "loguniform", "s4d", "normal", gate, None,
                   chunk, seed)
    inp = W.make_inputs(w)
    if mask is not None:
        inp["valid_len"] = np.array(mask, np.int32)
    h = np.random.default_rng(seed).standard_normal((batch, dim, N)).astype(np.float32) if h0 else None
    return w, inp, h


CASES = {
    "f32-n16": dict(batch=2, L=3000, dim=32, N=16),
    "f32-n16-mask-chunks": dict(batch=6, L=3000, dim=32, N=16, mask=[0, 100, 1024, 2999, 3000, 5000],
                                chunk=100),
    "bf16-gate-h0-chunks": dict(batch=3, L=2100, dim=48, N=16, dtype="bf16", gate=True, chunk=256,
                                h0=True, mask=[2100, 700, 1300]),
    "f32-n64-h0": dict(batch=1, L=1500, dim=8, N=64, h0=True),
    "f32-n4": dict(batch=2, L=1000, dim=64, N=4, chunk=64),
    "f32-n32-ragged": dict(batch=1, L=777, dim=40, N=32, chunk=333),
}


@pytest.mark.parametrize("segments", [1, 2, 3, 7, 0])
@pytest.mark.parametrize("name", sorted(CASES))
def test_split_matches_oracle(oracle, name, segments):
    w, inp, h0 = _case(**CASES[name])
    t = W.to_torch(inp, "cuda")
    h0t = torch.from_numpy(h0).cuda() if h0 is not None else None
    y, s, fin = S.scan_fwd_split(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                 t["valid_len"], time_segments=segments, chunk_len=w.chunk_len,
                                 h0=h0t, want_final=True)
    torch.cuda.synchronize()
    S.check_device_errors()
    y_ref, s_ref, f_ref = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                          inp["D"], inp["z"], inp["valid_len"],
                                          chunk_len=w.chunk_len, h0=h0, want_final=True)
    yg = _f64(y)
    assert _rel(yg, y_ref) <= TOL_Y[w.dtype]
    if s is not None:
        assert _rel(_f64(s), s_ref) <= TOL_STATES
    assert _rel(_f64(fin), f_ref) <= TOL_STATES
    if inp["valid_len"] is not None:
        for b, v in enumerate(inp["valid_len"]):
            v = min(max(int(v), 0), w.seqlen)
            assert np.all(yg[b, v:] == 0)


def test_plan_segments_and_workspace():
    segs, nbytes = S.split_plan(2, 3000, 32, 16, time_segments=7)
    assert segs == 7 and nbytes >= 2 * 2 * 7 * 32 * 16 * 4 + 2 * 7 * 32 * 4
    segs, nbytes = S.split_plan(2, 3000, 32, 16, time_segments=1000)  # clamped to whole tiles
    assert segs == (3000 + 63) // 64
    segs, nbytes = S.split_plan(8, 4096, 1024, 16, time_segments=1)
    assert (segs, nbytes) == (1, 0)


def test_split_argument_errors():
    w, inp, _ = _case(batch=1, L=640, dim=32, N=16)
    t = W.to_torch(inp, "cuda")
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(S.SsmError) as ei:
        S.scan_fwd_split(t["x"], t["delta"], t["A"], t["B"], t["C"], time_segments=4, workspace=small)
    assert ei.value.status == S.Status.ERR_SHAPE
    w1, inp1, _ = _case(batch=1, L=640, dim=32, N=1)  # no STREAM instance for one state
    t1 = W.to_torch(inp1, "cuda")
    with pytest.raises(S.SsmError) as ei:
        S.scan_fwd_split(t1["x"], t1["delta"], t1["A"], t1["B"], t1["C"], time_segments=2)
    assert ei.value.status == S.Status.ERR_UNSUPPORTED


def test_scan_fwd_routes_few_channel_rows_through_the_split(oracle):
    """scan_fwd with the library's choice of tier takes the time split when the
    rows leave the GPU mostly idle, and the result is the oracle's."""
    w, inp, _ = _case(batch=1, L=8192, dim=64, N=16, chunk=512, mask=[7000])
    segs, _ = S.split_plan(w.batch, w.seqlen, w.dim, w.dstate)
    assert segs > 1
    t = W.to_torch(inp, "cuda")
    y, s = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], None, t["valid_len"],
                      chunk_len=w.chunk_len)
    y1, s1 = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], None, t["valid_len"],
                        chunk_len=w.chunk_len, time_segments=1)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   None, inp["valid_len"], chunk_len=w.chunk_len)
    for yy, ss in ((y, s), (y1, s1)):
        assert _rel(_f64(yy), y_ref) <= 1e-5 and _rel(_f64(ss), s_ref) <= 1e-5


@pytest.mark.parametrize("key", sorted(W.SPLIT_WORKLOADS))
def test_split_full_size_whole_tensor(oracle, key):
    """The split workloads at full size through scan_fwd (which takes the time
    split for them), whole y and final state against the oracle."""
    w = W.SPLIT_WORKLOADS[key]
    inp = W.make_inputs(w)
    segs, _ = S.split_plan(w.batch, w.seqlen, w.dim, w.dstate)
    assert segs > 1
    t = W.to_torch(inp, "cuda")
    y, _, fin = S.scan_fwd_split(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                 t["valid_len"], time_segments=0, want_final=True)
    torch.cuda.synchronize()
    S.check_device_errors()
    yg, fg = _f64(y), _f64(fin)
    del y, fin, t
    y_ref, _, f_ref = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                      inp["D"], inp["z"], inp["valid_len"], want_final=True)
    assert _rel(yg, y_ref) <= TOL_Y[w.dtype]
    assert _rel(fg, f_ref) <= TOL_STATES
