"""The carried-state form of the forward (``ssm_scan_fwd_carry``) on a GPU.

The state before the first step may be given (h0) and the state after the last
step returned; a sequence scanned in two pieces, the second starting from the
first's final state, gives the whole sequence's result.  This is the serial
carry between sequence chunks of [P1] s3.1 (third level) and [P2] s2.4,
checked here against the fp64 oracle's own h0 / final-state output.
Tolerances as in test_parity: fp32 y 1e-5, bf16 y 1e-2, fp32 states 1e-5,
max-normalised.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

from test_parity import TIERS, TOL_STATES, TOL_Y, _edge, _tier, rel_err, tier_supported, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def _h0(batch, dim, n, seed=3):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((batch, dim, n)).astype(np.float32)


def _gpu(inp, kernel, h0):
    t = W.to_torch(inp, "cuda")
    k, shape = _tier(kernel)
    h = None if h0 is None else torch.from_numpy(h0).cuda()
    y, s, f = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                         t["valid_len"], chunk_len=inp["chunk_len"], kernel=k, h0=h,
                         want_final=True, **shape)
    torch.cuda.synchronize()
    return to_f64(y), (to_f64(s) if s is not None else None), to_f64(f)


CASES = {
    "fp32-mask-gate-states": dict(batch=4, L=513, dim=37, N=16, gate=True, mask=[513, 0, 200, 1],
                                  chunk=100),
    "bf16-n8": dict(batch=2, L=300, dim=64, N=8, dtype="bf16", chunk=64),
    "fp32-n64-ragged": dict(batch=1, L=517, dim=40, N=64, chunk=128),
    "fp32-n32-L1": dict(batch=3, L=1, dim=32, N=32),
}


@pytest.mark.parametrize("kernel", TIERS)
@pytest.mark.parametrize("name", sorted(CASES))
def test_h0_and_final_state(oracle, name, kernel):
    inp = _edge(**CASES[name])
    if not tier_supported(inp, kernel):
        pytest.skip(f"{kernel} does not take this shape")
    Bt, L, Dm = inp["x"].shape
    h0 = _h0(Bt, Dm, inp["B"].shape[-1])
    y_ref, s_ref, f_ref = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                          inp["D"], inp["z"], inp["valid_len"],
                                          chunk_len=inp["chunk_len"], h0=h0, want_final=True)
    y, s, f = _gpu(inp, kernel, h0)
    e = rel_err(y, y_ref)
    assert e <= TOL_Y[inp["dtype"]], f"y rel err {e:.3e}"
    if s_ref is not None:
        assert rel_err(s, s_ref) <= TOL_STATES
    assert rel_err(f, f_ref) <= TOL_STATES, f"final-state rel err {rel_err(f, f_ref):.3e}"
    if inp["valid_len"] is not None:
        for b, v in enumerate(inp["valid_len"]):
            v = min(max(int(v), 0), L)
            assert np.all(y[b, v:] == 0)
            if v == 0:  # no valid step: the final state is h0 itself
                assert np.array_equal(f[b], h0[b].astype(np.float64))


def _piece(inp, t0, t1):
    out = dict(inp)
    for k in ("x", "delta", "B", "C", "z"):
        if inp[k] is not None:
            out[k] = np.ascontiguousarray(inp[k][:, t0:t1])
    if inp["valid_len"] is not None:
        out["valid_len"] = np.clip(inp["valid_len"].astype(np.int64) - t0, 0,
                                   t1 - t0).astype(np.int32)
    out["chunk_len"] = 0
    return out


@pytest.mark.parametrize("kernel", TIERS)
@pytest.mark.parametrize("split", [1, 64, 200, 512])
def test_split_run_equals_whole_run(oracle, kernel, split):
    """Two calls chained by the final state reproduce one call over the whole
    sequence (the oracle's whole run is the reference)."""
    inp = _edge(**CASES["fp32-mask-gate-states"])
    inp["chunk_len"] = 0
    if not tier_supported(inp, kernel):
        pytest.skip(f"{kernel} does not take this shape")
    L = inp["x"].shape[1]
    y_ref, _ = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                               inp["z"], inp["valid_len"])
    p1, p2 = _piece(inp, 0, split), _piece(inp, split, L)
    y1, _, f1 = _gpu(p1, kernel, None)
    y2, _, f2 = _gpu(p2, kernel, f1.astype(np.float32))
    y = np.concatenate([y1, y2], axis=1)
    e = rel_err(y, y_ref)
    assert e <= TOL_Y["f32"], f"split at {split}: y rel err {e:.3e}"
