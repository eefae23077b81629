"""The decode step (``ssm_decode_step``) on a GPU, against the fp64 oracle.

One decode step is the scan of one step starting from the given state; a
sequence scanned up to step k and then decoded step by step from the scan's
final state follows the scan of the whole sequence ([P1] s3.1 third level:
the serial carry; [P2] s2.4).  Tolerances as in test_parity: fp32 y 1e-5,
bf16 y 1e-2, the fp32 state 1e-5, max-normalised.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

from test_parity import TOL_STATES, TOL_Y, _edge, rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def _step_inputs(inp, t):
    """Step t of a [batch, L, ...] input set as [batch, ...] arrays."""
    return {k: (np.ascontiguousarray(inp[k][:, t]) if inp[k] is not None else None)
            for k in ("x", "delta", "B", "C", "z")}


def _gpu_step(step, A, D, state):
    dev = "cuda"
    cv = lambda a: None if a is None else W.to_torch({"v": a}, dev)["v"]
    y = S.decode_step(cv(step["x"]), cv(step["delta"]), cv(A), cv(step["B"]), cv(step["C"]),
                      cv(D), cv(step["z"]), state=state)
    return y


CASES = {
    "fp32-n16": dict(batch=3, L=40, dim=40, N=16),
    "fp32-n1": dict(batch=2, L=20, dim=33, N=1),
    "fp32-n2-gate": dict(batch=2, L=20, dim=8, N=2, gate=True),
    "bf16-n64-gate": dict(batch=2, L=24, dim=24, N=64, dtype="bf16", gate=True),
    "bf16-n8": dict(batch=4, L=16, dim=64, N=8, dtype="bf16"),
    # bf16 with 16 states stores the outputs of channel pairs together; an odd
    # batch * dim leaves the last output alone
    "bf16-n16-gate-odd": dict(batch=3, L=10, dim=33, N=16, dtype="bf16", gate=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_one_step_equals_scan_of_one_step(oracle, name):
    inp = _edge(**CASES[name])
    Bt, L, Dm = inp["x"].shape
    N = inp["B"].shape[-1]
    h0 = np.random.default_rng(5).standard_normal((Bt, Dm, N)).astype(np.float32)
    one = {k: (v[:, :1] if isinstance(v, np.ndarray) and v.ndim == 3 else v) for k, v in inp.items()}
    y_ref, _, f_ref = oracle.scan_fwd(one["x"], one["delta"], inp["A"], one["B"], one["C"],
                                      inp["D"], one["z"], None, h0=h0, want_final=True)
    state = torch.from_numpy(h0.copy()).cuda()
    y = _gpu_step(_step_inputs(inp, 0), inp["A"], inp["D"], state)
    torch.cuda.synchronize()
    e = rel_err(to_f64(y), y_ref[:, 0])
    assert e <= TOL_Y[inp["dtype"]], f"y rel err {e:.3e}"
    es = rel_err(to_f64(state), f_ref)
    assert es <= TOL_STATES, f"state rel err {es:.3e}"


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_then_decode_follows_the_scan(oracle, name):
    inp = _edge(**CASES[name])
    Bt, L, Dm = inp["x"].shape
    k = L // 2
    y_ref, _, f_ref = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                      inp["D"], inp["z"], None, want_final=True)
    t = W.to_torch({kk: (np.ascontiguousarray(v[:, :k]) if isinstance(v, np.ndarray) and v.ndim == 3
                         else v) for kk, v in inp.items()}, "cuda")
    y_pre, _, state = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                 want_final=True)
    ys = [to_f64(y_pre)]
    for step in range(k, L):
        ys.append(to_f64(_gpu_step(_step_inputs(inp, step), inp["A"], inp["D"], state))[:, None])
    torch.cuda.synchronize()
    y = np.concatenate(ys, axis=1)
    e = rel_err(y, y_ref)
    assert e <= TOL_Y[inp["dtype"]], f"y rel err {e:.3e}"
    es = rel_err(to_f64(state), f_ref)
    assert es <= TOL_STATES, f"final state rel err {es:.3e}"


@pytest.mark.parametrize("key", sorted(W.DECODE_WORKLOADS))
def test_decode_full_size_whole_tensor(oracle, key):
    """One decode step of the benchmark's decode workloads (batch 1024, dim
    2048, 16 states) from the workload's state, whole y and state against the
    oracle's scan of one step."""
    w = W.DECODE_WORKLOADS[key]
    inp = W.make_inputs(w)
    h0 = W.make_state(w)
    y_ref, _, f_ref = oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                      inp["D"], inp["z"], None, h0=h0, want_final=True)
    state = torch.from_numpy(h0.copy()).cuda()
    y = _gpu_step(_step_inputs(inp, 0), inp["A"], inp["D"], state)
    torch.cuda.synchronize()
    e = rel_err(to_f64(y), y_ref[:, 0])
    assert e <= TOL_Y[inp["dtype"]], f"y rel err {e:.3e}"
    assert rel_err(to_f64(state), f_ref) <= TOL_STATES


def _offset(t):
    """The same values one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("name", ["fp32-n16", "bf16-n64-gate"])
def test_decode_with_unaligned_rows(oracle, name):
    """B and C rows that do not start on a 16-byte boundary (the entry point
    requires only their element alignment) take element loads."""
    inp = _edge(**CASES[name])
    Bt, L, Dm = inp["x"].shape
    N = inp["B"].shape[-1]
    h0 = np.random.default_rng(6).standard_normal((Bt, Dm, N)).astype(np.float32)
    one = {k: (v[:, :1] if isinstance(v, np.ndarray) and v.ndim == 3 else v) for k, v in inp.items()}
    y_ref, _, f_ref = oracle.scan_fwd(one["x"], one["delta"], inp["A"], one["B"], one["C"],
                                      inp["D"], one["z"], None, h0=h0, want_final=True)
    step = _step_inputs(inp, 0)
    cv = lambda a: None if a is None else W.to_torch({"v": a}, "cuda")["v"]
    state = torch.from_numpy(h0.copy()).cuda()
    y = S.decode_step(cv(step["x"]), cv(step["delta"]), cv(inp["A"]), _offset(cv(step["B"])),
                      _offset(cv(step["C"])), cv(inp["D"]), cv(step["z"]), state=state)
    torch.cuda.synchronize()
    assert rel_err(to_f64(y), y_ref[:, 0]) <= TOL_Y[inp["dtype"]]
    assert rel_err(to_f64(state), f_ref) <= TOL_STATES
