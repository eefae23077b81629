"""The fused step-size preparation on a GPU, against the fp64 oracle.

delta <- clip(softplus(delta + dt_bias[d])) inside the kernels ([P1] s3.3),
for every tier, with masking, gating and chunk states, and in the decode
step.  Tolerances as in test_parity: fp32 y 1e-5, bf16 y 1e-2, fp32 states
1e-5, max-normalised.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

from test_parity import TOL_STATES, TOL_Y, _edge, rel_err, tier_supported, to_f64

pytestmark = pytest.mark.gpu

TIERS = ["serial", "warpscan", "stream", "auto"]


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def _raw_delta(inp, seed=41):
    """Raw step inputs and a per-channel bias with the recipe of the benchmark
    workloads: softplus(0.5 N(0,1) + dt_bias), dt_bias = softplus^-1(U(1e-3, 0.1))."""
    rng = np.random.default_rng(seed)
    Bt, L, Dm = inp["x"].shape
    raw = (0.5 * rng.standard_normal((Bt, L, Dm))).astype(np.float32)
    bias = np.log(np.expm1(rng.uniform(1e-3, 1e-1, Dm))).astype(np.float32)
    if inp["dtype"] == "bf16":
        raw = W.f32_to_bf16_bits(raw)
    return raw, bias


CASES = {
    "fp32-mask-gate-states": dict(batch=4, L=513, dim=40, N=16, gate=True, mask=[513, 0, 200, 1],
                                  chunk=100),
    "bf16-gate": dict(batch=2, L=300, dim=64, N=16, dtype="bf16", gate=True, chunk=64),
    "fp32-n64": dict(batch=1, L=400, dim=32, N=64),
    "bf16-n8-mask": dict(batch=3, L=257, dim=64, N=8, dtype="bf16", mask=[5, 257, 128]),
}
PREPS = {"bias-softplus": dict(softplus=True, bias=True, clamp=None),
         "softplus-clamp": dict(softplus=True, bias=True, clamp=(2e-3, 0.05)),
         "bias-only": dict(softplus=False, bias=True, clamp=None)}


@pytest.mark.parametrize("prep", sorted(PREPS))
@pytest.mark.parametrize("kernel", TIERS)
@pytest.mark.parametrize("name", sorted(CASES))
def test_prepared_delta_matches_oracle(oracle, name, kernel, prep):
    inp = _edge(**CASES[name])
    if not tier_supported(inp, kernel):
        pytest.skip(f"{kernel} does not take this shape")
    pr = PREPS[prep]
    raw, bias = _raw_delta(inp)
    if not pr["softplus"]:  # bias only: keep the step positive
        raw = inp["delta"]
        bias = np.abs(bias) * 1e-3
    inp["delta"] = raw
    y_ref, s_ref = oracle.scan_fwd(inp["x"], raw, inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["valid_len"], chunk_len=inp["chunk_len"],
                                   dt_bias=bias, delta_softplus=pr["softplus"],
                                   delta_clamp=pr["clamp"])
    t = W.to_torch(inp, "cuda")
    y, s = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                      t["valid_len"], chunk_len=inp["chunk_len"], kernel=kernel,
                      dt_bias=torch.from_numpy(bias).cuda(), delta_softplus=pr["softplus"],
                      delta_clamp=pr["clamp"])
    torch.cuda.synchronize()
    y, s = to_f64(y), (to_f64(s) if s is not None else None)
    e = rel_err(y, y_ref)
    assert e <= TOL_Y[inp["dtype"]], f"y rel err {e:.3e}"
    if s_ref is not None:
        assert rel_err(s, s_ref) <= TOL_STATES
    if inp["valid_len"] is not None:
        for b, v in enumerate(inp["valid_len"]):
            assert np.all(y[b, min(max(int(v), 0), y.shape[1]):] == 0)


def test_forced_stream_shape_without_preparation_is_refused():
    inp = _edge(batch=1, L=64, dim=64, N=16)
    t = W.to_torch(inp, "cuda")
    with pytest.raises(S.SsmError) as ei:
        S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], kernel="stream",
                   channels_per_lane=4, delta_softplus=True)
    assert ei.value.status == S.Status.ERR_UNSUPPORTED


def test_decode_with_prepared_delta_follows_the_scan(oracle):
    inp = _edge(batch=2, L=24, dim=40, N=16, gate=True)
    raw, bias = _raw_delta(inp)
    inp["delta"] = raw
    Bt, L, Dm = inp["x"].shape
    k = 10
    y_ref, _, f_ref = oracle.scan_fwd(inp["x"], raw, inp["A"], inp["B"], inp["C"], inp["D"],
                                      inp["z"], None, want_final=True, dt_bias=bias,
                                      delta_softplus=True, delta_clamp=(1e-3, 0.08))
    cut = {kk: (np.ascontiguousarray(v[:, :k]) if isinstance(v, np.ndarray) and v.ndim == 3
                else v) for kk, v in inp.items()}
    t = W.to_torch(cut, "cuda")
    bias_t = torch.from_numpy(bias).cuda()
    y_pre, _, state = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                 want_final=True, dt_bias=bias_t, delta_softplus=True,
                                 delta_clamp=(1e-3, 0.08))
    ys = [to_f64(y_pre)]
    A, D = W.to_torch({"A": inp["A"], "D": inp["D"]}, "cuda").values()
    for step in range(k, L):
        st = W.to_torch({kk: np.ascontiguousarray(inp[kk][:, step]) for kk in
                         ("x", "delta", "B", "C", "z")}, "cuda")
        y = S.decode_step(st["x"], st["delta"], A, st["B"], st["C"], D, st["z"], state=state,
                          dt_bias=bias_t, delta_softplus=True, delta_clamp=(1e-3, 0.08))
        ys.append(to_f64(y)[:, None])
    torch.cuda.synchronize()
    e = rel_err(np.concatenate(ys, axis=1), y_ref)
    assert e <= TOL_Y["f32"], f"y rel err {e:.3e}"
    assert rel_err(to_f64(state), f_ref) <= TOL_STATES


@pytest.mark.parametrize("key", [2, 3])
def test_fused_delta_full_size_whole_tensor(oracle, key):
    """The benchmark's fused-preparation configuration at full size (raw delta
    and dt_bias from the workload's recipe), whole y and chunk states against
    the oracle."""
    w = W.WORKLOADS[key]
    inp = W.make_inputs(w)
    raw, bias = W.make_raw_delta(w)
    inp["delta"] = raw
    t = W.to_torch(inp, "cuda")
    y, s = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                      t["valid_len"], chunk_len=w.chunk_len,
                      dt_bias=torch.from_numpy(bias).cuda(), delta_softplus=True)
    torch.cuda.synchronize()
    S.check_device_errors()
    yg = to_f64(y)
    sg = to_f64(s) if s is not None else None
    del y, s, t
    y_ref, s_ref = oracle.scan_fwd(inp["x"], raw, inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["z"], inp["valid_len"], chunk_len=w.chunk_len,
                                   dt_bias=bias, delta_softplus=True)
    e = rel_err(yg, y_ref)
    assert e <= TOL_Y[w.dtype], f"workload {key}: y rel err {e:.3e}"
    if s_ref is not None:
        assert rel_err(sg, s_ref) <= TOL_STATES
