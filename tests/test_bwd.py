"""The backward (``ssm_scan_bwd``) on a GPU, against the fp64 oracle's backward.

Tolerances (max |g - g_ref| / max |g_ref| per gradient): the forward's fp32
bound is 1e-5; the backward runs a second recurrence of the same length and
adds the summed gradients (dA over batch and steps, dB and dC over channels,
dD) with fp32 atomics in no fixed order, so 1e-4 for every fp32 result, and
1e-2 for gradients stored in bf16 (dx, ddelta, dz with bf16 I/O: rounding of
the stored value, as for the forward's y).

Two kernels serve the backward: the TMA-tiled one for 16, 32 or 64 states,
chunks a multiple of 16 steps and 16-byte aligned buffers (every case below
that meets those), and the generic one for the rest (chunks of 1, 7, 100;
N of 1, 2, 8), which the ``misaligned`` variant also forces on tiled shapes
by placing x 4 (or 2) bytes past a 16-byte boundary.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

from test_parity import _edge, _poison_padding, rel_err, to_f64

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


CASES = {
    "fp32-gate-mask-h0-chunk100": dict(e=dict(batch=3, L=400, dim=40, N=16, gate=True,
                                              mask=[400, 0, 157]), chunk=100, h0=True),
    "fp32-n64-chunk64": dict(e=dict(batch=1, L=300, dim=24, N=64), chunk=64, h0=False),
    "bf16-gate-chunk256": dict(e=dict(batch=2, L=520, dim=64, N=16, dtype="bf16", gate=True),
                               chunk=256, h0=False),
    "fp32-n1-chunk1": dict(e=dict(batch=2, L=33, dim=33, N=1), chunk=1, h0=True),
    "fp32-n2-gate-chunk7": dict(e=dict(batch=2, L=60, dim=8, N=2, gate=True), chunk=7, h0=False),
    "bf16-n8-mask-chunk512": dict(e=dict(batch=3, L=1100, dim=32, N=8, dtype="bf16",
                                         mask=[1100, 5, 1024]), chunk=512, h0=True),
    # chunks of exactly one replay piece: the chunk states are the checkpoints
    "fp32-gate-mask-chunk16": dict(e=dict(batch=2, L=100, dim=24, N=16, gate=True,
                                          mask=[100, 37]), chunk=16, h0=True),
    # tiled: several channel blocks with a ragged last one, ragged L, valid
    # lengths inside a piece, on a piece boundary and zero
    "fp32-n16-mask-h0-chunk64": dict(e=dict(batch=4, L=333, dim=72, N=16,
                                            mask=[333, 0, 170, 64]), chunk=64, h0=True),
    "fp32-n32-gate-mask-chunk48": dict(e=dict(batch=2, L=200, dim=20, N=32, gate=True,
                                              mask=[200, 77]), chunk=48, h0=False),
    "bf16-n64-gate-mask-h0-chunk128": dict(e=dict(batch=2, L=300, dim=24, N=64, dtype="bf16",
                                                  gate=True, mask=[300, 129]), chunk=128,
                                           h0=True),
    "bf16-n32-chunk32": dict(e=dict(batch=2, L=90, dim=48, N=32, dtype="bf16"), chunk=32,
                             h0=False),
    # 32 checkpoints per chunk (one CTA per SM)
    "fp32-n16-gate-chunk512": dict(e=dict(batch=2, L=1100, dim=32, N=16, gate=True), chunk=512,
                                   h0=True),
    "fp32-n64-mask-chunk512": dict(e=dict(batch=2, L=1030, dim=16, N=64, mask=[1030, 517]),
                                   chunk=512, h0=True),
}


def _misaligned(t):
    """The same values one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


def _run_case(oracle, case, misalign=False, poison=False):
    inp = _edge(**case["e"])
    if poison:
        inp = _poison_padding(inp)
    Bt, L, Dm = inp["x"].shape
    N = inp["B"].shape[-1]
    rng = np.random.default_rng(61)
    dy = rng.standard_normal((Bt, L, Dm)).astype(np.float32)
    h0 = rng.standard_normal((Bt, Dm, N)).astype(np.float32) if case["h0"] else None
    bf16 = inp["dtype"] == "bf16"
    dy_io = W.f32_to_bf16_bits(dy) if bf16 else dy
    dy_ref = W.bf16_bits_to_f32(dy_io) if bf16 else dy
    ref = oracle.scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["z"], inp["valid_len"], dy=dy_ref.astype(np.float64), h0=h0)
    t = W.to_torch(inp, "cuda")
    h0t = torch.from_numpy(h0).cuda() if h0 is not None else None
    _, states = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["valid_len"], chunk_len=case["chunk"], h0=h0t)
    dyt = W.to_torch({"dy": dy_io}, "cuda")["dy"]
    xt = _misaligned(t["x"]) if misalign else t["x"]
    g = S.scan_bwd(xt, t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["valid_len"],
                   chunk_states=states, chunk_len=case["chunk"], dy=dyt, h0=h0t,
                   want_dh0=True)
    torch.cuda.synchronize()
    S.check_device_errors()
    for key in ("dx", "ddelta", "dz", "dA", "dB", "dC", "dD", "dh0"):
        if ref.get(key) is None and key != "dh0":
            assert g[key] is None
            continue
        want = ref[key]
        if key == "dh0" and want is None:
            # zero initial state: the gradient of h0 is still defined; check it
            # through the oracle run with an explicit zero state
            want = oracle.scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"],
                                   inp["D"], inp["z"], inp["valid_len"],
                                   dy=dy_ref.astype(np.float64),
                                   h0=np.zeros((Bt, Dm, N), np.float32))["dh0"]
        tol = TOL_BF16 if (bf16 and key in ("dx", "ddelta", "dz")) else TOL_F32
        got = to_f64(g[key])
        assert np.all(np.isfinite(got)), f"{key}: non-finite values"
        e = rel_err(got, want)
        assert e <= tol, f"{key}: rel err {e:.3e} > {tol}"
    if inp["valid_len"] is not None:
        for b, v in enumerate(inp["valid_len"]):
            v = min(max(int(v), 0), L)
            assert torch.all(g["dx"][b, v:] == 0) and torch.all(g["ddelta"][b, v:] == 0)
            if g["dz"] is not None:
                assert torch.all(g["dz"][b, v:] == 0)
            assert torch.all(g["dB"][b, v:] == 0) and torch.all(g["dC"][b, v:] == 0)
    return g


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(oracle, name):
    _run_case(oracle, CASES[name])


TILED = ["fp32-n16-mask-h0-chunk64", "bf16-n64-gate-mask-h0-chunk128",
         "fp32-n32-gate-mask-chunk48"]


@pytest.mark.parametrize("name", TILED)
def test_backward_generic_kernel_on_tiled_shapes(oracle, name):
    """The generic kernel on shapes the tiled one would take (x misaligned)."""
    _run_case(oracle, CASES[name], misalign=True)


@pytest.mark.parametrize("name", TILED)
@pytest.mark.parametrize("misalign", [False, True])
def test_backward_ignores_padding(oracle, name, misalign):
    """NaN and infinities at every step past valid_len of x, delta, z, B and C
    reach no gradient (padded steps are the identity, [P1] s2.3)."""
    _run_case(oracle, CASES[name], misalign=misalign, poison=True)


@pytest.mark.parametrize("key", [2, 3, 4])
def test_backward_full_size_whole_tensor(oracle, key):
    """Every gradient of the full-size workloads (the bench's chunk of 256 steps)
    against the oracle's backward, whole tensors."""
    w = W.WORKLOADS[key]
    chunk = 256
    inp = W.make_inputs(w)
    Bt, L, Dm = inp["x"].shape
    rng = np.random.default_rng(62)
    dy = rng.standard_normal((Bt, L, Dm)).astype(np.float32)
    bf16 = inp["dtype"] == "bf16"
    dy_io = W.f32_to_bf16_bits(dy) if bf16 else dy
    dy_ref = W.bf16_bits_to_f32(dy_io) if bf16 else dy
    t = W.to_torch(inp, "cuda")
    _, states = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["valid_len"], chunk_len=chunk)
    dyt = W.to_torch({"dy": dy_io}, "cuda")["dy"]
    g = S.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["valid_len"],
                   chunk_states=states, chunk_len=chunk, dy=dyt)
    torch.cuda.synchronize()
    S.check_device_errors()
    got = {k: to_f64(v) for k, v in g.items() if v is not None}
    del g, t, states, dyt
    ref = oracle.scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["z"], inp["valid_len"], dy=dy_ref.astype(np.float64))
    for key_g, v in got.items():
        tol = TOL_BF16 if (bf16 and key_g in ("dx", "ddelta", "dz")) else TOL_F32
        e = rel_err(v, ref[key_g])
        assert e <= tol, f"workload {key}: {key_g} rel err {e:.3e} > {tol}"
