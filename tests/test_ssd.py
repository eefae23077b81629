"""The SSD form (``ssm_ssd_fwd``, one decay per head, tensor-core products) on a
GPU, against the fp64 oracle's SSD form.

Tolerance, derived from the arithmetic: the products take bf16 operands (the
inputs as stored, delta-scaled B rows, the decay-weighted and masked block
matrix, x decayed to the block end, and the state entering a block), each
rounded once to 8 significant bits (relative 2^-9), and accumulate in fp32;
y is stored in bf16.  Sums of such terms stay within a few 2^-9 of the
largest output, so y is checked to 1e-2 max-normalised (the bound of every
bf16 output of the library) and the final state, which passes through the
same rounded operands but is stored in fp32, to 1e-2 as well.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_Y = 1e-2
TOL_STATE = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


BASE = W.SSD_WORKLOADS[1]
CASES = {
    # several blocks of 128 steps with a ragged tail, gate, initial state
    "b2-l300-h3-gate-h0": dict(w=dict(batch=2, seqlen=300, nheads=3, gate=True), h0=True),
    # masked rows: one empty, one ending inside a block, one ending on a block edge
    "b3-l384-h2-mask": dict(w=dict(batch=3, seqlen=384, nheads=2, gate=True), h0=True,
                            valid=[384, 0, 128]),
    "b2-l260-h2-mask-ragged": dict(w=dict(batch=2, seqlen=260, nheads=2, gate=False), h0=False,
                                   valid=[200, 131]),
    # valid lengths outside [0, L] are clamped
    "b2-l300-h1-mask-clamp": dict(w=dict(batch=2, seqlen=300, nheads=1, gate=True), h0=True,
                                  valid=[500, -5]),
    # exactly one block, no gate, no D
    "b1-l128-h1-noD": dict(w=dict(batch=1, seqlen=128, nheads=1, gate=False), h0=False,
                           no_d=True),
    # a single step
    "b2-l1-h2": dict(w=dict(batch=2, seqlen=1, nheads=2, gate=True), h0=True),
    # long enough for the decay between blocks to matter, several heads
    "b1-l1100-h4": dict(w=dict(batch=1, seqlen=1100, nheads=4, gate=True), h0=False),
    # 256 states: four 64-column parts of C and B, two state rows per TMEM lane
    "n256-b2-l300-h2-gate-h0": dict(w=dict(batch=2, seqlen=300, nheads=2, gate=True, dstate=256),
                                    h0=True),
    "n256-b3-l260-h1-mask": dict(w=dict(batch=3, seqlen=260, nheads=1, gate=False, dstate=256),
                                 h0=False, valid=[260, 0, 131]),
}


def _run(case):
    w = BASE.scaled(**case["w"])
    inp = W.make_ssd_inputs(w)
    if case.get("valid") is not None:
        inp["valid_len"] = np.array(case["valid"], np.int32)
    if case.get("no_d"):
        inp["D"] = None
    rng = np.random.default_rng(83)
    h0 = rng.standard_normal((w.batch, w.dim, w.dstate)).astype(np.float32) if case["h0"] else None
    t = W.to_torch(inp, "cuda")
    h0t = torch.from_numpy(h0).cuda() if h0 is not None else None
    y, fin = S.ssd_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                       t["valid_len"], nheads=w.nheads, h0=h0t, want_final=True)
    torch.cuda.synchronize()
    S.check_device_errors()
    return w, inp, h0, y, fin


@pytest.mark.parametrize("name", sorted(CASES))
def test_ssd_matches_oracle(oracle, name):
    case = CASES[name]
    w, inp, h0, y, fin = _run(case)
    y_ref, f_ref = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["valid_len"], h0, nheads=w.nheads,
                                  want_final=True)
    yg = y.float().cpu().numpy().astype(np.float64)
    fg = fin.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(yg)) and np.all(np.isfinite(fg))
    ey, ef = rel(yg, y_ref), rel(fg, f_ref)
    assert ey <= TOL_Y, f"y rel err {ey:.3e}"
    assert ef <= TOL_STATE, f"final state rel err {ef:.3e}"
    if inp["valid_len"] is not None:
        for b, v in enumerate(inp["valid_len"]):
            v = min(max(int(v), 0), w.seqlen)
            assert np.all(yg[b, v:] == 0)  # past valid_len the output is exactly 0


def test_ssd_split_equals_whole(oracle):
    """Running [0, 256) and then [256, L) from the first call's final state
    gives the single call's outputs: the carry between blocks is the state."""
    w = BASE.scaled(batch=2, seqlen=400, nheads=2, gate=True)
    inp = W.make_ssd_inputs(w)
    t = W.to_torch(inp, "cuda")
    y, fin = S.ssd_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], None,
                       nheads=w.nheads, want_final=True)
    k = 256
    part = {n: t[n][:, :k].contiguous() for n in ("x", "delta", "B", "C", "z")}
    rest = {n: t[n][:, k:].contiguous() for n in ("x", "delta", "B", "C", "z")}
    y1, f1 = S.ssd_fwd(part["x"], part["delta"], t["A"], part["B"], part["C"], t["D"], part["z"],
                       None, nheads=w.nheads, want_final=True)
    y2, f2 = S.ssd_fwd(rest["x"], rest["delta"], t["A"], rest["B"], rest["C"], t["D"], rest["z"],
                       None, nheads=w.nheads, h0=f1, want_final=True)
    torch.cuda.synchronize()
    # the same arithmetic on the same blocks: identical results
    assert torch.equal(torch.cat([y1, y2], dim=1), y)
    assert torch.equal(f2, fin)


def test_ssd_n256_split_equals_whole(oracle):
    """As above with 256 states: the state rows n and n + 128 share a TMEM lane."""
    w = BASE.scaled(batch=1, seqlen=384, nheads=2, gate=True, dstate=256)
    inp = W.make_ssd_inputs(w)
    t = W.to_torch(inp, "cuda")
    y, fin = S.ssd_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], None,
                       nheads=w.nheads, want_final=True)
    k = 128
    part = {n: t[n][:, :k].contiguous() for n in ("x", "delta", "B", "C", "z")}
    rest = {n: t[n][:, k:].contiguous() for n in ("x", "delta", "B", "C", "z")}
    _, f1 = S.ssd_fwd(part["x"], part["delta"], t["A"], part["B"], part["C"], t["D"], part["z"],
                      None, nheads=w.nheads, want_final=True)
    y2, f2 = S.ssd_fwd(rest["x"], rest["delta"], t["A"], rest["B"], rest["C"], t["D"], rest["z"],
                       None, nheads=w.nheads, h0=f1, want_final=True)
    torch.cuda.synchronize()
    assert torch.equal(y2, y[:, k:]) and torch.equal(f2, fin)


@pytest.mark.parametrize("key", sorted(W.SSD_WORKLOADS))
def test_ssd_full_size_whole_tensor(oracle, key):
    """The benchmark's workloads (128 and 256 states) at full size, in the
    launch configuration the benchmark times; the oracle computes every
    (batch row, head) and the whole of y is compared."""
    w = W.SSD_WORKLOADS[key]
    inp = W.make_ssd_inputs(w)
    t = W.to_torch(inp, "cuda")
    y = S.ssd_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], None,
                  nheads=w.nheads)
    torch.cuda.synchronize()
    S.check_device_errors()
    del t
    y_ref = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["z"], nheads=w.nheads)
    e = rel(y.float().cpu().numpy().astype(np.float64), y_ref)
    assert e <= TOL_Y, f"y rel err {e:.3e}"


def _halves(t, key):
    """Split the state dimension (last axis) of B or C in two contiguous halves."""
    return t[key][..., :64].contiguous(), t[key][..., 64:].contiguous()


def test_ssd_agrees_with_the_diagonal_scan(oracle):
    """With the head's step size and decay copied to its channels and states,
    the diagonal scan (STREAM tier, fp32 state) computes the same recurrence.
    The scan takes at most 64 states, so the 128 states are split in two and,
    without the gate, y is the sum of the two halves' outputs (D counted in
    one).  Both paths match the oracle, and each other within twice the bf16
    bound (two roundings of the summed outputs)."""
    w = BASE.scaled(batch=2, seqlen=640, nheads=2, gate=False)
    inp = W.make_ssd_inputs(w)
    t = W.to_torch(inp, "cuda")
    P, N = w.headdim, w.dstate
    y_ssd = S.ssd_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], None, None,
                      nheads=w.nheads)
    delta_full = t["delta"].repeat_interleave(P, dim=2).contiguous()
    A_half = t["A"].repeat_interleave(P)[:, None].expand(w.dim, N // 2).contiguous()
    (B1, B2), (C1, C2) = _halves(t, "B"), _halves(t, "C")
    y1, _ = S.scan_fwd(t["x"], delta_full, A_half, B1, C1, t["D"], None, None)
    y2, _ = S.scan_fwd(t["x"], delta_full, A_half, B2, C2, None, None, None)
    torch.cuda.synchronize()
    y_ref = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                           None, nheads=w.nheads)
    a = y_ssd.float().cpu().numpy().astype(np.float64)
    s2 = (y1.float() + y2.float()).cpu().numpy().astype(np.float64)
    assert rel(a, y_ref) <= TOL_Y
    assert rel(s2, y_ref) <= 2 * TOL_Y
    assert rel(a, s2) <= 2 * TOL_Y


def test_decode_continues_an_ssd_sequence(oracle):
    """The SSD form's final state, handed to the decode step (with the head's
    step size and decay copied to its channels and states, and the 128 states
    in two halves of 64 as for the scan), continues the sequence: decoding the
    last steps one by one gives the oracle's outputs for the whole sequence at
    those steps."""
    w = BASE.scaled(batch=2, seqlen=260, nheads=2, gate=False)
    inp = W.make_ssd_inputs(w)
    t = W.to_torch(inp, "cuda")
    P, N, k = w.headdim, w.dstate, 256
    pre = {n: t[n][:, :k].contiguous() for n in ("x", "delta", "B", "C")}
    _, state = S.ssd_fwd(pre["x"], pre["delta"], t["A"], pre["B"], pre["C"], t["D"], None, None,
                         nheads=w.nheads, want_final=True)
    st1, st2 = state[..., :64].contiguous(), state[..., 64:].contiguous()
    A_half = t["A"].repeat_interleave(P)[:, None].expand(w.dim, N // 2).contiguous()
    ys = []
    for s in range(k, w.seqlen):
        xs = t["x"][:, s].contiguous()
        dstep = t["delta"][:, s].repeat_interleave(P, dim=1).contiguous()
        Bs, Cs = t["B"][:, s], t["C"][:, s]
        ya = S.decode_step(xs, dstep, A_half, Bs[:, :64].contiguous(), Cs[:, :64].contiguous(),
                           t["D"], None, state=st1)
        yb = S.decode_step(xs, dstep, A_half, Bs[:, 64:].contiguous(), Cs[:, 64:].contiguous(),
                           None, None, state=st2)
        ys.append(ya.float() + yb.float())
    torch.cuda.synchronize()
    S.check_device_errors()
    y_ref = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], None,
                           nheads=w.nheads)
    got = torch.stack(ys, dim=1).cpu().numpy().astype(np.float64)
    assert rel(got, y_ref[:, k:]) <= 2 * TOL_Y
