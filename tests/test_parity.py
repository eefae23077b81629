"""Parity of the CUDA library with the fp64 oracle, through the C ABI, on a GPU.

Tolerances, from the path's precision contract (fp32 state and arithmetic):
  fp32 I/O:  max|y - y_ref| / max|y_ref| <= 1e-5
  bf16 I/O:  max|y - y_ref| / max|y_ref| <= 1e-2 (y is rounded to bf16)
  chunk states (fp32 always): max|s - s_ref| / max|s_ref| <= 1e-5
Outputs past valid_len must be exactly 0.
"""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# Tiers and STREAM launch shapes: "stream" takes the library's default shape,
# "stream-r4" four channels per thread, "stream-g8" eight states per thread,
# "stream-w4" four warps per CTA; "stream-tm" is the tier with B and C
# broadcast through tensor memory (channel pairs per lane), "stream-tm-r1" the
# same with one channel per lane.
TIERS = ["serial", "warpscan", "stream", "stream-r4", "stream-g8", "stream-w4", "stream-tm",
         "stream-tm-r1", "auto"]
_SHAPES = {"stream-r4": dict(channels_per_lane=4), "stream-g8": dict(states_per_lane=8),
           "stream-w4": dict(warps_per_block=4), "stream-tm-r1": dict(channels_per_lane=1)}


def _tier(kernel):
    """(tier, launch-shape keyword arguments) of a TIERS entry."""
    if kernel in _SHAPES:
        return ("stream-tm" if kernel.startswith("stream-tm") else "stream"), _SHAPES[kernel]
    return kernel, {}


TOL_Y = {"f32": 1e-5, "bf16": 1e-2}
TOL_STATES = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(inp: dict, kernel="auto", **kw):
    t = W.to_torch(inp, "cuda")
    k, shape = _tier(kernel)
    y, s = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                      t["valid_len"], chunk_len=inp["chunk_len"], kernel=k, **shape, **kw)
    torch.cuda.synchronize()
    return to_f64(y), (to_f64(s) if s is not None else None)


def run_oracle(oracle, inp: dict, threads=0):
    return oracle.scan_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["z"], inp["valid_len"], chunk_len=inp["chunk_len"],
                           threads=threads)


def rel_err(a, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(a - ref)) / den) if den > 0 else float(np.max(np.abs(a)))


def check(inp, y, s, y_ref, s_ref):
    tol = TOL_Y[inp["dtype"]]
    e = rel_err(y, y_ref)
    assert e <= tol, f"y rel err {e:.3e} > {tol}"
    if inp["valid_len"] is not None:
        L = y.shape[1]
        for b, v in enumerate(inp["valid_len"]):
            v = min(max(int(v), 0), L)
            assert np.all(y[b, v:] == 0), f"row {b}: nonzero output past valid_len {v}"
    if s_ref is not None:
        es = rel_err(s, s_ref)
        assert es <= TOL_STATES, f"chunk-state rel err {es:.3e} > {TOL_STATES}"
    return e


def tier_supported(inp, kernel):
    if kernel == "auto":
        return True
    Bt, L, Dm = inp["x"].shape
    k, shape = _tier(kernel)
    try:
        S.plan(Bt, L, Dm, inp["B"].shape[-1], dtype=inp["dtype"], gate=inp["z"] is not None,
               mask=inp["valid_len"] is not None, chunk_len=inp["chunk_len"], kernel=k, **shape)
        return True
    except S.SsmError as e:
        assert e.status == S.Status.ERR_UNSUPPORTED
        return False


# Scaled-down versions of the five workloads: several tiles of every tier and
# ragged tails in L and dim, small enough for the oracle to finish in seconds.
SMALL = {
    "w1-tiny-full": W.WORKLOADS[1],
    "w2-fp32": W.WORKLOADS[2].scaled(batch=2, seqlen=1000, dim=72),
    "w3-bf16-gate-states": W.WORKLOADS[3].scaled(batch=2, seqlen=700, dim=80),
    "w4-varlen": W.WORKLOADS[4].scaled(batch=6, seqlen=600, dim=48),
    "w5-long-n64": W.WORKLOADS[5].scaled(batch=1, seqlen=3000, dim=40),
}


def small_inputs(name):
    w = SMALL[name]
    inp = W.make_inputs(w)
    if w.mask is not None:  # span the edge cases: 0, 1, mid, L, > L
        inp["valid_len"] = np.array([0, 1, 64, 333, w.seqlen, w.seqlen + 100][:w.batch], np.int32)
    return inp


_ORACLE_CACHE = {}


def oracle_small(oracle, name):
    if name not in _ORACLE_CACHE:
        inp = small_inputs(name)
        _ORACLE_CACHE[name] = (inp, run_oracle(oracle, inp))
    return _ORACLE_CACHE[name]


@pytest.mark.parametrize("kernel", TIERS)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_workload_small(oracle, name, kernel):
    inp, (y_ref, s_ref) = oracle_small(oracle, name)
    if not tier_supported(inp, kernel):
        pytest.skip(f"{kernel} does not take this shape")
    y, s = run_gpu(inp, kernel)
    check(inp, y, s, y_ref, s_ref)


def _edge(batch, L, dim, N, dtype="f32", gate=False, mask=None, chunk=0, seed=7):
    w = W.Workload(0, "edge", batch, L, dim, N, dtype, "loguniform", "s4d", "normal", gate, None,
                   chunk, seed)
    inp = W.make_inputs(w)
    if mask is not None:
        inp["valid_len"] = np.array(mask, np.int32)
    return inp


EDGES = {
    "L1": dict(batch=2, L=1, dim=33, N=16),
    "L7-gate": dict(batch=1, L=7, dim=5, N=4, gate=True),
    "L31-N1": dict(batch=3, L=31, dim=64, N=1),
    "L33-N2-bf16": dict(batch=2, L=33, dim=48, N=2, dtype="bf16"),
    "N4-chunk1": dict(batch=1, L=40, dim=16, N=4, chunk=1),
    "N8-chunkL": dict(batch=2, L=100, dim=24, N=8, chunk=100),
    "N32-chunk-gtL": dict(batch=1, L=90, dim=40, N=32, chunk=1000),
    "N64-ragged": dict(batch=1, L=517, dim=9, N=64, chunk=128),
    "dim1": dict(batch=4, L=300, dim=1, N=16, chunk=64),
    "fp32-all-options": dict(batch=4, L=513, dim=37, N=16, gate=True, mask=[513, 0, 200, 1],
                             chunk=100),
    "bf16-mask-nogate": dict(batch=3, L=257, dim=64, N=16, dtype="bf16", mask=[5, 257, 128]),
    "chunk-not-mult-32": dict(batch=2, L=300, dim=32, N=16, chunk=48),
    "dim-odd-long": dict(batch=1, L=2500, dim=3, N=16, chunk=512),
}


@pytest.mark.parametrize("kernel", TIERS)
@pytest.mark.parametrize("name", sorted(EDGES))
def test_edge_cases(oracle, name, kernel):
    inp = _edge(**EDGES[name])
    if not tier_supported(inp, kernel):
        pytest.skip(f"{kernel} does not take this shape")
    y_ref, s_ref = run_oracle(oracle, inp)
    y, s = run_gpu(inp, kernel)
    check(inp, y, s, y_ref, s_ref)


def _poison_padding(inp):
    """Write NaN, +Inf and -Inf into every padded position (steps at or past
    valid_len) of x, delta, z, B and C.  Padded steps are the identity (1, 0)
    ([P1] s2.3, s5.3): nothing there may reach y or the state."""
    L = inp["x"].shape[1]
    for k in ("x", "delta", "z", "B", "C"):
        a = inp[k]
        if a is None:
            continue
        a = a.copy()
        for b, v in enumerate(inp["valid_len"]):
            v = min(max(int(v), 0), L)
            if v == L:
                continue
            n = a[b, v:].size
            if a.dtype == np.uint16:  # bf16 bit patterns: NaN, +Inf, -Inf
                pat = np.array([0x7FC0, 0x7F80, 0xFF80], np.uint16)
            else:
                pat = np.array([np.nan, np.inf, -np.inf], a.dtype)
            a[b, v:] = np.resize(pat, n).reshape(a[b, v:].shape)
        inp[k] = a
    return inp


@pytest.mark.parametrize("kernel", TIERS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nonfinite_padding_is_ignored(oracle, kernel, dtype):
    """Masked steps are a real identity: NaN and Inf in the padding of every
    input leave y exactly 0 there, the chunk states frozen and every valid
    output unchanged."""
    inp = _edge(batch=5, L=300, dim=48, N=16, dtype=dtype, gate=True,
                mask=[0, 1, 64, 150, 299], chunk=64, seed=11)
    clean = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    inp = _poison_padding(inp)
    if not tier_supported(inp, kernel):
        pytest.skip(f"{kernel} does not take this shape")
    y_ref, s_ref = run_oracle(oracle, clean)
    y, s = run_gpu(inp, kernel)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    check(inp, y, s, y_ref, s_ref)


def test_error_grows_slowly_with_length(oracle):
    """[P1] s4.4: the error against the reference stays at fp32 level as L grows
    from 256 to 8192.  Every decay is below 1, so the state forgets old
    rounding errors: the error must not grow with L the way a plain running sum
    would (linearly, 32x over this range), only stay at the fp32 level."""
    errs = []
    for L in (256, 1024, 4096, 8192):
        inp = _edge(batch=1, L=L, dim=64, N=16, seed=40)
        y_ref, _ = run_oracle(oracle, inp)
        y, _ = run_gpu(inp)
        errs.append(check(inp, y, None, y_ref, None))
    floor = 2.0 ** -23  # one fp32 rounding
    for e_short, e_long in zip(errs, errs[1:]):
        assert e_long <= 4 * max(e_short, 8 * floor), errs
    assert errs[-1] <= 8 * max(errs[0], 8 * floor), errs


def test_deterministic_bitwise():
    inp = W.make_inputs(SMALL["w2-fp32"])
    for kernel in TIERS:
        if not tier_supported(inp, kernel):
            continue
        y1, _ = run_gpu(inp, kernel)
        y2, _ = run_gpu(inp, kernel)
        assert np.array_equal(y1, y2), kernel


def test_tiers_agree_closely(oracle):
    """All tiers compute the same function; they may round differently.  fp32:
    y and the chunk states agree to a few fp32 roundings; bf16: the fp32
    results agree as closely, so the stored y differ by at most one bf16 ulp
    (2^-7 relative to the largest element)."""
    for name, tol_y in (("w2-fp32", 2e-6), ("w3-bf16-gate-states", 2.0 ** -7)):
        inp = small_inputs(name)
        outs = {k: run_gpu(inp, k) for k in TIERS if tier_supported(inp, k)}
        ref = outs["serial"]
        for k, (y, s) in outs.items():
            assert rel_err(y, ref[0]) <= tol_y, (name, k)
            if s is not None:
                assert rel_err(s, ref[1]) <= 2 * TOL_STATES, (name, k)


def test_host_entry_point_matches_device(oracle):
    inp = small_inputs("w4-varlen")
    t = W.to_torch(inp, "cpu")
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    y_h, s_h = S.scan_fwd_host(pinned["x"], pinned["delta"], pinned["A"], pinned["B"],
                               pinned["C"], pinned["D"], pinned["z"], pinned["valid_len"],
                               chunk_len=inp["chunk_len"])
    torch.cuda.synchronize()
    y_d, s_d = run_gpu(inp, time_segments=1)  # the host entry runs the unsplit tier per piece
    assert np.array_equal(to_f64(y_h), y_d)
    assert np.array_equal(to_f64(s_h), s_d)


@pytest.mark.parametrize("case", [
    dict(batch=1, L=8192, dim=64, N=16, gate=True, mask=[5000], chunk=256),
    dict(batch=3, L=6000, dim=40, N=8, dtype="bf16", mask=[6000, 0, 2345], chunk=100),
    dict(batch=2, L=7777, dim=32, N=64),
])
def test_host_entry_pipelined_pieces(oracle, case):
    """Long sequences go through several pipelined pieces chained by the
    carried state: the result is the device entry point's, bit for bit, and
    within tolerance of the oracle."""
    inp = _edge(**case)
    t = W.to_torch(inp, "cpu")
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    y_h, s_h = S.scan_fwd_host(pinned["x"], pinned["delta"], pinned["A"], pinned["B"],
                               pinned["C"], pinned["D"], pinned["z"], pinned["valid_len"],
                               chunk_len=inp["chunk_len"])
    torch.cuda.synchronize()
    y_d, s_d = run_gpu(inp, time_segments=1)  # the host entry runs the unsplit tier per piece
    assert np.array_equal(to_f64(y_h), y_d)
    if s_d is not None:
        assert np.array_equal(to_f64(s_h), s_d)
    y_ref, s_ref = run_oracle(oracle, inp)
    check(inp, to_f64(y_h), None if s_h is None else to_f64(s_h), y_ref, s_ref)


def test_host_entry_calls_in_flight():
    """Several end-to-end calls enqueued without waiting, alternating two
    streams and two workspaces (the calls share the library's copy streams):
    each returns, bit for bit, what the device entry point gives for its own
    inputs.  Consecutive calls get different inputs, so outputs that crossed
    over between calls, or a workspace overwritten while in use, would show."""
    case = dict(batch=2, L=8192, dim=64, N=16, gate=True, mask=[5000, 8192], chunk=256)
    inps = [_edge(**case, seed=s) for s in (11, 12, 13, 14)]
    pinned = []
    for inp in inps:
        t = W.to_torch(inp, "cpu")
        pinned.append({k: (v.pin_memory() if isinstance(v, torch.Tensor) else v)
                       for k, v in t.items()})
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    need = S.host_workspace_bytes(2, 8192, 64, 16, dtype="f32", has_D=True, gate=True, mask=True,
                                  chunk_len=256)
    wss = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in streams]
    outs = []
    for k, p in enumerate(pinned):
        outs.append(S.scan_fwd_host(p["x"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                    p["valid_len"], chunk_len=256, workspace=wss[k % 2],
                                    stream=streams[k % 2]))
    torch.cuda.synchronize()
    for inp, (y_h, s_h) in zip(inps, outs):
        y_d, s_d = run_gpu(inp, time_segments=1)
        assert np.array_equal(to_f64(y_h), y_d)
        assert np.array_equal(to_f64(s_h), s_d)


def test_stream_argument_is_respected():
    inp = W.make_inputs(SMALL["w2-fp32"])
    t = W.to_torch(inp, "cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        y, _ = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"])
    st.synchronize()
    y_ref, _ = run_gpu(inp)
    assert np.array_equal(to_f64(y), y_ref)


# Full-size workloads, in the launch configuration the benchmark times (AUTO),
# compared with the oracle on the whole of y and of the chunk states (the
# oracle runs every channel, one OpenMP thread per channel).
@pytest.mark.parametrize("key", [1, 2, 3, 4, 5])
def test_full_size_whole_tensor(oracle, key):
    w = W.WORKLOADS[key]
    inp = W.make_inputs(w)
    t = W.to_torch(inp, "cuda")
    y, s = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                      t["valid_len"], chunk_len=w.chunk_len)
    torch.cuda.synchronize()
    S.check_device_errors()
    del t
    y_ref, s_ref = run_oracle(oracle, inp)
    yg = to_f64(y)
    del y
    e = rel_err(yg, y_ref)
    assert e <= TOL_Y[w.dtype], f"workload {key}: y rel err {e:.3e}"
    if inp["valid_len"] is not None:
        for b, v in enumerate(inp["valid_len"]):
            assert np.all(yg[b, int(v):] == 0), f"workload {key}: row {b} past valid_len"
    if s is not None:
        es = rel_err(to_f64(s), s_ref)
        assert es <= TOL_STATES, f"workload {key}: state rel err {es:.3e}"


def test_length_ranked_rows_change_nothing_but_the_order():
    """Batches of at most 32 rows with valid lengths run their rows longest
    first; larger ones in index order.  The assignment of rows to CTAs is the
    only difference: the first 32 rows of a 33-row batch equal, bit for bit,
    the same 32 rows run as a batch of their own."""
    w = W.WORKLOADS[4].scaled(batch=33, seqlen=600, dim=48)
    inp = W.make_inputs(w)
    inp["valid_len"] = np.random.default_rng(9).integers(0, 700, size=33).astype(np.int32)
    t = W.to_torch(inp, "cuda")
    y33, s33 = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                          t["valid_len"], chunk_len=w.chunk_len, time_segments=1)
    sl = lambda v: v[:32].contiguous() if v is not None else None
    y32, s32 = S.scan_fwd(sl(t["x"]), sl(t["delta"]), t["A"], sl(t["B"]), sl(t["C"]), t["D"],
                          sl(t["z"]), sl(t["valid_len"]), chunk_len=w.chunk_len,
                          time_segments=1)
    torch.cuda.synchronize()
    assert torch.equal(y33[:32], y32)
    if s33 is not None:
        assert torch.equal(s33[:32], s32)
