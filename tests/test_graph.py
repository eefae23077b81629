"""The library's device entry points inside a CUDA graph: a decode loop (the
launch-bound inner loop of generation) and a forward, captured once and
replayed, give the same results bit for bit as the same calls made eagerly.
Every entry point works asynchronously on the caller's stream and plans on the
host, so the calls record into the graph like any kernel launch."""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

from test_parity import _edge

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


@pytest.mark.parametrize("dtype,gate", [("f32", False), ("bf16", True)])
def test_decode_loop_in_a_cuda_graph(dtype, gate):
    K = 12
    inp = _edge(batch=4, L=K, dim=96, N=16, dtype=dtype, gate=gate)
    t = W.to_torch(inp, "cuda")
    h0 = torch.randn(4, 96, 16, device="cuda")
    steps = [{k: (t[k][:, i].contiguous() if t[k] is not None else None)
              for k in ("x", "delta", "B", "C", "z")} for i in range(K)]

    def run(state, outs):
        for i, s in enumerate(steps):
            S.decode_step(s["x"], s["delta"], t["A"], s["B"], s["C"], t["D"], s["z"],
                          state=state, out=outs[i])

    outs_e = [torch.empty_like(s["x"]) for s in steps]
    state_e = h0.clone()
    run(state_e, outs_e)  # eager (also does the library's one-time lookups)

    outs_g = [torch.empty_like(s["x"]) for s in steps]
    state_g = h0.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            run(state_g, outs_g)
    torch.cuda.current_stream().wait_stream(side)
    state_g.copy_(h0)  # capture does not execute: start the replay from h0
    g.replay()
    torch.cuda.synchronize()
    S.check_device_errors()
    for a, b in zip(outs_e, outs_g):
        assert torch.equal(a, b)
    assert torch.equal(state_e, state_g)
    # a second replay continues from the state the first one left
    g.replay()
    torch.cuda.synchronize()
    state_e2 = state_e.clone()
    run(state_e2, outs_e)
    torch.cuda.synchronize()
    assert torch.equal(state_e2, state_g)


def test_forward_in_a_cuda_graph():
    inp = _edge(batch=4, L=700, dim=64, N=16, gate=True, mask=[700, 300, 1, 0], chunk=128)
    t = W.to_torch(inp, "cuda")
    y_e, s_e = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                          t["valid_len"], chunk_len=128, time_segments=1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            y_g, s_g = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                  t["valid_len"], chunk_len=128, time_segments=1)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    S.check_device_errors()
    assert torch.equal(y_e, y_g) and torch.equal(s_e, s_g)


def _capture(fn):
    """fn() captured once into a graph (on a side stream) and replayed once."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            out = fn()
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    S.check_device_errors()
    return out


def test_backward_in_a_cuda_graph():
    inp = _edge(batch=2, L=300, dim=64, N=16, gate=True, mask=[300, 170])
    t = W.to_torch(inp, "cuda")
    _, states = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["valid_len"], chunk_len=64, time_segments=1)
    dy = torch.randn_like(t["x"])

    def bwd():
        return S.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                          t["valid_len"], chunk_states=states, chunk_len=64, dy=dy,
                          want_dh0=True)

    g_e = bwd()
    torch.cuda.synchronize()
    g_g = _capture(bwd)
    for k in ("dx", "ddelta", "dz", "dh0"):
        assert torch.equal(g_e[k], g_g[k]), k
    for k in ("dA", "dB", "dC", "dD"):  # atomics: equal up to the order of the sums
        assert torch.allclose(g_e[k], g_g[k], rtol=1e-5, atol=1e-6), k


def test_ssd_in_a_cuda_graph():
    w = W.SSD_WORKLOADS[1].scaled(batch=2, seqlen=512, nheads=4)
    inp = W.make_ssd_inputs(w)
    t = W.to_torch(inp, "cuda")

    def ssd():
        return S.ssd_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                         t["valid_len"], nheads=w.nheads)

    y_e = ssd()
    torch.cuda.synchronize()
    y_g = _capture(ssd)
    assert torch.equal(y_e, y_g)
