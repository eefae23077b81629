"""selective_scan under torch.autograd: the gradients autograd returns are
the library's backward, equal to the oracle's backward within its tolerances,
for fp32 and bf16 I/O, with the gate, valid lengths and an initial state."""
import numpy as np
import pytest
import torch

import selective_state_space_fwd_gb300 as S
from selective_state_space_fwd_gb300 import workloads as W

from test_parity import _edge, rel_err, to_f64

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built(ssmlib, oracle):
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield


@pytest.mark.parametrize("dtype,gate,mask,chunk", [
    ("f32", True, [300, 170, 0], 64),
    ("bf16", True, None, 128),
    ("f32", False, [300, 1, 299], 100),  # a chunk the tiled backward does not take
])
def test_autograd_gradients_match_the_oracle(oracle, dtype, gate, mask, chunk):
    inp = _edge(batch=3, L=300, dim=48, N=16, dtype=dtype, gate=gate, mask=mask)
    Bt, L, Dm = inp["x"].shape
    N = inp["B"].shape[-1]
    rng = np.random.default_rng(71)
    h0 = rng.standard_normal((Bt, Dm, N)).astype(np.float32)
    dy = rng.standard_normal((Bt, L, Dm)).astype(np.float32)
    bf16 = dtype == "bf16"
    dy_io = W.f32_to_bf16_bits(dy) if bf16 else dy
    dy_ref = W.bf16_bits_to_f32(dy_io) if bf16 else dy
    ref = oracle.scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["z"], inp["valid_len"], dy=dy_ref.astype(np.float64), h0=h0)
    t = W.to_torch(inp, "cuda")
    leaves = {k: t[k].clone().requires_grad_(True)
              for k in ("x", "delta", "A", "B", "C", "D", "z") if t[k] is not None}
    h0t = torch.from_numpy(h0).cuda().requires_grad_(True)
    y = S.selective_scan(leaves["x"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"],
                         leaves["D"], leaves.get("z"), t["valid_len"], h0=h0t, chunk_len=chunk)
    dyt = W.to_torch({"dy": dy_io}, "cuda")["dy"]
    y.backward(dyt)
    torch.cuda.synchronize()
    S.check_device_errors()
    grads = {"dx": leaves["x"].grad, "ddelta": leaves["delta"].grad, "dA": leaves["A"].grad,
             "dB": leaves["B"].grad, "dC": leaves["C"].grad, "dD": leaves["D"].grad,
             "dh0": h0t.grad}
    if gate:
        grads["dz"] = leaves["z"].grad
    for key, g in grads.items():
        tol = TOL_BF16 if (bf16 and key in ("dx", "ddelta", "dz", "dB", "dC")) else TOL_F32
        e = rel_err(to_f64(g), ref[key])
        assert e <= tol, f"{key}: rel err {e:.3e} > {tol}"
