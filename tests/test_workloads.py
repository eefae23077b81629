"""The seeded input generator (CPU): determinism, independence of the tensor
streams, the stated distributions, and bf16 rounding checked against
PyTorch's own float32 -> bfloat16 conversion."""
import numpy as np
import torch

from selective_state_space_fwd_gb300 import workloads as W


def small(k, **kw):
    w = W.WORKLOADS[k]
    return w.scaled(**{"seqlen": 96, "dim": 40, **kw})


def test_deterministic():
    for k in W.WORKLOADS:
        a, b = W.make_inputs(small(k)), W.make_inputs(small(k))
        for key in ("x", "delta", "A", "B", "C", "D", "z", "valid_len"):
            if a[key] is None:
                assert b[key] is None
            else:
                assert np.array_equal(a[key], b[key]), (k, key)


def test_streams_independent_of_other_shapes():
    a = W.make_inputs(small(2, dim=40))
    b = W.make_inputs(small(2, dim=56))
    assert np.array_equal(a["B"], b["B"]) and np.array_equal(a["C"], b["C"])


def test_distributions():
    w = W.WORKLOADS[1]
    inp = W.make_inputs(w)
    d = inp["delta"]
    assert d.min() >= 1e-3 * (1 - 1e-6) and d.max() <= 1e-1 * (1 + 1e-6)
    assert np.array_equal(inp["A"], -np.tile(np.arange(1, 17, dtype=np.float32), (64, 1)))
    assert np.all(inp["D"] == 1)
    assert abs(inp["x"].mean()) < 0.05 and abs(inp["x"].std() - 1) < 0.05
    inp2 = W.make_inputs(small(2, seqlen=512, dim=256))
    assert inp2["delta"].min() > 0 and inp2["A"].max() < 0
    inp4 = W.make_inputs(W.WORKLOADS[4].scaled(seqlen=64, dim=8))
    v = inp4["valid_len"]
    assert v.dtype == np.int32 and v.min() >= 64 and v.max() <= 2048 and v.shape == (32,)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    f = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1.0, -2.5, 3.0e38, 1e-30, 0.0, 1.00390625, 1.01171875],
                                 np.float32)])
    ours = W.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_channel_slice_is_indexing():
    inp = W.make_inputs(small(4, seqlen=64, dim=8))
    s = W.channel_slice(inp, 5, 3)
    assert np.array_equal(s["x"][0, :, 0], inp["x"][5, :, 3])
    assert np.array_equal(s["B"][0], inp["B"][5])
    assert np.array_equal(s["A"][0], inp["A"][3])
    assert s["valid_len"][0] == inp["valid_len"][5]


def test_ssd_inputs_shapes_and_ranges():
    w = W.SSD_WORKLOADS[1].scaled(batch=2, seqlen=96, nheads=3)
    a, b = W.make_ssd_inputs(w), W.make_ssd_inputs(w)
    for k in ("x", "delta", "A", "B", "C", "D", "z"):
        assert np.array_equal(a[k], b[k]), k  # seeded
    assert a["x"].shape == (2, 96, 3 * 64) and a["x"].dtype == np.uint16
    assert a["delta"].shape == (2, 96, 3) and a["B"].shape == (2, 96, 128)
    assert a["A"].shape == (3,) and np.all((a["A"] <= -1.0) & (a["A"] >= -16.0))
    dt = W.bf16_bits_to_f32(a["delta"])
    assert np.all(dt > 0) and np.all(dt < 1.0)
    assert np.all(a["D"] == 1.0) and a["valid_len"] is None
