"""Pins of the fp64 oracle: checks against what the pages and the mathematics
fix, independently of the oracle's own loop.  Each pin is a function taking
``plant`` (0 = the real oracle, k > 0 = a build of the oracle with planted
mistake k) and raising AssertionError when the oracle disagrees.

Page keys:
  [P1] the article at pwwt.cn/news/6372990 on Mamba's hardware-aware algorithm
       and parallel associative scan.
  [P2] "Mamba并行扫描与硬件感知优化：从SSM递推到GPU高效实现" (bjdmk.com.cn/news/5218626).
  [P3] the article at m.nxbn.cn/news/191302 (only its unrolled-sum formula of
       s1 is used, as the brute-force form of the recurrence).
"""
from __future__ import annotations

import math
import os

import numpy as np

from oracle import ref_scan as R

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_closed_form() -> np.ndarray:
    vals = [float(l) for l in open(os.path.join(GOLDEN, "closed_form_a05_b1_L8.txt"))
            if l.strip() and not l.startswith("#")]
    return np.array(vals)


def golden_bf16() -> list[tuple[int, float]]:
    out = []
    for l in open(os.path.join(GOLDEN, "bf16_widening.txt")):
        if l.strip() and not l.startswith("#"):
            bits, val = l.split()
            out.append((int(bits, 16), float(val)))
    return out


def _fwd(x, delta, A, B, C, D=None, z=None, valid_len=None, chunk_len=0, plant=0, threads=1):
    return R.scan_fwd(x, delta, A, B, C, D, z, valid_len, chunk_len=chunk_len, threads=threads,
                      plant=plant)


def _rand_inputs(rng, batch, L, dim, N, gate=False, mask=None):
    x = rng.standard_normal((batch, L, dim)).astype(np.float32)
    delta = np.exp(rng.uniform(np.log(1e-2), np.log(0.5), (batch, L, dim))).astype(np.float32)
    A = -np.exp(rng.uniform(np.log(0.5), np.log(4.0), (dim, N))).astype(np.float32)
    B = rng.standard_normal((batch, L, N)).astype(np.float32)
    C = rng.standard_normal((batch, L, N)).astype(np.float32)
    D = rng.standard_normal(dim).astype(np.float32)
    z = rng.standard_normal((batch, L, dim)).astype(np.float32) if gate else None
    return x, delta, A, B, C, D, z


# ---------------------------------------------------------------------------
# The combine and the serial recurrence


def pin_closed_form_recurrence(plant=0):
    """[P1] s2.3 note, s4.1: a = 0.5, b = 1, 8 steps, h = 2 (1 - 0.5^k)."""
    h = R.linear_recurrence(np.full(8, 0.5), np.ones(8), plant=plant)
    assert np.array_equal(h, golden_closed_form()), h


def pin_closed_form_forward(plant=0):
    """The same closed form driven through the full forward: N = 1, dim = 1,
    delta = 1, A = -ln 2 (so exp(delta A) = 1/2), B = C = 1, x = 1, D = 0, so y_t = h_t."""
    L = 8
    one = np.ones((1, L, 1), np.float32)
    A = np.array([[-math.log(2.0)]], np.float32)
    y, _ = _fwd(one, one, A, np.ones((1, L, 1), np.float32), np.ones((1, L, 1), np.float32),
                D=np.zeros(1, np.float32), plant=plant)
    np.testing.assert_allclose(y[0, :, 0], golden_closed_form(), rtol=1e-7, atol=0)


def pin_combine_is_composition(plant=0):
    """[P1] s2.1, [P2] s2.2: combine((a1,b1),(a2,b2)) applied to h equals applying
    (a1,b1) first and (a2,b2) second."""
    rng = np.random.default_rng(11)
    for _ in range(200):
        a1, b1, a2, b2, h = rng.uniform(-2, 2, 5)
        a, b = R.combine(a1, b1, a2, b2, plant=plant)
        direct = a2 * (a1 * h + b1) + b2
        assert abs((a * h + b) - direct) <= 1e-12 * max(1.0, abs(direct)), (a1, b1, a2, b2)


def _tree_reduce(ops, rng, plant):
    if len(ops) == 1:
        return ops[0]
    k = int(rng.integers(1, len(ops)))
    l = _tree_reduce(ops[:k], rng, plant)
    r = _tree_reduce(ops[k:], rng, plant)
    return R.combine(l[0], l[1], r[0], r[1], plant=plant)


def pin_associativity_bruteforce(plant=0):
    """[P1] s2.1, [P2] s2.2: the combine is associative.  All five bracketings of
    four random ops agree, and random bracketings of up to 16 ops agree with the
    left fold, to 1e-12 in fp64."""
    rng = np.random.default_rng(12)
    c = lambda p, q: R.combine(p[0], p[1], q[0], q[1], plant=plant)
    for _ in range(50):
        o = [tuple(rng.uniform(-1.5, 1.5, 2)) for _ in range(4)]
        forms = [c(c(c(o[0], o[1]), o[2]), o[3]), c(c(o[0], c(o[1], o[2])), o[3]),
                 c(c(o[0], o[1]), c(o[2], o[3])), c(o[0], c(c(o[1], o[2]), o[3])),
                 c(o[0], c(o[1], c(o[2], o[3])))]
        for f in forms[1:]:
            assert abs(f[0] - forms[0][0]) < 1e-12 and abs(f[1] - forms[0][1]) < 1e-12
    for n in range(2, 17):
        ops = [tuple(rng.uniform(-1.2, 1.2, 2)) for _ in range(n)]
        left = ops[0]
        for o in ops[1:]:
            left = c(left, o)
        for _ in range(5):
            t = _tree_reduce(ops, rng, plant)
            assert abs(t[0] - left[0]) < 1e-12 and abs(t[1] - left[1]) < 1e-12


def pin_recurrence_is_prefix_of_combines(plant=0):
    """The serial recurrence from h = 0 equals the b part of the inclusive prefix
    of combines (h_t = prefix_t applied to 0), [P1] s2.2."""
    rng = np.random.default_rng(13)
    a = rng.uniform(0, 1, 40)
    b = rng.standard_normal(40)
    h = R.linear_recurrence(a, b, plant=plant)
    acc = (a[0], b[0])
    assert abs(h[0] - acc[1]) < 1e-12
    for t in range(1, 40):
        acc = R.combine(acc[0], acc[1], a[t], b[t], plant=plant)
        assert abs(h[t] - acc[1]) < 1e-12 * max(1, abs(acc[1]))


def pin_reverse_identity(plant=0):
    """[P1] s2.3: the backward recurrence g_t = a_{t+1} g_{t+1} + c_t (g_{L-1} = c_{L-1})
    equals the forward recurrence run on the flipped sequence with the a's
    shifted by one."""
    rng = np.random.default_rng(14)
    L = 33
    a = rng.uniform(0, 1, L)
    c = rng.standard_normal(L)
    g = np.empty(L)
    g[L - 1] = c[L - 1]
    for t in range(L - 2, -1, -1):
        g[t] = a[t + 1] * g[t + 1] + c[t]
    a_shift = np.concatenate([a[1:], [0.0]])  # the coefficient that multiplies g_{t+1}
    fwd = R.linear_recurrence(a_shift[::-1].copy(), c[::-1].copy(), plant=plant)
    np.testing.assert_allclose(fwd[::-1], g, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# The full forward


def pin_lti_convolution(plant=0):
    """[P1] s1.2, [P2] s1.3: with delta, B and C constant in time the SSM is a
    causal convolution, y_t = sum_k K_k x_{t-k} + D x_t with
    K_k = sum_n C_n exp(delta A_n)^k delta B_n.  Checked with numpy's convolution."""
    rng = np.random.default_rng(15)
    L, dim, N = 64, 3, 5
    x = rng.standard_normal((1, L, dim)).astype(np.float32)
    dts = np.array([0.05, 0.3, 1.0], np.float32)
    delta = np.broadcast_to(dts, (1, L, dim)).astype(np.float32).copy()
    A = -rng.uniform(0.2, 3.0, (dim, N)).astype(np.float32)
    Bn = rng.standard_normal(N).astype(np.float32)
    Cn = rng.standard_normal(N).astype(np.float32)
    B = np.broadcast_to(Bn, (1, L, N)).astype(np.float32).copy()
    C = np.broadcast_to(Cn, (1, L, N)).astype(np.float32).copy()
    D = rng.standard_normal(dim).astype(np.float32)
    y, _ = _fwd(x, delta, A, B, C, D=D, plant=plant)
    k = np.arange(L)
    for d in range(dim):
        dt = float(dts[d])
        abar = np.exp(dt * A[d].astype(np.float64))
        K = (Cn.astype(np.float64)[None, :] * abar[None, :] ** k[:, None]
             * (dt * Bn.astype(np.float64))[None, :]).sum(1)
        xd = x[0, :, d].astype(np.float64)
        ref = np.convolve(xd, K)[:L] + float(D[d]) * xd
        np.testing.assert_allclose(y[0, :, d], ref, rtol=1e-10, atol=1e-12)


def pin_unrolled_sum_bruteforce(plant=0):
    """[P3] s1 unrolled form, [P1] s2.1: h_T = sum_s (prod_{j=s+1..T} a_j) b_s
    with a_j = exp(delta_j A), b_s = delta_s B_s x_s, evaluated with explicit
    products on a tiny time-varying input; y = C h + D x."""
    rng = np.random.default_rng(16)
    batch, L, dim, N = 2, 11, 3, 4
    x, delta, A, B, C, D, _ = _rand_inputs(rng, batch, L, dim, N)
    y, _ = _fwd(x, delta, A, B, C, D=D, plant=plant)
    f = lambda v: v.astype(np.float64)
    for b in range(batch):
        for d in range(dim):
            for T in range(L):
                h = np.zeros(N)
                for s in range(T + 1):
                    prod = np.ones(N)
                    for j in range(s + 1, T + 1):
                        prod *= np.exp(f(delta[b, j, d]) * f(A[d]))
                    h += prod * f(delta[b, s, d]) * f(B[b, s]) * f(x[b, s, d])
                ref = float((f(C[b, T]) * h).sum() + f(D[d]) * f(x[b, T, d]))
                assert abs(y[b, T, d] - ref) <= 1e-11 * max(1.0, abs(ref)), (b, T, d)


def pin_d_residual(plant=0):
    """[P1] s1.1: with C = 0 the output is exactly D x; with D absent and C = 0 it is 0."""
    rng = np.random.default_rng(17)
    x, delta, A, B, C, D, _ = _rand_inputs(rng, 2, 9, 4, 3)
    C0 = np.zeros_like(C)
    y, _ = _fwd(x, delta, A, B, C0, D=D, plant=plant)
    np.testing.assert_array_equal(y, D.astype(np.float64)[None, None, :] * x.astype(np.float64))
    y0, _ = _fwd(x, delta, A, B, C0, D=None, plant=plant)
    assert np.all(y0 == 0)


def pin_gate(plant=0):
    """The gate multiplies the whole output by silu(z) = z sigmoid(z) (sigmoid
    from scipy), and z = 0 gives exactly 0."""
    from scipy.special import expit
    rng = np.random.default_rng(18)
    x, delta, A, B, C, D, z = _rand_inputs(rng, 2, 17, 5, 4, gate=True)
    y, _ = _fwd(x, delta, A, B, C, D=D, plant=plant)
    yg, _ = _fwd(x, delta, A, B, C, D=D, z=z, plant=plant)
    zz = z.astype(np.float64)
    np.testing.assert_allclose(yg, y * zz * expit(zz), rtol=1e-12, atol=1e-14)
    yz, _ = _fwd(x, delta, A, B, C, D=D, z=np.zeros_like(z), plant=plant)
    assert np.all(yz == 0)


def pin_masking(plant=0):
    """[P1] s2.3, s5.3: steps at or past valid_len are the identity (a=1, b=0):
    a row with valid_len = k matches an unpadded run of length k for t < k,
    its outputs after that are exactly 0 and its chunk states stay frozen at
    h_{k-1}.  valid_len is clamped to [0, L]."""
    rng = np.random.default_rng(19)
    batch, L, dim, N, chunk = 4, 24, 3, 4, 5
    x, delta, A, B, C, D, z = _rand_inputs(rng, batch, L, dim, N, gate=True)
    vl = np.array([7, 0, 30, -3], np.int32)  # 30 -> L, -3 -> 0
    y, s = _fwd(x, delta, A, B, C, D=D, z=z, valid_len=vl, chunk_len=chunk, plant=plant)
    for b, k in enumerate([7, 0, 24, 0]):
        if k > 0:
            yk, sk = _fwd(x[b:b + 1, :k].copy(), delta[b:b + 1, :k].copy(), A, B[b:b + 1, :k].copy(),
                          C[b:b + 1, :k].copy(), D=D, z=z[b:b + 1, :k].copy(), chunk_len=k,
                          plant=plant)
            np.testing.assert_allclose(y[b, :k], yk[0], rtol=1e-13, atol=1e-14)
            frozen = sk[0, -1]
        else:
            frozen = np.zeros((dim, N))
        assert np.all(y[b, k:] == 0)
        # chunks that end at or after k hold the frozen state
        for c in range(s.shape[1]):
            t_end = min((c + 1) * chunk, L) - 1
            if t_end >= k - 1 and k < L:
                np.testing.assert_allclose(s[b, c], frozen, rtol=1e-13, atol=1e-14)


def pin_chunk_states_and_carry(plant=0):
    """[P1] s3.4: chunk c stores h at step min((c+1) chunk, L) - 1; and [P2] s4.2:
    the state inside the next chunk equals its zero-start local state plus the
    running product of a times the carried state (h = h_local + cumprod(a) h_in)."""
    rng = np.random.default_rng(20)
    batch, L, dim, N, chunk = 2, 23, 3, 4, 6
    x, delta, A, B, C, D, _ = _rand_inputs(rng, batch, L, dim, N)
    _, s = _fwd(x, delta, A, B, C, D=D, chunk_len=chunk, plant=plant)
    assert s.shape == (batch, 4, dim, N)
    f = lambda v: v.astype(np.float64)
    for b in range(batch):
        for d in range(dim):
            a = np.exp(f(delta[b, :, d])[:, None] * f(A[d])[None, :])        # [L, N]
            bb = (f(delta[b, :, d]) * f(x[b, :, d]))[:, None] * f(B[b])        # [L, N]
            h = np.zeros(N)
            hs = []
            for t in range(L):
                h = a[t] * h + bb[t]
                hs.append(h.copy())
            hs = np.array(hs)
            for c in range(4):
                t_end = min((c + 1) * chunk, L) - 1
                np.testing.assert_allclose(s[b, c, d], hs[t_end], rtol=1e-12, atol=1e-14)
            for c in range(1, 4):  # carry identity across chunk c-1 -> c
                t0, t1 = c * chunk, min((c + 1) * chunk, L)
                hl = np.zeros(N)
                for t in range(t0, t1):
                    hl = a[t] * hl + bb[t]
                carried = hl + np.prod(a[t0:t1], axis=0) * s[b, c - 1, d]
                np.testing.assert_allclose(carried, s[b, c, d], rtol=1e-12, atol=1e-14)


def pin_bf16_widening(plant=0):
    """bf16 inputs are read as their exact values: known bit patterns widen to
    the hand-computed numbers, and a bf16 run equals the fp32 run on the
    widened values bit for bit."""
    vals = golden_bf16()
    bits = np.array([b for b, _ in vals], np.uint16).reshape(1, -1, 1)
    L = bits.shape[1]
    ones16 = np.full((1, L, 1), 0x3F80, np.uint16)  # 1.0
    zero16 = np.zeros((1, L, 1), np.uint16)
    A = np.zeros((1, 1), np.float32)  # a = 1
    # x = bits, delta = 1, B = 0, C = 0: y = D x with D = 1 -> y is the widened x
    y, _ = _fwd(bits, ones16, A, zero16, zero16, D=np.ones(1, np.float32), plant=plant)
    for i, (_, v) in enumerate(vals):
        assert y[0, i, 0] == v, (i, v)
    rng = np.random.default_rng(21)
    x, delta, A, B, C, D, z = _rand_inputs(rng, 2, 13, 3, 4, gate=True)
    from selective_state_space_fwd_gb300.workloads import f32_to_bf16_bits, bf16_bits_to_f32
    t16 = [f32_to_bf16_bits(t) for t in (x, delta, B, C, z)]
    t32 = [bf16_bits_to_f32(t) for t in t16]
    y16, _ = _fwd(t16[0], t16[1], A, t16[2], t16[3], D=D, z=t16[4], plant=plant)
    y32, _ = _fwd(t32[0], t32[1], A, t32[2], t32[3], D=D, z=t32[4], plant=plant)
    assert np.array_equal(y16, y32)


def pin_long_sequence_sane(plant=0):
    """[P1] s4.1: with a in (0,1) and b ~ N(0,1) a long run stays finite, and
    with a bounded by a_max the state is bounded by max|b| / (1 - a_max)."""
    rng = np.random.default_rng(22)
    L = 20000
    a = rng.uniform(0.0, 0.99, L)
    b = rng.standard_normal(L)
    h = R.linear_recurrence(a, b, plant=plant)
    assert np.all(np.isfinite(h))
    assert np.max(np.abs(h)) <= np.max(np.abs(b)) / (1 - 0.99) + 1e-9


def pin_initial_state_split(plant=0):
    """[P1] s3.1, s3.4, [P2] s2.4: running [0, L) equals running [0, k) and then
    [k, L) from the state after step k-1 (the carry between chunks), for the
    outputs, the final state and the chunk states; and with h0 given on a
    length-1 run, h = a h0 + b by hand."""
    rng = np.random.default_rng(23)
    batch, L, dim, N, k = 2, 30, 3, 4, 12
    x, delta, A, B, C, D, z = _rand_inputs(rng, batch, L, dim, N, gate=True)
    vl = np.array([30, 17], np.int32)
    y, st, fin = R.scan_fwd(x, delta, A, B, C, D, z, vl, chunk_len=6, want_final=True,
                            plant=plant)
    y1, st1, f1 = R.scan_fwd(x[:, :k].copy(), delta[:, :k].copy(), A, B[:, :k].copy(),
                             C[:, :k].copy(), D, z[:, :k].copy(), np.minimum(vl, k),
                             chunk_len=6, want_final=True, plant=plant)
    y2, st2, f2 = R.scan_fwd(x[:, k:].copy(), delta[:, k:].copy(), A, B[:, k:].copy(),
                             C[:, k:].copy(), D, z[:, k:].copy(),
                             np.clip(vl - k, 0, L - k).astype(np.int32), chunk_len=6,
                             want_final=True, h0=f1.astype(np.float32), plant=plant)
    # the carried state is rounded to fp32 once: compare with a tolerance
    np.testing.assert_allclose(y[:, :k], y1, rtol=0, atol=0)
    np.testing.assert_allclose(y[:, k:], y2, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(fin, f2, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(st[:, :2], st1, rtol=0, atol=0)
    np.testing.assert_allclose(st[:, 2:], st2, rtol=1e-6, atol=1e-7)
    one = np.ones((1, 1, 1), np.float32)
    h0 = np.array([[[0.75]]], np.float32)
    A1 = np.array([[-0.5]], np.float32)
    ys, _, fs = R.scan_fwd(one * 2, one * 0.5, A1, one * 3, one, None, None, None,
                           want_final=True, h0=h0, plant=plant)
    want = np.exp(0.5 * -0.5) * 0.75 + 0.5 * 3 * 2
    assert abs(fs[0, 0, 0] - want) < 1e-12 and abs(ys[0, 0, 0] - want) < 1e-12


def pin_softplus_closed_form(plant=0):
    """Fused step-size preparation, closed form: raw delta = 0 and no bias give
    the step softplus(0) = ln 2; with A = -1 the decay is exactly 1/2 and
    b = ln 2, so h_t = 2 ln 2 (1 - 2^-t) (the a = 1/2 closed form scaled by
    ln 2) and y_t = h_t with B = C = x = 1, D = 0."""
    L = 8
    one = np.ones((1, L, 1), np.float32)
    y, _ = R.scan_fwd(one, np.zeros((1, L, 1), np.float32), -np.ones((1, 1), np.float32), one,
                      one, np.zeros(1, np.float32), delta_softplus=True, plant=plant)
    want = 2.0 * math.log(2.0) * (1.0 - 0.5 ** np.arange(1, L + 1))
    np.testing.assert_allclose(y[0, :, 0], want, rtol=1e-12, atol=0)


def pin_softplus_and_bias_library(plant=0):
    """softplus(delta + dt_bias[d]) inside the oracle equals passing the step
    size computed beforehand with numpy's logaddexp(0, v) = ln(e^0 + e^v) (a
    library routine); the bias alone equals adding it beforehand.  The
    precomputed steps are rounded to fp32 once: compared within 1e-6."""
    rng = np.random.default_rng(31)
    batch, L, dim, N = 2, 40, 5, 4
    x, _, A, B, C, D, z = _rand_inputs(rng, batch, L, dim, N, gate=True)
    raw = (0.5 * rng.standard_normal((batch, L, dim))).astype(np.float32)
    bias = np.log(np.expm1(rng.uniform(1e-3, 1e-1, dim))).astype(np.float32)
    y, _ = R.scan_fwd(x, raw, A, B, C, D, z, dt_bias=bias, delta_softplus=True, plant=plant)
    pre = np.logaddexp(0.0, raw.astype(np.float64) + bias.astype(np.float64)).astype(np.float32)
    y_pre, _ = R.scan_fwd(x, pre, A, B, C, D, z, plant=plant)
    np.testing.assert_allclose(y, y_pre, rtol=1e-6, atol=1e-6 * np.max(np.abs(y_pre)))
    pos = np.exp(rng.uniform(np.log(1e-2), np.log(0.5), (batch, L, dim))).astype(np.float32)
    small = (0.1 * rng.uniform(0.0, 1.0, dim)).astype(np.float32)
    y_b, _ = R.scan_fwd(x, pos, A, B, C, D, z, dt_bias=small, plant=plant)
    y_b2, _ = R.scan_fwd(x, (pos.astype(np.float64) + small).astype(np.float32), A, B, C, D, z,
                         plant=plant)
    np.testing.assert_allclose(y_b, y_b2, rtol=1e-6, atol=1e-6 * np.max(np.abs(y_b2)))


def pin_delta_clamp(plant=0):
    """Clipping after softplus: with [lo, hi] = [c, c] every step size is c, so
    the run equals one with delta = c given directly; with a wide interval the
    clip changes nothing; a clip inside the range moves only the steps outside
    it (compared with the steps clipped beforehand by numpy)."""
    rng = np.random.default_rng(37)
    batch, L, dim, N = 2, 30, 4, 4
    x, _, A, B, C, D, z = _rand_inputs(rng, batch, L, dim, N, gate=True)
    raw = rng.standard_normal((batch, L, dim)).astype(np.float32)
    c = np.float32(0.125)
    y_c, _ = R.scan_fwd(x, raw, A, B, C, D, z, delta_softplus=True,
                        delta_clamp=(float(c), float(c)), plant=plant)
    y_k, _ = R.scan_fwd(x, np.full_like(raw, c), A, B, C, D, z, plant=plant)
    np.testing.assert_allclose(y_c, y_k, rtol=1e-12, atol=1e-12)
    y_w, _ = R.scan_fwd(x, raw, A, B, C, D, z, delta_softplus=True, delta_clamp=(0.0, 1e30),
                        plant=plant)
    y_n, _ = R.scan_fwd(x, raw, A, B, C, D, z, delta_softplus=True, plant=plant)
    np.testing.assert_array_equal(y_w, y_n)
    lo, hi = 0.3, 0.9
    y_m, _ = R.scan_fwd(x, raw, A, B, C, D, z, delta_softplus=True, delta_clamp=(lo, hi),
                        plant=plant)
    pre = np.clip(np.logaddexp(0.0, raw.astype(np.float64)), lo, hi).astype(np.float32)
    y_p, _ = R.scan_fwd(x, pre, A, B, C, D, z, plant=plant)
    np.testing.assert_allclose(y_m, y_p, rtol=1e-6, atol=1e-6 * np.max(np.abs(y_p)))


# ---------------------------------------------------------------------------
# The backward


def _bwd_problem(rng, gate=True, with_h0=True):
    batch, L, dim, N = 2, 5, 2, 3
    x, delta, A, B, C, D, z = _rand_inputs(rng, batch, L, dim, N, gate=gate)
    h0 = rng.standard_normal((batch, dim, N)).astype(np.float32) if with_h0 else None
    vl = np.array([5, 3], np.int32)
    dy = rng.standard_normal((batch, L, dim))
    return dict(x=x, delta=delta, A=A, B=B, C=C, D=D, z=z, valid_len=vl, h0=h0), dy


def _loss(args, dy, plant):
    y, _ = R.scan_fwd(args["x"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                      args["z"], args["valid_len"], h0=args["h0"], plant=plant)
    return float(np.sum(dy * y))


def pin_bwd_finite_differences(plant=0):
    """Every gradient of l = sum(dy * y) against central differences of the
    forward (each fp32 input moved up and down by about 1e-3 of its size; the
    difference quotient uses the moved values as stored)."""
    rng = np.random.default_rng(51)
    args, dy = _bwd_problem(rng)
    g = R.scan_bwd(args["x"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                   args["z"], args["valid_len"], dy=dy, h0=args["h0"], plant=plant)
    names = {"x": "dx", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "h0": "dh0"}
    for key, gname in names.items():
        base = args[key]
        fd = np.empty(base.shape)
        for idx in np.ndindex(base.shape):
            v = float(base[idx])
            step = max(abs(v), 0.1) * 1e-3
            up, dn = base.copy(), base.copy()
            up[idx] = np.float32(v + step)
            dn[idx] = np.float32(v - step)
            lu = _loss(dict(args, **{key: up}), dy, plant)
            ld = _loss(dict(args, **{key: dn}), dy, plant)
            fd[idx] = (lu - ld) / (float(up[idx]) - float(dn[idx]))
        got = g[gname]
        scale = max(np.max(np.abs(fd)), 1e-12)
        assert np.max(np.abs(got - fd)) <= 1e-4 * scale, (key, np.max(np.abs(got - fd)), scale)


def pin_bwd_homogeneity(plant=0):
    """Without gate and with h0 = 0, y is linear in x, in B and in C, so
    <dx, x> = <dy, y>, <dB, B> = <dC, C> = <dy, y - D x> and <dD, D> = <dy, D x>
    (Euler's identity for functions homogeneous of degree one)."""
    rng = np.random.default_rng(53)
    args, dy = _bwd_problem(rng, gate=False, with_h0=False)
    y, _ = R.scan_fwd(args["x"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                      None, args["valid_len"], plant=plant)
    g = R.scan_bwd(args["x"], args["delta"], args["A"], args["B"], args["C"], args["D"], None,
                   args["valid_len"], dy=dy, plant=plant)
    L = y.shape[1]
    mask = (np.arange(L)[None, :] < args["valid_len"][:, None])[:, :, None]
    dxy = args["D"][None, None, :].astype(np.float64) * args["x"] * mask
    tot = float(np.sum(dy * y))
    assert abs(float(np.sum(g["dx"] * args["x"])) - tot) <= 1e-10 * abs(tot) + 1e-12
    rest = float(np.sum(dy * (y - dxy)))
    assert abs(float(np.sum(g["dB"] * args["B"])) - rest) <= 1e-10 * abs(rest) + 1e-12
    assert abs(float(np.sum(g["dC"] * args["C"])) - rest) <= 1e-10 * abs(rest) + 1e-12
    dpart = float(np.sum(dy * dxy))
    assert abs(float(np.sum(g["dD"] * args["D"])) - dpart) <= 1e-10 * abs(dpart) + 1e-12


# ---------------------------------------------------------------------------
# The SSD form ([P2] s5.1-s5.2): one decay per head


def _ssd_problem(rng, batch=2, L=10, H=2, P=3, N=4, valid=(10, 6)):
    dim = H * P
    x = rng.standard_normal((batch, L, dim)).astype(np.float32)
    delta = np.exp(rng.uniform(np.log(1e-2), np.log(0.5), (batch, L, H))).astype(np.float32)
    A = -np.exp(rng.uniform(np.log(0.5), np.log(4.0), H)).astype(np.float32)
    B = rng.standard_normal((batch, L, N)).astype(np.float32)
    C = rng.standard_normal((batch, L, N)).astype(np.float32)
    D = rng.standard_normal(dim).astype(np.float32)
    z = rng.standard_normal((batch, L, dim)).astype(np.float32)
    h0 = rng.standard_normal((batch, dim, N)).astype(np.float32)
    vl = np.array(valid, np.int32)
    return dict(x=x, delta=delta, A=A, B=B, C=C, D=D, z=z, h0=h0, valid_len=vl, H=H)


def pin_ssd_closed_form(plant=0):
    """The a = 1/2, b = 1 closed form through the SSD form: one head of one
    channel, one state, delta = 1, A = -ln 2, B = C = x = 1, D = 0."""
    L = 8
    one = np.ones((1, L, 1), np.float32)
    y = R.ssd_fwd(one, one, np.array([-math.log(2.0)], np.float32), one, one,
                  D=np.zeros(1, np.float32), nheads=1, plant=plant)
    np.testing.assert_allclose(y[0, :, 0], golden_closed_form(), rtol=1e-7, atol=0)


def pin_ssd_quadratic_form(plant=0):
    """[P2] s5.1: the recurrence written out is one lower-triangular
    (semiseparable) matrix per head applied to the inputs,
    y_t = sum_{s<=t} (C_t . B_s) exp(A_h sum_{s<r<=t} delta_r) delta_s x_s
          + (C_t . h0) exp(A_h sum_{r<=t} delta_r) + D x_t, times silu(z_t),
    built here by brute force as a dense matrix, with the final state as the
    same sums taken at the last valid step."""
    rng = np.random.default_rng(71)
    a = _ssd_problem(rng)
    H = a["H"]
    y, fin = R.ssd_fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["valid_len"],
                       a["h0"], nheads=H, want_final=True, plant=plant)
    batch, L, dim = a["x"].shape
    P = dim // H
    x, dl, B, C = (a[k].astype(np.float64) for k in ("x", "delta", "B", "C"))
    A, D, z, h0 = (a[k].astype(np.float64) for k in ("A", "D", "z", "h0"))
    want = np.zeros((batch, L, dim))
    want_fin = np.zeros(fin.shape)
    for b in range(batch):
        Lv = int(a["valid_len"][b])
        for h in range(H):
            cs = np.concatenate([[0.0], np.cumsum(dl[b, :Lv, h])])  # cs[t+1] = sum_{r<=t}
            M = np.zeros((Lv, Lv))
            for t in range(Lv):
                for s_ in range(t + 1):
                    M[t, s_] = (C[b, t] @ B[b, s_]) * math.exp(A[h] * (cs[t + 1] - cs[s_ + 1])) \
                        * dl[b, s_, h]
            ch = slice(h * P, (h + 1) * P)
            yp = M @ x[b, :Lv, ch]
            yp += (C[b, :Lv] @ h0[b, ch].T) * np.exp(A[h] * cs[1:])[:, None]
            yp += D[ch][None, :] * x[b, :Lv, ch]
            zz = z[b, :Lv, ch]
            want[b, :Lv, ch] = yp * zz / (1.0 + np.exp(-zz))
            w = np.exp(A[h] * (cs[Lv] - cs[1:])) * dl[b, :Lv, h]  # weight of step s in the final state
            want_fin[b, ch] = math.exp(A[h] * cs[Lv]) * h0[b, ch] + (x[b, :Lv, ch] * w[:, None]).T @ B[b, :Lv]
    scale = np.max(np.abs(want))
    assert np.max(np.abs(y - want)) <= 1e-12 * scale, np.max(np.abs(y - want)) / scale
    fscale = np.max(np.abs(want_fin))
    assert np.max(np.abs(fin - want_fin)) <= 1e-12 * fscale


def pin_ssd_reduces_to_scan(plant=0):
    """With the head's step size and decay copied to each of its channels and
    states (delta[b,t,d] = delta[b,t,h], A[d,n] = A[h]), the SSD form is the
    diagonal scan pinned above: same y and final state, fp32 and bf16 inputs."""
    rng = np.random.default_rng(73)
    a = _ssd_problem(rng, batch=2, L=23, H=3, P=4, N=5, valid=(23, 9))
    H = a["H"]
    P = a["x"].shape[2] // H
    N = a["B"].shape[2]
    for bf16 in (False, True):
        cv = (lambda t: _to_bf16_bits(t)) if bf16 else (lambda t: t)
        x, dl, B, C, z = (cv(a[k]) for k in ("x", "delta", "B", "C", "z"))
        y, fin = R.ssd_fwd(x, dl, a["A"], B, C, a["D"], z, a["valid_len"], a["h0"], nheads=H,
                           want_final=True, plant=plant)
        dfull = np.repeat(dl, P, axis=2)
        Afull = np.repeat(a["A"], P)[:, None].repeat(N, axis=1).astype(np.float32)
        ys, _, fs = R.scan_fwd(x, dfull, Afull, B, C, a["D"], z, a["valid_len"], h0=a["h0"],
                               want_final=True)
        np.testing.assert_allclose(y, ys, rtol=0, atol=1e-13 * np.max(np.abs(ys)))
        np.testing.assert_allclose(fin, fs, rtol=0, atol=1e-13 * np.max(np.abs(fs)))


def _to_bf16_bits(a):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (numpy, for pins only)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


ALL_PINS = [pin_closed_form_recurrence, pin_closed_form_forward, pin_combine_is_composition,
            pin_associativity_bruteforce, pin_recurrence_is_prefix_of_combines,
            pin_reverse_identity, pin_lti_convolution, pin_unrolled_sum_bruteforce,
            pin_d_residual, pin_gate, pin_masking, pin_chunk_states_and_carry,
            pin_bf16_widening, pin_long_sequence_sane, pin_initial_state_split,
            pin_softplus_closed_form, pin_softplus_and_bias_library, pin_delta_clamp,
            pin_bwd_finite_differences, pin_bwd_homogeneity, pin_ssd_closed_form,
            pin_ssd_quadratic_form, pin_ssd_reduces_to_scan]
