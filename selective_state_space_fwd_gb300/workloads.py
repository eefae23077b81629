"""Seeded synthetic inputs for the selective-scan forward.

This module only draws random tensors with the stated distributions and
stores them in the I/O dtype.  It holds none of the scan's arithmetic, imports
neither the CUDA library nor the oracle, and is the one piece both sides
share: the tests and the benchmark feed the same arrays to the oracle and to
the GPU.

Five workloads (shapes and distributions of the method's usual settings:
S4D-real state matrices A[d, n] = -(n + 1), a positive step size delta, Gaussian
x, B, C):

  1 tiny-fp32     batch 1, L 256, dim 64, N 16; delta = exp(U(ln 1e-3, ln 1e-1));
                  D = 1; fp32; no gate, no mask.                           seed 0
  2 fp32          batch 8, L 4096, dim 1024, N 16; delta = softplus(0.5 N(0,1) +
                  dt_bias_d), dt_bias_d = softplus^-1(U(1e-3, 1e-1)); A = -exp(ln(n+1));
                  D ~ N(0,1); fp32; no gate.                               seed 1
  3 bf16-gated    batch 8, L 2048, dim 2048, N 16; as 2 plus z ~ N(0,1); bf16 I/O;
                  chunk states every 256 steps.                            seed 2
  4 varlen-bf16   batch 32, L_max 2048, dim 1536, N 16; as 3 with valid_len ~ U{64..2048};
                  padded positions are still filled with N(0,1) draws.     seed 3
  5 long-fp32     batch 2, L 32768, dim 2048, N 64; delta as in 1; A = -(n+1); D = 1; fp32.
                                                                           seed 4

The softplus in the delta recipe of workloads 2-4 is part of how the input is
drawn (the forward receives delta already positive); it is evaluated here in
fp64 with numpy and rounded to the I/O dtype like every other input.

Each tensor draws from its own stream, numpy PCG64 seeded with
(workload seed, tensor id), so a tensor does not depend on the shapes of the
others.  bf16 tensors are returned as uint16 arrays of bf16 bit patterns
(float32 rounded to nearest even).
"""
from __future__ import annotations

import dataclasses

import numpy as np

# tensor ids of the per-tensor streams
_X, _DELTA, _DTBIAS, _B, _C, _D, _Z, _VALID, _STATE = range(9)


@dataclasses.dataclass(frozen=True)
class Workload:
    key: int
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    dtype: str            # "f32" or "bf16"
    delta: str            # "loguniform" or "softplus"
    a_init: str           # "s4d" (-(n+1)) or "s4d_exp" (-exp(ln(n+1)))
    d_skip: str           # "ones" or "normal"
    gate: bool
    mask: tuple[int, int] | None  # valid_len ~ U{lo..hi}
    chunk_len: int
    seed: int

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def elements(self) -> int:
        return self.batch * self.seqlen * self.dim


WORKLOADS: dict[int, Workload] = {
    1: Workload(1, "tiny-fp32", 1, 256, 64, 16, "f32", "loguniform", "s4d", "ones", False, None,
                0, 0),
    2: Workload(2, "fp32-b8-l4096-d1024-n16", 8, 4096, 1024, 16, "f32", "softplus", "s4d_exp",
                "normal", False, None, 0, 1),
    3: Workload(3, "bf16-gated-b8-l2048-d2048-n16-chunk256", 8, 2048, 2048, 16, "bf16", "softplus",
                "s4d_exp", "normal", True, None, 256, 2),
    4: Workload(4, "varlen-bf16-b32-l2048-d1536-n16-chunk256", 32, 2048, 1536, 16, "bf16",
                "softplus", "s4d_exp", "normal", True, (64, 2048), 256, 3),
    5: Workload(5, "long-fp32-b2-l32768-d2048-n64", 2, 32768, 2048, 64, "f32", "loguniform", "s4d",
                "ones", False, None, 0, 4),
}

# Long sequences of few channels, for the time split of the forward (the rows
# alone leave most of the GPU idle): distributions of workloads 2 and 5.
SPLIT_WORKLOADS = {
    1: Workload(301, "long-few-channels-fp32-b1-l65536-d256-n16", 1, 65536, 256, 16, "f32",
                "softplus", "s4d_exp", "normal", False, None, 0, 31),
    2: Workload(302, "long-few-channels-fp32-b2-l32768-d512-n64", 2, 32768, 512, 64, "f32",
                "loguniform", "s4d", "ones", False, None, 0, 32),
}

# Decode steps (one step of the recurrence on a carried state): the inputs of
# one time step for every (batch row, channel), drawn like the scan workloads'
# (seqlen 1), plus a state [batch, dim, dstate] ~ N(0, 1) in fp32.  The state
# is larger than L2, as for a serving batch of 1024 sequences.
DECODE_WORKLOADS = {
    1: Workload(101, "decode-fp32-b1024-d2048-n16", 1024, 1, 2048, 16, "f32", "softplus",
                "s4d_exp", "normal", False, None, 0, 11),
    2: Workload(102, "decode-bf16-gated-b1024-d2048-n16", 1024, 1, 2048, 16, "bf16",
                "softplus", "s4d_exp", "normal", True, None, 0, 12),
    # one sequence's step of a generation loop: a 128 KB state, bound by launch
    # latency rather than HBM
    3: Workload(103, "decode-fp32-b1-d2048-n16", 1, 1, 2048, 16, "f32", "softplus",
                "s4d_exp", "normal", False, None, 0, 13),
}


@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    """A workload of the SSD form (one decay per head): channels in nheads heads
    of headdim, bf16 I/O.  Mamba 2's usual settings: headdim 64, dstate 128,
    A_h = -U(1, 16), delta = softplus(0.5 N(0,1) + dt_bias_h) with
    dt_bias_h = softplus^-1(U(1e-3, 1e-1)), D = 1, x, z, B, C ~ N(0, 1)."""
    key: int
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    gate: bool
    mask: tuple[int, int] | None
    seed: int

    def scaled(self, **kw) -> "SsdWorkload":
        return dataclasses.replace(self, **kw)

    @property
    def dim(self) -> int:
        return self.nheads * self.headdim

    @property
    def elements(self) -> int:
        return self.batch * self.seqlen * self.dim


SSD_WORKLOADS = {
    1: SsdWorkload(201, "ssd-bf16-gated-b8-l4096-h32-p64-n128", 8, 4096, 32, 64, 128, True, None,
                   21),
    2: SsdWorkload(202, "ssd-bf16-gated-b8-l4096-h32-p64-n256", 8, 4096, 32, 64, 256, True, None,
                   22),
}


def make_ssd_inputs(w: SsdWorkload) -> dict:
    """All inputs of an SSD workload: x, z [batch, L, nheads*headdim], delta
    [batch, L, nheads], B, C [batch, L, dstate] as bf16 bit patterns; A
    [nheads], D [nheads*headdim] fp32; valid_len int32 [batch] or None."""
    Bt, L, H, N = w.batch, w.seqlen, w.nheads, w.dstate
    act = (Bt, L, w.dim)
    x = _normal(_rng(w.seed, _X), act)
    u = _rng(w.seed, _DTBIAS).uniform(1e-3, 1e-1, H)
    dt_bias = np.log(np.expm1(u))
    g = _normal(_rng(w.seed, _DELTA), (Bt, L, H)).astype(np.float64)
    delta = _softplus64(0.5 * g + dt_bias[None, None, :]).astype(np.float32)
    A = -_rng(w.seed, _D).uniform(1.0, 16.0, H).astype(np.float32)
    Bm = _normal(_rng(w.seed, _B), (Bt, L, N))
    Cm = _normal(_rng(w.seed, _C), (Bt, L, N))
    D = np.ones(w.dim, dtype=np.float32)
    z = _normal(_rng(w.seed, _Z), act) if w.gate else None
    valid = None
    if w.mask is not None:
        lo, hi = w.mask
        valid = _rng(w.seed, _VALID).integers(lo, hi + 1, size=Bt).astype(np.int32)
    x, delta, Bm, Cm = (f32_to_bf16_bits(t) for t in (x, delta, Bm, Cm))
    z = f32_to_bf16_bits(z) if z is not None else None
    return dict(x=x, delta=delta, A=A, B=Bm, C=Cm, D=D, z=z, valid_len=valid, dtype="bf16",
                nheads=H)


def make_raw_delta(w: Workload):
    """For the softplus recipe: the step inputs before the fused preparation,
    raw = 0.5 N(0,1) [batch, L, dim] (I/O dtype) and dt_bias [dim] fp32, from
    the same streams as make_inputs' delta, so that softplus(raw + dt_bias)
    is that delta up to the rounding of raw and dt_bias."""
    if w.delta != "softplus":
        raise ValueError("only the softplus recipe has a raw form")
    shape = (w.batch, w.seqlen, w.dim)
    u = _rng(w.seed, _DTBIAS).uniform(1e-3, 1e-1, w.dim)
    bias = np.log(np.expm1(u)).astype(np.float32)
    rng = _rng(w.seed, _DELTA)
    raw = np.empty(shape, dtype=np.float32)
    r2 = raw.reshape(-1, w.dim)
    rows_per_chunk = max(1, (1 << 22) // w.dim)
    for r in range(0, r2.shape[0], rows_per_chunk):
        n = min(rows_per_chunk, r2.shape[0] - r)
        r2[r:r + n] = 0.5 * rng.standard_normal((n, w.dim))
    if w.dtype == "bf16":
        raw = f32_to_bf16_bits(raw)
    return raw, bias


def make_state(w: Workload) -> np.ndarray:
    """A carried state for decode workloads: fp32 [batch, dim, dstate] ~ N(0, 1)."""
    return _normal(_rng(w.seed, _STATE), (w.batch, w.dim, w.dstate)).astype(np.float32)


def _rng(seed: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, chunk=1 << 24) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    for s in range(0, out.size, chunk):
        out[s:s + chunk] = rng.standard_normal(min(chunk, out.size - s), dtype=np.float32)
    return out.reshape(shape)


def _softplus64(v: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, v)


def _delta(w: Workload, shape, chunk=1 << 22) -> np.ndarray:
    rng = _rng(w.seed, _DELTA)
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    if w.delta == "loguniform":
        lo, hi = np.log(1e-3), np.log(1e-1)
        for s in range(0, out.size, chunk):
            n = min(chunk, out.size - s)
            out[s:s + n] = np.exp(rng.uniform(lo, hi, n))
    elif w.delta == "softplus":
        # dt_bias_d = softplus^-1(u) = ln(expm1(u)), u ~ U(1e-3, 1e-1), one per channel
        u = _rng(w.seed, _DTBIAS).uniform(1e-3, 1e-1, shape[-1])
        dt_bias = np.log(np.expm1(u))
        flat_dim = shape[-1]
        rows_per_chunk = max(1, chunk // flat_dim)
        rows = out.size // flat_dim
        o2 = out.reshape(rows, flat_dim)
        for r in range(0, rows, rows_per_chunk):
            n = min(rows_per_chunk, rows - r)
            g = rng.standard_normal((n, flat_dim))
            o2[r:r + n] = _softplus64(0.5 * g + dt_bias[None, :])
    else:
        raise ValueError(w.delta)
    return out.reshape(shape)


def make_inputs(w: Workload) -> dict:
    """All inputs of workload ``w`` as numpy arrays, in the I/O dtype.

    Keys: x, delta, A, B, C, D, z (None without gate), valid_len (None without
    mask), plus 'dtype' and 'chunk_len'.  fp32 tensors are float32; bf16 tensors
    are uint16 bit patterns."""
    Bt, L, Dm, N = w.batch, w.seqlen, w.dim, w.dstate
    act = (Bt, L, Dm)
    x = _normal(_rng(w.seed, _X), act)
    delta = _delta(w, act)
    if w.a_init == "s4d":
        A = -np.tile(np.arange(1, N + 1, dtype=np.float64), (Dm, 1))
    elif w.a_init == "s4d_exp":
        A = -np.exp(np.log(np.tile(np.arange(1, N + 1, dtype=np.float64), (Dm, 1))))
    else:
        raise ValueError(w.a_init)
    A = A.astype(np.float32)
    Bm = _normal(_rng(w.seed, _B), (Bt, L, N))
    Cm = _normal(_rng(w.seed, _C), (Bt, L, N))
    if w.d_skip == "ones":
        D = np.ones(Dm, dtype=np.float32)
    else:
        D = _rng(w.seed, _D).standard_normal(Dm).astype(np.float32)
    z = _normal(_rng(w.seed, _Z), act) if w.gate else None
    valid = None
    if w.mask is not None:
        lo, hi = w.mask
        valid = _rng(w.seed, _VALID).integers(lo, hi + 1, size=Bt).astype(np.int32)
    if w.dtype == "bf16":
        x, delta, Bm, Cm = (f32_to_bf16_bits(t) for t in (x, delta, Bm, Cm))
        z = f32_to_bf16_bits(z) if z is not None else None
    elif w.dtype != "f32":
        raise ValueError(w.dtype)
    return dict(x=x, delta=delta, A=A, B=Bm, C=Cm, D=D, z=z, valid_len=valid, dtype=w.dtype,
                chunk_len=w.chunk_len)


def channel_slice(inp: dict, b: int, d: int) -> dict:
    """Inputs restricted to the single channel (b, d), batch 1 and dim 1.
    Pure indexing, for computing sampled reference outputs one channel at a time."""
    out = dict(inp)
    for k in ("x", "delta", "z"):
        if inp[k] is not None:
            out[k] = np.ascontiguousarray(inp[k][b:b + 1, :, d:d + 1])
    for k in ("B", "C"):
        out[k] = np.ascontiguousarray(inp[k][b:b + 1])
    out["A"] = np.ascontiguousarray(inp["A"][d:d + 1])
    out["D"] = np.ascontiguousarray(inp["D"][d:d + 1]) if inp["D"] is not None else None
    if inp["valid_len"] is not None:
        out["valid_len"] = np.ascontiguousarray(inp["valid_len"][b:b + 1])
    return out


def to_torch(inp: dict, device="cuda") -> dict:
    """Move a make_inputs() dict to PyTorch tensors (bf16 bit patterns become bfloat16)."""
    import torch

    def conv(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    out = {k: conv(v) if isinstance(v, np.ndarray) or v is None else v for k, v in inp.items()}
    return out
