"""ctypes front end of the fp64 CPU oracle (``ref_scan.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of the selective
scan forward that the CUDA library is checked against.  Only the test suite,
``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` leg may import
this module.  It imports nothing from the CUDA package and the CUDA package
imports nothing from it.

Arrays are numpy: fp32 tensors as ``float32``; bf16 tensors as ``uint16``
holding the raw bf16 bit patterns.  Results are ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_scan.c")
_LIB_CACHE: dict[str, ctypes.CDLL] = {}


def lib_path(plant: int = 0) -> str:
    name = "libref_scan.so" if plant == 0 else f"libref_scan_plant{plant}.so"
    return os.path.join(_HERE, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math).  ``plant`` > 0
    builds a mutant with one known mistake, for the tests that check the pins
    catch it."""
    out = lib_path(plant)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
               f"-DREF_PLANT={int(plant)}", _SRC, "-o", out + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)
    return out


def _load(plant: int = 0) -> ctypes.CDLL:
    key = str(plant)
    if key in _LIB_CACHE:
        return _LIB_CACHE[key]
    lib = ctypes.CDLL(build(plant))
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.ref_scan_fwd.restype = I32
    lib.ref_scan_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I32, I32]
    lib.ref_scan_fwd_full.restype = I32
    lib.ref_scan_fwd_full.argtypes = [P, P, P, I32, I32, ctypes.c_double, ctypes.c_double, P, P,
                                      P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I32, I32]
    lib.ref_scan_fwd_h0.restype = I32
    lib.ref_scan_fwd_h0.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64,
                                    I32, I32]
    lib.ref_ssd_fwd.restype = I32
    lib.ref_ssd_fwd.argtypes = [P] * 11 + [I64, I64, I64, I64, I64, I32, I32]
    lib.ref_scan_bwd.restype = I32
    lib.ref_scan_bwd.argtypes = [P] * 18 + [I64, I64, I64, I64, I32, I32]
    D = ctypes.c_double
    lib.ref_combine.restype = None
    lib.ref_combine.argtypes = [D, D, D, D, ctypes.POINTER(D), ctypes.POINTER(D)]
    lib.ref_linear_recurrence.restype = None
    lib.ref_linear_recurrence.argtypes = [P, P, I64, D, P]
    lib.ref_plant_id.restype = I32
    _LIB_CACHE[key] = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def combine(a1: float, b1: float, a2: float, b2: float, plant: int = 0) -> tuple[float, float]:
    """The affine composition: (a1, b1) first, then (a2, b2)."""
    ao, bo = ctypes.c_double(), ctypes.c_double()
    _load(plant).ref_combine(a1, b1, a2, b2, ctypes.byref(ao), ctypes.byref(bo))
    return ao.value, bo.value


def linear_recurrence(a, b, h0: float = 0.0, plant: int = 0) -> np.ndarray:
    """h_t = a_t h_{t-1} + b_t from h_{-1} = h0, for 1-D arrays a and b."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    assert a.shape == b.shape and a.ndim == 1
    h = np.empty_like(a)
    _load(plant).ref_linear_recurrence(_ptr(a), _ptr(b), a.shape[0], float(h0), _ptr(h))
    return h


def scan_fwd(x, delta, A, B, C, D=None, z=None, valid_len=None, chunk_len: int = 0,
             threads: int = 0, plant: int = 0, h0=None, want_final: bool = False,
             dt_bias=None, delta_softplus: bool = False, delta_clamp=None):
    """Run the oracle.  Returns ``(y, states)``: y is float64 [batch, L, dim];
    states is float64 [batch, ceil(L/chunk_len), dim, dstate], or None when
    ``chunk_len`` is 0.  With ``h0`` (float32 [batch, dim, dstate]) the state
    starts there instead of at 0; with ``want_final`` the result is
    ``(y, states, final)`` with the state after the last step.  ``dt_bias``
    (float32 [dim]) is added to delta, ``delta_softplus`` applies softplus to
    the sum and ``delta_clamp`` = (lo, hi) clips it, before delta is used."""
    if x.dtype == np.float32:
        dtype = 0
    elif x.dtype == np.uint16:
        dtype = 1
    else:
        raise TypeError("x must be float32 or uint16 (bf16 bits)")
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    for name, t, shape in (("delta", delta, (batch, L, dim)), ("B", B, (batch, L, dstate)),
                           ("C", C, (batch, L, dstate))):
        if t.shape != shape or t.dtype != x.dtype:
            raise ValueError(f"{name}: expected {shape} {x.dtype}, got {t.shape} {t.dtype}")
    if A.shape != (dim, dstate) or A.dtype != np.float32:
        raise ValueError("A must be float32 [dim, dstate]")
    if D is not None and (D.shape != (dim,) or D.dtype != np.float32):
        raise ValueError("D must be float32 [dim]")
    if z is not None and (z.shape != (batch, L, dim) or z.dtype != x.dtype):
        raise ValueError("z must match x")
    if valid_len is not None and (valid_len.shape != (batch,) or valid_len.dtype != np.int32):
        raise ValueError("valid_len must be int32 [batch]")
    if h0 is not None and (h0.shape != (batch, dim, dstate) or h0.dtype != np.float32):
        raise ValueError("h0 must be float32 [batch, dim, dstate]")
    if dt_bias is not None and (dt_bias.shape != (dim,) or dt_bias.dtype != np.float32):
        raise ValueError("dt_bias must be float32 [dim]")
    dt_bias = None if dt_bias is None else np.ascontiguousarray(dt_bias)
    arrs = [np.ascontiguousarray(t) if t is not None else None
            for t in (x, delta, A, B, C, D, z, valid_len, h0)]
    y = np.empty((batch, L, dim), dtype=np.float64)
    states = None
    if chunk_len > 0:
        states = np.empty((batch, (L + chunk_len - 1) // chunk_len, dim, dstate), dtype=np.float64)
    final = np.empty((batch, dim, dstate), dtype=np.float64) if want_final else None
    xa, da, Aa, Ba, Ca, Da, za, va, ha = arrs
    lo, hi = delta_clamp if delta_clamp is not None else (0.0, 0.0)
    rc = _load(plant).ref_scan_fwd_full(_ptr(xa), _ptr(da), _ptr(dt_bias), int(bool(delta_softplus)),
                                        int(delta_clamp is not None), float(lo), float(hi),
                                        _ptr(Aa), _ptr(Ba), _ptr(Ca), _ptr(Da), _ptr(za), _ptr(va),
                                        _ptr(ha), _ptr(y), _ptr(states), _ptr(final), batch, L, dim,
                                        dstate, int(chunk_len), dtype, int(threads))
    if rc != 0:
        raise RuntimeError("ref_scan_fwd failed")
    return (y, states, final) if want_final else (y, states)


def scan_bwd(x, delta, A, B, C, D=None, z=None, valid_len=None, dy=None, h0=None,
             threads: int = 0, plant: int = 0) -> dict:
    """Gradients of l = sum(dy * y) with respect to every input of the forward
    (delta used as given).  Returns a dict of float64 arrays: dx, ddelta, dA,
    dB, dC, dD (None without D), dz (None without gate), dh0 (None without h0)."""
    if x.dtype == np.float32:
        dtype = 0
    elif x.dtype == np.uint16:
        dtype = 1
    else:
        raise TypeError("x must be float32 or uint16 (bf16 bits)")
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    if dy.shape != (batch, L, dim):
        raise ValueError("dy must be [batch, L, dim]")
    arrs = [np.ascontiguousarray(t) if t is not None else None
            for t in (x, delta, A, B, C, D, z, valid_len, h0)]
    out = {"dx": np.empty((batch, L, dim)), "ddelta": np.empty((batch, L, dim)),
           "dA": np.empty((dim, dstate)), "dB": np.empty((batch, L, dstate)),
           "dC": np.empty((batch, L, dstate)), "dD": np.empty(dim) if D is not None else None,
           "dz": np.empty((batch, L, dim)) if z is not None else None,
           "dh0": np.empty((batch, dim, dstate)) if h0 is not None else None}
    rc = _load(plant).ref_scan_bwd(*[_ptr(t) for t in arrs], _ptr(dy), _ptr(out["dx"]),
                                   _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]),
                                   _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
                                   _ptr(out["dh0"]), batch, L, dim, dstate, dtype, int(threads))
    if rc != 0:
        raise RuntimeError("ref_scan_bwd failed")
    return out


def ssd_fwd(x, delta, A, B, C, D=None, z=None, valid_len=None, h0=None, nheads: int = 1,
            want_final: bool = False, threads: int = 0, plant: int = 0):
    """The SSD form of the scan: one decay per head.  x, z [batch, L, nheads *
    headdim]; delta [batch, L, nheads]; A float32 [nheads]; B, C [batch, L,
    dstate]; D float32 [nheads * headdim]; h0 float32 [batch, nheads * headdim,
    dstate].  Returns y (float64 [batch, L, dim]), and with ``want_final`` also
    the state after the last step (float64 [batch, dim, dstate])."""
    if x.dtype == np.float32:
        dtype = 0
    elif x.dtype == np.uint16:
        dtype = 1
    else:
        raise TypeError("x must be float32 or uint16 (bf16 bits)")
    batch, L, dim = x.shape
    if dim % nheads:
        raise ValueError("dim must be a multiple of nheads")
    headdim = dim // nheads
    dstate = B.shape[-1]
    for name, t, shape in (("delta", delta, (batch, L, nheads)), ("B", B, (batch, L, dstate)),
                           ("C", C, (batch, L, dstate))):
        if t.shape != shape or t.dtype != x.dtype:
            raise ValueError(f"{name}: expected {shape} {x.dtype}, got {t.shape} {t.dtype}")
    if A.shape != (nheads,) or A.dtype != np.float32:
        raise ValueError("A must be float32 [nheads]")
    if D is not None and (D.shape != (dim,) or D.dtype != np.float32):
        raise ValueError("D must be float32 [dim]")
    if z is not None and (z.shape != (batch, L, dim) or z.dtype != x.dtype):
        raise ValueError("z must match x")
    if valid_len is not None and (valid_len.shape != (batch,) or valid_len.dtype != np.int32):
        raise ValueError("valid_len must be int32 [batch]")
    if h0 is not None and (h0.shape != (batch, dim, dstate) or h0.dtype != np.float32):
        raise ValueError("h0 must be float32 [batch, dim, dstate]")
    arrs = [np.ascontiguousarray(t) if t is not None else None
            for t in (x, delta, A, B, C, D, z, valid_len, h0)]
    y = np.empty((batch, L, dim), dtype=np.float64)
    final = np.empty((batch, dim, dstate), dtype=np.float64) if want_final else None
    rc = _load(plant).ref_ssd_fwd(*[_ptr(t) for t in arrs], _ptr(y), _ptr(final), batch, L,
                                  nheads, headdim, dstate, dtype, int(threads))
    if rc != 0:
        raise RuntimeError("ref_ssd_fwd failed")
    return (y, final) if want_final else y


def plant_id(plant: int = 0) -> int:
    return _load(plant).ref_plant_id()
