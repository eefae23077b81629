"""ctypes binding of libssmscan (include/ssmscan.h): argument marshalling only.

Every step of the forward runs in the CUDA library.  Tensors are PyTorch CUDA
tensors (PyTorch provides device memory and streams); this module checks their
dtypes, shapes and devices, allocates outputs when the caller passes none, and
forwards raw pointers.  If the compiled library is missing the import fails
loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import enum
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssmscan.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "ssmscan.h")


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_SHAPE = 2
    ERR_UNSUPPORTED = 3
    ERR_ALIGN = 4
    ERR_CUDA = 5
    ERR_TIMEOUT = 6


class Kernel(enum.IntEnum):
    AUTO = 0
    SERIAL = 1
    WARPSCAN = 2
    STREAM = 3
    STREAM_TM = 4


class DType(enum.IntEnum):
    F32 = 0
    BF16 = 1


class SsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__(f"{where}: {self.status.name} ({status_string(status)})")


class Shapes(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("chunk_len", ctypes.c_int64)]


class Options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("warps_per_block", ctypes.c_int32),
                ("states_per_lane", ctypes.c_int32), ("channels_per_lane", ctypes.c_int32)]


_lib = None


class SsdShapes(ctypes.Structure):
    """ssm_ssd_shapes."""
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64)]


class DeltaPrep(ctypes.Structure):
    """ssm_delta_prep: the fused step-size preparation."""
    _fields_ = [("dt_bias", ctypes.c_void_p), ("softplus", ctypes.c_int32),
                ("clamp", ctypes.c_int32), ("lo", ctypes.c_float), ("hi", ctypes.c_float)]


def _prep(dt_bias, delta_softplus, delta_clamp, dim, dev):
    """A DeltaPrep for the keyword arguments, or None when nothing is asked."""
    if dt_bias is None and not delta_softplus and delta_clamp is None:
        return None
    import torch
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", (dim,), torch.float32, dev)
    lo, hi = delta_clamp if delta_clamp is not None else (0.0, 0.0)
    return DeltaPrep(_ptr(dt_bias).value if dt_bias is not None else None,
                     int(bool(delta_softplus)), int(delta_clamp is not None), float(lo), float(hi))


def load() -> ctypes.CDLL:
    """Load libssmscan.so (built in-tree by ``selective_state_space_fwd_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m selective_state_space_fwd_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    SP, OP = ctypes.POINTER(Shapes), ctypes.POINTER(Options)
    lib.ssm_scan_fwd.restype = I32
    lib.ssm_scan_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, SP, I32, P]
    lib.ssm_scan_fwd_ex.restype = I32
    lib.ssm_scan_fwd_ex.argtypes = [P, P, P, P, P, P, P, P, P, P, SP, I32, P, OP]
    lib.ssm_scan_fwd_carry.restype = I32
    lib.ssm_scan_fwd_carry.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, SP, I32, P, OP]
    DP = ctypes.POINTER(DeltaPrep)
    lib.ssm_scan_fwd_prep.restype = I32
    lib.ssm_scan_fwd_prep.argtypes = [P, P, DP, P, P, P, P, P, P, P, P, P, P, SP, I32, P, OP]
    lib.ssm_decode_step_prep.restype = I32
    lib.ssm_decode_step_prep.argtypes = [P, P, DP, P, P, P, P, P, P, P, I64, I64, I64, I32, P]
    lib.ssm_scan_fwd_host_static.restype = I32
    lib.ssm_scan_fwd_host_static.argtypes = [P, P, P, P, P, P, P, P, P, P, SP, I32, P]
    lib.ssm_scan_host_static_capacity.restype = SZ
    lib.ssm_scan_host_static_capacity.argtypes = []
    lib.ssm_ssd_fwd.restype = I32
    lib.ssm_ssd_fwd.argtypes = [P] * 11 + [ctypes.POINTER(SsdShapes), I32, P]
    lib.ssm_scan_bwd.restype = I32
    lib.ssm_scan_bwd.argtypes = [P] * 19 + [SP, I32, P]
    lib.ssm_decode_step.restype = I32
    lib.ssm_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, I64, I64, I64, I32, P]
    lib.ssm_scan_plan.restype = I32
    lib.ssm_scan_plan.argtypes = [SP, I32, I32, I32, I32, OP, ctypes.POINTER(I32),
                                  ctypes.POINTER(I64)]
    lib.ssm_scan_fwd_host.restype = I32
    lib.ssm_scan_fwd_host.argtypes = [P, P, P, P, P, P, P, P, P, P, SP, I32, P, SZ, P]
    lib.ssm_scan_host_workspace_bytes.restype = SZ
    lib.ssm_scan_host_workspace_bytes.argtypes = [SP, I32, I32, I32, I32, I32]
    lib.ssm_chunk_count.restype = I64
    lib.ssm_chunk_count.argtypes = [SP]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [I32]
    lib.ssm_kernel_name.restype = ctypes.c_char_p
    lib.ssm_kernel_name.argtypes = [I32]
    lib.ssm_version.restype = ctypes.c_char_p
    lib.ssm_version.argtypes = []
    lib.ssm_check_device_errors.restype = I32
    lib.ssm_check_device_errors.argtypes = []
    lib.ssm_scan_fwd_split.restype = I32
    lib.ssm_scan_fwd_split.argtypes = [P] * 12 + [SP, I32, I64, P, SZ, P]
    lib.ssm_scan_split_plan.restype = I32
    lib.ssm_scan_split_plan.argtypes = [SP, I32, I32, I64, ctypes.POINTER(I64),
                                        ctypes.POINTER(SZ)]
    lib.ssm_selftest_wait_timeout.restype = I32
    lib.ssm_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
    _lib = lib
    return lib


def declared_functions() -> list[str]:
    """Names of the functions include/ssmscan.h declares (for export checks)."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().ssm_status_string(int(status)).decode()


def kernel_name(kernel: int) -> str:
    return load().ssm_kernel_name(int(kernel)).decode()


def version() -> str:
    return load().ssm_version().decode()


def _shapes(batch, seqlen, dim, dstate, chunk_len) -> Shapes:
    return Shapes(int(batch), int(seqlen), int(dim), int(dstate), int(chunk_len))


def chunk_count(seqlen: int, chunk_len: int) -> int:
    s = _shapes(1, seqlen, 1, 1, chunk_len)
    return int(load().ssm_chunk_count(ctypes.byref(s)))


def check_device_errors() -> None:
    """Raise SsmError if a kernel's bounded wait gave up since the last check
    (synchronises the device)."""
    st = load().ssm_check_device_errors()
    if st != 0:
        raise SsmError(st, "ssm_check_device_errors")


def selftest_wait_timeout(polls: int = 1000, stream=None) -> None:
    """Run the bounded-wait self-test kernel: a wait on an mbarrier nothing
    arrives on gives up after ``polls`` polls and sets the sticky error word
    (read it with check_device_errors)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    with torch.cuda.device(stream.device):
        st = load().ssm_selftest_wait_timeout(int(polls), ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise SsmError(st, "ssm_selftest_wait_timeout")


def plan(batch, seqlen, dim, dstate, *, dtype="f32", gate=False, mask=False, chunk_len=0,
         kernel: Kernel | str = Kernel.AUTO, warps_per_block: int = 0,
         states_per_lane: int = 0, channels_per_lane: int = 0) -> tuple[Kernel, int]:
    """The tier and grid the library would launch for this call (no GPU needed)."""
    s = _shapes(batch, seqlen, dim, dstate, chunk_len)
    o = Options(int(_kernel(kernel)), int(warps_per_block), int(states_per_lane),
                int(channels_per_lane))
    k, g = ctypes.c_int32(), ctypes.c_int64()
    st = load().ssm_scan_plan(ctypes.byref(s), int(_dtype_code(dtype)), int(gate), int(mask),
                              int(chunk_len > 0), ctypes.byref(o), ctypes.byref(k),
                              ctypes.byref(g))
    if st != 0:
        raise SsmError(st, "ssm_scan_plan")
    return Kernel(k.value), int(g.value)


def _kernel(k) -> Kernel:
    return Kernel[k.upper().replace("-", "_")] if isinstance(k, str) else Kernel(k)


def _dtype_code(dtype) -> DType:
    if isinstance(dtype, str):
        return {"f32": DType.F32, "fp32": DType.F32, "float32": DType.F32,
                "bf16": DType.BF16, "bfloat16": DType.BF16}[dtype]
    import torch
    if dtype == torch.float32:
        return DType.F32
    if dtype == torch.bfloat16:
        return DType.BF16
    raise TypeError(f"unsupported dtype {dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, shape, dtype, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def scan_fwd(x, delta, A, B, C, D=None, z=None, valid_len=None, *, chunk_len: int = 0,
             out=None, out_states=None, kernel: Kernel | str = Kernel.AUTO,
             warps_per_block: int = 0, states_per_lane: int = 0, channels_per_lane: int = 0,
             stream=None, h0=None, want_final: bool = False, out_final=None, dt_bias=None,
             delta_softplus: bool = False, delta_clamp=None, time_segments: int | None = None):
    """The fused selective-scan forward on CUDA tensors.

    x, delta, z: [batch, L, dim]; B, C: [batch, L, dstate] (fp32 or bf16, all the
    same dtype); A: fp32 [dim, dstate]; D: fp32 [dim]; valid_len: int32 [batch].
    Returns ``(y, states)`` with y like x and states fp32
    [batch, ceil(L/chunk_len), dim, dstate] (None when chunk_len == 0).
    ``h0`` (fp32 [batch, dim, dstate]) is the state before the first step
    (zeros when None); with ``want_final`` the result is ``(y, states, final)``,
    final being the fp32 state after the last step.  ``dt_bias`` (fp32 [dim]),
    ``delta_softplus`` and ``delta_clamp`` = (lo, hi) ask for the fused
    step-size preparation of delta.
    With the library's choice of tier (AUTO, no launch-shape options, no
    step-size preparation) and ``time_segments`` None, a sequence whose batch
    rows leave most of the GPU idle runs through the time split
    (scan_fwd_split, workspace from PyTorch); ``time_segments`` = 1 keeps one
    segment, k > 1 asks for k.
    Runs on ``stream`` (default: the current PyTorch stream of x's device).
    """
    import torch
    lib = load()
    if x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    plain = (_kernel(kernel) == Kernel.AUTO and not (warps_per_block or states_per_lane
             or channels_per_lane) and dt_bias is None and not delta_softplus
             and delta_clamp is None)
    if plain and time_segments != 1 and x.dim() == 3 and B.dim() == 3:
        segs = time_segments or 0
        try:
            with torch.cuda.device(x.device):
                n, _ = split_plan(x.shape[0], x.shape[1], x.shape[2], B.shape[-1], dtype=x.dtype,
                                  gate=z is not None, time_segments=segs)
        except SsmError:
            n = 1  # the split does not take this shape: the tiers below do
        if n > 1:
            return scan_fwd_split(x, delta, A, B, C, D, z, valid_len, time_segments=segs,
                                  chunk_len=chunk_len, h0=h0, want_final=want_final, out=out,
                                  out_states=out_states, out_final=out_final, stream=stream)
    dev, dt = x.device, x.dtype
    code = _dtype_code(dt)
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    _check(x, "x", (batch, L, dim), dt, dev)
    _check(delta, "delta", (batch, L, dim), dt, dev)
    _check(B, "B", (batch, L, dstate), dt, dev)
    _check(C, "C", (batch, L, dstate), dt, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if z is not None:
        _check(z, "z", (batch, L, dim), dt, dev)
    if valid_len is not None:
        _check(valid_len, "valid_len", (batch,), torch.int32, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", (batch, L, dim), dt, dev)
    states = None
    if chunk_len > 0:
        nch = (L + chunk_len - 1) // chunk_len
        states = (torch.empty((batch, nch, dim, dstate), dtype=torch.float32, device=dev)
                  if out_states is None else out_states)
        _check(states, "out_states", (batch, nch, dim, dstate), torch.float32, dev)
    if h0 is not None:
        _check(h0, "h0", (batch, dim, dstate), torch.float32, dev)
    final = None
    if want_final or out_final is not None:
        final = (torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
                 if out_final is None else out_final)
        _check(final, "out_final", (batch, dim, dstate), torch.float32, dev)
    s = _shapes(batch, L, dim, dstate, chunk_len)
    o = Options(int(_kernel(kernel)), int(warps_per_block), int(states_per_lane),
                int(channels_per_lane))
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    prep = _prep(dt_bias, delta_softplus, delta_clamp, dim, dev)
    with torch.cuda.device(dev):
        if prep is not None:
            st = lib.ssm_scan_fwd_prep(_ptr(x), _ptr(delta), ctypes.byref(prep), _ptr(A), _ptr(B),
                                       _ptr(C), _ptr(D), _ptr(z), _ptr(valid_len), _ptr(h0),
                                       _ptr(y), _ptr(states), _ptr(final), ctypes.byref(s),
                                       int(code), ctypes.c_void_p(handle), ctypes.byref(o))
        elif h0 is None and final is None:
            st = lib.ssm_scan_fwd_ex(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(z), _ptr(valid_len), _ptr(y), _ptr(states),
                                     ctypes.byref(s), int(code), ctypes.c_void_p(handle),
                                     ctypes.byref(o))
        else:
            st = lib.ssm_scan_fwd_carry(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                        _ptr(D), _ptr(z), _ptr(valid_len), _ptr(h0), _ptr(y),
                                        _ptr(states), _ptr(final), ctypes.byref(s), int(code),
                                        ctypes.c_void_p(handle), ctypes.byref(o))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd_prep" if prep is not None else
                       "ssm_scan_fwd_carry" if final is not None or h0 is not None
                       else "ssm_scan_fwd")
    if want_final or out_final is not None:
        return y, states, final
    return y, states


def split_plan(batch, seqlen, dim, dstate, *, dtype="f32", gate=False,
               time_segments: int = 0) -> tuple[int, int]:
    """(segments, workspace bytes) of scan_fwd_split for these shapes
    (time_segments 0 = the library's choice for the current device)."""
    s = _shapes(batch, seqlen, dim, dstate, 0)
    segs, nbytes = ctypes.c_int64(), ctypes.c_size_t()
    st = load().ssm_scan_split_plan(ctypes.byref(s), int(_dtype_code(dtype)), int(gate),
                                    int(time_segments), ctypes.byref(segs), ctypes.byref(nbytes))
    if st != 0:
        raise SsmError(st, "ssm_scan_split_plan")
    return int(segs.value), int(nbytes.value)


def scan_fwd_split(x, delta, A, B, C, D=None, z=None, valid_len=None, *, time_segments: int = 0,
                   chunk_len: int = 0, h0=None, want_final: bool = False, workspace=None,
                   out=None, out_states=None, out_final=None, stream=None):
    """The forward with each sequence split into segments run by separate CTAs
    (aggregate pass, carry, output pass).  Arguments and results as scan_fwd
    with h0 / want_final; ``workspace`` (a CUDA uint8 tensor) is allocated
    here when None and the plan needs one."""
    import torch
    lib = load()
    if x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    dev, dt = x.device, x.dtype
    code = _dtype_code(dt)
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    for name, t, shape, tdt in (("x", x, (batch, L, dim), dt), ("delta", delta, (batch, L, dim), dt),
                                ("B", B, (batch, L, dstate), dt), ("C", C, (batch, L, dstate), dt),
                                ("A", A, (dim, dstate), torch.float32)):
        _check(t, name, shape, tdt, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if z is not None:
        _check(z, "z", (batch, L, dim), dt, dev)
    if valid_len is not None:
        _check(valid_len, "valid_len", (batch,), torch.int32, dev)
    if h0 is not None:
        _check(h0, "h0", (batch, dim, dstate), torch.float32, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", (batch, L, dim), dt, dev)
    states = None
    if chunk_len > 0:
        nch = (L + chunk_len - 1) // chunk_len
        states = (torch.empty((batch, nch, dim, dstate), dtype=torch.float32, device=dev)
                  if out_states is None else out_states)
        _check(states, "out_states", (batch, nch, dim, dstate), torch.float32, dev)
    final = None
    if want_final or out_final is not None:
        final = (torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
                 if out_final is None else out_final)
        _check(final, "out_final", (batch, dim, dstate), torch.float32, dev)
    with torch.cuda.device(dev):
        _, need = split_plan(batch, L, dim, dstate, dtype=dt, gate=z is not None,
                             time_segments=time_segments)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if workspace is not None and (workspace.device != dev or workspace.dtype != torch.uint8
                                      or not workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous uint8 tensor on x's device")
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        s = _shapes(batch, L, dim, dstate, chunk_len)
        st = lib.ssm_scan_fwd_split(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                    _ptr(z), _ptr(valid_len), _ptr(h0), _ptr(y), _ptr(states),
                                    _ptr(final), ctypes.byref(s), int(code), int(time_segments),
                                    _ptr(workspace),
                                    workspace.numel() if workspace is not None else 0,
                                    ctypes.c_void_p(handle))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd_split")
    if want_final or out_final is not None:
        return y, states, final
    return y, states


def host_workspace_bytes(batch, seqlen, dim, dstate, *, dtype="f32", has_D=True, gate=False,
                         mask=False, chunk_len=0) -> int:
    s = _shapes(batch, seqlen, dim, dstate, chunk_len)
    return int(load().ssm_scan_host_workspace_bytes(ctypes.byref(s), int(_dtype_code(dtype)),
                                                    int(has_D), int(gate), int(mask),
                                                    int(chunk_len > 0)))


def _check_host_inputs(x, delta, A, B, C, D, z, valid_len):
    """Dtype, shape, device (CPU) and contiguity of every input of the host
    entry points: the library reads each as a dense host array of that shape."""
    import torch
    cpu = torch.device("cpu")
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"x: dtype {x.dtype}, expected float32 or bfloat16")
    if x.dim() != 3:
        raise ValueError(f"x: shape {tuple(x.shape)}, expected [batch, L, dim]")
    dt = x.dtype
    batch, L, dim = x.shape
    if B.dim() != 3:
        raise ValueError(f"B: shape {tuple(B.shape)}, expected [batch, L, dstate]")
    dstate = B.shape[-1]
    for name, t, shape, tdt in (("x", x, (batch, L, dim), dt), ("delta", delta, (batch, L, dim), dt),
                                ("B", B, (batch, L, dstate), dt), ("C", C, (batch, L, dstate), dt),
                                ("A", A, (dim, dstate), torch.float32)):
        _check(t, name, shape, tdt, cpu)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, cpu)
    if z is not None:
        _check(z, "z", (batch, L, dim), dt, cpu)
    if valid_len is not None:
        _check(valid_len, "valid_len", (batch,), torch.int32, cpu)


def scan_fwd_host(x, delta, A, B, C, D=None, z=None, valid_len=None, *, chunk_len: int = 0,
                  out=None, out_states=None, workspace=None, stream=None):
    """End-to-end form on HOST tensors (pinned CPU tensors give async copies).

    The library copies inputs into ``workspace`` (a CUDA uint8 tensor; allocated
    here when None), runs the forward and copies y (and states) back into
    ``out`` / ``out_states`` (CPU tensors; allocated pinned when None), all on
    ``stream``.  The call returns once the work is enqueued: synchronise the
    stream before reading the outputs."""
    import torch
    lib = load()
    _check_host_inputs(x, delta, A, B, C, D, z, valid_len)
    dt = x.dtype
    code = _dtype_code(dt)
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    y = torch.empty((batch, L, dim), dtype=dt, pin_memory=True) if out is None else out
    _check(y, "out", (batch, L, dim), dt, torch.device("cpu"))
    states = None
    if chunk_len > 0:
        nch = (L + chunk_len - 1) // chunk_len
        states = (torch.empty((batch, nch, dim, dstate), dtype=torch.float32, pin_memory=True)
                  if out_states is None else out_states)
        _check(states, "out_states", (batch, nch, dim, dstate), torch.float32,
               torch.device("cpu"))
    need = host_workspace_bytes(batch, L, dim, dstate, dtype=dt, has_D=D is not None,
                                gate=z is not None, mask=valid_len is not None,
                                chunk_len=chunk_len)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    if workspace.device.type != "cuda" or workspace.dtype != torch.uint8 \
            or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    s = _shapes(batch, L, dim, dstate, chunk_len)
    with torch.cuda.device(workspace.device):
        st = lib.ssm_scan_fwd_host(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                   _ptr(z), _ptr(valid_len), _ptr(y), _ptr(states),
                                   ctypes.byref(s), int(code), _ptr(workspace),
                                   workspace.numel(), ctypes.c_void_p(handle))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd_host")
    return y, states


def decode_step(x, delta, A, B, C, D=None, z=None, *, state, out=None, stream=None,
                dt_bias=None, delta_softplus: bool = False, delta_clamp=None):
    """One step of the recurrence on a carried state, in place (decode).

    x, delta, z: [batch, dim]; B, C: [batch, dstate] (fp32 or bf16, all the
    same dtype); A: fp32 [dim, dstate]; D: fp32 [dim]; state: fp32
    [batch, dim, dstate], updated in place.  Returns y [batch, dim].  The
    step-size preparation arguments are those of scan_fwd."""
    import torch
    lib = load()
    if x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    dev, dt = x.device, x.dtype
    code = _dtype_code(dt)
    batch, dim = x.shape
    dstate = B.shape[-1]
    _check(x, "x", (batch, dim), dt, dev)
    _check(delta, "delta", (batch, dim), dt, dev)
    _check(B, "B", (batch, dstate), dt, dev)
    _check(C, "C", (batch, dstate), dt, dev)
    _check(A, "A", (dim, dstate), torch.float32, dev)
    _check(state, "state", (batch, dim, dstate), torch.float32, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if z is not None:
        _check(z, "z", (batch, dim), dt, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", (batch, dim), dt, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    prep = _prep(dt_bias, delta_softplus, delta_clamp, dim, dev)
    with torch.cuda.device(dev):
        st = lib.ssm_decode_step_prep(_ptr(x), _ptr(delta),
                                      ctypes.byref(prep) if prep is not None else None, _ptr(A),
                                      _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(state), _ptr(y),
                                      batch, dim, dstate, int(code), ctypes.c_void_p(handle))
    if st != 0:
        raise SsmError(st, "ssm_decode_step")
    return y


def scan_bwd(x, delta, A, B, C, D=None, z=None, valid_len=None, *, chunk_states, chunk_len: int,
             dy, h0=None, want_dh0: bool = False, stream=None) -> dict:
    """Every gradient of sum(dy * y) for the forward on these inputs (delta used
    as given).  ``chunk_states`` are the boundary states the forward wrote with
    the same ``chunk_len`` (1 .. 512).  Returns a dict: dx, ddelta, dz (None
    without gate) like x; dA, dB, dC, dD (None without D), dh0 (when wanted) in fp32."""
    import torch
    lib = load()
    dev, dt = x.device, x.dtype
    code = _dtype_code(dt)
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    nch = (L + chunk_len - 1) // chunk_len
    for name, t, shape, tdt in (("x", x, (batch, L, dim), dt), ("delta", delta, (batch, L, dim), dt),
                                ("B", B, (batch, L, dstate), dt), ("C", C, (batch, L, dstate), dt),
                                ("A", A, (dim, dstate), torch.float32), ("dy", dy, (batch, L, dim), dt),
                                ("chunk_states", chunk_states, (batch, nch, dim, dstate),
                                 torch.float32)):
        _check(t, name, shape, tdt, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if z is not None:
        _check(z, "z", (batch, L, dim), dt, dev)
    if valid_len is not None:
        _check(valid_len, "valid_len", (batch,), torch.int32, dev)
    if h0 is not None:
        _check(h0, "h0", (batch, dim, dstate), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x),
           "dz": torch.empty_like(x) if z is not None else None,
           "dA": torch.empty((dim, dstate), **f32), "dB": torch.empty((batch, L, dstate), **f32),
           "dC": torch.empty((batch, L, dstate), **f32),
           "dD": torch.empty((dim,), **f32) if D is not None else None,
           "dh0": torch.empty((batch, dim, dstate), **f32) if want_dh0 else None}
    s = _shapes(batch, L, dim, dstate, chunk_len)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(dev):
        st = lib.ssm_scan_bwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                              _ptr(valid_len), _ptr(h0), _ptr(chunk_states), _ptr(dy),
                              _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA"]),
                              _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
                              _ptr(out["dh0"]), ctypes.byref(s), int(code),
                              ctypes.c_void_p(handle))
    if st != 0:
        raise SsmError(st, "ssm_scan_bwd")
    return out


def ssd_fwd(x, delta, A, B, C, D=None, z=None, valid_len=None, *, nheads: int, h0=None,
            want_final: bool = False, out=None, out_final=None, stream=None):
    """The SSD form of the scan (one decay per head) on the tensor cores.

    x, z: bf16 [batch, L, nheads * headdim]; delta: bf16 [batch, L, nheads];
    A: fp32 [nheads]; B, C: bf16 [batch, L, dstate]; D: fp32 [nheads * headdim];
    valid_len: int32 [batch]; h0: fp32 [batch, nheads * headdim, dstate].
    Returns y, or (y, final_state) with ``want_final``."""
    import torch
    lib = load()
    if x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor")
    dev, dt = x.device, x.dtype
    code = _dtype_code(dt)
    batch, L, dim = x.shape
    if dim % nheads:
        raise ValueError("the channel count must be a multiple of nheads")
    headdim = dim // nheads
    dstate = B.shape[-1]
    for name, t, shape, tdt in (("x", x, (batch, L, dim), dt), ("delta", delta, (batch, L, nheads), dt),
                                ("B", B, (batch, L, dstate), dt), ("C", C, (batch, L, dstate), dt),
                                ("A", A, (nheads,), torch.float32)):
        _check(t, name, shape, tdt, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if z is not None:
        _check(z, "z", (batch, L, dim), dt, dev)
    if valid_len is not None:
        _check(valid_len, "valid_len", (batch,), torch.int32, dev)
    if h0 is not None:
        _check(h0, "h0", (batch, dim, dstate), torch.float32, dev)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", (batch, L, dim), dt, dev)
    fin = None
    if want_final:
        fin = torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev) \
            if out_final is None else out_final
        _check(fin, "out_final", (batch, dim, dstate), torch.float32, dev)
    s = SsdShapes(batch, L, nheads, headdim, dstate)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(dev):
        st = lib.ssm_ssd_fwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                             _ptr(valid_len), _ptr(h0), _ptr(y), _ptr(fin), ctypes.byref(s),
                             int(code), ctypes.c_void_p(handle))
    if st != 0:
        raise SsmError(st, "ssm_ssd_fwd")
    return (y, fin) if want_final else y


def static_capacity() -> int:
    """Bytes of the fixed workspace of scan_fwd_host_static."""
    return int(load().ssm_scan_host_static_capacity())


def scan_fwd_host_static(x, delta, A, B, C, D=None, z=None, valid_len=None, *, out, chunk_len=0,
                         out_states=None, stream=None):
    """scan_fwd_host without any allocation: the library's fixed device
    workspace, every step on ``stream`` (default: the current stream of the
    current device).  ``out`` (and ``out_states`` when chunk_len > 0) are
    caller-owned host tensors; nothing is allocated here.  The call runs with
    the stream's device current.  Calls that overlap in time race on the
    workspace."""
    import torch
    lib = load()
    _check_host_inputs(x, delta, A, B, C, D, z, valid_len)
    dt = x.dtype
    batch, L, dim = x.shape
    dstate = B.shape[-1]
    cpu = torch.device("cpu")
    _check(out, "out", (batch, L, dim), dt, cpu)
    if chunk_len > 0:
        nch = (L + chunk_len - 1) // chunk_len
        if out_states is None:
            raise ValueError("out_states is required when chunk_len > 0")
        _check(out_states, "out_states", (batch, nch, dim, dstate), torch.float32, cpu)
    if stream is None:
        stream = torch.cuda.current_stream()
    if not hasattr(stream, "device"):
        raise TypeError("stream must be a torch.cuda.Stream")
    s = _shapes(batch, L, dim, dstate, chunk_len)
    with torch.cuda.device(stream.device):
        st = lib.ssm_scan_fwd_host_static(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                          _ptr(z), _ptr(valid_len), _ptr(out), _ptr(out_states),
                                          ctypes.byref(s), int(_dtype_code(dt)),
                                          ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise SsmError(st, "ssm_scan_fwd_host_static")
    return out, out_states
