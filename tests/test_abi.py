"""C ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every function include/ssmscan.h declares, and rejects bad arguments with a
status before anything is launched."""
import ctypes

import pytest

from selective_state_space_fwd_gb300 import _binding as Bd

EXPECTED = {"ssm_scan_fwd", "ssm_scan_fwd_ex", "ssm_scan_fwd_carry", "ssm_scan_fwd_prep",
            "ssm_decode_step", "ssm_decode_step_prep", "ssm_scan_bwd", "ssm_scan_plan",
            "ssm_scan_fwd_host_static", "ssm_scan_host_static_capacity", "ssm_scan_fwd_host",
            "ssm_scan_host_workspace_bytes", "ssm_chunk_count", "ssm_status_string",
            "ssm_kernel_name", "ssm_version", "ssm_check_device_errors", "ssm_ssd_fwd",
            "ssm_selftest_wait_timeout", "ssm_scan_fwd_split", "ssm_scan_split_plan"}


def test_every_declared_symbol_is_exported(ssmlib):
    declared = set(Bd.declared_functions())
    assert EXPECTED <= declared, EXPECTED - declared
    lib = ctypes.CDLL(Bd.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in ssmscan.h but not exported"


def test_status_and_kernel_strings(ssmlib):
    for s in Bd.Status:
        assert Bd.status_string(s) and Bd.status_string(s) != "unknown status"
    for k in Bd.Kernel:
        assert Bd.kernel_name(k) != "unknown"
    assert Bd.version().count(".") == 2


def test_chunk_count(ssmlib):
    assert Bd.chunk_count(2048, 256) == 8
    assert Bd.chunk_count(2049, 256) == 9
    assert Bd.chunk_count(5, 0) == 0
    assert Bd.chunk_count(1, 7) == 1


FAKE = 0x10000  # never dereferenced: validation returns before any device work


def _call(x=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, valid=None, y=FAKE,
          states=None, shapes=(2, 8, 4, 16, 0), dtype=0, kernel=0, wpb=0, spl=0, cpl=0, shapes_ptr=True):
    lib = Bd.load()
    s = Bd.Shapes(*shapes)
    o = Bd.Options(kernel, wpb, spl, cpl)
    P = ctypes.c_void_p
    return lib.ssm_scan_fwd_ex(P(x), P(delta), P(A), P(B), P(C), P(D), P(z), P(valid), P(y),
                               P(states), ctypes.byref(s) if shapes_ptr else None, dtype, None,
                               ctypes.byref(o))


@pytest.mark.parametrize("kw,status", [
    (dict(shapes_ptr=False), Bd.Status.ERR_NULL),
    (dict(x=None), Bd.Status.ERR_NULL),
    (dict(delta=None), Bd.Status.ERR_NULL),
    (dict(A=None), Bd.Status.ERR_NULL),
    (dict(B=None), Bd.Status.ERR_NULL),
    (dict(C=None), Bd.Status.ERR_NULL),
    (dict(y=None), Bd.Status.ERR_NULL),
    (dict(shapes=(0, 8, 4, 16, 0)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, -1, 4, 16, 0)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 0, 4, 16, 0)), Bd.Status.ERR_SHAPE),  # an empty sequence
    (dict(shapes=(2, 8, 0, 16, 0)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 8, 4, 0, 0)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 8, 4, 16, -5)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(1 << 40, 1 << 20, 1 << 20, 16, 0)), Bd.Status.ERR_SHAPE),
    (dict(states=FAKE, shapes=(2, 8, 4, 16, 0)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 8, 4, 3, 0)), Bd.Status.ERR_UNSUPPORTED),
    (dict(shapes=(2, 8, 4, 128, 0)), Bd.Status.ERR_UNSUPPORTED),
    (dict(dtype=7), Bd.Status.ERR_UNSUPPORTED),
    (dict(kernel=99), Bd.Status.ERR_UNSUPPORTED),
    (dict(wpb=3), Bd.Status.ERR_UNSUPPORTED),
    (dict(wpb=-1), Bd.Status.ERR_UNSUPPORTED),
    (dict(spl=3), Bd.Status.ERR_UNSUPPORTED),
    (dict(spl=32), Bd.Status.ERR_UNSUPPORTED),
    (dict(cpl=3), Bd.Status.ERR_UNSUPPORTED),
    (dict(cpl=1), Bd.Status.ERR_UNSUPPORTED),
    (dict(cpl=8), Bd.Status.ERR_UNSUPPORTED),
    (dict(x=FAKE + 2), Bd.Status.ERR_ALIGN),
    (dict(y=FAKE + 1, dtype=1), Bd.Status.ERR_ALIGN),
    (dict(A=FAKE + 2, dtype=1), Bd.Status.ERR_ALIGN),
    (dict(D=FAKE + 3), Bd.Status.ERR_ALIGN),
    (dict(valid=FAKE + 2), Bd.Status.ERR_ALIGN),
    (dict(states=FAKE + 2, shapes=(2, 8, 4, 16, 4)), Bd.Status.ERR_ALIGN),
])
def test_argument_errors_return_status(ssmlib, kw, status):
    assert _call(**kw) == status


def _carry(h0=None, final=None, **kw):
    lib = Bd.load()
    s = Bd.Shapes(2, 8, 4, 16, 0)
    o = Bd.Options(0, 0, 0, 0)
    P = ctypes.c_void_p
    return lib.ssm_scan_fwd_carry(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, None, None,
                                  P(h0), P(FAKE), None, P(final), ctypes.byref(s), 0, None,
                                  ctypes.byref(o))


@pytest.mark.parametrize("kw,status", [
    (dict(h0=FAKE + 2), Bd.Status.ERR_ALIGN),
    (dict(final=FAKE + 1), Bd.Status.ERR_ALIGN),
    (dict(h0=FAKE + 6, final=FAKE), Bd.Status.ERR_ALIGN),
])
def test_carry_argument_errors_return_status(ssmlib, kw, status):
    assert _carry(**kw) == status


def _decode(x=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, state=FAKE, y=FAKE,
            batch=2, dim=4, dstate=16, dtype=0):
    P = ctypes.c_void_p
    return Bd.load().ssm_decode_step(P(x), P(delta), P(A), P(B), P(C), P(D), P(z), P(state),
                                     P(y), batch, dim, dstate, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), Bd.Status.ERR_NULL),
    (dict(state=None), Bd.Status.ERR_NULL),
    (dict(y=None), Bd.Status.ERR_NULL),
    (dict(batch=0), Bd.Status.ERR_SHAPE),
    (dict(dim=-3), Bd.Status.ERR_SHAPE),
    (dict(dstate=3), Bd.Status.ERR_UNSUPPORTED),
    (dict(dstate=128), Bd.Status.ERR_UNSUPPORTED),
    (dict(dtype=5), Bd.Status.ERR_UNSUPPORTED),
    (dict(state=FAKE + 8), Bd.Status.ERR_ALIGN),
    (dict(A=FAKE + 4), Bd.Status.ERR_ALIGN),
    (dict(x=FAKE + 1, dtype=1), Bd.Status.ERR_ALIGN),
    (dict(batch=1 << 40, dim=1 << 30), Bd.Status.ERR_SHAPE),
])
def test_decode_argument_errors_return_status(ssmlib, kw, status):
    assert _decode(**kw) == status


def _prep_call(prep):
    lib = Bd.load()
    s = Bd.Shapes(2, 8, 4, 16, 0)
    o = Bd.Options(0, 0, 0, 0)
    P = ctypes.c_void_p
    return lib.ssm_scan_fwd_prep(P(FAKE), P(FAKE), ctypes.byref(prep), P(FAKE), P(FAKE), P(FAKE),
                                 None, None, None, None, P(FAKE), None, None, ctypes.byref(s), 0,
                                 None, ctypes.byref(o))


@pytest.mark.parametrize("prep,status", [
    (Bd.DeltaPrep(FAKE + 2, 0, 0, 0.0, 0.0), Bd.Status.ERR_ALIGN),
    (Bd.DeltaPrep(None, 2, 0, 0.0, 0.0), Bd.Status.ERR_UNSUPPORTED),
    (Bd.DeltaPrep(None, 1, 3, 0.0, 1.0), Bd.Status.ERR_UNSUPPORTED),
    (Bd.DeltaPrep(None, 1, 1, 1.0, 0.5), Bd.Status.ERR_SHAPE),
    (Bd.DeltaPrep(None, 1, 1, float("nan"), 0.5), Bd.Status.ERR_SHAPE),
])
def test_prep_argument_errors_return_status(ssmlib, prep, status):
    assert _prep_call(prep) == status


def _bwd(shapes=(2, 8, 4, 16, 4), z=None, dz=None, states=FAKE, dA=FAKE, x=FAKE, dtype=0):
    P = ctypes.c_void_p
    s = Bd.Shapes(*shapes)
    return Bd.load().ssm_scan_bwd(P(x), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(z), None,
                                  None, P(states), P(FAKE), P(FAKE), P(FAKE), P(dA), P(FAKE),
                                  P(FAKE), None, P(dz), None, ctypes.byref(s), dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(shapes=(2, 8, 4, 16, 0)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 0, 4, 16, 4)), Bd.Status.ERR_SHAPE),  # an empty sequence
    (dict(shapes=(2, 8, 4, 16, 513)), Bd.Status.ERR_UNSUPPORTED),
    (dict(states=None), Bd.Status.ERR_NULL),
    (dict(dA=None), Bd.Status.ERR_NULL),
    (dict(z=FAKE, dz=None), Bd.Status.ERR_NULL),
    (dict(x=FAKE + 2), Bd.Status.ERR_ALIGN),
    (dict(dA=FAKE + 2), Bd.Status.ERR_ALIGN),
])
def test_bwd_argument_errors_return_status(ssmlib, kw, status):
    assert _bwd(**kw) == status


def _ssd(x=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, valid=None, h0=None,
         y=FAKE, final=None, shapes=(2, 256, 4, 64, 128), dtype=1, shapes_ptr=True):
    P = ctypes.c_void_p
    s = Bd.SsdShapes(*shapes)
    return Bd.load().ssm_ssd_fwd(P(x), P(delta), P(A), P(B), P(C), P(D), P(z), P(valid), P(h0),
                                 P(y), P(final), ctypes.byref(s) if shapes_ptr else None, dtype,
                                 None)


@pytest.mark.parametrize("kw,status", [
    (dict(shapes_ptr=False), Bd.Status.ERR_NULL),
    (dict(x=None), Bd.Status.ERR_NULL),
    (dict(delta=None), Bd.Status.ERR_NULL),
    (dict(A=None), Bd.Status.ERR_NULL),
    (dict(y=None), Bd.Status.ERR_NULL),
    (dict(shapes=(0, 256, 4, 64, 128)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, -1, 4, 64, 128)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 0, 4, 64, 128)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(2, 256, 0, 64, 128)), Bd.Status.ERR_SHAPE),
    (dict(shapes=(1 << 40, 1 << 30, 4, 64, 128)), Bd.Status.ERR_SHAPE),
    (dict(dtype=0), Bd.Status.ERR_UNSUPPORTED),
    (dict(dtype=7), Bd.Status.ERR_UNSUPPORTED),
    (dict(shapes=(2, 256, 4, 32, 128)), Bd.Status.ERR_UNSUPPORTED),
    (dict(shapes=(2, 256, 4, 64, 16)), Bd.Status.ERR_UNSUPPORTED),
    (dict(x=FAKE + 8), Bd.Status.ERR_ALIGN),
    (dict(B=FAKE + 2), Bd.Status.ERR_ALIGN),
    (dict(y=FAKE + 4), Bd.Status.ERR_ALIGN),
    (dict(z=FAKE + 8), Bd.Status.ERR_ALIGN),
    (dict(delta=FAKE + 1), Bd.Status.ERR_ALIGN),
    (dict(h0=FAKE + 2), Bd.Status.ERR_ALIGN),
])
def test_ssd_argument_errors_return_status(ssmlib, kw, status):
    assert _ssd(**kw) == status


def test_plan_serial_always_available(ssmlib):
    for n in (1, 2, 4, 8, 16, 32, 64):
        k, g = Bd.plan(3, 100, 70, n, kernel="serial")
        assert k == Bd.Kernel.SERIAL and g == (3 * 70 + 127) // 128


def test_plan_auto_picks_a_tier(ssmlib):
    for n in (1, 16, 64):
        k, g = Bd.plan(8, 4096, 1024, n)
        assert k in (Bd.Kernel.SERIAL, Bd.Kernel.WARPSCAN, Bd.Kernel.STREAM) and g > 0


def test_host_workspace_bytes(ssmlib):
    b = Bd.host_workspace_bytes(2, 8, 4, 16, dtype="f32", has_D=True, gate=True, mask=True,
                                chunk_len=4)
    # x, delta, z; B, C; A; D; valid_len; y; chunk states; two carried states
    need = 3 * 2 * 8 * 4 * 4 + 2 * 2 * 8 * 16 * 4 + 4 * 16 * 4 + 4 * 4 + 2 * 4 + 2 * 8 * 4 * 4 \
        + 2 * 2 * 4 * 16 * 4 + 2 * 2 * 4 * 16 * 4
    assert need <= b <= need + 12 * 256
    assert Bd.host_workspace_bytes(0, 8, 4, 16) == 0


def test_no_fallback_without_the_library(monkeypatch, tmp_path):
    """Without the compiled library every entry fails loudly: there is no CPU path."""
    import numpy as np
    import torch
    monkeypatch.setattr(Bd, "_lib", None)
    monkeypatch.setattr(Bd, "LIB_PATH", str(tmp_path / "libssmscan.so"))
    with pytest.raises(ImportError):
        Bd.load()
    x = torch.from_numpy(np.zeros((1, 4, 2), np.float32))
    with pytest.raises(ImportError):
        Bd.scan_fwd(x, x, torch.zeros(2, 4), torch.zeros(1, 4, 4), torch.zeros(1, 4, 4))
    with pytest.raises(ImportError):
        Bd.ssd_fwd(x, x, torch.zeros(1), torch.zeros(1, 4, 4), torch.zeros(1, 4, 4), nheads=1)


def test_host_workspace_bytes_overflow_is_refused(ssmlib):
    """A workspace whose size would wrap size_t is reported as 0 (and refused by
    both host entry points) rather than as a small wrapped total."""
    # every element count is below 2^60, but six regions of them do not fit in 64 bits
    dim = (1 << 20) - 1  # x, delta, z, y: four regions of almost 2^62 bytes each
    assert Bd.host_workspace_bytes(1 << 20, 1 << 20, dim, 16, dtype="f32", gate=True) == 0
    lib = Bd.load()
    s = Bd.Shapes(1 << 20, 1 << 20, dim, 16, 0)
    P = ctypes.c_void_p
    st = lib.ssm_scan_fwd_host_static(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None,
                                      P(FAKE), None, P(FAKE), None, ctypes.byref(s), 0, None)
    assert st == Bd.Status.ERR_SHAPE
    st = lib.ssm_scan_fwd_host(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), None,
                               P(FAKE), None, ctypes.byref(s), 0, P(0x100000), 1 << 62, None)
    assert st == Bd.Status.ERR_SHAPE


def _host_args(**over):
    import torch
    a = dict(x=torch.zeros(2, 8, 4), delta=torch.zeros(2, 8, 4), A=torch.zeros(4, 16),
             B=torch.zeros(2, 8, 16), C=torch.zeros(2, 8, 16), D=torch.zeros(4),
             z=None, valid_len=None)
    a.update(over)
    return a


@pytest.mark.parametrize("entry", ["scan_fwd_host", "scan_fwd_host_static"])
@pytest.mark.parametrize("over,exc", [
    (lambda t: dict(A=t.zeros(4, 16, dtype=t.float64)), TypeError),
    (lambda t: dict(x=t.zeros(2, 4, 8).transpose(1, 2)), ValueError),
    (lambda t: dict(delta=t.zeros(2, 8, 4, dtype=t.bfloat16)), TypeError),
    (lambda t: dict(valid_len=t.zeros(2, dtype=t.int64)), TypeError),
    (lambda t: dict(D=t.zeros(5)), ValueError),
    (lambda t: dict(B=t.zeros(2, 8, 16)[:, :, :8]), ValueError),
    (lambda t: dict(x=t.zeros(2, 8, 4, dtype=t.float64)), TypeError),
])
def test_host_entries_check_every_input(ssmlib, entry, over, exc):
    """Both host entry points refuse a wrong dtype, shape or layout of any input
    before the library reads the host buffers (no GPU is touched)."""
    import torch
    a = _host_args(**over(torch))
    fn = getattr(Bd, entry)
    kw = {"out": torch.zeros(2, 8, 4)} if entry == "scan_fwd_host_static" else {}
    with pytest.raises(exc):
        fn(a["x"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["valid_len"], **kw)


def test_selftest_poll_bound(ssmlib):
    """The bounded-wait self-test refuses a poll count above its bound before
    launching anything."""
    assert Bd.load().ssm_selftest_wait_timeout((1 << 20) + 1, None) == Bd.Status.ERR_SHAPE


def test_split_argument_errors_return_status(ssmlib):
    """The time-split entry validates before launching anything."""
    lib = Bd.load()
    P = ctypes.c_void_p
    s = Bd.Shapes(2, 640, 32, 16, 0)

    def call(x=FAKE, y=FAKE, segs=2, ws=None, nbytes=0, shapes=s, h0=None):
        return lib.ssm_scan_fwd_split(P(x), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, None, None,
                                      P(h0), P(y), None, None, ctypes.byref(shapes), 0, segs, P(ws),
                                      nbytes, None)
    assert call(x=None) == Bd.Status.ERR_NULL
    assert call(y=None) == Bd.Status.ERR_NULL
    assert call(segs=-1) == Bd.Status.ERR_SHAPE
    assert call(h0=FAKE + 2) == Bd.Status.ERR_ALIGN
    assert call(shapes=Bd.Shapes(2, 0, 32, 16, 0)) == Bd.Status.ERR_SHAPE
    with pytest.raises(Bd.SsmError) as ei:  # checked before the plan looks at the device
        Bd.split_plan(2, 640, 32, 16, time_segments=-3)
    assert ei.value.status in (Bd.Status.ERR_SHAPE, Bd.Status.ERR_UNSUPPORTED)
