"""Benchmark of the fused selective-scan forward (libssmscan) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2] [--kernel auto]
    python bench.py --impl reference ...     # the fp64 CPU oracle as the reference arm

A step is one forward over one batch of the workload (workload 2 by default:
fp32, batch 8, L 4096, dim 1024, N 16).  Inputs are resident in HBM before the
timed region; each step's kernel is bracketed by CUDA events on the launch
stream and L2 is flushed between steps (a 256 MiB memset outside the events).
Prints one JSON line.  Under torchrun every rank runs its own copy of the
workload (weak scaling, no collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan fwd B·L·D elems/s and achieved % of roofline, 1×GB300"
UNIT = "elements/s"
# Nominal per-SM unit rates of GB300 (sm_103a): MUFU ex2 32 lanes/clk/SM, fp32
# FMA 128 lanes/clk/SM.  Used only when the probe kernels cannot run; the
# roofline normally takes the rates measured on the GPU by unit_rates().
NOMINAL_RATES = {"ex2_per_clk_sm": 32.0, "fp32_per_clk_sm": 128.0, "lds_bytes_per_clk_sm": 128.0}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def measured_capture(kernel: str, workload: str) -> dict | None:
    """The ncu capture of one launch recorded in profiles/traffic.json for this
    kernel and workload, if it was taken on the kernel sources as they are now
    (sha256 of each listed file); None otherwise."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f)
    for e in entries:
        if e.get("kernel") != kernel or e.get("workload") != workload:
            continue
        ok = True
        for rel, sha in e.get("sources", {}).items():
            fp = os.path.join(ROOT, rel)
            if not os.path.exists(fp) or hashlib.sha256(open(fp, "rb").read()).hexdigest() != sha:
                ok = False
                break
        if ok:
            return e
    return None


def measured_traffic(kernel: str, workload: str) -> int | None:
    """DRAM bytes (read + write) per launch from the ncu capture of this kernel
    and workload (measured_capture); None without a current capture."""
    e = measured_capture(kernel, workload)
    return None if e is None else int(e["dram_read_bytes"]) + int(e["dram_write_bytes"])


def smem_port(kernel: str, workload: str, t_meas: float, rates: dict, sms: int,
              sm_mhz: float) -> dict | None:
    """The shared-memory port floor of a launch: ncu's shared-memory wavefronts
    (128 bytes each) of the current capture, delivered at the measured 16-byte
    load rate, with the CTAs spread evenly over the SMs (the busiest SM holds
    ceil(grid / SMs) of them).  `frac` = floor / measured time.  None without a
    current capture that counted the wavefronts."""
    e = measured_capture(kernel, workload)
    if e is None or "smem_wavefronts" not in e or "grid" not in e:
        return None
    wf, grid = float(e["smem_wavefronts"]), int(e["grid"])
    per_sm = -(-grid // sms) * wf / grid
    rate = float(rates.get("lds_bytes_per_clk_sm", NOMINAL_RATES["lds_bytes_per_clk_sm"]))
    floor_s = per_sm * 128.0 / rate / (sm_mhz * 1e6)
    return {"wavefronts": int(wf), "grid": grid, "lds_bytes_per_clk_sm": rate,
            "floor_us": floor_s * 1e6, "frac": floor_s / t_meas}


def algorithmic_counts(w, inp) -> dict:
    """Work the method must do for one forward (independent of the kernel):
    valid (b,t,d) elements, exps, fp32 ops and HBM bytes (inputs read once,
    y and chunk states written once; the O(B L D N) state is never stored)."""
    L, Dm, N = w.seqlen, w.dim, w.dstate
    if inp["valid_len"] is not None:
        valid_rows = int(np.clip(inp["valid_len"], 0, L).sum())
    else:
        valid_rows = w.batch * L
    ev = valid_rows * Dm
    es = 2 if w.dtype == "bf16" else 4
    n_act_in = 3 if w.gate else 2
    nch = (L + w.chunk_len - 1) // w.chunk_len if w.chunk_len else 0
    bytes_ = (n_act_in * ev * es                  # x, delta (, z) of valid steps
              + w.batch * L * Dm * es              # y, every step
              + 2 * valid_rows * N * es            # B, C rows of valid steps
              + Dm * N * 4 + Dm * 4                # A, D
              + (w.batch * 4 if inp["valid_len"] is not None else 0)
              + w.batch * nch * Dm * N * 4)        # chunk states
    exps = ev * N + (ev if w.gate else 0)
    fp32 = 4 * ev * N + 2 * ev + (4 * ev if w.gate else 0)
    return dict(elements=w.batch * L * Dm, valid_elements=ev, n_elements=ev * N, exps=exps,
                fp32_ops=fp32, bytes=bytes_)


def unit_rates() -> tuple[dict, str]:
    """MUFU ex2 results and fp32 FMA lane-operations per SM clock, measured on
    the current GPU by the throughput probes of libssmprobe.so
    (selective_state_space_fwd_gb300/probe/unit_rates.cu); the nominal rates
    when the probes cannot run."""
    import ctypes
    try:
        from selective_state_space_fwd_gb300 import build as B
        lib = ctypes.CDLL(B.build_probe())
        e, f, f2 = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        n = ctypes.c_int()
        rc = lib.ssmprobe_unit_rates(ctypes.byref(e), ctypes.byref(f), ctypes.byref(f2),
                                     ctypes.byref(n))
        if rc != 0 or not (e.value > 0 and f.value > 0 and f2.value > 0):
            raise RuntimeError(f"probe status {rc}")
        ld, ldb = ctypes.c_double(), ctypes.c_double()
        rc = lib.ssmprobe_lds_rates(ctypes.byref(ld), ctypes.byref(ldb))
        if rc != 0 or not (ld.value > 0 and ldb.value > 0):
            raise RuntimeError(f"lds probe status {rc}")
    except Exception as ex:  # no GPU, no compiler: the nominal figures, said so
        return dict(NOMINAL_RATES, error=str(ex)[:80]), "nominal"
    return {"ex2_per_clk_sm": e.value, "fp32_per_clk_sm": max(f.value, f2.value),
            "ffma_per_clk_sm": f.value, "ffma2_lanes_per_clk_sm": f2.value,
            "lds_bytes_per_clk_sm": ld.value, "lds_bcast_bytes_per_clk_sm": ldb.value}, "measured"


def roof(counts, peaks, sms, sm_mhz, rates=NOMINAL_RATES) -> dict:
    hbm = peaks["hbm_gbs"] * 1e9
    clk = sm_mhz * 1e6
    t_hbm = counts["bytes"] / hbm
    t_mufu = counts["exps"] / (rates["ex2_per_clk_sm"] * sms * clk)
    t_fp32 = counts["fp32_ops"] / (rates["fp32_per_clk_sm"] * sms * clk)
    return dict(t_hbm=t_hbm, t_mufu=t_mufu, t_fp32=t_fp32, t_roof=max(t_hbm, t_mufu, t_fp32))


def _rates_text(rates) -> str:
    return (f"{rates['ex2_per_clk_sm']:.1f} ex2 and {rates['fp32_per_clk_sm']:.1f} fp32 "
            f"lanes/clk/SM")


def roofline(counts, t_meas, peaks, rates, sms, sm_mhz) -> dict:
    """The roofline against whichever term binds (the largest of HBM bytes at
    the measured copy bandwidth, exps at the MUFU rate, fp32 operations at the
    fp32 rate): achieved rate of that term, its peak, and their ratio, which
    equals roof time / measured time."""
    r = roof(counts, peaks, sms, sm_mhz, rates)
    clk = sm_mhz * 1e6
    terms = {"hbm": r["t_hbm"], "mufu": r["t_mufu"], "fp32": r["t_fp32"]}
    bound = max(terms, key=terms.get)
    if bound == "hbm":
        out = {"bound": "hbm", "achieved": counts["bytes"] / t_meas / 1e9,
               "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    elif bound == "mufu":
        out = {"bound": "alu", "alu_unit": "MUFU ex2", "achieved": counts["exps"] / t_meas / 1e9,
               "peak": rates["ex2_per_clk_sm"] * sms * clk / 1e9, "unit": "Gex2/s"}
    else:
        out = {"bound": "alu", "alu_unit": "fp32 FMA pipe",
               "achieved": counts["fp32_ops"] / t_meas / 1e9,
               "peak": rates["fp32_per_clk_sm"] * sms * clk / 1e9, "unit": "Gop/s fp32"}
    out["frac"] = out["achieved"] / out["peak"]
    out.update({"roof_us": {"hbm": r["t_hbm"] * 1e6, "mufu": r["t_mufu"] * 1e6,
                            "fp32": r["t_fp32"] * 1e6},
                "frac_of_roof": r["t_roof"] / t_meas,
                "algorithmic": {"bytes": counts["bytes"], "exps": counts["exps"],
                                "fp32_ops": counts["fp32_ops"]}})
    return out


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 7]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows]
        smax = max(float(r[1]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[4 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[2]) for r in rows)}


def cpu_sample_inputs(inp: dict, channels: int) -> dict:
    """The first ``channels`` channels of every batch row: a bounded sample of
    the same workload for the oracle (pure indexing)."""
    out = dict(inp)
    for k in ("x", "delta", "z"):
        if inp[k] is not None:
            out[k] = np.ascontiguousarray(inp[k][:, :, :channels])
    out["A"] = np.ascontiguousarray(inp["A"][:channels])
    out["D"] = np.ascontiguousarray(inp["D"][:channels]) if inp["D"] is not None else None
    return out


def time_oracle(inp: dict, target_s: float, threads: int) -> dict:
    """Time the oracle on a bounded channel sample sized for about target_s."""
    from oracle import ref_scan
    ref_scan.build()
    Bt, L, Dm = inp["x"].shape

    def run(ch):
        s = cpu_sample_inputs(inp, ch)
        t0 = time.perf_counter()
        ref_scan.scan_fwd(s["x"], s["delta"], s["A"], s["B"], s["C"], s["D"], s["z"],
                          s["valid_len"], chunk_len=inp["chunk_len"], threads=threads)
        return time.perf_counter() - t0

    ch = 1
    dt = run(ch)
    while dt < 0.5 and ch < Dm:
        ch = min(Dm, ch * 4)
        dt = run(ch)
    ch_target = int(min(Dm, max(1, ch * target_s / max(dt, 1e-6))))
    if ch_target != ch:
        ch = ch_target
        dt = run(ch)
    elems = Bt * L * ch
    return {"value": elems / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"all {Bt} batch rows x first {ch} of {Dm} channels x {L} steps "
                      f"({elems} elements, {dt:.1f} s)", "seconds": dt}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--kernel", default="auto")
    ap.add_argument("--warps-per-block", type=int, default=0)
    ap.add_argument("--states-per-lane", type=int, default=0)
    ap.add_argument("--channels-per-lane", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--e2e-inflight", type=int, default=2,
                    help="forward end-to-end calls in flight (own stream, workspace, outputs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="--op decode: also time consecutive steps captured in a CUDA graph "
                         "against the same steps launched one by one (no L2 flush: the steps "
                         "of one generation loop)")
    ap.add_argument("--fused-delta", action="store_true",
                    help="softplus workloads: pass the raw step inputs and dt_bias and let the "
                         "kernel apply softplus(raw + dt_bias)")
    ap.add_argument("--op", default="scan", choices=["scan", "decode", "bwd", "ssd", "split"],
                    help="scan: the forward (default); decode: one recurrence step on a "
                         "carried state (--workload picks a decode workload); bwd: the "
                         "backward, replaying from chunk states (--bwd-chunk); ssd: the "
                         "SSD form (one decay per head) on the tensor cores; split: a long "
                         "sequence of few channels split across CTAs (--split-workload)")
    ap.add_argument("--split-workload", type=int, default=1,
                    help="with --op split: 1 = b1 L65536 d256 N16, 2 = b2 L32768 d512 N64")
    ap.add_argument("--bwd-chunk", type=int, default=256)
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload, not the other full-size forwards")
    ap.add_argument("--split-batch", action="store_true",
                    help="under torchrun: split one workload's batch rows across the ranks "
                         "(strong scaling) instead of one replica per rank")
    ap.add_argument("--ssd-workload", type=int, default=1,
                    help="with --op ssd: 1 = 128 states, 2 = 256 states")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (identity when not distributed).
    Each rank runs its own replica of the workload, so the job's time is the
    slowest rank's time; this is the only collective the benchmark uses."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: int, ms: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes
    units_per_rank units, and the job takes the slowest rank's ms."""
    return world * units_per_rank / (ms * 1e-3)


def shard_rows(batch: int, rank: int, world: int) -> tuple[int, int]:
    """Batch rows [lo, hi) of a rank when one workload is split across ranks by
    batch row (rows are independent recurrences; no data-path exchange)."""
    per, extra = divmod(batch, world)
    lo = rank * per + min(rank, extra)
    return lo, lo + per + (1 if rank < extra else 0)


def slice_rows(inp: dict, lo: int, hi: int) -> dict:
    """Batch rows [lo, hi) of a make_inputs() dict (pure indexing: x, delta, z,
    B, C and valid_len have the batch as their first axis)."""
    out = dict(inp)
    for k in ("x", "delta", "z", "B", "C", "valid_len"):
        if inp.get(k) is not None:
            out[k] = np.ascontiguousarray(inp[k][lo:hi])
    return out


def args_kernel(args, S, w):
    """The tier the library launches for this workload and the forced options."""
    k, _ = S.plan(w.batch, w.seqlen, w.dim, w.dstate, dtype=w.dtype, gate=w.gate,
                  mask=w.mask is not None, chunk_len=w.chunk_len, kernel=args.kernel,
                  warps_per_block=args.warps_per_block, states_per_lane=args.states_per_lane,
                  channels_per_lane=args.channels_per_lane)
    return k


def time_forward(args, S, w, inp, prep, dev, stream, flush, K, warmup, clocks_index=0,
                 barrier=None) -> dict:
    """K timed forwards of workload w on device-resident inputs: CUDA events on
    the launch stream around each call, L2 flushed between calls (outside the
    events), SM clocks sampled during the timed region, which `barrier` (all
    ranks) and a device synchronise bracket on both sides."""
    import torch
    from selective_state_space_fwd_gb300 import workloads as W
    t = W.to_torch(inp, dev)
    y = torch.empty_like(t["x"])
    nch = (w.seqlen + w.chunk_len - 1) // w.chunk_len if w.chunk_len else 0
    states = (torch.empty((w.batch, nch, w.dim, w.dstate), dtype=torch.float32, device=dev)
              if w.chunk_len else None)

    def step():
        S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["valid_len"],
                   chunk_len=w.chunk_len, out=y, out_states=states, kernel=args.kernel,
                   warps_per_block=args.warps_per_block,
                   states_per_lane=args.states_per_lane, channels_per_lane=args.channels_per_lane,
                   stream=stream, **prep)

    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            step()
            if not args.no_flush:
                flush.zero_()
    torch.cuda.synchronize(dev)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if barrier is not None:
        barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(clocks_index)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            ev0[i].record(stream)
            step()
            ev1[i].record(stream)
            if not args.no_flush:
                flush.zero_()
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    if barrier is not None:
        barrier()
    S.check_device_errors()
    per_step = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]  # ms, one launch each
    return {"ms": sum(per_step) / K, "t": t, "clocks": clk, "wall": wall, "launches": K,
            "per_step": {"min": min(per_step), "median": statistics.median(per_step),
                         "max": max(per_step)}}


def reference_arm(args, w):
    """The fp64 CPU oracle, as it stands, on the host cores (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from selective_state_space_fwd_gb300 import workloads as W
    inp = W.make_inputs(w)
    threads = os.cpu_count() or 1
    steps, warm = max(1, args.steps), max(0, args.warmup)
    budget = 150.0 / (steps + warm)  # whole run within a few minutes
    probe = time_oracle(inp, min(budget, 5.0), threads)
    rate = probe["value"]
    ch = max(1, min(w.dim, int(budget * rate / (w.batch * w.seqlen))))
    from oracle import ref_scan
    s = cpu_sample_inputs(inp, ch)

    def step():
        ref_scan.scan_fwd(s["x"], s["delta"], s["A"], s["B"], s["C"], s["D"], s["z"],
                          s["valid_len"], chunk_len=inp["chunk_len"], threads=threads)

    for _ in range(warm):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = (time.perf_counter() - t0) / steps
    elems = w.batch * w.seqlen * ch
    val = elems / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "dim": w.dim,
                       "dstate": w.dstate},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"each step: all {w.batch} batch rows x first {ch} of "
                                       f"{w.dim} channels x {w.seqlen} steps ({elems} elements)"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DECODE_METRIC = "decode step: B*D (batch row, channel) updates/s and achieved % of HBM roofline, 1xGB300"


def decode_counts(w) -> dict:
    """Algorithmic bytes of one decode step: the state read and written once,
    the step's inputs read, y written."""
    es = 2 if w.dtype == "bf16" else 4
    B_, D_, N_ = w.batch, w.dim, w.dstate
    act = (3 if w.gate else 2) * B_ * D_ * es
    return {"elements": B_ * D_,
            "bytes": 2 * B_ * D_ * N_ * 4 + act + 2 * B_ * N_ * es + D_ * N_ * 4 + D_ * 4
                     + B_ * D_ * es}


def decode_main(args):
    """One decode step per timed step, on device buffers; the state stays resident."""
    import torch
    import selective_state_space_fwd_gb300 as S
    from selective_state_space_fwd_gb300 import build as B
    from selective_state_space_fwd_gb300 import workloads as W
    rank, world, local = dist_env()
    w = W.DECODE_WORKLOADS[args.workload]
    if args.impl == "reference":
        if rank == 0:
            decode_reference(args, w)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    S.load()
    inp = W.make_inputs(w)
    t = W.to_torch(inp, dev)
    flat = {k: (t[k].reshape(w.batch, -1) if t[k] is not None else None)
            for k in ("x", "delta", "B", "C", "z")}
    state = torch.from_numpy(W.make_state(w)).to(dev)
    y = torch.empty_like(flat["x"])
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        S.decode_step(flat["x"], flat["delta"], t["A"], flat["B"], flat["C"], t["D"], flat["z"],
                      state=state, out=y, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
            flush.zero_()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for i in range(K):
            ev0[i].record(stream)
            step()
            ev1[i].record(stream)
            if not args.no_flush:
                flush.zero_()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per_step = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms = sum(per_step) / K
    c = decode_counts(w)
    graph = None
    if args.graph:
        # consecutive steps of one generation loop, back to back: launched one
        # by one through the binding, and captured once into a CUDA graph
        G, R = 64, 8
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            g0.record(stream)
            for _ in range(G * R):
                step()
            g1.record(stream)
        torch.cuda.synchronize(dev)
        eager_ms = g0.elapsed_time(g1) / (G * R)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(cg, stream=stream):
                for _ in range(G):
                    step()
            for _ in range(3):
                cg.replay()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            g0.record(stream)
            for _ in range(R):
                cg.replay()
            g1.record(stream)
        torch.cuda.synchronize(dev)
        graph = {"steps_per_graph": G, "replays": R, "ms_per_step": g0.elapsed_time(g1) / (G * R),
                 "eager_ms_per_step": eager_ms,
                 "l2": "not flushed (consecutive steps of one generation loop)"}
    # end to end: the step's inputs from pinned host memory, y back, every step
    th = {k: (v.reshape(w.batch, -1).cpu().pin_memory() if v is not None else None)
          for k, v in flat.items()}
    y_h = torch.empty(tuple(y.shape), dtype=y.dtype, pin_memory=True)
    dbuf = {k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in th.items()}

    def step_host():
        with torch.cuda.stream(stream):
            for k, v in th.items():
                if v is not None:
                    dbuf[k].copy_(v, non_blocking=True)
            S.decode_step(dbuf["x"], dbuf["delta"], t["A"], dbuf["B"], dbuf["C"], t["D"],
                          dbuf["z"], state=state, out=y, stream=stream)
            y_h.copy_(y, non_blocking=True)

    for _ in range(3):
        step_host()
    torch.cuda.synchronize(dev)
    KE = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        step_host()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1) / KE
    peaks, peaks_src = load_peaks()
    achieved = c["bytes"] / (ms * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": c["elements"] / (ms * 1e-3), "unit": "updates/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.dtype == "f32" else "bf16-io/f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "gate": w.gate, "state_bytes": w.batch * w.dim * w.dstate * 4,
                   "l2": "flushed between steps (256 MiB memset outside the timed events)"
                         if not args.no_flush else "not flushed"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": measured_traffic("decode", w.name),
                     "peak_source": peaks_src, "kernel": "decode",
                     "algorithmic": {"bytes": c["bytes"]}},
        "cpu_baseline": None if args.no_cpu_baseline else decode_cpu(w, args.cpu_seconds),
        "e2e": {"value": c["elements"] / (ms_e2e * 1e-3), "unit": "updates/s",
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in th.values()
                                          if v is not None),
                "d2h_bytes_per_step": y_h.numel() * y_h.element_size(), "ms_per_step": ms_e2e},
        "gpu_launches": K, "clocks": clk,
        "per_step_ms": {"min": min(per_step), "median": statistics.median(per_step),
                        "max": max(per_step)},
    }
    if graph is not None:
        line["graph"] = graph
    print(json.dumps(line), flush=True)


def _decode_sample(w, rows):
    """The first `rows` batch rows of a decode workload, as oracle inputs (seqlen 1)."""
    from selective_state_space_fwd_gb300 import workloads as W
    inp = W.make_inputs(w)
    st = W.make_state(w)
    cut = {k: (np.ascontiguousarray(inp[k][:rows]) if inp[k] is not None else None)
           for k in ("x", "delta", "B", "C", "z")}
    return cut, inp["A"], inp["D"], np.ascontiguousarray(st[:rows])


def decode_cpu(w, seconds: float) -> dict:
    """The oracle (one-step scan from the state) on a bounded row sample."""
    from oracle import ref_scan
    threads = os.cpu_count() or 1
    rows = max(1, min(w.batch, 64))
    s, A, D, st = _decode_sample(w, rows)
    t0 = time.perf_counter()
    n = 0
    while True:
        ref_scan.scan_fwd(s["x"], s["delta"], A, s["B"], s["C"], D, s["z"], None, h0=st,
                          want_final=True, threads=threads)
        n += 1
        if time.perf_counter() - t0 > min(seconds, 5.0):
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": rows * w.dim / dt, "unit": "updates/s", "cores": threads, "kind": "oracle",
            "sample": f"first {rows} of {w.batch} batch rows x {w.dim} channels, one step"}


def decode_reference(args, w):
    """The oracle as the reference arm of the decode measurement."""
    cpu = decode_cpu(w, 150.0 / max(1, args.steps + args.warmup))
    line = {"impl": "reference", "metric": DECODE_METRIC, "value": cpu["value"],
            "unit": "updates/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name}, "cpu_baseline": cpu,
            "e2e": {"value": cpu["value"], "unit": "updates/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


BWD_METRIC = "selective-scan backward: B*L*D elems/s and achieved % of roofline, 1xGB300"
BWD_FP32_PER_NELT = 10  # lambda, d delta (2), dx, dB, dC, dA, the carry, the replayed update (2)


def bwd_counts(w, inp, chunk: int) -> dict:
    """Algorithmic work of the backward: one exp per valid (t, d, n) (the decay,
    reused by the replayed update and the adjoint), about ten fp32 operations
    per valid (t, d, n); bytes: the forward's inputs, dy and the chunk states
    read once, every gradient written once."""
    L, Dm, N, Bt = w.seqlen, w.dim, w.dstate, w.batch
    vl = np.clip(inp["valid_len"], 0, L) if inp["valid_len"] is not None else np.full(Bt, L)
    ev = int(vl.sum()) * Dm
    es = 2 if w.dtype == "bf16" else 4
    nact = 3 if w.gate else 2
    nch = (L + chunk - 1) // chunk
    rd = (nact + 1) * Bt * L * Dm * es + 2 * Bt * L * N * es + Dm * N * 4 + Dm * 4 \
        + Bt * nch * Dm * N * 4 + Bt * 4
    wr = nact * Bt * L * Dm * es + 2 * Bt * L * N * 4 + Dm * N * 4 + Dm * 4
    return {"elements": Bt * L * Dm, "n_elements": ev * N, "exps": ev * N,
            "fp32_ops": BWD_FP32_PER_NELT * ev * N, "bytes": rd + wr}


def bwd_cpu(w, chunk: int, seconds: float) -> dict:
    """The oracle's backward on a bounded channel sample of the workload (the
    first channels of every batch row; dB and dC are then partial sums over
    those channels, which does not change the work per element)."""
    from oracle import ref_scan
    from selective_state_space_fwd_gb300 import workloads as W
    threads = os.cpu_count() or 1
    inp = W.make_inputs(w)
    Bt, L, Dm = inp["x"].shape
    rng = np.random.default_rng(7)

    def run(ch):
        s = cpu_sample_inputs(inp, ch)
        dy = rng.standard_normal((Bt, L, ch))
        t0 = time.perf_counter()
        ref_scan.scan_bwd(s["x"], s["delta"], s["A"], s["B"], s["C"], s["D"], s["z"],
                          s["valid_len"], dy=dy, threads=threads)
        return time.perf_counter() - t0

    ch = 1
    dt = run(ch)
    while dt < 0.5 and ch < Dm:
        ch = min(Dm, ch * 4)
        dt = run(ch)
    ch_target = int(min(Dm, max(1, ch * min(seconds, 20.0) / max(dt, 1e-6))))
    if ch_target != ch:
        ch = ch_target
        dt = run(ch)
    elems = Bt * L * ch
    return {"value": elems / dt, "unit": "elements/s", "cores": threads, "kind": "oracle",
            "sample": f"all {Bt} batch rows x first {ch} of {Dm} channels x {L} steps "
                      f"({elems} elements, {dt:.1f} s)"}


def bwd_main(args):
    """The backward on device buffers, after one forward that writes the chunk states."""
    import torch
    import selective_state_space_fwd_gb300 as S
    from selective_state_space_fwd_gb300 import build as Bld
    from selective_state_space_fwd_gb300 import workloads as W
    rank, world, local = dist_env()
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        if rank == 0:
            cpu = bwd_cpu(w, args.bwd_chunk, 150.0 / max(1, args.steps + args.warmup))
            print(json.dumps({"impl": "reference", "metric": BWD_METRIC, "value": cpu["value"],
                              "unit": "elements/s", "n_gpus": 1, "steps": args.steps,
                              "warmup": args.warmup, "ms_per_step": None,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": "f64", "data": "synthetic",
                              "config": {"workload": w.name, "chunk_len": args.bwd_chunk},
                              "cpu_baseline": cpu,
                              "e2e": {"value": cpu["value"], "unit": "elements/s",
                                      "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                  flush=True)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Bld.build()
    S.load()
    inp = W.make_inputs(w)
    t = W.to_torch(inp, dev)
    chunk = args.bwd_chunk
    _, states = S.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                           t["valid_len"], chunk_len=chunk)
    gen = torch.Generator(device=dev).manual_seed(7)
    dy = torch.randn(tuple(t["x"].shape), generator=gen, device=dev).to(t["x"].dtype)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        return S.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                          t["valid_len"], chunk_states=states, chunk_len=chunk, dy=dy,
                          stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
            flush.zero_()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for i in range(K):
            ev0[i].record(stream)
            step()
            ev1[i].record(stream)
            if not args.no_flush:
                flush.zero_()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per_step = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms = sum(per_step) / K
    c = bwd_counts(w, inp, chunk)
    peaks, peaks_src = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    rates, rates_src = unit_rates()
    roofline_ = roofline(c, ms * 1e-3, peaks, rates, sms, mhz)
    roofline_.update({"traffic": measured_traffic("bwd", w.name), "kernel": "bwd",
                      "smem_port": smem_port("bwd", w.name, ms * 1e-3, rates, sms, mhz),
                      "peak_source": f"{peaks_src} HBM copy GB/s; {rates_src} unit rates "
                                     f"{_rates_text(rates)} x {sms} SMs x {mhz:.0f} MHz"})
    # end to end: the backward's inputs in from pinned host memory, every gradient out
    host = {k: v.cpu().pin_memory() for k, v in (("x", t["x"]), ("delta", t["delta"]),
                                                  ("B", t["B"]), ("C", t["C"]), ("dy", dy),
                                                  ("states", states))}
    if t["z"] is not None:
        host["z"] = t["z"].cpu().pin_memory()
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    outs = step()
    outs_h = {k: torch.empty(tuple(v.shape), dtype=v.dtype, pin_memory=True)
              for k, v in outs.items() if v is not None}

    def step_host():
        with torch.cuda.stream(stream):
            for k, v in host.items():
                dbuf[k].copy_(v, non_blocking=True)
            g = S.scan_bwd(dbuf["x"], dbuf["delta"], t["A"], dbuf["B"], dbuf["C"], t["D"],
                           dbuf.get("z"), t["valid_len"], chunk_states=dbuf["states"],
                           chunk_len=chunk, dy=dbuf["dy"], stream=stream)
            for k, v in outs_h.items():
                v.copy_(g[k], non_blocking=True)

    for _ in range(2):
        step_host()
    torch.cuda.synchronize(dev)
    KE = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        step_host()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1) / KE
    line = {"metric": BWD_METRIC, "value": c["elements"] / (ms * 1e-3), "unit": UNIT, "n_gpus": 1,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w.dtype == "f32" else "bf16-io/f32", "data": "synthetic",
            "config": {"workload": w.name, "chunk_len": chunk, "gate": w.gate,
                       "masked": w.mask is not None,
                       "l2": "flushed between steps (256 MiB memset outside the timed events)"},
            "roofline": roofline_,
            "cpu_baseline": None if args.no_cpu_baseline else bwd_cpu(w, chunk, args.cpu_seconds),
            "e2e": {"value": c["elements"] / (ms_e2e * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
                    "d2h_bytes_per_step": sum(v.numel() * v.element_size()
                                              for v in outs_h.values()),
                    "ms_per_step": ms_e2e},
            "gpu_launches": K, "clocks": clk,
            "per_step_ms": {"min": min(per_step), "median": statistics.median(per_step),
                            "max": max(per_step)}}
    print(json.dumps(line), flush=True)


SSD_METRIC = "SSD (one decay per head) fwd: B*L*D elems/s and achieved % of roofline, 1xGB300"


def ssd_counts(w) -> dict:
    """Algorithmic work of the SSD form with blocks of 128 steps.  Bytes: x, z
    read and y written once (bf16), delta per (t, head), B and C rows once.
    Tensor flops: C B^T once per (batch row, block) (shared by the heads),
    then per head the block matrix times x, C times the entering state and the
    state update (2 flops per multiply-add)."""
    Q = 128
    Bt, L, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    nb = (L + Q - 1) // Q
    act = Bt * L * H * P
    nbytes = 2 * act * (3 if w.gate else 2) + 2 * Bt * L * H + 2 * 2 * Bt * L * N + 4 * H + 4 * H * P
    flops = Bt * nb * 2 * Q * Q * N + Bt * H * nb * (2 * Q * Q * P + 2 * 2 * Q * N * P)
    return {"elements": act, "bytes": nbytes, "flops": flops}


def _ssd_sample(inp, w, pairs):
    subs = []
    P = w.headdim
    for b, h in pairs:
        ch = slice(h * P, (h + 1) * P)
        subs.append(tuple(np.ascontiguousarray(a) for a in (
            inp["x"][b:b + 1, :, ch], inp["delta"][b:b + 1, :, h:h + 1], inp["A"][h:h + 1],
            inp["B"][b:b + 1], inp["C"][b:b + 1], inp["D"][ch],
            inp["z"][b:b + 1, :, ch] if inp["z"] is not None else None)))
    return subs


def ssd_cpu(w, inp, seconds: float) -> dict:
    """The oracle's SSD form on a bounded sample of (batch row, head) pairs."""
    from oracle import ref_scan
    threads = os.cpu_count() or 1
    pairs = [(b % w.batch, (7 * b) % w.nheads) for b in range(16)]
    subs = _ssd_sample(inp, w, pairs)
    t0 = time.perf_counter()
    n = 0
    while True:
        for sub in subs:
            ref_scan.ssd_fwd(*sub, nheads=1, threads=threads)
            n += 1
        if time.perf_counter() - t0 > min(seconds, 20.0):
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": w.seqlen * w.headdim / dt, "unit": "elements/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{len(pairs)} (batch row, head) pairs x {w.headdim} channels x "
                      f"{w.seqlen} steps, cycled for about {min(seconds, 20.0):.0f} s"}


def ssd_main(args):
    """The SSD form on device buffers (inputs larger than L2), then end to end."""
    import torch
    import selective_state_space_fwd_gb300 as S
    from selective_state_space_fwd_gb300 import build as Bld
    from selective_state_space_fwd_gb300 import workloads as W
    rank, world, local = dist_env()
    w = W.SSD_WORKLOADS[args.ssd_workload]
    inp = W.make_ssd_inputs(w)
    if args.impl == "reference":
        if rank == 0:
            cpu = ssd_cpu(w, inp, 150.0 / max(1, args.steps + args.warmup))
            print(json.dumps({"impl": "reference", "metric": SSD_METRIC, "value": cpu["value"],
                              "unit": "elements/s", "n_gpus": 1, "steps": args.steps,
                              "warmup": args.warmup, "ms_per_step": None,
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": "f64", "data": "synthetic",
                              "config": {"workload": w.name}, "cpu_baseline": cpu,
                              "e2e": {"value": cpu["value"], "unit": "elements/s",
                                      "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                  flush=True)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Bld.build()
    S.load()
    t = W.to_torch(inp, dev)
    y = torch.empty_like(t["x"])
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(tt, out):
        S.ssd_fwd(tt["x"], tt["delta"], t["A"], tt["B"], tt["C"], t["D"], tt["z"], None,
                  nheads=w.nheads, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(t, y)
            flush.zero_()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for i in range(K):
            ev0[i].record(stream)
            step(t, y)
            ev1[i].record(stream)
            if not args.no_flush:
                flush.zero_()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    S.check_device_errors()
    per_step = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms = sum(per_step) / K
    c = ssd_counts(w)
    peaks, peaks_src = load_peaks()
    t_hbm = c["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = c["flops"] / (peaks["bf16_tflops"] * 1e12)
    sec = ms * 1e-3
    if t_hbm >= t_tc:
        ach = c["bytes"] / sec / 1e9
        roofline = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / peaks["hbm_gbs"]}
    else:
        ach = c["flops"] / sec / 1e12
        roofline = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"]}
    roofline.update({"traffic": measured_traffic("ssd", w.name), "kernel": "ssd",
                     "peak_source": peaks_src,
                     "roof_us": {"hbm": t_hbm * 1e6, "tensor_bf16": t_tc * 1e6},
                     "frac_of_roof": max(t_hbm, t_tc) / sec,
                     "tensor_tflops": c["flops"] / sec / 1e12,
                     "algorithmic": {"bytes": c["bytes"], "flops": c["flops"]}})
    # end to end: every input from pinned host memory, y back, every step
    names = ("x", "delta", "B", "C", "z")
    host = {k: t[k].cpu().pin_memory() for k in names if t[k] is not None}
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    y_h = torch.empty(tuple(y.shape), dtype=y.dtype, pin_memory=True)

    def step_host():
        with torch.cuda.stream(stream):
            for k, v in host.items():
                dbuf[k].copy_(v, non_blocking=True)
            step({k: dbuf.get(k) for k in names}, y)
            y_h.copy_(y, non_blocking=True)

    for _ in range(2):
        step_host()
    torch.cuda.synchronize(dev)
    KE = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        step_host()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1) / KE
    line = {
        "metric": SSD_METRIC, "value": c["elements"] / sec, "unit": "elements/s", "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16-io/bf16-mma/f32-acc",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen,
                   "nheads": w.nheads, "headdim": w.headdim, "dstate": w.dstate,
                   "gate": w.gate, "block": 128,
                   "l2": "flushed between steps (256 MiB memset outside the timed events)"
                         if not args.no_flush else "not flushed"},
        "roofline": roofline,
        "cpu_baseline": None if args.no_cpu_baseline else ssd_cpu(w, inp, args.cpu_seconds),
        "e2e": {"value": c["elements"] / (ms_e2e * 1e-3), "unit": "elements/s",
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
                "d2h_bytes_per_step": y_h.numel() * y_h.element_size(), "ms_per_step": ms_e2e},
        "gpu_launches": K, "clocks": clk,
        "per_step_ms": {"min": min(per_step), "median": statistics.median(per_step),
                        "max": max(per_step)},
    }
    print(json.dumps(line), flush=True)


SPLIT_METRIC = ("selective-scan fwd, sequence split across CTAs: B*L*D elems/s and achieved % "
                "of roofline, 1xGB300")


def split_main(args):
    """The time split on a long sequence of few channels: scan_fwd with the
    library's choice (the split) against one segment, device buffers."""
    from selective_state_space_fwd_gb300 import workloads as W
    w = W.SPLIT_WORKLOADS[args.split_workload]
    if args.impl == "reference":
        reference_arm(args, w)
        return
    import torch
    import selective_state_space_fwd_gb300 as S
    from selective_state_space_fwd_gb300 import build as B
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()
    S.load()
    inp = W.make_inputs(w)
    t = W.to_torch(inp, dev)
    segs, nbytes = S.split_plan(w.batch, w.seqlen, w.dim, w.dstate, dtype=w.dtype, gate=w.gate)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    y = torch.empty_like(t["x"])
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(nseg, K):
        def step():
            S.scan_fwd_split(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                             t["valid_len"], time_segments=nseg, out=y, workspace=ws, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                step()
                flush.zero_()
        torch.cuda.synchronize(dev)
        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        clocks = ClockSampler(local)
        with torch.cuda.stream(stream):
            for i in range(K):
                ev0[i].record(stream)
                step()
                ev1[i].record(stream)
                flush.zero_()
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        S.check_device_errors()
        per = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
        return sum(per) / K, clk, per

    ms, clk, per = timed(segs, args.steps)
    ms1, _, _ = timed(1, max(3, min(args.steps, 10)))
    counts = algorithmic_counts(w, inp)
    peaks, peaks_src = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    rates, rates_src = unit_rates()
    rl = roofline(counts, ms * 1e-3, peaks, rates, sms, mhz)
    rl.update({"kernel": "stream (aggregate pass, carry, output pass)", "traffic": None,
               "peak_source": f"{peaks_src} HBM copy GB/s; {rates_src} unit rates "
                              f"{_rates_text(rates)} x {sms} SMs x {mhz:.0f} MHz"})
    # end to end: inputs from pinned host memory, the split forward, y back
    th = {k: (v.cpu().pin_memory() if isinstance(v, torch.Tensor) else None)
          for k, v in t.items() if k in ("x", "delta", "A", "B", "C", "D")}
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in th.items() if v is not None}
    y_h = torch.empty(tuple(y.shape), dtype=y.dtype, pin_memory=True)

    def step_host():
        with torch.cuda.stream(stream):
            for k, v in th.items():
                dbuf[k].copy_(v, non_blocking=True)
            S.scan_fwd_split(dbuf["x"], dbuf["delta"], dbuf["A"], dbuf["B"], dbuf["C"], dbuf["D"],
                             time_segments=segs, out=y, workspace=ws, stream=stream)
            y_h.copy_(y, non_blocking=True)

    for _ in range(2):
        step_host()
    torch.cuda.synchronize(dev)
    KE = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        step_host()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1) / KE
    cpu = None
    if not args.no_cpu_baseline:
        cpu = time_oracle(inp, args.cpu_seconds, os.cpu_count() or 1)
        cpu.pop("seconds", None)
    line = {
        "metric": SPLIT_METRIC, "value": counts["elements"] / (ms * 1e-3), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.dtype == "f32" else "bf16-io/f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "dim": w.dim,
                   "dstate": w.dstate, "segments": segs,
                   "l2": "flushed between steps (256 MiB memset outside the timed events)"},
        "roofline": rl, "cpu_baseline": cpu,
        "unsplit": {"ms_per_step": ms1, "value": counts["elements"] / (ms1 * 1e-3)},
        "e2e": {"value": counts["elements"] / (ms_e2e * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in th.values()
                                          if v is not None),
                "d2h_bytes_per_step": y_h.numel() * y_h.element_size(), "ms_per_step": ms_e2e},
        "gpu_launches": 3 * args.steps, "clocks": clk,
        "per_step_ms": {"min": min(per), "median": statistics.median(per), "max": max(per)},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.op == "decode":
        decode_main(args)
        return
    if args.op == "bwd":
        bwd_main(args)
        return
    if args.op == "ssd":
        ssd_main(args)
        return
    if args.op == "split":
        split_main(args)
        return
    from selective_state_space_fwd_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, w)
        return

    import torch
    import torch.distributed as dist
    import selective_state_space_fwd_gb300 as S
    from selective_state_space_fwd_gb300 import build as B

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    B.build()
    S.load()

    inp = W.make_inputs(w)
    full_valid = inp["valid_len"]
    if args.split_batch and world > 1:
        # one workload split across ranks by batch row: rank r scans rows [lo, hi)
        # (the rows are independent recurrences; no data-path exchange)
        lo, hi = shard_rows(w.batch, rank, world)
        inp = slice_rows(inp, lo, hi)
    prep = {}
    if args.fused_delta:
        raw, bias = W.make_raw_delta(w)
        if args.split_batch and world > 1:
            raw = np.ascontiguousarray(raw[lo:hi])
        inp["delta"] = raw
        prep = {"dt_bias": torch.from_numpy(bias).to(dev), "delta_softplus": True}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    wr = w.scaled(batch=int(inp["x"].shape[0]))  # this rank's rows
    res = time_forward(args, S, wr, inp, prep, dev, stream, flush, args.steps, args.warmup,
                       clocks_index=local, barrier=dist.barrier if world > 1 else None)
    ms = max_over_ranks(res["ms"], dev)
    res_launches, res_clocks, res_wall = res["launches"], res["clocks"], res["wall"]
    res_per_step = res["per_step"]
    res_kernel = args_kernel(args, S, wr)
    counts = algorithmic_counts(w, {"valid_len": full_valid})
    if args.fused_delta:  # one exp and one log per valid (b, t, d)
        counts["exps"] += 2 * counts["valid_elements"]
        counts["bytes"] += w.dim * 4
    if args.split_batch and world > 1:
        value = counts["elements"] / (ms * 1e-3)  # the whole workload, shared by the ranks
    else:
        value = job_rate(world, counts["elements"], ms)
    t = res["t"]
    nch = (w.seqlen + w.chunk_len - 1) // w.chunk_len if w.chunk_len else 0

    # End to end through the C ABI with host buffers: H2D of the step's inputs from
    # pinned memory, the forward, D2H of y (and chunk states), every step.
    th = W.to_torch(inp, "cpu")
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in th.items()}
    # NF calls in flight, as a serving loop issues them: call k runs on stream
    # k % NF with its own workspace and output buffers, so that its copies in
    # overlap the previous call's last kernel and copies out (the library's
    # copy streams keep the calls' copies in order).
    NF = max(1, args.e2e_inflight)
    y_hs = [torch.empty(tuple(t["x"].shape), dtype=t["x"].dtype, pin_memory=True)
            for _ in range(NF)]
    s_hs = [torch.empty((wr.batch, nch, w.dim, w.dstate), dtype=torch.float32, pin_memory=True)
            if w.chunk_len else None for _ in range(NF)]
    y_h, s_h = y_hs[0], s_hs[0]
    del res, t
    torch.cuda.empty_cache()
    ws_bytes = S.host_workspace_bytes(wr.batch, w.seqlen, w.dim, w.dstate, dtype=w.dtype,
                                      has_D=True, gate=w.gate, mask=w.mask is not None,
                                      chunk_len=w.chunk_len)
    wss = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in range(NF)]
    streams = [stream] + [torch.cuda.Stream(dev) for _ in range(NF - 1)]

    def step_host(k):
        j = k % NF
        S.scan_fwd_host(pinned["x"], pinned["delta"], pinned["A"], pinned["B"], pinned["C"],
                        pinned["D"], pinned["z"], pinned["valid_len"], chunk_len=w.chunk_len,
                        out=y_hs[j], out_states=s_hs[j], workspace=wss[j], stream=streams[j])

    for k in range(3 * NF):
        step_host(k)
    torch.cuda.synchronize(dev)
    KE = max(1, args.e2e_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for sj in streams[1:]:
        sj.wait_event(e0)
    for k in range(KE):
        step_host(k)
    for sj in streams[1:]:
        stream.wait_stream(sj)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / KE, dev)
    # every in-flight slot returned the same y as the device-timed forward
    for yk in y_hs[1:min(NF, KE)]:
        if not torch.equal(yk, y_h):
            raise RuntimeError("end-to-end calls in flight returned different outputs")
    es = 2 if w.dtype == "bf16" else 4
    h2d = sum(v.numel() * v.element_size() for k, v in pinned.items()
              if isinstance(v, torch.Tensor))
    d2h = y_h.numel() * es + (s_h.numel() * 4 if s_h is not None else 0)
    del wss, pinned, th, y_hs, s_hs
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peaks_src = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz_peak = float(peaks.get("sm_max_mhz", 2070.0))
    rates, rates_src = unit_rates()
    peak_text = (f"{peaks_src} HBM copy GB/s; {rates_src} unit rates {_rates_text(rates)} "
                 f"x {sms} SMs x {sm_mhz_peak:.0f} MHz")
    rl = roofline(counts, ms * 1e-3, peaks, rates, sms, sm_mhz_peak)
    rl.update({
        "traffic": measured_traffic(S.kernel_name(res_kernel), w.name),
        "smem_port": smem_port(S.kernel_name(res_kernel), w.name, ms * 1e-3, rates, sms,
                               sm_mhz_peak),
        "peak_source": peak_text, "unit_rates": rates,
        "kernel": S.kernel_name(res_kernel),
        "warps_per_block": args.warps_per_block, "states_per_lane": args.states_per_lane,
        "channels_per_lane": args.channels_per_lane})
    # The other full-size workloads of the same forward (device-timed only, the
    # same timing rules), each with its own roofline.
    per_config = {}
    forced = args.kernel != "auto" or args.warps_per_block or args.states_per_lane \
        or args.channels_per_lane
    if not args.no_per_config and world == 1 and not args.fused_delta and not forced:
        for key in sorted(W.WORKLOADS):
            if key in (1, args.workload):
                continue
            wk = W.WORKLOADS[key]
            ik = W.make_inputs(wk)
            rk = time_forward(args, S, wk, ik, {}, dev, stream, flush,
                              max(3, min(args.steps, 20)), 3, clocks_index=local)
            ck = algorithmic_counts(wk, ik)
            rlk = roofline(ck, rk["ms"] * 1e-3, peaks, rates, sms, sm_mhz_peak)
            kk = args_kernel(args, S, wk)
            per_config[wk.name] = {
                "ms_per_step": rk["ms"], "value": ck["elements"] / (rk["ms"] * 1e-3),
                "unit": UNIT, "valid_elements_per_s": ck["valid_elements"] / (rk["ms"] * 1e-3),
                "kernel": S.kernel_name(kk), "clocks": rk["clocks"],
                "roofline": dict({k: rlk[k] for k in ("bound", "achieved", "peak", "unit",
                                                      "frac", "frac_of_roof", "roof_us")},
                                 traffic=measured_traffic(S.kernel_name(kk), wk.name),
                                 smem_port=smem_port(S.kernel_name(kk), wk.name,
                                                     rk["ms"] * 1e-3, rates, sms, sm_mhz_peak)),
                "gpu_launches": rk["launches"]}
            del rk, ik
            torch.cuda.empty_cache()
    cpu = None
    if not args.no_cpu_baseline:
        cpu = time_oracle(inp, args.cpu_seconds, os.cpu_count() or 1)
        cpu.pop("seconds", None)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if args.split_batch and world > 1 else "weak",
        "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16-io/f32",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "dim": w.dim,
                   "dstate": w.dstate, "gate": w.gate, "chunk_len": w.chunk_len,
                   "masked": w.mask is not None,
                   "delta": "fused: softplus(raw + dt_bias) in the kernel" if args.fused_delta
                            else "given (already positive)",
                   "l2": "flushed between steps (256 MiB memset outside the timed events)"
                         if not args.no_flush else "not flushed",
                   "parallelism": (f"batch rows split over {world} ranks" if args.split_batch
                                   else f"replicas x{world}") if world > 1 else "single GPU"},
        "roofline": rl,
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(1 if args.split_batch else world, counts["elements"], ms_e2e),
                "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_e2e, "calls_in_flight": NF},
        "gpu_launches": res_launches,
        "clocks": res_clocks,
        "timed_wall_s": res_wall,
        "per_step_ms": res_per_step,
        "per_config": per_config,
    }
    if counts["valid_elements"] != counts["elements"]:
        line["valid_elements_per_s"] = job_rate(world, counts["valid_elements"], ms)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
