"""Build libssmscan.so in-tree with nvcc for sm_103a (GB300).

    python -m selective_state_space_fwd_gb300.build [--force]

Each translation unit under csrc/ compiles in parallel; the objects link into
``selective_state_space_fwd_gb300/libssmscan.so`` against the shared CUDA
runtime (the same soname PyTorch loads, so one runtime serves both).  No
cmake, no torch extension machinery: the library has a plain C ABI.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libssmscan.so")
# measurement harness: unit-rate probes the benchmark's roofline uses
PROBE_SRC = os.path.join(PKG, "probe", "unit_rates.cu")
PROBE_LIB = os.path.join(PKG, "libssmprobe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssmscan")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    out = sources()
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    out += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    out.append(os.path.abspath(__file__))
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build_probe(force: bool = False) -> str:
    """libssmprobe.so: the MUFU ex2, fp32 FMA and shared-memory load rate probes."""
    if (not force and os.path.exists(PROBE_LIB)
            and os.path.getmtime(PROBE_LIB) >= max(os.path.getmtime(PROBE_SRC),
                                                   os.path.getmtime(os.path.abspath(__file__)))):
        return PROBE_LIB
    nvcc = _nvcc()
    tmp = PROBE_LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
           "-o", tmp, PROBE_SRC, "-Xlinker", f"-rpath,{_cuda_lib_dir(nvcc)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on unit_rates.cu:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


def build(force: bool = False, verbose: bool = False) -> str:
    build_probe(force)
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OBJ, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose:
        common += ["-Xptxas", "-v"]
    common += os.environ.get("SSM_NVCC_EXTRA", "").split()  # extra defines for comparison builds

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJ, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([nvcc, *common, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
