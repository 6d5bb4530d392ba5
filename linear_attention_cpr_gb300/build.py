"""Build the in-tree CUDA library (sm_103a) with nvcc: ``python -m linear_attention_cpr_gb300.build``.

Translation units compile in parallel into ``_build/`` and link into
``_build/libcprgdn.so`` (the C ABI of include/cpr_gdn.h) and ``_build/libcprprobe.so``
(the FP32-pipe peak probe used for roofline denominators).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(BUILD, "libcprgdn.so")
PROBE_LIB = os.path.join(BUILD, "libcprprobe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-cudart", "shared",
                     f"-I{INCLUDE}"]
LIB_UNITS = ["api.cu", "prefill.cu", "decode.cu", "backward.cu", "backward_tc.cu", "noalloc.cu", "pik.cu"]
PROBE_UNITS = ["probe_peaks.cu"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return hs


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources + [__file__])


def _build_lib(out: str, units: list[str], verbose: bool) -> None:
    srcs = [os.path.join(CSRC, u) for u in units]
    if not _stale(out, srcs + _headers()):
        return
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        log, _ = p.communicate()
        if p.returncode != 0:
            failed.append((cmd, log.decode(errors="replace")))
    if failed:
        msg = "\n\n".join(" ".join(c) + "\n" + log for c, log in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = f"{out}.{os.getpid()}.tmp"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    if verbose:
        print(" ".join(link), flush=True)
    subprocess.run(link, check=True)
    os.replace(tmp, out)


def build(verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libcprgdn.so."""
    _build_lib(LIB, LIB_UNITS, verbose)
    if all(os.path.exists(os.path.join(CSRC, u)) for u in PROBE_UNITS):
        _build_lib(PROBE_LIB, PROBE_UNITS, verbose)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
