"""fp64 CPU oracle of the Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this module.
The CUDA library never imports, links or calls it, and this module never imports the
CUDA library; the two share only the seeded input generators, which hold none of the
method's arithmetic.

The arithmetic lives in ``cpr_oracle.c`` (plain C, fp64).  This module compiles it
with the host C compiler on first use and calls it through ``ctypes``.

Functions (all inputs are converted to float64 exactly; layouts as in cpr_oracle.c):

``recurrent``   the plain gated delta rule, token by token, over a packed batch;
                returns (o, state_out, boundary_states).  Pinned by brute force,
                closed forms and invariants in tests/test_oracle_pins.py.
``chunked``     the CPR schedule (chunk update U at every full chunk, token recurrence
                inside chunks) in fp64; agrees with ``recurrent`` to rounding.
``bruteforce``  materialised products of per-token transition matrices for one
                (sequence, head); tiny sizes only.

Modules beside it: ``oracle.pik`` (the deterministic K-split product: fp32 tree, exact
product, error bound) and ``oracle.backward`` (the exact adjoint of the recurrence, for
the backward pass).

Sources: "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"; "SkyRL IsoExec: vLLM 与 Megatron
的 logprob 差 ...", section "Gated DeltaNet 的第三条路：chunkwise-parallel recurrent";
recurrence of the Gated Delta Networks paper (Yang, Kautz & Hatamizadeh, ICLR 2025).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)


def lib_path(mutant: int = 0) -> str:
    name = "libcproracle.so" if mutant == 0 else f"libcproracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile cpr_oracle.c (optionally with a planted mistake, for the pin tests)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP: single-threaded
    os.replace(tmp, out)
    return out


def _lib(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant not in _libs:
            lib = ctypes.CDLL(build(mutant))
            for fn in ("oracle_gdn_recurrent", "oracle_gdn_chunked"):
                f = getattr(lib, fn)
                f.restype = ctypes.c_int
                f.argtypes = [_D, _D, _D, _D, _D, _I32, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, ctypes.c_int, _D, _D, _D, _D, ctypes.c_int]
            lib.oracle_gdn_bruteforce.restype = ctypes.c_int
            lib.oracle_gdn_bruteforce.argtypes = [_D, _D, _D, _D, _D, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, _D, _D, _D]
            lib.oracle_num_chunks.restype = ctypes.c_int64
            lib.oracle_num_chunks.argtypes = [_I32, ctypes.c_int, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            _libs[mutant] = lib
        return _libs[mutant]


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor: exact widening on the CPU
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_D)


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def num_chunks(cu_seqlens, C: int) -> int:
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return int(_lib().oracle_num_chunks(cu.ctypes.data_as(_I32), len(cu) - 1, C))


def _run(fn_name, q, k, v, g, beta, cu_seqlens, C, state_in, boundaries, n_threads, mutant):
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = len(cu) - 1
    if k.shape != (T, H, dk) or v.shape[:2] != (T, H) or g.shape != (T, H) or beta.shape != (T, H):
        raise ValueError("oracle: inconsistent input shapes")
    if N < 0 or int(cu[-1]) != T:
        raise ValueError("oracle: cu_seqlens[-1] must equal the token count")
    s_in = None if state_in is None else _f64(state_in).reshape(N, H, dk, dv)
    o = np.zeros((T, H, dv))
    s_out = np.zeros((N, H, dk, dv))
    bnd = np.zeros((num_chunks(cu, C), H, dk, dv)) if boundaries else None
    rc = getattr(_lib(mutant), fn_name)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), cu.ctypes.data_as(_I32), N, H, dk, dv, C,
        _ptr(s_in), _ptr(o), _ptr(s_out), _ptr(bnd), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"{fn_name} failed with code {rc}")
    return o, s_out, bnd


def recurrent(q, k, v, g, beta, cu_seqlens, C, state_in=None, boundaries=True, n_threads=0, mutant=0):
    """Plain fp64 recurrence.  Returns (o [T,H,dv], state_out [N,H,dk,dv], boundary [n_chunks,H,dk,dv])."""
    return _run("oracle_gdn_recurrent", q, k, v, g, beta, cu_seqlens, C, state_in, boundaries,
                n_threads, mutant)


def chunked(q, k, v, g, beta, cu_seqlens, C, state_in=None, boundaries=True, n_threads=0, mutant=0):
    """CPR schedule in fp64 (chunk update at each full chunk).  Same returns as ``recurrent``."""
    return _run("oracle_gdn_chunked", q, k, v, g, beta, cu_seqlens, C, state_in, boundaries,
                n_threads, mutant)


def bruteforce(q, k, v, g, beta, S0=None, mutant=0):
    """One (sequence, head): q,k [T,dk], v [T,dv], g,beta [T], S0 [dk,dv].  Returns (o [T,dv], S_T [dk,dv])."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, dk = q.shape
    dv = v.shape[1]
    s0 = None if S0 is None else _f64(S0).reshape(dk, dv)
    o = np.zeros((T, dv))
    st = np.zeros((dk, dv))
    rc = _lib(mutant).oracle_gdn_bruteforce(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), T, dk, dv,
                                            _ptr(s0), _ptr(o), _ptr(st))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_bruteforce failed with code {rc}")
    return o, st
