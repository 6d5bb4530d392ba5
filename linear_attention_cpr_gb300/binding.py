"""Thin Python binding of the C ABI in include/cpr_gdn.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors are torch
tensors on the current CUDA device; torch supplies device memory and the stream, and
every step of the layer runs in the library's CUDA kernels.  There is no fallback: if
the compiled library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

CPR_DTYPE_BF16 = 0
CPR_DTYPE_F32 = 1
DEV_BAD_CU_SEQLENS = 1
DEV_BOUNDARY_CAPACITY = 2
DEV_BAD_POS = 4

EXPORTED = (
    "cpr_gdn_supported", "cpr_gdn_version", "cpr_gdn_strerror", "cpr_gdn_num_chunks",
    "cpr_gdn_prefill_workspace_size", "cpr_gdn_decode_workspace_size", "cpr_gdn_prefill",
    "cpr_gdn_ring_from_prefill", "cpr_gdn_decode", "cpr_gdn_device_status", "cpr_gdn_set_profile_events",
    "cpr_gdn_prefill_noalloc", "cpr_gdn_prefill_noalloc_status", "cpr_gdn_prefill_continue", "cpr_gdn_prefill_grouped",
    "cpr_gdn_ring_from_prefill_grouped", "cpr_gdn_decode_grouped", "cpr_gdn_prefill_continue_grouped",
    "cpr_pik_workspace_size", "cpr_pik_gemm", "cpr_pik_combine", "cpr_gdn_set_wait_test",
    "cpr_gdn_backward_workspace_size", "cpr_gdn_backward_supported", "cpr_gdn_backward",
)
NOALLOC_SCRATCH_BYTES = 16 << 20  # CPR_GDN_NOALLOC_SCRATCH_BYTES


class CprError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed: {text} ({code})")
        self.code = code


class _Ring(ctypes.Structure):
    _fields_ = [("S_b", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libcprgdn.so (built by ``linear_attention_cpr_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library {path} is not built; run "
                               "`python -m linear_attention_cpr_gb300.build` (nvcc, sm_103a)")
        _build.build()
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ, U32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint32
    sig = {
        "cpr_gdn_supported": (ctypes.c_int, [I32, I32, I32, I32]),
        "cpr_gdn_version": (I32, []),
        "cpr_gdn_strerror": (ctypes.c_char_p, [I32]),
        "cpr_gdn_num_chunks": (I64, [P, I32, I32]),
        "cpr_gdn_prefill_workspace_size": (SZ, [I64, I32, I32, I32, I32, I32]),
        "cpr_gdn_decode_workspace_size": (SZ, [I32, I32, I32, I32, I32]),
        "cpr_gdn_prefill": (I32, [P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, P, P, P, P, I64, P, SZ, P]),
        "cpr_gdn_ring_from_prefill": (I32, [P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, P, P,
                                            ctypes.POINTER(_Ring), P]),
        "cpr_gdn_decode": (I32, [P, P, P, P, P, P, ctypes.POINTER(_Ring), P, I32, I32, I32, I32, I32, I32, P, P,
                                 SZ, P]),
        "cpr_gdn_device_status": (I32, [P, ctypes.POINTER(ctypes.c_uint32), P]),
        "cpr_gdn_set_profile_events": (I32, [ctypes.POINTER(ctypes.c_void_p), I32]),
        "cpr_gdn_prefill_noalloc": (I32, [P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, P, P, P, P, I64, P]),
        "cpr_gdn_prefill_noalloc_status": (I32, [ctypes.POINTER(ctypes.c_uint32), P]),
        "cpr_gdn_set_wait_test": (I32, [U32, ctypes.c_uint64]),
        "cpr_gdn_backward_workspace_size": (SZ, [I64, I32, I32, I32, I32, I32]),
        "cpr_gdn_backward_supported": (ctypes.c_int, [I32, I32, I32, I32]),
        "cpr_gdn_backward": (I32, [P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, P, I64, P, P, P, P, P, P, P,
                                   P, P, SZ, P]),
        "cpr_gdn_prefill_continue": (I32, [P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, P, P,
                                           ctypes.POINTER(_Ring), P, P, I64, P, SZ, P]),
        "cpr_gdn_prefill_grouped": (I32, [P, P, P, P, P, P, I32, I64, I32, I32, U32, I32, I32, I32, I32, P, P, P, P,
                                          I64, P, SZ, P]),
        "cpr_gdn_ring_from_prefill_grouped": (I32, [P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, I32, P, P,
                                                    ctypes.POINTER(_Ring), P]),
        "cpr_gdn_decode_grouped": (I32, [P, P, P, P, P, P, ctypes.POINTER(_Ring), P, I32, I32, I32, U32, I32, I32,
                                         I32, I32, P, P, SZ, P]),
        "cpr_gdn_prefill_continue_grouped": (I32, [P, P, P, P, P, P, I32, I64, I32, I32, U32, I32, I32, I32, I32, P,
                                                   P, ctypes.POINTER(_Ring), P, P, I64, P, SZ, P]),
        "cpr_pik_workspace_size": (SZ, []),
        "cpr_pik_gemm": (I32, [P, P, P, I32, I32, I32, I32, I32, I32, P, P]),
        "cpr_pik_combine": (I32, [P, I32, I64, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise CprError(fn, code, load_library().cpr_gdn_strerror(code).decode())


QK_L2NORM = 1  # CPR_QK_L2NORM


def _flags(qk_l2norm: bool) -> int:
    return QK_L2NORM if qk_l2norm else 0


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CPR_DTYPE_BF16
    if t.dtype == torch.float32:
        return CPR_DTYPE_F32
    raise TypeError(f"unsupported element type {t.dtype} (bf16 or fp32)")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if t.numel() == 0:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def cpr_gdn_supported(dk: int, dv: int, C: int, dtype=torch.bfloat16) -> bool:
    code = CPR_DTYPE_BF16 if dtype == torch.bfloat16 else CPR_DTYPE_F32
    return bool(load_library().cpr_gdn_supported(dk, dv, C, code))


def cpr_gdn_version() -> int:
    return int(load_library().cpr_gdn_version())


def cpr_gdn_strerror(code: int) -> str:
    return load_library().cpr_gdn_strerror(code).decode()


def cpr_gdn_num_chunks(cu_seqlens_host, C: int) -> int:
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).cpu().contiguous()
    n = int(load_library().cpr_gdn_num_chunks(cu.data_ptr(), cu.numel() - 1, C))
    if n < 0:
        raise CprError("cpr_gdn_num_chunks", n, cpr_gdn_strerror(n))
    return n


def cpr_gdn_prefill_workspace_size(total_tokens: int, n_seqs: int, H: int, dk: int, dv: int, C: int) -> int:
    return int(load_library().cpr_gdn_prefill_workspace_size(total_tokens, n_seqs, H, dk, dv, C))


def cpr_gdn_decode_workspace_size(B: int, H: int, dk: int, dv: int, C: int) -> int:
    return int(load_library().cpr_gdn_decode_workspace_size(B, H, dk, dv, C))


def cpr_gdn_prefill(q, k, v, g, beta, cu_seqlens, C: int, state_in=None, *, out=None, state_out=None,
                    boundary_states=None, workspace=None, n_chunks: int | None = None, qk_l2norm: bool = False,
                    stream=None):
    """CPR prefill.  Returns (out, state_out, boundary_states, workspace).

    ``cu_seqlens`` is an int32 CUDA tensor.  ``n_chunks`` (the batch's chunk count) is
    read from a host copy of cu_seqlens when not given and boundary_states is None.
    """
    T, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[-1]  # value heads; H / Hk value heads share each query/key head
    N = cu_seqlens.numel() - 1
    dev = q.device
    if out is None:
        out = torch.empty(T, H, dv, dtype=q.dtype, device=dev)
    if state_out is None:
        state_out = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    if boundary_states is None:
        if n_chunks is None:
            n_chunks = cpr_gdn_num_chunks(cu_seqlens.cpu(), C)
        boundary_states = torch.empty(max(n_chunks, 1), H, dk, dv, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(cpr_gdn_prefill_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)
    code = load_library().cpr_gdn_prefill_grouped(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, Hk, _flags(qk_l2norm), dk, dv, C,
        _dtype_code(q), _ptr(state_in), _ptr(out), _ptr(state_out), _ptr(boundary_states), boundary_states.shape[0],
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check("cpr_gdn_prefill_grouped", code)
    return out, state_out, boundary_states, workspace


def cpr_gdn_backward_workspace_size(total_tokens: int, n_seqs: int, H: int, dk: int, dv: int, C: int) -> int:
    return int(load_library().cpr_gdn_backward_workspace_size(total_tokens, n_seqs, H, dk, dv, C))


def cpr_gdn_backward_supported(dk: int, dv: int, C: int, dtype=torch.bfloat16) -> bool:
    code = CPR_DTYPE_BF16 if dtype == torch.bfloat16 else CPR_DTYPE_F32
    return bool(load_library().cpr_gdn_backward_supported(dk, dv, C, code))


def cpr_gdn_backward(q, k, v, g, beta, cu_seqlens, C: int, boundary_states, d_out, d_state_out=None, *,
                     grads=None, d_state_in=True, workspace=None, stream=None):
    """CPR backward.  Returns (dict(dq, dk, dv, dg, dbeta, d_state_in), workspace).

    ``boundary_states`` are the forward's (cpr_gdn_prefill on the same batch and C);
    ``d_out`` has the element type of q; gradients are fp32.  ``grads`` may hold
    preallocated outputs under those names; ``d_state_in=False`` skips that output."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = q.device
    gr = dict(grads or {})
    gr.setdefault("dq", torch.empty(T, H, dk, dtype=torch.float32, device=dev))
    gr.setdefault("dk", torch.empty(T, H, dk, dtype=torch.float32, device=dev))
    gr.setdefault("dv", torch.empty(T, H, dv, dtype=torch.float32, device=dev))
    gr.setdefault("dg", torch.empty(T, H, dtype=torch.float32, device=dev))
    gr.setdefault("dbeta", torch.empty(T, H, dtype=torch.float32, device=dev))
    if d_state_in is True:
        gr.setdefault("d_state_in", torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev))
    if workspace is None:
        workspace = torch.empty(cpr_gdn_backward_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)
    code = load_library().cpr_gdn_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv, C, _dtype_code(q),
        _ptr(boundary_states), boundary_states.shape[0], _ptr(d_out), _ptr(d_state_out), _ptr(gr["dq"]),
        _ptr(gr["dk"]), _ptr(gr["dv"]), _ptr(gr["dg"]), _ptr(gr["dbeta"]), _ptr(gr.get("d_state_in")),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check("cpr_gdn_backward", code)
    return gr, workspace


@dataclass
class Ring:
    """Decode ring buffers (see cpr_gdn_ring in include/cpr_gdn.h)."""
    S_b: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor

    @staticmethod
    def empty(B: int, H: int, dk: int, dv: int, C: int, dtype=torch.bfloat16, device="cuda") -> "Ring":
        return Ring(S_b=torch.zeros(B, H, dk, dv, dtype=torch.float32, device=device),
                    k=torch.zeros(B, H, C, dk, dtype=dtype, device=device),
                    v=torch.zeros(B, H, C, dv, dtype=dtype, device=device),
                    g=torch.zeros(B, H, C, dtype=torch.float32, device=device),
                    beta=torch.zeros(B, H, C, dtype=torch.float32, device=device))

    def _c(self) -> _Ring:
        return _Ring(_ptr(self.S_b), _ptr(self.k), _ptr(self.v), _ptr(self.g), _ptr(self.beta))

    def clone(self) -> "Ring":
        return Ring(*(t.clone() for t in (self.S_b, self.k, self.v, self.g, self.beta)))

    def index(self, idx) -> "Ring":
        return Ring(*(t[idx].contiguous() for t in (self.S_b, self.k, self.v, self.g, self.beta)))


def cpr_gdn_ring_from_prefill(k, v, g, beta, cu_seqlens, C: int, boundary_states, state_out, ring: Ring | None = None,
                              stream=None) -> Ring:
    T, Hk, dk = k.shape
    H, dv = v.shape[1], v.shape[-1]
    N = cu_seqlens.numel() - 1
    if ring is None:
        ring = Ring.empty(N, H, dk, dv, C, dtype=k.dtype, device=k.device)
    rc = ring._c()
    code = load_library().cpr_gdn_ring_from_prefill_grouped(
        _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, Hk, dk, dv, C, _dtype_code(k),
        _ptr(boundary_states), _ptr(state_out), ctypes.byref(rc), _stream(stream))
    _check("cpr_gdn_ring_from_prefill_grouped", code)
    return ring


def continue_chunks(cu_seqlens_host, pos0_host, C: int) -> int:
    """Chunks of the remainders of a continuation (what its boundary_states must hold)."""
    cu = [int(x) for x in cu_seqlens_host]
    p0 = [int(x) for x in pos0_host]
    n = 0
    for i in range(len(cu) - 1):
        L = cu[i + 1] - cu[i]
        f = 0 if p0[i] % C == 0 else min(C - p0[i] % C, L)
        n += -(-(L - f) // C)
    return n


def cpr_gdn_prefill_continue(q, k, v, g, beta, cu_seqlens, pos0, C: int, state, ring: Ring, *, out=None,
                             boundary_states=None, workspace=None, n_chunks: int | None = None,
                             qk_l2norm: bool = False, stream=None):
    """Continuation prefill: each sequence continues from absolute position pos0[n] with
    ``state`` and ``ring`` (updated in place).  Returns (out, boundary_states, workspace).

    ``cu_seqlens`` and ``pos0`` are int32 CUDA tensors; ``n_chunks`` (the remainders' chunk
    count) is read from host copies of both when not given and boundary_states is None.
    """
    T, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[-1]
    N = cu_seqlens.numel() - 1
    dev = q.device
    if out is None:
        out = torch.empty(T, H, dv, dtype=q.dtype, device=dev)
    if boundary_states is None:
        if n_chunks is None:
            n_chunks = continue_chunks(cu_seqlens.cpu(), pos0.cpu(), C)
        boundary_states = torch.empty(max(n_chunks, 1), H, dk, dv, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(cpr_gdn_prefill_workspace_size(T, N, H, dk, dv, C), dtype=torch.uint8, device=dev)
    rc = ring._c()
    code = load_library().cpr_gdn_prefill_continue_grouped(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, Hk, _flags(qk_l2norm), dk, dv, C,
        _dtype_code(q), _ptr(pos0), _ptr(state), ctypes.byref(rc), _ptr(out), _ptr(boundary_states),
        boundary_states.shape[0],
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check("cpr_gdn_prefill_continue_grouped", code)
    return out, boundary_states, workspace


def cpr_gdn_decode(q, k, v, g, beta, state, ring: Ring, pos, C: int, *, out=None, workspace=None,
                   qk_l2norm: bool = False, stream=None):
    """One decode step for B sequences; ``state`` and ``ring`` are updated in place.  Returns (out, workspace)."""
    B, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[-1]
    if out is None:
        out = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = torch.empty(cpr_gdn_decode_workspace_size(B, H, dk, dv, C), dtype=torch.uint8, device=q.device)
    rc = ring._c()
    code = load_library().cpr_gdn_decode_grouped(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), ctypes.byref(rc), _ptr(pos), B, H, Hk,
        _flags(qk_l2norm), dk, dv, C, _dtype_code(q), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("cpr_gdn_decode_grouped", code)
    return out, workspace


def cpr_gdn_set_wait_test(extra_publications: int, limit_ns: int = 0) -> None:
    """Timeout-test hook: while extra_publications > 0 the prefill's intra-chunk items
    wait for publications that never come and give up after limit_ns (0: about 4 s),
    recording CPR_DEV_TIMEOUT.  (0, 0) restores normal operation."""
    _check("cpr_gdn_set_wait_test", load_library().cpr_gdn_set_wait_test(int(extra_publications), int(limit_ns)))


def cpr_gdn_device_status(workspace, stream=None) -> int:
    st = ctypes.c_uint32(0)
    code = load_library().cpr_gdn_device_status(_ptr(workspace), ctypes.byref(st), _stream(stream))
    _check("cpr_gdn_device_status", code)
    return int(st.value)


def cpr_gdn_set_profile_events(events) -> None:
    """Record the given torch.cuda.Event objects between the library's kernels (None: off)."""
    lib = load_library()
    if events is None:
        _check("cpr_gdn_set_profile_events", lib.cpr_gdn_set_profile_events(None, 0))
        return
    for e in events:  # make sure every event handle exists
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("cpr_gdn_set_profile_events", lib.cpr_gdn_set_profile_events(arr, len(events)))


def cpr_gdn_prefill_noalloc(q, k, v, g, beta, cu_seqlens, C: int, state_in=None, *, out, state_out,
                            boundary_states, stream=None):
    """Prefill without a caller workspace: the library's static scratch is used instead.

    For callers that must not allocate device memory while the layer runs (their runtime
    owns a fixed memory pool, or an allocation's device synchronisation is unacceptable).
    The caller passes every output buffer; this call allocates nothing.  Problems needing
    more than NOALLOC_SCRATCH_BYTES of scratch raise CprError (CPR_ERR_WORKSPACE).  The
    first call on a device looks up the scratch's address (make it before any stream
    capture); calls that overlap on the GPU race on the shared scratch.
    """
    T, H, dk = q.shape
    dv = v.shape[-1]
    if v.shape[1] != H:
        raise ValueError("cpr_gdn_prefill_noalloc takes one query/key head per value head")
    N = cu_seqlens.numel() - 1
    code = load_library().cpr_gdn_prefill_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H, dk, dv, C, _dtype_code(q),
        _ptr(state_in), _ptr(out), _ptr(state_out), _ptr(boundary_states), boundary_states.shape[0],
        _stream(stream))
    _check("cpr_gdn_prefill_noalloc", code)
    return out, state_out, boundary_states


def cpr_gdn_prefill_noalloc_status(stream=None) -> int:
    """Status word (CPR_DEV_* bits) of the last cpr_gdn_prefill_noalloc call on the current
    device, read from the library's scratch (waits for the stream)."""
    st = ctypes.c_uint32(0)
    code = load_library().cpr_gdn_prefill_noalloc_status(ctypes.byref(st), _stream(stream))
    _check("cpr_gdn_prefill_noalloc_status", code)
    return int(st.value)


def cpr_pik_workspace_size() -> int:
    return int(load_library().cpr_pik_workspace_size())


def cpr_pik_gemm(x, w, n_leaves: int, leaves=None, *, out=None, workspace=None, stream=None):
    """Deterministic K-split product Y = X W^T (x bf16 [M, K], w bf16 [N, K]; fp32 result):
    the subtree root of leaves [lo, hi) = ``leaves`` of the fixed n_leaves-leaf tree, or
    the whole product when ``leaves`` is None.  Returns (out, workspace)."""
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("x and w disagree on K")
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("x and w must be bf16")
    lo, hi = (0, n_leaves) if leaves is None else leaves
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(cpr_pik_workspace_size(), dtype=torch.uint8, device=x.device)
    code = load_library().cpr_pik_gemm(_ptr(x), _ptr(w), _ptr(out), M, N, K, n_leaves, lo, hi, _ptr(workspace),
                                       _stream(stream))
    _check("cpr_pik_gemm", code)
    return out, workspace


def cpr_pik_combine(parts, *, out=None, stream=None):
    """The top of the fixed tree over the subtree roots parts[0..P) (fp32 [P, ...]);
    returns out (fp32, the shape of parts[0])."""
    if parts.dtype != torch.float32:
        raise TypeError("parts must be fp32")
    P = parts.shape[0]
    if out is None:
        out = torch.empty(parts.shape[1:], dtype=torch.float32, device=parts.device)
    count = out.numel()
    if parts.numel() != P * count:
        raise ValueError("out must hold one part")
    code = load_library().cpr_pik_combine(_ptr(parts), P, count, _ptr(out), _stream(stream))
    _check("cpr_pik_combine", code)
    return out
