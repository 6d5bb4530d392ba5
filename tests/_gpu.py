"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and compare it with
the fp64 oracle (tolerances) and with itself (bit for bit)."""
from __future__ import annotations

import numpy as np
import torch

import linear_attention_cpr_gb300 as cpr
import oracle
from linear_attention_cpr_gb300 import inputs

# Tolerances against the fp64 oracle (unit-scale inputs): outputs rounded to bf16 within
# 2e-3 absolute; every (sequence, head) final state within 1e-4 relative Frobenius.
# fp32 outputs (the tiny workload) are held to 2e-5.
O_TOL_BF16 = 2e-3
O_TOL_F32 = 2e-5
STATE_RTOL = 1e-4


def dev():
    return torch.device("cuda", 0)


def to_dev(d: dict) -> dict:
    return {k: v.to(dev()) for k, v in d.items()}


def prefill(x: dict, C: int, state_in=None, n_chunks=None):
    out, st, bnd, ws = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                           state_in=state_in, n_chunks=n_chunks)
    torch.cuda.synchronize()
    status = cpr.cpr_gdn_device_status(ws)
    assert status == 0, f"device status {status}"
    return out, st, bnd


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    a, b = a.contiguous(), b.contiguous()
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    return bool(torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                            b.view(torch.uint8) if b.dtype != torch.uint8 else b))


def assert_close_to_oracle(o_gpu, st_gpu, o_ref, st_ref, o_tol, bnd_gpu=None, bnd_ref=None, what=""):
    o = o_gpu.float().cpu().double().numpy()
    err = np.abs(o - o_ref)
    max_err = float(err.max()) if err.size else 0.0
    assert max_err <= o_tol, f"{what}: max|do| = {max_err:.3e} > {o_tol} (max|o| = {np.abs(o_ref).max():.3f})"
    s = st_gpu.cpu().double().numpy()
    num = np.sqrt(((s - st_ref) ** 2).sum(axis=(-2, -1)))
    den = np.sqrt((st_ref ** 2).sum(axis=(-2, -1)))
    rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
    print(f"parity {what}: max|do| {max_err:.3e} (tol {o_tol}), state rel Frobenius {float(rel.max()):.3e}")
    assert float(rel.max()) <= STATE_RTOL, f"{what}: state rel Frobenius {float(rel.max()):.3e}"
    if bnd_gpu is not None:
        b = bnd_gpu.cpu().double().numpy()[: bnd_ref.shape[0]]
        num = np.sqrt(((b - bnd_ref) ** 2).sum(axis=(-2, -1)))
        den = np.sqrt((bnd_ref ** 2).sum(axis=(-2, -1)))
        rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
        assert float(rel.max()) <= STATE_RTOL, f"{what}: boundary rel Frobenius {float(rel.max()):.3e}"
    return max_err


def tokens(T, H, dk, dv, dtype, seed):
    q, k, v, g, beta = inputs.random_tokens(T, H, dk, dv, dtype=dtype, seed=seed)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def pack(seqs: list[dict]) -> dict:
    """Concatenate per-sequence token dicts into one packed batch (with cu_seqlens)."""
    out = {k: torch.cat([s[k] for s in seqs], dim=0).contiguous() for k in ("q", "k", "v", "g", "beta")}
    out["cu_seqlens"] = inputs.cu_seqlens_of([s["q"].shape[0] for s in seqs])
    return out


def slice_tokens(x: dict, a: int, b: int) -> dict:
    return {k: x[k][a:b].contiguous() for k in ("q", "k", "v", "g", "beta")}


def decode_run(prefix_seqs: list[dict], steps: list[dict], C: int, state_in=None):
    """Prefill the prefixes, build the ring, then run len(steps) decode steps.

    steps[s] holds the s-th new token of every sequence (q,k [B,H,dk] ...).
    Returns (list of per-step outputs [B,H,dv], final state [B,H,dk,dv]).
    """
    x = to_dev(pack(prefix_seqs))
    B = len(prefix_seqs)
    out, st, bnd = prefill(x, C, state_in=state_in)
    ring = cpr.cpr_gdn_ring_from_prefill(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd, st)
    state = st.clone()
    pos = torch.tensor([s["q"].shape[0] for s in prefix_seqs], dtype=torch.int32, device=dev())
    outs = []
    ws = None
    for tok in steps:
        t = to_dev(tok)
        o, ws = cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C, workspace=ws)
        outs.append(o.clone())
        pos += 1
    torch.cuda.synchronize()
    if ws is not None:
        assert cpr.cpr_gdn_device_status(ws) == 0
    return outs, state, ring
