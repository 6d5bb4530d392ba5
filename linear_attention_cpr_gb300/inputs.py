"""Seeded synthetic inputs shaped like the CPR Gated DeltaNet workloads.

This module holds no arithmetic of the method: it only draws the layer's inputs.  It is
the one module that both the CUDA path's callers and the fp64 oracle's callers use, so
that both see the same values.

Value recipe (every workload):
  q, k ~ N(0, 1), each (token, head) vector L2-normalised over its dk entries; q is then
  scaled by dk**-0.5;  v ~ N(0, 1);  g = log(alpha) = -0.5 * softplus(N(0, 1));
  beta = sigmoid(N(0, 1));  initial state S_0 = 0.  q, k, v are rounded to bf16 unless
  the workload is fp32; g and beta stay fp32.  Draw order: q, k, v, g, beta.

The pages measure real model activations (the hybrid model's GDN layers during RL on a
math-problem dataset); those are not available, and these synthetic tensors stand in for them
with the shapes the pages' per-layer table quotes (1 x 10,240 tokens for the trainer,
5 x 2,048 for rollout prefill, 256 sequences x 1 token for rollout decode).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    H: int
    dk: int
    dv: int
    C: int
    dtype: torch.dtype
    seqlens: list[int]
    decode_steps: int = 0
    seed: int = 0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))


def _lengths_uniform(n: int, lo: int, hi: int, seed: int) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def _lengths_loguniform(n: int, lo: int, hi: int, seed: int) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def workload(name: str) -> Workload:
    """The five named workloads (sizes exactly as the benchmark configuration lists them)."""
    if name == "tiny":
        return Workload("tiny", H=2, dk=32, dv=32, C=16, dtype=torch.float32, seqlens=[256],
                        decode_steps=256, note="B=1, T=256, fp32; prefill vs 256 decode steps")
    if name == "trainer_fwd":
        return Workload("trainer_fwd", H=16, dk=128, dv=128, C=64, dtype=torch.bfloat16,
                        seqlens=[10240], note="1 x 10,240 tokens")
    if name == "rollout_prefill":
        return Workload("rollout_prefill", H=16, dk=128, dv=128, C=64, dtype=torch.bfloat16,
                        seqlens=[2048] * 5, note="5 x 2,048 tokens packed")
    if name == "rollout_decode":
        return Workload("rollout_decode", H=16, dk=128, dv=128, C=64, dtype=torch.bfloat16,
                        seqlens=_lengths_uniform(256, 1, 4096, seed=0), decode_steps=512,
                        note="256 sequences x 1 token, prior lengths U[1,4096], 512 steps")
    if name == "varlen_stress":
        return Workload("varlen_stress", H=32, dk=128, dv=128, C=64, dtype=torch.bfloat16,
                        seqlens=_lengths_loguniform(32, 64, 8192, seed=0), decode_steps=128,
                        note="32 packed sequences, lengths log-uniform in [64, 8192]")
    raise KeyError(name)


WORKLOADS = ("tiny", "trainer_fwd", "rollout_prefill", "rollout_decode", "varlen_stress")


def cu_seqlens_of(seqlens) -> torch.Tensor:
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def draw_tokens(T: int, H: int, dk: int, dv: int, dtype: torch.dtype, gen: torch.Generator,
                device="cpu"):
    """(q, k, v, g, beta) for T tokens: q,k [T,H,dk], v [T,H,dv] in ``dtype``; g, beta [T,H] fp32."""
    f32 = torch.float32
    q = torch.randn(T, H, dk, generator=gen, dtype=f32, device=device)
    k = torch.randn(T, H, dk, generator=gen, dtype=f32, device=device)
    v = torch.randn(T, H, dv, generator=gen, dtype=f32, device=device)
    g_raw = torch.randn(T, H, generator=gen, dtype=f32, device=device)
    b_raw = torch.randn(T, H, generator=gen, dtype=f32, device=device)
    q = torch.nn.functional.normalize(q, dim=-1) * (dk ** -0.5)
    k = torch.nn.functional.normalize(k, dim=-1)
    g = -0.5 * torch.nn.functional.softplus(g_raw)
    beta = torch.sigmoid(b_raw)
    return (q.to(dtype).contiguous(), k.to(dtype).contiguous(), v.to(dtype).contiguous(),
            g.contiguous(), beta.contiguous())


def prefill_inputs(w: Workload, seed: int | None = None, device="cpu"):
    """Packed prefill inputs of a workload: dict(q, k, v, g, beta, cu_seqlens)."""
    gen = torch.Generator(device=device).manual_seed(w.seed if seed is None else seed)
    q, k, v, g, beta = draw_tokens(w.total_tokens, w.H, w.dk, w.dv, w.dtype, gen, device)
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens_of(w.seqlens).to(device))


def decode_inputs(w: Workload, step: int, seed: int | None = None, device="cpu"):
    """One decode step's new tokens for every sequence: q,k [B,H,dk], v [B,H,dv], g,beta [B,H]."""
    base = w.seed if seed is None else seed
    gen = torch.Generator(device=device).manual_seed(1_000_003 * (step + 1) + base)
    q, k, v, g, beta = draw_tokens(len(w.seqlens), w.H, w.dk, w.dv, w.dtype, gen, device)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def random_tokens(T: int, H: int, dk: int, dv: int, dtype=torch.float32, seed: int = 0, device="cpu"):
    """Tokens with the workload value recipe for arbitrary small shapes (tests)."""
    gen = torch.Generator(device=device).manual_seed(seed)
    return draw_tokens(T, H, dk, dv, dtype, gen, device)


def gemm_operands(M: int, N: int, K: int, seed: int = 0, device="cpu"):
    """Operands of the deterministic K-split product Y = X W^T: x [M, K] and w [N, K] in
    bf16, entries N(0, 1) rounded to bf16 (the scale of normalised activations and of a
    unit-variance weight; the product's entries then have standard deviation sqrt(K)).
    Draw order: x, then w."""
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=gen).to(torch.bfloat16)
    w = torch.randn(N, K, generator=gen).to(torch.bfloat16)
    return x.to(device), w.to(device)
