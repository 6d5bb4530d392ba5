"""CPU oracle of the deterministic K-split GEMM ("pik").

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this module.  The CUDA library
never imports or calls it, and this module never imports the CUDA library.

Source: "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section on the fixed
binary reduction tree (tensor parallelism: the pik implementation); "SkyRL IsoExec: vLLM
与 Megatron 的 logprob 差 ...", section on the unified model.  K is cut into contiguous
leaves; each leaf's partial product is accumulated in fp32 on the tensor cores; a fixed
binary tree over the leaves combines the partials, and the rank-to-leaf mapping is fixed.

Functions:

``leaf_bounds``    the K range of each leaf (contiguous, equal);
``rank_leaves``    the leaves a rank owns for a given rank count (contiguous block);
``tree_sum``       the fixed tree over adjacent parts, in fp32 rounded to nearest, exactly
                   as the method fixes it (bit-exact reference for the combine step);
``gemm_exact``     X W^T in fp64 from bf16-exact inputs: the value every correct pik result
                   approximates (products of bf16 values are exact in fp64, and the sums
                   over K lose at most fp64 rounding);
``error_bound``    a bound on |pik - exact| for fp32 accumulation over K terms plus the
                   tree's additions (standard gamma_n bound, n = K + log2(leaves)).

What the pages leave open, and the reading taken: the tensor cores' own rounding inside
one MMA instruction is the hardware's; the oracle therefore pins the GEMM to the exact
product within the accumulation bound, and pins the tree bit-exactly.
"""
from __future__ import annotations

import numpy as np


def leaf_bounds(K: int, n_leaves: int) -> list[tuple[int, int]]:
    """[(k_begin, k_end)] of each leaf: K cut into n_leaves contiguous, equal leaves."""
    if n_leaves < 1 or K % n_leaves:
        raise ValueError("K must split into n_leaves equal leaves")
    step = K // n_leaves
    return [(i * step, (i + 1) * step) for i in range(n_leaves)]


def rank_leaves(rank: int, n_ranks: int, n_leaves: int) -> tuple[int, int]:
    """Leaves [lo, hi) that rank `rank` of `n_ranks` owns: a contiguous block of
    n_leaves / n_ranks leaves in rank order (a complete subtree of the fixed tree)."""
    if n_ranks < 1 or n_leaves % n_ranks or not 0 <= rank < n_ranks:
        raise ValueError("the rank count must divide the leaf count")
    per = n_leaves // n_ranks
    return rank * per, (rank + 1) * per


def tree_sum(parts: list[np.ndarray]) -> np.ndarray:
    """The fixed binary tree over adjacent parts (a power of two of them): level by level,
    part 2i + 1 is added to part 2i in float32 with round-to-nearest, until one remains."""
    n = len(parts)
    if n < 1 or n & (n - 1):
        raise ValueError("the tree needs a power-of-two number of parts")
    level = [np.asarray(p, dtype=np.float32) for p in parts]
    while len(level) > 1:
        level = [np.add(level[2 * i], level[2 * i + 1], dtype=np.float32) for i in range(len(level) // 2)]
    return level[0]


def gemm_exact(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """X W^T in fp64 (x: [M, K], w: [N, K], both already bf16-representable)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def error_bound(x: np.ndarray, w: np.ndarray, n_leaves: int) -> np.ndarray:
    """Elementwise bound on |pik(x, w) - gemm_exact(x, w)|: gamma_n |X| |W|^T with
    n = K + log2(n_leaves) fp32 roundings on any path and u = 2^-24, doubled to allow the
    tensor cores a truncating rather than a rounding accumulator (u = 2^-23)."""
    K = x.shape[1]
    n = K + int(np.log2(n_leaves)) + 1
    u = 2.0 ** -23
    gamma = n * u / (1.0 - n * u)
    return gamma * (np.abs(np.asarray(x, np.float64)) @ np.abs(np.asarray(w, np.float64)).T)
