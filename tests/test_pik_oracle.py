"""Pins of the pik oracle (oracle/pik.py) and the pik entry points' host-side checks (CPU).

The tree is pinned by hand-worked fp32 cases whose result changes with any other pairing
or order; the exact product by closed forms and brute force; the error bound by a plain
fp32 accumulation that must stay inside it; the rank-to-leaf mapping by its invariants.
"""
import ctypes
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import pik


def test_tree_pairs_neighbours_first():
    # 1e8 + 1 rounds to 1e8 in fp32 (spacing 8 there), and -1e8 + 1 to -1e8: the tree
    # ((a + b) + (c + d)) gives 0.  Left to right gives 1; strided pairs ((a + c) + (b + d))
    # give 2; the exact sum is 2.
    parts = [np.float32(1e8), np.float32(1), np.float32(-1e8), np.float32(1)]
    assert pik.tree_sum(parts) == np.float32(0.0)
    seq = np.float32(0)
    for p in parts:
        seq = np.float32(seq + p)
    assert seq == np.float32(1.0)


def test_tree_eight_parts_hand_worked():
    # level 1: (2^24 + 1) -> 2^24 (tie to even), (1 + 1) = 2, (-2^24 + 3) exact, (1 + 1) = 2
    # level 2: 2^24 + 2 exact, -2^24 + 5 exact;  level 3: 7.
    # Left to right: 2^24 + 1 + 1 + 1 stays 2^24 (each addition ties to even), then
    # + (-2^24 + 3) = 3, + 0 + 1 + 1 = 5.
    t = float(2 ** 24)
    parts = [t, 1.0, 1.0, 1.0, -t + 3.0, 0.0, 1.0, 1.0]
    parts = [np.float32(p) for p in parts]
    assert pik.tree_sum(parts) == np.float32(7.0)
    # and the pairwise structure: ((p0+p1)+(p2+p3)) + ((p4+p5)+(p6+p7))
    f = np.float32
    manual = f(f(f(parts[0] + parts[1]) + f(parts[2] + parts[3])) + f(f(parts[4] + parts[5]) + f(parts[6] + parts[7])))
    assert manual == np.float32(7.0)
    seq = np.float32(0)
    for p in parts:
        seq = np.float32(seq + p)
    assert seq == np.float32(5.0)


def test_tree_rank_invariance():
    rng = np.random.default_rng(0)
    leaves = [rng.standard_normal(257).astype(np.float32) * np.float32(10.0 ** rng.integers(-3, 4)) for _ in range(8)]
    whole = pik.tree_sum(leaves)
    for n_ranks in (1, 2, 4, 8):
        roots = []
        for r in range(n_ranks):
            lo, hi = pik.rank_leaves(r, n_ranks, 8)
            roots.append(pik.tree_sum(leaves[lo:hi]))
        assert np.array_equal(pik.tree_sum(roots), whole)


def test_tree_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        pik.tree_sum([np.zeros(2, np.float32)] * 3)


def test_leaf_and_rank_ranges():
    assert pik.leaf_bounds(512, 4) == [(0, 128), (128, 256), (256, 384), (384, 512)]
    for L in (1, 2, 4, 8):
        for P in (p for p in (1, 2, 4, 8) if L % p == 0):
            owned = [pik.rank_leaves(r, P, L) for r in range(P)]
            assert owned[0][0] == 0 and owned[-1][1] == L
            assert all(a[1] == b[0] for a, b in zip(owned, owned[1:]))
            assert all(hi - lo == L // P and lo % (hi - lo) == 0 for lo, hi in owned)
    with pytest.raises(ValueError):
        pik.rank_leaves(0, 3, 8)


def _bf16(a):
    """Round fp32 values to bf16 (nearest even) and return them as fp64."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def test_gemm_exact_closed_forms():
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((5, 64)))
    assert np.array_equal(pik.gemm_exact(x, np.eye(64)), x)
    h = np.array([[1.0]])
    for _ in range(3):
        h = np.block([[h, h], [h, -h]])
    assert np.array_equal(pik.gemm_exact(h, h), 8.0 * np.eye(8))  # H H^T = 8 I
    assert np.array_equal(pik.gemm_exact(np.ones((3, 96)), np.ones((2, 96))), np.full((3, 2), 96.0))


def test_gemm_exact_brute_force():
    rng = np.random.default_rng(2)
    x = _bf16(rng.standard_normal((3, 16)))
    w = _bf16(rng.standard_normal((4, 16)))
    ref = [[sum(Fraction(float(x[i, k])) * Fraction(float(w[j, k])) for k in range(16)) for j in range(4)]
           for i in range(3)]
    got = pik.gemm_exact(x, w)
    for i, j in itertools.product(range(3), range(4)):
        assert abs(Fraction(float(got[i, j])) - ref[i][j]) <= abs(ref[i][j]) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


def test_error_bound_covers_fp32_accumulation():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((4, 1024)))
    w = _bf16(rng.standard_normal((3, 1024)))
    exact = pik.gemm_exact(x, w)
    bound = pik.error_bound(x, w, 4)
    # a plain left-to-right fp32 accumulation per leaf, then the tree
    parts = []
    for k0, k1 in pik.leaf_bounds(1024, 4):
        acc = np.zeros((4, 3), np.float32)
        for k in range(k0, k1):
            acc = np.float32(acc + np.outer(x[:, k], w[:, k]).astype(np.float32))
        parts.append(acc)
    got = pik.tree_sum(parts).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound)
    assert np.all(bound > 0)
    # the bound is not vacuous: far below the magnitude scale |X||W|^T
    scale = np.abs(x) @ np.abs(w).T
    assert np.all(bound < 1e-3 * scale)


def test_entry_points_reject_bad_arguments():
    from linear_attention_cpr_gb300 import build
    build.build()
    import linear_attention_cpr_gb300 as cpr
    lib = cpr.load_library()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    ws = ctypes.c_void_p(1 << 21)
    bad = [
        (128, 128, 100, 1, 0, 1),   # K not a multiple of 64 * n_leaves
        (128, 128, 512, 3, 0, 3),   # leaf count not a power of two
        (128, 128, 512, 4, 1, 3),   # two leaves not aligned on a subtree
        (128, 128, 512, 4, 0, 3),   # three leaves
        (128, 128, 512, 4, 2, 6),   # beyond the leaves
        (0, 128, 512, 4, 0, 4),     # empty M
        (128, 128, 512, 16, 0, 16), # more than eight leaves
    ]
    for M, N, K, L, lo, hi in bad:
        assert lib.cpr_pik_gemm(fake, fake, fake, M, N, K, L, lo, hi, ws, None) == -1, (M, N, K, L, lo, hi)
    assert lib.cpr_pik_gemm(fake, fake, fake, 128, 128, 512, 4, 0, 4, None, None) == -4
    assert lib.cpr_pik_gemm(ctypes.c_void_p((1 << 20) + 8), fake, fake, 128, 128, 512, 4, 0, 4, ws, None) == -3
    assert lib.cpr_pik_combine(fake, 3, 16, fake, None) == -1
    assert lib.cpr_pik_combine(fake, 2, -1, fake, None) == -1
    assert lib.cpr_pik_combine(ctypes.c_void_p((1 << 20) + 4), 2, 16, fake, None) == -3
    assert lib.cpr_pik_combine(fake, 2, 0, fake, None) == 0
    assert lib.cpr_pik_workspace_size() >= 4


def _tree_pins_hold(tree):
    f = np.float32
    a = [f(1e8), f(1), f(-1e8), f(1)]
    t = float(2 ** 24)
    b = [f(p) for p in (t, 1.0, 1.0, 1.0, -t + 3.0, 0.0, 1.0, 1.0)]
    return tree(a) == f(0.0) and tree(b) == f(7.0)


def test_tree_pins_catch_planted_mistakes():
    def left_to_right(parts):
        acc = np.float32(parts[0])
        for p in parts[1:]:
            acc = np.float32(acc + p)
        return acc

    def strided(parts):  # pairs (i, i + n/2) first
        level = [np.float32(p) for p in parts]
        while len(level) > 1:
            h = len(level) // 2
            level = [np.float32(level[i] + level[i + h]) for i in range(h)]
        return level[0]

    def in_fp64(parts):
        return np.float32(sum(float(p) for p in parts))

    def right_first(parts):  # the tree with the operands of each addition swapped
        level = [np.float32(p) for p in parts]
        while len(level) > 1:
            level = [np.float32(level[2 * i + 1] + level[2 * i]) for i in range(len(level) // 2)]
        return level[0]

    assert _tree_pins_hold(pik.tree_sum)
    for mutant in (left_to_right, strided, in_fp64):
        assert not _tree_pins_hold(mutant), mutant.__name__
    # fp32 addition commutes: swapping operands is not a mistake and must pass
    assert _tree_pins_hold(right_first)


def test_binding_checks_before_any_device_work():
    import torch

    import linear_attention_cpr_gb300 as cpr
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        cpr.cpr_pik_gemm(x.float(), torch.zeros(4, 64, dtype=torch.bfloat16), 1)
    with pytest.raises(ValueError):
        cpr.cpr_pik_gemm(x, torch.zeros(4, 128, dtype=torch.bfloat16), 1)  # K disagrees
    with pytest.raises(TypeError):
        cpr.cpr_pik_combine(torch.zeros(2, 8, dtype=torch.float64))
