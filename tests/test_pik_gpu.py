"""The deterministic K-split product (pik) on the GPU, through the C ABI:
  - against the exact product (fp64 oracle) within the fp32-accumulation bound, on
    aligned and ragged shapes and every leaf count;
  - bit for bit the same result for every rank count that divides the leaf count (each
    rank's subtree root computed alone, then the top of the tree), and from call to call;
  - the combine step bit for bit against the oracle's fp32 tree;
  - the full-size product on sampled rows."""
import numpy as np
import pytest
import torch

import _gpu
import linear_attention_cpr_gb300 as cpr
from linear_attention_cpr_gb300 import build, inputs
from oracle import pik

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    cpr.load_library()


def _run(x, w, L, leaves=None):
    y, ws = cpr.cpr_pik_gemm(x, w, L, leaves)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    return y


def _check_oracle(x, w, y, L, rows=None):
    xs, ws_ = x.float().cpu().double().numpy(), w.float().cpu().double().numpy()
    yy = y.cpu().double().numpy()
    if rows is not None:
        xs, yy = xs[rows], yy[rows]
    exact = pik.gemm_exact(xs, ws_)
    bound = pik.error_bound(xs, ws_, L)
    err = np.abs(yy - exact)
    assert np.all(err <= bound), f"max err {err.max()} vs bound at that element {bound.flat[err.argmax()]}"


@pytest.mark.parametrize("M,N,K,L", [
    (128, 128, 64, 1),      # one tile, one stage
    (256, 256, 1024, 4),    # several tiles and stages per leaf
    (200, 136, 512, 4),     # ragged rows and columns
    (1, 1, 512, 8),         # a single element
    (300, 70, 2048, 8),     # ragged, eight leaves (64-column tiles)
    (130, 260, 384, 2),     # ragged, two leaves of three stages
])
def test_matches_exact_product(M, N, K, L):
    dev = _gpu.dev()
    x, w = inputs.gemm_operands(M, N, K, seed=M + N + K, device=dev)
    y = _run(x, w, L)
    _check_oracle(x, w, y, L)


@pytest.mark.parametrize("L", [2, 4, 8])
def test_rank_count_invariance(L):
    M, N, K = 384, 320, 64 * L * 5
    dev = _gpu.dev()
    x, w = inputs.gemm_operands(M, N, K, seed=L, device=dev)
    whole = _run(x, w, L)
    assert _gpu.bits_equal(whole, _run(x, w, L))  # call to call
    P = 1
    while P <= L:
        parts = torch.empty(P, M, N, dtype=torch.float32, device=dev)
        for r in range(P):
            lo, hi = pik.rank_leaves(r, P, L)
            cpr.cpr_pik_gemm(x, w, L, (lo, hi), out=parts[r])
        y = cpr.cpr_pik_combine(parts)
        torch.cuda.synchronize()
        assert _gpu.bits_equal(y, whole), f"{P} ranks of {L} leaves"
        P *= 2


def test_leaf_roots_are_the_oracle_tree_of_single_leaves():
    # every subtree root equals the oracle's fp32 tree over the single-leaf results
    L, M, N, K = 8, 256, 192, 64 * 8 * 3
    dev = _gpu.dev()
    x, w = inputs.gemm_operands(M, N, K, seed=11, device=dev)
    single = [_run(x, w, L, (l, l + 1)).cpu().numpy() for l in range(L)]
    for size in (2, 4, 8):
        for lo in range(0, L, size):
            root = _run(x, w, L, (lo, lo + size)).cpu().numpy()
            assert np.array_equal(root, pik.tree_sum(single[lo:lo + size])), (lo, size)


@pytest.mark.parametrize("P,count", [(1, 7), (2, 1000), (4, 4096 + 3), (8, 65536)])
def test_combine_bitwise(P, count):
    g = torch.Generator().manual_seed(P * 1000 + count)
    scale = torch.tensor([10.0 ** e for e in (-3, 0, 5, 8)])[torch.randint(0, 4, (P, count), generator=g)]
    parts = (torch.randn(P, count, generator=g) * scale).float()
    y = cpr.cpr_pik_combine(parts.to(_gpu.dev()))
    torch.cuda.synchronize()
    ref = pik.tree_sum([parts[p].numpy() for p in range(P)])
    assert np.array_equal(y.cpu().numpy(), ref)


def test_combine_in_place():
    g = torch.Generator().manual_seed(5)
    parts = torch.randn(4, 4096, generator=g).to(_gpu.dev())
    ref = pik.tree_sum([parts[p].cpu().numpy() for p in range(4)])
    cpr.cpr_pik_combine(parts, out=parts[0])
    torch.cuda.synchronize()
    assert np.array_equal(parts[0].cpu().numpy(), ref)


def test_rejects_bad_arguments():
    dev = _gpu.dev()
    x, w = inputs.gemm_operands(128, 128, 320, device=dev)
    with pytest.raises(cpr.CprError):
        cpr.cpr_pik_gemm(x, w, 4)          # K = 320 is not a multiple of 64 * 4
    with pytest.raises(cpr.CprError):
        cpr.cpr_pik_gemm(x, w, 5)
    x, w = inputs.gemm_operands(128, 128, 512, device=dev)
    with pytest.raises(cpr.CprError):
        cpr.cpr_pik_gemm(x, w, 4, (1, 3))  # not a subtree


@pytest.mark.slow
def test_full_size_sampled_rows():
    # the size bench.py times: M = N = K = 8192, eight leaves; rows checked one by one
    M = N = K = 8192
    dev = _gpu.dev()
    x, w = inputs.gemm_operands(M, N, K, seed=0, device=dev)
    y = _run(x, w, 8)
    rows = np.array([0, 1, 127, 128, 4095, 5000, 8190, 8191])
    _check_oracle(x, w, y, 8, rows=rows)
    parts = torch.empty(2, M, N, dtype=torch.float32, device=dev)
    for r in range(2):
        cpr.cpr_pik_gemm(x, w, 8, pik.rank_leaves(r, 2, 8), out=parts[r])
    assert _gpu.bits_equal(cpr.cpr_pik_combine(parts), y)
