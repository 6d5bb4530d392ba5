"""The fp64 oracle against brute force, exact arithmetic, a hand-derived example,
closed forms and invariants of the gated delta rule (CPU only)."""
import numpy as np
import pytest

import _pins
import oracle


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    ok, detail = pin()
    assert ok, detail


def test_packing_invariance_exact():
    """Each (sequence, head) is computed alone: packing changes no bit of the oracle."""
    lens = [7, 30, 1, 18]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, beta, cu, s0 = _pins.random_problem(31, int(cu[-1]), 3, 6, 5, cu=cu)
    o, st, bnd = oracle.recurrent(q, k, v, g, beta, cu, C=8, state_in=s0)
    c = 0
    for n, L in enumerate(lens):
        sl = slice(int(cu[n]), int(cu[n + 1]))
        o1, st1, b1 = oracle.recurrent(q[sl], k[sl], v[sl], g[sl], beta[sl], [0, L], C=8,
                                       state_in=s0[n:n + 1])
        assert np.array_equal(o1, o[sl]) and np.array_equal(st1[0], st[n])
        assert np.array_equal(b1, bnd[c:c + len(b1)])
        c += len(b1)
    assert c == len(bnd)


def test_empty_sequences_keep_state():
    q, k, v, g, beta, _, s0 = _pins.random_problem(37, 4, 1, 4, 4, cu=[0, 0, 4, 4])
    cu = np.array([0, 0, 4, 4], dtype=np.int32)
    o, st, bnd = oracle.recurrent(q, k, v, g, beta, cu, C=2, state_in=s0)
    assert np.array_equal(st[0], s0[0]) and np.array_equal(st[2], s0[2])
    assert bnd.shape[0] == 2


def test_threads_do_not_change_bits():
    q, k, v, g, beta, cu, s0 = _pins.random_problem(41, 50, 4, 8, 8, cu=[0, 20, 50])
    a = oracle.recurrent(q, k, v, g, beta, cu, C=16, state_in=s0, n_threads=1)
    b = oracle.recurrent(q, k, v, g, beta, cu, C=16, state_in=s0, n_threads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_rejects_bad_cu_seqlens():
    q, k, v, g, beta, _, _ = _pins.random_problem(43, 4, 1, 2, 2)
    with pytest.raises(ValueError):
        oracle.recurrent(q, k, v, g, beta, [0, 3], C=2)
    with pytest.raises(RuntimeError):
        oracle.recurrent(q, k, v, g, beta, [0, 3, 2, 4], C=2)
