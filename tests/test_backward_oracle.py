"""Pins of the backward oracle (oracle/backward.py, the exact adjoint of the gated delta
rule), CPU only: central finite differences of the pinned forward oracle, a single-token
closed form, and planted mistakes that the pins must catch."""
import numpy as np
import pytest

import oracle
from oracle import backward


def _problem(seed, lens=(4, 2), H=2, dk=3, dv=2):
    rng = np.random.default_rng(seed)
    T, N = sum(lens), len(lens)
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    x = dict(
        q=rng.standard_normal((T, H, dk)) * dk ** -0.5,
        k=k,
        v=rng.standard_normal((T, H, dv)),
        g=-0.5 * np.log1p(np.exp(rng.standard_normal((T, H)))),
        beta=1.0 / (1.0 + np.exp(-rng.standard_normal((T, H)))),
        state_in=rng.standard_normal((N, H, dk, dv)) * 0.5,
    )
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    d_out = rng.standard_normal((T, H, dv))
    d_state = rng.standard_normal((N, H, dk, dv))
    return x, cu, d_out, d_state


def _loss(x, cu, d_out, d_state):
    o, st, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, 4, state_in=x["state_in"],
                                boundaries=False)
    return float(np.sum(d_out * o) + np.sum(d_state * st))


def _fd_grads(x, cu, d_out, d_state, h=1e-6):
    out = {}
    for name in ("q", "k", "v", "g", "beta", "state_in"):
        grad = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            grad[idx] = (_loss(xp, cu, d_out, d_state) - _loss(xm, cu, d_out, d_state)) / (2 * h)
        out[name] = grad
    return out


_NAMES = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "state_in": "d_state_in"}


def _matches_fd(grads, fd):
    return all(np.allclose(grads[_NAMES[n]], fd[n], rtol=1e-6, atol=1e-7) for n in fd)


@pytest.fixture(scope="module")
def case():
    oracle.build()
    x, cu, d_out, d_state = _problem(0)
    return x, cu, d_out, d_state, _fd_grads(x, cu, d_out, d_state)


def test_backward_matches_finite_differences(case):
    x, cu, d_out, d_state, fd = case
    grads = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, d_out, d_state,
                                        state_in=x["state_in"])
    for n in fd:
        np.testing.assert_allclose(grads[_NAMES[n]], fd[n], rtol=1e-6, atol=1e-7, err_msg=n)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4])
def test_finite_differences_catch_planted_mistakes(case, mutant):
    x, cu, d_out, d_state, fd = case
    grads = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, d_out, d_state,
                                        state_in=x["state_in"], mutant=mutant)
    assert not _matches_fd(grads, fd)


def test_single_token_closed_form():
    # S_0 = 0, one token: o = beta (k . q) v, S_1 = beta v k^T.  With L = dO . o:
    #   dq = beta (dO . v) k,  dk = beta (dO . v) q,  dv = beta (k . q) dO,
    #   dbeta = (k . q)(dO . v),  dg = 0,
    #   dL/dS_0 = alpha (dO q^T - beta (k . q) dO k^T)   (S is dv x dk; stored transposed)
    rng = np.random.default_rng(3)
    dk_, dv_ = 4, 3
    q, k, v = rng.standard_normal((1, 1, dk_)), rng.standard_normal((1, 1, dk_)), rng.standard_normal((1, 1, dv_))
    g, beta = np.array([[-0.3]]), np.array([[0.7]])
    dO = rng.standard_normal((1, 1, dv_))
    gr = backward.recurrent_backward(q, k, v, g, beta, [0, 1], dO)
    qq, kk, vv, d = q[0, 0], k[0, 0], v[0, 0], dO[0, 0]
    b, a = 0.7, np.exp(-0.3)
    np.testing.assert_allclose(gr["dq"][0, 0], b * (d @ vv) * kk, rtol=1e-13)
    np.testing.assert_allclose(gr["dk"][0, 0], b * (d @ vv) * qq, rtol=1e-13)
    np.testing.assert_allclose(gr["dv"][0, 0], b * (kk @ qq) * d, rtol=1e-13)
    np.testing.assert_allclose(gr["dbeta"][0, 0], (kk @ qq) * (d @ vv), rtol=1e-13)
    assert gr["dg"][0, 0] == 0.0
    dS0 = a * (np.outer(d, qq) - b * (kk @ qq) * np.outer(d, kk))
    np.testing.assert_allclose(gr["d_state_in"][0, 0], dS0.T, rtol=1e-13, atol=1e-15)


def test_zero_upstream_gives_zero_gradients():
    x, cu, d_out, d_state = _problem(5)
    gr = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, np.zeros_like(d_out),
                                     state_in=x["state_in"])
    assert all(not np.any(gr[n]) for n in gr)


@pytest.mark.parametrize("C", [1, 2, 3, 4, 8])
def test_chunked_schedule_equals_token_adjoint(C):
    x, cu, d_out, d_state = _problem(7, lens=(9, 0, 5, 1), H=2, dk=4, dv=3)
    ref = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, d_out, d_state,
                                      state_in=x["state_in"])
    got = backward.chunked_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, d_out, C, d_state,
                                    state_in=x["state_in"])
    for name in ref:
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-10, atol=1e-12, err_msg=name)
    assert got["chain_mismatch"] < 1e-12


@pytest.mark.parametrize("C,lens,dk,dv", [(1, (9, 0, 5, 1), 4, 3), (3, (9, 0, 5, 1), 4, 3), (8, (9, 0, 5, 1), 4, 3),
                                          (16, (40, 17), 8, 6)])
def test_wy_chunk_adjoint_equals_token_adjoint(C, lens, dk, dv):
    # every chunk's adjoint through the WY form (matrix products only) = the token adjoint
    x, cu, d_out, d_state = _problem(11, lens=lens, H=2, dk=dk, dv=dv)
    ref = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, d_out, d_state,
                                      state_in=x["state_in"])
    got = backward.wy_chunked_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, d_out, C, d_state,
                                       state_in=x["state_in"])
    for name in ref:
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-9, atol=1e-11, err_msg=name)


def test_chain_terms_in_wy_form():
    # the chain's per-chunk terms from the forward's WY intermediates: the chunk map
    # M = P = gamma_n I - W^T diag(d) K, and the propagated queries
    # P_t q_t = (diag(gamma) Q - ((Q K^T) o D) W)_t, against the products of the token
    # transitions A_t = alpha_t (I - beta_t k_t k_t^T)
    rng = np.random.default_rng(13)
    n, dk, dv = 7, 5, 4
    K = rng.standard_normal((n, dk))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    Q = rng.standard_normal((n, dk))
    V = rng.standard_normal((n, dv))
    g = -0.5 * np.log1p(np.exp(rng.standard_normal(n)))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(n)))
    f = backward._wy_chunk_forward(np.zeros((dv, dk)), Q, K, V, g, b)
    P, qt = np.eye(dk), []
    for t in range(n):
        P = P @ (np.exp(g[t]) * (np.eye(dk) - b[t] * np.outer(K[t], K[t])))
        qt.append(P @ Q[t])
    M = f["gam"][-1] * np.eye(dk) - f["W"].T @ (f["d"][:, None] * K)
    np.testing.assert_allclose(M, P, rtol=1e-12, atol=1e-14)
    Qt = f["gam"][:, None] * Q - f["Pm"] @ f["W"]
    np.testing.assert_allclose(Qt, np.array(qt), rtol=1e-12, atol=1e-14)
