"""fp64 CPU oracle of the backward pass of the gated delta rule (the layer's gradients).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU legs may import this module.  The CUDA library never imports or calls it, and this
module never imports the CUDA library.

Source: the pages time a CPR backward for the trainer ("IsoExec: Eliminating
Trainer-Inference Mismatch in SkyRL", section "Chunkwise-Parallel Recurrent (CPR) Gated
DeltaNet", per-layer table) but do not describe its algorithm.  The reading taken: CPR's
forward is the token recurrence of the Gated Delta Networks paper (Yang, Kautz &
Hatamizadeh, ICLR 2025) evaluated in a fixed order, so its backward is the adjoint of
that recurrence, run in reverse time; this module computes that adjoint exactly (fp64),
whatever chunk grid a GPU schedule uses.

Forward, per (sequence, head), S of shape dv x dk:
    S~_t = alpha_t S_{t-1},  alpha_t = exp(g_t)
    r_t  = v_t - S~_t k_t,   u_t = beta_t r_t
    S_t  = S~_t + u_t k_t^T,  o_t = S_t q_t
Reverse time, from dS = dL/dS_T (zero if the final state is unused):
    dS   += do_t q_t^T          dq_t  = S_t^T do_t
    du    = dS k_t              dk_t  = dS^T u_t
    dbeta_t = r_t . du          dr    = beta_t du,  dv_t = dr
    dS~   = dS - dr k_t^T       dk_t -= S~_t^T dr
    dg_t  = alpha_t <dS~, S_{t-1}>
    dS    = alpha_t dS~         (dL/dS_{t-1})
and dL/dS_0 is the last dS.  States are stored as [dk, dv] (element (j, i) holds S[i][j]),
as in the forward oracle.

``mutant`` plants one mistake for the pin tests: 1, the sign of the S~^T dr term of dk;
2, dg left out; 3, dq from the state before the token's update; 4, the decay left out of
the state's gradient.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def recurrent_backward(q, k, v, g, beta, cu_seqlens, d_out, d_state_out=None, state_in=None, mutant: int = 0):
    """Gradients of L = sum(d_out * o) + sum(d_state_out * state_out) with respect to every
    input of the plain recurrence over a packed batch.

    q, k [T, H, dk]; v, d_out [T, H, dv]; g, beta [T, H]; cu_seqlens [N + 1];
    state_in, d_state_out [N, H, dk, dv] or None (zeros).
    Returns dict(dq, dk, dv, dg, dbeta, d_state_in) in the same layouts."""
    q, k, v, g, beta, d_out = (_f64(x) for x in (q, k, v, g, beta, d_out))
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    s_in = np.zeros((N, H, dk, dv)) if state_in is None else _f64(state_in)
    ds_out = np.zeros((N, H, dk, dv)) if d_state_out is None else _f64(d_state_out)
    grads = {name: np.zeros_like(x) for name, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    d_state_in = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            t0, t1 = cu[n], cu[n + 1]
            S = s_in[n, h].T.copy()  # dv x dk
            prev, tilde, res, after = [], [], [], []
            for t in range(t0, t1):
                a = np.exp(g[t, h])
                St = a * S
                r = v[t, h] - St @ k[t, h]
                prev.append(S)
                tilde.append(St)
                res.append(r)
                S = St + np.outer(beta[t, h] * r, k[t, h])
                after.append(S)
            dS = ds_out[n, h].T.copy()
            for i in range(t1 - t0 - 1, -1, -1):
                t = t0 + i
                kt, qt, bt, a = k[t, h], q[t, h], beta[t, h], np.exp(g[t, h])
                r, St, Sp, Sa = res[i], tilde[i], prev[i], after[i]
                u = bt * r
                dS = dS + np.outer(d_out[t, h], qt)
                grads["dq"][t, h] = (Sp if mutant == 3 else Sa).T @ d_out[t, h]
                du = dS @ kt
                dkt = dS.T @ u
                grads["dbeta"][t, h] = r @ du
                dr = bt * du
                grads["dv"][t, h] = dr
                dSt = dS - np.outer(dr, kt)
                dkt = dkt + St.T @ dr if mutant == 1 else dkt - St.T @ dr
                grads["dk"][t, h] = dkt
                grads["dg"][t, h] = 0.0 if mutant == 2 else a * np.sum(dSt * Sp)
                dS = dSt if mutant == 4 else a * dSt
            d_state_in[n, h] = dS.T
    grads["d_state_in"] = d_state_in
    return grads


def chunked_backward(q, k, v, g, beta, cu_seqlens, d_out, C, d_state_out=None, state_in=None):
    """The same gradients by the chunk schedule a GPU backward would run (fp64):
    1. boundary states S_b by the forward recurrence (what a forward pass saves);
    2. per chunk, its transition P = A_1 ... A_n (A_t = alpha_t (I - beta_t k_t k_t^T) acting
       on the right of the row-vector state, S_t = S_{t-1} A_t + beta_t v_t k_t^T) and
       qt_t = P_t q_t (P_t = A_1 ... A_t);
    3. a reverse chain over each sequence's chunks: dS_b = dS_{b+1} P^T + sum_t do_t qt_t^T,
       from dS at the sequence's end;
    4. per chunk, the reverse token recurrence of ``recurrent_backward`` from dS_{b+1},
       with the states recomputed from S_b.
    Returns the dict of ``recurrent_backward`` plus ``chain_mismatch``: the largest
    difference between the chain's dS_b and the one each chunk's reverse recurrence arrives
    at (both exact up to rounding)."""
    q, k, v, g, beta, d_out = (_f64(x) for x in (q, k, v, g, beta, d_out))
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    s_in = np.zeros((N, H, dk, dv)) if state_in is None else _f64(state_in)
    ds_out = np.zeros((N, H, dk, dv)) if d_state_out is None else _f64(d_state_out)
    out = {name: np.zeros_like(x) for name, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    d_state_in = np.zeros((N, H, dk, dv))
    mismatch = 0.0
    eye = np.eye(dk)
    for n in range(N):
        for h in range(H):
            t0, t1 = cu[n], cu[n + 1]
            starts = list(range(t0, t1, C))
            # 1. boundary states
            S = s_in[n, h].T.copy()
            bounds = []
            for c0 in starts:
                bounds.append(S.copy())
                for t in range(c0, min(c0 + C, t1)):
                    a = np.exp(g[t, h])
                    St = a * S
                    S = St + np.outer(beta[t, h] * (v[t, h] - St @ k[t, h]), k[t, h])
            # 2. per-chunk transitions and propagated queries
            Ps, qts = [], []
            for c0 in starts:
                P = eye.copy()
                qt = []
                for t in range(c0, min(c0 + C, t1)):
                    A = np.exp(g[t, h]) * (eye - beta[t, h] * np.outer(k[t, h], k[t, h]))
                    P = P @ A
                    qt.append(P @ q[t, h])
                Ps.append(P)
                qts.append(qt)
            # 3. reverse chain: dS at every chunk's end, then its start
            d_end = [None] * len(starts)
            dS = ds_out[n, h].T.copy()
            d_start = [None] * len(starts)
            for j in range(len(starts) - 1, -1, -1):
                d_end[j] = dS.copy()
                c0 = starts[j]
                dS = dS @ Ps[j].T
                for i, t in enumerate(range(c0, min(c0 + C, t1))):
                    dS = dS + np.outer(d_out[t, h], qts[j][i])
                d_start[j] = dS.copy()
            d_state_in[n, h] = dS.T if starts else ds_out[n, h]
            # 4. per-chunk reverse token recurrence from the chunk's end adjoint
            for j, c0 in enumerate(starts):
                c1 = min(c0 + C, t1)
                sub = slice(c0, c1)
                gr = recurrent_backward(q[sub, h:h + 1], k[sub, h:h + 1], v[sub, h:h + 1], g[sub, h:h + 1],
                                        beta[sub, h:h + 1], [0, c1 - c0], d_out[sub, h:h + 1],
                                        d_state_out=d_end[j].T[None, None], state_in=bounds[j].T[None, None])
                for name in ("dq", "dk", "dv", "dg", "dbeta"):
                    out[name][sub, h] = gr[name][:, 0]
                mismatch = max(mismatch, float(np.max(np.abs(gr["d_state_in"][0, 0] - d_start[j].T))))
    out["d_state_in"] = d_state_in
    out["chain_mismatch"] = mismatch
    return out


def _wy_chunk_forward(Sb, Q, K, V, g, b):
    """One chunk of n tokens in the WY form (fp64): S_b (dv x dk) and the chunk's
    q, k [n, dk], v [n, dv], g, beta [n].  Returns the intermediates the adjoint needs."""
    n = len(g)
    G = np.cumsum(g)
    gam = np.exp(G)
    low = np.tril(np.ones((n, n)), -1)  # i < r
    lowd = np.tril(np.ones((n, n)))     # i <= r
    E = np.exp(G[:, None] - G[None, :]) * lowd
    KK = K @ K.T
    L = KK * E * low
    A = b[:, None] * L
    T = np.linalg.inv(np.eye(n) + A)
    Ut = T @ (b[:, None] * V)
    W = T @ ((b * gam)[:, None] * K)
    U = Ut - W @ Sb.T
    Pm = (Q @ K.T) * E  # lower with diagonal
    O = gam[:, None] * (Q @ Sb.T) + Pm @ U
    d = np.exp(G[-1] - G)
    S_end = gam[-1] * Sb + U.T @ (d[:, None] * K)
    return dict(G=G, gam=gam, low=low, E=E, KK=KK, L=L, T=T, Ut=Ut, W=W, U=U, Pm=Pm, O=O, d=d, S_end=S_end)


def _wy_chunk_backward(Sb, Q, K, V, g, b, dO, dS_end):
    """Adjoint of one chunk in the WY form: returns (dS_b, dq, dk, dv, dg, dbeta)."""
    f = _wy_chunk_forward(Sb, Q, K, V, g, b)
    G, gam, low, E, KK, L, T, W, U, Pm, d = (f[x] for x in ("G", "gam", "low", "E", "KK", "L", "T", "W", "U", "Pm", "d"))
    n = len(g)
    dSb = np.zeros_like(Sb)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dgam, dd, db = np.zeros(n), np.zeros(n), np.zeros(n)
    # S_end = gam_last S_b + U^T diag(d) K
    dSb += gam[-1] * dS_end
    dgam[-1] += np.sum(dS_end * Sb)
    dU = (d[:, None] * K) @ dS_end.T
    UdS = U @ dS_end
    dK += d[:, None] * UdS
    dd += np.sum(UdS * K, axis=1)
    # O = diag(gam) Q S_b^T + Pm U
    dQ += gam[:, None] * (dO @ Sb)
    dSb += dO.T @ (gam[:, None] * Q)
    dgam += np.sum(dO * (Q @ Sb.T), axis=1)
    dPm = (dO @ U.T) * np.tril(np.ones((n, n)))
    dU += Pm.T @ dO
    dQK = dPm * E
    dQ += dQK @ K
    dK += dQK.T @ Q
    dE = dPm * (Q @ K.T)
    # U = Ut - W S_b^T
    dUt = dU
    dW = -dU @ Sb
    dSb += -dU.T @ W
    # Ut = T diag(b) V,  W = T diag(b gam) K
    bV, bgK = b[:, None] * V, (b * gam)[:, None] * K
    dT = dUt @ bV.T + dW @ bgK.T
    TdUt, TdW = T.T @ dUt, T.T @ dW
    dV += b[:, None] * TdUt
    db += np.sum(TdUt * V, axis=1) + gam * np.sum(TdW * K, axis=1)
    dK += (b * gam)[:, None] * TdW
    dgam += b * np.sum(TdW * K, axis=1)
    # T = (I + A)^-1,  A = diag(b) L  (strictly lower)
    dA = -(T.T @ dT @ T.T) * low
    db += np.sum(dA * L, axis=1)
    dL = b[:, None] * dA
    # L = (K K^T) o E o low
    dKK = dL * E * low
    dK += (dKK + dKK.T) @ K
    dE += dL * KK * low
    # the gates: gam_r = e^{G_r}, d_i = e^{G_last - G_i}, E_ri = e^{G_r - G_i}
    dG = gam * dgam
    dG[-1] += np.sum(d * dd)
    dG -= d * dd
    ED = E * dE
    dG += np.sum(ED, axis=1) - np.sum(ED, axis=0)
    dg = np.cumsum(dG[::-1])[::-1]  # G = cumsum(g)
    return dSb, dQ, dK, dV, dg, db


def wy_chunked_backward(q, k, v, g, beta, cu_seqlens, d_out, C, d_state_out=None, state_in=None):
    """The same gradients with every chunk's adjoint taken through the WY form (fp64):
    the in-chunk work is matrix products (what tensor cores would run), and each chunk
    hands dS_b to the previous one.  Same returns as ``recurrent_backward``."""
    q, k, v, g, beta, d_out = (_f64(x) for x in (q, k, v, g, beta, d_out))
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    s_in = np.zeros((N, H, dk, dv)) if state_in is None else _f64(state_in)
    ds_out = np.zeros((N, H, dk, dv)) if d_state_out is None else _f64(d_state_out)
    out = {name: np.zeros_like(x) for name, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    d_state_in = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            t0, t1 = cu[n], cu[n + 1]
            starts = list(range(t0, t1, C))
            bounds, S = [], s_in[n, h].T.copy()
            for c0 in starts:
                bounds.append(S)
                sl = slice(c0, min(c0 + C, t1))
                S = _wy_chunk_forward(S, q[sl, h], k[sl, h], v[sl, h], g[sl, h], beta[sl, h])["S_end"]
            dS = ds_out[n, h].T.copy()
            for j in range(len(starts) - 1, -1, -1):
                sl = slice(starts[j], min(starts[j] + C, t1))
                dS, dQ, dK, dV, dg, db = _wy_chunk_backward(bounds[j], q[sl, h], k[sl, h], v[sl, h], g[sl, h],
                                                            beta[sl, h], d_out[sl, h], dS)
                out["dq"][sl, h], out["dk"][sl, h], out["dv"][sl, h] = dQ, dK, dV
                out["dg"][sl, h], out["dbeta"][sl, h] = dg, db
            d_state_in[n, h] = dS.T
    out["d_state_in"] = d_state_in
    return out
