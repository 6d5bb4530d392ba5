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
