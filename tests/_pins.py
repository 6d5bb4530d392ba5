"""Pins of the fp64 oracle against facts fixed by the mathematics, not by the oracle itself.

Each pin returns (ok, detail).  tests/test_oracle_pins.py asserts every pin on the real
oracle; tests/test_oracle_mutants.py builds the oracle with planted mistakes and checks
that every mistake makes at least one pin fail.

The recurrence is the gated delta rule named by "IsoExec: Eliminating Trainer-Inference
Mismatch in SkyRL", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet", in the
form of the Gated Delta Networks paper:
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _unit_rows(a):
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


def random_problem(seed, T, H, dk, dv, cu=None, state=True):
    r = _rng(seed)
    q = _unit_rows(r.standard_normal((T, H, dk))) * dk ** -0.5
    k = _unit_rows(r.standard_normal((T, H, dk)))
    v = r.standard_normal((T, H, dv))
    g = -0.5 * np.log1p(np.exp(r.standard_normal((T, H))))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))
    cu = np.array([0, T] if cu is None else cu, dtype=np.int32)
    s0 = r.standard_normal((len(cu) - 1, H, dk, dv)) * 0.3 if state else None
    return q, k, v, g, beta, cu, s0


def _close(a, b, tol):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 0.0)
    return err <= tol * scale, err


# --- brute force: materialised transition products (T <= 8, d <= 4) -------------------

def pin_bruteforce(mutant=0):
    worst = 0.0
    for seed, (T, dk, dv) in enumerate([(1, 2, 2), (3, 3, 2), (5, 4, 4), (8, 4, 3), (7, 2, 4)]):
        q, k, v, g, beta, cu, s0 = random_problem(100 + seed, T, 1, dk, dv)
        o, st, _ = oracle.recurrent(q, k, v, g, beta, cu, C=4, state_in=s0, mutant=mutant)
        ob, stb = oracle.bruteforce(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0=s0[0, 0])
        ok1, e1 = _close(o[:, 0], ob, 1e-12)
        ok2, e2 = _close(st[0, 0], stb, 1e-12)
        worst = max(worst, e1, e2)
        if not (ok1 and ok2):
            return False, f"recurrence vs transition products: {max(e1, e2):.3e} at T={T}"
    return True, f"max err {worst:.3e}"


# --- exact rational brute force, independent of the C code ----------------------------

def _exact_states(q, k, v, alpha, beta, S0):
    """S_t by the transition-product form in exact rational arithmetic (math layout)."""
    T, dk = len(k), len(k[0])
    dv = len(v[0])
    Mt = []
    for t in range(T):
        Mt.append([[alpha[t] * ((1 if r == c else 0) - beta[t] * k[t][r] * k[t][c]) for c in range(dk)]
                   for r in range(dk)])

    def mm(A, B):
        return [[sum(A[i][l] * B[l][j] for l in range(len(B))) for j in range(len(B[0]))]
                for i in range(len(A))]

    outs, states = [], []
    for t in range(T):
        P = [[Fraction(int(r == c)) for c in range(dk)] for r in range(dk)]
        for s in range(t + 1):
            P = mm(P, Mt[s])
        S = mm(S0, P)
        for s in range(t + 1):
            term = [[beta[s] * v[s][i] * k[s][j] for j in range(dk)] for i in range(dv)]
            for u in range(s + 1, t + 1):
                term = mm(term, Mt[u])
            S = [[S[i][j] + term[i][j] for j in range(dk)] for i in range(dv)]
        states.append(S)
        outs.append([sum(S[i][j] * q[t][j] for j in range(dk)) for i in range(dv)])
    return outs, states


def pin_exact_rational(mutant=0):
    r = _rng(7)
    T, dk, dv = 4, 3, 2
    # dyadic rationals: exactly representable, so the oracle sees the same numbers
    k = (r.integers(-8, 9, (T, dk)) / 8.0)
    q = (r.integers(-8, 9, (T, dk)) / 8.0)
    v = (r.integers(-8, 9, (T, dv)) / 4.0)
    beta = np.array([0.5, 0.25, 0.75, 1.0])
    g = np.log(np.array([1.0, 0.5, 0.75, 0.25]))
    alpha = [Fraction(math.exp(x)) for x in g]  # the exact double the oracle exponentiates to
    S0 = (r.integers(-4, 5, (dk, dv)) / 4.0)
    F = lambda a: [[Fraction(float(x)) for x in row] for row in a]
    S0m = [[Fraction(float(S0[j, i])) for j in range(dk)] for i in range(dv)]
    outs, states = _exact_states(F(q), F(k), F(v), alpha, [Fraction(float(b)) for b in beta], S0m)
    o, st, _ = oracle.recurrent(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                                [0, T], C=2, state_in=S0[None, None], mutant=mutant)
    ref_o = np.array([[float(x) for x in row] for row in outs])
    ref_s = np.array([[float(states[-1][i][j]) for i in range(dv)] for j in range(dk)])
    ok1, e1 = _close(o[:, 0], ref_o, 1e-13)
    ok2, e2 = _close(st[0, 0], ref_s, 1e-13)
    return ok1 and ok2, f"exact rational brute force: {max(e1, e2):.3e}"


# --- hand-derived worked example (tests/golden) ---------------------------------------

def load_golden(name="gdn_hand_example.txt"):
    rec = {"token": [], "out": [], "boundary": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key in ("dk", "dv", "C"):
                rec[key] = int(vals[0])
            elif key in rec:
                rec[key].append([float(x) for x in vals])
            else:
                rec[key] = [float(x) for x in vals]
    return rec


def pin_golden(mutant=0):
    gd = load_golden()
    dk, dv, C = gd["dk"], gd["dv"], gd["C"]
    tok = np.array(gd["token"])
    T = len(tok)
    k, v, q = tok[:, 0:dk], tok[:, dk:dk + dv], tok[:, dk + dv:2 * dk + dv]
    alpha, beta = tok[:, -2], tok[:, -1]
    g = np.log(alpha)
    o, st, bnd = oracle.recurrent(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                                  [0, T], C=C, mutant=mutant)
    ok1, e1 = _close(o[:, 0], np.array(gd["out"]), 1e-14)
    ok2, e2 = _close(st[0, 0].reshape(-1), np.array(gd["state_out"]), 1e-14)
    ok3, e3 = _close(bnd[:, 0].reshape(len(gd["boundary"]), -1), np.array(gd["boundary"]), 1e-14)
    return ok1 and ok2 and ok3, f"hand example: o {e1:.1e} state {e2:.1e} boundary {e3:.1e}"


# --- closed forms ----------------------------------------------------------------------

def pin_beta_zero_decay(mutant=0):
    """beta = 0: S_t = (alpha_1 ... alpha_t) S_0, o_t = S_t q_t."""
    q, k, v, g, beta, cu, s0 = random_problem(11, 9, 2, 4, 3)
    beta[:] = 0.0
    o, st, _ = oracle.recurrent(q, k, v, g, beta, cu, C=4, state_in=s0, mutant=mutant)
    G = np.cumsum(g, axis=0)  # [T, H]
    want_s = np.exp(G[-1])[:, None, None] * s0[0]
    want_o = np.einsum("th,hji,thj->thi", np.exp(G), s0[0], q)
    ok1, e1 = _close(st[0], want_s, 1e-13)
    ok2, e2 = _close(o, want_o, 1e-13)
    return ok1 and ok2, f"pure decay: {max(e1, e2):.3e}"


def pin_orthonormal_recall(mutant=0):
    """alpha = beta = 1, orthonormal keys: S k_i returns the last v written to k_i."""
    r = _rng(5)
    dk, dv, T = 4, 3, 10
    Q, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = Q.T  # rows orthonormal
    which = r.integers(0, dk, T)
    k = keys[which][:, None]
    v = r.standard_normal((T, 1, dv))
    qi = r.integers(0, dk, T)
    q = keys[qi][:, None]
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    o, st, _ = oracle.recurrent(q, k, v, g, beta, [0, T], C=4, mutant=mutant)
    worst = 0.0
    for t in range(T):
        last = [s for s in range(t + 1) if which[s] == qi[t]]
        want = v[last[-1], 0] if last else np.zeros(dv)
        ok, e = _close(o[t, 0], want, 1e-12)
        worst = max(worst, e)
        if not ok:
            return False, f"recall failed at t={t}: {e:.3e}"
    return True, f"recall: {worst:.3e}"


def pin_beta_one_unit_key(mutant=0):
    """beta = 1 with a unit key (any alpha, any history): S_t k_t = v_t."""
    q, k, v, g, beta, cu, s0 = random_problem(13, 12, 2, 5, 4)
    beta[:] = 1.0
    q = k.copy()  # read back along the key just written
    o, _, _ = oracle.recurrent(q, k, v, g, beta, cu, C=4, state_in=s0, mutant=mutant)
    ok, e = _close(o, v, 1e-12)
    return ok, f"write-then-read: {e:.3e}"


def pin_single_token(mutant=0):
    """From S_0 = 0, one token: S_1 = beta v k^T and o = beta v (k . q)."""
    q, k, v, g, beta, cu, _ = random_problem(17, 1, 3, 4, 5, state=False)
    o, st, _ = oracle.recurrent(q, k, v, g, beta, cu, C=4, mutant=mutant)
    want_o = beta[0][:, None] * v[0] * np.sum(k[0] * q[0], axis=-1)[:, None]
    want_s = beta[0][:, None, None] * np.einsum("hj,hi->hji", k[0], v[0])
    ok1, e1 = _close(o[0], want_o, 1e-14)
    ok2, e2 = _close(st[0], want_s, 1e-14)
    return ok1 and ok2, f"single token: {max(e1, e2):.3e}"


# --- the CPR schedule in fp64 agrees with the plain recurrence -------------------------

def pin_chunked_equals_recurrent(mutant=0):
    lens = [0, 1, 5, 16, 17, 40, 64, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, g, beta, cu, s0 = random_problem(19, T, 2, 8, 6, cu=cu)
    worst = 0.0
    for C in (1, 2, 3, 8, 16, 64):
        a = oracle.recurrent(q, k, v, g, beta, cu, C=C, state_in=s0, mutant=mutant)
        b = oracle.chunked(q, k, v, g, beta, cu, C=C, state_in=s0, mutant=mutant)
        for x, y, what in zip(a, b, ("o", "state_out", "boundary")):
            ok, e = _close(y, x, 1e-11)
            worst = max(worst, e)
            if not ok:
                return False, f"chunked vs recurrent {what} at C={C}: {e:.3e}"
    return True, f"chunked == recurrent to {worst:.3e}"


def pin_boundary_is_prefix_state(mutant=0):
    """boundary[chunk j of sequence n] equals the final state after the first j*C tokens."""
    lens = [23, 9]
    cu = np.array([0, 23, 32], dtype=np.int32)
    q, k, v, g, beta, cu, s0 = random_problem(23, 32, 1, 4, 4, cu=cu)
    C = 4
    _, _, bnd = oracle.recurrent(q, k, v, g, beta, cu, C=C, state_in=s0, mutant=mutant)
    c = 0
    for n, L in enumerate(lens):
        t0 = int(cu[n])
        for j in range(-(-L // C)):
            if j == 0:
                want = s0[n]
            else:
                sl = slice(t0, t0 + j * C)
                _, ob = oracle.bruteforce(q[sl, 0], k[sl, 0], v[sl, 0], g[sl, 0], beta[sl, 0], S0=s0[n, 0])
                want = ob[None]
            ok, e = _close(bnd[c], want, 1e-12)
            if not ok:
                return False, f"boundary {c} (seq {n}, chunk {j}): {e:.3e}"
            c += 1
    return True, "boundary states match prefix brute force"


def pin_continuation(mutant=0):
    """Running a prefix, then continuing from its final state, equals one run (decode form)."""
    q, k, v, g, beta, cu, s0 = random_problem(29, 20, 2, 4, 4)
    o, st, _ = oracle.recurrent(q, k, v, g, beta, cu, C=4, state_in=s0, mutant=mutant)
    split = 13
    o1, st1, _ = oracle.recurrent(q[:split], k[:split], v[:split], g[:split], beta[:split], [0, split],
                                  C=4, state_in=s0, mutant=mutant)
    o2, st2, _ = oracle.recurrent(q[split:], k[split:], v[split:], g[split:], beta[split:],
                                  [0, 20 - split], C=4, state_in=st1, mutant=mutant)
    ok1, e1 = _close(np.concatenate([o1, o2]), o, 0.0)
    ok2, e2 = _close(st2, st, 0.0)
    return ok1 and ok2, f"continuation: {max(e1, e2):.3e}"


ALL_PINS = [pin_bruteforce, pin_exact_rational, pin_golden, pin_beta_zero_decay,
            pin_orthonormal_recall, pin_beta_one_unit_key, pin_single_token,
            pin_chunked_equals_recurrent, pin_boundary_is_prefix_state, pin_continuation]
