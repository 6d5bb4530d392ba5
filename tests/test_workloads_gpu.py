"""The five benchmark workloads at full size, in the launch configuration bench.py times.

Each is checked against the fp64 oracle (whole, or on sampled sequences where the oracle
would take minutes) and against itself bit for bit (prefill == decode, packed == alone,
permuted and regrouped batches).
"""
import numpy as np
import pytest
import torch

import _gpu
import linear_attention_cpr_gb300 as cpr
import oracle
from linear_attention_cpr_gb300 import build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    cpr.load_library()
    oracle.build()


def _cpu(x):
    return {k: v.cpu() for k, v in x.items()}


def _seq(x, cu, n):
    a, b = int(cu[n]), int(cu[n + 1])
    return {k: x[k][a:b].contiguous() for k in ("q", "k", "v", "g", "beta")}


def test_trainer_fwd_full_vs_oracle_and_repeatable():
    w = inputs.workload("trainer_fwd")
    x = inputs.prefill_inputs(w, device="cuda")
    a = _gpu.prefill(x, w.C)
    xc = _cpu(x)
    o_ref, st_ref, bnd_ref = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], w.C)
    err = _gpu.assert_close_to_oracle(a[0], a[1], o_ref, st_ref, _gpu.O_TOL_BF16, a[2], bnd_ref, what="trainer_fwd")
    print(f"trainer_fwd max|do| = {err:.3e}")
    b = _gpu.prefill(x, w.C)
    for u, v in zip(a, b):
        assert _gpu.bits_equal(u, v)


def test_rollout_prefill_packed_equals_alone_and_oracle():
    w = inputs.workload("rollout_prefill")
    x = inputs.prefill_inputs(w, device="cuda")
    o, st, bnd = _gpu.prefill(x, w.C)
    cu = x["cu_seqlens"].cpu()
    for n in range(len(w.seqlens)):
        s = _seq(x, cu, n)
        s["cu_seqlens"] = inputs.cu_seqlens_of([w.seqlens[n]]).cuda()
        o1, st1, b1 = _gpu.prefill(s, w.C)
        assert _gpu.bits_equal(o1, o[int(cu[n]):int(cu[n + 1])])
        assert _gpu.bits_equal(st1[0], st[n])
        assert _gpu.bits_equal(b1, bnd[32 * n:32 * (n + 1)])
    xc = _cpu(x)
    o_ref, st_ref, bnd_ref = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], w.C)
    _gpu.assert_close_to_oracle(o, st, o_ref, st_ref, _gpu.O_TOL_BF16, bnd, bnd_ref, what="rollout_prefill")


def test_rollout_decode_resync_bitwise_and_oracle():
    """256 sequences, prior lengths U[1,4096]; 64 decode steps (every sequence crosses a
    chunk boundary); sampled sequences re-run as one prefill of prior + new tokens."""
    w = inputs.workload("rollout_decode")
    C, H, d = w.C, w.H, w.dk
    x = inputs.prefill_inputs(w, device="cuda")
    n_chunks = cpr.cpr_gdn_num_chunks(inputs.cu_seqlens_of(w.seqlens), C)
    _, st, bnd, ws = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                         n_chunks=n_chunks)
    ring = cpr.cpr_gdn_ring_from_prefill(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd, st)
    state = st.clone()
    pos = torch.tensor(w.seqlens, dtype=torch.int32, device="cuda")
    M = 64
    toks = [inputs.decode_inputs(w, s, device="cuda") for s in range(M)]
    outs = []
    dws = None
    for s in range(M):
        t = toks[s]
        o, dws = cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C, workspace=dws)
        outs.append(o.clone())
        pos += 1
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(dws) == 0
    cu = x["cu_seqlens"].cpu()
    lens = np.array(w.seqlens)
    # sequences whose prior length leaves the boundary at several different step offsets
    picks = sorted({int(np.argmin(lens)), int(np.argmax(lens))} |
                   {int(i) for i in np.where(lens % C == 0)[0][:1]} |
                   {int(i) for i in np.where(lens % C == C - 1)[0][:1]} | {3, 77, 200})
    for n in picks:
        s = _seq(x, cu, n)
        full = {k: torch.cat([s[k], torch.stack([toks[j][k][n] for j in range(M)])]).contiguous() for k in s}
        full["cu_seqlens"] = inputs.cu_seqlens_of([w.seqlens[n] + M]).cuda()
        of, stf, _ = _gpu.prefill(full, C)
        L = w.seqlens[n]
        for j in range(M):
            assert _gpu.bits_equal(outs[j][n], of[L + j]), f"seq {n} (L={L}) step {j}"
        assert _gpu.bits_equal(state[n], stf[0]), f"seq {n} final state"
        if n in picks[:3]:
            fc = _cpu(full)
            o_ref, st_ref, _ = oracle.recurrent(fc["q"], fc["k"], fc["v"], fc["g"], fc["beta"], fc["cu_seqlens"], C,
                                                boundaries=False)
            _gpu.assert_close_to_oracle(of, stf, o_ref, st_ref, _gpu.O_TOL_BF16, what=f"decode seq {n}")


def test_varlen_stress_permutations_and_regrouping():
    w = inputs.workload("varlen_stress")
    C = w.C
    x = inputs.prefill_inputs(w, device="cuda")
    cu = x["cu_seqlens"].cpu()
    N = len(w.seqlens)
    o, st, bnd = _gpu.prefill(x, C)
    seqs = [_seq(x, cu, n) for n in range(N)]
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(N, generator=g).tolist()
    xp = _gpu.pack([seqs[i] for i in perm])
    xp = {k: v.cuda() for k, v in xp.items()}
    op, stp, _ = _gpu.prefill(xp, C)
    cup = xp["cu_seqlens"].cpu()
    for j, n in enumerate(perm):
        assert _gpu.bits_equal(op[int(cup[j]):int(cup[j + 1])], o[int(cu[n]):int(cu[n + 1])])
        assert _gpu.bits_equal(stp[j], st[n])
    # decode 128 steps: whole batch vs permuted batch vs two regrouped halves
    M = 128
    toks = [inputs.decode_inputs(w, s, device="cuda") for s in range(M)]

    def run_decode(order):
        sub = [seqs[i] for i in order]
        pre = {k: v.cuda() for k, v in _gpu.pack(sub).items()}
        _, s0, b0 = _gpu.prefill(pre, C)
        ring = cpr.cpr_gdn_ring_from_prefill(pre["k"], pre["v"], pre["g"], pre["beta"], pre["cu_seqlens"], C, b0, s0)
        state = s0.clone()
        pos = torch.tensor([w.seqlens[i] for i in order], dtype=torch.int32, device="cuda")
        idx = torch.tensor(order, device="cuda")
        res = []
        for s in range(M):
            t = {k: v.index_select(0, idx).contiguous() for k, v in toks[s].items()}
            out, _ = cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C)
            res.append(out.clone())
            pos += 1
        torch.cuda.synchronize()
        return torch.stack(res, 1), state  # [B, M, H, dv]

    base_o, base_s = run_decode(list(range(N)))
    po, ps = run_decode(perm)
    for j, n in enumerate(perm):
        assert _gpu.bits_equal(po[j], base_o[n]) and _gpu.bits_equal(ps[j], base_s[n])
    half = perm[: N // 2], perm[N // 2:]
    for grp in half:
        go, gs = run_decode(list(grp))
        for j, n in enumerate(grp):
            assert _gpu.bits_equal(go[j], base_o[n]) and _gpu.bits_equal(gs[j], base_s[n])
    # oracle on three sampled sequences (prefill + decode tokens)
    lens = np.array(w.seqlens)
    for n in (int(np.argmin(lens)), int(np.argsort(lens)[N // 2]), 5):
        s = _cpu(seqs[n])
        full = {k: torch.cat([s[k], torch.stack([toks[j][k][n].cpu() for j in range(M)])]) for k in s}
        o_ref, st_ref, _ = oracle.recurrent(full["q"], full["k"], full["v"], full["g"], full["beta"],
                                            [0, w.seqlens[n] + M], C, boundaries=False)
        L = w.seqlens[n]
        got = torch.cat([o[int(cu[n]):int(cu[n + 1])], base_o[n]])
        _gpu.assert_close_to_oracle(got, base_s[n:n + 1], o_ref, st_ref, _gpu.O_TOL_BF16, what=f"varlen seq {n}")
        assert got.shape[0] == L + M


def test_long_single_sequence():
    """One 65,536-token sequence (1,024 chained chunk updates), two heads."""
    d, C, H, T = 128, 64, 2, 65536
    q, k, v, g, beta = inputs.random_tokens(T, H, d, d, dtype=torch.bfloat16, seed=3, device="cuda")
    x = dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=inputs.cu_seqlens_of([T]).cuda())
    o, st, bnd = _gpu.prefill(x, C)
    xc = _cpu(x)
    o_ref, st_ref, bnd_ref = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], C)
    _gpu.assert_close_to_oracle(o, st, o_ref, st_ref, _gpu.O_TOL_BF16, bnd, bnd_ref, what="long sequence")
