"""Parity of the CUDA path (through the C ABI) with the fp64 oracle and with itself.

Small cases spanning several chunks and a ragged tail, every built shape.  Bitwise
checks follow the CPR contract ("IsoExec: Eliminating Trainer-Inference Mismatch in
SkyRL", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": prefill, trainer
forward and decode are bitwise exact): prefill == decode, packed == alone, and results
independent of batch position.
"""
import numpy as np
import pytest
import torch

import _gpu
import linear_attention_cpr_gb300 as cpr
import oracle
from linear_attention_cpr_gb300 import build, inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    (32, 16, torch.float32),
    (32, 16, torch.bfloat16),
    (64, 32, torch.bfloat16),
    (128, 16, torch.bfloat16),
    (128, 32, torch.bfloat16),
    (128, 64, torch.bfloat16),
    (128, 64, torch.float32),
]
IDS = [f"d{d}-C{C}-{str(t).split('.')[-1]}" for d, C, t in SHAPES]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    cpr.load_library()
    oracle.build()


def _otol(dtype):
    return _gpu.O_TOL_F32 if dtype == torch.float32 else _gpu.O_TOL_BF16


def _lens(C):
    return [1, C - 1, C, C + 1, 2 * C, 3 * C + 5, 7]


@pytest.mark.parametrize("d,C,dtype", SHAPES, ids=IDS)
def test_prefill_matches_oracle(d, C, dtype):
    H = 3
    seqs = [_gpu.tokens(L, H, d, d, dtype, seed=10 + i) for i, L in enumerate(_lens(C))]
    x = _gpu.pack(seqs)
    N = len(seqs)
    gen = torch.Generator().manual_seed(5)
    s0 = 0.3 * torch.randn(N, H, d, d, generator=gen)
    out, st, bnd = _gpu.prefill(_gpu.to_dev(x), C, state_in=s0.cuda())
    o_ref, st_ref, bnd_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                              state_in=s0)
    assert bnd.shape[0] == bnd_ref.shape[0]
    _gpu.assert_close_to_oracle(out, st, o_ref, st_ref, _otol(dtype), bnd, bnd_ref, what=f"d{d} C{C}")


@pytest.mark.parametrize("d,C,dtype", SHAPES, ids=IDS)
def test_decode_equals_prefill_bitwise(d, C, dtype):
    """Prefill of L + M tokens == prefill of L tokens, ring, then M decode steps (bits)."""
    H = 2
    prefix = [0, 1, C - 1, C, C + 3, 2 * C]
    M = 2 * C + 3
    full = [_gpu.tokens(L + M, H, d, d, dtype, seed=100 + i) for i, L in enumerate(prefix)]
    pre = [_gpu.slice_tokens(f, 0, L) for f, L in zip(full, prefix)]
    steps = []
    for s in range(M):
        steps.append({key: torch.stack([f[key][L + s] for f, L in zip(full, prefix)]) for key in full[0]})
    outs, state, ring = _gpu.decode_run(pre, steps, C)
    xf = _gpu.to_dev(_gpu.pack(full))
    o_full, st_full, bnd_full = _gpu.prefill(xf, C)
    cu = xf["cu_seqlens"].cpu()
    for n, L in enumerate(prefix):
        for s in range(M):
            assert _gpu.bits_equal(outs[s][n], o_full[int(cu[n]) + L + s]), f"seq {n} step {s}"
        assert _gpu.bits_equal(state[n], st_full[n]), f"final state of seq {n}"
    # ...and both are within tolerance of the oracle
    xc = _gpu.pack(full)
    o_ref, st_ref, _ = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], C,
                                        boundaries=False)
    _gpu.assert_close_to_oracle(o_full, st_full, o_ref, st_ref, _otol(dtype), what="full prefill")


@pytest.mark.parametrize("d,C,dtype", [SHAPES[3], SHAPES[5]], ids=[IDS[3], IDS[5]])
def test_packing_and_position_invariance_bitwise(d, C, dtype):
    H = 4
    lens = [3 * C + 1, C, 5, 2 * C + 7, 1, C - 1]
    seqs = [_gpu.tokens(L, H, d, d, dtype, seed=200 + i) for i, L in enumerate(lens)]
    o_all, st_all, bnd_all = _gpu.prefill(_gpu.to_dev(_gpu.pack(seqs)), C)
    cu = inputs.cu_seqlens_of(lens)
    cch = np.concatenate([[0], np.cumsum([-(-L // C) for L in lens])])
    # one at a time
    for n, s in enumerate(seqs):
        o1, st1, b1 = _gpu.prefill(_gpu.to_dev(_gpu.pack([s])), C)
        assert _gpu.bits_equal(o1, o_all[int(cu[n]):int(cu[n + 1])])
        assert _gpu.bits_equal(st1[0], st_all[n])
        assert _gpu.bits_equal(b1, bnd_all[cch[n]:cch[n + 1]])
    # permuted order and a different grouping
    perm = [4, 1, 5, 0, 3, 2]
    o_p, st_p, _ = _gpu.prefill(_gpu.to_dev(_gpu.pack([seqs[i] for i in perm])), C)
    cu_p = inputs.cu_seqlens_of([lens[i] for i in perm])
    for j, n in enumerate(perm):
        assert _gpu.bits_equal(o_p[int(cu_p[j]):int(cu_p[j + 1])], o_all[int(cu[n]):int(cu[n + 1])])
        assert _gpu.bits_equal(st_p[j], st_all[n])


def test_tiny_workload_prefill_vs_256_decode_steps():
    """B=1, T=256, H=2, dk=dv=32, C=16, fp32, seed 0: prefill vs 256 decode steps."""
    w = inputs.workload("tiny")
    x = inputs.prefill_inputs(w)
    out, st, bnd = _gpu.prefill(_gpu.to_dev(x), w.C)
    o_ref, st_ref, bnd_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], w.C)
    _gpu.assert_close_to_oracle(out, st, o_ref, st_ref, _gpu.O_TOL_F32, bnd, bnd_ref, what="tiny")
    steps = [{k: x[k][t:t + 1] for k in ("q", "k", "v", "g", "beta")} for t in range(256)]
    empty = {k: x[k][:0] for k in ("q", "k", "v", "g", "beta")}
    outs, state, _ = _gpu.decode_run([empty], steps, w.C)
    for t in range(256):
        assert _gpu.bits_equal(outs[t][0], out[t]), f"token {t}"
    assert _gpu.bits_equal(state[0], st[0])


def test_state_in_none_is_zero_state():
    d, C = 128, 64
    x = _gpu.to_dev(_gpu.pack([_gpu.tokens(150, 2, d, d, torch.bfloat16, seed=7)]))
    a = _gpu.prefill(x, C)
    b = _gpu.prefill(x, C, state_in=torch.zeros(1, 2, d, d, device="cuda"))
    for u, v in zip(a, b):
        assert _gpu.bits_equal(u, v)


def test_empty_sequences_pass_state_through():
    d, C = 128, 64
    lens = [0, 70, 0]
    seqs = [_gpu.tokens(L, 2, d, d, torch.bfloat16, seed=30 + i) for i, L in enumerate(lens)]
    s0 = torch.randn(3, 2, d, d, device="cuda")
    out, st, bnd = _gpu.prefill(_gpu.to_dev(_gpu.pack(seqs)), C, state_in=s0)
    assert _gpu.bits_equal(st[0], s0[0]) and _gpu.bits_equal(st[2], s0[2])
    assert bnd.shape[0] == 2 and _gpu.bits_equal(bnd[0], s0[1])


def test_repeat_runs_identical():
    d, C = 128, 64
    x = _gpu.to_dev(_gpu.pack([_gpu.tokens(L, 4, d, d, torch.bfloat16, seed=40 + L) for L in (300, 64, 129)]))
    a = _gpu.prefill(x, C)
    b = _gpu.prefill(x, C)
    for u, v in zip(a, b):
        assert _gpu.bits_equal(u, v)


def test_device_checks_record_status():
    d, C, H = 128, 64, 2
    x = _gpu.to_dev(_gpu.pack([_gpu.tokens(L, H, d, d, torch.bfloat16, seed=50) for L in (10, 10, 10)]))
    # decreasing cu_seqlens: no chunk is processed, status bit 1
    bad = torch.tensor([0, 20, 10, 30], dtype=torch.int32, device="cuda")
    out, st, bnd, ws = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], bad, C, n_chunks=3)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) & 1
    # too few boundary rows: status bit 2
    small = torch.empty(2, H, d, d, device="cuda")
    out, st, bnd, ws = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                           boundary_states=small)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) & 2
    # negative decode position: status bit 4, sequence skipped
    ring = cpr.Ring.empty(3, H, d, d, C, device="cuda")
    state = torch.zeros(3, H, d, d, device="cuda")
    t = _gpu.to_dev(_gpu.tokens(3, H, d, d, torch.bfloat16, seed=51))
    pos = torch.tensor([0, -1, 5], dtype=torch.int32, device="cuda")
    o, ws = cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) & 4
    assert torch.count_nonzero(state[1]) == 0
    # a clean call clears it
    pos = torch.tensor([0, 1, 5], dtype=torch.int32, device="cuda")
    o, ws = cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], state, ring, pos, C, workspace=ws)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0


def test_decay_exp_error_bound():
    """The decay exponential e^x = 2^(x log2 e) (ex2.approx) against fp64 exp on x <= 0.
    Rounding x log2 e to fp32 moves the exponent by up to |x log2 e| 2^-24, a relative
    error of about |x| 2^-24 in e^x; ex2.approx adds at most 2^-22.  So the bound is
    2^-21 + |x| 2^-23 (twice the sum) wherever e^x is a normal float, and 1 exactly at 0."""
    import ctypes

    probe = ctypes.CDLL(build.PROBE_LIB)
    probe.cpr_probe_decay_exp.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    x = torch.cat([torch.zeros(1), -torch.logspace(-8, 1.9, 200000, dtype=torch.float64).float()]).cuda()
    y = torch.empty_like(x)
    assert probe.cpr_probe_decay_exp(x.data_ptr(), y.data_ptr(), x.numel(), None) == 0
    torch.cuda.synchronize()
    ref = torch.exp(x.double())
    rel = ((y.double() - ref).abs() / ref).cpu()
    normal = (ref > 1.2e-38).cpu()
    bound = 2.0 ** -21 + x.abs().double().cpu() * 2.0 ** -23
    excess = (rel - bound)[normal]
    assert float(excess.max()) <= 0.0, float((rel / bound)[normal].max())
    assert float(y[0]) == 1.0


@pytest.mark.parametrize("case", ["beta_zero", "alpha_one", "whole_chunks"])
def test_degenerate_inputs_match_oracle(case):
    """Degenerate cases of the recurrence, on the main shape (d128, C64, bf16):
    beta = 0 leaves only the decay, S_t = (prod alpha) S_0 (checked in closed form too);
    alpha = 1 (g = 0) is the ungated delta rule; lengths that are multiples of C end on a
    chunk update (state_out is U's result, not a stepped state)."""
    d, C, H = 128, 64, 2
    lens = [2 * C, C, 3 * C] if case == "whole_chunks" else [C + 7, 2 * C + 1]
    seqs = [_gpu.tokens(L, H, d, d, torch.bfloat16, seed=60 + i) for i, L in enumerate(lens)]
    for s in seqs:
        if case == "beta_zero":
            s["beta"] = torch.zeros_like(s["beta"])
        if case == "alpha_one":
            s["g"] = torch.zeros_like(s["g"])
    x = _gpu.pack(seqs)
    gen = torch.Generator().manual_seed(61)
    s0 = 0.3 * torch.randn(len(lens), H, d, d, generator=gen)
    out, st, bnd = _gpu.prefill(_gpu.to_dev(x), C, state_in=s0.cuda())
    o_ref, st_ref, bnd_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                              state_in=s0)
    _gpu.assert_close_to_oracle(out, st, o_ref, st_ref, _gpu.O_TOL_BF16, bnd, bnd_ref, what=case)
    if case == "beta_zero":
        cu = x["cu_seqlens"]
        for n in range(len(lens)):
            decay = torch.exp(x["g"][int(cu[n]):int(cu[n + 1])].double().sum(0))  # [H]
            want = decay[:, None, None] * s0[n].double()
            got = st[n].cpu().double()
            rel = ((got - want).norm() / want.norm()).item()
            assert rel <= _gpu.STATE_RTOL, rel
