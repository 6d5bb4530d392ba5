"""The CPR backward on the GPU, through the C ABI, against the fp64 oracle of the exact
adjoint (oracle/backward.py, pinned by finite differences of the forward oracle), and
against itself.

The pages time a trainer backward ("IsoExec: Eliminating Trainer-Inference Mismatch in
SkyRL", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet", per-layer table, row
"Trainer Fwd+Bwd") without describing it; the gradients are those of the recurrence, so
the oracle is its exact adjoint.  The kernels take the forward's boundary states (from
cpr_gdn_prefill) as the saved states, as a trainer does.

Tolerance (fp32 arithmetic against fp64, derived in the design notes): for every
gradient tensor, relative Frobenius error <= 1e-4 and every element within 1e-3 of the
tensor's largest magnitude.  Bitwise: the same gradients from run to run and for a
sequence alone or packed with others in any order."""
import numpy as np
import pytest
import torch

import _gpu
import linear_attention_cpr_gb300 as cpr
import oracle
from linear_attention_cpr_gb300 import build, inputs
from oracle import backward

pytestmark = pytest.mark.gpu

GRAD_RTOL = 1e-4
GRAD_MAXTOL = 1e-3
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_state_in")

SHAPES = [
    (32, 16, torch.float32),
    (32, 16, torch.bfloat16),
    (64, 32, torch.bfloat16),
    (128, 16, torch.bfloat16),
    (128, 32, torch.float32),
    (128, 64, torch.bfloat16),
]
IDS = [f"d{d}-C{C}-{str(t).split('.')[-1]}" for d, C, t in SHAPES]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    cpr.load_library()
    oracle.build()


def _upstream(T, N, H, d, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    d_out = torch.randn(T, H, d, generator=gen).to(dtype)
    d_state = 0.5 * torch.randn(N, H, d, d, generator=gen)
    return d_out, d_state


def _check(gr, ref, what, names=NAMES):
    for name in names:
        g = gr[name].double().cpu().numpy()
        r = ref[name]
        scale = float(np.abs(r).max())
        if scale == 0.0:
            assert float(np.abs(g).max()) == 0.0, f"{what} {name}: nonzero where the oracle is zero"
            continue
        rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
        mx = float(np.abs(g - r).max()) / scale
        print(f"backward {what} {name}: rel Frobenius {rel:.2e}, max/scale {mx:.2e}")
        assert rel <= GRAD_RTOL, f"{what} {name}: relative Frobenius error {rel:.3e}"
        assert mx <= GRAD_MAXTOL, f"{what} {name}: max error {mx:.3e} of the largest magnitude"


def _run(x, C, s0, d_out, d_state, dev):
    xd = _gpu.to_dev(x)
    _, _, bnd = _gpu.prefill(xd, C, state_in=None if s0 is None else s0.to(dev))
    gr, ws = cpr.cpr_gdn_backward(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], xd["cu_seqlens"], C, bnd,
                                  d_out.to(dev), None if d_state is None else d_state.to(dev))
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    return gr


@pytest.mark.parametrize("d,C,dtype", SHAPES, ids=IDS)
def test_backward_matches_oracle(d, C, dtype):
    H = 2
    lens = [1, C - 1, C, C + 1, 2 * C, 3 * C + 5, 0, 7]
    seqs = [_gpu.tokens(L, H, d, d, dtype, seed=60 + i) for i, L in enumerate(lens)]
    x = _gpu.pack(seqs)
    N, T = len(lens), sum(lens)
    s0 = 0.3 * torch.randn(N, H, d, d, generator=torch.Generator().manual_seed(3))
    d_out, d_state = _upstream(T, N, H, d, dtype, seed=4)
    gr = _run(x, C, s0, d_out, d_state, _gpu.dev())
    ref = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], d_out.float(),
                                      d_state_out=d_state, state_in=s0)
    _check(gr, ref, f"d{d} C{C}")


def test_backward_without_state_gradients():
    # no upstream state gradient and no initial state: the chain starts from zero
    d, C, H, dtype = 128, 64, 2, torch.bfloat16
    lens = [200, 64]
    x = _gpu.pack([_gpu.tokens(L, H, d, d, dtype, seed=80 + i) for i, L in enumerate(lens)])
    d_out, _ = _upstream(sum(lens), len(lens), H, d, dtype, seed=5)
    gr = _run(x, C, None, d_out, None, _gpu.dev())
    ref = backward.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], d_out.float())
    _check(gr, ref, "no state grads")


def test_backward_is_deterministic_and_packing_invariant():
    d, C, H, dtype = 128, 64, 2, torch.bfloat16
    lens = [130, 64, 1, 77]
    seqs = [_gpu.tokens(L, H, d, d, dtype, seed=90 + i) for i, L in enumerate(lens)]
    ups = [_upstream(L, 1, H, d, dtype, seed=100 + i) for i, L in enumerate(lens)]
    dev = _gpu.dev()

    def batch(order):
        x = _gpu.pack([seqs[i] for i in order])
        d_out = torch.cat([ups[i][0] for i in order])
        d_state = torch.cat([ups[i][1] for i in order])
        return _run(x, C, None, d_out, d_state, dev)

    a = batch([0, 1, 2, 3])
    b = batch([0, 1, 2, 3])
    for name in NAMES:
        assert _gpu.bits_equal(a[name], b[name]), f"{name} differs from run to run"
    perm = [2, 0, 3, 1]
    p = batch(perm)
    starts = np.concatenate([[0], np.cumsum(lens)])
    pstarts = np.concatenate([[0], np.cumsum([lens[i] for i in perm])])
    for pos, i in enumerate(perm):
        alone = batch([i])
        sl, psl = slice(starts[i], starts[i + 1]), slice(pstarts[pos], pstarts[pos + 1])
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            assert _gpu.bits_equal(alone[name], a[name][sl]), f"{name}: sequence {i} alone != packed"
            assert _gpu.bits_equal(alone[name], p[name][psl]), f"{name}: sequence {i} permuted != alone"
        assert _gpu.bits_equal(alone["d_state_in"][0], p["d_state_in"][pos])


def test_backward_trainer_size_sampled_heads():
    # the trainer workload (1 x 10,240 tokens, H=16, d=128, C=64): every head on the GPU,
    # two heads against the oracle's WY-chunked adjoint (fp64; pinned against the
    # token-level adjoint)
    w = inputs.workload("trainer_fwd")
    x = inputs.prefill_inputs(w)
    T, H, d, C = w.total_tokens, w.H, w.dk, w.C
    d_out, _ = _upstream(T, 1, H, d, w.dtype, seed=7)
    gr = _run(x, C, None, d_out, None, _gpu.dev())
    for h in (0, 11):
        sub = {k: x[k][:, h:h + 1].contiguous() for k in ("q", "k", "v", "g", "beta")}
        ref = backward.wy_chunked_backward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], x["cu_seqlens"],
                                           d_out[:, h:h + 1].float(), C)
        got = {n: gr[n][:, h:h + 1] for n in ("dq", "dk", "dv", "dg", "dbeta")}
        got["d_state_in"] = gr["d_state_in"][:, h:h + 1]
        _check(got, ref, f"trainer_fwd head {h}")
