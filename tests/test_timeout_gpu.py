"""The failure path of the waits on other CTAs (the prefill's, and the backward's fused
launch's), on the GPU, without a fault.

An intra-chunk item waits (bounded) until the chain CTAs publish its chunk's boundary
state.  The library's test hook makes every item wait for one publication more than the
chain ever makes, with a 2 ms limit: each wait runs out, the items are skipped, the call
records CPR_DEV_TIMEOUT in its status word and returns, and the context stays usable (a
normal call right after gives the oracle's result).  Nothing is in flight when an item
gives up: its chunk's staging copies have been waited for before the wait begins."""
import numpy as np
import pytest
import torch

import _gpu
import linear_attention_cpr_gb300 as cpr
import oracle
from linear_attention_cpr_gb300 import build

pytestmark = pytest.mark.gpu

CPR_DEV_TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    cpr.load_library()


def test_item_wait_runs_out_and_reports_timeout():
    C, H, d = 64, 2, 128
    lens = [150, 64, 37]
    xc = _gpu.pack([_gpu.tokens(L, H, d, d, torch.bfloat16, seed=40 + i) for i, L in enumerate(lens)])
    x = _gpu.to_dev(xc)
    T, N = sum(lens), len(lens)
    n_chunks = cpr.cpr_gdn_num_chunks(xc["cu_seqlens"], C)
    sentinel = 7.0
    out = torch.full((T, H, d), sentinel, dtype=torch.bfloat16, device="cuda")
    st = torch.full((N, H, d, d), sentinel, device="cuda")
    bnd = torch.empty(n_chunks, H, d, d, device="cuda")
    ws = torch.empty(cpr.cpr_gdn_prefill_workspace_size(T, N, H, d, d, C), dtype=torch.uint8, device="cuda")
    cpr.cpr_gdn_set_wait_test(1, 2_000_000)
    try:
        cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, out=out, state_out=st,
                            boundary_states=bnd, workspace=ws)
        torch.cuda.synchronize()
    finally:
        cpr.cpr_gdn_set_wait_test(0, 0)
    status = cpr.cpr_gdn_device_status(ws)
    assert status & CPR_DEV_TIMEOUT, f"status {status}: the timeout was not reported"
    # every item gave up: no output was written, nor the final state of a sequence whose
    # last chunk is partial (an item writes it); the chain's own results are unaffected
    assert bool((out.float() == sentinel).all()), "an item wrote outputs after its wait ran out"
    for n, L in enumerate(lens):
        if L % C:
            assert bool((st[n] == sentinel).all())
    o_ref, st_ref, b_ref = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], C)
    b = bnd.cpu().double().numpy()
    rel = np.linalg.norm(b - b_ref, axis=(-2, -1)) / np.maximum(np.linalg.norm(b_ref, axis=(-2, -1)), 1e-300)
    assert float(rel.max()) <= _gpu.STATE_RTOL

    # the context is still usable, and the hook is off again: a normal call is correct
    out2, st2, bnd2 = _gpu.prefill(x, C)
    _gpu.assert_close_to_oracle(out2, st2, o_ref, st_ref, _gpu.O_TOL_BF16, bnd2, b_ref, what="after timeout")


def test_backward_gradient_wait_runs_out_and_reports_timeout():
    # the backward's fused launch (d = 128, C = 64, bf16): each chunk's gradients wait for
    # the reverse chain to publish its state adjoint; with the hook every wait runs out, no
    # gradient of a token is written, the chain's own result (d_state_in) is unaffected
    from oracle import backward
    C, H, d = 64, 2, 128
    lens = [150, 64, 37]
    xc = _gpu.pack([_gpu.tokens(L, H, d, d, torch.bfloat16, seed=50 + i) for i, L in enumerate(lens)])
    x = _gpu.to_dev(xc)
    T, N = sum(lens), len(lens)
    gen = torch.Generator().manual_seed(6)
    d_out = torch.randn(T, H, d, generator=gen).to(torch.bfloat16)
    d_state = 0.5 * torch.randn(N, H, d, d, generator=gen)
    _, _, bnd = _gpu.prefill(x, C)
    sentinel = 7.0
    grads = {"dq": torch.full((T, H, d), sentinel, device="cuda"), "dk": torch.full((T, H, d), sentinel, device="cuda"),
             "dv": torch.full((T, H, d), sentinel, device="cuda"), "dg": torch.full((T, H), sentinel, device="cuda"),
             "dbeta": torch.full((T, H), sentinel, device="cuda"),
             "d_state_in": torch.full((N, H, d, d), sentinel, device="cuda")}
    cpr.cpr_gdn_set_wait_test(1, 2_000_000)
    try:
        _, ws = cpr.cpr_gdn_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd,
                                     d_out.cuda(), d_state.cuda(), grads=grads)
        torch.cuda.synchronize()
    finally:
        cpr.cpr_gdn_set_wait_test(0, 0)
    status = cpr.cpr_gdn_device_status(ws)
    assert status & CPR_DEV_TIMEOUT, f"status {status}: the timeout was not reported"
    for name in ("dq", "dk", "dv", "dg", "dbeta"):
        assert bool((grads[name] == sentinel).all()), f"{name} written after its wait ran out"
    ref = backward.recurrent_backward(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"],
                                      d_out.float(), d_state_out=d_state)
    g = grads["d_state_in"].double().cpu().numpy()
    r = ref["d_state_in"]
    assert float(np.linalg.norm(g - r) / np.linalg.norm(r)) <= 1e-4

    # the context is still usable, and the hook is off again
    gr, ws2 = cpr.cpr_gdn_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd,
                                   d_out.cuda(), d_state.cuda())
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws2) == 0
    for name in ("dq", "dk", "dv", "dg", "dbeta", "d_state_in"):
        gg = gr[name].double().cpu().numpy()
        rr = ref[name]
        assert float(np.linalg.norm(gg - rr) / np.linalg.norm(rr)) <= 1e-4, name
