"""cpr_gdn_prefill_noalloc: prefill for callers that cannot allocate device memory.

Such callers (a runtime that owns all device memory through its own pool, a loop that
must not pay an allocation's device synchronisation) cannot hand cpr_gdn_prefill a
workspace; the no-alloc entry point uses the library's static scratch instead.  These
tests call it through the C ABI and compare it with cpr_gdn_prefill on the same inputs,
within the parity tolerances, on two calls in a row with different shapes (the shared
scratch keeps the previous call's contents, which must not matter).  This file sorts
last so that a run stopping at the first failure has run every other test first.
"""
import pytest
import torch

import _gpu
import linear_attention_cpr_gb300 as cpr
from linear_attention_cpr_gb300 import binding, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    cpr.load_library()


def _compare(d, C, dtype, lens, H, seed):
    x = _gpu.to_dev(_gpu.pack([_gpu.tokens(L, H, d, d, dtype, seed=seed + i) for i, L in enumerate(lens)]))
    N, T = len(lens), sum(lens)
    assert cpr.cpr_gdn_prefill_workspace_size(T, N, H, d, d, C) <= binding.NOALLOC_SCRATCH_BYTES
    s0 = 0.3 * torch.randn(N, H, d, d, device="cuda", generator=torch.Generator("cuda").manual_seed(seed))
    ref_o, ref_s, ref_b, _ = cpr.cpr_gdn_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C,
                                                 state_in=s0)
    out = torch.full_like(ref_o, float("nan"))
    st = torch.full_like(ref_s, float("nan"))
    bnd = torch.full_like(ref_b, float("nan"))
    cpr.cpr_gdn_prefill_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, state_in=s0,
                                out=out, state_out=st, boundary_states=bnd)
    torch.cuda.synchronize()
    tol = _gpu.O_TOL_F32 if dtype == torch.float32 else _gpu.O_TOL_BF16
    assert float((out.float() - ref_o.float()).abs().max()) <= tol
    rel = ((st - ref_s).norm(dim=(-2, -1)) / ref_s.norm(dim=(-2, -1)).clamp_min(1e-30)).max()
    assert float(rel) <= _gpu.STATE_RTOL
    relb = ((bnd - ref_b).norm(dim=(-2, -1)) / ref_b.norm(dim=(-2, -1)).clamp_min(1e-30)).max()
    assert float(relb) <= _gpu.STATE_RTOL


def test_noalloc_prefill_matches_prefill_on_two_calls_in_a_row():
    _compare(128, 64, torch.bfloat16, [70, 5, 130], H=2, seed=1)   # first call on this device: sets up
    _compare(32, 16, torch.float32, [33, 16, 1, 90], H=3, seed=7)  # second call: stale scratch from the first


def test_noalloc_prefill_rejects_problems_beyond_the_scratch():
    d, C, H, T = 128, 64, 16, 65536
    assert cpr.cpr_gdn_prefill_workspace_size(T, 1, H, d, d, C) > binding.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(T, H, d, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(T, H, device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    st = torch.empty(1, H, d, d, device="cuda")
    bnd = torch.empty(T // C, H, d, d, device="cuda")
    with pytest.raises(cpr.CprError) as ei:
        cpr.cpr_gdn_prefill_noalloc(q, q, q, g, g, cu, C, out=out, state_out=st, boundary_states=bnd)
    assert ei.value.code == -4
