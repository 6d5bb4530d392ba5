"""cpr_gdn_prefill_noalloc: prefill for callers that cannot allocate device memory.

Such callers (a runtime that owns all device memory through its own pool, a loop that
must not pay an allocation's device synchronisation) cannot hand cpr_gdn_prefill a
workspace; the no-alloc entry point uses the library's static scratch instead.  These
tests call it through the C ABI and compare it with cpr_gdn_prefill on the same inputs
bit for bit (both run the same kernels, so stale contents of the shared scratch must not
change a single bit), on two calls in a row with different shapes, and read the
no-alloc status word after each call.  This file sorts last so that a run stopping at
the first failure has run every other test first.
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
    assert cpr.cpr_gdn_prefill_noalloc_status() == 0
    assert _gpu.bits_equal(out, ref_o), "outputs differ from cpr_gdn_prefill"
    assert _gpu.bits_equal(st, ref_s), "final states differ from cpr_gdn_prefill"
    assert _gpu.bits_equal(bnd, ref_b), "boundary states differ from cpr_gdn_prefill"


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
