"""Grouped value heads (H value heads over Hk query/key heads, value head h reading
query/key head h / (H / Hk)): every path gives, bit for bit, what it gives with each
query/key head repeated for its value heads, and the fp64 oracle (on those repeated
inputs) within the usual tolerances."""
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


def _grouped_inputs(d, C, dtype, lengths, Hk, G, seed):
    H = Hk * G
    T = sum(lengths)
    dev = _gpu.dev()
    q, k, v, g, beta = inputs.random_tokens(T, H, d, d, dtype=dtype, seed=seed, device=dev)
    q, k = q[:, :Hk].contiguous(), k[:, :Hk].contiguous()  # Hk query/key heads
    x = dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=inputs.cu_seqlens_of(lengths).to(dev))
    xe = dict(x, q=q.repeat_interleave(G, dim=1).contiguous(), k=k.repeat_interleave(G, dim=1).contiguous())
    return x, xe


@pytest.mark.parametrize("d,C,dtype", [(128, 64, torch.bfloat16), (32, 16, torch.float32)],
                         ids=["d128_C64_bf16", "d32_C16_f32"])
def test_grouped_heads_equal_repeated_heads_bitwise(d, C, dtype):
    Hk, G = 2, 3
    lengths = [3 * C + 5, 2 * C, C - 1]
    x, xe = _grouped_inputs(d, C, dtype, lengths, Hk, G, seed=5)
    o, st, bnd = _gpu.prefill(x, C)
    oe, ste, bnde = _gpu.prefill(xe, C)
    assert _gpu.bits_equal(o, oe) and _gpu.bits_equal(st, ste) and _gpu.bits_equal(bnd, bnde)
    ring = cpr.cpr_gdn_ring_from_prefill(x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], C, bnd, st)
    ringe = cpr.cpr_gdn_ring_from_prefill(xe["k"], xe["v"], xe["g"], xe["beta"], xe["cu_seqlens"], C, bnde, ste)
    for a, b in zip((ring.S_b, ring.k, ring.v, ring.g, ring.beta), (ringe.S_b, ringe.k, ringe.v, ringe.g, ringe.beta)):
        assert _gpu.bits_equal(a, b)
    # decode across a resync
    pos = torch.tensor(lengths, dtype=torch.int32, device=_gpu.dev())
    for step in range(C + 2):
        q, k, v, g, beta = inputs.random_tokens(len(lengths), Hk * G, d, d, dtype=dtype, seed=500 + step,
                                                device=_gpu.dev())
        q, k = q[:, :Hk].contiguous(), k[:, :Hk].contiguous()
        oa, _ = cpr.cpr_gdn_decode(q, k, v, g, beta, st, ring, pos.clone(), C)
        ob, _ = cpr.cpr_gdn_decode(q.repeat_interleave(G, 1).contiguous(), k.repeat_interleave(G, 1).contiguous(),
                                   v, g, beta, ste, ringe, pos.clone(), C)
        pos += 1
        assert _gpu.bits_equal(oa, ob), f"decode step {step}"
    assert _gpu.bits_equal(st, ste)
    # a continuation of every sequence
    more, more_e = _grouped_inputs(d, C, dtype, [C + 3, 5, 2 * C], Hk, G, seed=9)
    o2, b2, ws = cpr.cpr_gdn_prefill_continue(more["q"], more["k"], more["v"], more["g"], more["beta"],
                                              more["cu_seqlens"], pos, C, st, ring)
    o2e, b2e, wse = cpr.cpr_gdn_prefill_continue(more_e["q"], more_e["k"], more_e["v"], more_e["g"], more_e["beta"],
                                                 more_e["cu_seqlens"], pos, C, ste, ringe)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0 and cpr.cpr_gdn_device_status(wse) == 0
    assert _gpu.bits_equal(o2, o2e) and _gpu.bits_equal(st, ste) and _gpu.bits_equal(b2, b2e)


def test_grouped_heads_match_oracle():
    d, C, dtype = 128, 64, torch.bfloat16
    x, xe = _grouped_inputs(d, C, dtype, [4 * C + 17, C + 1], Hk=4, G=2, seed=13)
    o, st, bnd = _gpu.prefill(x, C)
    xc = {k: v.cpu() for k, v in xe.items()}
    o_ref, st_ref, bnd_ref = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], C)
    _gpu.assert_close_to_oracle(o, st, o_ref, st_ref, _gpu.O_TOL_BF16, bnd, bnd_ref, what="grouped heads")


def test_grouped_heads_rejected_when_not_dividing():
    d, C = 32, 16
    x, _ = _grouped_inputs(d, C, torch.float32, [C], Hk=2, G=2, seed=1)
    v3 = torch.cat([x["v"], x["v"][:, :1]], 1).contiguous()  # 5 value heads over 2 query/key heads
    g3 = torch.cat([x["g"], x["g"][:, :1]], 1).contiguous()
    b3 = torch.cat([x["beta"], x["beta"][:, :1]], 1).contiguous()
    with pytest.raises(cpr.CprError):
        cpr.cpr_gdn_prefill(x["q"], x["k"], v3, g3, b3, x["cu_seqlens"], C)
