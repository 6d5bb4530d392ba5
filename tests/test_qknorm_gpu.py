"""The in-kernel L2 normalisation of queries and keys (CPR_QK_L2NORM): with raw (not
normalised) queries and keys, prefill matches the fp64 oracle run on normalised inputs
(k / sqrt(sum k^2 + 1e-6), q / sqrt(sum q^2 + 1e-6) * dk^-1/2), and prefill, decode and the
continuation give the same bits as each other."""
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


def _raw_tokens(T, H, d, dtype, seed):
    """Tokens with unit-normal, unnormalised queries and keys (values, decays as usual)."""
    gen = torch.Generator().manual_seed(seed)
    _, _, v, g, beta = inputs.random_tokens(T, H, d, d, dtype=dtype, seed=seed)
    q = torch.randn(T, H, d, generator=gen).to(dtype)
    k = torch.randn(T, H, d, generator=gen).to(dtype)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def _normalised_f64(x, d):
    """The normalisation in fp64, for the oracle."""
    def l2(t):
        t = t.double()
        return t / torch.sqrt((t * t).sum(-1, keepdim=True) + 1e-6)
    return dict(x, q=l2(x["q"]) * d ** -0.5, k=l2(x["k"]))


@pytest.mark.parametrize("d,C,dtype", [(128, 64, torch.bfloat16), (32, 16, torch.float32)],
                         ids=["d128_C64_bf16", "d32_C16_f32"])
def test_qk_l2norm_matches_oracle_and_decode_bitwise(d, C, dtype):
    H = 2
    prefix = [0, C - 1, C + 3]
    M = C + 2
    full = [_raw_tokens(L + M, H, d, dtype, seed=40 + i) for i, L in enumerate(prefix)]
    xf = _gpu.to_dev(_gpu.pack(full))
    o_full, st_full, bnd_full, ws = cpr.cpr_gdn_prefill(xf["q"], xf["k"], xf["v"], xf["g"], xf["beta"],
                                                        xf["cu_seqlens"], C, qk_l2norm=True)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    # the oracle on inputs normalised in fp64
    xc = _gpu.pack(full)
    xn = _normalised_f64(xc, d)
    o_ref, st_ref, _ = oracle.recurrent(xn["q"], xn["k"], xn["v"], xn["g"], xn["beta"], xc["cu_seqlens"], C,
                                        boundaries=False)
    otol = _gpu.O_TOL_BF16 if dtype == torch.bfloat16 else _gpu.O_TOL_F32
    _gpu.assert_close_to_oracle(o_full, st_full, o_ref, st_ref, otol, what="qk l2norm prefill")
    # prefix prefill, ring, then decode steps: the same bits
    pre = _gpu.to_dev(_gpu.pack([_gpu.slice_tokens(f, 0, L) for f, L in zip(full, prefix)]))
    _, st, bnd, _ = cpr.cpr_gdn_prefill(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], pre["cu_seqlens"], C,
                                        qk_l2norm=True)
    ring = cpr.cpr_gdn_ring_from_prefill(pre["k"], pre["v"], pre["g"], pre["beta"], pre["cu_seqlens"], C, bnd, st)
    pos = torch.tensor(prefix, dtype=torch.int32, device=_gpu.dev())
    cu = xf["cu_seqlens"].cpu()
    for s in range(M):
        t = _gpu.to_dev({key: torch.stack([f[key][L + s] for f, L in zip(full, prefix)]) for key in full[0]})
        o, _ = cpr.cpr_gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], st, ring, pos, C, qk_l2norm=True)
        pos += 1
        for n, L in enumerate(prefix):
            assert _gpu.bits_equal(o[n], o_full[int(cu[n]) + L + s]), f"seq {n} step {s}"
    assert _gpu.bits_equal(st, st_full)


def test_qk_l2norm_continuation_bitwise():
    d, C, dtype, H = 128, 64, torch.bfloat16, 2
    lengths, splits = [3 * C + 9, 2 * C], [C + 20, 2 * C - 3]
    seqs = [_raw_tokens(L, H, d, dtype, seed=70 + i) for i, L in enumerate(lengths)]
    xf = _gpu.to_dev(_gpu.pack(seqs))
    o_full, st_full, _, _ = cpr.cpr_gdn_prefill(xf["q"], xf["k"], xf["v"], xf["g"], xf["beta"], xf["cu_seqlens"], C,
                                                qk_l2norm=True)
    first = _gpu.to_dev(_gpu.pack([_gpu.slice_tokens(s, 0, p) for s, p in zip(seqs, splits)]))
    second = _gpu.to_dev(_gpu.pack([_gpu.slice_tokens(s, p, L) for s, p, L in zip(seqs, splits, lengths)]))
    _, st, bnd, _ = cpr.cpr_gdn_prefill(first["q"], first["k"], first["v"], first["g"], first["beta"],
                                        first["cu_seqlens"], C, qk_l2norm=True)
    ring = cpr.cpr_gdn_ring_from_prefill(first["k"], first["v"], first["g"], first["beta"], first["cu_seqlens"], C,
                                         bnd, st)
    pos0 = torch.tensor(splits, dtype=torch.int32, device=_gpu.dev())
    o2, _, ws = cpr.cpr_gdn_prefill_continue(second["q"], second["k"], second["v"], second["g"], second["beta"],
                                             second["cu_seqlens"], pos0, C, st, ring, qk_l2norm=True)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    assert _gpu.bits_equal(st, st_full)
    c2, cf = second["cu_seqlens"].tolist(), xf["cu_seqlens"].tolist()
    for n, p in enumerate(splits):
        assert _gpu.bits_equal(o2[c2[n]:c2[n + 1]], o_full[cf[n] + p:cf[n + 1]]), f"seq {n}"
