"""Continuation prefill (a rollout's chunked prefill): splitting each sequence at any
position into a prefill and a continuation gives the one-shot prefill's outputs, final
state, boundary states and ring bit for bit, and decode then carries on identically.
The one-shot path itself is pinned to the fp64 oracle by the other GPU tests; one case
here is also checked against the oracle directly."""
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


def _pack(parts):
    """Concatenate per-sequence token dicts into packed inputs with cu_seqlens."""
    keys = ("q", "k", "v", "g", "beta")
    lens = [p["q"].shape[0] for p in parts]
    x = {k: torch.cat([p[k] for p in parts], 0).contiguous() for k in keys}
    x["cu_seqlens"] = inputs.cu_seqlens_of(lens).to(x["q"].device)
    return x


def _split_case(d, C, dtype, lengths, splits, seed):
    H = 2
    dev = _gpu.dev()
    T = sum(lengths)
    q, k, v, g, beta = inputs.random_tokens(T, H, d, d, dtype=dtype, seed=seed, device=dev)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    full = dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=inputs.cu_seqlens_of(lengths).to(dev))
    seqs = [{n: t[cu[i]:cu[i + 1]] for n, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta))}
            for i in range(len(lengths))]
    first = _pack([{n: t[:s] for n, t in sq.items()} for sq, s in zip(seqs, splits)])
    second = _pack([{n: t[s:] for n, t in sq.items()} for sq, s in zip(seqs, splits)])
    return full, first, second, cu


@pytest.mark.parametrize("d,C,dtype", [(128, 64, torch.bfloat16), (64, 32, torch.float32), (32, 16, torch.float32)],
                         ids=["d128_C64_bf16", "d64_C32_f32", "d32_C16_f32"])
def test_continuation_equals_one_shot_bitwise(d, C, dtype):
    # splits: at 0, inside the first chunk, at a boundary, inside a later chunk, at the
    # end; remainders that stay inside the chunk, complete it exactly, or run past it
    lengths = [5 * C + 7, 3 * C, 2 * C + 1, C - 3, 4 * C, 3 * C + C // 2, 2 * C]
    splits = [C + 3, 0, C, C - 5, 4 * C, 2 * C + C // 2 + 2, C // 2]
    full, first, second, cu = _split_case(d, C, dtype, lengths, splits, seed=7)
    H = full["q"].shape[1]
    o_full, st_full, bnd_full = _gpu.prefill(full, C)
    ring_full = cpr.cpr_gdn_ring_from_prefill(full["k"], full["v"], full["g"], full["beta"], full["cu_seqlens"], C,
                                              bnd_full, st_full)
    o1, st1, bnd1 = _gpu.prefill(first, C)
    ring = cpr.cpr_gdn_ring_from_prefill(first["k"], first["v"], first["g"], first["beta"], first["cu_seqlens"], C,
                                         bnd1, st1)
    pos0 = torch.tensor(splits, dtype=torch.int32, device=_gpu.dev())
    state = st1.clone()
    o2, bnd2, ws = cpr.cpr_gdn_prefill_continue(second["q"], second["k"], second["v"], second["g"], second["beta"],
                                                second["cu_seqlens"], pos0, C, state, ring)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    # outputs: the first and second parts of each sequence, against the one-shot run
    c1 = first["cu_seqlens"].tolist()
    c2 = second["cu_seqlens"].tolist()
    for n, s in enumerate(splits):
        a = cu[n]
        assert _gpu.bits_equal(o1[c1[n]:c1[n + 1]], o_full[a:a + s]), f"seq {n}: first part"
        assert _gpu.bits_equal(o2[c2[n]:c2[n + 1]], o_full[a + s:cu[n + 1]]), f"seq {n}: continuation"
    assert _gpu.bits_equal(state, st_full), "final states"
    # boundary states of the chunks that start inside the continuation
    cf = [0]
    for L in [cu[i + 1] - cu[i] for i in range(len(splits))]:
        cf.append(cf[-1] + -(-L // C))
    j2 = 0
    for n, s in enumerate(splits):
        L = cu[n + 1] - cu[n]
        first_full_chunk = -(-s // C)  # chunks of the whole sequence that start at or after s
        n_rest = -(-L // C) - first_full_chunk
        for j in range(n_rest):
            assert _gpu.bits_equal(bnd2[j2 + j], bnd_full[cf[n] + first_full_chunk + j]), f"seq {n} boundary {j}"
        j2 += n_rest
    # the ring: S_b and the slots of each sequence's final partial chunk
    assert _gpu.bits_equal(ring.S_b, ring_full.S_b), "ring S_b"
    for n in range(len(splits)):
        rem = (cu[n + 1] - cu[n]) % C
        for name in ("k", "v", "g", "beta"):
            a, b = getattr(ring, name)[n][:, :rem], getattr(ring_full, name)[n][:, :rem]
            assert _gpu.bits_equal(a.contiguous(), b.contiguous()), f"ring {name} seq {n}"
    # decode carries on identically after both
    st_a, st_b = state.clone(), st_full.clone()
    ring_a, ring_b = ring.clone(), ring_full.clone()
    pos = torch.tensor([cu[n + 1] - cu[n] for n in range(len(splits))], dtype=torch.int32, device=_gpu.dev())
    for step in range(C + 2):
        t = inputs.random_tokens(len(splits), H, d, d, dtype=dtype, seed=1000 + step, device=_gpu.dev())
        oa, _ = cpr.cpr_gdn_decode(*t, st_a, ring_a, pos.clone(), C)
        ob, _ = cpr.cpr_gdn_decode(*t, st_b, ring_b, pos.clone(), C)
        pos += 1
        assert _gpu.bits_equal(oa, ob), f"decode step {step}"
    assert _gpu.bits_equal(st_a, st_b)


def test_continuation_matches_oracle():
    d, C, dtype = 128, 64, torch.bfloat16
    lengths = [3 * C + 5, 2 * C + 9]
    splits = [C + 40, 2 * C + 1]
    full, first, second, cu = _split_case(d, C, dtype, lengths, splits, seed=11)
    o1, st1, bnd1 = _gpu.prefill(first, C)
    ring = cpr.cpr_gdn_ring_from_prefill(first["k"], first["v"], first["g"], first["beta"], first["cu_seqlens"], C,
                                         bnd1, st1)
    pos0 = torch.tensor(splits, dtype=torch.int32, device=_gpu.dev())
    state = st1.clone()
    o2, _, ws = cpr.cpr_gdn_prefill_continue(second["q"], second["k"], second["v"], second["g"], second["beta"],
                                             second["cu_seqlens"], pos0, C, state, ring)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) == 0
    xc = {k: v.cpu() for k, v in full.items()}
    o_ref, st_ref, _ = oracle.recurrent(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], xc["cu_seqlens"], C)
    c2 = second["cu_seqlens"].tolist()
    o_cont = torch.cat([o2[c2[n]:c2[n + 1]] for n in range(len(splits))], 0)
    ref_cont = np.concatenate([o_ref[cu[n] + splits[n]:cu[n + 1]] for n in range(len(splits))], 0)
    _gpu.assert_close_to_oracle(o_cont, state, ref_cont, st_ref, _gpu.O_TOL_BF16, what="continuation")


def test_continuation_bad_position_records_status_and_writes_nothing():
    d, C, dtype = 32, 16, torch.float32
    lengths, splits = [2 * C + 3, C], [5, 0]
    full, first, second, cu = _split_case(d, C, dtype, lengths, splits, seed=3)
    o1, st1, bnd1 = _gpu.prefill(first, C)
    ring = cpr.cpr_gdn_ring_from_prefill(first["k"], first["v"], first["g"], first["beta"], first["cu_seqlens"], C,
                                         bnd1, st1)
    state = st1.clone()
    ring0 = ring.clone()
    pos0 = torch.tensor([5, -1], dtype=torch.int32, device=_gpu.dev())
    out = torch.full((second["q"].shape[0], 2, d), 7.0, dtype=dtype, device=_gpu.dev())
    _, _, ws = cpr.cpr_gdn_prefill_continue(second["q"], second["k"], second["v"], second["g"], second["beta"],
                                            second["cu_seqlens"], pos0, C, state, ring, out=out)
    torch.cuda.synchronize()
    assert cpr.cpr_gdn_device_status(ws) & cpr.binding.DEV_BAD_POS
    assert _gpu.bits_equal(state, st1) and _gpu.bits_equal(ring.S_b, ring0.S_b) and _gpu.bits_equal(ring.k, ring0.k)
    assert bool((out == 7.0).all())
