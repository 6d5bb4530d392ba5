"""The bench's algorithmic work counts (the numerators of every roofline figure), pinned to
counts worked by hand from the method's definition (CPU only)."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_prefill_counts_trainer_fwd():
    b = _bench()
    T, H, d, C = 10240, 16, 128, 64
    nbytes, flops = b.prefill_algorithmic(T, 1, H, d, d, T // C)
    # q, k, v in and o out (bf16): T H (3 d + d) 2 = 167,772,160
    # g, beta (fp32): 2 T H 4 = 1,310,720
    # 160 boundary states + 1 final state, fp32 d x d: 161 x 16 x 65,536 = 168,820,736
    assert nbytes == 167_772_160 + 1_310_720 + 168_820_736 == 337_903_616
    # S k (2), alpha S + u k^T (3), S q (2) flops per state element per token-head
    assert flops == 7 * d * d * T * H == 18_790_481_920


def test_decode_counts_rollout_decode():
    b = _bench()
    B, H, d, C = 256, 16, 128, 64
    # per (sequence, head): state read + written 2 x 65,536; q, k, v 3 x 256; g, beta 8;
    # o 256; the ring slot (k, v) 512 and its g, beta 8  ->  132,624 bytes
    assert b.decode_algorithmic(B, H, d, d, C, 0) == B * H * 132_624
    # one resync: the ring chunk (k, v, g, beta) 64 x 520, S_b read 65,536, S_b and the
    # state written 2 x 65,536 per head
    one = b.decode_algorithmic(B, H, d, d, C, 1) - b.decode_algorithmic(B, H, d, d, C, 0)
    assert one == H * (64 * 520 + 3 * 65_536)


def test_backward_counts_trainer_fwd():
    b = _bench()
    H, d, C, nc = 16, 128, 64, 160
    f = b.backward_algorithmic(nc, H, d, d, C)
    # chunk maps: 4 x (64 x 64 x 128) + 2 x (64 x 128 x 128) + 64^3 / 6 multiply-adds
    assert f["chunk_maps"] == 2 * (4 * 524_288 + 2 * 1_048_576 + 43_690) * nc * H
    # chain: one 128 x 128 by 128 x 128 product per chunk and head
    assert f["reverse_chain"] == 2 * 2_097_152 * nc * H
    # chunk gradients: 10 x 524,288 + 5 x 1,048,576 + 2 x 262,144 + 43,690
    assert f["chunk_grads"] == 2 * (5_242_880 + 5_242_880 + 524_288 + 43_690) * nc * H
