"""The C-ABI library loads and exports every entry point that include/cpr_gdn.h declares,
and its host-side logic answers without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest
import torch

import linear_attention_cpr_gb300 as cpr
from linear_attention_cpr_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def _declared():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(cpr_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return cpr.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"{name} missing from {binding.library_path()}"
    assert set(names) == set(binding.EXPORTED)


def test_version_and_strerror(lib):
    assert cpr.cpr_gdn_version() >= 1
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(cpr.cpr_gdn_strerror(code), str)


def test_supported_shapes(lib):
    assert cpr.cpr_gdn_supported(128, 128, 64)
    assert cpr.cpr_gdn_supported(32, 32, 16, torch.float32)
    assert not cpr.cpr_gdn_supported(96, 96, 64)
    assert not cpr.cpr_gdn_supported(128, 128, 48)


def test_num_chunks_host(lib):
    assert cpr.cpr_gdn_num_chunks([0, 0, 1, 64, 129], 64) == 0 + 1 + 1 + 2
    assert cpr.cpr_gdn_num_chunks([0, 10240], 64) == 160
    with pytest.raises(cpr.CprError):
        cpr.cpr_gdn_num_chunks([0, 5, 3], 4)


def test_workspace_size_monotone(lib):
    a = cpr.cpr_gdn_prefill_workspace_size(10240, 1, 16, 128, 128, 64)
    b = cpr.cpr_gdn_prefill_workspace_size(20480, 1, 16, 128, 128, 64)
    assert 0 < a < b
    assert a % 256 == 0
    assert cpr.cpr_gdn_prefill_workspace_size(-1, 1, 16, 128, 128, 64) == 0
    assert cpr.cpr_gdn_decode_workspace_size(256, 16, 128, 128, 64) >= 4


def _raw_prefill(lib, **kw):
    args = dict(q=16, k=16, v=16, g=16, beta=16, cu=16, N=1, T=64, H=2, dk=128, dv=128, C=64, dtype=0,
                state_in=None, out=16, state_out=16, bnd=16, cap=1, ws=16, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    return lib.cpr_gdn_prefill(*args.values())


def test_prefill_rejects_on_host(lib):
    # every call below is refused by host-side checks before anything is enqueued
    assert _raw_prefill(lib, dk=96, dv=96) == -2
    assert _raw_prefill(lib, C=48) == -2
    assert _raw_prefill(lib, dtype=7) == -1
    assert _raw_prefill(lib, H=0) == -1
    assert _raw_prefill(lib, q=None) == -1
    assert _raw_prefill(lib, ws_bytes=16) == -4
    assert _raw_prefill(lib, q=18) == -3
    assert _raw_prefill(lib, g=18) == -3
    assert _raw_prefill(lib, N=0) == 0  # empty batch: nothing to do


def test_decode_rejects_on_host(lib):
    ring = binding._Ring(16, 16, 16, 16, 16)
    ws = lib.cpr_gdn_decode_workspace_size(4, 2, 128, 128, 64)
    base = [16, 16, 16, 16, 16, 16, ctypes.byref(ring), 16, 4, 2, 128, 128, 64, 0, 16, 16, ws, None]
    # `base` itself is never passed: its pointers are placeholders, only rejected variants run
    bad = list(base)
    bad[10], bad[11] = 96, 96
    assert lib.cpr_gdn_decode(*bad) == -2
    bad = list(base)
    bad[16] = 0
    assert lib.cpr_gdn_decode(*bad) == -4
    bad = list(base)
    bad[0] = 20
    assert lib.cpr_gdn_decode(*bad) == -3
    bad = list(base)
    bad[8] = 0
    assert lib.cpr_gdn_decode(*bad) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.load_library()
