"""The C-ABI library builds, loads and exports every entry point that
include/moe.h declares (CPU only; no compute calls)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from moe_expert_layer_histogram_gb300 import _build
    _build.build()
    import moe_expert_layer_histogram_gb300 as m
    return m.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("moe_create", "moe_prepare_weights", "moe_forward", "moe_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_uses_the_same_names():
    import moe_expert_layer_histogram_gb300 as m
    for n in _declared():
        assert hasattr(m, n), n


def test_status_strings(lib):
    import moe_expert_layer_histogram_gb300 as m
    for code in range(8):
        assert m.moe_status_string(code)
    assert m.moe_status_string(0) == "ok"


def test_no_cpu_fallback_without_library(tmp_path, monkeypatch):
    import moe_expert_layer_histogram_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        m.lib()


def test_static_routing_refuses_misaligned_pointers_on_the_host(lib):
    # argument errors are found on the host before any CUDA call, so this
    # runs without a GPU: every pointer must be 4-byte aligned
    import moe_expert_layer_histogram_gb300 as m
    good = 1 << 20
    for bad in range(5):
        ptrs = [good] * 5
        ptrs[bad] = good + 2
        code = lib.moe_route_permute_static(ptrs[0], 8, 16, 2, ptrs[1], ptrs[2], ptrs[3],
                                            ptrs[4], None)
        assert code == 1, (bad, code)
    assert lib.moe_route_permute_static(good, 4097, 16, 2, good, good, good, good, None) == 2
    assert lib.moe_route_permute_static(good, 0, 16, 2, good, good, good, good, None) == 0
    assert m.moe_status_string(1) == "invalid argument"


def test_config_rejects_negative_test_fields(lib):
    import ctypes
    import moe_expert_layer_histogram_gb300 as m
    for field in ("max_ctas", "test_fail_alloc_at", "test_stall_gemm"):
        cfg = m.MoEConfig(16, 256, 128, 8, 2, 0, 0.0, 0, 0, 0, 0, 0)
        setattr(cfg, field, -1)
        h = ctypes.c_void_p()
        assert lib.moe_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
        assert not h.value
