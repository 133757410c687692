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
