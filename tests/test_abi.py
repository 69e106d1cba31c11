"""Host-side checks of the C ABI: the library builds, loads and exports every
entry point the header declares; sizing calls work without a GPU."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(collider_[a-z_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from sparse_backward_gemm_gb300 import build
    build.build()
    import sparse_backward_gemm_gb300 as cl
    return cl


def test_every_declared_symbol_is_exported(lib):
    L = lib.lib()
    declared = _declared()
    assert len(declared) >= 18
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(lib.EXPORTED)


def test_sizing_calls(lib):
    assert lib.collider_compact_workspace_size(4, 2048) == 0
    assert lib.collider_compact_workspace_size(1, 5_000_000) > 0
    assert lib.collider_linear_workspace_size(lib.BF16, 8192, 2048, 5632) > 0
    assert lib.collider_attn_workspace_size(4, 2048, 32, 4, 64) > 0
    import workloads
    s = workloads.WORKLOADS["tinyllama_layer"]
    d = lib.LayerDesc(arch=lib.ARCH_LLAMA, B=s.B, T=s.T, D=s.D, H=s.H, Hkv=s.Hkv, dh=s.dh, F=s.F,
                      rotary_dim=s.rotary_dim, rope_base=s.rope_base, norm=lib.NORM_RMS, eps=s.eps,
                      act=lib.ACT_SWIGLU)
    n = lib.collider_layer_workspace_size(d)
    assert 100 << 20 < n < 4 << 30
    d.dh = 96            # unsupported head dim -> 0
    assert lib.collider_layer_workspace_size(d) == 0


def test_binding_has_no_fallback(lib):
    src = open(os.path.join(ROOT, "sparse_backward_gemm_gb300", "collider.py")).read()
    assert "oracle" not in src and "numpy" not in src
