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
    # the dense forward's scratch: f32 outputs of the QKV, output and down
    # projections (the up projection writes the saved bf16 [g | u] itself), lse,
    # RoPE table
    nf = lib.collider_layer_fwd_workspace_size(d)
    M = s.B * s.T
    f32_acc = 4 * M * (s.Nqkv + 2 * s.D)
    assert f32_acc <= nf < f32_acc + (16 << 20)
    d.dh = 96            # unsupported head dim -> 0
    assert lib.collider_layer_workspace_size(d) == 0
    assert lib.collider_layer_fwd_workspace_size(d) == 0


def test_forward_argument_errors_need_no_gpu(lib):
    """Argument errors come back synchronously, before any CUDA call."""
    import workloads
    s = workloads.WORKLOADS["phi15_layer"]
    d = lib.LayerDesc(arch=lib.ARCH_PHI, B=s.B, T=s.T, D=s.D, H=s.H, Hkv=s.Hkv, dh=s.dh, F=s.F,
                      rotary_dim=s.rotary_dim, rope_base=s.rope_base, norm=lib.NORM_LAYER, eps=s.eps,
                      act=lib.ACT_GELU_TANH, qkv_bias=1, out_bias=1, mlp_bias=1)
    fake = 1 << 20   # never dereferenced: validation fails first
    params = lib.LayerParams(norm1_w=fake, norm1_b=fake, w_qkv=fake, b_qkv=fake, w_o=fake, b_o=None,
                             w_up=fake, b_up=fake, w_down=fake, b_down=fake)
    acts = lib.LayerActs(a=fake, mean1=fake, rstd1=fake, qkv=fake, o=fake, lse=fake, up=fake)
    with pytest.raises(lib.ColliderError) as e:      # b_o missing although out_bias is set
        lib.collider_layer_fwd(d, params, fake, fake + 4096, acts, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "bias" in str(e.value)
    params.b_o = fake + 8                           # misaligned
    with pytest.raises(lib.ColliderError) as e:
        lib.collider_layer_fwd(d, params, fake, fake + 4096, acts, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "aligned" in str(e.value)
    params.b_o = fake
    with pytest.raises(lib.ColliderError) as e:      # no workspace
        lib.collider_layer_fwd(d, params, fake, fake + 4096, acts, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "workspace" in str(e.value)
    with pytest.raises(lib.ColliderError) as e:      # y aliasing x
        lib.collider_layer_fwd(d, params, fake, fake, acts, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "alias" in str(e.value)
    d.act = lib.ACT_SWIGLU                          # phi blocks use GELU
    with pytest.raises(lib.ColliderError) as e:
        lib.collider_layer_fwd(d, params, fake, fake + 4096, acts, None, stream=0)
    assert e.value.status == lib.ERR_UNSUPPORTED


def test_layer_backward_saved_set_errors_need_no_gpu(lib):
    """A Llama block's saved set may leave out a, b and s (recomputed), but not
    h or rstd2, and not a, b or s in a dense call (which reads them in place);
    a Phi block needs a.  All refused before any CUDA call."""
    import workloads
    s = workloads.WORKLOADS["tinyllama_layer"]
    d = lib.LayerDesc(arch=lib.ARCH_LLAMA, B=s.B, T=s.T, D=s.D, H=s.H, Hkv=s.Hkv, dh=s.dh, F=s.F,
                      rotary_dim=s.rotary_dim, rope_base=s.rope_base, norm=lib.NORM_RMS, eps=s.eps,
                      act=lib.ACT_SWIGLU)
    fake = 1 << 20   # never dereferenced: validation fails first
    w = lib.LayerWeights(**{f: fake for f, _ in lib.LayerWeights._fields_})
    g = lib.LayerGrads(**{f: fake for f, _ in lib.LayerGrads._fields_})
    sv = lib.LayerSaved(**{f: fake for f, _ in lib.LayerSaved._fields_})
    sv.mean1 = None
    sv.a = sv.b = sv.s = None
    with pytest.raises(lib.ColliderError) as e:      # dense call without a, b, s
        lib.collider_layer_bwd(d, w, sv, fake, lib.ROWS_FULL, None, None, None, g, lib.ROWS_FULL, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "dense" in str(e.value)
    with pytest.raises(lib.ColliderError) as e:      # filtered: a, b, s may be absent; the workspace is next
        lib.collider_layer_bwd(d, w, sv, fake, lib.ROWS_FULL, fake, fake, fake, g, lib.ROWS_FULL, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "workspace" in str(e.value)
    sv.h = None
    with pytest.raises(lib.ColliderError) as e:      # h is needed
        lib.collider_layer_bwd(d, w, sv, fake, lib.ROWS_FULL, fake, fake, fake, g, lib.ROWS_FULL, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "h" in str(e.value)
    p = workloads.WORKLOADS["phi15_layer"]
    dp = lib.LayerDesc(arch=lib.ARCH_PHI, B=p.B, T=p.T, D=p.D, H=p.H, Hkv=p.Hkv, dh=p.dh, F=p.F,
                       rotary_dim=p.rotary_dim, rope_base=p.rope_base, norm=lib.NORM_LAYER, eps=p.eps,
                       act=lib.ACT_GELU_TANH)
    svp = lib.LayerSaved(**{f: fake for f, _ in lib.LayerSaved._fields_})
    svp.a = None
    with pytest.raises(lib.ColliderError) as e:      # a Phi block needs a
        lib.collider_layer_bwd(dp, w, svp, fake, lib.ROWS_FULL, fake, fake, fake, g, lib.ROWS_FULL, None, stream=0)
    assert e.value.status == lib.ERR_INVALID_ARG and "phi" in str(e.value)


def test_binding_has_no_fallback(lib):
    src = open(os.path.join(ROOT, "sparse_backward_gemm_gb300", "collider.py")).read()
    assert "oracle" not in src and "numpy" not in src
