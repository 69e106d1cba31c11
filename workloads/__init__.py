"""Seeded synthetic workloads for the filtered transformer backward.

This module is shared by both sides of every parity check (the fp64 CPU
oracle and the CUDA library), so it holds NO arithmetic of the method
itself: it only draws random numbers, rounds them to their storage type,
and builds the per-token keep-masks.  Everything the backward computes lives
elsewhere.

Shapes follow the decoder models named in "Enhancing Token Filtering
Efficiency in Large Language Model Training with Collider" (abstract:
TinyLlama-1.1B, Qwen2.5-1.5B, Phi1.5-1.4B); the token filter itself (Fig. 2b,
backward filtering of the loss) is stood in for by seeded random scores.

Seeds: tensor ``k`` of workload ``c`` is drawn from PCG64(1000*c + k), with
the ordinals listed in :func:`layer_weights`, :func:`layer_inputs` and
:func:`stack_tensors`.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "LayerShape", "LinearShape", "StackShape", "WORKLOADS", "bf16_representable",
    "gumbel_keep_mask", "span_keep_mask", "keep_mask", "normal", "linear_inputs",
    "layer_weights", "layer_inputs", "stack_tensors", "n_filtered",
]


# --------------------------------------------------------------------------
# workload shapes
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class LinearShape:
    """One linear layer Y = X.W, W stored [in, out] row-major."""
    seed_base: int
    B: int
    T: int
    K: int          # in features
    N: int          # out features
    f: float        # filtered fraction per sequence
    mask: str = "gumbel"
    dtype: str = "f32"

    @property
    def M(self) -> int:
        return self.B * self.T


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One pre-norm decoder block.

    arch "llama": x -> RMSNorm -> QKV -> RoPE -> causal GQA -> O-proj -> +x
                   -> RMSNorm -> [gate|up] -> SwiGLU -> down -> +h
    arch "phi":   x -> LayerNorm = a; out = x + Attn(a) + MLP(a)  (parallel
                   block, GELU-tanh MLP, partial RoPE, biases everywhere)
    """
    seed_base: int
    arch: str
    B: int
    T: int
    D: int
    H: int
    Hkv: int
    dh: int
    F: int
    rotary_dim: int
    rope_base: float
    norm: str        # "rms" | "ln"
    eps: float
    act: str         # "swiglu" | "gelu"
    qkv_bias: bool
    out_bias: bool
    mlp_bias: bool
    f: float
    mask: str = "gumbel"

    @property
    def M(self) -> int:
        return self.B * self.T

    @property
    def Nqkv(self) -> int:
        return (self.H + 2 * self.Hkv) * self.dh

    @property
    def Nup(self) -> int:
        """Width of the first MLP projection ([gate|up] for SwiGLU)."""
        return 2 * self.F if self.act == "swiglu" else self.F

    def with_(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class StackShape:
    """L decoder blocks + final norm + untied LM head + token embedding."""
    seed_base: int
    layer: LayerShape
    L: int
    V: int

    def with_(self, **kw) -> "StackShape":
        return dataclasses.replace(self, **kw)


_TINYLLAMA = LayerShape(seed_base=2000, arch="llama", B=4, T=2048, D=2048, H=32, Hkv=4,
                        dh=64, F=5632, rotary_dim=64, rope_base=10000.0, norm="rms",
                        eps=1e-5, act="swiglu", qkv_bias=False, out_bias=False,
                        mlp_bias=False, f=0.4, mask="gumbel")

WORKLOADS = {
    # 1: single linear layer, fp32 end to end
    "linear_fp32": LinearShape(seed_base=1000, B=1, T=128, K=256, N=256, f=0.4),
    # 2: TinyLlama-1.1B-shaped block, batch 4 x 2048
    "tinyllama_layer": _TINYLLAMA,
    # 3: Qwen2.5-1.5B-shaped block (QKV bias, head_dim 128), batch 2 x 4096
    "qwen25_layer": LayerShape(seed_base=3000, arch="llama", B=2, T=4096, D=1536, H=12,
                               Hkv=2, dh=128, F=8960, rotary_dim=128, rope_base=1e6,
                               norm="rms", eps=1e-6, act="swiglu", qkv_bias=True,
                               out_bias=False, mlp_bias=False, f=0.4, mask="gumbel"),
    # 4: Phi-1.5-shaped parallel block, span masks, ratio sweep 0/.2/.4/.6
    "phi15_layer": LayerShape(seed_base=4000, arch="phi", B=4, T=2048, D=2048, H=32,
                              Hkv=32, dh=64, F=8192, rotary_dim=32, rope_base=10000.0,
                              norm="ln", eps=1e-5, act="gelu", qkv_bias=True,
                              out_bias=True, mlp_bias=True, f=0.4, mask="span"),
    # 5: 22-layer TinyLlama-shaped stack, 1 x 8192, vocab 32000
    "tinyllama_stack": StackShape(seed_base=5000, layer=_TINYLLAMA.with_(B=1, T=8192, seed_base=5000),
                                  L=22, V=32000),
}


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------
def bf16_representable(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (ties to even); returned as float32.

    Only used to make generated inputs exactly representable in bf16, so both
    sides of a comparison start from identical values.
    """
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    # NaN stays NaN (not produced by the generators, kept for safety)
    return np.where(np.isnan(a), a, out).reshape(np.shape(x))


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal(shape, std: float, seed: int, bf16: bool = True, mean: float = 0.0) -> np.ndarray:
    """N(mean, std^2) samples as float32 (bf16-representable when ``bf16``)."""
    a = _rng(seed).standard_normal(size=shape, dtype=np.float64) * std + mean
    a = a.astype(np.float32)
    return bf16_representable(a) if bf16 else a


# --------------------------------------------------------------------------
# keep-masks (stand-in for the token filter's decision)
# --------------------------------------------------------------------------
def n_filtered(T: int, f: float) -> int:
    """Filtered tokens per sequence: floor(f*T) (exact 40% of 128 is not an integer)."""
    return int(math.floor(f * T + 1e-9))


def gumbel_keep_mask(B: int, T: int, f: float, seed: int) -> np.ndarray:
    """Per-token Gumbel(0,1) scores; the lowest floor(f*T) of each sequence are
    filtered (ties: lower position first).  Returns uint8 [B, T], 1 = kept."""
    g = _rng(seed).gumbel(size=(B, T))
    nf = n_filtered(T, f)
    keep = np.ones((B, T), dtype=np.uint8)
    pos = np.arange(T)
    for b in range(B):
        order = np.lexsort((pos, g[b]))      # primary: score, secondary: position
        keep[b, order[:nf]] = 0
    return keep


def span_keep_mask(B: int, T: int, f: float, seed: int, mean_len: float = 16.0) -> np.ndarray:
    """Filtered tokens come in contiguous spans: repeatedly draw a start
    ~ U[0,T) and a length ~ Geometric(p=1/mean_len) (support >= 1) and filter
    [s, s+len) clipped to the sequence, truncating the last span so that
    exactly floor(f*T) tokens per sequence are filtered.  uint8 [B, T]."""
    rng = _rng(seed)
    nf = n_filtered(T, f)
    keep = np.ones((B, T), dtype=np.uint8)
    for b in range(B):
        left = nf
        while left > 0:
            s = int(rng.integers(0, T))
            ln = int(rng.geometric(1.0 / mean_len))
            for t in range(s, min(T, s + ln)):
                if left == 0:
                    break
                if keep[b, t]:
                    keep[b, t] = 0
                    left -= 1
    return keep


def keep_mask(B: int, T: int, f: float, kind: str, seed: int) -> np.ndarray:
    if kind == "gumbel":
        return gumbel_keep_mask(B, T, f, seed)
    if kind == "span":
        return span_keep_mask(B, T, f, seed)
    raise ValueError(kind)


# --------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------
def linear_inputs(s: LinearShape):
    """Single-linear workload: X, W ~ N(0, 1/256) (variance), dY ~ N(0,1), fp32.

    Ordinals: 0 mask, 1 X, 2 W, 3 dY."""
    sb = s.seed_base
    keep = keep_mask(s.B, s.T, s.f, s.mask, sb + 0)
    std = math.sqrt(1.0 / 256.0)
    X = normal((s.M, s.K), std, sb + 1, bf16=False)
    W = normal((s.K, s.N), std, sb + 2, bf16=False)
    dY = normal((s.M, s.N), 1.0, sb + 3, bf16=False)
    return dict(keep=keep, X=X, W=W, dY=dY)


def layer_weights(s: LayerShape, seed_base: int | None = None) -> dict:
    """Random-init block weights, all bf16-representable float32, layout [in, out].

    Ordinals (added to the seed base): 10 norm1 gamma, 11 norm1 beta, 12 W_qkv,
    13 b_qkv, 14 W_o, 15 b_o, 16 norm2 gamma, 17 W_up ([gate|up] or fc1),
    18 b_up, 19 W_down (fc2), 20 b_down.  Std 0.02; gamma = 1 + N(0, 0.02).
    """
    sb = s.seed_base if seed_base is None else seed_base
    std = 0.02
    w = dict(
        norm1_w=normal((s.D,), std, sb + 10, mean=1.0),
        w_qkv=normal((s.D, s.Nqkv), std, sb + 12),
        w_o=normal((s.H * s.dh, s.D), std, sb + 14),
        w_up=normal((s.D, s.Nup), std, sb + 17),
        w_down=normal((s.F, s.D), std, sb + 19),
    )
    if s.norm == "ln":
        w["norm1_b"] = normal((s.D,), std, sb + 11)
    if s.arch == "llama":
        w["norm2_w"] = normal((s.D,), std, sb + 16, mean=1.0)
    if s.qkv_bias:
        w["b_qkv"] = normal((s.Nqkv,), std, sb + 13)
    if s.out_bias:
        w["b_o"] = normal((s.D,), std, sb + 15)
    if s.mlp_bias:
        w["b_up"] = normal((s.Nup,), std, sb + 18)
        w["b_down"] = normal((s.D,), std, sb + 20)
    return w


def layer_inputs(s: LayerShape) -> dict:
    """Block input x ~ N(0,1), upstream gradient dOut ~ N(0,1) (bf16), keep-mask.

    Ordinals: 0 mask, 1 x, 2 dOut."""
    sb = s.seed_base
    keep = keep_mask(s.B, s.T, s.f, s.mask, sb + 0)
    x = normal((s.M, s.D), 1.0, sb + 1)
    dout = normal((s.M, s.D), 1.0, sb + 2)
    return dict(keep=keep, x=x, dout=dout)


def stack_tensors(s: StackShape) -> dict:
    """Stack workload: token ids (T+1, uniform over the vocabulary: inputs are
    ids[:T], targets ids[1:]), embedding E [V, D], per-layer weights, final
    norm gamma, LM head W_lm [D, V] (untied), keep-mask.

    Ordinals: 0 mask, 1 ids, 2 E, 3 final gamma, 4 W_lm; layer l uses seed base
    seed_base + 100*(l+1) with the ordinals of :func:`layer_weights`."""
    ls = s.layer
    sb = s.seed_base
    keep = keep_mask(ls.B, ls.T, ls.f, ls.mask, sb + 0)
    ids = _rng(sb + 1).integers(0, s.V, size=(ls.B, ls.T + 1), dtype=np.int64)
    E = normal((s.V, ls.D), 0.02, sb + 2)
    normf_w = normal((ls.D,), 0.02, sb + 3, mean=1.0)
    w_lm = normal((ls.D, s.V), 0.02, sb + 4)
    layers = [layer_weights(ls, seed_base=sb + 100 * (l + 1)) for l in range(s.L)]
    return dict(keep=keep, ids=ids[:, :ls.T].astype(np.int32).reshape(-1),
                targets=ids[:, 1:].astype(np.int32).reshape(-1), E=E,
                normf_w=normf_w, w_lm=w_lm, layers=layers)
