"""Thin ctypes binding of libcollider (``include/collider.h``).

Argument marshalling only: every step of the filtered backward runs in the
library's CUDA kernels.  Each function takes the same arguments as the C entry
point of the same name; buffers may be torch tensors (their ``data_ptr()`` is
passed), plain integers (device addresses) or None (NULL).  ``stream``
defaults to torch's current CUDA stream.  A non-OK status raises
:class:`ColliderError` carrying the library's message.  There is no fallback:
if ``libcollider.so`` is missing, importing the binding's entry points fails.
"""
from __future__ import annotations

import ctypes as C
import os

__all__ = [
    "ColliderError", "lib", "LIB_PATH", "ROWS_FULL", "ROWS_COMPACT", "F32", "BF16",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_TIMEOUT",
    "ARCH_LLAMA", "ARCH_PHI", "NORM_RMS", "NORM_LAYER", "ACT_SWIGLU", "ACT_GELU_TANH",
    "LayerDesc", "LayerWeights", "LayerSaved", "LayerGrads", "LayerParams", "LayerActs", "EXPORTED",
    "collider_last_error", "collider_check", "collider_selftest_wait_timeout", "collider_launch_count",
    "collider_profile_enable", "collider_profile_count", "collider_profile_get", "collider_profile_get_span",
    "collider_select_keep", "collider_compact_workspace_size", "collider_compact", "collider_compact_noalloc",
    "collider_gather_rows",
    "collider_scatter_rows", "collider_linear_workspace_size", "collider_linear_bwd",
    "collider_attn_workspace_size", "collider_attn_bwd", "collider_layer_workspace_size",
    "collider_layer_bwd", "collider_layer_fwd_workspace_size", "collider_layer_fwd",
    "collider_stack_workspace_size", "collider_stack_bwd",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcollider.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(5)
_STATUS = {1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT"}
F32, BF16 = 0, 1
ROWS_FULL, ROWS_COMPACT = 0, 1
ARCH_LLAMA, ARCH_PHI = 0, 1
NORM_RMS, NORM_LAYER = 0, 1
ACT_SWIGLU, ACT_GELU_TANH = 0, 1


class ColliderError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"COLLIDER_ERR_{_STATUS.get(status, status)}: {msg}")
        self.status = status


class LayerDesc(C.Structure):
    _fields_ = [("arch", C.c_int), ("B", C.c_int), ("T", C.c_int), ("D", C.c_int), ("H", C.c_int),
                ("Hkv", C.c_int), ("dh", C.c_int), ("F", C.c_int), ("rotary_dim", C.c_int),
                ("rope_base", C.c_float), ("norm", C.c_int), ("eps", C.c_float), ("act", C.c_int),
                ("qkv_bias", C.c_int), ("out_bias", C.c_int), ("mlp_bias", C.c_int)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("norm1_w", "w_qkv", "w_o", "norm2_w", "w_up", "w_down")]


class LayerSaved(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("x", "a", "mean1", "rstd1", "qkv", "o", "lse", "h", "b",
                                          "rstd2", "up", "s")]


class LayerGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("dx", "dnorm1_w", "dnorm1_b", "dw_qkv", "db_qkv", "dw_o",
                                          "db_o", "dnorm2_w", "dw_up", "db_up", "dw_down", "db_down")]


class LayerParams(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("norm1_w", "norm1_b", "w_qkv", "b_qkv", "w_o", "b_o", "norm2_w",
                                          "w_up", "b_up", "w_down", "b_down")]


class LayerActs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("a", "mean1", "rstd1", "qkv", "o", "lse", "h", "b", "rstd2", "up",
                                          "s")]


P = C.c_void_p
I = C.c_int
SZ = C.c_size_t
# name -> (restype, argtypes)
_SIGS = {
    "collider_last_error": (C.c_char_p, []),
    "collider_check": (I, [P]),
    "collider_selftest_wait_timeout": (I, [P]),
    "collider_launch_count": (C.c_longlong, [I]),
    "collider_profile_enable": (I, [I]),
    "collider_profile_count": (I, []),
    "collider_profile_get": (I, [I, C.POINTER(C.c_char_p), C.POINTER(C.c_longlong), C.POINTER(C.c_float)]),
    "collider_profile_get_span": (I, [I, C.POINTER(C.c_float), C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "collider_select_keep": (I, [P, I, I, I, P, P]),
    "collider_compact_workspace_size": (SZ, [I, I]),
    "collider_compact": (I, [P, I, I, P, P, P, P, SZ, P]),
    "collider_compact_noalloc": (I, [P, I, I, P, P, P, P]),
    "collider_gather_rows": (I, [P, SZ, P, SZ, SZ, I, P, P, P]),
    "collider_scatter_rows": (I, [P, SZ, P, SZ, SZ, I, P, P, P]),
    "collider_linear_workspace_size": (SZ, [I, I, I, I]),
    "collider_linear_bwd": (I, [I, I, I, I, P, I, P, P, I, P, P, P, I, P, P, P, SZ, P]),
    "collider_attn_workspace_size": (SZ, [I, I, I, I, I]),
    "collider_attn_bwd": (I, [I, I, I, I, I, I, C.c_float, I, C.c_float, P, P, P, P, P, I, I, I, I, P,
                              P, P, P, P, P, P, I, P, SZ, P]),
    "collider_layer_workspace_size": (SZ, [C.POINTER(LayerDesc)]),
    "collider_layer_bwd": (I, [C.POINTER(LayerDesc), C.POINTER(LayerWeights), C.POINTER(LayerSaved), P, I,
                               P, P, P, C.POINTER(LayerGrads), I, P, SZ, P]),
    "collider_layer_fwd_workspace_size": (SZ, [C.POINTER(LayerDesc)]),
    "collider_layer_fwd": (I, [C.POINTER(LayerDesc), C.POINTER(LayerParams), P, P, C.POINTER(LayerActs), P, SZ,
                               P]),
    "collider_stack_workspace_size": (SZ, [C.POINTER(LayerDesc), I, I]),
    "collider_stack_bwd": (I, [C.POINTER(LayerDesc), I, I, C.POINTER(LayerWeights), C.POINTER(LayerSaved),
                               P, P, P, P, P, P, P, P, P, P, P, C.POINTER(LayerGrads), P, P, P, P, SZ, P]),
}
EXPORTED = tuple(_SIGS)

_lib = None


def lib() -> C.CDLL:
    """Load libcollider.so (built in-tree); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m sparse_backward_gemm_gb300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != OK:
        raise ColliderError(status, lib().collider_last_error().decode())


def _nbytes(ws):
    if ws is None:
        return 0
    if hasattr(ws, "numel"):
        return ws.numel() * ws.element_size()
    raise TypeError("pass the workspace as a tensor (its size is taken from it)")


# --------------------------------------------------------------------------
def collider_last_error() -> str:
    return lib().collider_last_error().decode()


def collider_check(stream=None) -> None:
    _check(lib().collider_check(_stream(stream)))


def collider_selftest_wait_timeout(stream=None) -> None:
    _check(lib().collider_selftest_wait_timeout(_stream(stream)))


def collider_launch_count(reset: int = 0) -> int:
    return lib().collider_launch_count(reset)


def collider_profile_enable(on: int) -> None:
    lib().collider_profile_enable(int(on))


def collider_profile_count() -> int:
    return lib().collider_profile_count()


def collider_profile_get_span(i: int):
    """Returns (start_ms, end_ms, stream_index) of profile record i on the timeline of record 0."""
    a, b, k = C.c_float(), C.c_float(), C.c_int()
    if lib().collider_profile_get_span(i, C.byref(a), C.byref(b), C.byref(k)) != 0:
        raise IndexError(i)
    return a.value, b.value, k.value


def collider_profile_get(i: int):
    """Returns (name, (M, N, K, dyn), ms) of profile record i."""
    name = C.c_char_p()
    mnk = (C.c_longlong * 4)()
    ms = C.c_float()
    if lib().collider_profile_get(i, C.byref(name), mnk, C.byref(ms)) != 0:
        raise IndexError(i)
    return name.value.decode(), tuple(mnk), ms.value


def collider_select_keep(scores, B, T, n_filter, mask, stream=None) -> None:
    _check(lib().collider_select_keep(_ptr(scores), B, T, n_filter, _ptr(mask), _stream(stream)))


def collider_compact_workspace_size(B: int, T: int) -> int:
    return lib().collider_compact_workspace_size(B, T)


def collider_compact(mask, B, T, idx, cu_kept, n_kept, ws=None, stream=None) -> None:
    _check(lib().collider_compact(_ptr(mask), B, T, _ptr(idx), _ptr(cu_kept), _ptr(n_kept), _ptr(ws),
                                  _nbytes(ws), _stream(stream)))


def collider_compact_noalloc(mask, B, T, idx, cu_kept, n_kept, stream=None) -> None:
    """collider_compact without a workspace and without any allocation (scratch
    is a fixed array inside the library; B*T <= 2^30)."""
    _check(lib().collider_compact_noalloc(_ptr(mask), B, T, _ptr(idx), _ptr(cu_kept), _ptr(n_kept),
                                          _stream(stream)))


def collider_gather_rows(src, src_ld_bytes, dst, dst_ld_bytes, row_bytes, M, idx, n_kept, stream=None) -> None:
    _check(lib().collider_gather_rows(_ptr(src), src_ld_bytes, _ptr(dst), dst_ld_bytes, row_bytes, M, _ptr(idx),
                                      _ptr(n_kept), _stream(stream)))


def collider_scatter_rows(compact, compact_ld_bytes, full, full_ld_bytes, row_bytes, M, idx, n_kept,
                          stream=None) -> None:
    _check(lib().collider_scatter_rows(_ptr(compact), compact_ld_bytes, _ptr(full), full_ld_bytes, row_bytes, M,
                                       _ptr(idx), _ptr(n_kept), _stream(stream)))


def collider_linear_workspace_size(dtype, M, K, N) -> int:
    return lib().collider_linear_workspace_size(dtype, M, K, N)


def collider_linear_bwd(dtype, M, K, N, X, x_rows, W, dY, dy_rows, idx, n_kept, dX, dx_rows, dW, db, ws,
                        stream=None) -> None:
    _check(lib().collider_linear_bwd(dtype, M, K, N, _ptr(X), x_rows, _ptr(W), _ptr(dY), dy_rows, _ptr(idx),
                                     _ptr(n_kept), _ptr(dX), dx_rows, _ptr(dW), _ptr(db), _ptr(ws), _nbytes(ws),
                                     _stream(stream)))


def collider_attn_workspace_size(B, T, H, Hkv, dh) -> int:
    return lib().collider_attn_workspace_size(B, T, H, Hkv, dh)


def collider_attn_bwd(B, T, H, Hkv, dh, causal, scale, rotary_dim, rope_base, Q, K, V, O, dO, q_ld, kv_ld, do_ld,
                      in_rows, lse, idx, cu_kept, n_kept, dQ, dK, dV, out_rows, ws, stream=None) -> None:
    _check(lib().collider_attn_bwd(B, T, H, Hkv, dh, causal, scale, rotary_dim, rope_base, _ptr(Q), _ptr(K),
                                   _ptr(V), _ptr(O), _ptr(dO), q_ld, kv_ld, do_ld, in_rows, _ptr(lse), _ptr(idx),
                                   _ptr(cu_kept), _ptr(n_kept), _ptr(dQ), _ptr(dK), _ptr(dV), out_rows, _ptr(ws),
                                   _nbytes(ws), _stream(stream)))


def collider_layer_workspace_size(desc: LayerDesc) -> int:
    return lib().collider_layer_workspace_size(C.byref(desc))


def collider_layer_bwd(desc, weights, saved, dOut, dout_rows, idx, cu_kept, n_kept, grads, dx_rows, ws,
                       stream=None) -> None:
    _check(lib().collider_layer_bwd(C.byref(desc), C.byref(weights), C.byref(saved), _ptr(dOut), dout_rows,
                                    _ptr(idx), _ptr(cu_kept), _ptr(n_kept), C.byref(grads), dx_rows, _ptr(ws),
                                    _nbytes(ws), _stream(stream)))


def collider_layer_fwd_workspace_size(desc: LayerDesc) -> int:
    return lib().collider_layer_fwd_workspace_size(C.byref(desc))


def collider_layer_fwd(desc, params, x, y, acts, ws, stream=None) -> None:
    _check(lib().collider_layer_fwd(C.byref(desc), C.byref(params), _ptr(x), _ptr(y), C.byref(acts), _ptr(ws),
                                    _nbytes(ws), _stream(stream)))


def collider_stack_workspace_size(desc: LayerDesc, L: int, V: int) -> int:
    return lib().collider_stack_workspace_size(C.byref(desc), L, V)


def collider_stack_bwd(desc, L, V, weights, saved, logits, targets, ids, y, xL, rstdf, normf_w, w_lm, idx,
                       cu_kept, n_kept, grads, dnormf_w, dw_lm, dE, ws, stream=None) -> None:
    """weights / saved / grads: ctypes arrays of LayerWeights / LayerSaved / LayerGrads (length L)."""
    _check(lib().collider_stack_bwd(C.byref(desc), L, V, weights, saved, _ptr(logits), _ptr(targets), _ptr(ids),
                                    _ptr(y), _ptr(xL), _ptr(rstdf), _ptr(normf_w), _ptr(w_lm), _ptr(idx),
                                    _ptr(cu_kept), _ptr(n_kept), grads, _ptr(dnormf_w), _ptr(dw_lm), _ptr(dE),
                                    _ptr(ws), _nbytes(ws), _stream(stream)))
