"""ctypes marshalling for the C oracle (test infrastructure only).

Inputs are host torch tensors or numpy arrays in the I/O dtype; every result
is a float64 numpy array.  The functions follow the definitions written out
at the top of ``addln_oracle.c`` ("算子融合与Kernel合并" 4.2 for LayerNorm,
"算子融合的收益量化" section 1 for the residual add).
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np
import torch

from .build import build_oracle

_DT = {"fp32": 0, "fp16": 1, "bf16": 2}
_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            lib.oracle_decode.argtypes = [_P, ctypes.c_int, _I64, _P]
            lib.oracle_round.argtypes = [_P, ctypes.c_int, _I64, _P]
            lib.oracle_add.argtypes = [_P, _P, ctypes.c_int, _I64, ctypes.c_int, _P]
            lib.oracle_layernorm.argtypes = [_P, _P, _P, _I64, _I64, ctypes.c_double, _P, _P, _P]
            lib.oracle_add_layernorm.argtypes = [_P, _P, ctypes.c_int, _P, _P, _I64, _I64,
                                                 ctypes.c_double, ctypes.c_int, _P, _P, _P, _P]
            lib.oracle_softmax.argtypes = [_P, ctypes.c_int, _I64, _I64, _P, _P, _P]
            lib.oracle_bias_gelu_residual.argtypes = [_P, _P, ctypes.c_int, _P, _I64, _I64,
                                                      ctypes.c_int, _P]
            lib.oracle_add_layernorm_bwd.argtypes = [_P, _P, _P, _P, _P, _P, ctypes.c_int, _I64,
                                                     _I64, _P, _P, _P]
            for f in ("oracle_decode", "oracle_round", "oracle_add", "oracle_layernorm",
                      "oracle_add_layernorm", "oracle_softmax", "oracle_bias_gelu_residual",
                      "oracle_add_layernorm_bwd"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _raw(t, dtype: str) -> np.ndarray:
    """Contiguous host array holding the raw encoding of ``t`` in ``dtype``."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if dtype == "fp32":
            assert t.dtype == torch.float32, t.dtype
            return t.numpy()
        assert t.dtype == {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype], t.dtype
        return t.view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(t)
    if dtype == "fp32":
        assert a.dtype == np.float32
    else:
        assert a.dtype in (np.uint16, np.int16, np.float16) and a.itemsize == 2
    return a


def _f32(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous().to(torch.float32).numpy()
    return np.ascontiguousarray(t, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: bad argument (oracle returned {rc})")


def oracle_decode(t, dtype: str) -> np.ndarray:
    src = _raw(t, dtype)
    out = np.empty(src.shape, dtype=np.float64)
    _check(load().oracle_decode(_ptr(src), _DT[dtype], src.size, _ptr(out)), "oracle_decode")
    return out


def oracle_round(v, dtype: str) -> np.ndarray:
    """Round fp64 values to ``dtype`` (nearest, ties to even); result in fp64."""
    src = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(src.shape, dtype=np.float64)
    _check(load().oracle_round(_ptr(src), _DT[dtype], src.size, _ptr(out)), "oracle_round")
    return out


def oracle_add(x, r, dtype: str, round_A: bool = False) -> np.ndarray:
    xs, rs = _raw(x, dtype), _raw(r, dtype)
    assert xs.shape == rs.shape
    out = np.empty(xs.shape, dtype=np.float64)
    _check(load().oracle_add(_ptr(xs), _ptr(rs), _DT[dtype], xs.size, int(round_A), _ptr(out)),
           "oracle_add")
    return out


def oracle_layernorm(a, gamma, beta, eps: float) -> dict:
    """LayerNorm of fp64 rows ``a`` ([rows, H]).  Returns y, mean, rstd."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    rows, H = a.shape
    g, b = _f32(gamma), _f32(beta)
    assert g.shape == (H,) and b.shape == (H,)
    y = np.empty((rows, H), dtype=np.float64)
    mean = np.empty(rows, dtype=np.float64)
    rstd = np.empty(rows, dtype=np.float64)
    _check(load().oracle_layernorm(_ptr(a), _ptr(g), _ptr(b), rows, H, float(eps),
                                   _ptr(y), _ptr(mean), _ptr(rstd)), "oracle_layernorm")
    return {"y": y, "mean": mean, "rstd": rstd}


def oracle_add_layernorm(x, r, gamma, beta, eps: float, dtype: str, round_A: bool = False,
                         want_y: bool = True, want_a: bool = True, want_stats: bool = True) -> dict:
    """The fused operation on host rows.  Returns fp64 arrays y, a (A rounded
    to ``dtype``), mean, rstd (each None when not requested)."""
    xs, rs = _raw(x, dtype), _raw(r, dtype)
    assert xs.shape == rs.shape and xs.ndim == 2
    rows, H = xs.shape
    g, b = _f32(gamma), _f32(beta)
    assert g.shape == (H,) and b.shape == (H,)
    y = np.empty((rows, H), dtype=np.float64) if want_y else None
    a = np.empty((rows, H), dtype=np.float64) if want_a else None
    mean = np.empty(rows, dtype=np.float64) if want_stats else None
    rstd = np.empty(rows, dtype=np.float64) if want_stats else None
    _check(load().oracle_add_layernorm(_ptr(xs), _ptr(rs), _DT[dtype], _ptr(g), _ptr(b), rows, H,
                                       float(eps), int(round_A), _ptr(y), _ptr(a), _ptr(mean),
                                       _ptr(rstd)), "oracle_add_layernorm")
    return {"y": y, "a": a, "mean": mean, "rstd": rstd}


def oracle_softmax(x, dtype: str) -> dict:
    """Row softmax of host rows ``x`` ([rows, H] in dtype): fp64 y, and the
    per-row max and exp-sum ("算子融合与Kernel合并" 4.3, fused_softmax)."""
    xs = _raw(x, dtype)
    assert xs.ndim == 2
    rows, H = xs.shape
    y = np.empty((rows, H), dtype=np.float64)
    mx = np.empty(rows, dtype=np.float64)
    sm = np.empty(rows, dtype=np.float64)
    _check(load().oracle_softmax(_ptr(xs), _DT[dtype], rows, H, _ptr(y), _ptr(mx), _ptr(sm)),
           "oracle_softmax")
    return {"y": y, "max": mx, "sum": sm}


def oracle_bias_gelu_residual(x, r, bias, dtype: str, round_intermediates: bool = False) -> np.ndarray:
    """Y = GELU(X + bias) + R (exact erf GELU) in fp64, [rows, H]; with
    round_intermediates, X + bias and its GELU are rounded to the dtype first
    (the unfused chain that stores them)."""
    xs, rs = _raw(x, dtype), _raw(r, dtype)
    assert xs.shape == rs.shape and xs.ndim == 2
    rows, H = xs.shape
    b = _f32(bias)
    assert b.shape == (H,)
    y = np.empty((rows, H), dtype=np.float64)
    _check(load().oracle_bias_gelu_residual(_ptr(xs), _ptr(rs), _DT[dtype], _ptr(b), rows, H,
                                            int(round_intermediates), _ptr(y)),
           "oracle_bias_gelu_residual")
    return y


def oracle_add_layernorm_bwd(dy, a, mean, rstd, gamma, dtype: str, dres=None) -> dict:
    """Backward of the fused operation (textbook derivative) in fp64: dx
    ([rows, H], = dX = dR), dgamma, dbeta ([H]).  a is the stored sum A in the
    dtype; mean, rstd are the saved fp32 statistics."""
    dys, As = _raw(dy, dtype), _raw(a, dtype)
    assert dys.shape == As.shape and dys.ndim == 2
    rows, H = dys.shape
    m, rs, g = _f32(mean), _f32(rstd), _f32(gamma)
    assert m.shape == (rows,) and rs.shape == (rows,) and g.shape == (H,)
    dr = _raw(dres, dtype) if dres is not None else None
    dx = np.empty((rows, H), dtype=np.float64)
    dg = np.empty(H, dtype=np.float64)
    db = np.empty(H, dtype=np.float64)
    _check(load().oracle_add_layernorm_bwd(_ptr(dys), _ptr(As), _ptr(m), _ptr(rs), _ptr(g),
                                           _ptr(dr), _DT[dtype], rows, H, _ptr(dx), _ptr(dg),
                                           _ptr(db)), "oracle_add_layernorm_bwd")
    return {"dx": dx, "dgamma": dg, "dbeta": db}
