"""Thin ctypes binding over the C ABI in include/addln.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libaddln.so``.  Tensors are PyTorch CUDA tensors (PyTorch
supplies device memory and the current stream); raw integer device pointers
are accepted too.  There is no CPU fallback: if the library is missing this
module raises on import of the first function call.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libaddln.so")

FP32, FP16, BF16 = 0, 1, 2
DTYPE_CODE = {torch.float32: FP32, torch.float16: FP16, torch.bfloat16: BF16}

OK = 0
ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_EPS, ERR_ALIAS = -1, -2, -3, -4, -5
ERR_LAUNCH, ERR_UNSUPPORTED, ERR_DEVICE_TIMEOUT, ERR_CUDA = -6, -7, -8, -9
ERR_WORKSPACE = -10
ERR_BOUNDS = -11

PATH_AUTO, PATH_WARP_VEC, PATH_CTA_TMA, PATH_CTA_VEC, PATH_SCALAR = 0, 1, 2, 3, 4

# Every symbol include/addln.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
SIGNATURES = {
    "add_layernorm_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                         ctypes.c_float, ctypes.c_int, _P]),
    "add_layernorm_fwd_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                              ctypes.c_float, ctypes.c_int, _P, _I64, _P]),
    "add_layernorm_fwd_host_workspace_size": (ctypes.c_int64, [_I64, _I64, ctypes.c_int,
                                                               ctypes.c_int, ctypes.c_int]),
    "add_layernorm_fwd_host_last_mode": (ctypes.c_int, []),
    "add_fwd": (ctypes.c_int, [_P, _P, _P, _I64, ctypes.c_int, _P]),
    "layernorm_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, ctypes.c_float,
                                     ctypes.c_int, _P]),
    "softmax_fwd": (ctypes.c_int, [_P, _P, _I64, _I64, ctypes.c_int, _P]),
    "bias_gelu_residual_fwd": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, ctypes.c_int, _P]),
    "bias_add_fwd": (ctypes.c_int, [_P, _P, _P, _I64, _I64, ctypes.c_int, _P]),
    "gelu_fwd": (ctypes.c_int, [_P, _P, _I64, ctypes.c_int, _P]),
    "add_layernorm_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                         ctypes.c_int, _P, _I64, _P]),
    "add_layernorm_bwd_workspace_size": (ctypes.c_int64, [_I64, _I64, ctypes.c_int]),
    "add_layernorm_bwd_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                                 ctypes.c_int, _P]),
    "addln_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "addln_max_hidden": (ctypes.c_int64, [ctypes.c_int]),
    "addln_get_device_error": (ctypes.c_int, [_P]),
    "addln_bounds_checked": (ctypes.c_int, []),
    "addln_bounds_violation": (ctypes.c_uint64, []),
    "addln_set_force_path": (ctypes.c_int, [ctypes.c_int]),
    "addln_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "addln_set_grid_cap": (ctypes.c_int64, [ctypes.c_int64]),
    "addln_set_pdl": (ctypes.c_int, [ctypes.c_int]),
    "addln_set_cta_shape": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "addln_set_warp_rows": (ctypes.c_int, [ctypes.c_int]),
    "addln_last_path": (ctypes.c_char_p, []),
    "addln_last_cuda_error": (ctypes.c_char_p, []),
}

_lib = None
_lock = threading.Lock()


class AddLNError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {strerror(code)} (code {code})"
        if code in (ERR_LAUNCH, ERR_CUDA):
            msg += f": {lib().addln_last_cuda_error().decode()}"
        super().__init__(msg)


def load(path: str):
    """A ctypes handle on the library at `path` with every header signature
    set (the normal build through lib(); the bounds-checked build's tests
    load theirs here)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                _lib = load(LIB_PATH)
    return _lib


def strerror(code: int) -> str:
    return lib().addln_strerror(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != OK:
        raise AddLNError(rc, where)


def _rows_shape(x):
    if x.dim() < 1:
        raise ValueError("x must have at least one dimension (the hidden dim)")
    H = x.shape[-1]
    rows = x.numel() // H if H else 0
    return rows, H


def _require(t, name, dtype=None, like=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if like is not None and t.numel() != like.numel():
        raise ValueError(f"{name} has {t.numel()} elements, expected {like.numel()}")


def add_layernorm_fwd(x, r, gamma, beta, y, resid_out=None, mean=None, rstd=None,
                      eps: float = 1e-5, stream=None, rows=None, H=None, dtype=None):
    """Fused residual-Add + LayerNorm into caller-provided outputs.

    With tensors, rows and H come from x's shape ([..., H]) and dtype from
    x.dtype.  With raw device pointers, pass rows, H and dtype explicitly.
    """
    if isinstance(x, torch.Tensor):
        rows_, H_ = _rows_shape(x)
        dtype_ = DTYPE_CODE.get(x.dtype)
        if dtype_ is None:
            raise ValueError(f"unsupported dtype {x.dtype}")
        for t, n in ((x, "x"), (r, "r"), (y, "y"), (resid_out, "resid_out")):
            if t is not None and isinstance(t, torch.Tensor):
                _require(t, n, x.dtype, like=x)
        for t, n in ((gamma, "gamma"), (beta, "beta")):
            if isinstance(t, torch.Tensor):
                _require(t, n, torch.float32)
                if t.numel() != H_:
                    raise ValueError(f"{n} must have H={H_} elements")
        for t, n in ((mean, "mean"), (rstd, "rstd")):
            if isinstance(t, torch.Tensor):
                _require(t, n, torch.float32)
                if t.numel() != rows_:
                    raise ValueError(f"{n} must have rows={rows_} elements")
        rows = rows_ if rows is None else rows
        H = H_ if H is None else H
        dtype = dtype_ if dtype is None else dtype
    rc = lib().add_layernorm_fwd(_ptr(x), _ptr(r), _ptr(gamma), _ptr(beta), _ptr(y),
                                 _ptr(resid_out), _ptr(mean), _ptr(rstd), int(rows), int(H),
                                 float(eps), int(dtype), _stream(stream))
    _check(rc, "add_layernorm_fwd")


def _require_host(t, name, dtype=None, like=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if like is not None and t.numel() != like.numel():
        raise ValueError(f"{name} has {t.numel()} elements, expected {like.numel()}")


def add_layernorm_fwd_host_workspace_size(rows: int, H: int, dtype: int, want_resid: bool = False,
                                          want_stats: bool = False) -> int:
    n = int(lib().add_layernorm_fwd_host_workspace_size(int(rows), int(H), int(dtype),
                                                         int(bool(want_resid)), int(bool(want_stats))))
    if n < 0:
        raise AddLNError(n, "add_layernorm_fwd_host_workspace_size")
    return n


HOST_PIPELINED = 1
HOST_MAPPED = 2


def add_layernorm_fwd_host_last_mode() -> int:
    """HOST_MAPPED or HOST_PIPELINED: how the last add_layernorm_fwd_host call
    moved its data (0 before any call)."""
    return int(lib().add_layernorm_fwd_host_last_mode())


def add_layernorm_fwd_host(x, r, gamma, beta, y, resid_out=None, mean=None, rstd=None,
                           eps: float = 1e-5, workspace=None, stream=None):
    """add_layernorm_fwd from host tensors to host tensors.

    The host-device traffic happens inside the call: read and written in
    place by the kernel when every row buffer is pinned and the GPU can reach
    host memory, else copied in pipelined chunks.  `workspace` is a CUDA uint8
    tensor of at least add_layernorm_fwd_host_workspace_size(...) bytes
    (allocated here when omitted).  Synchronise `stream` (default: the
    current stream) before reading the outputs.
    """
    rows, H = _rows_shape(x)
    dtype = DTYPE_CODE.get(x.dtype)
    if dtype is None:
        raise ValueError(f"unsupported dtype {x.dtype}")
    for t, n in ((x, "x"), (r, "r"), (y, "y"), (resid_out, "resid_out")):
        if t is not None:
            _require_host(t, n, x.dtype, like=x)
    for t, n in ((gamma, "gamma"), (beta, "beta")):
        _require_host(t, n, torch.float32)
        if t.numel() != H:
            raise ValueError(f"{n} must have H={H} elements")
    for t, n in ((mean, "mean"), (rstd, "rstd")):
        if t is not None:
            _require_host(t, n, torch.float32)
            if t.numel() != rows:
                raise ValueError(f"{n} must have rows={rows} elements")
    need = add_layernorm_fwd_host_workspace_size(rows, H, dtype, resid_out is not None,
                                                 mean is not None or rstd is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = lib().add_layernorm_fwd_host(_ptr(x), _ptr(r), _ptr(gamma), _ptr(beta), _ptr(y),
                                      _ptr(resid_out), _ptr(mean), _ptr(rstd), int(rows), int(H),
                                      float(eps), int(dtype), _ptr(workspace),
                                      int(workspace.numel() * workspace.element_size()),
                                      _stream(stream))
    _check(rc, "add_layernorm_fwd_host")


def layernorm_fwd(a, gamma, beta, y, mean=None, rstd=None, eps: float = 1e-5, stream=None,
                  rows=None, H=None, dtype=None):
    """LayerNorm of a stored [rows, H] tensor (second kernel of the unfused chain)."""
    if isinstance(a, torch.Tensor):
        rows_, H_ = _rows_shape(a)
        _require(a, "a")
        _require(y, "y", a.dtype, like=a)
        rows = rows_ if rows is None else rows
        H = H_ if H is None else H
        dtype = DTYPE_CODE[a.dtype] if dtype is None else dtype
    rc = lib().layernorm_fwd(_ptr(a), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(mean), _ptr(rstd),
                             int(rows), int(H), float(eps), int(dtype), _stream(stream))
    _check(rc, "layernorm_fwd")


def add_fwd(x, r, a, stream=None, n=None, dtype=None):
    """A = X + R elementwise (first kernel of the unfused chain)."""
    if isinstance(x, torch.Tensor):
        _require(x, "x")
        _require(r, "r", x.dtype, like=x)
        _require(a, "a", x.dtype, like=x)
        n = x.numel() if n is None else n
        dtype = DTYPE_CODE[x.dtype] if dtype is None else dtype
    _check(lib().add_fwd(_ptr(x), _ptr(r), _ptr(a), int(n), int(dtype), _stream(stream)), "add_fwd")


def softmax_fwd(x, y, stream=None, rows=None, H=None, dtype=None):
    """Row softmax of x ([..., H]) into y."""
    if isinstance(x, torch.Tensor):
        rows_, H_ = _rows_shape(x)
        _require(x, "x")
        _require(y, "y", x.dtype, like=x)
        rows = rows_ if rows is None else rows
        H = H_ if H is None else H
        dtype = DTYPE_CODE[x.dtype] if dtype is None else dtype
    _check(lib().softmax_fwd(_ptr(x), _ptr(y), int(rows), int(H), int(dtype), _stream(stream)),
           "softmax_fwd")


def softmax(x, stream=None):
    """Allocate y with PyTorch and run softmax_fwd."""
    y = torch.empty_like(x)
    softmax_fwd(x, y, stream=stream)
    return y


def bias_gelu_residual_fwd(x, r, bias, y, stream=None, rows=None, H=None, dtype=None):
    """Y = GELU(X + bias) + R in one kernel."""
    if isinstance(x, torch.Tensor):
        rows_, H_ = _rows_shape(x)
        _require(x, "x")
        _require(r, "r", x.dtype, like=x)
        _require(y, "y", x.dtype, like=x)
        _require(bias, "bias", torch.float32)
        if bias.numel() != H_:
            raise ValueError(f"bias must have H={H_} elements")
        rows = rows_ if rows is None else rows
        H = H_ if H is None else H
        dtype = DTYPE_CODE[x.dtype] if dtype is None else dtype
    _check(lib().bias_gelu_residual_fwd(_ptr(x), _ptr(r), _ptr(bias), _ptr(y), int(rows), int(H),
                                        int(dtype), _stream(stream)), "bias_gelu_residual_fwd")


def bias_add_fwd(x, bias, t, stream=None):
    rows, H = _rows_shape(x)
    _require(x, "x")
    _require(t, "t", x.dtype, like=x)
    _check(lib().bias_add_fwd(_ptr(x), _ptr(bias), _ptr(t), rows, H, DTYPE_CODE[x.dtype],
                              _stream(stream)), "bias_add_fwd")


def gelu_fwd(t, u, stream=None):
    _require(t, "t")
    _require(u, "u", t.dtype, like=t)
    _check(lib().gelu_fwd(_ptr(t), _ptr(u), t.numel(), DTYPE_CODE[t.dtype], _stream(stream)),
           "gelu_fwd")


def bias_gelu_residual(x, r, bias, stream=None):
    """Allocate Y with PyTorch and run bias_gelu_residual_fwd."""
    y = torch.empty_like(x)
    bias_gelu_residual_fwd(x, r, bias, y, stream=stream)
    return y


def bias_gelu_residual_unfused(x, r, bias, t=None, y=None, stream=None):
    """The three-kernel chain: T = X + bias, T = GELU(T), Y = T + R, each a
    separate HBM round trip (T is stored in the I/O dtype)."""
    t = torch.empty_like(x) if t is None else t
    y = torch.empty_like(x) if y is None else y
    bias_add_fwd(x, bias, t, stream=stream)
    gelu_fwd(t, t, stream=stream)
    add_fwd(t, r, y, stream=stream)
    return y


def add_layernorm_bwd_workspace_size(rows: int, H: int, dtype: int) -> int:
    n = int(lib().add_layernorm_bwd_workspace_size(int(rows), int(H), int(dtype)))
    if n < 0:
        raise AddLNError(n, "add_layernorm_bwd_workspace_size")
    return n


def bwd_workspace(rows: int, H: int, dtype, device=None):
    """A workspace for add_layernorm_bwd on rows x H of dtype (a torch dtype)."""
    nbytes = add_layernorm_bwd_workspace_size(rows, H, DTYPE_CODE[dtype])
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device or "cuda")


def add_layernorm_bwd(dy, a, mean, rstd, gamma, dx, dgamma=None, dbeta=None, dres=None,
                      workspace=None, stream=None):
    """Backward of add_layernorm_fwd into caller-provided dx (and dgamma,
    dbeta).  workspace: a CUDA tensor of at least
    add_layernorm_bwd_workspace_size(rows, H, dtype) bytes, reusable call
    after call (bwd_workspace makes one; allocated here when None and dgamma
    is wanted)."""
    rows, H = _rows_shape(dy)
    _require(dy, "dy")
    for t, n in ((a, "a"), (dx, "dx"), (dres, "dres")):
        if t is not None:
            _require(t, n, dy.dtype, like=dy)
    dt = DTYPE_CODE[dy.dtype]
    if dgamma is not None and workspace is None:
        workspace = bwd_workspace(rows, H, dy.dtype, dy.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().add_layernorm_bwd(_ptr(dy), _ptr(a), _ptr(mean), _ptr(rstd), _ptr(gamma),
                                   _ptr(dres), _ptr(dx), _ptr(dgamma), _ptr(dbeta), rows, H, dt,
                                   _ptr(workspace), wbytes, _stream(stream)), "add_layernorm_bwd")


NOALLOC_SCRATCH_BYTES = 32 << 20


def add_layernorm_bwd_noalloc(dy, a, mean, rstd, gamma, dx, dgamma=None, dbeta=None, dres=None,
                              stream=None):
    """add_layernorm_bwd with the library's built-in scratch buffer instead of
    a workspace, for callers that cannot allocate device memory.  Calls that
    can overlap on the GPU share that buffer and must be serialised."""
    rows, H = _rows_shape(dy)
    _require(dy, "dy")
    for t, n in ((a, "a"), (dx, "dx"), (dres, "dres")):
        if t is not None:
            _require(t, n, dy.dtype, like=dy)
    _check(lib().add_layernorm_bwd_noalloc(_ptr(dy), _ptr(a), _ptr(mean), _ptr(rstd), _ptr(gamma),
                                           _ptr(dres), _ptr(dx), _ptr(dgamma), _ptr(dbeta), rows,
                                           H, DTYPE_CODE[dy.dtype], _stream(stream)),
           "add_layernorm_bwd_noalloc")


def add_layernorm_backward(dy, a, mean, rstd, gamma, dres=None, stream=None):
    """Allocate outputs with PyTorch; returns (dx, dgamma, dbeta)."""
    dx = torch.empty_like(dy)
    H = dy.shape[-1]
    dg = torch.empty(H, dtype=torch.float32, device=dy.device)
    db = torch.empty(H, dtype=torch.float32, device=dy.device)
    add_layernorm_bwd(dy, a, mean, rstd, gamma, dx, dg, db, dres=dres, stream=stream)
    return dx, dg, db


def addln_max_hidden(dtype: int) -> int:
    return int(lib().addln_max_hidden(int(dtype)))


def addln_get_device_error(stream=None) -> int:
    return int(lib().addln_get_device_error(_stream(stream)))


def addln_set_force_path(path: int) -> int:
    return int(lib().addln_set_force_path(int(path)))


def addln_set_wait_limit_ns(ns: int) -> int:
    return int(lib().addln_set_wait_limit_ns(int(ns)))


def addln_set_grid_cap(ctas: int) -> int:
    return int(lib().addln_set_grid_cap(int(ctas)))


def addln_set_pdl(on: bool) -> int:
    return int(lib().addln_set_pdl(int(bool(on))))


def addln_set_cta_shape(threads: int, stages: int) -> int:
    return int(lib().addln_set_cta_shape(int(threads), int(stages)))


def addln_set_warp_rows(rows: int) -> int:
    """Test and benchmark only: rows a warp takes on the warp-per-row vector
    path (0 = by shape, 1 or 2 forced).  Returns the previous setting."""
    rc = int(lib().addln_set_warp_rows(int(rows)))
    if rc < 0:
        raise AddLNError(rc, "addln_set_warp_rows")
    return rc


def addln_last_path() -> str:
    return lib().addln_last_path().decode()


def addln_last_cuda_error() -> str:
    return lib().addln_last_cuda_error().decode()


def addln_strerror(code: int) -> str:
    return strerror(code)


# --------------------------------------------------------------- convenience
def add_layernorm(x, r, gamma, beta, eps: float = 1e-5, want_resid: bool = False,
                  want_stats: bool = False, stream=None):
    """Allocate outputs with PyTorch and run add_layernorm_fwd.

    Returns (y, resid_out or None, mean or None, rstd or None).
    """
    y = torch.empty_like(x)
    a = torch.empty_like(x) if want_resid else None
    rows, _ = _rows_shape(x)
    mean = torch.empty(rows, dtype=torch.float32, device=x.device) if want_stats else None
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device) if want_stats else None
    add_layernorm_fwd(x, r, gamma, beta, y, a, mean, rstd, eps=eps, stream=stream)
    return y, a, mean, rstd


def add_then_layernorm(x, r, gamma, beta, eps: float = 1e-5, want_stats: bool = False,
                       stream=None):
    """The unfused two-kernel chain: A = X + R to memory, then LayerNorm(A).

    Returns (y, a, mean or None, rstd or None).
    """
    a = torch.empty_like(x)
    y = torch.empty_like(x)
    rows, _ = _rows_shape(x)
    mean = torch.empty(rows, dtype=torch.float32, device=x.device) if want_stats else None
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device) if want_stats else None
    add_fwd(x, r, a, stream=stream)
    layernorm_fwd(a, gamma, beta, y, mean, rstd, eps=eps, stream=stream)
    return y, a, mean, rstd
