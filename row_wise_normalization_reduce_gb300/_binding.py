"""ctypes binding of libnrm.so (include/nrm.h).

Argument marshalling only: every step of every operator runs in the CUDA
library.  torch provides the device memory and the current stream.  If the
library is missing the first call raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnrm.so")

NRM_F32, NRM_F16, NRM_BF16 = 0, 1, 2
PLAN_AUTO, PLAN_GENERIC, PLAN_WARP, PLAN_CTA, PLAN_TMA, PLAN_PERSIST, PLAN_WRAW, PLAN_CLUSTER = range(8)
PLAN_NAMES = {0: "auto", 1: "generic", 2: "warp", 3: "cta", 4: "tma", 5: "persist", 6: "wraw",
              7: "cluster"}

_DT = {torch.float32: NRM_F32, torch.float16: NRM_F16, torch.bfloat16: NRM_BF16}

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int


class NrmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


def _declare(lib):
    lib.ln_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _INT, _P]
    lib.rms_fwd.argtypes = [_P, _P, _P, _P, _I64, _I64, _F, _INT, _P]
    lib.add_rms_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _INT, _P]
    lib.bn_fwd_train_workspace_size.argtypes = [_I64, _I64, _I64, _INT]
    lib.bn_fwd_train_workspace_size.restype = ctypes.c_size_t
    lib.bn_fwd_train.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, _INT,
                                 _P, ctypes.c_size_t, _P]
    for f in ("ln_fwd", "rms_fwd", "add_rms_fwd", "bn_fwd_train"):
        getattr(lib, f).restype = _INT
    lib.bn_fwd_train_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F,
                                         _F, _INT, _P]
    lib.bn_fwd_train_noalloc.restype = _INT
    lib.bn_fwd_infer.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _INT, _P]
    lib.bn_fwd_infer.restype = _INT
    lib.bn_bwd_workspace_size.argtypes = [_I64, _I64, _I64, _INT]
    lib.bn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.bn_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P,
                           ctypes.c_size_t, _P]
    lib.bn_bwd.restype = _INT
    lib.softmax_fwd.argtypes = [_P, _P, _P, _P, _I64, _I64, _INT, _P]
    lib.softmax_fwd.restype = _INT
    lib.ln_fwd_ld.argtypes = [_P, _I64, _P, _P, _P, _I64, _P, _P, _I64, _I64, _F, _INT, _P]
    lib.rms_fwd_ld.argtypes = [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _F, _INT, _P]
    lib.add_rms_fwd_ld.argtypes = [_P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _P, _I64, _I64,
                                   _F, _INT, _P]
    lib.softmax_fwd_ld.argtypes = [_P, _I64, _P, _I64, _P, _P, _I64, _I64, _INT, _P]
    for f in ("ln_fwd_ld", "rms_fwd_ld", "add_rms_fwd_ld", "softmax_fwd_ld"):
        getattr(lib, f).restype = _INT
    lib.bn_fwd_partial_stats.argtypes = [_P, _P, _I64, _I64, _I64, _INT, _P, ctypes.c_size_t, _P]
    lib.bn_fwd_apply_stats.argtypes = [_P, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _I64, _I64, _I64,
                                       _F, _F, _INT, _P]
    lib.bn_bwd_partial_sums.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _INT, _P,
                                        ctypes.c_size_t, _P]
    lib.bn_bwd_apply_sums.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _I64, _I64,
                                      _I64, _INT, _P]
    for f in ("bn_fwd_partial_stats", "bn_fwd_apply_stats", "bn_bwd_partial_sums",
              "bn_bwd_apply_sums"):
        getattr(lib, f).restype = _INT
    lib.add_rms_fwd_host_workspace_size.argtypes = [_I64, _INT]
    lib.add_rms_fwd_host_workspace_size.restype = ctypes.c_size_t
    lib.add_rms_fwd_host.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _INT, _P,
                                     ctypes.c_size_t, _P]
    lib.add_rms_fwd_host.restype = _INT
    lib.nrm_status_string.argtypes = [_INT]
    lib.nrm_status_string.restype = ctypes.c_char_p
    lib.nrm_force_plan.argtypes = [_INT, _INT, _INT, _INT, _INT]
    lib.nrm_force_plan.restype = _INT
    lib.nrm_last_plan.argtypes = [ctypes.POINTER(_INT)] * 5
    lib.nrm_last_plan.restype = None
    lib.nrm_set_wait_limit.argtypes = [ctypes.c_uint]
    lib.nrm_set_wait_limit.restype = ctypes.c_uint
    lib.nrm_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint), _INT]
    lib.nrm_device_fault.restype = _INT
    lib.nrm_set_pointer_checks.argtypes = [_INT]
    lib.nrm_set_pointer_checks.restype = _INT
    lib.nrm_set_bn_group_bytes.argtypes = [ctypes.c_size_t]
    lib.nrm_set_bn_group_bytes.restype = ctypes.c_size_t
    return lib


def lib():
    """The loaded libnrm.so (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it first "
                        "(python -c 'import __graft_entry__ as g; g.build()')")
                _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(status: int) -> str:
    return lib().nrm_status_string(status).decode()


def _check(status: int, where: str):
    if status != 0:
        raise NrmError(status, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _param(p, n, dtype, device, name):
    if p is None:
        return None
    _cuda(p, name)
    if p.dtype != dtype or p.numel() != n or p.device != device:
        raise ValueError(f"{name} must be [{n}] {dtype} on {device}")
    return p


def _rows_view(x: torch.Tensor):
    n = x.shape[-1]
    return x.numel() // n if n else 0, n


def _rows(t: torch.Tensor, name: str):
    """(rows, N, row stride) of a row-operator tensor: contiguous, or 2-D with
    unit column stride (a column slice or a padded buffer)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    n = t.shape[-1]
    if t.is_contiguous():
        return (t.numel() // n if n else 0), n, n
    if t.dim() == 2 and t.stride(1) == 1 and t.stride(0) >= n:
        return t.shape[0], n, t.stride(0)
    raise ValueError(f"{name} must be contiguous, or 2-D with unit column stride")


def _same_rows(t, x, name):
    if t.shape != x.shape or t.dtype != x.dtype or t.device != x.device:
        raise ValueError(f"{name} must match x in shape, dtype and device")
    return _rows(t, name)[2]


# ---------------------------------------------------------------------------
# Operators (same names as the C ABI).
# ---------------------------------------------------------------------------
def ln_fwd(x, gamma=None, beta=None, eps=1e-5, *, out=None, mean=None, rstd=None,
           want_stats=True, stream=None):
    """LayerNorm over the last dimension of x.  Returns (y, mean, rstd).  x
    (and out) may be 2-D views with a row stride (ln_fwd_ld)."""
    rows, n, ldx = _rows(x, "x")
    gamma = _param(gamma, n, x.dtype, x.device, "gamma")
    beta = _param(beta, n, x.dtype, x.device, "beta")
    y = torch.empty(x.shape, device=x.device, dtype=x.dtype) if out is None else out
    ldy = _same_rows(y, x, "out")
    if want_stats:
        mean = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32) if mean is None else mean
        rstd = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32) if rstd is None else rstd
    with torch.cuda.device(x.device):
        st = lib().ln_fwd_ld(_ptr(x), ldx, _ptr(gamma), _ptr(beta), _ptr(y), ldy, _ptr(mean),
                             _ptr(rstd), rows, n, eps, _dtype_code(x),
                             stream if stream is not None else _stream(x.device))
    _check(st, "ln_fwd")
    return y, mean, rstd


def rms_fwd(x, w=None, eps=1e-6, *, out=None, rstd=None, want_stats=False, stream=None):
    """RMSNorm over the last dimension of x.  Returns (y, rstd or None)."""
    rows, n, ldx = _rows(x, "x")
    w = _param(w, n, x.dtype, x.device, "w")
    y = torch.empty(x.shape, device=x.device, dtype=x.dtype) if out is None else out
    ldy = _same_rows(y, x, "out")
    if want_stats and rstd is None:
        rstd = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32)
    with torch.cuda.device(x.device):
        st = lib().rms_fwd_ld(_ptr(x), ldx, _ptr(w), _ptr(y), ldy, _ptr(rstd), rows, n, eps,
                              _dtype_code(x), stream if stream is not None else _stream(x.device))
    _check(st, "rms_fwd")
    return y, rstd


def add_rms_fwd(x, residual, w=None, eps=1e-6, *, residual_out=None, out=None, rstd=None,
                want_stats=False, stream=None):
    """residual_out = x + residual (rounded to x.dtype); y = RMSNorm(residual_out, w).
    Returns (residual_out, y, rstd or None).  Pass residual_out=residual to update
    the residual stream in place."""
    rows, n, ldx = _rows(x, "x")
    ldr = _same_rows(residual, x, "residual")
    w = _param(w, n, x.dtype, x.device, "w")
    ro = torch.empty(x.shape, device=x.device, dtype=x.dtype) if residual_out is None else residual_out
    ldro = _same_rows(ro, x, "residual_out")
    y = torch.empty(x.shape, device=x.device, dtype=x.dtype) if out is None else out
    ldy = _same_rows(y, x, "out")
    if want_stats and rstd is None:
        rstd = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32)
    with torch.cuda.device(x.device):
        st = lib().add_rms_fwd_ld(_ptr(x), ldx, _ptr(residual), ldr, _ptr(w), _ptr(ro), ldro,
                                  _ptr(y), ldy, _ptr(rstd), rows, n, eps, _dtype_code(x),
                                  stream if stream is not None else _stream(x.device))
    _check(st, "add_rms_fwd")
    return ro, y, rstd


def add_rms_fwd_host_workspace(n, dtype, device=None):
    """Device staging buffer for add_rms_fwd_host on rows of length n."""
    nbytes = lib().add_rms_fwd_host_workspace_size(n, _DT[dtype])
    return torch.empty(max(nbytes, 256), dtype=torch.uint8,
                       device=device if device is not None else torch.device("cuda"))


def add_rms_fwd_host(x, residual, w=None, eps=1e-6, *, residual_out=None, out=None, rstd=None,
                     workspace=None, stream=None, synchronize=True):
    """add_rms_fwd on HOST tensors (pinned memory is fastest), streamed through
    the current device in chunks.  w and rstd are device tensors.  Returns
    (residual_out, y); with synchronize=False they are complete only once the
    stream is."""
    if x.is_cuda or residual.is_cuda:
        raise ValueError("x and residual must be host tensors")
    if not (x.is_contiguous() and residual.is_contiguous()):
        raise ValueError("x and residual must be contiguous")
    if residual.shape != x.shape or residual.dtype != x.dtype:
        raise ValueError("residual must match x in shape and dtype")
    rows, n = _rows_view(x)
    device = torch.device("cuda", torch.cuda.current_device())
    w = _param(w, n, x.dtype, device, "w")
    ro = torch.empty_like(x) if residual_out is None else residual_out
    y = torch.empty_like(x) if out is None else out
    for t, name in ((ro, "residual_out"), (y, "out")):
        if t.is_cuda or not t.is_contiguous() or t.shape != x.shape or t.dtype != x.dtype:
            raise ValueError(f"{name} must be a contiguous host tensor like x")
    ws = add_rms_fwd_host_workspace(n, x.dtype, device) if workspace is None else workspace
    s = stream if stream is not None else _stream(device)
    st = lib().add_rms_fwd_host(_ptr(x), _ptr(residual), _ptr(w), _ptr(ro), _ptr(y), _ptr(rstd),
                                rows, n, eps, _dtype_code(x), _ptr(ws),
                                ws.numel() * ws.element_size(), s)
    _check(st, "add_rms_fwd_host")
    if synchronize:
        torch.cuda.current_stream(device).synchronize() if stream is None else \
            torch.cuda.synchronize(device)
    return ro, y


def bn_fwd_train_workspace_size(batch, c, hw, dtype=torch.float32) -> int:
    return lib().bn_fwd_train_workspace_size(batch, c, hw, _DT[dtype])


def _bn_train_tensors(x, gamma, beta, running_mean, running_var, out, save_mean, save_rstd):
    """Checks shared by both training-forward entry points; allocates the
    outputs that are None.  Returns (batch, c, hw, gamma, beta, y, save_mean,
    save_rstd)."""
    _cuda(x, "x")
    if x.dim() < 2:
        raise ValueError("x must be [batch, C, ...]")
    batch, c = x.shape[0], x.shape[1]
    hw = x.numel() // (batch * c) if batch * c else 0
    gamma = _param(gamma, c, x.dtype, x.device, "gamma")
    beta = _param(beta, c, x.dtype, x.device, "beta")
    for t, name in ((running_mean, "running_mean"), (running_var, "running_var"),
                    (save_mean, "save_mean"), (save_rstd, "save_rstd")):
        if t is not None:
            _cuda(t, name)
            if t.dtype != torch.float32 or t.numel() != c or t.device != x.device:
                raise ValueError(f"{name} must be [{c}] float32 on {x.device}")
    if out is not None:
        _cuda(out, "out")
        if out.shape != x.shape or out.dtype != x.dtype or out.device != x.device:
            raise ValueError("out must be like x")
    y = torch.empty_like(x) if out is None else out
    save_mean = torch.empty(c, device=x.device, dtype=torch.float32) if save_mean is None else save_mean
    save_rstd = torch.empty(c, device=x.device, dtype=torch.float32) if save_rstd is None else save_rstd
    return batch, c, hw, gamma, beta, y, save_mean, save_rstd


def bn_fwd_train(x, gamma=None, beta=None, running_mean=None, running_var=None, eps=1e-5,
                 momentum=0.1, *, out=None, save_mean=None, save_rstd=None, workspace=None,
                 stream=None):
    """BatchNorm2d training forward over NCHW x.  Returns (y, save_mean, save_rstd);
    running_mean / running_var (binary32) are updated in place when given."""
    batch, c, hw, gamma, beta, y, save_mean, save_rstd = _bn_train_tensors(
        x, gamma, beta, running_mean, running_var, out, save_mean, save_rstd)
    need = lib().bn_fwd_train_workspace_size(batch, c, hw, _dtype_code(x))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    with torch.cuda.device(x.device):
        st = lib().bn_fwd_train(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(save_mean),
                                _ptr(save_rstd), _ptr(running_mean), _ptr(running_var), batch, c,
                                hw, eps, momentum, _dtype_code(x), _ptr(workspace),
                                workspace.numel() * workspace.element_size(),
                                stream if stream is not None else _stream(x.device))
    _check(st, "bn_fwd_train")
    return y, save_mean, save_rstd


def bn_fwd_train_noalloc(x, gamma=None, beta=None, running_mean=None, running_var=None,
                         eps=1e-5, momentum=0.1, *, out, save_mean, save_rstd, stream=None):
    """bn_fwd_train for callers that cannot allocate device memory at call time:
    every output is passed in (same checks as bn_fwd_train), and the library
    keeps the partial statistics in a fixed array of its own (batch * C <=
    65536).  Returns (y, save_mean, save_rstd)."""
    if out is None or save_mean is None or save_rstd is None:
        raise ValueError("bn_fwd_train_noalloc allocates nothing: pass out, save_mean and save_rstd")
    batch, c, hw, gamma, beta, y, save_mean, save_rstd = _bn_train_tensors(
        x, gamma, beta, running_mean, running_var, out, save_mean, save_rstd)
    with torch.cuda.device(x.device):
        st = lib().bn_fwd_train_noalloc(
            _ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(save_mean), _ptr(save_rstd),
            _ptr(running_mean), _ptr(running_var), batch, c, hw, eps, momentum, _dtype_code(x),
            stream if stream is not None else _stream(x.device))
    _check(st, "bn_fwd_train_noalloc")
    return y, save_mean, save_rstd


def softmax_fwd(x, *, out=None, row_max=None, row_sum=None, want_stats=False, stream=None):
    """Softmax over the last dimension of x.  Returns (y, row_max, row_sum);
    the statistics are None unless requested or passed in."""
    rows, n, ldx = _rows(x, "x")
    y = torch.empty(x.shape, device=x.device, dtype=x.dtype) if out is None else out
    ldy = _same_rows(y, x, "out")
    if want_stats:
        if row_max is None:
            row_max = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32)
        if row_sum is None:
            row_sum = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32)
    with torch.cuda.device(x.device):
        st = lib().softmax_fwd_ld(_ptr(x), ldx, _ptr(y), ldy, _ptr(row_max), _ptr(row_sum),
                                  rows, n, _dtype_code(x),
                                  stream if stream is not None else _stream(x.device))
    _check(st, "softmax_fwd")
    return y, row_max, row_sum


def _nchw(x):
    _cuda(x, "x")
    if x.dim() < 2:
        raise ValueError("x must be [batch, C, ...]")
    batch, c = x.shape[0], x.shape[1]
    hw = 1
    for d in x.shape[2:]:
        hw *= d
    return batch, c, hw


def _stat(t, c, device, name):
    _cuda(t, name)
    if t.dtype != torch.float32 or t.numel() != c or t.device != device:
        raise ValueError(f"{name} must be [{c}] float32 on {device}")
    return t


def bn_fwd_infer(x, running_mean, running_var, gamma=None, beta=None, eps=1e-5, *, out=None,
                 stream=None):
    """BatchNorm2d inference forward over NCHW x with the running statistics.
    Returns y."""
    batch, c, hw = _nchw(x)
    gamma = _param(gamma, c, x.dtype, x.device, "gamma")
    beta = _param(beta, c, x.dtype, x.device, "beta")
    running_mean = _stat(running_mean, c, x.device, "running_mean")
    running_var = _stat(running_var, c, x.device, "running_var")
    y = torch.empty_like(x) if out is None else out
    with torch.cuda.device(x.device):
        st = lib().bn_fwd_infer(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(running_mean),
                                _ptr(running_var), batch, c, hw, eps, _dtype_code(x),
                                stream if stream is not None else _stream(x.device))
    _check(st, "bn_fwd_infer")
    return y


def bn_bwd_workspace_size(batch, c, hw, dtype=torch.float32) -> int:
    return lib().bn_bwd_workspace_size(batch, c, hw, _DT[dtype])


def bn_bwd(dy, x, save_mean, save_rstd, gamma=None, *, out=None, dgamma=None, dbeta=None,
           workspace=None, stream=None):
    """BatchNorm2d training backward over NCHW tensors, from the statistics the
    training forward saved.  Returns (dx, dgamma, dbeta)."""
    batch, c, hw = _nchw(x)
    _cuda(dy, "dy")
    if dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy must match x in shape and dtype")
    gamma = _param(gamma, c, x.dtype, x.device, "gamma")
    save_mean = _stat(save_mean, c, x.device, "save_mean")
    save_rstd = _stat(save_rstd, c, x.device, "save_rstd")
    dx = torch.empty_like(x) if out is None else out
    dgamma = torch.empty(c, device=x.device, dtype=torch.float32) if dgamma is None else dgamma
    dbeta = torch.empty(c, device=x.device, dtype=torch.float32) if dbeta is None else dbeta
    need = lib().bn_bwd_workspace_size(batch, c, hw, _dtype_code(x))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    with torch.cuda.device(x.device):
        st = lib().bn_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(save_mean), _ptr(save_rstd),
                          _ptr(dx), _ptr(dgamma), _ptr(dbeta), batch, c, hw, _dtype_code(x),
                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                          stream if stream is not None else _stream(x.device))
    _check(st, "bn_bwd")
    return dx, dgamma, dbeta


def _scratch(batch, c, hw, dtype, device, workspace):
    need = max(lib().bn_fwd_train_workspace_size(batch, c, hw, _DT[dtype]), 16)
    if workspace is None:
        return torch.empty(need, device=device, dtype=torch.uint8)
    return workspace


def bn_fwd_partial_stats(x, *, out=None, workspace=None, stream=None):
    """Per-channel (count, mean, M2) of this process's batch, [C, 3] float64."""
    batch, c, hw = _nchw(x)
    stats = torch.empty(c, 3, device=x.device, dtype=torch.float64) if out is None else out
    ws = _scratch(batch, c, hw, x.dtype, x.device, workspace)
    with torch.cuda.device(x.device):
        st = lib().bn_fwd_partial_stats(_ptr(x), _ptr(stats), batch, c, hw, _dtype_code(x),
                                        _ptr(ws), ws.numel() * ws.element_size(),
                                        stream if stream is not None else _stream(x.device))
    _check(st, "bn_fwd_partial_stats")
    return stats


def bn_fwd_apply_stats(x, parts, gamma=None, beta=None, running_mean=None, running_var=None,
                       eps=1e-5, momentum=0.1, *, out=None, save_mean=None, save_rstd=None,
                       stream=None):
    """Training forward of the local batch from the exchanged [nparts, C, 3]
    float64 statistics.  Returns (y, save_mean, save_rstd)."""
    batch, c, hw = _nchw(x)
    if parts.dtype != torch.float64 or parts.dim() != 3 or parts.shape[1:] != (c, 3):
        raise ValueError(f"parts must be [nparts, {c}, 3] float64")
    _cuda(parts, "parts")
    gamma = _param(gamma, c, x.dtype, x.device, "gamma")
    beta = _param(beta, c, x.dtype, x.device, "beta")
    y = torch.empty_like(x) if out is None else out
    save_mean = torch.empty(c, device=x.device, dtype=torch.float32) if save_mean is None else save_mean
    save_rstd = torch.empty(c, device=x.device, dtype=torch.float32) if save_rstd is None else save_rstd
    with torch.cuda.device(x.device):
        st = lib().bn_fwd_apply_stats(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), _ptr(parts),
                                      parts.shape[0], _ptr(save_mean), _ptr(save_rstd),
                                      _ptr(running_mean), _ptr(running_var), batch, c, hw, eps,
                                      momentum, _dtype_code(x),
                                      stream if stream is not None else _stream(x.device))
    _check(st, "bn_fwd_apply_stats")
    return y, save_mean, save_rstd


def bn_bwd_partial_sums(dy, x, save_mean, save_rstd, *, out=None, workspace=None, stream=None):
    """Per-channel (sum dy, sum dy * xhat) of this process's batch, [C, 2] float64."""
    batch, c, hw = _nchw(x)
    _cuda(dy, "dy")
    sums = torch.empty(c, 2, device=x.device, dtype=torch.float64) if out is None else out
    ws = _scratch(batch, c, hw, x.dtype, x.device, workspace)
    with torch.cuda.device(x.device):
        st = lib().bn_bwd_partial_sums(_ptr(dy), _ptr(x), _ptr(save_mean), _ptr(save_rstd),
                                       _ptr(sums), batch, c, hw, _dtype_code(x), _ptr(ws),
                                       ws.numel() * ws.element_size(),
                                       stream if stream is not None else _stream(x.device))
    _check(st, "bn_bwd_partial_sums")
    return sums


def bn_bwd_apply_sums(dy, x, save_mean, save_rstd, parts, count, gamma=None, *, out=None,
                      dgamma=None, dbeta=None, stream=None):
    """Backward of the local batch from the exchanged [nparts, C, 2] float64
    sums and the global count.  Returns (dx, dgamma, dbeta)."""
    batch, c, hw = _nchw(x)
    _cuda(dy, "dy")
    if parts.dtype != torch.float64 or parts.dim() != 3 or parts.shape[1:] != (c, 2):
        raise ValueError(f"parts must be [nparts, {c}, 2] float64")
    gamma = _param(gamma, c, x.dtype, x.device, "gamma")
    dx = torch.empty_like(x) if out is None else out
    dgamma = torch.empty(c, device=x.device, dtype=torch.float32) if dgamma is None else dgamma
    dbeta = torch.empty(c, device=x.device, dtype=torch.float32) if dbeta is None else dbeta
    with torch.cuda.device(x.device):
        st = lib().bn_bwd_apply_sums(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(save_mean),
                                     _ptr(save_rstd), _ptr(parts), parts.shape[0], count,
                                     _ptr(dx), _ptr(dgamma), _ptr(dbeta), batch, c, hw,
                                     _dtype_code(x),
                                     stream if stream is not None else _stream(x.device))
    _check(st, "bn_bwd_apply_sums")
    return dx, dgamma, dbeta


# ---------------------------------------------------------------------------
# Plan control (tests and measurements).
# ---------------------------------------------------------------------------
def force_plan(plan: int = PLAN_AUTO, threads: int = 0, packs: int = 0, stages: int = 0,
               groups: int = 0):
    _check(lib().nrm_force_plan(plan, threads, packs, stages, groups), "nrm_force_plan")


def last_plan():
    """(plan, threads, packs, stages, groups) of this thread's last row-operator call."""
    v = [_INT() for _ in range(5)]
    lib().nrm_last_plan(*[ctypes.byref(x) for x in v])
    return tuple(x.value for x in v)


def set_wait_limit(tries: int) -> int:
    return lib().nrm_set_wait_limit(tries)


def device_fault(clear: bool = True) -> int:
    """Fault bits recorded by kernels on the current device (synchronizes)."""
    v = ctypes.c_uint()
    _check(lib().nrm_device_fault(ctypes.byref(v), 1 if clear else 0), "nrm_device_fault")
    return v.value


def set_bn_group_bytes(nbytes: int) -> int:
    """Input bytes per channel group of the streaming BatchNorm plans (0: default)."""
    return lib().nrm_set_bn_group_bytes(nbytes)


def set_pointer_checks(enable: bool) -> bool:
    return bool(lib().nrm_set_pointer_checks(1 if enable else 0))
