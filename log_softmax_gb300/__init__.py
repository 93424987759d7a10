"""GB300 (sm_103a) logsumexp library: Python binding of liblse.so.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of liblse.so (built from csrc/ by ``log_softmax_gb300.build``); torch
is used for device memory and streams.  There is no CPU fallback: if the
library is missing or the device is not supported, calls raise.

C-ABI entry points (declared in include/lse.h), same names here:
    lse_reduce(x, out, outer, R, inner, stream=None)
    log_softmax_lastdim(x, out, rows, cols, stream=None)
    log_softmax_lastdim_host(x, out, rows, cols, stream=None)   (host tensors)
    softmax_lastdim(x, out, rows, cols, stream=None)
    log_softmax_dim(x, out, outer, R, inner, stream=None)
    gn_act_lse(y, gamma, beta, out, N, C, HW, G, eps, stream=None)
    gn_act_lse_noalloc(y, gamma, beta, out, N, C, HW, G, eps, stream=None)
    group_norm(y, gamma, beta, out, N, C, HW, G, eps, stream=None)
    gn_act_residual(y, gamma, beta, out, N, C, HW, G, eps, stream=None)
    conv2d_3x3(x, w, b, y, N, Cin, H, W, Cout, stream=None)
    conv_gn_act_lse(x, w, b, gamma, beta, out, N, Cin, H, W, Cout, G, eps, stream=None)
Conveniences that allocate the output with torch:
    logsumexp(x, dim=0), log_softmax(x, dim=-1), softmax(x),
    gn_act_lse_forward(y, gamma, beta, G, eps), group_norm_forward(...),
    gn_act_residual_forward(...), conv2d_3x3_forward(x, w, b),
    conv_gn_act_lse_forward(x, w, b, gamma, beta, G, eps)
Given host (CPU) tensors, a convenience returns a host result after synchronising,
and raises LseError(LSE_ERR_TIMEOUT) if a bounded wait in a kernel gave up on the
device; given CUDA tensors it returns at once and lse_device_status() reports.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblse.so")

STATUS = {
    0: "LSE_OK", 1: "LSE_ERR_NULL", 2: "LSE_ERR_SIZE", 3: "LSE_ERR_ALIGN", 4: "LSE_ERR_CUDA",
    5: "LSE_ERR_UNSUPPORTED", 6: "LSE_ERR_VALUE", 7: "LSE_ERR_TIMEOUT",
}

EXPORTS = ("lse_reduce", "log_softmax_lastdim", "log_softmax_lastdim_host", "softmax_lastdim",
           "log_softmax_dim", "gn_act_lse", "gn_act_lse_noalloc", "group_norm", "gn_act_residual",
           "conv2d_3x3", "conv_gn_act_lse",
           "lse_release_workspace", "lse_device_status", "lse_status_string", "lse_last_cuda_error",
           "lse_version")


class LseError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{fn} failed: {name}{(' (' + detail + ')') if detail else ''}")


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads liblse.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m log_softmax_gb300.build` "
            "(the library has no CPU fallback)")
    lib = ctypes.CDLL(path)
    i64, vp, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    lib.lse_reduce.argtypes = [vp, vp, i64, i64, i64, vp]
    lib.log_softmax_lastdim.argtypes = [vp, vp, i64, i64, vp]
    lib.log_softmax_lastdim_host.argtypes = [vp, vp, i64, i64, vp]
    lib.log_softmax_lastdim_host.restype = ctypes.c_int
    lib.softmax_lastdim.argtypes = [vp, vp, i64, i64, vp]
    lib.log_softmax_dim.argtypes = [vp, vp, i64, i64, i64, vp]
    lib.gn_act_lse.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, vp]
    lib.conv2d_3x3.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp]
    lib.conv_gn_act_lse.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp]
    lib.group_norm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, vp]
    lib.gn_act_residual.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, vp]
    lib.gn_act_lse_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, vp]
    lib.gn_act_lse_noalloc.restype = ctypes.c_int
    lib.lse_release_workspace.argtypes = []
    lib.lse_device_status.argtypes = [vp]
    lib.lse_status_string.argtypes = [ctypes.c_int]
    lib.lse_status_string.restype = ctypes.c_char_p
    lib.lse_last_cuda_error.argtypes = []
    lib.lse_version.argtypes = []
    for name in ("lse_reduce", "log_softmax_lastdim", "softmax_lastdim", "log_softmax_dim",
                 "gn_act_lse", "group_norm", "gn_act_residual", "conv2d_3x3", "conv_gn_act_lse",
                 "lse_release_workspace",
                 "lse_device_status", "lse_last_cuda_error", "lse_version"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(t):
    """Device address of a tensor (or None / int passed through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t)}")
    if t.numel() > 0 and not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if t.numel() > 0 and t.dtype != torch.float32:
        raise TypeError(f"tensor must be float32, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _device_of(t):
    """Makes the tensor's device current for the call (the library works on the
    current device); a no-op for anything that is not a CUDA tensor."""
    if isinstance(t, torch.Tensor) and t.is_cuda:
        return torch.cuda.device(t.device)
    return contextlib.nullcontext()


def _stream(stream, like=None):
    if stream is None:
        dev = like.device if isinstance(like, torch.Tensor) and like.is_cuda else None
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, rc: int):
    if rc != 0:
        lib = load_library()
        detail = ""
        if rc == 4:
            detail = f"cudaError {lib.lse_last_cuda_error()}"
        raise LseError(fn, rc, detail)


# ----------------------------------------------------------------- C-ABI, same names

def lse_reduce(x, out, outer: int, R: int, inner: int, stream=None) -> None:
    """out[o, i] = logsumexp over r of x[o, r, i]; x (outer, R, inner), out (outer, inner)."""
    lib = load_library()
    with _device_of(x):
        rc = lib.lse_reduce(_ptr(x), _ptr(out), int(outer), int(R), int(inner), _stream(stream, x))
    _check("lse_reduce", rc)


def log_softmax_lastdim(x, out, rows: int, cols: int, stream=None) -> None:
    """out[r, j] = x[r, j] - logsumexp_k x[r, k] over a contiguous (rows, cols) tensor."""
    lib = load_library()
    with _device_of(x):
        rc = lib.log_softmax_lastdim(_ptr(x), _ptr(out), int(rows), int(cols), _stream(stream, x))
    _check("log_softmax_lastdim", rc)


def softmax_lastdim(x, out, rows: int, cols: int, stream=None) -> None:
    """out[r, j] = exp(x[r, j] - logsumexp_k x[r, k]) over a contiguous (rows, cols) tensor."""
    lib = load_library()
    with _device_of(x):
        rc = lib.softmax_lastdim(_ptr(x), _ptr(out), int(rows), int(cols), _stream(stream, x))
    _check("softmax_lastdim", rc)


def log_softmax_dim(x, out, outer: int, R: int, inner: int, stream=None) -> None:
    """out[o, r, i] = x[o, r, i] - logsumexp over r' of x[o, r', i]; x and out (outer, R, inner)."""
    lib = load_library()
    with _device_of(x):
        rc = lib.log_softmax_dim(_ptr(x), _ptr(out), int(outer), int(R), int(inner),
                                 _stream(stream, x))
    _check("log_softmax_dim", rc)


def _host_ptr(t):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("expected a CPU tensor")
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError("tensor must be contiguous float32")
    return t.data_ptr() if t.numel() > 0 else None


def log_softmax_lastdim_host(x, out, rows: int, cols: int, stream=None) -> None:
    """log_softmax_lastdim on host (CPU) tensors, pipelined through the device; `out`
    is complete once `stream` (default: the current stream) is."""
    lib = load_library()
    rc = lib.log_softmax_lastdim_host(_host_ptr(x), _host_ptr(out), int(rows), int(cols),
                                      _stream(stream))
    _check("log_softmax_lastdim_host", rc)


def gn_act_lse(y, gamma, beta, out, N: int, C: int, HW: int, G: int, eps: float,
               stream=None) -> None:
    """GroupNorm -> tanh -> hardswish -> +y -> logsumexp over channels; out is [N, HW]."""
    lib = load_library()
    with _device_of(y):
        rc = lib.gn_act_lse(_ptr(y), _ptr(gamma), _ptr(beta), _ptr(out), int(N), int(C), int(HW),
                            int(G), float(eps), _stream(stream, y))
    _check("gn_act_lse", rc)


def group_norm(y, gamma, beta, out, N: int, C: int, HW: int, G: int, eps: float,
               stream=None) -> None:
    """GroupNorm forward with per-channel affine; out has y's shape [N, C, HW]."""
    lib = load_library()
    with _device_of(y):
        rc = lib.group_norm(_ptr(y), _ptr(gamma), _ptr(beta), _ptr(out), int(N), int(C), int(HW),
                            int(G), float(eps), _stream(stream, y))
    _check("group_norm", rc)


def gn_act_residual(y, gamma, beta, out, N: int, C: int, HW: int, G: int, eps: float,
                    stream=None) -> None:
    """y + hardswish(tanh(GroupNorm(y))); out has y's shape [N, C, HW]."""
    lib = load_library()
    with _device_of(y):
        rc = lib.gn_act_residual(_ptr(y), _ptr(gamma), _ptr(beta), _ptr(out), int(N), int(C),
                                 int(HW), int(G), float(eps), _stream(stream, y))
    _check("gn_act_residual", rc)


def conv2d_3x3(x, w, b, y, N: int, Cin: int, H: int, W: int, Cout: int, stream=None) -> None:
    """Conv2d 3x3, stride 1, no padding, with bias: x [N,Cin,H,W] -> y [N,Cout,H-2,W-2]."""
    lib = load_library()
    with _device_of(x):
        rc = lib.conv2d_3x3(_ptr(x), _ptr(w), _ptr(b), _ptr(y), int(N), int(Cin), int(H), int(W), int(Cout),
                            _stream(stream, x))
    _check("conv2d_3x3", rc)


def conv_gn_act_lse(x, w, b, gamma, beta, out, N: int, Cin: int, H: int, W: int, Cout: int, G: int,
                    eps: float, stream=None) -> None:
    """Conv2d 3x3 (valid, bias) -> GroupNorm -> tanh -> hardswish -> + conv output ->
    logsumexp over channels; out is [N, H-2, W-2]."""
    lib = load_library()
    with _device_of(x):
        rc = lib.conv_gn_act_lse(_ptr(x), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta), _ptr(out), int(N), int(Cin),
                                 int(H), int(W), int(Cout), int(G), float(eps), _stream(stream, x))
    _check("conv_gn_act_lse", rc)


def gn_act_lse_noalloc(y, gamma, beta, out, N: int, C: int, HW: int, G: int, eps: float,
                       stream=None) -> None:
    """gn_act_lse for callers that must not allocate device memory: the statistics
    use a fixed array inside the library (N*G <= 65536; calls on one device share it,
    so calls that may overlap on the GPU must be ordered)."""
    lib = load_library()
    with _device_of(y):
        rc = lib.gn_act_lse_noalloc(_ptr(y), _ptr(gamma), _ptr(beta), _ptr(out), int(N), int(C),
                                    int(HW), int(G), float(eps), _stream(stream, y))
    _check("gn_act_lse_noalloc", rc)


def lse_release_workspace() -> None:
    _check("lse_release_workspace", load_library().lse_release_workspace())


def lse_device_status(stream=None) -> int:
    """Synchronises the stream; returns the library's device status code and clears it."""
    return load_library().lse_device_status(_stream(stream))


def lse_status_string(status: int) -> str:
    return load_library().lse_status_string(int(status)).decode()


def lse_version() -> int:
    return load_library().lse_version()


def lse_last_cuda_error() -> int:
    """cudaError_t of the last LSE_ERR_CUDA on this thread (0 if none)."""
    return load_library().lse_last_cuda_error()


# ----------------------------------------------------------------- conveniences

def _to_device(t: torch.Tensor, device):
    if t.is_cuda:
        return t.contiguous(), False
    return t.contiguous().to(device, non_blocking=True), True


def _raise_on_device_timeout(fn: str, stream) -> None:
    """After a synchronisation: reads (and clears) the library's device status and
    raises LseError(LSE_ERR_TIMEOUT) when a bounded wait in a kernel gave up, since
    that call's outputs are then unspecified.  The status word is per device, so a
    timeout of another call on the same device that completed meanwhile is
    reported here too."""
    rc = load_library().lse_device_status(stream)
    if rc != 0:
        raise LseError(fn, rc, "a kernel's bounded wait gave up; the outputs are unspecified"
                       if rc == 7 else "")


def _result(dev_out: torch.Tensor, was_host: bool, out, fn: str = "call"):
    """Returns the device result, or copies it to host memory (`out` if given, else
    a new pinned tensor) when the input came from the host.  The host path
    synchronises, so it also checks the device status (see _raise_on_device_timeout);
    a device result is returned while the call may still run, unchecked."""
    if not was_host:
        return dev_out
    host = out if out is not None else torch.empty(dev_out.shape, dtype=dev_out.dtype,
                                                   pin_memory=True)
    stream = torch.cuda.current_stream(dev_out.device)
    host.copy_(dev_out.view(host.shape), non_blocking=True)
    stream.synchronize()
    with torch.cuda.device(dev_out.device):
        _raise_on_device_timeout(fn, stream.cuda_stream)
    return host


def _device_out(shape, xd: torch.Tensor, was_host: bool, out):
    if out is not None and not was_host:
        if tuple(out.shape) != tuple(shape) or not out.is_cuda:
            raise ValueError(f"out must be a CUDA tensor of shape {tuple(shape)}")
        return out
    return torch.empty(shape, dtype=torch.float32, device=xd.device)


def logsumexp(x: torch.Tensor, dim: int = 0, keepdim: bool = False, out=None,
              device="cuda") -> torch.Tensor:
    """torch.logsumexp(x, dim) for fp32 x.  A CPU tensor (pinned, for an asynchronous
    copy) is copied to `device`, reduced there, and the result copied back to host
    memory (`out` if given)."""
    xd, host = _to_device(x, device)
    dim = dim % xd.ndim if xd.ndim else 0
    shape = list(xd.shape)
    outer = 1
    for s in shape[:dim]:
        outer *= s
    R = shape[dim] if shape else 1
    inner = 1
    for s in shape[dim + 1:]:
        inner *= s
    out_shape = shape[:dim] + ([1] if keepdim else []) + shape[dim + 1:]
    res = _device_out(out_shape, xd, host, out)
    lse_reduce(xd, res, outer, R, inner)
    return _result(res, host, out, "logsumexp")


def _split(shape, dim):
    """(outer, R, inner) of a contiguous tensor of `shape` around axis `dim`."""
    outer = 1
    for s in shape[:dim]:
        outer *= s
    inner = 1
    for s in shape[dim + 1:]:
        inner *= s
    return outer, (shape[dim] if shape else 1), inner


def log_softmax(x: torch.Tensor, out=None, device="cuda", *, dim: int = -1) -> torch.Tensor:
    """log_softmax of fp32 x over axis `dim` (default the last).  CPU input is copied
    to `device` and the result back to host memory (`out` if given); for the last
    axis the copies are pipelined with the computation by the library."""
    if x.ndim and dim % x.ndim != x.ndim - 1:
        xd, host = _to_device(x, device)
        outer, R, inner = _split(list(xd.shape), dim % xd.ndim)
        res = _device_out(xd.shape, xd, host, out)
        log_softmax_dim(xd, res, outer, R, inner)
        return _result(res, host, out, "log_softmax")
    if not x.is_cuda:
        # host in, host out: the library pipelines chunks through the device
        xh = x.contiguous()
        cols = xh.shape[-1] if xh.ndim else 1
        rows = xh.numel() // cols if cols else 0
        oh = out if out is not None else torch.empty(xh.shape, dtype=torch.float32,
                                                     pin_memory=xh.is_pinned())
        with torch.cuda.device(torch.device(device)):
            stream = torch.cuda.current_stream()
            log_softmax_lastdim_host(xh, oh, rows, cols, stream=stream)
            stream.synchronize()
            _raise_on_device_timeout("log_softmax", stream.cuda_stream)
        return oh
    xd, host = _to_device(x, device)
    cols = xd.shape[-1] if xd.ndim else 1
    rows = xd.numel() // cols if cols else 0
    res = _device_out(xd.shape, xd, host, out)
    log_softmax_lastdim(xd, res, rows, cols)
    return _result(res, host, out, "log_softmax")


def softmax(x: torch.Tensor, out=None, device="cuda") -> torch.Tensor:
    """softmax over the last axis of fp32 x (any leading shape), as exp(x - logsumexp)."""
    xd, host = _to_device(x, device)
    cols = xd.shape[-1] if xd.ndim else 1
    rows = xd.numel() // cols if cols else 0
    res = _device_out(xd.shape, xd, host, out)
    softmax_lastdim(xd, res, rows, cols)
    return _result(res, host, out, "softmax")


def _gn_call(fn, y, gamma, beta, G, eps, out, device):
    yd, host = _to_device(y, device)
    gd, _ = _to_device(gamma, yd.device)
    bd, _ = _to_device(beta, yd.device)
    N, C = yd.shape[0], yd.shape[1]
    HW = 1
    for s in yd.shape[2:]:
        HW *= s
    res = _device_out(yd.shape, yd, host, out)
    fn(yd, gd, bd, res, N, C, HW, G, eps)
    return _result(res, host, out, fn.__name__)


def group_norm_forward(y: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, G: int,
                       eps: float = 1e-5, out=None, device="cuda") -> torch.Tensor:
    """GroupNorm(G, eps) with affine gamma/beta of y [N, C, *spatial]; same shape out."""
    return _gn_call(group_norm, y, gamma, beta, G, eps, out, device)


def gn_act_residual_forward(y: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, G: int,
                            eps: float = 1e-5, out=None, device="cuda") -> torch.Tensor:
    """y + hardswish(tanh(GroupNorm(y))) for y [N, C, *spatial]; same shape out."""
    return _gn_call(gn_act_residual, y, gamma, beta, G, eps, out, device)


def conv2d_3x3_forward(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor, out=None,
                       device="cuda") -> torch.Tensor:
    """Conv2d(Cin, Cout, 3) (stride 1, no padding, bias) of x [N, Cin, H, W]."""
    xd, host = _to_device(x, device)
    wd, _ = _to_device(w, xd.device)
    bd, _ = _to_device(b, xd.device)
    N, Cin, H, W = xd.shape
    Cout = wd.shape[0]
    res = _device_out((N, Cout, H - 2, W - 2), xd, host, out)
    conv2d_3x3(xd, wd, bd, res, N, Cin, H, W, Cout)
    return _result(res, host, out, "conv2d_3x3_forward")


def conv_gn_act_lse_forward(x: torch.Tensor, w: torch.Tensor, b: torch.Tensor, gamma: torch.Tensor,
                            beta: torch.Tensor, G: int, eps: float = 1e-5, out=None,
                            device="cuda") -> torch.Tensor:
    """The chain from the convolution's input x [N, Cin, H, W]; returns [N, 1, H-2, W-2]."""
    xd, host = _to_device(x, device)
    wd, bd, gd, betad = (_to_device(t, xd.device)[0] for t in (w, b, gamma, beta))
    N, Cin, H, W = xd.shape
    res = _device_out((N, 1, H - 2, W - 2), xd, host, out)
    conv_gn_act_lse(xd, wd, bd, gd, betad, res, N, Cin, H, W, wd.shape[0], G, eps)
    return _result(res, host, out, "conv_gn_act_lse_forward")


def gn_act_lse_forward(y: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, G: int,
                       eps: float = 1e-5, out=None, device="cuda") -> torch.Tensor:
    """GroupNorm(G, eps, affine gamma/beta) -> tanh -> hardswish -> +y -> logsumexp over
    dim 1 with keepdim, for y of shape [N, C, *spatial]; returns [N, 1, *spatial]."""
    yd, host = _to_device(y, device)
    gd, _ = _to_device(gamma, yd.device)
    bd, _ = _to_device(beta, yd.device)
    N, C = yd.shape[0], yd.shape[1]
    spatial = list(yd.shape[2:])
    HW = 1
    for s in spatial:
        HW *= s
    res = _device_out([N, 1] + spatial, yd, host, out)
    gn_act_lse(yd, gd, bd, res, N, C, HW, G, eps)
    return _result(res, host, out, "gn_act_lse_forward")
