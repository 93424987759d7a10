"""Oracle for the logsumexp hot path (test infrastructure only).

A plain C implementation in double precision (``lse_oracle.c``) behind ctypes.
Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package; the product library never does.

Each function takes fp32 numpy arrays (or CPU torch tensors) and returns float64
numpy arrays.  See ``lse_oracle.c`` for the passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "lse_oracle.c")
_LIB = os.path.join(_HERE, "liblse_oracle.so")
_lock = threading.Lock()
_default = None

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]


def compile_oracle(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library (IEEE double, no fast-math)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle unless an up-to-date build exists."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, _LIB)
    return _LIB


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().cpu().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle takes float32 inputs, got {a.dtype}")
    return a


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class Oracle:
    """One loaded oracle library (the committed one, or a test's planted mutant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_lse_reduce.argtypes = [vp, vp, i64, i64, i64]
        lib.oracle_log_softmax.argtypes = [vp, vp, i64, i64]
        lib.oracle_row_lse.argtypes = [vp, vp, i64, i64]
        lib.oracle_gn_act_lse.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64,
                                          ctypes.c_double, vp, vp]
        lib.oracle_softmax.argtypes = [vp, vp, i64, i64]
        lib.oracle_log_softmax_dim.argtypes = [vp, vp, i64, i64, i64]
        for name in ("oracle_group_norm", "oracle_gn_act_residual"):
            getattr(lib, name).argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_double]
        lib.oracle_conv2d.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64]
        lib.oracle_conv_gn_act_lse.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                               ctypes.c_double]
        for f in (lib.oracle_lse_reduce, lib.oracle_log_softmax, lib.oracle_row_lse,
                  lib.oracle_gn_act_lse, lib.oracle_softmax, lib.oracle_log_softmax_dim,
                  lib.oracle_group_norm, lib.oracle_gn_act_residual, lib.oracle_conv2d,
                  lib.oracle_conv_gn_act_lse):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def lse_reduce(self, x, outer: int, R: int, inner: int) -> np.ndarray:
        """logsumexp over the middle axis of x viewed as (outer, R, inner) -> (outer, inner)."""
        x = _f32(x)
        assert x.size == outer * R * inner
        out = np.empty((outer, inner), dtype=np.float64)
        rc = self.lib.oracle_lse_reduce(_p(x), _p(out), outer, R, inner)
        if rc != 0:
            raise ValueError(f"oracle_lse_reduce rejected its arguments (rc={rc})")
        return out

    def logsumexp_dim0(self, x) -> np.ndarray:
        """logsumexp over dim 0 of an N-d tensor (the (R, B, D) form) -> shape x.shape[1:]."""
        x = _f32(x)
        R = x.shape[0]
        inner = int(np.prod(x.shape[1:])) if x.ndim > 1 else 1
        return self.lse_reduce(x, 1, R, inner).reshape(x.shape[1:])

    def log_softmax(self, x) -> np.ndarray:
        """log_softmax over the last axis of a 2-d (rows, cols) array."""
        x = _f32(x)
        rows, cols = x.shape
        out = np.empty((rows, cols), dtype=np.float64)
        rc = self.lib.oracle_log_softmax(_p(x), _p(out), rows, cols)
        if rc != 0:
            raise ValueError(f"oracle_log_softmax rejected its arguments (rc={rc})")
        return out

    def row_lse(self, x) -> np.ndarray:
        """logsumexp of each row of a 2-d (rows, cols) array."""
        x = _f32(x)
        rows, cols = x.shape
        out = np.empty((rows,), dtype=np.float64)
        rc = self.lib.oracle_row_lse(_p(x), _p(out), rows, cols)
        if rc != 0:
            raise ValueError(f"oracle_row_lse rejected its arguments (rc={rc})")
        return out

    def gn_act_lse(self, y, gamma, beta, G: int, eps: float = 1e-5, return_stats: bool = False):
        """GroupNorm -> tanh -> hardswish -> +y -> logsumexp over channels.

        y is (N, C, H, W) or (N, C, HW); returns (N, 1, *spatial) in float64, and with
        return_stats also the (N, G) mean and rstd.  eps is rounded to fp32 first, as
        the CUDA path receives it."""
        y = _f32(y)
        gamma = _f32(gamma)
        beta = _f32(beta)
        N, C = y.shape[0], y.shape[1]
        spatial = y.shape[2:]
        HW = int(np.prod(spatial)) if len(spatial) else 1
        assert gamma.size == C and beta.size == C
        out = np.empty((N, HW), dtype=np.float64)
        mean = np.empty((N, G), dtype=np.float64)
        rstd = np.empty((N, G), dtype=np.float64)
        rc = self.lib.oracle_gn_act_lse(_p(y), _p(gamma), _p(beta), _p(out), N, C, HW, G,
                                        float(np.float32(eps)), _p(mean), _p(rstd))
        if rc != 0:
            raise ValueError(f"oracle_gn_act_lse rejected its arguments (rc={rc})")
        out = out.reshape((N, 1) + tuple(spatial))
        if return_stats:
            return out, mean, rstd
        return out


    def softmax(self, x) -> np.ndarray:
        """softmax over the last axis of a 2-d (rows, cols) array."""
        x = _f32(x)
        rows, cols = x.shape
        out = np.empty((rows, cols), dtype=np.float64)
        rc = self.lib.oracle_softmax(_p(x), _p(out), rows, cols)
        if rc != 0:
            raise ValueError(f"oracle_softmax rejected its arguments (rc={rc})")
        return out

    def log_softmax_dim(self, x, outer: int, R: int, inner: int) -> np.ndarray:
        """log_softmax over the middle axis of x viewed as (outer, R, inner)."""
        x = _f32(x)
        assert x.size == outer * R * inner
        out = np.empty((outer, R, inner), dtype=np.float64)
        rc = self.lib.oracle_log_softmax_dim(_p(x), _p(out), outer, R, inner)
        if rc != 0:
            raise ValueError(f"oracle_log_softmax_dim rejected its arguments (rc={rc})")
        return out

    def _gn_elementwise(self, fn, y, gamma, beta, G, eps):
        y = _f32(y)
        gamma = _f32(gamma)
        beta = _f32(beta)
        N, C = y.shape[0], y.shape[1]
        HW = int(np.prod(y.shape[2:])) if y.ndim > 2 else 1
        out = np.empty(y.shape, dtype=np.float64)
        rc = fn(_p(y), _p(gamma), _p(beta), _p(out), N, C, HW, G, float(np.float32(eps)))
        if rc != 0:
            raise ValueError(f"oracle rejected its arguments (rc={rc})")
        return out

    def group_norm(self, y, gamma, beta, G: int, eps: float = 1e-5) -> np.ndarray:
        """GroupNorm with per-channel affine, y of shape (N, C, *spatial)."""
        return self._gn_elementwise(self.lib.oracle_group_norm, y, gamma, beta, G, eps)

    def gn_act_residual(self, y, gamma, beta, G: int, eps: float = 1e-5) -> np.ndarray:
        """y + hardswish(tanh(GroupNorm(y))), y of shape (N, C, *spatial)."""
        return self._gn_elementwise(self.lib.oracle_gn_act_residual, y, gamma, beta, G, eps)


    def conv2d(self, x, w, b) -> np.ndarray:
        """Valid stride-1 Conv2d with bias: x [N, Cin, H, W], w [Cout, Cin, KH, KW], b [Cout]."""
        x, w, b = _f32(x), _f32(w), _f32(b)
        N, Cin, H, W = x.shape
        Cout, Cin2, KH, KW = w.shape
        assert Cin2 == Cin and b.size == Cout
        out = np.empty((N, Cout, H - KH + 1, W - KW + 1), dtype=np.float64)
        rc = self.lib.oracle_conv2d(_p(x), _p(w), _p(b), _p(out), N, Cin, H, W, Cout, KH, KW)
        if rc != 0:
            raise ValueError(f"oracle_conv2d rejected its arguments (rc={rc})")
        return out

    def conv_gn_act_lse(self, x, w, b, gamma, beta, G: int, eps: float = 1e-5) -> np.ndarray:
        """Conv2d 3x3 (valid, bias) -> GroupNorm -> tanh -> hardswish -> +y -> channel
        logsumexp (keepdim): [N, 1, H - 2, W - 2]."""
        x, w, b, gamma, beta = _f32(x), _f32(w), _f32(b), _f32(gamma), _f32(beta)
        N, Cin, H, W = x.shape
        Cout = w.shape[0]
        assert w.shape == (Cout, Cin, 3, 3) and b.size == Cout and gamma.size == Cout and beta.size == Cout
        out = np.empty((N, 1, H - 2, W - 2), dtype=np.float64)
        rc = self.lib.oracle_conv_gn_act_lse(_p(x), _p(w), _p(b), _p(gamma), _p(beta), _p(out), N, Cin,
                                             H, W, Cout, G, float(np.float32(eps)))
        if rc != 0:
            raise ValueError(f"oracle_conv_gn_act_lse rejected its arguments (rc={rc})")
        return out


def default() -> Oracle:
    """The committed oracle, compiled on first use."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def lse_reduce(x, outer: int, R: int, inner: int) -> np.ndarray:
    return default().lse_reduce(x, outer, R, inner)


def logsumexp_dim0(x) -> np.ndarray:
    return default().logsumexp_dim0(x)


def log_softmax(x) -> np.ndarray:
    return default().log_softmax(x)


def row_lse(x) -> np.ndarray:
    return default().row_lse(x)


def gn_act_lse(y, gamma, beta, G: int, eps: float = 1e-5, return_stats: bool = False):
    return default().gn_act_lse(y, gamma, beta, G, eps, return_stats)


def softmax(x) -> np.ndarray:
    return default().softmax(x)


def log_softmax_dim(x, outer: int, R: int, inner: int) -> np.ndarray:
    return default().log_softmax_dim(x, outer, R, inner)


def group_norm(y, gamma, beta, G: int, eps: float = 1e-5) -> np.ndarray:
    return default().group_norm(y, gamma, beta, G, eps)


def gn_act_residual(y, gamma, beta, G: int, eps: float = 1e-5) -> np.ndarray:
    return default().gn_act_residual(y, gamma, beta, G, eps)


def conv2d(x, w, b) -> np.ndarray:
    return default().conv2d(x, w, b)


def conv_gn_act_lse(x, w, b, gamma, beta, G: int, eps: float = 1e-5) -> np.ndarray:
    return default().conv_gn_act_lse(x, w, b, gamma, beta, G, eps)
