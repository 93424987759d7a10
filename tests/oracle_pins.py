"""Pins for the oracle: facts fixed by the pages and by mathematics, not by the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with the fact.  ``test_oracle_pins.py`` runs them on the
committed oracle; ``test_oracle_mutants.py`` runs them on oracles with a planted
mistake and requires that some pin fails for every mutant.

Independent references used here:
  * closed forms (constant input gives c + ln R; two values give
    max + log1p(exp(-|a - b|)); log_softmax of a constant row is -ln cols);
  * invariants (shift invariance, sum of exp(log_softmax) = 1, bounds
    max <= lse <= max + ln R);
  * brute force in 60-digit decimal arithmetic with no max subtraction;
  * library routines in float64 (torch.logsumexp, torch.log_softmax,
    torch.nn.functional.group_norm / hardswish, numpy population variance).
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

getcontext().prec = 60


def _rng(seed):
    return np.random.default_rng(seed)


def _dec_lse(values) -> float:
    """ln(sum(exp(v))) in 60-digit decimal, no max subtraction."""
    s = sum(Decimal(float(v)).exp() for v in values)
    return float(s.ln())


def _close(a, b, rtol=1e-13, atol=1e-13):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    bad = ~(np.abs(a - b) <= atol + rtol * np.abs(b))
    assert not bad.any(), f"max diff {np.max(np.abs(a - b))} at {np.argwhere(bad)[:5].tolist()}"


# --------------------------------------------------------------------- form 1 (dim-0 / strided)

def pin_lse_constant(orc):
    """constant c over R values: lse = c + ln R (also c = +-1000, where exp overflows)."""
    for R in (1, 2, 3, 4, 7, 32):
        for c in (0.0, 2.5, -7.25, 1000.0, -1000.0, 88.5):
            x = np.full((2, R, 3), c, dtype=np.float32)
            out = orc.lse_reduce(x, 2, R, 3)
            _close(out, np.full((2, 3), c + math.log(R)))


def pin_lse_two_values(orc):
    """lse(a, b) = max(a, b) + log1p(exp(-|a - b|))."""
    pairs = [(0.0, 0.0), (1.0, -1.0), (-3.5, 20.0), (100.0, 99.0), (-50.0, -80.0), (7.0, 7.0)]
    x = np.array([[a for a, _ in pairs], [b for _, b in pairs]], dtype=np.float32)  # (R=2, inner)
    out = orc.lse_reduce(x, 1, 2, len(pairs))[0]
    ref = [max(a, b) + math.log1p(math.exp(-abs(a - b))) for a, b in pairs]
    _close(out, ref)


def pin_lse_bruteforce(orc):
    """x (outer, R, inner) with distinct values: each output is the decimal ln-sum-exp of
    exactly the values x[o, :, i] (catches a wrong stride or a transposed index)."""
    rng = _rng(11)
    for outer, R, inner in ((2, 3, 5), (1, 4, 1), (3, 1, 2), (2, 7, 3)):
        x = rng.uniform(-30, 30, size=(outer, R, inner)).astype(np.float32)
        out = orc.lse_reduce(x, outer, R, inner)
        ref = np.array([[_dec_lse(x[o, :, i]) for i in range(inner)] for o in range(outer)])
        _close(out, ref, rtol=1e-14, atol=1e-14)


def pin_lse_shift(orc):
    """lse(x + k) = lse(x) + k (x on a 1/8 grid so that x + k is exact in fp32)."""
    rng = _rng(12)
    x = (rng.integers(-128, 128, size=(1, 9, 6)) / 8.0).astype(np.float32)
    base = orc.lse_reduce(x, 1, 9, 6)
    for k in (1024.0, -1024.0, 3.0):
        _close(orc.lse_reduce(x + np.float32(k), 1, 9, 6), base + k, rtol=1e-14, atol=1e-12)


def pin_lse_bounds(orc):
    """max <= lse <= max + ln R."""
    rng = _rng(13)
    x = rng.normal(0, 5, size=(3, 17, 11)).astype(np.float32)
    out = orc.lse_reduce(x, 3, 17, 11)
    mx = x.astype(np.float64).max(axis=1)
    assert np.all(out >= mx) and np.all(out <= mx + math.log(17) + 1e-12)


def pin_lse_torch(orc):
    """agrees with torch.logsumexp in float64 (a library routine) on random shapes."""
    rng = _rng(14)
    for shape in ((4, 10, 32), (5, 3, 7), (33, 2, 9), (1, 6, 4)):
        x = rng.normal(0, 3, size=shape).astype(np.float32)
        ref = torch.logsumexp(torch.from_numpy(x).double(), dim=0).numpy()
        _close(orc.logsumexp_dim0(x), ref, rtol=1e-13, atol=1e-13)


def pin_lse_special(orc):
    """NaN wins, then +inf, then an all -inf set gives -inf; -inf entries add nothing."""
    inf, nan = float("inf"), float("nan")
    cols = [
        ([1.0, nan, 2.0], nan),
        ([nan, inf, 0.0], nan),
        ([inf, 1.0, -inf], inf),
        ([-inf, -inf, -inf], -inf),
        ([-inf, 0.0, -inf], 0.0),
        ([-inf, 1.0, 2.0], 2.0 + math.log1p(math.exp(-1.0))),
    ]
    x = np.array([c for c, _ in cols], dtype=np.float32).T.copy()  # (R=3, inner)
    out = orc.lse_reduce(x, 1, 3, len(cols))[0]
    for got, (_, want) in zip(out, cols):
        if math.isnan(want):
            assert math.isnan(got), got
        elif math.isinf(want):
            assert got == want, (got, want)
        else:
            assert abs(got - want) <= 1e-14, (got, want)


# --------------------------------------------------------------------- form 2 (log_softmax)

def pin_lsm_constant(orc):
    """a constant row gives -ln cols everywhere."""
    for cols in (1, 2, 5, 4096):
        x = np.full((3, cols), -2.75, dtype=np.float32)
        _close(orc.log_softmax(x), np.full((3, cols), -math.log(cols)), atol=1e-12)


def pin_lsm_normalised(orc):
    """sum_j exp(out_j) = 1 and out_j - out_k = x_j - x_k."""
    rng = _rng(21)
    x = rng.normal(0, 2, size=(4, 257)).astype(np.float32)
    out = orc.log_softmax(x)
    _close(np.exp(out).sum(axis=1), np.ones(4), atol=1e-12)
    d = x.astype(np.float64) - out
    _close(d - d[:, :1], np.zeros_like(d), atol=1e-12)


def pin_lsm_bruteforce(orc):
    """tiny rows against decimal arithmetic with no max subtraction."""
    rng = _rng(22)
    for rows, cols in ((1, 1), (2, 3), (3, 8), (1, 5)):
        x = rng.uniform(-40, 40, size=(rows, cols)).astype(np.float32)
        out = orc.log_softmax(x)
        ref = np.array([[float(x[r, j]) - _dec_lse(x[r]) for j in range(cols)]
                        for r in range(rows)])
        _close(out, ref, rtol=1e-14, atol=1e-13)
        _close(orc.row_lse(x), [_dec_lse(x[r]) for r in range(rows)], rtol=1e-14, atol=1e-14)


def pin_lsm_torch(orc):
    """agrees with torch.log_softmax in float64 (a library routine)."""
    rng = _rng(23)
    x = rng.normal(0, 2, size=(6, 1000)).astype(np.float32)
    x[rng.random(size=x.shape) < 0.01] = -np.inf
    ref = torch.log_softmax(torch.from_numpy(x).double(), dim=1).numpy()
    out = orc.log_softmax(x)
    finite = np.isfinite(ref)
    _close(out[finite], ref[finite], atol=1e-12)
    assert np.array_equal(np.isneginf(out), np.isneginf(ref))


def pin_lsm_special(orc):
    """-inf entries -> -inf; +inf in a row -> NaN at the +inf, -inf elsewhere;
    NaN in a row -> NaN everywhere; an all -inf row -> NaN everywhere."""
    inf, nan = float("inf"), float("nan")
    x = np.array([[0.0, -inf, 1.0],
                  [inf, 1.0, -inf],
                  [1.0, nan, 2.0],
                  [-inf, -inf, -inf]], dtype=np.float32)
    out = orc.log_softmax(x)
    assert out[0, 1] == -inf
    _close(out[0, [0, 2]], [-math.log1p(math.e), 1.0 - math.log(1 + math.e)], atol=1e-14)
    assert math.isnan(out[1, 0]) and out[1, 1] == -inf and out[1, 2] == -inf
    assert np.isnan(out[2]).all()
    assert np.isnan(out[3]).all()


# --------------------------------------------------------------------- form 3 (GN chain)

def _torch_chain(y, gamma, beta, G, eps):
    """GroupNorm -> tanh -> hardswish -> +y -> logsumexp(dim=1, keepdim) with float64
    library routines."""
    y64 = torch.from_numpy(y).double()
    z = F.group_norm(y64, G, torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(),
                     eps=float(np.float32(eps)))
    r = y64 + F.hardswish(torch.tanh(z))
    return torch.logsumexp(r, dim=1, keepdim=True).numpy()


def pin_gn_torch(orc):
    """agrees with float64 torch group_norm/tanh/hardswish/logsumexp composition for
    several group counts (catches the group assignment, variance kind, eps placement,
    per-channel affine, residual and channel reduction)."""
    rng = _rng(31)
    for (N, C, H, W, G) in ((2, 8, 3, 5, 4), (1, 8, 4, 4, 2), (2, 6, 2, 3, 6), (1, 4, 5, 1, 1),
                            (3, 64, 2, 2, 16)):
        y = rng.normal(0.3, 1.7, size=(N, C, H, W)).astype(np.float32)
        gamma = rng.uniform(0.5, 1.5, size=C).astype(np.float32)
        beta = rng.normal(0, 0.3, size=C).astype(np.float32)
        _close(orc.gn_act_lse(y, gamma, beta, G, 1e-5), _torch_chain(y, gamma, beta, G, 1e-5),
               rtol=1e-12, atol=1e-12)


def pin_gn_stats(orc):
    """(N, G) mean and rstd equal numpy's mean and population variance per group,
    rstd = 1 / sqrt(var + eps)."""
    rng = _rng(32)
    N, C, HW, G, eps = 3, 12, 7, 3, 1e-2
    y = rng.normal(2.0, 3.0, size=(N, C, HW)).astype(np.float32)
    _, mean, rstd = orc.gn_act_lse(y, np.ones(C, np.float32), np.zeros(C, np.float32), G, eps,
                                   return_stats=True)
    grp = y.astype(np.float64).reshape(N, G, -1)
    _close(mean, grp.mean(axis=2), rtol=1e-13, atol=1e-13)
    _close(rstd, 1.0 / np.sqrt(grp.var(axis=2, ddof=0) + float(np.float32(eps))), rtol=1e-12)


def pin_gn_zero_gamma(orc):
    """gamma = 0: the normalised branch is the constant beta_c, so
    out = lse_c(y_c + hardswish(tanh(beta_c))), with hardswish and tanh from torch."""
    rng = _rng(33)
    N, C, HW, G = 2, 8, 5, 4
    y = rng.normal(0, 1, size=(N, C, HW)).astype(np.float32)
    beta = rng.normal(0, 1, size=C).astype(np.float32)
    out = orc.gn_act_lse(y, np.zeros(C, np.float32), beta, G, 1e-5)[:, 0, :]
    h = F.hardswish(torch.tanh(torch.from_numpy(beta).double())).numpy()
    ref = np.array([[_dec_lse(y[n, :, p].astype(np.float64) + h) for p in range(HW)]
                    for n in range(N)])
    _close(out, ref, rtol=1e-13, atol=1e-13)


def pin_gn_single_channel(orc):
    """C = G = 1, HW = 1: variance 0, so z = beta and out = y + hardswish(tanh(beta))."""
    for yv, b in ((0.5, 0.25), (-3.0, -2.0), (10.0, 0.0)):
        y = np.array([[[yv]]], dtype=np.float32)
        out = orc.gn_act_lse(y, np.array([1.3], np.float32), np.array([b], np.float32), 1, 1e-5)
        t = math.tanh(float(np.float32(b)))
        want = float(np.float32(yv)) + t * min(max(t + 3.0, 0.0), 6.0) / 6.0
        _close(out.reshape(-1), [want], atol=1e-14)


# --------------------------------------------------------------------- softmax, other axes, GroupNorm alone

def pin_softmax_normalised(orc):
    """rows sum to 1 and out_j / out_k = exp(x_j - x_k); a constant row gives 1/cols."""
    rng = _rng(41)
    x = rng.normal(0, 3, size=(5, 77)).astype(np.float32)
    out = orc.softmax(x)
    _close(out.sum(axis=1), np.ones(5), atol=1e-13)
    _close(out / out[:, :1], np.exp(x.astype(np.float64) - x[:, :1].astype(np.float64)),
           rtol=1e-12, atol=0)
    _close(orc.softmax(np.full((2, 6), 4.5, np.float32)), np.full((2, 6), 1 / 6), atol=1e-15)


def pin_softmax_torch(orc):
    """agrees with torch.softmax in float64, with -inf entries and an all -inf row."""
    rng = _rng(42)
    x = rng.normal(0, 2, size=(5, 300)).astype(np.float32)
    x[rng.random(size=x.shape) < 0.02] = -np.inf
    x[4, :] = -np.inf
    ref = torch.softmax(torch.from_numpy(x).double(), dim=1).numpy()
    out = orc.softmax(x)
    assert np.array_equal(np.isnan(out), np.isnan(ref))
    fin = ~np.isnan(ref)
    _close(out[fin], ref[fin], atol=1e-14)


def pin_softmax_special(orc):
    """softmax = exp(log_softmax): a row holding +inf gives NaN at the +inf and 0 elsewhere
    (torch's (x - max) / sum gives NaN throughout; the reading follows log_softmax); a NaN
    row gives NaN; -inf entries give exactly 0."""
    inf, nan = float("inf"), float("nan")
    x = np.array([[1.0, inf, 2.0], [1.0, nan, 2.0], [0.0, -inf, 0.0]], dtype=np.float32)
    out = orc.softmax(x)
    assert math.isnan(out[0, 1]) and out[0, 0] == 0.0 and out[0, 2] == 0.0
    assert np.isnan(out[1]).all()
    assert out[2, 1] == 0.0
    _close(out[2, [0, 2]], [0.5, 0.5], atol=1e-15)


def pin_log_softmax_dim_torch(orc):
    """log_softmax over the middle axis agrees with torch.log_softmax(dim=1) in float64."""
    rng = _rng(43)
    for outer, R, inner in ((2, 5, 7), (1, 33, 3), (3, 4, 1), (2, 1, 5)):
        x = rng.normal(0, 4, size=(outer, R, inner)).astype(np.float32)
        ref = torch.log_softmax(torch.from_numpy(x).double(), dim=1).numpy()
        _close(orc.log_softmax_dim(x, outer, R, inner), ref, atol=1e-13)


def pin_log_softmax_dim_bruteforce(orc):
    """each output x[o,r,i] - ln(sum over r' of exp x[o,r',i]) in 60-digit decimal."""
    rng = _rng(44)
    x = rng.uniform(-25, 25, size=(2, 3, 4)).astype(np.float32)
    out = orc.log_softmax_dim(x, 2, 3, 4)
    ref = np.array([[[float(x[o, r, i]) - _dec_lse(x[o, :, i]) for i in range(4)] for r in range(3)]
                    for o in range(2)])
    _close(out, ref, rtol=1e-14, atol=1e-13)


def pin_group_norm_torch(orc):
    """GroupNorm alone agrees with torch.nn.functional.group_norm in float64."""
    rng = _rng(45)
    for (N, C, H, W, G) in ((2, 8, 3, 5, 4), (1, 6, 2, 2, 3), (2, 4, 1, 7, 1), (1, 16, 4, 4, 16)):
        y = rng.normal(1.5, 2.0, size=(N, C, H, W)).astype(np.float32)
        gamma = rng.uniform(0.5, 1.5, size=C).astype(np.float32)
        beta = rng.normal(0, 0.3, size=C).astype(np.float32)
        ref = F.group_norm(torch.from_numpy(y).double(), G, torch.from_numpy(gamma).double(),
                           torch.from_numpy(beta).double(), eps=float(np.float32(1e-5))).numpy()
        _close(orc.group_norm(y, gamma, beta, G, 1e-5), ref, rtol=1e-12, atol=1e-12)


def pin_group_norm_moments(orc):
    """with gamma = 1, beta = 0 every group of the output has mean 0 and population variance
    var / (var + eps), var from numpy."""
    rng = _rng(46)
    N, C, HW, G, eps = 2, 6, 9, 3, 0.5
    y = rng.normal(3, 1.5, size=(N, C, HW)).astype(np.float32)
    out = orc.group_norm(y, np.ones(C, np.float32), np.zeros(C, np.float32), G, eps).reshape(N, G, -1)
    var = y.astype(np.float64).reshape(N, G, -1).var(axis=2)
    _close(out.mean(axis=2), np.zeros((N, G)), atol=1e-13)
    _close(out.var(axis=2), var / (var + eps), rtol=1e-12)


def pin_gn_act_residual_torch(orc):
    """y + hardswish(tanh(GroupNorm(y))) agrees with the float64 torch composition."""
    rng = _rng(47)
    N, C, H, W, G = 2, 8, 3, 4, 2
    y = rng.normal(0, 1, size=(N, C, H, W)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, size=C).astype(np.float32)
    beta = rng.normal(0, 0.3, size=C).astype(np.float32)
    y64 = torch.from_numpy(y).double()
    z = F.group_norm(y64, G, torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(),
                     eps=float(np.float32(1e-5)))
    ref = (y64 + F.hardswish(torch.tanh(z))).numpy()
    _close(orc.gn_act_residual(y, gamma, beta, G, 1e-5), ref, rtol=1e-12, atol=1e-12)


def pin_gn_non_finite(orc):
    """NaN, +inf or -inf in a group makes that group NaN and leaves the others alone, as
    float64 torch.nn.functional.group_norm gives; through the channel lse (which spans
    every group) the whole sample is NaN."""
    rng = _rng(48)
    N, C, H, W, G = 4, 8, 3, 3, 4
    y = rng.normal(0, 1, size=(N, C, H, W)).astype(np.float32)
    y[0, 2, 1, 1] = np.nan       # sample 0, group 1
    y[1, 0, 0, 0] = np.inf       # sample 1, group 0
    y[2, 7, 2, 2] = -np.inf      # sample 2, group 3
    gamma = rng.uniform(0.5, 1.5, size=C).astype(np.float32)
    beta = rng.normal(0, 0.3, size=C).astype(np.float32)
    y64 = torch.from_numpy(y).double()
    z = F.group_norm(y64, G, torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(),
                     eps=float(np.float32(1e-5))).numpy()
    got = np.asarray(orc.group_norm(y, gamma, beta, G, 1e-5), dtype=np.float64).reshape(z.shape)
    assert np.array_equal(np.isnan(got), np.isnan(z))
    assert int(np.isnan(got).sum()) == 3 * 2 * 9
    fin = ~np.isnan(z)
    _close(got[fin], z[fin], rtol=1e-12, atol=1e-12)
    lse = np.asarray(orc.gn_act_lse(y, gamma, beta, G, 1e-5), dtype=np.float64).reshape(N, -1)
    assert np.isnan(lse[:3]).all() and np.isfinite(lse[3]).all()


# --------------------------------------------------------------------- Conv2d and the conv-fed chain

def pin_conv_torch(orc):
    """Valid stride-1 Conv2d with bias agrees with float64 torch.nn.functional.conv2d
    (non-square planes, Cin != Cout, a non-square kernel)."""
    rng = _rng(61)
    x = rng.normal(0, 1, size=(2, 3, 6, 9)).astype(np.float32)
    w = rng.uniform(-0.5, 0.5, size=(5, 3, 3, 2)).astype(np.float32)
    b = rng.normal(0, 1, size=5).astype(np.float32)
    ref = F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                   torch.from_numpy(b).double()).numpy()
    _close(orc.conv2d(x, w, b), ref, rtol=1e-13, atol=1e-13)


def pin_conv_delta(orc):
    """A weight that is 1 at (co, ci, u, v) and 0 elsewhere copies channel ci shifted by
    (u, v) into channel co: y[n, co, i, j] = x[n, ci, i + u, j + v] + b[co]; no other
    channel receives anything but its bias.  Fixes the index order of every operand."""
    rng = _rng(62)
    x = rng.normal(0, 1, size=(2, 3, 5, 7)).astype(np.float32)
    for co, ci, u, v in ((0, 2, 0, 1), (3, 0, 2, 0), (1, 1, 1, 2)):
        w = np.zeros((4, 3, 3, 3), dtype=np.float32)
        w[co, ci, u, v] = 1.0
        b = np.arange(4, dtype=np.float32) * 0.25
        y = orc.conv2d(x, w, b)
        exp = np.broadcast_to(b.astype(np.float64)[None, :, None, None], y.shape).copy()
        exp[:, co] += x[:, ci, u:u + 3, v:v + 5].astype(np.float64)
        _close(y, exp, rtol=0, atol=0)


def pin_conv_constant(orc):
    """Constant input c gives b[co] + c * sum of w[co] at every output pixel."""
    rng = _rng(63)
    w = rng.uniform(-1, 1, size=(4, 2, 3, 3)).astype(np.float32)
    b = rng.normal(0, 1, size=4).astype(np.float32)
    c = 1.75
    x = np.full((1, 2, 4, 6), c, dtype=np.float32)
    y = orc.conv2d(x, w, b)
    exp = b.astype(np.float64) + c * w.astype(np.float64).reshape(4, -1).sum(1)
    _close(y, np.broadcast_to(exp[None, :, None, None], y.shape), rtol=1e-14, atol=1e-14)


def pin_conv_chain_torch(orc):
    """Conv2d -> GroupNorm -> tanh -> hardswish -> + conv output -> logsumexp over channels,
    keepdim, agrees with the float64 torch composition of the same layers."""
    rng = _rng(64)
    N, Cin, H, W, Cout, G = 2, 3, 7, 6, 8, 4
    x = rng.normal(0, 1, size=(N, Cin, H, W)).astype(np.float32)
    w = rng.uniform(-0.3, 0.3, size=(Cout, Cin, 3, 3)).astype(np.float32)
    b = rng.uniform(-0.3, 0.3, size=Cout).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, size=Cout).astype(np.float32)
    beta = rng.normal(0, 0.3, size=Cout).astype(np.float32)
    y = F.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(), torch.from_numpy(b).double())
    z = F.group_norm(y, G, torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(),
                     eps=float(np.float32(1e-5)))
    ref = torch.logsumexp(y + F.hardswish(torch.tanh(z)), dim=1, keepdim=True).numpy()
    _close(orc.conv_gn_act_lse(x, w, b, gamma, beta, G, 1e-5), ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------- stored closed forms

def pin_golden_closed_forms(orc):
    """cases in tests/golden/closed_forms.json: inputs with an expected value written as a
    closed-form expression (evaluated here with the math module)."""
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    env = {k: getattr(math, k) for k in ("log", "exp", "log1p", "tanh", "sqrt")}
    env["hs"] = lambda t: t * min(max(t + 3.0, 0.0), 6.0) / 6.0
    for case in cases:
        x = np.array(case["x"], dtype=np.float32)
        want = np.array([eval(e, {"__builtins__": {}}, env) for e in case["expect"]])
        if case["op"] == "lse_dim0":
            got = orc.logsumexp_dim0(x).reshape(-1)
        elif case["op"] == "log_softmax":
            got = orc.log_softmax(x).reshape(-1)
        elif case["op"] == "gn_act_lse":
            got = orc.gn_act_lse(x, np.array(case["gamma"], np.float32),
                                 np.array(case["beta"], np.float32), case["G"],
                                 case["eps"]).reshape(-1)
        else:
            raise KeyError(case["op"])
        _close(got, want, rtol=1e-13, atol=1e-13)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
