"""softmax_lastdim, log_softmax_dim, group_norm and gn_act_residual against the
oracle, element by element, through the C ABI (GPU only).

Same bar and the same kind of cases as the three forms: several tiles and a
ragged tail, every kernel the dispatch can pick, unaligned addresses and the
special values.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def lib():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300 as L
    L.load_library()
    torch.cuda.set_device(0)
    yield L
    assert L.lse_device_status() == 0


@pytest.fixture
def env(monkeypatch):
    return monkeypatch


def _misaligned(t: torch.Tensor) -> torch.Tensor:
    buf = torch.empty(t.numel() + 1, dtype=torch.float32, device=DEV)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _softmax(L, x_cpu, misalign=False):
    rows, cols = x_cpu.shape
    x = x_cpu.to(DEV)
    out = torch.full((rows, cols), float("nan"), device=DEV)
    if misalign:
        x, out = _misaligned(x), _misaligned(out)
    L.softmax_lastdim(x, out, rows, cols)
    torch.cuda.synchronize()
    return out.cpu()


def _lsm_dim(L, x_cpu, outer, R, inner, misalign=False):
    x = x_cpu.reshape(outer, R, inner).to(DEV)
    out = torch.full((outer, R, inner), float("nan"), device=DEV)
    if misalign:
        x, out = _misaligned(x), _misaligned(out)
    L.log_softmax_dim(x, out, outer, R, inner)
    torch.cuda.synchronize()
    return out.cpu()


# ----------------------------------------------------------------------------- softmax

SM_COLS = [1, 3, 4, 33, 1000, 4097, 16384, 16385, 32768, 32772, 70001, 393216]


@pytest.mark.parametrize("cols", SM_COLS)
def test_softmax_parity(lib, cols):
    rows = max(2, min(37, 2_000_000 // cols))
    x = synth.normal((rows, cols), seed=cols + 100, var=4.0)
    x.masked_fill_(synth.bernoulli_mask((rows, cols), seed=cols + 101, p=0.01), float("-inf"))
    x[:, 0] = 0.5
    assert_parity(_softmax(lib, x), oracle.softmax(x), f"softmax cols={cols}")


@pytest.mark.parametrize("variant", ["1", "3", "6", "7", "8", "2", "4", "5"])
def test_softmax_variants(lib, env, variant):
    """Registers, streaming and warp-specialised kernels (whole-slice buffers or a ring
    of chunk slots); the variants without a softmax output fall back to the default
    choice."""
    env.setenv("LSE_LSM_VARIANT", variant)
    for rows, cols in ((7, 4096), (5, 393216), (3, 100003)):
        x = synth.normal((rows, cols), seed=rows * cols, var=9.0)
        assert_parity(_softmax(lib, x), oracle.softmax(x), f"softmax v{variant} {rows}x{cols}")


@pytest.mark.parametrize("cols", [5, 129, 4097, 70001])
def test_softmax_misaligned(lib, cols):
    x = synth.normal((9, cols), seed=cols + 7)
    assert_parity(_softmax(lib, x, misalign=True), oracle.softmax(x), f"softmax misaligned {cols}")


def test_softmax_special_rows(lib):
    inf, nan = float("inf"), float("nan")
    for cols in (8, 4096, 40000, 393216):
        x = synth.normal((6, cols), seed=cols + 3)
        x[0, 3] = -inf
        x[1, 5] = inf
        x[2, 7] = nan
        x[3, :] = -inf
        x[4, :] = 7.0
        x[5, 1] = 1e30
        assert_parity(_softmax(lib, x), oracle.softmax(x), f"softmax special cols={cols}")


def test_softmax_rows_sum_to_one(lib):
    x = synth.normal((16, 393216), seed=31, var=25.0)
    p = _softmax(lib, x).double()
    assert torch.allclose(p.sum(1), torch.ones(16, dtype=torch.float64), atol=1e-4)
    assert (p >= 0).all()


def test_softmax_convenience(lib):
    x = synth.normal((3, 5, 1000), seed=41)
    got = lib.softmax(x.to(DEV))
    assert got.shape == x.shape
    assert_parity(got.reshape(15, 1000), oracle.softmax(x.reshape(15, 1000)), "softmax()")


# ----------------------------------------------------------------------------- log_softmax over an axis

DIM_SHAPES = [
    (1, 4, 320),
    (1, 32, 4096),      # a slice of the dim-0 workload's shape
    (3, 17, 33),        # ragged inner, outer > 1
    (2, 7, 1000),
    (1, 1, 64),         # R = 1: every output is 0 (or NaN)
    (1, 5000, 3),       # long R, tiny inner
    (4, 300, 8),
    (1, 9, 4097),       # inner not a multiple of 4: scalar kernel
    (2, 64, 12),
    (5, 2000, 1),       # inner = 1: the row kernels
    (2, 70000, 1),
]


@pytest.mark.parametrize("outer,R,inner", DIM_SHAPES)
@pytest.mark.parametrize("misalign", [False, True])
def test_log_softmax_dim_parity(lib, outer, R, inner, misalign):
    x = synth.uniform((outer, R, inner), seed=outer * 7 + R * 3 + inner, lo=-20, hi=20)
    got = _lsm_dim(lib, x, outer, R, inner, misalign)
    assert_parity(got, oracle.log_softmax_dim(x, outer, R, inner), f"lsm dim {outer,R,inner}")


@pytest.mark.parametrize("one_walk", ["0", "1"], ids=["two-walks", "one-walk"])
@pytest.mark.parametrize("outer,R,inner", [(1, 8, 1000), (3, 16, 260), (1, 32, 4096), (2, 64, 12),
                                           (2, 32, 40000)])
def test_log_softmax_dim_walks(lib, env, one_walk, outer, R, inner):
    """R = 8 x the thread rows: the tile kept in registers (one walk) or walked twice
    through L2; both give the oracle's result, ragged inner tiles included."""
    env.setenv("LSE_STRIDED_ONE_WALK", one_walk)
    x = synth.uniform((outer, R, inner), seed=outer * 5 + R + inner, lo=-20, hi=20)
    got = _lsm_dim(lib, x, outer, R, inner, False)
    assert_parity(got, oracle.log_softmax_dim(x, outer, R, inner), f"lsm dim {outer, R, inner} walks {one_walk}")


def test_log_softmax_dim_special_values(lib):
    inf, nan = float("inf"), float("nan")
    cols = [[1.0, nan, 2.0, 0.0], [nan, inf, 0.0, 1.0], [inf, 1.0, -inf, 0.0],
            [-inf, -inf, -inf, -inf], [-inf, 0.0, -inf, -inf], [-inf, 1.0, 2.0, -inf],
            [1e30, -1e30, 3.0, 1e30], [-1e30, -1e30, -1e30, -1e30]]
    x = torch.tensor(cols, dtype=torch.float32).T.contiguous()   # (R=4, inner=8)
    for rep in (1, 3, 20):
        xx = x.repeat(rep, 1)
        R = 4 * rep
        got = _lsm_dim(lib, xx, 1, R, 8)
        assert_parity(got, oracle.log_softmax_dim(xx, 1, R, 8), f"lsm dim special R={R}")


def test_log_softmax_dim_convenience_every_axis(lib):
    x = synth.normal((3, 5, 7, 9), seed=55, var=9.0)
    for dim in range(4):
        got = lib.log_softmax(x.to(DEV), dim=dim)
        ref = torch.log_softmax(x.double(), dim=dim).numpy()
        assert_parity(got, ref, f"log_softmax dim={dim}")


def test_log_softmax_dim_columns_normalised(lib):
    x = synth.normal((2, 256, 4096), seed=57, var=16.0)
    got = _lsm_dim(lib, x, 2, 256, 4096).double()
    s = torch.exp(got).sum(1)
    assert torch.allclose(s, torch.ones_like(s), atol=1e-5)


# ----------------------------------------------------------------------------- GroupNorm and the chain

GN_CASES = [
    (2, 64, 12, 12, 16),
    (2, 64, 126, 126, 16),   # two samples of the chain's shape
    (3, 8, 5, 7, 4),         # HW = 35: scalar kernels
    (2, 6, 4, 4, 3),
    (1, 4, 1, 1, 1),
    (2, 32, 9, 9, 32),       # one channel per group
    (1, 20, 33, 3, 5),       # C not a multiple of 4: channel tail
    (19, 16, 8, 8, 4),       # more samples than the lag
]


def _gn(L, fn, inp, G, eps=1e-5, misalign=False):
    y = inp["y"].to(DEV)
    out = torch.full(y.shape, float("nan"), device=DEV)
    if misalign:
        y, out = _misaligned(y), _misaligned(out)
    N, C = y.shape[0], y.shape[1]
    HW = y[0, 0].numel()
    getattr(L, fn)(y, inp["gamma"].to(DEV), inp["beta"].to(DEV), out, N, C, HW, G, eps)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("variant", ["0", "3"])
@pytest.mark.parametrize("fn", ["group_norm", "gn_act_residual"])
@pytest.mark.parametrize("N,C,H,W,G", GN_CASES)
def test_gn_elementwise_parity(lib, env, fn, N, C, H, W, G, variant):
    """The default (slab rows in tensor memory where HW % 4 == 0 and the pointers are
    16-byte aligned, else the bulk-copy work queue) and the bulk-copy work queue itself."""
    env.setenv("LSE_GN_VARIANT", variant)
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = _gn(lib, fn, inp, G)
    ref = getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"{fn} {N,C,H,W,G}")


@pytest.mark.parametrize("fn", ["group_norm", "gn_act_residual"])
def test_gn_elementwise_misaligned(lib, fn):
    N, C, H, W, G = 2, 8, 4, 8, 2
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = _gn(lib, fn, inp, G, misalign=True)
    assert_parity(got, getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-5),
                  f"{fn} misaligned")


@pytest.mark.parametrize("variant", ["0", "2", "3"])
@pytest.mark.parametrize("fn", ["group_norm", "gn_act_residual"])
def test_gn_elementwise_non_finite(lib, env, fn, variant):
    """NaN, +inf or -inf in a group makes exactly that group NaN (its mean or variance is
    NaN); the other groups and samples match the oracle."""
    env.setenv("LSE_GN_VARIANT", variant)
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 16, 6, 7))
    y = inp["y"].clone()
    y[0, 5, 2, 3] = float("nan")
    y[1, 1, 0, 0] = float("inf")
    y[2, 10, 5, 6] = float("-inf")
    inp["y"] = y
    got = _gn(lib, fn, inp, 4)
    nan = torch.isnan(got)
    assert int(nan.sum()) == 3 * 4 * 42
    assert bool(nan[0, 4:8].all() and nan[1, 0:4].all() and nan[2, 8:12].all())
    assert_parity(got, getattr(oracle, fn)(y, inp["gamma"], inp["beta"], 4, 1e-5), f"{fn} non-finite y")


@pytest.mark.parametrize("cfg", [{"LSE_GN_VARIANT": "2", "LSE_GN_PARTS": "5", "LSE_GN_LAG": "0"},
                                 {"LSE_GN_VARIANT": "2", "LSE_GN_PARTS": "16", "LSE_GN_LAG": "100",
                                  "LSE_GN_CTAS_PER_SM": "1"},
                                 {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "1", "LSE_GNT_LAG": "0"},
                                 {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "2", "LSE_GNT_LAG": "3",
                                  "LSE_GNT_CTAS_PER_SM": "1"},
                                 {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "6", "LSE_GNT_LAG": "100"}],
                         ids=["queue-p5", "queue-p16", "tma-s1", "tma-s2", "tma-s6"])
@pytest.mark.parametrize("fn", ["group_norm", "gn_act_residual"])
def test_gn_elementwise_configs(lib, env, cfg, fn):
    for k, v in cfg.items():
        env.setenv(k, v)
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(5, 64, 20, 20))
    got = _gn(lib, fn, inp, 16)
    assert_parity(got, getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], 16, 1e-5),
                  f"{fn} {cfg}")


GN_ROW_CASES = [
    (5, 64, 20, 20, 16),     # slabs of 1,600 floats: one CTA or a few per slab
    (3, 64, 126, 126, 16),   # the full image: slabs of 63,504 floats over several CTAs
    (7, 32, 40, 40, 8),      # ragged last slice
    (2, 8, 64, 64, 2),       # slabs of 16,384 floats
    (40, 16, 32, 32, 4),     # 160 slabs: more rows than SMs
    (300, 4, 16, 16, 1),     # 300 one-group samples: the CTAs loop over rows
    (2, 6, 4, 4, 3),         # two channels per group, 32-float slabs
]


@pytest.mark.parametrize("cfg", [{}, {"LSE_GNR_GROUP": "2"}, {"LSE_GNR_GROUP": "19"},
                                 {"LSE_GNR_GROUP": "3", "LSE_GNR_CHUNK": "1024"}],
                         ids=["plan", "gs2", "gs19", "gs3-chunk1k"])
@pytest.mark.parametrize("fn", ["group_norm", "gn_act_residual"])
@pytest.mark.parametrize("N,C,H,W,G", GN_ROW_CASES)
def test_gn_rows_parity(lib, env, fn, N, C, H, W, G, cfg):
    """The (sample, group) slabs as rows parked in tensor memory (LSE_GN_VARIANT=6)."""
    env.setenv("LSE_GN_VARIANT", "6")
    for k, v in cfg.items():
        env.setenv(k, v)
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = _gn(lib, fn, inp, G)
    ref = getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"{fn} rows {N,C,H,W,G} {cfg}")


@pytest.mark.parametrize("fn", ["group_norm", "gn_act_residual"])
def test_gn_rows_non_finite(lib, env, fn):
    """test_gn_elementwise_non_finite with 48 pixels (HW % 4 == 0: the row kernel takes it)."""
    env.setenv("LSE_GN_VARIANT", "6")
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 16, 6, 8))
    y = inp["y"].clone()
    y[0, 5, 2, 3] = float("nan")
    y[1, 1, 0, 0] = float("inf")
    y[2, 10, 5, 6] = float("-inf")
    inp["y"] = y
    got = _gn(lib, fn, inp, 4)
    nan = torch.isnan(got)
    assert int(nan.sum()) == 3 * 4 * 48
    assert bool(nan[0, 4:8].all() and nan[1, 0:4].all() and nan[2, 8:12].all())
    assert_parity(got, getattr(oracle, fn)(y, inp["gamma"], inp["beta"], 4, 1e-5), f"{fn} rows non-finite y")


@pytest.mark.parametrize("variant", ["0", "6"])
def test_group_norm_large_mean(lib, env, variant):
    """Mean 100 times the spread (1e2 and 0.5): the mean is subtracted before scaling and the
    variance is not E[y^2] - E[y]^2 (which in fp32 would be off by ~1e-3 relative here).
    The regime stays where an fp32 GroupNorm can meet the tolerance: z inherits the mean's
    half-ulp times rstd * gamma (8e-6 here; 3e-4 at mean 1e3 and spread 0.1, the chain's
    own large-mean test, where the output's magnitude widens the tolerance)."""
    env.setenv("LSE_GN_VARIANT", variant)
    N, C, H, W, G = 2, 16, 40, 40, 4
    inp = {"y": synth.normal((N, C, H, W), seed=81, mean=1.0e2, var=0.25),
           "gamma": synth.uniform((C,), seed=82, lo=0.5, hi=1.5),
           "beta": synth.normal((C,), seed=83, var=0.1)}
    for fn in ("group_norm", "gn_act_residual"):
        got = _gn(lib, fn, inp, G)
        assert_parity(got, getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-5),
                      f"{fn} mean 1e3 v{variant}")


@pytest.mark.parametrize("variant", ["0", "6"])
def test_group_norm_wide_range(lib, env, variant):
    env.setenv("LSE_GN_VARIANT", variant)
    N, C, H, W, G = 2, 16, 20, 20, 4
    inp = {"y": synth.normal((N, C, H, W), seed=77, mean=30.0, var=25.0),
           "gamma": synth.uniform((C,), seed=78, lo=-3.0, hi=3.0),
           "beta": synth.normal((C,), seed=79, var=4.0)}
    for fn in ("group_norm", "gn_act_residual"):
        got = _gn(lib, fn, inp, G, eps=1e-3)
        assert_parity(got, getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-3),
                      f"{fn} wide")


def test_group_norm_moments(lib):
    """With gamma = 1, beta = 0 every group of the output has mean 0 and
    population variance var / (var + eps)."""
    N, C, H, W, G = 3, 32, 16, 16, 8
    y = synth.normal((N, C, H, W), seed=81, mean=-4.0, var=9.0)
    inp = {"y": y, "gamma": torch.ones(C), "beta": torch.zeros(C)}
    z = _gn(lib, "group_norm", inp, G).double().reshape(N, G, -1)
    var = y.double().reshape(N, G, -1).var(dim=2, unbiased=False)
    assert torch.allclose(z.mean(2), torch.zeros(N, G, dtype=torch.float64), atol=1e-5)
    assert torch.allclose(z.var(2, unbiased=False), var / (var + 1e-5), atol=1e-5)


def test_group_norm_constant_group(lib):
    y = torch.full((1, 4, 3, 3), 2.0)
    inp = {"y": y, "gamma": torch.ones(4), "beta": torch.tensor([0.0, 0.5, -1.0, 2.0])}
    got = _gn(lib, "group_norm", inp, 2)
    assert_parity(got, oracle.group_norm(y, inp["gamma"], inp["beta"], 2, 1e-5), "gn constant")


def test_gn_chain_consistency(lib):
    """The lse over channels of gn_act_residual's output is gn_act_lse's output."""
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 64, 30, 30))
    r = _gn(lib, "gn_act_residual", inp, 16).to(DEV)
    lse = lib.logsumexp(r, dim=1, keepdim=True)
    full = lib.gn_act_lse_forward(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), 16, 1e-5)
    assert (lse - full).abs().max().item() < 1e-5


def test_gn_conveniences(lib):
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(2, 16, 6, 10))
    args = (inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), 4, 1e-5)
    assert_parity(lib.group_norm_forward(*args),
                  oracle.group_norm(inp["y"], inp["gamma"], inp["beta"], 4, 1e-5), "group_norm_forward")
    assert_parity(lib.gn_act_residual_forward(*args),
                  oracle.gn_act_residual(inp["y"], inp["gamma"], inp["beta"], 4, 1e-5),
                  "gn_act_residual_forward")
