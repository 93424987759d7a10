"""Tensors past 2^31 elements (GPU only).

Every entry point accepts sizes up to INT64_MAX / 4 elements, so every kernel must
address its data with 64-bit offsets.  Each case below puts some outputs (or the
inputs they read) beyond element 2^31 and compares sampled rows, columns or samples
on both sides of that boundary with the oracle; every output is also checked
against a property that holds at any size.  The largest case holds about 20 GB on
the device.
"""
import math

import pytest
import torch

import oracle
import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BIG = 1 << 31


@pytest.fixture(scope="module")
def lib():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300 as L
    L.load_library()
    torch.cuda.set_device(0)
    yield L
    assert L.lse_device_status() == 0
    torch.cuda.empty_cache()


@pytest.fixture(autouse=True)
def _release():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _rows_across(rows, cols):
    """Row indices around the first row that holds element 2^31, and the ends."""
    k = BIG // cols
    return sorted({0, 1, k - 1, k, k + 1, rows - 2, rows - 1})


@pytest.mark.parametrize("fn,rows,cols", [("log_softmax_lastdim", 8192, 270336),   # long rows
                                          ("log_softmax_lastdim", 524416, 4096),   # short rows
                                          ("softmax_lastdim", 8192, 270336)])
def test_rows_past_2_31(lib, fn, rows, cols):
    assert rows * cols > BIG
    workload = "log_softmax_4096x393216" if cols > 4096 else "log_softmax_256x4096"
    x = synth.make_inputs(workload, shape=(rows, cols), device=DEV)["x"]
    out = torch.empty_like(x)
    getattr(lib, fn)(x, out, rows, cols)
    torch.cuda.synchronize()
    rs = _rows_across(rows, cols)
    ref = (oracle.log_softmax if fn == "log_softmax_lastdim" else oracle.softmax)(x[rs].cpu())
    assert_parity(out[rs].cpu(), ref, f"{fn} rows {rs}")
    step = max(1, (1 << 28) // cols)
    for r0 in range(0, rows, step):
        o = out[r0:r0 + step].double()
        s = (torch.exp(o) if fn == "log_softmax_lastdim" else o).sum(dim=1)
        assert bool(((s - 1).abs() < 1e-4).all()), (r0, float((s - 1).abs().max()))
    del x, out


@pytest.mark.parametrize("fn", ["log_softmax_lastdim", "softmax_lastdim", "row_lse"])
def test_rows_of_40m(lib, fn):
    """Rows of 40 million floats (160 MB), far past what shared memory can stage: the
    streaming row kernels, compared with the oracle element by element."""
    rows, cols = 2, 40_000_000
    x = synth.make_inputs("log_softmax_4096x393216", shape=(rows, cols), device=DEV)["x"]
    xc = x.cpu()
    if fn == "row_lse":
        out = torch.empty(rows, device=DEV)
        lib.lse_reduce(x, out, rows, cols, 1)
        ref = oracle.lse_reduce(xc.view(rows, cols, 1), rows, cols, 1)
    else:
        out = torch.empty_like(x)
        getattr(lib, fn)(x, out, rows, cols)
        ref = (oracle.log_softmax if fn == "log_softmax_lastdim" else oracle.softmax)(xc)
    torch.cuda.synchronize()
    assert_parity(out.cpu().view(ref.shape), ref, f"{fn} rows of {cols}")
    del x, out


@pytest.mark.parametrize("outer,R,inner", [(1, 4, 540_000_000), (65_600, 8, 4096)])
def test_lse_reduce_past_2_31(lib, outer, R, inner):
    assert outer * R * inner > BIG
    x = synth.make_inputs("lse_dim0_32x8192x4096", shape=(outer * R, inner), device=DEV)["x"]
    x = x.view(outer, R, inner)
    out = torch.empty(outer, inner, device=DEV)
    lib.lse_reduce(x, out, outer, R, inner)
    torch.cuda.synchronize()
    # sampled (o, i) whose inputs lie before and after element 2^31
    os_ = sorted({0, outer // 2, outer - 1})
    is_ = torch.tensor(sorted({0, 1, inner // 2, inner - 2, inner - 1}), device=DEV)
    for o in os_:
        cols = x[o][:, is_].cpu().contiguous()
        ref = oracle.lse_reduce(cols, 1, R, cols.shape[1])[0]
        assert_parity(out[o, is_].cpu(), ref, f"lse_reduce outer {o}")
    # every output: max <= lse <= max + ln R
    for o0 in range(0, outer, max(1, outer // 8)):
        blk = x[o0:o0 + max(1, outer // 8)]
        mx = blk.amax(dim=1)
        ob = out[o0:o0 + max(1, outer // 8)]
        assert bool(((ob >= mx - 1e-5 * mx.abs()) & (ob <= mx + math.log(R) + 1e-5)).all())
        del mx
    del x, out


def test_log_softmax_dim_past_2_31(lib):
    outer, R, inner = 1, 4, 540_000_000
    x = synth.make_inputs("log_softmax_dim0_32x8192x4096", shape=(R, inner), device=DEV)["x"]
    out = torch.empty_like(x)
    lib.log_softmax_dim(x, out, outer, R, inner)
    torch.cuda.synchronize()
    idx = torch.tensor([0, 1, inner // 2, inner - 2, inner - 1], device=DEV)
    cols = x[:, idx].cpu().contiguous()
    assert_parity(out[:, idx].cpu(), oracle.log_softmax_dim(cols, 1, R, cols.shape[1])[0], "columns across 2^31")
    for c0 in range(0, inner, 1 << 26):
        s = torch.exp(out[:, c0:c0 + (1 << 26)].double()).sum(dim=0)
        assert bool(((s - 1).abs() < 1e-5).all()), (c0, float((s - 1).abs().max()))
    del x, out


@pytest.mark.parametrize("fn", ["gn_act_lse", "group_norm", "gn_act_residual"])
def test_group_norm_forms_past_2_31(lib, fn):
    N, C, H, W, G = 540, 64, 250, 250, 16
    assert N * C * H * W > BIG
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W), device=DEV)
    y, gamma, beta = inp["y"], inp["gamma"], inp["beta"]
    out = torch.empty((N, 1, H, W) if fn == "gn_act_lse" else (N, C, H, W), device=DEV)
    getattr(lib, fn)(y, gamma, beta, out, N, C, H * W, G, 1e-5)
    torch.cuda.synchronize()
    first = BIG // (C * H * W)  # the first sample that holds element 2^31
    for n in sorted({0, first, first + 1, N - 1}):
        ref = getattr(oracle, fn)(y[n:n + 1].cpu(), gamma.cpu(), beta.cpu(), G, 1e-5)
        assert_parity(out[n:n + 1].cpu(), ref, f"{fn} sample {n}")
    if fn == "gn_act_lse":
        ymax = y.amax(dim=1, keepdim=True)
        assert bool((out <= ymax + 2.0 / 3.0 + math.log(C) + 1e-4).all())
        assert bool((out >= ymax - 1.0 / 3.0 - 1e-4).all())
    elif fn == "gn_act_residual":
        for n0 in range(0, N, 64):
            d = out[n0:n0 + 64] - y[n0:n0 + 64]
            assert bool(((d >= -1.0 / 3.0 - 1e-6) & (d <= 2.0 / 3.0 + 1e-6)).all())
    else:
        # every (n, g): (z - beta) / gamma has mean 0
        for n0 in range(0, N, 64):
            zn = ((out[n0:n0 + 64] - beta.view(1, C, 1, 1)) / gamma.view(1, C, 1, 1)).view(-1, G, C // G * H * W)
            assert float(zn.double().mean(dim=2).abs().max()) < 1e-4
    del y, out


@pytest.mark.parametrize("fn", ["conv2d_3x3", "conv_gn_act_lse"])
def test_conv_forms_past_2_31(lib, fn):
    N, Cin, H, W, Cout, G = 2200, 8, 128, 128, 64, 16
    OH, OW = H - 2, W - 2
    assert N * Cout * OH * OW > BIG
    inp = synth.make_inputs("conv_gn_act_lse_128x8x128x128", shape=(N, Cin, H, W), device=DEV)
    x, w, b, gamma, beta = (inp[k] for k in ("x", "w", "bias", "gamma", "beta"))
    first = BIG // (Cout * OH * OW)  # the first sample whose y holds element 2^31
    samples = sorted({0, first, first + 1, N - 1})
    if fn == "conv2d_3x3":
        y = torch.empty(N, Cout, OH, OW, device=DEV)
        lib.conv2d_3x3(x, w, b, y, N, Cin, H, W, Cout)
        torch.cuda.synchronize()
        for n in samples:
            assert_parity(y[n:n + 1].cpu(), oracle.conv2d(x[n:n + 1].cpu(), w.cpu(), b.cpu()), f"conv2d sample {n}")
        assert not bool(torch.isnan(y).any())
        del y
    else:
        out = torch.empty(N, 1, OH, OW, device=DEV)
        lib.conv_gn_act_lse(x, w, b, gamma, beta, out, N, Cin, H, W, Cout, G, 1e-5)
        torch.cuda.synchronize()
        for n in samples:
            ref = oracle.conv_gn_act_lse(x[n:n + 1].cpu(), w.cpu(), b.cpu(), gamma.cpu(), beta.cpu(), G, 1e-5)
            assert_parity(out[n:n + 1].cpu(), ref, f"conv chain sample {n}")
        assert bool(torch.isfinite(out).all())
        del out
    del x
