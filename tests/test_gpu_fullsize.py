"""The bench workloads at full size, in the launch configuration the bench times
(GPU only).  Outputs the oracle can afford are checked element by element on a
seeded sample; every output is checked against properties that hold at any size.
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


def test_lse_dim0_4x10x32(lib):
    x = synth.make_inputs("lse_dim0_4x10x32")["x"]
    out = torch.empty(10, 32, device=DEV)
    lib.lse_reduce(x.to(DEV), out, 1, 4, 320)
    assert_parity(out, oracle.logsumexp_dim0(x), "(4,10,32)")


def test_log_softmax_256x4096(lib):
    x = synth.make_inputs("log_softmax_256x4096")["x"]
    out = torch.empty(256, 4096, device=DEV)
    lib.log_softmax_lastdim(x.to(DEV), out, 256, 4096)
    assert_parity(out, oracle.log_softmax(x), "(256,4096)")


def test_lse_dim0_32x8192x4096(lib):
    x = synth.make_inputs("lse_dim0_32x8192x4096", device=DEV)["x"]
    R, inner = 32, 8192 * 4096
    out = torch.empty(8192, 4096, device=DEV)
    lib.lse_reduce(x, out, 1, R, inner)
    torch.cuda.synchronize()
    # sampled outputs against the oracle
    g = torch.Generator().manual_seed(303)
    idx = torch.randint(0, inner, (8192,), generator=g)
    idx = torch.cat([idx, torch.tensor([0, 1, 2, 3, inner - 4, inner - 3, inner - 2, inner - 1])])
    cols = x.view(R, inner)[:, idx.to(DEV)].cpu().contiguous()
    ref = oracle.lse_reduce(cols, 1, R, cols.shape[1])[0]
    assert_parity(out.view(-1)[idx.to(DEV)].cpu(), ref, "sampled")
    # every output: max <= lse <= max + ln R
    mx = x.view(R, inner).amax(dim=0)
    o = out.view(-1)
    assert bool(((o >= mx - 1e-5 * mx.abs()) & (o <= mx + math.log(R) + 1e-5)).all())
    del x, mx


def test_log_softmax_4096x393216(lib):
    rows, cols = 4096, 393216
    x = synth.make_inputs("log_softmax_4096x393216", device=DEV)["x"]
    out = torch.empty_like(x)
    lib.log_softmax_lastdim(x, out, rows, cols)
    torch.cuda.synchronize()
    # a seeded sample of 256 full rows, the first and the last among them
    g = torch.Generator().manual_seed(404)
    rows_s = sorted(set([0, rows - 1] + torch.randperm(rows - 2, generator=g)[:254].add(1).tolist()))
    assert len(rows_s) == 256
    for k in range(0, 256, 64):
        part = rows_s[k:k + 64]
        assert_parity(out[part].cpu(), oracle.log_softmax(x[part].cpu()), f"sampled rows {k}..{k + 63}")
    # every row: sum exp = 1 and out - x constant along the row
    for r0 in range(0, rows, 512):
        o = out[r0:r0 + 512].double()
        s = torch.exp(o).sum(dim=1)
        assert bool(((s - 1).abs() < 1e-4).all()), float((s - 1).abs().max())
        d = (x[r0:r0 + 512].double() - o)
        assert bool(((d - d[:, :1]).abs() < 5e-5).all())
    del x, out


@pytest.mark.parametrize("variant", ["0", "5", "7"])
def test_gn_act_lse_128x64x126x126(lib, monkeypatch, variant):
    monkeypatch.setenv("LSE_GN_VARIANT", variant)
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", device=DEV)
    y, gamma, beta = inp["y"], inp["gamma"], inp["beta"]
    N, C, H, W = y.shape
    out = torch.empty(N, 1, H, W, device=DEV)
    lib.gn_act_lse(y, gamma, beta, out, N, C, H * W, 16, 1e-5)
    torch.cuda.synchronize()
    for n in (0, 77, N - 1):
        ref = oracle.gn_act_lse(y[n:n + 1].cpu(), gamma.cpu(), beta.cpu(), 16, 1e-5)
        assert_parity(out[n:n + 1].cpu(), ref, f"sample {n}")
    # every output: max_c r <= out <= max_c r + ln C, with r bounded by y +- 2/3
    ymax = y.amax(dim=1, keepdim=True)
    assert bool((out <= ymax + 2.0 / 3.0 + math.log(C) + 1e-4).all())
    assert bool((out >= ymax - 1.0 / 3.0 - 1e-4).all())


# ----------------------------------------------------------------------------- the NEXT rows at full size

def test_softmax_4096x393216(lib):
    rows, cols = 4096, 393216
    x = synth.make_inputs("softmax_4096x393216", device=DEV)["x"]
    out = torch.empty_like(x)
    lib.softmax_lastdim(x, out, rows, cols)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(505)
    rows_s = sorted(set([0, rows - 1] + torch.randperm(rows - 2, generator=g)[:254].add(1).tolist()))
    for k in range(0, len(rows_s), 64):
        part = rows_s[k:k + 64]
        assert_parity(out[part].cpu(), oracle.softmax(x[part].cpu()), f"sampled rows {k}..{k + 63}")
    # every row sums to one, every entry in [0, 1]
    for r0 in range(0, rows, 512):
        s = out[r0:r0 + 512].double().sum(dim=1)
        assert bool(((s - 1).abs() < 1e-4).all()), float((s - 1).abs().max())
    assert bool(((out >= 0) & (out <= 1)).all())
    del x, out


def test_log_softmax_dim0_32x8192x4096(lib):
    x = synth.make_inputs("log_softmax_dim0_32x8192x4096", device=DEV)["x"]
    R, inner = 32, 8192 * 4096
    out = torch.empty_like(x)
    lib.log_softmax_dim(x, out, 1, R, inner)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(606)
    idx = torch.cat([torch.randint(0, inner, (4096,), generator=g),
                     torch.tensor([0, 1, 2, 3, inner - 4, inner - 3, inner - 2, inner - 1])]).to(DEV)
    cols = x.view(R, inner)[:, idx].cpu().contiguous()
    assert_parity(out.view(R, inner)[:, idx].cpu(), oracle.log_softmax_dim(cols, 1, R, cols.shape[1])[0],
                  "sampled columns")
    # every column: sum over the axis of exp = 1
    for c0 in range(0, inner, 1 << 24):
        s = torch.exp(out.view(R, inner)[:, c0:c0 + (1 << 24)].double()).sum(dim=0)
        assert bool(((s - 1).abs() < 1e-5).all()), float((s - 1).abs().max())
    del x, out


@pytest.mark.parametrize("fn,workload", [("group_norm", "group_norm_128x64x126x126"),
                                         ("gn_act_residual", "gn_act_residual_128x64x126x126")])
def test_gn_elementwise_full(lib, fn, workload):
    inp = synth.make_inputs(workload, device=DEV)
    y, gamma, beta = inp["y"], inp["gamma"], inp["beta"]
    N, C, H, W = y.shape
    out = torch.empty_like(y)
    getattr(lib, fn)(y, gamma, beta, out, N, C, H * W, 16, 1e-5)
    torch.cuda.synchronize()
    for n in (0, 64, N - 1):
        ref = getattr(oracle, fn)(y[n:n + 1].cpu(), gamma.cpu(), beta.cpu(), 16, 1e-5)
        assert_parity(out[n:n + 1].cpu(), ref, f"{fn} sample {n}")
    if fn == "group_norm":
        # every (n, g): ((z - beta) / gamma) has mean 0 and variance var / (var + eps)
        zn = ((out - beta.view(1, C, 1, 1)) / gamma.view(1, C, 1, 1)).double().view(N, 16, -1)
        var = y.double().view(N, 16, -1).var(dim=2, unbiased=False)
        assert float(zn.mean(dim=2).abs().max()) < 1e-4
        assert float((zn.var(dim=2, unbiased=False) - var / (var + 1e-5)).abs().max()) < 1e-4
    else:
        # every element: out - y = hardswish(tanh(z)) lies in [-1/3, 2/3]
        d = out - y
        assert bool(((d >= -1.0 / 3.0 - 1e-6) & (d <= 2.0 / 3.0 + 1e-6)).all())
    del y, out


def test_conv_gn_act_lse_128x8x128x128(lib):
    inp = synth.make_inputs("conv_gn_act_lse_128x8x128x128", device=DEV)
    x, w, b, gamma, beta = (inp[k] for k in ("x", "w", "bias", "gamma", "beta"))
    N, Cin, H, W = x.shape
    out = torch.empty(N, 1, H - 2, W - 2, device=DEV)
    lib.conv_gn_act_lse(x, w, b, gamma, beta, out, N, Cin, H, W, 64, 16, 1e-5)
    torch.cuda.synchronize()
    for n in (0, 91, N - 1):
        ref = oracle.conv_gn_act_lse(x[n:n + 1].cpu(), w.cpu(), b.cpu(), gamma.cpu(), beta.cpu(), 16, 1e-5)
        assert_parity(out[n:n + 1].cpu(), ref, f"conv chain sample {n}")
    # every output: the chain's bounds around max_c y (y from the library's conv)
    y = torch.empty(N, 64, H - 2, W - 2, device=DEV)
    lib.conv2d_3x3(x, w, b, y, N, Cin, H, W, 64)
    ymax = y.amax(dim=1, keepdim=True)
    assert bool((out <= ymax + 2.0 / 3.0 + math.log(64) + 1e-4).all())
    assert bool((out >= ymax - 1.0 / 3.0 - 1e-4).all())
    del x, y, out
