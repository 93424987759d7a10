"""Out-of-bounds writes (GPU only): every entry point writes into the middle of a
buffer whose guard regions on both sides hold a sentinel, on ragged shapes and
on aligned and unaligned addresses; the guards must be intact afterwards and
the outputs must match the oracle.  (compute-sanitizer is not available here;
this is the check that stands in for its out-of-bounds detection.)
"""
import pytest
import torch

import oracle
import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SENTINEL = -12345.5


@pytest.fixture(scope="module", autouse=True)
def lib():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300 as L
    L.load_library()
    torch.cuda.set_device(0)
    yield L
    assert L.lse_device_status() == 0


def _guarded(shape, shift):
    """A view of `shape` inside a larger buffer, `shift` floats past a 1 KB guard."""
    n = 1
    for s in shape:
        n *= s
    pad = 256 + shift
    buf = torch.full((n + pad + 256,), SENTINEL, device=DEV)
    return buf, buf[pad:pad + n].view(shape), pad, n


def _intact(buf, pad, n):
    torch.cuda.synchronize()
    return bool((buf[:pad] == SENTINEL).all()) and bool((buf[pad + n:] == SENTINEL).all())


@pytest.mark.parametrize("shift", [0, 1])
def test_row_ops(lib, shift, monkeypatch):
    for variant in ("0", "7", "8", "3", "1"):
        monkeypatch.setenv("LSE_LSM_VARIANT", variant)
        for rows, cols in ((3, 5), (7, 4099), (5, 70001), (3, 393216)):
            x = synth.normal((rows, cols), seed=rows + cols)
            for name, fn, ref in (("log_softmax", lib.log_softmax_lastdim, oracle.log_softmax),
                                  ("softmax", lib.softmax_lastdim, oracle.softmax)):
                buf, out, pad, n = _guarded((rows, cols), shift)
                fn(x.to(DEV), out, rows, cols)
                assert _intact(buf, pad, n), f"{name} {rows}x{cols} wrote outside its output"
                assert_parity(out.cpu(), ref(x), f"{name} {rows}x{cols}")


@pytest.mark.parametrize("shift", [0, 1])
def test_strided_ops(lib, shift):
    for outer, R, inner in ((2, 5, 33), (1, 32, 4100), (3, 300, 8)):
        x = synth.uniform((outer, R, inner), seed=R + inner, lo=-5, hi=5)
        buf, out, pad, n = _guarded((outer, inner), shift)
        lib.lse_reduce(x.to(DEV), out, outer, R, inner)
        assert _intact(buf, pad, n)
        assert_parity(out.cpu(), oracle.lse_reduce(x, outer, R, inner), "lse_reduce")
        buf, out, pad, n = _guarded((outer, R, inner), shift)
        lib.log_softmax_dim(x.to(DEV), out, outer, R, inner)
        assert _intact(buf, pad, n)
        assert_parity(out.cpu(), oracle.log_softmax_dim(x, outer, R, inner), "log_softmax_dim")


@pytest.mark.parametrize("shift", [0, 1])
def test_groupnorm_ops(lib, shift, monkeypatch):
    for variant in ("0", "1", "2", "3", "4", "5", "6", "7"):
        monkeypatch.setenv("LSE_GN_VARIANT", variant)
        for N, C, H, W, G in ((3, 64, 12, 12, 16), (2, 8, 5, 7, 4), (5, 16, 8, 8, 4)):
            inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
            y, g, b = (inp[k].to(DEV) for k in ("y", "gamma", "beta"))
            buf, out, pad, n = _guarded((N, 1, H, W), shift)
            lib.gn_act_lse(y, g, b, out, N, C, H * W, G, 1e-5)
            assert _intact(buf, pad, n), f"gn_act_lse v{variant}"
            assert_parity(out.cpu(), oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5), "gn")
            for fn in ("group_norm", "gn_act_residual"):
                buf, out, pad, n = _guarded((N, C, H, W), shift)
                getattr(lib, fn)(y, g, b, out, N, C, H * W, G, 1e-5)
                assert _intact(buf, pad, n), f"{fn} v{variant}"
                assert_parity(out.cpu(), getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-5), fn)


@pytest.mark.parametrize("shift", [0, 1])
def test_conv_ops(lib, shift, monkeypatch):
    for chain in ("1", "2", "3"):
        monkeypatch.setenv("LSE_CONV_CHAIN", chain)
        for N, H, W in ((2, 9, 11), (1, 130, 131)):
            inp = synth.make_inputs("conv_gn_act_lse_128x8x128x128", shape=(N, 8, H, W))
            x, w, b, g, be = (inp[k].to(DEV) for k in ("x", "w", "bias", "gamma", "beta"))
            buf, y, pad, n = _guarded((N, 64, H - 2, W - 2), shift)
            lib.conv2d_3x3(x, w, b, y, N, 8, H, W, 64)
            assert _intact(buf, pad, n), "conv2d_3x3"
            assert_parity(y.cpu(), oracle.conv2d(inp["x"], inp["w"], inp["bias"]), "conv2d")
            buf, out, pad, n = _guarded((N, 1, H - 2, W - 2), shift)
            lib.conv_gn_act_lse(x, w, b, g, be, out, N, 8, H, W, 64, 16, 1e-5)
            assert _intact(buf, pad, n), f"conv_gn_act_lse chain {chain}"
            assert_parity(out.cpu(), oracle.conv_gn_act_lse(inp["x"], inp["w"], inp["bias"], inp["gamma"],
                                                            inp["beta"], 16, 1e-5), "conv chain")
