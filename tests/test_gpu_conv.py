"""Conv2d 3x3 on the tensor cores (and the chain fed by it) against the oracle,
element by element, through the C ABI (GPU only)."""
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


def _inputs(N, Cin, H, W, Cout, seed=0):
    inp = synth.make_inputs("conv_gn_act_lse_128x8x128x128", shape=(N, Cin, H, W))
    if Cout != inp["w"].shape[0] or seed:
        bound = 1.0 / np.sqrt(Cin * 9)
        inp["w"] = synth.uniform((Cout, Cin, 3, 3), 300 + seed, -bound, bound)
        inp["bias"] = synth.uniform((Cout,), 400 + seed, -bound, bound)
        inp["gamma"] = synth.uniform((Cout,), 500 + seed, 0.5, 1.5)
        inp["beta"] = synth.normal((Cout,), 600 + seed, var=0.1)
    return inp


def _conv(L, inp, misalign=False):
    x, w, b = (inp[k].to(DEV) for k in ("x", "w", "bias"))
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    y = torch.full((N, Cout, H - 2, W - 2), float("nan"), device=DEV)
    if misalign:
        def mis(t):
            buf = torch.empty(t.numel() + 1, device=DEV)
            v = buf[1:].view(t.shape)
            v.copy_(t)
            return v
        x, w, b, y = mis(x), mis(w), mis(b), mis(y)
    L.conv2d_3x3(x, w, b, y, N, Cin, H, W, Cout)
    torch.cuda.synchronize()
    return y.cpu()


CONV_SHAPES = [
    (2, 8, 16, 20, 64),     # several 128-pixel tiles, the chain's channel counts
    (1, 8, 128, 128, 64),   # one full sample of the chain's input
    (3, 3, 7, 9, 16),       # K = 27 padded to 32, one partial tile
    (2, 1, 5, 5, 32),       # K = 9 padded to 16
    (1, 8, 130, 131, 128),  # Cout = 128, ragged last tile (three MMAs per tap)
    (5, 4, 12, 3, 48),      # OW = 1
    (2, 8, 14, 18, 80),     # Cout = 80: three MMAs per tap, 128 accumulator columns
    (1, 8, 5, 1024, 64),    # W = 1024, the widest accepted: the window is loaded directly
    (1, 8, 4, 1024, 128),   # the same with the largest Cout
    (1, 8, 6, 900, 64),     # the widest that keeps the bulk-copy window at Cout = 64
    (2, 8, 3, 40, 32),      # H = 3: one output row
    (3, 5, 3, 3, 16),       # a 1 x 1 output per sample
]


@pytest.mark.parametrize("N,Cin,H,W,Cout", CONV_SHAPES)
def test_conv2d_parity(lib, N, Cin, H, W, Cout):
    inp = _inputs(N, Cin, H, W, Cout)
    got = _conv(lib, inp)
    ref = oracle.conv2d(inp["x"], inp["w"], inp["bias"])
    assert_parity(got, ref, f"conv2d {N, Cin, H, W, Cout}")


def test_conv2d_misaligned(lib):
    inp = _inputs(2, 8, 9, 11, 64)
    assert_parity(_conv(lib, inp, misalign=True), oracle.conv2d(inp["x"], inp["w"], inp["bias"]),
                  "conv2d misaligned")


def test_conv2d_wide_values(lib):
    """Inputs of scale 30 and weights of scale 1: the split keeps fp32 accuracy.  Outputs
    here are sums of products of scale ~15 whose fp32 accumulation alone rounds at ~1e-6
    of the largest output, so the bar adds that term to the usual one."""
    N, Cin, H, W, Cout = 2, 8, 10, 12, 64
    inp = {"x": synth.normal((N, Cin, H, W), 71, var=900.0),
           "w": synth.uniform((Cout, Cin, 3, 3), 72, -1.0, 1.0),
           "bias": synth.normal((Cout,), 73)}
    got = _conv(lib, inp)
    ref = oracle.conv2d(inp["x"], inp["w"], inp["bias"])
    err = np.abs(got.double().numpy() - ref)
    assert (err <= 2e-5 + 2e-6 * np.abs(ref) + 1e-6 * np.abs(ref).max()).all(), err.max()


def test_conv2d_forward_convenience(lib):
    inp = _inputs(2, 8, 14, 15, 64)
    got = lib.conv2d_3x3_forward(inp["x"].to(DEV), inp["w"].to(DEV), inp["bias"].to(DEV))
    assert_parity(got, oracle.conv2d(inp["x"], inp["w"], inp["bias"]), "conv2d_3x3_forward")


# ----------------------------------------------------------------------------- the chain from x

CHAIN_CASES = [
    (2, 8, 16, 20, 64, 16),     # the chain's channel counts, several tiles
    (2, 8, 128, 128, 64, 16),   # two full samples of the chain's shape
    (3, 8, 9, 11, 32, 8),       # 4 channels per group, Cout = 32
    (2, 8, 12, 14, 64, 64),     # 1 channel per group
    (2, 8, 12, 14, 64, 4),      # 16 channels per group
    (1, 8, 20, 7, 48, 6),       # 8 channels per group, Cout = 48
    (1, 8, 20, 22, 128, 16),    # Cout = 128: the unstacked products in every epilogue
    (1, 8, 5, 1024, 64, 16),    # W = 1024
]


def _chain(L, inp, G, eps=1e-5):
    x, w, b, g, be = (inp[k].to(DEV) for k in ("x", "w", "bias", "gamma", "beta"))
    N, Cin, H, W = x.shape
    out = torch.full((N, 1, H - 2, W - 2), float("nan"), device=DEV)
    L.conv_gn_act_lse(x, w, b, g, be, out, N, Cin, H, W, w.shape[0], G, eps)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("chain", ["1", "2", "3"], ids=["y-round-trip", "y-free", "y-then-queue"])
@pytest.mark.parametrize("N,Cin,H,W,Cout,G", CHAIN_CASES)
def test_conv_chain_parity(lib, N, Cin, H, W, Cout, G, chain, monkeypatch):
    monkeypatch.setenv("LSE_CONV_CHAIN", chain)
    inp = _inputs(N, Cin, H, W, Cout, seed=1 if Cout != 64 else 0)
    got = _chain(lib, inp, G)
    ref = oracle.conv_gn_act_lse(inp["x"], inp["w"], inp["bias"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"conv chain {N, Cin, H, W, Cout, G}")


def test_conv2d_nan_input(lib):
    """A NaN input pixel makes NaN exactly the outputs whose window holds it, in every channel."""
    inp = _inputs(2, 8, 14, 16, 64)
    inp["x"] = inp["x"].clone()
    inp["x"][0, 3, 5, 7] = float("nan")
    got = _conv(lib, inp)
    assert int(torch.isnan(got).sum()) == 9 * 64
    assert_parity(got, oracle.conv2d(inp["x"], inp["w"], inp["bias"]), "conv2d with a NaN input")


@pytest.mark.parametrize("chain", ["1", "2", "3"], ids=["y-round-trip", "y-free", "y-then-queue"])
def test_conv_chain_nan_input(lib, chain, monkeypatch):
    """A NaN in one sample's input reaches every group mean of that sample, so the
    whole sample's output is NaN; the other sample is untouched."""
    monkeypatch.setenv("LSE_CONV_CHAIN", chain)
    inp = _inputs(2, 8, 14, 16, 64)
    inp["x"] = inp["x"].clone()
    inp["x"][0, 3, 5, 7] = float("nan")
    got = _chain(lib, inp, 16)
    assert bool(torch.isnan(got[0]).all()) and not bool(torch.isnan(got[1]).any())
    ref = oracle.conv_gn_act_lse(inp["x"], inp["w"], inp["bias"], inp["gamma"], inp["beta"], 16, 1e-5)
    assert_parity(got, ref, "conv chain with a NaN input")


def test_conv_chain_other_cin_is_two_calls(lib):
    """Cin other than the layer's 8 is not fused: the call reports it, and the two
    calls it stands for give the chain."""
    inp = _inputs(2, 3, 12, 10, 64, seed=2)
    with pytest.raises(lib.LseError):
        _chain(lib, inp, 16)
    y = _conv(lib, inp).to(DEV)
    got = lib.gn_act_lse_forward(y, inp["gamma"].to(DEV), inp["beta"].to(DEV), 16, 1e-5)
    ref = oracle.conv_gn_act_lse(inp["x"], inp["w"], inp["bias"], inp["gamma"], inp["beta"], 16, 1e-5)
    assert_parity(got, ref, "conv then chain, Cin = 3")


def test_conv_chain_matches_two_steps(lib):
    """The fused call equals conv2d_3x3 followed by gn_act_lse on its output."""
    inp = _inputs(3, 8, 40, 36, 64)
    y = _conv(lib, inp).to(DEV)
    two = lib.gn_act_lse_forward(y, inp["gamma"].to(DEV), inp["beta"].to(DEV), 16, 1e-5).cpu()
    one = _chain(lib, inp, 16)
    assert (one - two).abs().max().item() < 1e-5


def test_conv_chain_forward_convenience(lib):
    inp = _inputs(2, 8, 18, 17, 64)
    got = lib.conv_gn_act_lse_forward(*(inp[k].to(DEV) for k in ("x", "w", "bias", "gamma", "beta")), 16)
    assert got.shape == (2, 1, 16, 15)
    assert_parity(got, oracle.conv_gn_act_lse(inp["x"], inp["w"], inp["bias"], inp["gamma"], inp["beta"], 16),
                  "conv_gn_act_lse_forward")


@pytest.mark.parametrize("tma", ["0", "1"])
def test_conv2d_window_paths(lib, tma, monkeypatch):
    """Raw windows fetched by bulk copies one tile ahead, or loaded directly."""
    monkeypatch.setenv("LSE_CONV_TMA", tma)
    for shape in ((3, 8, 20, 24, 64), (1, 8, 130, 132, 64), (2, 3, 9, 12, 16)):
        inp = _inputs(*shape, seed=3)
        assert_parity(_conv(lib, inp), oracle.conv2d(inp["x"], inp["w"], inp["bias"]), f"conv tma={tma} {shape}")


@pytest.mark.parametrize("ws", ["0", "1"], ids=["tile-slots", "pipeline"])
def test_conv2d_pipeline_paths(lib, ws, monkeypatch):
    """The pipelined kernel (warp roles, rings of four raw windows, split windows and
    accumulators) and the tile-slot kernel: several tiles per CTA so that every ring
    wraps, fewer tiles than SMs, every stacked Cout, unstacked Cout 96 (three products per
    tap), a ragged last tile, the widest rows its rings take; Cout 112 and 128 and planes
    of H W % 4 != 0 (no bulk copies) take the tile-slot kernel either way."""
    monkeypatch.setenv("LSE_CONV_WS", ws)
    for shape in ((12, 8, 128, 128, 64), (1, 8, 20, 24, 64), (4, 8, 32, 47, 16), (3, 5, 40, 36, 32),
                  (2, 8, 60, 70, 48), (1, 8, 130, 131, 128), (2, 8, 50, 180, 64), (2, 8, 61, 70, 48),
                  (4, 8, 64, 64, 128), (3, 8, 20, 36, 96), (1, 8, 128, 128, 112), (2, 8, 30, 132, 128),
                  (2, 8, 12, 140, 128)):
        inp = _inputs(*shape, seed=5)
        assert_parity(_conv(lib, inp), oracle.conv2d(inp["x"], inp["w"], inp["bias"]), f"conv ws={ws} {shape}")
