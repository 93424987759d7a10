"""Concurrent calls (GPU only): scratch, counters and per-device state are never shared.

Two streams run the same entry point on different data with no ordering between
them, and two host threads call the library in a loop on their own streams (ctypes
releases the interpreter lock during the foreign call, so the calls really overlap
on the host).  Every result is compared with the oracle.
"""
import threading

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


def _gn_case(seed, N=5, C=64, H=20, W=20):
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    inp["y"] = inp["y"] * (1.0 + seed) + seed
    return inp


def _conv_case(seed, N=2, Cin=8, H=24, W=30):
    inp = synth.make_inputs("conv_gn_act_lse_128x8x128x128", shape=(N, Cin, H, W))
    inp["x"] = synth.normal((N, Cin, H, W), 400 + seed)
    return inp


def _run(lib, kind, inp, stream):
    """Copy the inputs in and enqueue one call, all on `stream` (so the call is
    ordered after its copies and nothing else); returns the output and the device
    tensors to keep alive until the stream is synchronised."""
    with torch.cuda.stream(stream):
        if kind == "log_softmax_long":
            x = inp["x"].to(DEV)
            out = torch.empty_like(x)
            lib.log_softmax_lastdim(x, out, x.shape[0], x.shape[1], stream=stream)
            return out, (x,)
        if kind == "lse_reduce":
            x = inp["x"].to(DEV)
            out = torch.empty(x.shape[1], device=DEV)
            lib.lse_reduce(x, out, 1, x.shape[0], x.shape[1], stream=stream)
            return out, (x,)
        if kind == "gn_act_lse":
            y, g, b = (inp[k].to(DEV) for k in ("y", "gamma", "beta"))
            N, C, H, W = y.shape
            out = torch.empty(N, 1, H, W, device=DEV)
            lib.gn_act_lse(y, g, b, out, N, C, H * W, 16, 1e-5, stream=stream)
            return out, (y, g, b)
        if kind == "conv_gn_act_lse":
            t = {k: inp[k].to(DEV) for k in ("x", "w", "bias", "gamma", "beta")}
            N, Cin, H, W = t["x"].shape
            out = torch.empty(N, 1, H - 2, W - 2, device=DEV)
            lib.conv_gn_act_lse(t["x"], t["w"], t["bias"], t["gamma"], t["beta"], out, N, Cin, H, W, 64, 16,
                                1e-5, stream=stream)
            return out, tuple(t.values())
    raise KeyError(kind)


def _reference(kind, inp):
    if kind == "log_softmax_long":
        return oracle.log_softmax(inp["x"])
    if kind == "lse_reduce":
        return oracle.lse_reduce(inp["x"], 1, inp["x"].shape[0], inp["x"].shape[1])[0]
    if kind == "gn_act_lse":
        return oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], 16, 1e-5)
    return oracle.conv_gn_act_lse(inp["x"], inp["w"], inp["bias"], inp["gamma"], inp["beta"], 16, 1e-5)


def _draw(kind, seed):
    if kind == "log_softmax_long":
        return {"x": synth.normal((24, 393216), 500 + seed)}
    if kind == "lse_reduce":
        return {"x": synth.uniform((32, 90001), 600 + seed, -20.0, 20.0)}
    if kind == "gn_act_lse":
        return _gn_case(seed)
    return _conv_case(seed)


KINDS = ["log_softmax_long", "lse_reduce", "gn_act_lse", "conv_gn_act_lse"]


@pytest.mark.parametrize("kind", KINDS)
def test_two_streams_unordered(lib, kind):
    """The same entry point on two streams at once, three calls each, no ordering."""
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    draws = [[_draw(kind, 10 * s + k) for k in range(3)] for s in range(2)]
    torch.cuda.synchronize()
    pending = []
    for k in range(3):
        for s in range(2):
            pending.append((draws[s][k], _run(lib, kind, draws[s][k], streams[s])))
    torch.cuda.synchronize()
    for i, (inp, (out, _)) in enumerate(pending):
        assert_parity(out.cpu(), _reference(kind, inp), f"{kind}, call {i}")


def test_two_host_threads(lib):
    """Two host threads, each with its own stream, alternate entry points in a loop."""
    errors = []
    results = [[], []]

    def worker(t):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            for it in range(6):
                kind = KINDS[(it + t) % len(KINDS)]
                inp = _draw(kind, 100 * t + it)
                out, keep = _run(lib, kind, inp, s)
                s.synchronize()
                results[t].append((kind, out.cpu(), inp))
                del keep
        except Exception as e:  # reported below, on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads)
    assert not errors, errors
    for t in range(2):
        assert len(results[t]) == 6
        for kind, got, inp in results[t]:
            assert_parity(got, _reference(kind, inp), f"thread {t} {kind}")
