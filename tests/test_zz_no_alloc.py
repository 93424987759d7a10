"""gn_act_lse_noalloc, the entry point for callers that must not allocate device
memory (a plugin whose host framework owns all device memory, or a
latency-critical path that cannot take an allocation's cost or failure), gives
what gn_act_lse gives.

It is called through the C ABI twice in a row, on different inputs, and each
result is compared with the allocating entry point's on the same input, within
the parity tolerance of the other tests.  This file is collected last so that a
run stopping at its first failure has already run every other test; it also
passes on its own in a fresh process (the first call does the per-device set-up).
"""
import ctypes

import pytest
import torch

import oracle
import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_allocating_entry_point():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300 as L
    lib = L.load_library()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream

    cases = [(2, 64, 12, 12, 16, 0), (3, 8, 5, 7, 4, 1)]   # second: HW % 4 != 0
    for N, C, H, W, G, seed_shift in cases:
        inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W), device=DEV)
        # different data for the two shapes: shift the draw by the case index
        y = inp["y"] * (1.0 + 0.5 * seed_shift) + seed_shift
        gamma, beta = inp["gamma"], inp["beta"]
        ref = torch.empty(N, 1, H, W, device=DEV)
        got = torch.full((N, 1, H, W), float("nan"), device=DEV)
        rc = lib.gn_act_lse(_p(y), _p(gamma), _p(beta), _p(ref), N, C, H * W, G, 1e-5, stream)
        assert rc == 0, L.lse_status_string(rc)
        rc = lib.gn_act_lse_noalloc(_p(y), _p(gamma), _p(beta), _p(got), N, C, H * W, G, 1e-5,
                                    stream)
        assert rc == 0, L.lse_status_string(rc)
        torch.cuda.synchronize()
        assert_parity(got.cpu(), ref.cpu().double().numpy(), f"noalloc vs gn_act_lse {N,C,H,W,G}")

    # non-finite values: NaN / +inf / -inf in one group of samples 0 / 1 / 2 make those
    # samples NaN, as in the oracle; sample 3 stays finite
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 16, 6, 7))
    y = inp["y"].clone()
    y[0, 5, 2, 3], y[1, 1, 0, 0], y[2, 10, 5, 6] = float("nan"), float("inf"), float("-inf")
    yd, gd, bd = y.to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV)
    got = torch.empty(4, 1, 6, 7, device=DEV)
    rc = lib.gn_act_lse_noalloc(_p(yd), _p(gd), _p(bd), _p(got), 4, 16, 42, 4, 1e-5, stream)
    assert rc == 0, L.lse_status_string(rc)
    torch.cuda.synchronize()
    assert_parity(got.cpu(), oracle.gn_act_lse(y, inp["gamma"], inp["beta"], 4, 1e-5), "noalloc, non-finite y")

    # beyond the fixed scratch (N * G > 65536): rejected before any launch
    big = torch.empty(4, device=DEV)
    rc = lib.gn_act_lse_noalloc(_p(big), _p(big), _p(big), _p(big), 65537, 16, 1, 16, 1e-5, stream)
    assert rc == 2, L.lse_status_string(rc)
