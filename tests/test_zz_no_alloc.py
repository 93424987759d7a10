"""gn_act_lse_noalloc, the entry point for callers that must not allocate device
memory (a plugin whose host framework owns all device memory, or a
latency-critical path that cannot take an allocation's cost or failure), gives
the chain's result.

It is called through the C ABI twice in a row, on different inputs, and each
result is compared with the oracle element by element (the parity tolerance of
the other tests) and, as an extra check, with the allocating entry point's on
the same input.  A third call fills the fixed scratch to its last entry
(N * G = 65536, so every entry of the array is written and read back), and one
more than that is rejected before any launch.  This file is collected last so
that a run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process (the first call does the per-device
set-up).
"""
import ctypes

import pytest
import torch

import oracle
import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LSE_ERR_SIZE = 2
MAX_GROUPS = 65536


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300 as L
    torch.cuda.set_device(0)
    return L, L.load_library()


def _inputs(N, C, H, W, shift):
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    # different data for each case: scale and shift the draw by the case index
    return inp["y"] * (1.0 + 0.5 * shift) + shift, inp["gamma"], inp["beta"]


def _both(L, lib, y, gamma, beta, G, stream):
    """The no-allocation call and gn_act_lse on the same device copy of the inputs."""
    N, C, H, W = y.shape
    yd, gd, bd = y.to(DEV), gamma.to(DEV), beta.to(DEV)
    ref = torch.empty(N, 1, H, W, device=DEV)
    got = torch.full((N, 1, H, W), float("nan"), device=DEV)
    rc = lib.gn_act_lse_noalloc(_p(yd), _p(gd), _p(bd), _p(got), N, C, H * W, G, 1e-5, stream)
    assert rc == 0, L.lse_status_string(rc)
    rc = lib.gn_act_lse(_p(yd), _p(gd), _p(bd), _p(ref), N, C, H * W, G, 1e-5, stream)
    assert rc == 0, L.lse_status_string(rc)
    torch.cuda.synchronize()
    return got.cpu(), ref.cpu()


def test_noalloc_matches_the_oracle_twice_in_a_row(lib):
    L, c = lib
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(2, 64, 12, 12, 16, 0), (3, 8, 5, 7, 4, 1)]   # second: HW % 4 != 0
    for N, C, H, W, G, shift in cases:
        y, gamma, beta = _inputs(N, C, H, W, shift)
        got, ref = _both(L, c, y, gamma, beta, G, stream)
        assert_parity(got, oracle.gn_act_lse(y, gamma, beta, G, 1e-5), f"noalloc vs oracle {N, C, H, W, G}")
        assert_parity(got, ref.double().numpy(), f"noalloc vs gn_act_lse {N, C, H, W, G}")


def test_noalloc_non_finite_values(lib):
    # NaN / +inf / -inf in one group of samples 0 / 1 / 2 make those samples NaN, as in
    # the oracle; sample 3 stays finite
    L, c = lib
    stream = torch.cuda.current_stream().cuda_stream
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 16, 6, 7))
    y = inp["y"].clone()
    y[0, 5, 2, 3], y[1, 1, 0, 0], y[2, 10, 5, 6] = float("nan"), float("inf"), float("-inf")
    got, _ = _both(L, c, y, inp["gamma"], inp["beta"], 4, stream)
    assert_parity(got, oracle.gn_act_lse(y, inp["gamma"], inp["beta"], 4, 1e-5), "noalloc, non-finite y")


def test_noalloc_fills_the_fixed_scratch_and_rejects_more(lib):
    L, c = lib
    stream = torch.cuda.current_stream().cuda_stream
    # N * G == 65536: every entry of the fixed array is written, then read back
    N, C, G, H, W = MAX_GROUPS // 16, 16, 16, 2, 2
    y, gamma, beta = _inputs(N, C, H, W, 2)
    got, ref = _both(L, c, y, gamma, beta, G, stream)
    assert_parity(got, oracle.gn_act_lse(y, gamma, beta, G, 1e-5), "noalloc at N*G = 65536")
    assert_parity(got, ref.double().numpy(), "noalloc vs gn_act_lse at N*G = 65536")

    # one group more than the array holds: rejected on the host, nothing launched
    out = torch.full((4,), 7.0, device=DEV)
    small = torch.zeros(4, device=DEV)
    rc = c.gn_act_lse_noalloc(_p(small), _p(small), _p(small), _p(out), MAX_GROUPS + 1, 1, 1, 1, 1e-5, stream)
    assert rc == LSE_ERR_SIZE, L.lse_status_string(rc)
    rc = c.gn_act_lse_noalloc(_p(small), _p(small), _p(small), _p(out), 4097, 16, 1, 16, 1e-5, stream)
    assert rc == LSE_ERR_SIZE, L.lse_status_string(rc)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
