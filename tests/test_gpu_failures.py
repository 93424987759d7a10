"""Failure paths, made on the host or by a bounded wait that runs out; nothing
here faults, traps or hangs a GPU (GPU only).

- an exhausted scratch pool (a test hook makes the library's allocation fail)
  must come back as LSE_ERR_CUDA with cudaErrorMemoryAllocation, with nothing
  enqueued, and the library must work normally afterwards;
- a statistics wait whose target nothing reaches must give up after about one
  second, record LSE_ERR_TIMEOUT in the device status (read and cleared by
  lse_device_status) and leave the context usable.
"""
import pytest
import torch

import oracle
import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CUDA_ERROR_MEMORY_ALLOCATION = 2


@pytest.fixture(scope="module", autouse=True)
def lib():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300 as L
    L.load_library()
    torch.cuda.set_device(0)
    yield L
    assert L.lse_device_status() == 0


def _gn_inputs():
    return synth.make_inputs("gn_act_lse_128x64x126x126", shape=(3, 64, 12, 12))


def _gn_call(L, inp, out):
    L.gn_act_lse(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), out, 3, 64, 144, 16, 1e-5)


def test_allocation_failure_is_reported(lib, monkeypatch):
    inp = _gn_inputs()
    out = torch.full((3, 1, 12, 12), 7.0, device=DEV)
    x = synth.normal((4, 393216), seed=9, device=DEV)
    xo = torch.full_like(x, 7.0)
    monkeypatch.setenv("LSE_TEST_FAIL_ALLOC", "1")
    for call in (lambda: _gn_call(lib, inp, out),
                 lambda: lib.log_softmax_lastdim(x, xo, 4, 393216),
                 lambda: lib.group_norm(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV),
                                        torch.empty(3, 64, 12, 12, device=DEV), 3, 64, 144, 16, 1e-5)):
        with pytest.raises(lib.LseError) as e:
            call()
        assert e.value.status == 4
        assert lib.lse_last_cuda_error() == CUDA_ERROR_MEMORY_ALLOCATION
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((xo == 7.0).all())  # nothing was enqueued
    monkeypatch.delenv("LSE_TEST_FAIL_ALLOC")
    _gn_call(lib, inp, out)
    torch.cuda.synchronize()
    assert_parity(out.cpu(), oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], 16, 1e-5), "after")
    assert lib.lse_device_status() == 0


def test_bounded_wait_timeout_is_reported(lib, monkeypatch):
    inp = _gn_inputs()
    out = torch.empty(3, 1, 12, 12, device=DEV)
    monkeypatch.setenv("LSE_GN_VARIANT", "2")           # the work-queue kernel and its statistics wait
    monkeypatch.setenv("LSE_TEST_UNREACHABLE_WAIT", "1")
    _gn_call(lib, inp, out)                              # enqueued: the wait runs out on the device
    assert lib.lse_device_status() == 7                  # LSE_ERR_TIMEOUT, then cleared
    assert lib.lse_status_string(7) != "unknown status"
    monkeypatch.delenv("LSE_TEST_UNREACHABLE_WAIT")
    _gn_call(lib, inp, out)                              # the context is still usable
    torch.cuda.synchronize()
    assert lib.lse_device_status() == 0
    assert_parity(out.cpu(), oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], 16, 1e-5), "after")


def test_timeout_raises_through_a_convenience(lib, monkeypatch):
    """A convenience that returns a host result synchronises, so it reads the device
    status: a bounded wait that ran out becomes LseError(LSE_ERR_TIMEOUT) instead of
    a silently unspecified result, and the next call works."""
    inp = _gn_inputs()
    monkeypatch.setenv("LSE_GN_VARIANT", "2")
    monkeypatch.setenv("LSE_TEST_UNREACHABLE_WAIT", "1")
    with pytest.raises(lib.LseError) as e:
        lib.gn_act_lse_forward(inp["y"].pin_memory(), inp["gamma"], inp["beta"], 16, 1e-5)
    assert e.value.status == 7
    assert lib.lse_device_status() == 0                  # the status was read and cleared
    monkeypatch.delenv("LSE_TEST_UNREACHABLE_WAIT")
    got = lib.gn_act_lse_forward(inp["y"].pin_memory(), inp["gamma"], inp["beta"], 16, 1e-5)
    assert not got.is_cuda
    assert_parity(got, oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], 16, 1e-5), "after the timeout")
