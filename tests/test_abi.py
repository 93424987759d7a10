"""The C-ABI library loads, exports what include/lse.h declares, and rejects bad
arguments on the host before touching CUDA (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lse.h")


@pytest.fixture(scope="module")
def lib():
    from log_softmax_gb300 import build
    build.build()
    import log_softmax_gb300
    return log_softmax_gb300.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("lse_reduce", "log_softmax_lastdim", "gn_act_lse", "lse_status_string",
              "lse_last_cuda_error", "softmax_lastdim", "log_softmax_dim", "group_norm",
              "gn_act_residual", "log_softmax_lastdim_host", "gn_act_lse_noalloc"):
        assert n in names, names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in lse.h but not exported"


def test_python_binding_names_match(lib):
    import log_softmax_gb300 as L
    for name in declared_functions():
        assert callable(getattr(L, name, None)), f"binding lacks {name}"


def test_status_strings(lib):
    import log_softmax_gb300 as L
    for code in range(8):
        assert L.lse_status_string(code) and L.lse_status_string(code) != "unknown status"
    assert L.lse_status_string(99) == "unknown status"


# Each case fails validation before any CUDA call, so it runs without a GPU.
LSE_REDUCE_ERRORS = [
    ((None, None, -1, 3, 3), 2),      # negative size
    ((None, None, 2, 0, 3), 2),       # empty reduced axis with outputs
    ((None, None, 2, 3, 3), 1),       # null pointers
    ((2, 8, 2, 3, 3), 3),             # x not 4-byte aligned
    ((None, None, 2**40, 2**40, 2**10), 2),  # element count overflows int64
    ((None, None, 0, 5, 3), 0),       # no outputs: ok, nothing launched
    ((None, None, 5, 0, 0), 0),
]


@pytest.mark.parametrize("args,want", LSE_REDUCE_ERRORS)
def test_lse_reduce_validation(lib, args, want):
    assert lib.lse_reduce(*args, None) == want


LSM_ERRORS = [
    ((None, None, -1, 4), 2),
    ((None, None, 4, -4), 2),
    ((None, None, 4, 4), 1),
    ((16, 34, 4, 4), 3),
    ((None, None, 2**62, 4), 2),
    ((None, None, 0, 7), 0),
    ((None, None, 7, 0), 0),
]


@pytest.mark.parametrize("args,want", LSM_ERRORS)
def test_log_softmax_validation(lib, args, want):
    assert lib.log_softmax_lastdim(*args, None) == want
    assert lib.log_softmax_lastdim_host(*args, None) == want
    assert lib.softmax_lastdim(*args, None) == want


LSM_DIM_ERRORS = [
    ((None, None, -1, 3, 3), 2),
    ((None, None, 2, -3, 3), 2),
    ((None, None, 2, 3, -3), 2),
    ((None, None, 2, 0, 3), 0),       # empty reduced axis: no outputs either
    ((None, None, 2, 3, 3), 1),
    ((2, 8, 2, 3, 3), 3),
    ((16, 34, 2, 3, 1), 3),           # inner = 1 goes to the row path, same checks
    ((None, None, 2**40, 2**40, 2**10), 2),
    ((None, None, 0, 5, 3), 0),
]


@pytest.mark.parametrize("args,want", LSM_DIM_ERRORS)
def test_log_softmax_dim_validation(lib, args, want):
    assert lib.log_softmax_dim(*args, None) == want


GN_ERRORS = [
    ((1, 6, 4, 4, 1e-5), 2),           # C % G != 0
    ((1, 0, 4, 1, 1e-5), 2),           # C = 0
    ((1, 8, 4, 0, 1e-5), 2),           # G = 0
    ((-1, 8, 4, 4, 1e-5), 2),
    ((1, 16384, 4, 4, 1e-5), 2),       # more channels than the apply table holds
    ((1, 8, 4, 4, -1.0), 6),           # eps < 0
    ((1, 8, 4, 4, float("nan")), 6),
    ((1, 8, 4, 4, float("inf")), 6),
    ((0, 8, 4, 4, 1e-5), 0),           # no outputs
    ((1, 8, 4, 4, 1e-5), 1),           # null pointers
]


@pytest.mark.parametrize("args,want", GN_ERRORS)
def test_gn_act_lse_validation(lib, args, want):
    N, C, HW, G, eps = args
    assert lib.gn_act_lse(None, None, None, None, N, C, HW, G, eps, None) == want
    assert lib.group_norm(None, None, None, None, N, C, HW, G, eps, None) == want
    assert lib.gn_act_residual(None, None, None, None, N, C, HW, G, eps, None) == want
    # the no-allocation entry point checks gn_act_lse's rules first, with the same codes
    assert lib.gn_act_lse_noalloc(None, None, None, None, N, C, HW, G, eps, None) == want


NOALLOC_LIMIT_ERRORS = [
    ((65537, 1, 1, 1, 1e-5), 2),       # one group more than the fixed scratch holds
    ((4097, 16, 1, 16, 1e-5), 2),
    ((65537, 1, 1, 1, -1.0), 6),       # a bad eps is reported first, as gn_act_lse does
    ((4097, 16, 0, 16, 1e-5), 2),      # no outputs, but past the limit: still rejected
]


@pytest.mark.parametrize("args,want", NOALLOC_LIMIT_ERRORS)
def test_gn_act_lse_noalloc_limit(lib, args, want):
    N, C, HW, G, eps = args
    # aligned stand-in addresses: the call must return before touching any of them
    assert lib.gn_act_lse_noalloc(16, 16, 16, 16, N, C, HW, G, eps, None) == want


CONV_ERRORS = [
    ((1, 8, 2, 8, 64), 2),        # H < 3
    ((1, 0, 8, 8, 64), 2),        # Cin = 0
    ((-1, 8, 8, 8, 64), 2),
    ((1, 9, 8, 8, 64), 5),        # Cin > 8: no tensor-core path
    ((1, 8, 8, 8, 40), 5),        # Cout not a multiple of 16
    ((1, 8, 8, 8, 256), 5),       # Cout > 128
    ((1, 8, 8, 1025, 64), 5),     # W > 1024: the staged window would not fit
    ((0, 8, 8, 8, 64), 0),        # no outputs
    ((1, 8, 8, 8, 64), 1),        # null pointers
]


@pytest.mark.parametrize("args,want", CONV_ERRORS)
def test_conv2d_validation(lib, args, want):
    N, Cin, H, W, Cout = args
    assert lib.conv2d_3x3(None, None, None, None, N, Cin, H, W, Cout, None) == want
    assert lib.conv_gn_act_lse(None, None, None, None, None, None, N, Cin, H, W, Cout, 16 if Cout % 16 == 0
                               else 1, 1e-5, None) == want


CONV_CHAIN_ERRORS = [
    ((1, 8, 8, 8, 64, 5, 1e-5), 2),     # Cout % G != 0
    ((1, 8, 8, 8, 64, 2, 1e-5), 5),     # 32 channels per group: not a divisor of 16
    ((1, 8, 8, 8, 64, 16, -1.0), 6),    # eps < 0
    ((1, 8, 8, 8, 64, 0, 1e-5), 2),
    ((1, 8, 8, 8, 64, 16, 1e-5), 1),    # null pointers
    ((1, 4, 8, 8, 64, 16, 1e-5), 5),    # Cin != 8: conv2d_3x3 then gn_act_lse instead
]


@pytest.mark.parametrize("args,want", CONV_CHAIN_ERRORS)
def test_conv_chain_validation(lib, args, want):
    N, Cin, H, W, Cout, G, eps = args
    assert lib.conv_gn_act_lse(None, None, None, None, None, None, N, Cin, H, W, Cout, G, eps, None) == want


def test_binding_raises_on_error(lib):
    import torch

    import log_softmax_gb300 as L
    with pytest.raises(L.LseError) as e:
        L.lse_reduce(None, None, 2, 0, 3, stream=0)
    assert e.value.status == 2
    with pytest.raises(ValueError):
        L.log_softmax_lastdim(torch.zeros(2, 3), torch.zeros(2, 3), 2, 3, stream=0)


def test_missing_library_fails_loudly(tmp_path):
    import log_softmax_gb300 as L
    saved = L._lib
    try:
        L._lib = None
        with pytest.raises(ImportError):
            L.load_library(str(tmp_path / "liblse.so"))
    finally:
        L._lib = saved


def test_product_does_not_import_oracle():
    """The CUDA path and its binding never import or load the oracle."""
    pkg = os.path.join(ROOT, "log_softmax_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
