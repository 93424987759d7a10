"""CUDA path against the oracle, element by element, through the C ABI (GPU only).

Sizes here are ones the oracle finishes in seconds but that still span several
tiles, clusters and a ragged tail; every kernel variant and the special values
are covered.  Full-size workloads are in test_gpu_fullsize.py.
"""
import math
import os

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
    """Same values at a device address 4 bytes past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=torch.float32, device=DEV)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _lse_reduce(L, x_cpu, outer, R, inner, misalign=False):
    x = x_cpu.to(DEV)
    out = torch.full((outer, inner), float("nan"), device=DEV)
    if misalign:
        x = _misaligned(x)
        out = _misaligned(out)
    L.lse_reduce(x, out, outer, R, inner)
    torch.cuda.synchronize()
    return out.cpu()


def _log_softmax(L, x_cpu, misalign=False):
    rows, cols = x_cpu.shape
    x = x_cpu.to(DEV)
    out = torch.full((rows, cols), float("nan"), device=DEV)
    if misalign:
        x = _misaligned(x)
        out = _misaligned(out)
    L.log_softmax_lastdim(x, out, rows, cols)
    torch.cuda.synchronize()
    return out.cpu()


# ----------------------------------------------------------------------------- form 1

LSE_SHAPES = [
    (1, 4, 320),        # the (4, 10, 32) task, flattened
    (1, 32, 4096),      # 32 x 4096 slice of the large strided case
    (3, 17, 33),        # ragged inner, outer > 1
    (2, 7, 1000),
    (1, 1, 64),         # R = 1: lse is x itself
    (1, 5000, 3),       # long R, tiny inner: thread rows split R
    (4, 300, 8),
    (1, 9, 4097),       # inner not a multiple of 4: scalar kernel
    (5, 2000, 1),       # inner = 1: row statistic kernels
    (2, 70000, 1),      # inner = 1, long rows: streaming row kernel
]


@pytest.mark.parametrize("outer,R,inner", LSE_SHAPES)
@pytest.mark.parametrize("misalign", [False, True])
def test_lse_reduce_parity(lib, outer, R, inner, misalign):
    x = synth.uniform((outer, R, inner), seed=outer * 1000 + R + inner, lo=-20, hi=20)
    got = _lse_reduce(lib, x, outer, R, inner, misalign)
    assert_parity(got, oracle.lse_reduce(x, outer, R, inner), f"lse_reduce {outer,R,inner}")


def test_lse_dim0_small_workload(lib):
    x = synth.make_inputs("lse_dim0_4x10x32")["x"]
    got = lib.logsumexp(x.to(DEV), dim=0)
    assert got.shape == (10, 32)
    assert_parity(got, oracle.logsumexp_dim0(x), "lse dim0 (4,10,32)")


def test_logsumexp_other_dims(lib):
    x = synth.normal((3, 5, 7, 9), seed=5, var=9.0)
    for dim in range(4):
        got = lib.logsumexp(x.to(DEV), dim=dim)
        ref = torch.logsumexp(x.double(), dim=dim).numpy()
        assert_parity(got, ref, f"dim {dim}")


def test_lse_reduce_special_values(lib):
    inf, nan = float("inf"), float("nan")
    cols = [[1.0, nan, 2.0, 0.0], [nan, inf, 0.0, 1.0], [inf, 1.0, -inf, 0.0],
            [-inf, -inf, -inf, -inf], [-inf, 0.0, -inf, -inf], [-inf, 1.0, 2.0, -inf],
            [1e30, -1e30, 3.0, 1e30], [-1e30, -1e30, -1e30, -1e30]]
    x = torch.tensor(cols, dtype=torch.float32).T.contiguous()   # (R=4, inner=8)
    for R_chunks in (1, 3):  # also with the reduced axis repeated (longer R, same answer + log)
        xx = x.repeat(R_chunks, 1)
        got = _lse_reduce(lib, xx.reshape(1, 4 * R_chunks, 8), 1, 4 * R_chunks, 8)
        ref = oracle.lse_reduce(xx, 1, 4 * R_chunks, 8)
        assert_parity(got, ref, "special")


def test_lse_reduce_constant(lib):
    for R in (1, 3, 32, 257):
        x = torch.full((2, R, 12), 3.25)
        got = _lse_reduce(lib, x, 2, R, 12)
        assert_parity(got, np.full((2, 12), 3.25 + math.log(R)), f"const R={R}")


# ----------------------------------------------------------------------------- form 2

LSM_COLS = [1, 3, 4, 5, 31, 32, 33, 127, 128, 129, 512, 1000, 1023, 2048, 4096, 4097, 8192,
            16384, 16385, 32768, 32769, 32772, 60000, 131072, 393216]


@pytest.mark.parametrize("cols", LSM_COLS)
def test_log_softmax_parity(lib, cols):
    rows = max(2, min(37, 2_000_000 // cols))
    x = synth.normal((rows, cols), seed=cols, var=4.0)
    x.masked_fill_(synth.bernoulli_mask((rows, cols), seed=cols + 1, p=0.01), float("-inf"))
    x[:, 0] = 0.5  # no row is entirely -inf
    got = _log_softmax(lib, x)
    assert_parity(got, oracle.log_softmax(x), f"log_softmax cols={cols}")


@pytest.mark.parametrize("cols", [5, 129, 4097, 16385, 70001])
def test_log_softmax_misaligned(lib, cols):
    rows = 9
    x = synth.normal((rows, cols), seed=cols + 7)
    got = _log_softmax(lib, x, misalign=True)
    assert_parity(got, oracle.log_softmax(x), f"misaligned cols={cols}")


def test_log_softmax_small_workload(lib):
    x = synth.make_inputs("log_softmax_256x4096")["x"]
    got = _log_softmax(lib, x)
    assert_parity(got, oracle.log_softmax(x), "log_softmax (256,4096)")


LONG_ROW_CONFIGS = [
    # cluster shared memory (DSMEM merge)
    {"LSE_LSM_VARIANT": "2"}, {"LSE_LSM_VARIANT": "2", "LSE_LSM_CLUSTER": "1"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_CLUSTER": "2"}, {"LSE_LSM_VARIANT": "2", "LSE_LSM_CLUSTER": "4"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_CLUSTER": "8"}, {"LSE_LSM_VARIANT": "2", "LSE_LSM_CLUSTER": "16"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_THREADS": "256"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_THREADS": "1024", "LSE_LSM_CHUNK": "2048"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_CLUSTER": "8", "LSE_LSM_THREADS": "1024", "LSE_LSM_CHUNK": "16384"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_NBUF": "2"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_NBUF": "2", "LSE_LSM_CLUSTER": "4", "LSE_LSM_THREADS": "256"},
    {"LSE_LSM_VARIANT": "2", "LSE_LSM_NBUF": "2", "LSE_LSM_CLUSTER": "16", "LSE_LSM_CHUNK": "2048"},
    # streaming
    {"LSE_LSM_VARIANT": "3"},
    # group shared memory (global-memory merge), single and double buffered
    {"LSE_LSM_VARIANT": "4"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_NBUF": "1"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_NBUF": "2"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "2", "LSE_LSM_NBUF": "1"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "3", "LSE_LSM_NBUF": "2"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "5"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "8", "LSE_LSM_NBUF": "1"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "19", "LSE_LSM_NBUF": "2"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "32"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_NBUF": "3"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_NBUF": "3", "LSE_LSM_GROUP": "6", "LSE_LSM_CHUNK": "2048"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_NBUF": "3", "LSE_LSM_GROUP": "24", "LSE_LSM_THREADS": "512"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "8", "LSE_LSM_THREADS": "512", "LSE_LSM_CHUNK": "4096"},
    # warp-specialised group
    {"LSE_LSM_VARIANT": "6"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_GROUP": "2"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_GROUP": "7", "LSE_WS_FW": "8", "LSE_WS_NB": "2"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_GROUP": "16", "LSE_WS_SW": "8", "LSE_LSM_CHUNK": "2048"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_FW": "8", "LSE_WS_SW": "8"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "2"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "2", "LSE_WS_GROUP": "5", "LSE_WS_FW": "8"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "3", "LSE_WS_GROUP": "24", "LSE_WS_SW": "8"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "3", "LSE_WS_GROUP": "3", "LSE_LSM_CHUNK": "2048"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "4", "LSE_WS_GROUP": "40", "LSE_WS_FW": "12"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "5", "LSE_WS_GROUP": "38", "LSE_WS_FW": "16"},
    {"LSE_LSM_VARIANT": "6", "LSE_WS_NB": "0", "LSE_WS_FW": "4", "LSE_WS_SW": "4"},
    # warp-specialised group with a ring of chunk slots
    {"LSE_LSM_VARIANT": "7"},
    {"LSE_LSM_VARIANT": "7", "LSE_WS_GROUP": "19"},
    {"LSE_LSM_VARIANT": "7", "LSE_WS_GROUP": "3", "LSE_RING_CHUNK": "4096"},
    {"LSE_LSM_VARIANT": "7", "LSE_WS_GROUP": "40", "LSE_RING_CHUNK": "512"},
    # warp-specialised group with its rows parked in tensor memory
    {"LSE_LSM_VARIANT": "8"},
    {"LSE_LSM_VARIANT": "8", "LSE_WS_GROUP": "19"},
    {"LSE_LSM_VARIANT": "8", "LSE_WS_GROUP": "3", "LSE_TMEM_CHUNK": "4096"},
    {"LSE_LSM_VARIANT": "8", "LSE_WS_GROUP": "40", "LSE_TMEM_CHUNK": "1024"},
    # group with an L2 re-read
    {"LSE_LSM_VARIANT": "5"},
    {"LSE_LSM_VARIANT": "5", "LSE_L2_GROUP": "1"},
    {"LSE_LSM_VARIANT": "5", "LSE_L2_GROUP": "3", "LSE_L2_THREADS": "256"},
    {"LSE_LSM_VARIANT": "5", "LSE_L2_GROUP": "32", "LSE_L2_THREADS": "1024"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "16", "LSE_LSM_THREADS": "1024", "LSE_LSM_CHUNK": "2048"},
    {"LSE_LSM_VARIANT": "4", "LSE_LSM_GROUP": "2", "LSE_LSM_THREADS": "512", "LSE_LSM_CHUNK": "16384",
     "LSE_LSM_NBUF": "1"},
]


@pytest.mark.parametrize("cfg", LONG_ROW_CONFIGS,
                         ids=["-".join(f"{k[8:]}{v}" for k, v in c.items()) for c in LONG_ROW_CONFIGS])
def test_log_softmax_variants(lib, env, cfg):
    """Each long-row kernel configuration, several rows per cluster / group so that
    the persistent loop refills its shared-memory buffers."""
    for k, v in cfg.items():
        env.setenv(k, v)
    rows, cols = 300, 65536 + 4
    x = synth.normal((rows, cols), seed=99)
    got = _log_softmax(lib, x)
    assert_parity(got, oracle.log_softmax(x), f"config {cfg}")


@pytest.mark.parametrize("cluster", ["1", "2", "4", "8"])
def test_stream_cluster_sizes(lib, env, cluster):
    env.setenv("LSE_LSM_VARIANT", "3")
    env.setenv("LSE_STREAM_CLUSTER", cluster)
    x = synth.normal((5, 100003), seed=3)
    assert_parity(_log_softmax(lib, x), oracle.log_softmax(x), f"stream CL={cluster}")
    y = synth.normal((3, 100000), seed=4)
    got = _lse_reduce(lib, y.reshape(3, 100000, 1), 3, 100000, 1)
    assert_parity(got.reshape(-1), oracle.row_lse(y), f"row lse CL={cluster}")


def test_log_softmax_special_rows(lib):
    inf, nan = float("inf"), float("nan")
    for cols in (8, 4096, 40000, 393216):
        x = synth.normal((6, cols), seed=cols)
        x[0, 3] = -inf
        x[1, 5] = inf
        x[2, 7] = nan
        x[3, :] = -inf
        x[4, :] = 7.0
        x[5, 1] = 1e30
        got = _log_softmax(lib, x)
        assert_parity(got, oracle.log_softmax(x), f"special rows cols={cols}")


def test_log_softmax_shift_and_normalisation(lib):
    x = synth.normal((16, 50000), seed=21)
    a = _log_softmax(lib, x).double()
    b = _log_softmax(lib, x + 1000.0).double()
    assert torch.allclose(torch.exp(a).sum(1), torch.ones(16, dtype=torch.float64), atol=1e-5)
    assert (a - b).abs().max() < 2e-3  # x + 1000 rounds x to ~6e-5 in fp32


# ----------------------------------------------------------------------------- form 3

GN_CASES = [
    (2, 64, 12, 12, 16),
    (2, 64, 126, 126, 16),   # two samples of the full chain shape
    (3, 8, 5, 7, 4),         # HW = 35, not a multiple of 4: scalar kernels
    (2, 6, 4, 4, 3),
    (1, 4, 1, 1, 1),
    (2, 32, 9, 9, 32),       # one channel per group
    (1, 20, 33, 3, 5),       # C not a multiple of 8: channel tail
]


@pytest.mark.parametrize("N,C,H,W,G", GN_CASES)
def test_gn_act_lse_parity(lib, N, C, H, W, G):
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = lib.gn_act_lse_forward(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), G, 1e-5)
    ref = oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"gn {N,C,H,W,G}")


GN_CONFIGS = [
    {"LSE_GN_VARIANT": "1"},                                    # statistics kernel + apply kernel
    {"LSE_GN_VARIANT": "2"},                                    # work queue, default parts / lag
    {"LSE_GN_VARIANT": "2", "LSE_GN_PARTS": "1", "LSE_GN_LAG": "0"},
    {"LSE_GN_VARIANT": "2", "LSE_GN_PARTS": "7", "LSE_GN_LAG": "2"},
    {"LSE_GN_VARIANT": "2", "LSE_GN_PARTS": "16", "LSE_GN_LAG": "100", "LSE_GN_CTAS_PER_SM": "1"},
    {"LSE_GN_VARIANT": "2", "LSE_GN_THREADS": "512", "LSE_GN_LAG": "3"},
    {"LSE_GN_VARIANT": "2", "LSE_GN_THREADS": "1024", "LSE_GN_PARTS": "3"},
    {"LSE_GN_VARIANT": "0"},                                    # the default choice
    {"LSE_GN_VARIANT": "3"},                                    # work queue, bulk-copy staging
    {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "1", "LSE_GNT_LAG": "0"},
    {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "2", "LSE_GNT_LAG": "2", "LSE_GNT_CTAS_PER_SM": "1"},
    {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "6", "LSE_GNT_LAG": "100"},
    {"LSE_GN_VARIANT": "3", "LSE_GNT_SLOTS": "8", "LSE_GNT_CTAS_PER_SM": "1"},
    {"LSE_GN_VARIANT": "4"},                                    # sample slices in shared memory
    {"LSE_GN_VARIANT": "4", "LSE_SLAB_NB": "2"},
    {"LSE_GN_VARIANT": "4", "LSE_SLAB_GROUP": "2"},
    {"LSE_GN_VARIANT": "5"},                                    # tiles parked in tensor memory
    {"LSE_GN_VARIANT": "5", "LSE_GNM_SLOTS": "2"},
    {"LSE_GN_VARIANT": "7"},                                    # the whole grid on one sample at a time
    {"LSE_GN_VARIANT": "7", "LSE_GNS_SLOTS": "3"},
]


@pytest.mark.parametrize("cfg", GN_CONFIGS,
                         ids=["-".join(f"{k[7:]}{v}" for k, v in c.items()) for c in GN_CONFIGS])
@pytest.mark.parametrize("N,C,H,W,G", [(5, 64, 20, 20, 16), (3, 8, 5, 7, 4), (2, 6, 1, 1, 3)])
def test_gn_act_lse_variants(lib, env, cfg, N, C, H, W, G):
    for k, v in cfg.items():
        env.setenv(k, v)
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = lib.gn_act_lse_forward(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), G, 1e-5)
    ref = oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"gn {cfg} {N,C,H,W,G}")


def _non_finite_gn_input():
    """Four samples of y[., 16, 6, 7] (4 channels per group at G = 4): a NaN in sample 0
    group 1, +inf in sample 1 group 0, -inf in sample 2 group 2, sample 3 finite."""
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 16, 6, 7))
    y = inp["y"].clone()
    y[0, 5, 2, 3] = float("nan")
    y[1, 1, 0, 0] = float("inf")
    y[2, 10, 5, 6] = float("-inf")
    return y, inp["gamma"], inp["beta"]


@pytest.mark.parametrize("variant", ["0", "1", "2", "3", "4", "7"])
def test_gn_act_lse_non_finite(lib, env, variant):
    """A non-finite value makes its group's mean or variance NaN, so every channel of that
    group is NaN at every pixel and the sample's channel lse is NaN everywhere; the
    finite sample is unaffected (the oracle's plain definition, variance over all values)."""
    env.setenv("LSE_GN_VARIANT", variant)
    y, gamma, beta = _non_finite_gn_input()
    got = lib.gn_act_lse_forward(y.to(DEV), gamma.to(DEV), beta.to(DEV), 4, 1e-5).cpu()
    assert all(bool(torch.isnan(got[n]).all()) for n in range(3))
    assert not bool(torch.isnan(got[3]).any())
    assert_parity(got, oracle.gn_act_lse(y, gamma, beta, 4, 1e-5), f"non-finite y, variant {variant}")


@pytest.mark.parametrize("N,C,H,W,G", [
    (3, 64, 33, 40, 16),    # 6 tiles, the last with 40 pixels
    (2, 12, 16, 16, 3),     # 3 channel blocks: the two channel halves differ
    (1, 4, 2, 2, 1),        # one block of four channels, one 4-pixel tile
    (2, 32, 32, 32, 8),     # 8 tile buffers
    (7, 64, 20, 20, 4),     # 16 channels per group
    (6, 64, 126, 126, 16),  # the full image: 63 tiles per sample
    (6000, 4, 16, 16, 2),   # ~40 tiles per CTA: the announcement ring wraps
])
def test_gn_tmem_shapes(lib, env, N, C, H, W, G):
    """The tile queue with tiles parked in tensor memory on ragged and extreme shapes."""
    env.setenv("LSE_GN_VARIANT", "5")
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = lib.gn_act_lse_forward(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), G, 1e-5)
    ref = oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"gn tmem {N,C,H,W,G}")


@pytest.mark.parametrize("N,C,H,W,G,slots", [
    (3, 64, 33, 40, 16, 0),     # slices of 8 and 12 pixels
    (2, 12, 16, 16, 3, 0),      # 6 channels per apply half: pairs only, no batch of 8
    (1, 4, 2, 2, 1, 0),         # one quad: a grid of one CTA
    (2, 32, 32, 32, 8, 0),
    (7, 64, 20, 20, 4, 0),      # 16 channels per group
    (2, 64, 12, 12, 64, 0),     # one channel per group, 64 groups: both table lanes
    (2, 60, 10, 10, 15, 0),     # 15 groups of 4
    (6, 64, 126, 126, 16, 0),   # the full image: slices of 104 and 108 pixels
    (3, 64, 160, 152, 16, 0),   # slices of 160 pixels: two apply blocks (128 + 32)
    (50, 8, 16, 16, 2, 3),      # three slots: the ring wraps 16 times
])
def test_gn_sweep_shapes(lib, env, N, C, H, W, G, slots):
    """The whole grid on one sample at a time (slices of every channel in shared memory,
    grid-wide fp64 sums) on ragged and extreme shapes."""
    env.setenv("LSE_GN_VARIANT", "7")
    if slots:
        env.setenv("LSE_GNS_SLOTS", str(slots))
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    got = lib.gn_act_lse_forward(inp["y"].to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), G, 1e-5)
    ref = oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5)
    assert_parity(got, ref, f"gn sweep {N,C,H,W,G}")


def test_gn_tmem_non_finite(lib, env):
    """The non-finite samples of test_gn_act_lse_non_finite with 48 pixels (a multiple of
    4, so that the tensor-memory kernel takes them): NaN samples stay NaN everywhere."""
    env.setenv("LSE_GN_VARIANT", "5")
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(4, 16, 6, 8))
    y = inp["y"].clone()
    y[0, 5, 2, 3] = float("nan")
    y[1, 1, 0, 0] = float("inf")
    y[2, 10, 5, 6] = float("-inf")
    got = lib.gn_act_lse_forward(y.to(DEV), inp["gamma"].to(DEV), inp["beta"].to(DEV), 4, 1e-5).cpu()
    assert all(bool(torch.isnan(got[n]).all()) for n in range(3))
    assert not bool(torch.isnan(got[3]).any())
    assert_parity(got, oracle.gn_act_lse(y, inp["gamma"], inp["beta"], 4, 1e-5), "non-finite y, variant 5")


@pytest.mark.parametrize("variant", ["0", "1", "2", "3"])
@pytest.mark.parametrize("N,H,W,G", [(2, 3, 4, 512), (1, 2, 2, 8192), (2, 3, 3, 64)])
def test_gn_max_channels(lib, env, variant, N, H, W, G):
    """C = 8192, the largest accepted: the per-channel table fills 128 KB of shared memory
    in every kernel variant (HW = 9: the scalar kernels)."""
    env.setenv("LSE_GN_VARIANT", variant)
    C = 8192
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    y, g, b = (inp[k].to(DEV) for k in ("y", "gamma", "beta"))
    got = lib.gn_act_lse_forward(y, g, b, G, 1e-5).cpu()
    assert_parity(got, oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5), f"C=8192 G={G} v{variant}")
    for fn in ("group_norm", "gn_act_residual"):
        out = torch.full((N, C, H, W), float("nan"), device=DEV)
        getattr(lib, fn)(y, g, b, out, N, C, H * W, G, 1e-5)
        torch.cuda.synchronize()
        assert_parity(out.cpu(), getattr(oracle, fn)(inp["y"], inp["gamma"], inp["beta"], G, 1e-5),
                      f"{fn} C=8192 G={G} v{variant}")


@pytest.mark.parametrize("variant", ["0", "5", "7"])
def test_gn_act_lse_wide_range(lib, env, variant):
    """Large gamma and shifted data: z spans about [-60, 60] (tanh saturates),
    a non-zero mean exercises the statistics."""
    env.setenv("LSE_GN_VARIANT", variant)
    N, C, H, W, G = 2, 16, 20, 20, 4
    y = synth.normal((N, C, H, W), seed=77, mean=30.0, var=25.0)
    gamma = synth.uniform((C,), seed=78, lo=-12.0, hi=12.0)
    beta = synth.normal((C,), seed=79, var=4.0)
    got = lib.gn_act_lse_forward(y.to(DEV), gamma.to(DEV), beta.to(DEV), G, 1e-3)
    assert_parity(got, oracle.gn_act_lse(y, gamma, beta, G, 1e-3), "gn wide")


@pytest.mark.parametrize("variant", ["0", "5", "7"])
def test_gn_act_lse_large_mean_small_spread(lib, env, variant):
    """Groups whose mean (1e3) is 1e4 times their spread (std 0.1, so rstd ~ 10): z stays
    accurate (the mean is subtracted before scaling, and the tile-queue kernel merges its
    tiles' means relative to one of them), and the channel lse near 1e3 keeps within the
    relative part of the tolerance despite the rounding of the exponent's shift
    (m log2 e).  (Beyond a ratio of ~1e5 no fp32 GroupNorm is accurate: the mean itself
    is only known to half an ulp, e.g. 5e-4 at 1e4.)  40 x 40 pixels: 7 tiles of 256."""
    env.setenv("LSE_GN_VARIANT", variant)
    N, C, H, W, G = 2, 16, 40, 40, 4
    y = synth.normal((N, C, H, W), seed=81, mean=1.0e3, var=1.0e-2)
    gamma = synth.uniform((C,), seed=82, lo=0.5, hi=1.5)
    beta = synth.normal((C,), seed=83, var=0.1)
    got = lib.gn_act_lse_forward(y.to(DEV), gamma.to(DEV), beta.to(DEV), G, 1e-5)
    assert_parity(got, oracle.gn_act_lse(y, gamma, beta, G, 1e-5), "gn mean 1e3, std 0.1")


@pytest.mark.parametrize("variant", ["0", "5", "7"])
@pytest.mark.parametrize("scale", [1.0e3, 1.0e6, 1.0e15])
def test_gn_act_lse_large_values(lib, env, scale, variant):
    """y of magnitude up to 1e15 with channels far apart: the running max and its
    rescale carry the channel lse (terms span many binades).  32 x 32 pixels: 4 tiles."""
    env.setenv("LSE_GN_VARIANT", variant)
    N, C, H, W, G = 2, 24, 32, 32, 6
    y = synth.normal((N, C, H, W), seed=84) * scale
    gamma = synth.uniform((C,), seed=85, lo=0.5, hi=1.5)
    beta = synth.normal((C,), seed=86, var=0.1)
    got = lib.gn_act_lse_forward(y.to(DEV), gamma.to(DEV), beta.to(DEV), G, 1e-5)
    assert_parity(got, oracle.gn_act_lse(y, gamma, beta, G, 1e-5), f"gn scale {scale}")


@pytest.mark.parametrize("variant", ["0", "5", "7"])
def test_gn_act_lse_constant_group(lib, env, variant):
    """Zero variance in a group: z = beta exactly (eps keeps rstd finite).  20 x 20
    pixels: two tiles, whose merged M2 stays exactly 0."""
    env.setenv("LSE_GN_VARIANT", variant)
    y = torch.full((1, 4, 20, 20), 2.0)
    gamma = torch.ones(4)
    beta = torch.tensor([0.0, 0.5, -1.0, 2.0])
    got = lib.gn_act_lse_forward(y.to(DEV), gamma.to(DEV), beta.to(DEV), 2, 1e-5)
    assert_parity(got, oracle.gn_act_lse(y, gamma, beta, 2, 1e-5), "gn constant")


def test_gn_act_lse_misaligned(lib):
    N, C, H, W, G = 2, 8, 4, 8, 2
    inp = synth.make_inputs("gn_act_lse_128x64x126x126", shape=(N, C, H, W))
    y = _misaligned(inp["y"].to(DEV))
    out = _misaligned(torch.empty(N, 1, H, W, device=DEV))
    lib.gn_act_lse(y, inp["gamma"].to(DEV), inp["beta"].to(DEV), out, N, C, H * W, G, 1e-5)
    torch.cuda.synchronize()
    assert_parity(out.cpu(), oracle.gn_act_lse(inp["y"], inp["gamma"], inp["beta"], G, 1e-5),
                  "gn misaligned")


# ----------------------------------------------------------------------------- streams, host API

def test_side_stream_and_host_tensors(lib):
    x = synth.normal((64, 5000), seed=1)
    s = torch.cuda.Stream()
    xd = x.to(DEV)
    out = torch.empty_like(xd)
    with torch.cuda.stream(s):
        lib.log_softmax_lastdim(xd, out, 64, 5000, stream=s)
    s.synchronize()
    assert_parity(out.cpu(), oracle.log_softmax(x), "side stream")
    got = lib.log_softmax(x.pin_memory())   # host in, host out
    assert not got.is_cuda
    assert_parity(got, oracle.log_softmax(x), "host tensors")


def test_repeat_calls_are_deterministic(lib):
    x = synth.normal((40, 393216), seed=11, device=DEV)
    a = torch.empty_like(x)
    b = torch.empty_like(x)
    lib.log_softmax_lastdim(x, a, 40, 393216)
    lib.log_softmax_lastdim(x, b, 40, 393216)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_log_softmax_persistent_long_rows(lib):
    """More rows than resident clusters: each cluster loops over rows and refills
    its shared-memory slice while writing the previous row."""
    x = synth.normal((64, 393216), seed=12)
    assert_parity(_log_softmax(lib, x), oracle.log_softmax(x), "64 x 393216")


@pytest.mark.parametrize("rows,cols,chunk_mb,pinned", [
    (37, 100000, "1", True),      # many chunks, last one short
    (5, 393216, "1", False),      # pageable buffers, one row per chunk
    (300, 4099, "", True),        # one chunk, unaligned rows
    (9, 65536, "2", True),
])
def test_log_softmax_host_pipeline(lib, env, rows, cols, chunk_mb, pinned):
    """Host buffers in and out, pipelined through device staging buffers."""
    env.setenv("LSE_HOST_CHUNK_MB", chunk_mb)
    x = synth.normal((rows, cols), seed=rows + cols)
    if pinned:
        x = x.pin_memory()
    out = torch.full((rows, cols), float("nan"))
    if pinned:
        out = out.pin_memory()
    s = torch.cuda.current_stream()
    lib.log_softmax_lastdim_host(x, out, rows, cols, stream=s)
    s.synchronize()
    assert_parity(out, oracle.log_softmax(x), f"host pipeline {rows}x{cols}")
    got = lib.log_softmax(x)   # the convenience routes host tensors through the same entry
    assert not got.is_cuda
    assert_parity(got, oracle.log_softmax(x), "host convenience")
