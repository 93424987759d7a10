"""Host-side arithmetic of bench.py (no GPU): the e2e ceiling a host link allows."""
import pytest

import bench


def test_e2e_ceiling_both_directions():
    # 10 GB in and 10 GB out on a link doing 200 / 200 GB/s one way and 300 GB/s both ways:
    # the two directions at once bound the step at 20 GB / 300 GB/s
    link = {"h2d_gbs": 200.0, "d2h_gbs": 200.0, "both_gbs": 300.0}
    assert bench.e2e_ceiling(20e9, 10e9, 10e9, link) == pytest.approx(300.0)


def test_e2e_ceiling_one_direction_dominates():
    # a reduction: 4 GB in, 0.1 GB out; the copy in alone takes 4 / 200 s
    link = {"h2d_gbs": 200.0, "d2h_gbs": 190.0, "both_gbs": 340.0}
    assert bench.e2e_ceiling(4.1e9, 4e9, 0.1e9, link) == pytest.approx(4.1e9 / (4e9 / 200e9) / 1e9)


def test_e2e_ceiling_slow_return():
    # the way back is the slow one
    link = {"h2d_gbs": 200.0, "d2h_gbs": 50.0, "both_gbs": 240.0}
    assert bench.e2e_ceiling(2e9, 1e9, 1e9, link) == pytest.approx(2e9 / (1e9 / 50e9) / 1e9)


def test_oracle_on_threads():
    """The all-cores CPU baseline: the oracle on two threads, each on its own share."""
    import synth
    w = synth.WORKLOADS["log_softmax_256x4096"]
    sample = {"x": synth.normal((8, 4096), 2)}
    b, s, used, done = bench.time_oracle_threads(w, sample, 0.2, 1, 2)
    assert used == 2 and done >= 2 and b == done * 8 * 4096 and s > 0
    w = synth.WORKLOADS["gn_act_lse_128x64x126x126"]
    inp = synth.make_inputs(w, shape=(3, 64, 6, 6))
    b, s, used, done = bench.time_oracle_threads(w, inp, 0.2, 1, 8)
    assert used == 3 and done >= 3 and b > 0
