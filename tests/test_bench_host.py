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


def test_clock_summary_keeps_the_timed_window():
    # samples every 2 ms; the window holds four of them, one with a power-cap reason
    samples = [(0.000 + 0.002 * i, 2070.0 - (i == 7) * 300, 2070.0, ["sw_power_cap"] if i == 6 else [], 900.0 + i)
               for i in range(20)]
    c = bench.summarize_clocks(samples, [(0.0095, 0.0155)])
    assert c["samples"] == 3 and c["window"] == "timed region"
    assert c["sm_mhz"] == 2070.0 and c["sm_mhz_min"] == 1770.0 and c["reasons"] == ["sw_power_cap"]
    assert c["power_w_max"] == 907.0
    # two windows are pooled
    c = bench.summarize_clocks(samples, [(0.0, 0.001), (0.037, 0.039)])
    assert c["samples"] == 2


def test_clock_summary_without_samples_in_the_window():
    samples = [(1.0, 1900.0, 2070.0, [], None)]
    c = bench.summarize_clocks(samples, [(5.0, 6.0)])
    assert c["samples"] == 1 and c["window"].startswith("whole run")
    assert bench.summarize_clocks([], [(0.0, 1.0)])["samples"] == 0


def test_conv_chain_counts_the_method_bytes():
    import synth
    w = synth.WORKLOADS["conv_gn_act_lse_128x8x128x128"]
    # x once, weights + bias + gamma + beta, out [128, 126, 126]
    assert bench.algorithmic_bytes(w) == 4 * (128 * 8 * 128 * 128 + 64 * (72 + 3) + 128 * 126 * 126)
    assert bench.design_bytes(w) - bench.algorithmic_bytes(w) == 8 * 128 * 64 * 126 * 126
    assert bench.conv_flops(w) == 2 * 128 * 64 * 126 * 126 * 72
