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
