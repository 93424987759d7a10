"""The special-function rates behind the bench's roofline of the GroupNorm chain
(bench.SFU_EX2_PER_CLK_PER_SM, bench.SFU_RCP_PER_CLK_PER_SM), measured on the GPU
at hand by a throughput kernel (tests/gpu_probes/sfu_rates.cu) at the device's
maximum SM clock: the base-2 exponential runs at twice the reciprocal's rate.
The timed kernel runs at the clock the GPU chooses, so the check allows 20 %."""
import os
import shutil
import subprocess

import pytest

import bench

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_sfu_rates(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "sfu_rates")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    os.path.join(HERE, "gpu_probes", "sfu_rates.cu")], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout
    rates = dict(line.split()[:2] for line in out.splitlines() if line.split()[0] in ("ex2", "rcp"))
    ex2, rcp = float(rates["ex2"]), float(rates["rcp"])
    assert abs(ex2 - bench.SFU_EX2_PER_CLK_PER_SM) <= 0.2 * bench.SFU_EX2_PER_CLK_PER_SM, out
    assert abs(rcp - bench.SFU_RCP_PER_CLK_PER_SM) <= 0.2 * bench.SFU_RCP_PER_CLK_PER_SM, out
