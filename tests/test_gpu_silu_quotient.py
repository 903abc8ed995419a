"""The conv's SiLU forms sigmoid through the quotient t / (1 + t) with the
hardware's approximate reciprocal and one correction (Markstein, IBM J. Res.
Dev. 34, 1990). The oracle's fp32 mirror takes that quotient as an IEEE
division, so the two agree bit for bit only if the step is correctly
rounded for every t the exp can produce. This test runs the library's own
step (silu_negquot in common.cuh) over every float t in [0, 1] on the GPU
and requires no difference from the IEEE quotient."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gated_deltanet_linear_14_gb300", "csrc")


@pytest.mark.gpu
def test_silu_quotient_correctly_rounded_for_every_t(tmp_path):
    from gated_deltanet_linear_14_gb300 import build as gbuild
    exe = str(tmp_path / "silu_quotient_check")
    src = os.path.join(ROOT, "tests", "cuda", "silu_quotient_check.cu")
    cmd = [gbuild.nvcc()] + gbuild.ARCH + gbuild.NVCC_FLAGS + [src, "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    m = re.search(r"values (\d+) differences (\d+)", out)
    assert m, out
    assert int(m.group(1)) == 0x3F800001
    assert int(m.group(2)) == 0, out
