"""Register budget of the main kernel's instances, from ptxas's own summary.

The main kernel runs 16 warps per SM, so every instance is held to 128
registers, and the allocation of these multi-path kernels moves with small
source changes. This compiles the kernel file for sm_103a with `-Xptxas -v`
(about 20 s, no GPU) and checks the spill bytes each instance is recorded
with: none for the linear, narrow sinc, nearest, height-map nearest and wide
sinc kernels, at most 8/8 bytes for the height map and 12/20 for the
height-map sinc kernel.
"""

import os
import re
import subprocess
import tempfile

import pytest

from domain_backprojection_sarbp_gb300 import build

KERNELS = os.path.join(build.CSRC, "sarbp_kernels.cu")

# instance -> (spill store bytes, spill load bytes) allowed
SPILL_BUDGET = {
    0: (0, 0),    # linear
    1: (0, 0),    # windowed sinc, narrow geometry
    2: (0, 0),    # nearest
    3: (8, 8),    # height map, linear
    4: (12, 20),  # height map, windowed sinc
    5: (0, 0),    # height map, nearest
    6: (0, 0),    # windowed sinc, wide geometry
}


@pytest.fixture(scope="module")
def ptxas_summary():
    try:
        cc = build.nvcc()
    except RuntimeError as e:
        pytest.skip(str(e))
    with tempfile.TemporaryDirectory() as d:
        cmd = [cc] + build.FLAGS + ["-Xptxas", "-v", "-c", KERNELS, "-o", os.path.join(d, "k.o")]
        out = subprocess.run(cmd, capture_output=True, text=True, check=True)
    text = out.stdout + out.stderr
    spills, regs = {}, {}
    current = None
    lines = text.splitlines()
    for i, line in enumerate(lines):
        m = re.search(r"Function properties for (\S+)", line)
        if m and i + 1 < len(lines):
            s = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", lines[i + 1])
            if s:
                spills[m.group(1)] = (int(s.group(1)), int(s.group(2)))
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            current = m.group(1)
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            regs[current] = int(m.group(1))
            current = None

    def instance(name):
        m = re.search(r"bp_kernelILi(\d+)E", name)
        return int(m.group(1)) if m else None

    by_instance = {}
    for name, r in regs.items():
        n = instance(name)
        if n is not None:
            by_instance[n] = (r, spills.get(name))
    return by_instance


def test_every_instance_is_compiled(ptxas_summary):
    assert sorted(ptxas_summary) == sorted(SPILL_BUDGET)


@pytest.mark.parametrize("n", sorted(SPILL_BUDGET))
def test_spills_within_budget(ptxas_summary, n):
    regs, spill = ptxas_summary[n]
    assert regs <= 128, (n, regs)
    assert spill is not None, n
    stores, loads = spill
    max_stores, max_loads = SPILL_BUDGET[n]
    assert stores <= max_stores and loads <= max_loads, (n, spill)
