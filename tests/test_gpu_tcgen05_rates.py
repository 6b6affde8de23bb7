"""Issue and completion rates of tcgen05.mma on one SM (needs a GB300 and nvcc).

The probe behind the prefill kernel's tile shapes and the measured-and-rejected experiments: an
M 128 N 128 K 16 MMA runs at the SM's dense bf16 rate, N 64 with both operands in shared memory
does not; changing accumulator, shape or operand layout between groups of MMAs costs nothing.
The pipe does not run ahead of the issuing thread: the attention order with each MMA's
descriptors built in the issue loop runs at about half the rate it reaches with them built
before the loop, and a second commit per group of MMAs slows the stream where one does not."""
import json
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tcgen05_mma_rates(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = tmp_path / "tcgen05_mma_rates"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-o", str(exe), os.path.join(HERE, "probes", "tcgen05_mma_rates.cu")],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120,
                         check=True).stdout
    print(out)
    rows = {r["mode"]: r for r in (json.loads(x) for x in out.splitlines() if x.startswith("{"))}
    assert sorted(rows) == list(range(11))
    assert all(r["status"] == 0 for r in rows.values())
    peak = 128 * 128 * 16 * 2 / 64  # one M128 N128 K16 MMA per 64 cycles: 8,192 flop/cycle
    assert rows[1]["flop_per_cycle"] > 0.85 * peak
    assert rows[2]["flop_per_cycle"] > 0.85 * peak
    # precomputed descriptors: the attention order and one commit per group at the mix's rate
    assert rows[8]["flop_per_cycle"] > 0.9 * rows[4]["flop_per_cycle"]
    assert rows[9]["flop_per_cycle"] > 0.9 * rows[4]["flop_per_cycle"]
