"""Staging the selected K/V rows: cp.async row gathers against the TMA
tile::gather4 load (four rows of 64 columns per instruction), on random
256-byte rows of an L2-resident tensor, the access pattern of the sparse
attention kernels. Both must gather the same bytes; the rate each reaches
per SM is printed (pytest -s): the measurement behind the attention kernels'
use of cp.async for this step."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu


def test_gather_methods_agree_and_report_rates(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gpu_probes", "gather_rows.cu")
    exe = str(tmp_path / "gather_rows")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe, src],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "cp.async, 7 warps" in r.stdout and "TMA gather4" in r.stdout
