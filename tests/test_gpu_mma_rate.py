"""Rate of one tcgen05.mma kind::f16 instruction by shape: M = 128 with
N = 128 (the shape of every GEMM in the attention kernels, whose N is the
128-key tile or d = 128) against N = 256, operands in shared memory or A in
TMEM. The per-instruction rates are printed (pytest -s): the measurement
behind the attention kernels' tensor ceiling."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu


def test_mma_rate_probe_runs_and_accumulates_zero(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gpu_probes", "mma_rate.cu")
    exe = str(tmp_path / "mma_rate")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe, src],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    for name in ("ss N=128", "ss N=256", "ts N=128", "ts N=256"):
        assert name in r.stdout
