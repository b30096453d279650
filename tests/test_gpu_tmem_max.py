"""The TMEM load with a max reduction (tcgen05.ld.red ... .max.f32) returns, per thread, the maximum of the
32 columns it loads: the property the Index Branch max-pool and the Main Branch softmax maxima rely on.
Builds tests/tmem_max_probe.cu with nvcc for sm_103a and runs it (one warp, in-bounds)."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
def test_tmem_load_max_reduction():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "tmem_max_probe")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-o", exe,
                        os.path.join(HERE, "tmem_max_probe.cu")], check=True, capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "values mismatched 0 of 1024, reductions mismatched 0 of 32" in r.stdout, r.stdout
