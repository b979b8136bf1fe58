"""The C ABI from C: tests/c_abi_check.c is compiled against include/qknr.h,
libqknr.so and the oracle's C library, then run on the GPU. It checks
qknr_apply against the oracle element by element, qknr_apply_host against
qknr_apply bit for bit, and qknr_apply_checked's position report, with no
Python between the caller and the kernels."""
import os
import shutil
import subprocess
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_c_consumer(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    import qk_rmsnorm_rope_gb300 as q
    lib_dir = os.path.dirname(q.library_path())
    oracle_dir = os.path.dirname(oracle.build())
    exe = str(tmp_path / "c_abi_check")
    subprocess.run([nvcc, "-O2", os.path.join(ROOT, "tests", "c_abi_check.c"), "-I",
                    os.path.join(ROOT, "include"), "-L", lib_dir, "-lqknr", "-L", oracle_dir,
                    "-lqknr_oracle", "-lm", "-Xlinker", f"-rpath,{lib_dir}:{oracle_dir}", "-o", exe],
                   check=True, capture_output=True, text=True, timeout=600)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "all passed" in r.stdout
