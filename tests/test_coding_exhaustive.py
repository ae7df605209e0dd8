"""The E4M3 coding routine every quantizer uses, checked on the GPU against
CUDA's correctly rounded division on every (BF16 x, BF16 amax) pair (2^31
cases): the whole input domain of the weight, activation and KV quantizers."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_coding_matches_division_on_whole_domain(tmp_path, W):
    exe = str(tmp_path / "check_coding")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    os.path.join(HERE, "cuda", "check_coding.cu"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
