"""The polynomial exp2 of the attention softmax (two lanes per paired instruction),
against CUDA's exp2f: maximum relative error below 1e-4 over [-125, 8] (the fitted bound
is 7.5e-5; exp2f itself is accurate to a couple of fp32 ulps), both lanes identical, and a
negligible value for -inf."""
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_soft_exp2_matches_exp2f(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    exe = tmp_path / "soft_exp2_check"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    os.path.join(HERE, "cuda", "soft_exp2_check.cu"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    err = float(out[out.index("max_rel_err") + 1])
    neg_inf = float(out[out.index("neg_inf") + 1])
    assert err < 1e-4, out
    assert int(out[out.index("lane_mismatch") + 1]) == 0, out
    assert 0.0 <= neg_inf < 1e-37
