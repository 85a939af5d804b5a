"""The C ABI used from plain C: tests/c_client/ssim_client.c, compiled with gcc
against include/gbssim.h, the built libgbssim.so and the CUDA runtime, runs
the forward, the stored and the recompute backward on a small pair that it
generates from a closed formula; its printed mean and gradients must match
the oracle on the same pair, restated here."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from test_gpu_parity import GRAD_RTOL, MEAN_TOL

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pair():
    C, H, W = 2, 24, 30
    c, i, j = np.meshgrid(np.arange(C), np.arange(H), np.arange(W), indexing="ij")
    x = (0.5 + 0.4 * np.sin(0.37 * i + 0.11 * j + c)).astype(np.float32)
    y = (x.astype(np.float64) + 0.05 * np.cos(0.23 * i - 0.19 * j + 2.0 * c)).astype(np.float32)
    return x[None].astype(np.float64), y[None].astype(np.float64)


def test_c_client_matches_the_oracle(oracle_mod, tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _build

    lib = _build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "ssim_client")
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-O2", "-o", exe, os.path.join(ROOT, "tests", "c_client", "ssim_client.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", libdir, "-l:" + os.path.basename(lib), "-L", os.path.join(cuda, "lib64"),
                    "-lcudart", "-lm", f"-Wl,-rpath,{libdir}:{os.path.join(cuda, 'lib64')}"],
                   check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    vals = np.array([float(v) for v in out])
    x, y = _pair()
    n = x.size
    assert vals.size == 1 + 2 * n
    ref_mean = oracle_mod.ssim2d(x, y, "valid")
    g1, _ = oracle_mod.ssim2d_grad(x, y, [-1.0], "valid", want_grad2=False)
    assert abs(vals[0] - ref_mean[0]) <= MEAN_TOL
    for k, label in ((1, "stored"), (1 + n, "recompute")):
        g = vals[k:k + n].reshape(x.shape)
        err = np.max(np.abs(g - g1)) / np.max(np.abs(g1))
        assert err <= GRAD_RTOL, f"{label}: {err:.3e}"
