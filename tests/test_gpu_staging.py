"""The two ways the 2D and 3D kernels stage their inputs, and the bounded
staging wait.

On 16-byte aligned images with W % 4 == 0 the kernels stage rows and slice
tiles with tensor copies (one thread per block issues them; a transaction
barrier tracks them) -- in 3D the XY statistics kernel only in valid padding,
the adjoint kernel in both (its tiles of the derivative field start at
negative coordinates in same padding); otherwise, or when the staging hook asks
for it, every thread issues cp.async copies.  Both must give the oracle's results.  A wait for a tensor copy is
bounded: when it runs out, the kernel's blocks stop, the device records the
failure, the affected means come out NaN, and the context stays usable.  The
hook's mode 2 makes every wait run out by announcing 16 bytes more than the
copies deliver; no fault is involved.  The hook exists only in the test build
of the library (libgbssim_test.so), which these tests load.
"""
import ctypes

import numpy as np
import pytest

from test_gpu_parity import _assert_parity, _oracle, _run
from workloads import dl_vector, make_inputs, uniform_pair

pytestmark = pytest.mark.gpu

STAGING_TIMEOUT = 1  # GBSSIM_DEV_STAGING_TIMEOUT


@pytest.fixture(scope="module")
def lib():
    """The test build of the library (the staging hook is not part of the
    product library); every package call in this module goes to it."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    with _abi.using_test_library() as test_lib:
        yield test_lib


def _status(lib):
    flags = ctypes.c_uint(0xFFFFFFFF)
    assert lib.gbssim_device_status(ctypes.byref(flags)) == 0
    return flags.value


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape,padding", [((1, 3, 64, 64), "valid"), ((1, 3, 64, 64), "same"),
                                           ((2, 1, 129, 12), "valid"),
                                           ((1, 2, 130, 236), "same"),
                                           ((1, 1, 75, 500), "valid")])
def test_both_staging_paths_match_the_oracle(lib, oracle_mod, shape, padding, mode):
    import torch

    x, y = uniform_pair(shape, 950 + shape[3], std=0.08)
    dl = np.linspace(-1.0, 0.5, shape[0])
    ref = _oracle(oracle_mod, x, y, dl, padding, True, want_map=True)
    lib.gbssim_tune_staging(mode)
    try:
        for path in ("saved", "recompute"):
            got = _run(torch.device("cuda:0"), x, y, dl, padding, True, path, want_map=True)
            _assert_parity(got, ref, True, f"mode {mode} {shape} {padding} {path}")
    finally:
        lib.gbssim_tune_staging(0)


def test_cp_async_staging_on_the_1080p_pair(lib, oracle_mod):
    import torch

    x, y = make_inputs("splat1080_valid")
    dl = dl_vector("splat1080_valid")
    ref = _oracle(oracle_mod, x, y, dl, "valid", False)
    lib.gbssim_tune_staging(1)
    try:
        got = _run(torch.device("cuda:0"), x, y, dl, "valid", False, "saved")
    finally:
        lib.gbssim_tune_staging(0)
    _assert_parity(got, ref, False, "cp.async staging, 1080p")


def test_staging_wait_runs_out_and_the_context_survives(lib, oracle_mod):
    import torch

    dev = torch.device("cuda:0")
    assert _status(lib) == 0, "an earlier call recorded a staging timeout"
    x, y = uniform_pair((2, 1, 64, 64), 990, std=0.08)
    dl = np.array([-1.0, 0.5])
    lib.gbssim_tune_staging(2)
    try:
        stalled = _run(dev, x, y, dl, "valid", False, "saved")
    finally:
        lib.gbssim_tune_staging(0)
    assert _status(lib) & STAGING_TIMEOUT
    assert np.all(np.isnan(stalled["mean"]))
    assert _status(lib) == 0  # reading the status cleared it
    # the same call without the stall, on the same context
    got = _run(dev, x, y, dl, "valid", False, "saved")
    ref = _oracle(oracle_mod, x, y, dl, "valid", False)
    _assert_parity(got, ref, False, "after a staging timeout")
    assert _status(lib) == 0


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape,padding", [((1, 1, 13, 20, 36), "valid"),
                                           ((2, 1, 12, 12, 12), "valid"),
                                           ((1, 1, 13, 20, 36), "same"),
                                           ((1, 2, 7, 24, 16), "same")])
def test_both_3d_staging_paths_match_the_oracle(lib, oracle_mod, shape, padding, mode):
    import torch

    x, y = uniform_pair(shape, 970 + shape[4], std=0.08)
    dl = np.linspace(-1.0, 0.5, shape[0])
    ref = _oracle(oracle_mod, x, y, dl, padding, True, want_map=True)
    lib.gbssim_tune_staging(mode)
    try:
        for path in ("saved", "recompute"):
            got = _run(torch.device("cuda:0"), x, y, dl, padding, True, path, want_map=True)
            _assert_parity(got, ref, True, f"3D mode {mode} {shape} {padding} {path}")
    finally:
        lib.gbssim_tune_staging(0)


def test_3d_staging_wait_runs_out_and_the_context_survives(lib, oracle_mod):
    import torch

    dev = torch.device("cuda:0")
    assert _status(lib) == 0, "an earlier call recorded a staging timeout"
    x, y = uniform_pair((1, 1, 14, 16, 16), 991, std=0.08)
    dl = np.array([-1.0])
    lib.gbssim_tune_staging(2)
    try:
        stalled = _run(dev, x, y, dl, "valid", False, "saved")
    finally:
        lib.gbssim_tune_staging(0)
    assert _status(lib) & STAGING_TIMEOUT
    assert np.all(np.isnan(stalled["mean"]))
    assert _status(lib) == 0
    got = _run(dev, x, y, dl, "valid", False, "saved")
    ref = _oracle(oracle_mod, x, y, dl, "valid", False)
    _assert_parity(got, ref, False, "3D after a staging timeout")
    assert _status(lib) == 0


def test_pyramid_staging_wait_runs_out_and_the_context_survives(lib, oracle_mod):
    """The per-octave stage's one launch for all octaves takes the same failure
    path: every octave's means come out NaN, then the same call recovers."""
    import torch

    import differentiable_image_quality_gb300 as pkg

    dev = torch.device("cuda:0")
    assert _status(lib) == 0, "an earlier call recorded a staging timeout"
    x, y = uniform_pair((1, 2, 64, 64), 992, std=0.08)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    lib.gbssim_tune_staging(2)
    try:
        stalled, _ = pkg.ssim_pyramid(tx, ty, "valid", 2)
        torch.cuda.synchronize()
    finally:
        lib.gbssim_tune_staging(0)
    assert _status(lib) & STAGING_TIMEOUT
    assert np.all(np.isnan(stalled.cpu().numpy()))
    assert _status(lib) == 0
    means, _ = pkg.ssim_pyramid(tx, ty, "valid", 2)
    ref = oracle_mod.ssim2d_pyramid(x, y, "valid", 2)
    assert np.max(np.abs(means.cpu().numpy() - ref)) <= 1e-5
    assert _status(lib) == 0
