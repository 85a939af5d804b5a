"""GPU parity of the per-octave stage (ssim_pyramid) against the CPU oracle.

Every call goes through the C ABI.  Bars: the per-image means of l, cs and S
within 1e-5 of the oracle's (the loss's mean bar); the maps of octave 0 within
5e-6 absolute (the 2D SSIM map's bar), those of the downscaled octaves within
1e-5.  The kernels shift each window's values by one value per 11-row band and
8-column group, exact in real arithmetic, and take cs as 1 - D / (sigma11 +
sigma22 + C2) with D from the blurred squared difference of the two images,
which carries no rounding of their common level.  Measured at most 5.1e-6 at
the downscaled octaves of the 1080p blob render, 2.5e-6 at octave 0.  Bands lie
on one 11-row grid per image, so the values do not depend on the launch plan.
The GPU downscales in float32, the oracle in double from the same float32
inputs.
"""
import numpy as np
import pytest

from workloads import make_inputs, uniform_pair

pytestmark = pytest.mark.gpu

MEAN_TOL = 1e-5
MAP_TOL = 5e-6           # octave 0
OCTAVE_MAP_TOL = 1e-5    # octaves 1, 2, ... (downscaled: smaller features)


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    _abi.load()
    return torch.device("cuda:0")


def _gpu(dev, x, y, padding, octaves, want_maps=True):
    import torch

    import differentiable_image_quality_gb300 as pkg

    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    means, maps = pkg.ssim_pyramid(tx, ty, padding, octaves, want_maps=want_maps)
    torch.cuda.synchronize()
    return means.cpu().numpy(), None if maps is None else [m.cpu().numpy() for m in maps]


def _check(got, ref, octaves, label):
    gm, gmaps = got
    rm, rmaps = ref
    assert gm.shape == (octaves, 3, rm.shape[2])
    dm = np.max(np.abs(gm.astype(np.float64) - rm))
    assert dm <= MEAN_TOL, f"{label}: means off by {dm:.3e}"
    if gmaps is not None:
        for o in range(octaves):
            assert gmaps[o].shape == rmaps[o].shape, (label, o)
            assert np.all(np.isfinite(gmaps[o])), f"{label}: octave {o} map not finite"
            d = np.max(np.abs(gmaps[o].astype(np.float64) - rmaps[o]))
            tol = MAP_TOL if o == 0 else OCTAVE_MAP_TOL
            assert d <= tol, f"{label}: octave {o} maps off by {d:.3e}"


CASES = [
    # (shape, padding, octaves, seed): ragged downscales, several strips, tiny octaves
    ((1, 3, 64, 64), "valid", 2, 1),
    ((2, 2, 45, 50), "valid", 3, 2),
    ((1, 1, 13, 9), "same", 4, 3),
    ((1, 2, 37, 301), "same", 3, 4),
    ((2, 1, 90, 263), "valid", 4, 5),
    ((1, 1, 1, 1), "same", 2, 6),
    ((3, 1, 11, 11), "valid", 1, 7),
    ((1, 2, 100, 140), "same", 7, 8),    # two octave-chain launches (5 + 1 octaves)
    ((1, 1, 300, 517), "same", 10, 9),   # two chain launches (5 + 4), two octave launches (8 + 2)
    ((2, 1, 70, 33), "same", 6, 10),     # octave tiles wider than the image
]


@pytest.mark.parametrize("shape,padding,octaves,seed", CASES)
def test_pyramid_parity_small(dev, oracle_mod, shape, padding, octaves, seed):
    x, y = uniform_pair(shape, 900 + seed, std=0.08)
    got = _gpu(dev, x, y, padding, octaves)
    ref = oracle_mod.ssim2d_pyramid(x, y, padding, octaves, want_maps=True)
    _check(got, ref, octaves, f"{shape} {padding} x{octaves}")


@pytest.mark.parametrize("name,padding", [("splat1080_valid", "valid"), ("splat1080_same", "same")])
def test_pyramid_parity_1080p_six_octaves(dev, oracle_mod, name, padding):
    """The 1080p splatting pair through six octaves (1080 x 1920 .. 34 x 60)."""
    x, y = make_inputs(name)
    got = _gpu(dev, x, y, padding, 6)
    ref = oracle_mod.ssim2d_pyramid(x, y, padding, 6, want_maps=True)
    _check(got, ref, 6, f"{name} x6")


def test_pyramid_octave_zero_matches_forward(dev):
    import torch

    import differentiable_image_quality_gb300 as pkg

    x, y = uniform_pair((2, 3, 70, 131), 77, std=0.05)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    mean = torch.empty(2, device=dev)
    pkg.ssim_fwd(tx, ty, "same", mean)
    means, _ = pkg.ssim_pyramid(tx, ty, "same", 3)
    torch.cuda.synchronize()
    assert np.max(np.abs(means[0, 2].cpu().numpy() - mean.cpu().numpy())) < 1e-6


def test_pyramid_deterministic_and_rejects_bad_octaves(dev):
    import torch

    import differentiable_image_quality_gb300 as pkg

    x, y = uniform_pair((1, 2, 100, 120), 31, std=0.1)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    a, ma = pkg.ssim_pyramid(tx, ty, "valid", 3, want_maps=True)
    b, mb = pkg.ssim_pyramid(tx, ty, "valid", 3, want_maps=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    for u, v in zip(ma, mb):
        assert torch.equal(u, v)
    with pytest.raises(ValueError):
        pkg.ssim_pyramid(tx, ty, "valid", 5)  # octave 4 would be 7 x 8 < 11
    with pytest.raises(ValueError):
        pkg.ssim_pyramid(tx, ty, "valid", 0)
