"""Pins of the oracle's per-octave stage (2x downscale, l / cs / S maps).

The ssimulacra2 hand-off page runs, per octave of a 2x pyramid, a blur, the
pointwise sigma11 / sigma22 / sigma12 and a three-output error-map kernel; it
prints no formula for the downscale or the maps.  The oracle reads the
downscale as the 2x2 box mean (ragged edges over their in-range pixels) and
the maps as SSIM's luminance term l, contrast-structure term cs and S = l * cs.
These checks tie that reading to things outside the oracle:

* the downscale against a hand-worked example and torch's avg_pool2d with
  ceil_mode (which averages a ragged window over its in-range pixels);
* l and cs against closed forms (x = y gives 1 and 1; constant images give
  the luminance formula and cs = 1; y = x + k gives cs = 1), against S from
  the oracle's SSIM map, and against a torch float64 conv2d statement;
* the whole pyramid against avg_pool2d + conv2d octave by octave.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy import ndimage

from workloads import uniform_pair

SIGMA = 1.5
C1 = 0.01**2
C2 = 0.03**2


def rel_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def torch_pool(x):
    """2x2 means with ragged windows averaged over their in-range pixels."""
    t = torch.from_numpy(np.asarray(x, np.float64))
    return F.avg_pool2d(t, 2, 2, ceil_mode=True).numpy()


def torch_components(x, y, padding):
    """(l, cs) maps of NCHW float64 arrays with conv2d of the sampled Gaussian."""
    w = ndimage.gaussian_filter1d(np.eye(11)[5], SIGMA, mode="constant", truncate=5.0 / SIGMA)
    C = x.shape[1]
    win = torch.from_numpy(np.outer(w, w))[None, None].repeat(C, 1, 1, 1)
    pad = 0 if padding == "valid" else 5
    tx, ty = torch.from_numpy(x), torch.from_numpy(y)

    def blur(t):
        return F.conv2d(t, win, padding=pad, groups=C)

    mu1, mu2 = blur(tx), blur(ty)
    s11 = blur(tx * tx) - mu1 * mu1
    s22 = blur(ty * ty) - mu2 * mu2
    s12 = blur(tx * ty) - mu1 * mu2
    l = (2 * mu1 * mu2 + C1) / (mu1 * mu1 + mu2 * mu2 + C1)
    cs = (2 * s12 + C2) / (s11 + s22 + C2)
    return l.numpy(), cs.numpy()


# -------------------------------------------------------------- downscale

def test_downscale_worked_example(oracle_mod):
    # 3 x 5 plane 0..14: blocks (0,0) = (0+1+5+6)/4, (0,2) = (4+9)/2,
    # (1,0) = (10+11)/2, (1,2) = 14 alone
    out = oracle_mod.downscale2x(np.arange(15.0).reshape(3, 5))
    np.testing.assert_array_equal(out, [[3.0, 5.0, 6.5], [10.5, 12.5, 14.0]])


@pytest.mark.parametrize("shape", [(8, 8), (7, 10), (1, 1), (1, 5), (5, 1), (13, 17)])
def test_downscale_matches_avg_pool_ceil(oracle_mod, shape):
    f = np.random.default_rng(11).random(shape)
    ref = torch_pool(f[None, None])[0, 0]
    assert ref.shape == ((shape[0] + 1) // 2, (shape[1] + 1) // 2)
    assert np.max(np.abs(oracle_mod.downscale2x(f) - ref)) < 1e-15


def test_downscale_keeps_constants_and_even_sums(oracle_mod):
    assert np.all(oracle_mod.downscale2x(np.full((9, 6), 0.375)) == 0.375)
    f = np.random.default_rng(2).random((10, 12))
    assert abs(4.0 * oracle_mod.downscale2x(f).sum() - f.sum()) < 1e-12


# ------------------------------------------------------------- components

@pytest.mark.parametrize("padding", ["valid", "same"])
def test_components_of_identical_images_are_one(oracle_mod, padding):
    x, _ = uniform_pair((2, 2, 17, 14), 5, std=0.0)
    means, maps = oracle_mod.ssim2d_components(x, x, padding, want_maps=True)
    assert np.max(np.abs(maps - 1.0)) < 1e-12
    assert np.max(np.abs(means - 1.0)) < 1e-12


def test_components_constant_images_closed_form(oracle_mod):
    a, b = 0.3, 0.7
    x = np.full((1, 1, 15, 16), a)
    y = np.full((1, 1, 15, 16), b)
    means, maps = oracle_mod.ssim2d_components(x, y, "valid", want_maps=True)
    lum = (2 * a * b + C1) / (a * a + b * b + C1)
    assert np.max(np.abs(maps[0] - lum)) < 1e-12
    assert np.max(np.abs(maps[1] - 1.0)) < 1e-9   # sigma terms vanish: cs = C2 / C2
    assert abs(means[2, 0] - lum) < 1e-9


def test_components_shifted_copy_has_unit_cs(oracle_mod):
    x, _ = uniform_pair((1, 2, 19, 21), 8, std=0.0)
    y = np.asarray(x, np.float64) * 0.5 + 0.1
    z = y + 0.2
    _, maps = oracle_mod.ssim2d_components(y, z, "valid", want_maps=True)
    assert np.max(np.abs(maps[1] - 1.0)) < 1e-9


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_components_product_is_the_ssim_map(oracle_mod, padding):
    x, y = uniform_pair((2, 3, 18, 23), 9, std=0.1)
    means, maps = oracle_mod.ssim2d_components(x, y, padding, want_maps=True)
    ref_mean, ref_map = oracle_mod.ssim2d(x, y, padding, want_map=True)
    assert np.max(np.abs(maps[0] * maps[1] - ref_map)) < 1e-13
    assert np.max(np.abs(maps[2] - ref_map)) < 1e-13
    assert np.max(np.abs(means[2] - ref_mean)) < 1e-13
    np.testing.assert_allclose(means[0], maps[0].mean(axis=(1, 2, 3)), rtol=0, atol=1e-13)


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_components_match_torch_conv2d(oracle_mod, padding):
    x, y = uniform_pair((1, 2, 21, 17), 12, std=0.08)
    _, maps = oracle_mod.ssim2d_components(x, y, padding, want_maps=True)
    l, cs = torch_components(np.asarray(x, np.float64), np.asarray(y, np.float64), padding)
    assert np.max(np.abs(maps[0] - l)) < 1e-11
    assert np.max(np.abs(maps[1] - cs)) < 1e-9


# ---------------------------------------------------------------- pyramid

@pytest.mark.parametrize("padding,hw,octaves", [("valid", (45, 50), 3), ("same", (13, 9), 4)])
def test_pyramid_matches_pool_and_conv(oracle_mod, padding, hw, octaves):
    x, y = uniform_pair((2, 2) + hw, 21, std=0.07)
    means, maps = oracle_mod.ssim2d_pyramid(x, y, padding, octaves, want_maps=True)
    assert means.shape == (octaves, 3, 2)
    tx, ty = np.asarray(x, np.float64), np.asarray(y, np.float64)
    for o in range(octaves):
        if o:
            tx, ty = torch_pool(tx), torch_pool(ty)
        l, cs = torch_components(tx, ty, padding)
        assert maps[o].shape[-2:] == l.shape[-2:]
        assert np.max(np.abs(maps[o][0] - l)) < 1e-11
        assert np.max(np.abs(maps[o][1] - cs)) < 1e-8
        np.testing.assert_allclose(means[o][2], (l * cs).mean(axis=(1, 2, 3)), rtol=0, atol=1e-9)


def test_pyramid_octave_zero_is_the_forward(oracle_mod):
    x, y = uniform_pair((1, 3, 30, 26), 3, std=0.05)
    means = oracle_mod.ssim2d_pyramid(x, y, "valid", 1)
    assert np.max(np.abs(means[0, 2] - oracle_mod.ssim2d(x, y, "valid"))) < 1e-14
