"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each check ties one part of the oracle to mathematics or to an independent
library routine, chosen so that a plausible slip (a dropped constant, a wrong
sign, a shifted or transposed index, a wrong normaliser) fails at least one:

* the window against scipy's sampled-Gaussian filter, and its symmetry / sum;
* the direct 2D/3D blur against scipy.ndimage.gaussian_filter (zero padding),
  torch's float64 conv2d, and a separable numpy recomputation;
* the adjoint against the identity <B u, v> = <u, B^T v> and torch's
  conv_transpose2d (the "full" correlation named in TriSSIM README, "How it works");
* SSIM against closed forms: SSIM(x, x) = 1, symmetry, constant images, a
  constant-plus-image pair, a scaled pair y = a*x, and x constant;
* the derivatives and the chain rule against central finite differences and
  torch float64 autograd; grad = 0 at y = x; grad2(x, y) = grad1(y, x).
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
TRUNC = 5.0 / SIGMA  # scipy's radius = int(truncate * sigma + 0.5) = 5 -> 11 taps


def scipy_blur(f, padding):
    """Zero-padded Gaussian filter of scipy; 'valid' keeps the windows that fit."""
    out = ndimage.gaussian_filter(np.asarray(f, np.float64), SIGMA, mode="constant", cval=0.0,
                                  truncate=TRUNC)
    if padding == "valid":
        out = out[(slice(5, -5),) * out.ndim]
    return out


def rel_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------------- window

def test_window_matches_scipy_sampled_gaussian(oracle_mod):
    w = oracle_mod.gauss_window()
    impulse = np.zeros(41)
    impulse[20] = 1.0
    ref = ndimage.gaussian_filter1d(impulse, SIGMA, mode="constant", truncate=TRUNC)[15:26]
    assert np.max(np.abs(w - ref)) < 1e-15
    assert abs(w.sum() - 1.0) < 1e-15
    np.testing.assert_array_equal(w, w[::-1])
    assert np.argmax(w) == 5 and np.all(np.diff(w[:6]) > 0)


# ------------------------------------------------------------------- blur

@pytest.mark.parametrize("padding", ["valid", "same"])
@pytest.mark.parametrize("shape", [(11, 11), (16, 23), (37, 12)])
def test_blur2d_matches_scipy(oracle_mod, padding, shape):
    f = np.random.default_rng(7).random(shape)
    assert rel_err(oracle_mod.blur2d(f, padding), scipy_blur(f, padding)) < 1e-13


def test_blur2d_same_tiny_images(oracle_mod):
    for shape in [(1, 1), (1, 7), (3, 2), (6, 6)]:
        f = np.random.default_rng(1).random(shape)
        assert rel_err(oracle_mod.blur2d(f, "same"), scipy_blur(f, "same")) < 1e-13


def test_blur2d_valid_matches_torch_conv2d_and_separable(oracle_mod):
    f = np.random.default_rng(3).random((29, 34))
    w = ndimage.gaussian_filter1d(np.eye(11)[5], SIGMA, mode="constant", truncate=TRUNC)
    win = torch.from_numpy(np.outer(w, w))[None, None]
    ref = F.conv2d(torch.from_numpy(f)[None, None], win)[0, 0].numpy()
    out = oracle_mod.blur2d(f, "valid")
    assert rel_err(out, ref) < 1e-13
    # separable: rows then columns, each a 1D valid correlation
    rows = np.stack([np.correlate(r, w, "valid") for r in f])
    sep = np.stack([np.correlate(c, w, "valid") for c in rows.T]).T
    assert rel_err(out, sep) < 1e-13


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_blur3d_matches_scipy(oracle_mod, padding):
    f = np.random.default_rng(11).random((13, 12, 15))
    assert rel_err(oracle_mod.blur3d(f, padding), scipy_blur(f, padding)) < 1e-13


# ---------------------------------------------------------------- adjoint

@pytest.mark.parametrize("padding", ["valid", "same"])
@pytest.mark.parametrize("shape", [(11, 11), (19, 26), (12, 40)])
def test_adjoint_identity_2d(oracle_mod, padding, shape):
    rng = np.random.default_rng(5)
    u = rng.standard_normal(shape)
    Ho, Wo = (oracle_mod.out_extent(s, padding) for s in shape)
    v = rng.standard_normal((Ho, Wo))
    lhs = float(np.sum(oracle_mod.blur2d(u, padding) * v))
    rhs = float(np.sum(u * oracle_mod.blur2d_adjoint(v, *shape, padding)))
    assert abs(lhs - rhs) <= 1e-13 * max(abs(lhs), 1.0)


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_adjoint_identity_3d(oracle_mod, padding):
    rng = np.random.default_rng(6)
    shape = (12, 13, 11)
    u = rng.standard_normal(shape)
    v = rng.standard_normal(tuple(oracle_mod.out_extent(s, padding) for s in shape))
    lhs = float(np.sum(oracle_mod.blur3d(u, padding) * v))
    rhs = float(np.sum(u * oracle_mod.blur3d_adjoint(v, *shape, padding)))
    assert abs(lhs - rhs) <= 1e-13 * max(abs(lhs), 1.0)


def test_adjoint_valid_is_conv_transpose(oracle_mod):
    rng = np.random.default_rng(8)
    H, W = 23, 31
    g = rng.standard_normal((H - 10, W - 10))
    w = ndimage.gaussian_filter1d(np.eye(11)[5], SIGMA, mode="constant", truncate=TRUNC)
    win = torch.from_numpy(np.outer(w, w))[None, None]
    ref = F.conv_transpose2d(torch.from_numpy(g)[None, None], win)[0, 0].numpy()
    assert rel_err(oracle_mod.blur2d_adjoint(g, H, W, "valid"), ref) < 1e-13


# ---------------------------------------------------------- SSIM forward

@pytest.mark.parametrize("padding", ["valid", "same"])
def test_ssim_of_image_with_itself_is_one(oracle_mod, padding):
    x, _ = uniform_pair((2, 3, 17, 14), 21)
    mean, smap = oracle_mod.ssim2d(x, x, padding, want_map=True)
    assert np.max(np.abs(smap - 1.0)) < 1e-12
    assert np.max(np.abs(mean - 1.0)) < 1e-12
    v, _ = uniform_pair((1, 2, 12, 11, 13), 22)
    m3 = oracle_mod.ssim3d(v, v, padding)
    assert np.max(np.abs(m3 - 1.0)) < 1e-12


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_ssim_symmetric(oracle_mod, padding):
    x, y = uniform_pair((1, 2, 15, 18), 23, std=0.2)
    m1, s1 = oracle_mod.ssim2d(x, y, padding, want_map=True)
    m2, s2 = oracle_mod.ssim2d(y, x, padding, want_map=True)
    assert np.max(np.abs(s1 - s2)) < 1e-14 and np.max(np.abs(m1 - m2)) < 1e-14


def test_ssim_constant_images_closed_form(oracle_mod):
    # sigma11 = e11 - mu1^2 is zero only up to rounding of an n-term sum
    # (|err| <= n * 1.1e-16), and S divides it by ~C2 = 9e-4: 121 terms give
    # <= 1.5e-11, 1331 terms <= 1.6e-10.  Dropping C1 would move S by ~1e-4.
    for a, b in [(0.2, 0.7), (1.0, 0.0), (0.5, 0.5), (0.0, 0.0)]:
        x = np.full((1, 1, 14, 13), a)
        y = np.full((1, 1, 14, 13), b)
        expect = (2 * a * b + C1) / (a * a + b * b + C1)
        mean, smap = oracle_mod.ssim2d(x, y, "valid", want_map=True)
        assert np.max(np.abs(smap - expect)) < 1.5e-11
        assert abs(mean[0] - expect) < 1.5e-11
        m3 = oracle_mod.ssim3d(x[:, :, :11, None, :11] * np.ones((1, 1, 1, 12, 1)),
                               y[:, :, :11, None, :11] * np.ones((1, 1, 1, 12, 1)), "valid")
        assert abs(m3[0] - expect) < 1.6e-10


def _moments(x, y, padding):
    mu1, mu2 = scipy_blur(x, padding), scipy_blur(y, padding)
    s11 = scipy_blur(x * x, padding) - mu1 * mu1
    return mu1, mu2, s11


def test_ssim_shifted_copy_closed_form(oracle_mod):
    # y = x + k: sigma22 = sigma12 = sigma11, so the contrast-structure factor is 1.
    # Only valid windows see y as x + k everywhere (zero padding breaks the shift).
    padding = "valid"
    x = np.random.default_rng(31).random((19, 17)) * 0.5
    k = 0.3
    y = x + k
    mu1 = scipy_blur(x, padding)
    expect = (2 * mu1 * (mu1 + k) + C1) / (mu1**2 + (mu1 + k) ** 2 + C1)
    _, smap = oracle_mod.ssim2d(x[None, None], y[None, None], padding, want_map=True)
    assert rel_err(smap[0, 0], expect) < 1e-12


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_ssim_scaled_copy_closed_form(oracle_mod, padding):
    # y = a*x: mu2 = a mu1, sigma22 = a^2 sigma11, sigma12 = a sigma11 (all paddings).
    x = np.random.default_rng(32).random((16, 21))
    a = 0.6
    mu1, _, s11 = _moments(x, a * x, padding)
    expect = ((2 * a * mu1 * mu1 + C1) * (2 * a * s11 + C2)
              / (((1 + a * a) * mu1 * mu1 + C1) * ((1 + a * a) * s11 + C2)))
    _, smap = oracle_mod.ssim2d(x[None, None], (a * x)[None, None], padding, want_map=True)
    assert rel_err(smap[0, 0], expect) < 1e-10


def test_ssim_one_constant_image_closed_form(oracle_mod):
    # x = a everywhere (valid windows): sigma11 = sigma12 = 0.
    y = np.random.default_rng(33).random((18, 15))
    a = 0.4
    x = np.full_like(y, a)
    mu2 = scipy_blur(y, "valid")
    s22 = scipy_blur(y * y, "valid") - mu2 * mu2
    expect = (2 * a * mu2 + C1) * C2 / ((a * a + mu2 * mu2 + C1) * (s22 + C2))
    _, smap = oracle_mod.ssim2d(x[None, None], y[None, None], "valid", want_map=True)
    assert rel_err(smap[0, 0], expect) < 1e-10


def test_mean_normaliser_and_channels(oracle_mod):
    # mean[n] averages channels and output pixels: constant planes with different
    # constants per channel give the average of the per-channel closed forms.
    vals = [(0.1, 0.9), (0.5, 0.4), (0.8, 0.8)]
    x = np.stack([np.full((12, 16), a) for a, _ in vals])[None]
    y = np.stack([np.full((12, 16), b) for _, b in vals])[None]
    expect = np.mean([(2 * a * b + C1) / (a * a + b * b + C1) for a, b in vals])
    assert abs(oracle_mod.ssim2d(x, y, "valid")[0] - expect) < 1.5e-11


def test_stats_are_blurred_raw_moments(oracle_mod):
    x, y = uniform_pair((1, 1, 14, 16), 34)
    st = oracle_mod.ssim2d_stats(x, y, "same")[0, 0]
    x64, y64 = x[0, 0].astype(np.float64), y[0, 0].astype(np.float64)
    for k, f in enumerate([x64, y64, x64 * x64, y64 * y64, x64 * y64]):
        assert rel_err(st[k], scipy_blur(f, "same")) < 1e-13


# --------------------------------------------------------- derivatives

def test_pointwise_partials_finite_differences(oracle_mod):
    rng = np.random.default_rng(40)
    for _ in range(20):
        mu1, mu2 = rng.random(2)
        m = np.array([mu1, mu2, mu1 * mu1 + rng.random() * 0.05,
                      mu2 * mu2 + rng.random() * 0.05, mu1 * mu2 + rng.normal() * 0.01])
        _, d = oracle_mod.ssim_point(*m)
        for k in range(5):
            h = 1e-6
            mp, mm = m.copy(), m.copy()
            mp[k] += h
            mm[k] -= h
            fd = (oracle_mod.ssim_point(*mp)[0] - oracle_mod.ssim_point(*mm)[0]) / (2 * h)
            assert abs(fd - d[k]) <= 1e-7 * max(1.0, abs(d[k]))


def _fd_grad_2d(oracle_mod, x, y, dL, padding, which):
    h = 1e-5
    base = (x, y)
    g = np.zeros_like(base[which])
    flat = g.reshape(-1)
    for t in range(flat.size):
        plus = [base[0].copy(), base[1].copy()]
        minus = [base[0].copy(), base[1].copy()]
        plus[which].reshape(-1)[t] += h
        minus[which].reshape(-1)[t] -= h
        fp = float(np.dot(dL, oracle_mod.ssim2d(plus[0], plus[1], padding)))
        fm = float(np.dot(dL, oracle_mod.ssim2d(minus[0], minus[1], padding)))
        flat[t] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("padding,hw", [("same", (8, 8)), ("same", (16, 16)),
                                        ("valid", (12, 12)), ("valid", (16, 16)),
                                        ("valid", (13, 11))])
def test_grad2d_finite_differences(oracle_mod, padding, hw):
    x, y = uniform_pair((2, 2) + hw, 41, std=0.1)
    x, y = x.astype(np.float64), y.astype(np.float64)
    dL = np.array([-1.0, 0.37])
    g1, g2 = oracle_mod.ssim2d_grad(x, y, dL, padding, want_grad2=True)
    for which, g in ((0, g1), (1, g2)):
        fd = _fd_grad_2d(oracle_mod, x, y, dL, padding, which)
        assert rel_err(g, fd) < 1e-7


def _fd_grad_3d(oracle_mod, x, y, padding):
    h = 1e-5
    g = np.zeros_like(x)
    flat = g.reshape(-1)
    for t in range(flat.size):
        xp, xm = x.copy(), x.copy()
        xp.reshape(-1)[t] += h
        xm.reshape(-1)[t] -= h
        flat[t] = -(oracle_mod.ssim3d(xp, y, padding)[0]
                    - oracle_mod.ssim3d(xm, y, padding)[0]) / (2 * h)
    return g


@pytest.mark.parametrize("padding,dhw", [("valid", (12, 12, 12)), ("same", (7, 8, 6))])
def test_grad3d_finite_differences(oracle_mod, padding, dhw):
    x, y = uniform_pair((1, 1) + dhw, 42, std=0.1)
    x, y = x.astype(np.float64), y.astype(np.float64)
    g1, g2 = oracle_mod.ssim3d_grad(x, y, [-1.0], padding, want_grad2=True)
    assert rel_err(g1, _fd_grad_3d(oracle_mod, x, y, padding)) < 1e-7
    g2_swapped, _ = oracle_mod.ssim3d_grad(y, x, [-1.0], padding, want_grad2=False)
    assert rel_err(g2, g2_swapped) < 1e-13


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_grad_zero_at_identical_images(oracle_mod, padding):
    x, _ = uniform_pair((1, 3, 20, 17), 43)
    g1, g2 = oracle_mod.ssim2d_grad(x, x, [-1.0], padding)
    # Typical |grad| for distinct images here is ~1e-4; at y = x it vanishes.
    assert np.max(np.abs(g1)) < 1e-15 and np.max(np.abs(g2)) < 1e-15


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_grad2_is_grad1_with_images_swapped(oracle_mod, padding):
    x, y = uniform_pair((2, 1, 15, 19), 44, std=0.15)
    dL = np.array([-0.5, 2.0])
    g1, g2 = oracle_mod.ssim2d_grad(x, y, dL, padding)
    h1, _ = oracle_mod.ssim2d_grad(y, x, dL, padding, want_grad2=False)
    assert rel_err(g2, h1) < 1e-13


def _torch_ssim_mean(x, y, padding):
    """An independent float64 autograd SSIM: conv2d with scipy's window."""
    w = ndimage.gaussian_filter1d(np.eye(11)[5], SIGMA, mode="constant", truncate=TRUNC)
    C = x.shape[1]
    win = torch.from_numpy(np.outer(w, w)).expand(C, 1, 11, 11).contiguous()
    pad = 5 if padding == "same" else 0
    blur = lambda t: F.conv2d(t, win, padding=pad, groups=C)
    mu1, mu2 = blur(x), blur(y)
    s11 = blur(x * x) - mu1 * mu1
    s22 = blur(y * y) - mu2 * mu2
    s12 = blur(x * y) - mu1 * mu2
    S = ((2 * mu1 * mu2 + C1) * (2 * s12 + C2)) / ((mu1**2 + mu2**2 + C1) * (s11 + s22 + C2))
    return S.mean(dim=(1, 2, 3))


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_grad2d_matches_torch_autograd(oracle_mod, padding):
    x, y = uniform_pair((2, 3, 24, 31), 45, std=0.1)
    dL = np.array([-1.0, -0.25])
    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    ty = torch.tensor(y, dtype=torch.float64, requires_grad=True)
    m = _torch_ssim_mean(tx, ty, padding)
    (m * torch.from_numpy(dL)).sum().backward()
    mean = oracle_mod.ssim2d(x, y, padding)
    g1, g2 = oracle_mod.ssim2d_grad(x, y, dL, padding)
    assert np.max(np.abs(mean - m.detach().numpy())) < 1e-13
    assert rel_err(g1, tx.grad.numpy()) < 1e-11
    assert rel_err(g2, ty.grad.numpy()) < 1e-11


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_grad_at_equals_full_grad(oracle_mod, padding):
    x, y = uniform_pair((2, 2, 21, 18), 46, std=0.1)
    dL = np.array([-1.0, 0.5])
    g1, g2 = oracle_mod.ssim2d_grad(x, y, dL, padding)
    idx = np.random.default_rng(0).choice(x.size, 60, replace=False)
    idx = np.concatenate([idx, [0, x.size - 1, 17, 18 * 21]])
    a1, a2 = oracle_mod.ssim2d_grad_at(x, y, dL, padding, idx)
    assert rel_err(a1, g1.reshape(-1)[idx]) < 1e-12
    assert rel_err(a2, g2.reshape(-1)[idx]) < 1e-12
    v1, v2 = uniform_pair((1, 2, 12, 13, 11), 47, std=0.1)
    h1, h2 = oracle_mod.ssim3d_grad(v1, v2, [-1.0], padding)
    idx3 = np.random.default_rng(1).choice(v1.size, 25, replace=False)
    b1, b2 = oracle_mod.ssim3d_grad_at(v1, v2, [-1.0], padding, idx3)
    assert rel_err(b1, h1.reshape(-1)[idx3]) < 1e-12
    assert rel_err(b2, h2.reshape(-1)[idx3]) < 1e-12


def test_bad_arguments_rejected(oracle_mod):
    x = np.zeros((1, 1, 10, 12))
    with pytest.raises(ValueError):
        oracle_mod.ssim2d(x, x, "valid")  # H < 11
    with pytest.raises(ValueError):
        oracle_mod.ssim2d(x, x, "reflect")


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_ssim3d_map_at_matches_the_full_map(oracle_mod, padding):
    """The sampled 3D map (used where the whole map is too large) is the full
    map's value at each index: both are the direct 1331-term window sums, and
    the full map is itself pinned above (closed forms, scipy, finite
    differences of its mean)."""
    rng = np.random.default_rng(77)
    x = rng.random((2, 2, 13, 12, 14))
    y = np.clip(x + rng.normal(0, 0.05, x.shape), 0, 1)
    _, full = oracle_mod.ssim3d(x, y, padding, want_map=True)
    idx = rng.integers(0, full.size, size=200)
    idx[:3] = (0, full.size - 1, full.size // 2)
    got = oracle_mod.ssim3d_map_at(x, y, padding, idx)
    np.testing.assert_allclose(got, full.reshape(-1)[idx], rtol=0, atol=1e-14)
    with pytest.raises(ValueError):
        oracle_mod.ssim3d_map_at(x, y, padding, [full.size])
