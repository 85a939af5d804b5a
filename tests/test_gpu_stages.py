"""Stage-by-stage parity of the 2D gradient kernel (validation in the order of
the ssimulacra2 GPU hand-off page: the blurred statistics first, then what is
built on them).

The test build of the library (libgbssim_test.so) runs the gradient-mode
kernel of the stored forward with grad2 and also writes, for every output
pixel, the window's statistics mu1, mu2, sigma11 + sigma22, sigma12 and the
derivatives of S with respect to the unshifted moments mu1, mu2, E[x^2]
(= E[y^2]), E[xy].  They are
compared with the oracle's blurred statistics (oracle.ssim2d_stats, a direct
121-term window) and with its pointwise SSIM derivatives (oracle.ssim_point),
so that an error in one stage shows up in that stage, before it reaches S, the
mean or the gradients.

Bars.  The statistics are sums of 121 float32 products of values in [0, 1]
(shifted before squaring): within 1e-6 absolute.  The derivatives of S scale
like 1 / (sigma11 + sigma22 + C2), up to ~1e3 in flat regions, and the kernel
forms them from shifted moments: dS/dmu1 = g_m1 - 2 s dS/dE[x^2] - t dS/dE[xy]
is a difference of terms as large as the largest derivative.  So every
derivative is held to 5e-5 of the largest magnitude among all four over the
image (the scale of the terms its float32 rounding acts on).  The rounding of
a window's shifted second moments grows with their size, which is largest in a
flat window whose band value lies across an edge from most of its pixels:
measured 2.2e-5 on the crop of the blob render below, 1.2e-6 on the uniform
pairs.  (There the kernel's own outputs lose nothing where the two images
agree -- the chain rule meets dS/dE[(x-y)^2] through x - y -- but the dump's
derivatives with respect to the raw moments carry the rounding of sigma11 +
sigma22: 6.3e-5 on a white background whose bands take their shift from a
black border.)
"""
import numpy as np
import pytest

from workloads import make_inputs, uniform_pair

pytestmark = pytest.mark.gpu

STAT_TOL = 1e-6
DERIV_RTOL = 5e-5


@pytest.fixture(scope="module")
def test_lib():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    return _abi.load_test()


def _dump(lib, x, y, padding):
    import torch

    dev = torch.device("cuda:0")
    N, C, H, W = x.shape
    ho, wo = (H - 10, W - 10) if padding == "valid" else (H, W)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    stats = torch.full((N, C, ho, wo, 4), float("nan"), device=dev)
    grads = torch.full((N, C, ho, wo, 4), float("nan"), device=dev)
    f1, f2 = torch.empty_like(tx), torch.empty_like(ty)
    st = lib.gbssim_test_stage_dump2d(tx.data_ptr(), ty.data_ptr(), N, C, H, W,
                                      0 if padding == "valid" else 1, stats.data_ptr(),
                                      grads.data_ptr(), f1.data_ptr(), f2.data_ptr(),
                                      torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, lib.gbssim_strerror(st)
    torch.cuda.synchronize()
    return stats.cpu().numpy().astype(np.float64), grads.cpu().numpy().astype(np.float64)


def _oracle_stages(oracle_mod, x, y, padding):
    """(stats, derivs) of the oracle in the dump's layout: [N, C, Ho, Wo, 4]."""
    st = oracle_mod.ssim2d_stats(x, y, padding)  # (N, C, 5, Ho, Wo)
    mu1, mu2, e11, e22, e12 = (st[:, :, i] for i in range(5))
    stats = np.stack([mu1, mu2, e11 + e22 - mu1 * mu1 - mu2 * mu2, e12 - mu1 * mu2], axis=-1)
    derivs = np.empty(stats.shape)
    flat_st = st.transpose(0, 1, 3, 4, 2).reshape(-1, 5)
    flat_d = derivs.reshape(-1, 4)
    for i, (a, b, c, d, e) in enumerate(flat_st):
        _, g = oracle_mod.ssim_point(a, b, c, d, e)
        assert g[2] == g[3]  # dS/dE[x^2] = dS/dE[y^2]: S sees only sigma11 + sigma22
        flat_d[i] = (g[0], g[1], g[2], g[4])
    return stats, derivs


def _check(got, ref, label):
    gs, gd = got
    rs, rd = ref
    assert np.all(np.isfinite(gs)) and np.all(np.isfinite(gd)), f"{label}: pixels not written"
    names = ("mu1", "mu2", "sigma11 + sigma22", "sigma12")
    for i, n in enumerate(names):
        err = np.max(np.abs(gs[..., i] - rs[..., i]))
        assert err <= STAT_TOL, f"{label}: {n} off by {err:.3e}"
    names = ("dS/dmu1", "dS/dmu2", "dS/dE[x^2]", "dS/dE[xy]")
    scale = np.max(np.abs(rd))
    for i, n in enumerate(names):
        err = np.max(np.abs(gd[..., i] - rd[..., i])) / scale
        assert err <= DERIV_RTOL, f"{label}: {n} relative error {err:.3e}"


@pytest.mark.parametrize("shape,padding,seed", [
    ((1, 2, 40, 148), "valid", 1),
    ((1, 2, 40, 148), "same", 2),
    ((2, 1, 75, 260), "same", 3),   # several strips, several row steps
    ((1, 1, 12, 12), "valid", 4),
    ((1, 1, 3, 8), "same", 5),
])
def test_stages_match_the_oracle(test_lib, oracle_mod, shape, padding, seed):
    x, y = uniform_pair(shape, 1200 + seed, std=0.08)
    _check(_dump(test_lib, x, y, padding), _oracle_stages(oracle_mod, x, y, padding),
           f"{shape} {padding}")


def test_stages_on_a_crop_of_the_blob_render(test_lib, oracle_mod):
    """Flat, saturated and dark regions: where the statistics' float32
    cancellation would show first."""
    x, y = make_inputs("splat1080_same")
    x = np.ascontiguousarray(x[:, :, 300:372, 600:900])
    y = np.ascontiguousarray(y[:, :, 300:372, 600:900])
    _check(_dump(test_lib, x, y, "same"), _oracle_stages(oracle_mod, x, y, "same"),
           "blob render crop")
