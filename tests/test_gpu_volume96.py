"""GPU parity of the 3D loss through the autograd API on a batch of volumes.

Two 3-channel 96^3 volumes (same padding): the shape of the 3D example that the
fused-SSIM pages give for volumetric inputs.  The inputs are trilinear noise
(a 12^3 grid of U[0, 1] values upsampled to 96^3) and a noisy copy
(sigma 0.03, clamped).  The volume is small enough for the whole oracle, so
every output voxel and every input gradient is compared:
  - fused_ssim3d(img1, img2) and its backward: the loss is the mean over the
    two images, so dLoss/dmean[n] = 1/2; img2 also requires a gradient;
  - per_image=True: the per-image means;
  - train=False (no saved fields, the backward recomputes);
  - the map of the C-ABI forward (ssim3d_fwd) element by element.
The bars are the 3D parity bars: means 1e-5, maps 3e-5, gradients 1e-4 of the
largest oracle gradient.
"""
import numpy as np
import pytest

from workloads import noisy_copy, trilinear_noise_volume

pytestmark = pytest.mark.gpu

MEAN_TOL = 1e-5
MAP_TOL_3D = 3e-5
GRAD_RTOL = 1e-4
SHAPE = (2, 3, 96, 96, 96)


@pytest.fixture(scope="module")
def ref(oracle_mod):
    rng = np.random.default_rng(9603)
    a = trilinear_noise_volume(rng, *SHAPE, coarse=12)
    b = noisy_copy(rng, a, 0.03)
    x = np.ascontiguousarray(a, dtype=np.float32)
    y = np.ascontiguousarray(b, dtype=np.float32)
    mean, smap = oracle_mod.ssim3d(x, y, "same", want_map=True)
    g1, g2 = oracle_mod.ssim3d_grad(x, y, np.full(SHAPE[0], 1.0 / SHAPE[0]), "same")
    return {"x": x, "y": y, "mean": mean, "map": smap, "g1": g1, "g2": g2}


@pytest.fixture(scope="module")
def pkg():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiable_image_quality_gb300 as pkg
    from differentiable_image_quality_gb300 import _build

    _build.build()
    return pkg


def _grad_err(got, want):
    return float(np.max(np.abs(got.astype(np.float64) - want)) / np.max(np.abs(want)))


@pytest.mark.parametrize("train", [True, False])
def test_volume96_loss_and_gradients(pkg, ref, train):
    import torch

    dev = torch.device("cuda:0")
    tx = torch.from_numpy(ref["x"]).to(dev).requires_grad_(True)
    ty = torch.from_numpy(ref["y"]).to(dev).requires_grad_(True)
    loss = pkg.fused_ssim3d(tx, ty, padding="same", train=train)
    loss.backward()
    torch.cuda.synchronize()
    assert abs(loss.item() - float(np.mean(ref["mean"]))) <= MEAN_TOL
    for name, t in (("g1", tx), ("g2", ty)):
        got = t.grad.cpu().numpy()
        assert np.all(np.isfinite(got)), name
        err = _grad_err(got, ref[name])
        assert err <= GRAD_RTOL, f"train={train} {name}: relative error {err:.3e}"


def test_volume96_per_image_means(pkg, ref):
    import torch

    dev = torch.device("cuda:0")
    tx = torch.from_numpy(ref["x"]).to(dev)
    ty = torch.from_numpy(ref["y"]).to(dev)
    with torch.no_grad():
        m = pkg.fused_ssim3d(tx, ty, padding="same", train=False, per_image=True)
    assert m.shape == (SHAPE[0],)
    assert np.max(np.abs(m.cpu().numpy() - ref["mean"])) <= MEAN_TOL


def test_volume96_map(pkg, ref):
    import torch

    dev = torch.device("cuda:0")
    tx = torch.from_numpy(ref["x"]).to(dev)
    ty = torch.from_numpy(ref["y"]).to(dev)
    mean = torch.full((SHAPE[0],), float("nan"), device=dev)
    smap = torch.full(SHAPE, float("nan"), device=dev)
    pkg.ssim3d_fwd(tx, ty, "same", mean, out_map=smap)
    torch.cuda.synchronize()
    got = smap.cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got.astype(np.float64) - ref["map"])))
    assert err <= MAP_TOL_3D, f"map off by {err:.3e}"
    assert np.max(np.abs(mean.cpu().numpy() - ref["mean"])) <= MEAN_TOL
