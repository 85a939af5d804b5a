"""GPU parity on a volume whose intermediate fields exceed the L2 cache.

At 1x1x256^3 (valid padding) the 3D path's two per-slice fields -- the
XY-blurred statistics and the Z adjoint of the derivatives, 246^2 x 256
float4 each, 248 MB -- no longer fit in the GPU's 129 MB L2, so they go through
HBM between the kernels.  The whole oracle is too slow at this size; it is
compared where it can be evaluated point by point:
  - the SSIM map at sampled output voxels (oracle.ssim3d_map_at), within the
    3D map bar;
  - the gradient of the mean at sampled input voxels (oracle.ssim3d_grad_at),
    both backward paths, within 1e-4 of the largest sampled oracle gradient;
  - the mean against the float64 mean of the GPU's own map (the reduction),
    which together with the sampled map pins the mean.
The samples include the volume's corners, faces and edges.
"""
import numpy as np
import pytest

from workloads import dl_vector, make_inputs

pytestmark = pytest.mark.gpu

MAP_TOL_3D = 3e-5
GRAD_RTOL = 1e-4
N_SAMPLES = 3000


@pytest.fixture(scope="module")
def volume_run(oracle_mod):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiable_image_quality_gb300 as pkg
    from differentiable_image_quality_gb300 import _build

    _build.build()
    dev = torch.device("cuda:0")
    x, y = make_inputs("volume256_valid")
    dl = dl_vector("volume256_valid")
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    tdl = torch.from_numpy(dl).to(dev)
    D = x.shape[2]
    mean = torch.full((1,), float("nan"), device=dev)
    smap = torch.full((1, 1, D - 10, D - 10, D - 10), float("nan"), device=dev)
    saved = torch.empty(pkg.saved_bytes(x.shape, False) // 4, device=dev)
    pkg.ssim3d_fwd(tx, ty, "valid", mean, out_map=smap, saved=saved)
    g_saved = torch.full_like(tx, float("nan"))
    pkg.ssim3d_bwd(tdl, tx, ty, "valid", g_saved, saved=saved)
    g_rec = torch.full_like(tx, float("nan"))
    pkg.ssim3d_bwd(tdl, tx, ty, "valid", g_rec)
    torch.cuda.synchronize()
    return {"x": x, "y": y, "dl": dl, "mean": mean.cpu().numpy(), "map": smap.cpu().numpy(),
            "g_saved": g_saved.cpu().numpy(), "g_rec": g_rec.cpu().numpy()}


def _samples(shape, seed):
    """Flat indices into `shape` (the last three axes spatial): random ones plus
    every corner, face centre and edge midpoint."""
    rng = np.random.default_rng(seed)
    D, H, W = shape[-3:]
    pts = [(d, h, w) for d in (0, D // 2, D - 1) for h in (0, H // 2, H - 1)
           for w in (0, W // 2, W - 1)]
    flat = [np.ravel_multi_index((0, 0) + p, shape) for p in pts]
    flat += list(rng.integers(0, int(np.prod(shape)), size=N_SAMPLES - len(flat)))
    return np.asarray(flat, dtype=np.int64)


def test_large_volume_map_and_mean(volume_run, oracle_mod):
    got_map = volume_run["map"]
    assert np.all(np.isfinite(got_map))
    # the mean is the float64 mean of the map the kernels produced
    assert abs(float(volume_run["mean"][0]) - float(np.mean(got_map.astype(np.float64)))) <= 1e-6
    idx = _samples(got_map.shape, 256)
    ref = oracle_mod.ssim3d_map_at(volume_run["x"], volume_run["y"], "valid", idx)
    err = np.max(np.abs(got_map.reshape(-1)[idx].astype(np.float64) - ref))
    assert err <= MAP_TOL_3D, f"map at sampled voxels off by {err:.3e}"


@pytest.mark.parametrize("path", ["g_saved", "g_rec"])
def test_large_volume_gradient_at_samples(volume_run, oracle_mod, path):
    got = volume_run[path]
    assert np.all(np.isfinite(got))
    idx = _samples(got.shape, 257)
    ref, _ = oracle_mod.ssim3d_grad_at(volume_run["x"], volume_run["y"], volume_run["dl"], "valid",
                                       idx, want_grad2=False)
    scale = np.max(np.abs(ref))
    err = np.max(np.abs(got.reshape(-1)[idx].astype(np.float64) - ref)) / scale
    assert err <= GRAD_RTOL, f"{path}: gradient at sampled voxels, relative error {err:.3e}"
