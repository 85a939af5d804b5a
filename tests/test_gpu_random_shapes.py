"""GPU parity on a seeded sweep of random shapes.

The fixed cases elsewhere cover the edges the kernels' geometry suggests; this
sweep draws N, C, H, W (and D), the padding and the base-pointer alignment at
random from a fixed seed, so that combinations nobody chose by hand go through
every path too: the stored and the recompute backward, the single call, the
forward-only map, and the per-octave stage.  Same bars as the fixed cases.
"""
import numpy as np
import pytest

from test_gpu_parity import MAP_TOL, OCTAVE_MAP_TOL, _assert_parity, _oracle
from workloads import uniform_pair

pytestmark = pytest.mark.gpu

N_2D, N_3D = 14, 12


def _draw_2d(i):
    rng = np.random.default_rng(5000 + i)
    padding = "valid" if rng.random() < 0.5 else "same"
    lo = 11 if padding == "valid" else 1
    H = int(rng.integers(lo, 160))
    W = int(rng.integers(lo, 420))
    N, C = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    offset = int(rng.choice([0, 0, 1, 3]))  # floats past a 256-byte boundary
    return (N, C, H, W), padding, offset


def _draw_3d(i):
    rng = np.random.default_rng(6000 + i)
    padding = "valid" if rng.random() < 0.6 else "same"
    lo = 11 if padding == "valid" else 1
    D, H, W = (int(rng.integers(lo, 30)) for _ in range(3))
    N, C = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    return (N, C, D, H, W), padding


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    _abi.load()
    return torch.device("cuda:0")


def _on_device(a, dev, offset):
    """a as a CUDA tensor whose data starts `offset` floats into its storage."""
    import torch

    n = a.size
    buf = torch.empty(n + offset, device=dev)
    t = buf[offset:].view(a.shape)
    t.copy_(torch.from_numpy(a))
    return t


@pytest.mark.parametrize("i", range(N_2D))
def test_random_2d(dev, oracle_mod, i):
    import torch

    import differentiable_image_quality_gb300 as pkg

    shape, padding, offset = _draw_2d(i)
    N = shape[0]
    x, y = uniform_pair(shape, 7000 + i, std=0.1)
    dl = np.linspace(-1.0, 0.7, N)
    ref = _oracle(oracle_mod, x, y, dl, padding, True, want_map=True)
    tx, ty = _on_device(x, dev, offset), _on_device(y, dev, offset)
    tdl = torch.from_numpy(dl.astype(np.float32)).to(dev)
    ho = shape[2] - 10 if padding == "valid" else shape[2]
    wo = shape[3] - 10 if padding == "valid" else shape[3]
    label = f"{shape} {padding} offset {offset}"

    # stored backward
    mean = torch.full((N,), float("nan"), device=dev)
    smap = torch.full((N, shape[1], ho, wo), float("nan"), device=dev)
    saved = torch.empty(pkg.saved_bytes(shape, True) // 4, device=dev)
    pkg.ssim_fwd(tx, ty, padding, mean, out_map=smap, saved=saved, want_grad2=True)
    g1, g2 = torch.full_like(tx, float("nan")), torch.full_like(ty, float("nan"))
    pkg.ssim_bwd(tdl, tx, ty, padding, g1, g2, saved=saved)
    # recompute backward and single call
    r1, r2 = torch.full_like(tx, float("nan")), torch.full_like(ty, float("nan"))
    pkg.ssim_bwd(tdl, tx, ty, padding, r1, r2)
    m3 = torch.full((N,), float("nan"), device=dev)
    s1 = torch.full_like(tx, float("nan"))
    pkg.ssim_fwd_bwd(tx, ty, padding, tdl, m3, s1)
    # forward only, with the map
    m4 = torch.full((N,), float("nan"), device=dev)
    map4 = torch.full((N, shape[1], ho, wo), float("nan"), device=dev)
    pkg.ssim_fwd(tx, ty, padding, m4, out_map=map4)
    torch.cuda.synchronize()

    c = lambda t: t.cpu().numpy()  # noqa: E731
    _assert_parity({"mean": c(mean), "g1": c(g1), "g2": c(g2), "map": c(smap)}, ref, True,
                   label + " stored")
    _assert_parity({"mean": c(mean), "g1": c(r1), "g2": c(r2)}, ref, True, label + " recompute")
    _assert_parity({"mean": c(m3), "g1": c(s1)}, ref, False, label + " single call")
    dm = np.max(np.abs(c(m4).astype(np.float64) - ref["mean"]))
    assert dm <= 1e-5, f"{label} forward only: mean off by {dm:.3e}"
    dmap = np.max(np.abs(c(map4).astype(np.float64) - ref["map"]))
    assert dmap <= MAP_TOL, f"{label} forward only: map off by {dmap:.3e}"


@pytest.mark.parametrize("i", range(N_3D))
def test_random_3d(dev, oracle_mod, i):
    import torch

    import differentiable_image_quality_gb300 as pkg

    shape, padding = _draw_3d(i)
    N = shape[0]
    x, y = uniform_pair(shape, 8000 + i, std=0.1)
    dl = np.linspace(-1.0, 0.7, N)
    ref = _oracle(oracle_mod, x, y, dl, padding, True)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    tdl = torch.from_numpy(dl.astype(np.float32)).to(dev)
    mean = torch.full((N,), float("nan"), device=dev)
    saved = torch.empty(pkg.saved_bytes(shape, True) // 4, device=dev)
    pkg.ssim3d_fwd(tx, ty, padding, mean, saved=saved, want_grad2=True)
    g1, g2 = torch.full_like(tx, float("nan")), torch.full_like(ty, float("nan"))
    pkg.ssim3d_bwd(tdl, tx, ty, padding, g1, g2, saved=saved)
    r1 = torch.full_like(tx, float("nan"))
    pkg.ssim3d_bwd(tdl, tx, ty, padding, r1)
    torch.cuda.synchronize()
    c = lambda t: t.cpu().numpy()  # noqa: E731
    label = f"{shape} {padding}"
    _assert_parity({"mean": c(mean), "g1": c(g1), "g2": c(g2)}, ref, True, label + " stored")
    _assert_parity({"mean": c(mean), "g1": c(r1)}, ref, False, label + " recompute")


@pytest.mark.parametrize("i", range(10))
def test_random_pyramid(dev, oracle_mod, i):
    import differentiable_image_quality_gb300 as pkg

    shape, padding, offset = _draw_2d(100 + i)
    H, W = shape[2], shape[3]
    lo = 11 if padding == "valid" else 1
    octaves = 1
    while octaves < 10 and min(pkg.pyramid_extents(H, W, octaves + 1)[-1]) >= lo:
        octaves += 1
    x, y = uniform_pair(shape, 9000 + i, std=0.1)
    tx, ty = _on_device(x, dev, offset), _on_device(y, dev, offset)
    means, maps = pkg.ssim_pyramid(tx, ty, padding, octaves, want_maps=True)
    rm, rmaps = oracle_mod.ssim2d_pyramid(x, y, padding, octaves, want_maps=True)
    assert np.max(np.abs(means.cpu().numpy() - rm)) <= 1e-5, (shape, padding, octaves)
    for o in range(octaves):
        tol = MAP_TOL if o == 0 else OCTAVE_MAP_TOL
        assert np.max(np.abs(maps[o].cpu().numpy() - rmaps[o])) <= tol, (shape, o)
