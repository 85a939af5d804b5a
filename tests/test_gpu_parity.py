"""GPU parity: the CUDA library against the CPU oracle, element by element.

Every call goes through the C ABI (via the thin torch wrappers).  Bars, from
the loss's specification: |mean_gpu - mean_oracle| <= 1e-5 for every image;
max |grad_gpu - grad_oracle| <= 1e-4 * max |grad_oracle| for each gradient.
The SSIM map has no stated bar.  The kernels evaluate the contrast-structure
factor as cs = 1 - D / (sigma11 + sigma22 + C2) with D = sigma11 + sigma22 -
2 sigma12 taken from the blurred squared difference E[(x - y)^2]: D carries
no rounding of the images' common level, so where the images agree (the flat
windows, whose denominator is ~C2 = 9e-4) cs is near exact, and the float32
rounding of sigma11 + sigma22 moves S only in proportion to D / (sigma11 +
sigma22 + C2).  The 2D kernels also shift each 11-row band of an 8-column group
of windows by one pixel of that neighbourhood (bands on one grid per image, so
the results do not depend on the launch plan); the 3D kernels shift by 1/2.
Measured on the full workloads: 2D maps at most 2.4e-6 (the 1080p pairs, both
paddings), the downscaled octaves of the per-octave stage at most 5.1e-6,
3D maps at most 1.2e-5 (128^3).  Bars: 2D maps 5e-6, octave maps 1e-5, 3D maps
3e-5.
"""
import numpy as np
import pytest

from workloads import WORKLOADS, dl_vector, make_inputs, uniform_pair

pytestmark = pytest.mark.gpu

MEAN_TOL = 1e-5
GRAD_RTOL = 1e-4
MAP_TOL = 5e-6      # 2D maps
OCTAVE_MAP_TOL = 1e-5  # maps of the downscaled octaves
MAP_TOL_3D = 3e-5   # 3D maps


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    _abi.load()
    return torch.device("cuda:0")


def _run(dev, x, y, dl, padding, want_grad2, path, want_map=False):
    """One forward + backward through the C ABI; path 'saved' or 'recompute'."""
    import torch

    import differentiable_image_quality_gb300 as pkg

    tx = torch.from_numpy(x).to(dev)
    ty = torch.from_numpy(y).to(dev)
    tdl = torch.from_numpy(np.ascontiguousarray(dl, dtype=np.float32)).to(dev)
    N = x.shape[0]
    is3d = x.ndim == 5
    fwd = pkg.ssim3d_fwd if is3d else pkg.ssim_fwd
    bwd = pkg.ssim3d_bwd if is3d else pkg.ssim_bwd
    mean = torch.full((N,), float("nan"), device=dev)
    smap = None
    if want_map:
        ext = [s - 10 if padding == "valid" else s for s in x.shape[2:]]
        smap = torch.full((N, x.shape[1], *ext), float("nan"), device=dev)
    saved = None
    if path == "saved":
        saved = torch.empty(pkg.saved_bytes(x.shape, want_grad2) // 4, device=dev)
    fwd(tx, ty, padding, mean, out_map=smap, saved=saved, want_grad2=want_grad2)
    g1 = torch.full_like(tx, float("nan"))
    g2 = torch.full_like(ty, float("nan")) if want_grad2 else None
    bwd(tdl, tx, ty, padding, g1, g2, saved=saved)
    torch.cuda.synchronize()
    out = {"mean": mean.cpu().numpy(), "g1": g1.cpu().numpy()}
    if want_grad2:
        out["g2"] = g2.cpu().numpy()
    if want_map:
        out["map"] = smap.cpu().numpy()
    return out


def _oracle(oracle_mod, x, y, dl, padding, want_grad2, want_map=False):
    if x.ndim == 5:
        mean = oracle_mod.ssim3d(x, y, padding, want_map=want_map)
        g1, g2 = oracle_mod.ssim3d_grad(x, y, dl, padding, want_grad2)
    else:
        mean = oracle_mod.ssim2d(x, y, padding, want_map=want_map)
        g1, g2 = oracle_mod.ssim2d_grad(x, y, dl, padding, want_grad2)
    smap = None
    if want_map:
        mean, smap = mean
    return {"mean": mean, "g1": g1, "g2": g2, "map": smap}


def _assert_parity(got, ref, want_grad2, label=""):
    dm = np.max(np.abs(got["mean"].astype(np.float64) - ref["mean"]))
    assert dm <= MEAN_TOL, f"{label} mean off by {dm:.3e}"
    for k in ("g1", "g2") if want_grad2 else ("g1",):
        scale = np.max(np.abs(ref[k]))
        err = np.max(np.abs(got[k].astype(np.float64) - ref[k])) / scale
        assert np.all(np.isfinite(got[k])), f"{label} {k} has non-finite values"
        assert err <= GRAD_RTOL, f"{label} {k} relative error {err:.3e}"
    if "map" in got and ref.get("map") is not None:
        dmap = np.max(np.abs(got["map"].astype(np.float64) - ref["map"]))
        tol = MAP_TOL_3D if got["map"].ndim == 5 else MAP_TOL
        assert dmap <= tol, f"{label} map off by {dmap:.3e}"


SMALL_2D = [
    # (shape, padding, seed) -- several strips (118 / 128 columns), ragged tails
    ((1, 3, 64, 64), "valid", 1),
    ((1, 3, 64, 64), "same", 2),
    ((2, 2, 37, 301), "valid", 3),
    ((2, 2, 37, 301), "same", 4),
    ((1, 1, 250, 257), "valid", 5),
    ((1, 1, 250, 257), "same", 6),
    ((3, 1, 11, 11), "valid", 7),     # one output pixel per plane
    ((1, 4, 11, 130), "valid", 8),
    ((1, 1, 1, 1), "same", 9),
    ((2, 1, 3, 1), "same", 10),
    ((1, 2, 5, 139), "same", 11),
    ((1, 1, 129, 12), "valid", 12),   # tall and narrow
    ((1, 1, 130, 236), "same", 13),   # exactly two gradient strips
]


@pytest.mark.parametrize("path", ["saved", "recompute"])
@pytest.mark.parametrize("shape,padding,seed", SMALL_2D)
def test_parity_small_2d(dev, oracle_mod, shape, padding, seed, path):
    x, y = uniform_pair(shape, 500 + seed, std=0.08)
    dl = np.linspace(-1.0, 0.5, shape[0])
    got = _run(dev, x, y, dl, padding, True, path, want_map=True)
    ref = _oracle(oracle_mod, x, y, dl, padding, True, want_map=True)
    _assert_parity(got, ref, True, f"{shape} {padding} {path}")


@pytest.mark.parametrize("seg_rows", [22, 23, 40, 57])
@pytest.mark.parametrize("padding", ["valid", "same"])
def test_parity_forced_row_segments(dev, oracle_mod, padding, seg_rows):
    """Short row segments: the 20-row warm-up and segment ownership of the mean."""
    from differentiable_image_quality_gb300 import _abi

    x, y = uniform_pair((2, 2, 97, 150), 600 + seg_rows, std=0.1)
    dl = np.array([-1.0, -0.3])
    with _abi.using_test_library() as lib:  # the segment hook is in the test build only
        lib.gbssim_tune_seg_rows(seg_rows)
        try:
            for path in ("saved", "recompute"):
                got = _run(dev, x, y, dl, padding, True, path, want_map=True)
                ref = _oracle(oracle_mod, x, y, dl, padding, True, want_map=True)
                _assert_parity(got, ref, True, f"seg_rows={seg_rows} {padding} {path}")
        finally:
            lib.gbssim_tune_seg_rows(0)


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_pixels_do_not_depend_on_the_plan(dev, padding):
    """The 2D kernels' bands lie on one 11-row grid per image, so every window's
    shift, and with it every map value and gradient element, comes out the same
    bit for bit whatever the row segmentation (forced here to several lengths,
    some not multiples of 11).  The means sum per-segment partials, grouped by
    the plan: they may differ in their last bits."""
    from differentiable_image_quality_gb300 import _abi

    x, y = uniform_pair((1, 2, 150, 300), 700, std=0.1)
    dl = np.array([-1.0])
    runs = []
    with _abi.using_test_library() as lib:
        for seg_rows in (0, 22, 30, 47):
            lib.gbssim_tune_seg_rows(seg_rows)
            try:
                runs.append([_run(dev, x, y, dl, padding, True, path, want_map=True)
                             for path in ("saved", "recompute")])
            finally:
                lib.gbssim_tune_seg_rows(0)
    for seg_rows, got in zip((22, 30, 47), runs[1:]):
        for g, r, path in zip(got, runs[0], ("saved", "recompute")):
            label = f"{padding} seg_rows={seg_rows} {path}"
            assert np.array_equal(g["map"], r["map"]), label
            assert np.array_equal(g["g1"], r["g1"]) and np.array_equal(g["g2"], r["g2"]), label
            assert np.max(np.abs(g["mean"] - r["mean"])) <= 1e-6, label


@pytest.mark.parametrize("shape,padding,seed", [
    ((1, 3, 64, 64), "valid", 31), ((2, 2, 37, 300), "same", 32), ((1, 1, 250, 256), "valid", 33),
    ((1, 2, 130, 236), "same", 34), ((1, 1, 11, 12), "valid", 35)])
def test_forward_kernels_agree(dev, oracle_mod, shape, padding, seed):
    """Forward only and the per-octave stage on images staged by tensor copies
    run the split forward kernel; the test build can force the stream kernel
    there.  Both must match the oracle."""
    import torch

    import differentiable_image_quality_gb300 as pkg
    from differentiable_image_quality_gb300 import _abi

    x, y = uniform_pair(shape, 500 + seed, std=0.08)
    N = shape[0]
    ref_mean, ref_map = oracle_mod.ssim2d(x, y, padding, want_map=True)
    octs = 1
    while octs < 3 and min(pkg.pyramid_extents(shape[2], shape[3], octs + 1)[-1]) >= (
            11 if padding == "valid" else 1):
        octs += 1
    ref_pm, ref_pmaps = oracle_mod.ssim2d_pyramid(x, y, padding, octs, want_maps=True)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    with _abi.using_test_library() as lib:
        for split in (1, 0):
            lib.gbssim_tune_fwd_split(split)
            try:
                mean = torch.full((N,), float("nan"), device=dev)
                ho, wo = ref_map.shape[2:]
                smap = torch.full((N, shape[1], ho, wo), float("nan"), device=dev)
                pkg.ssim_fwd(tx, ty, padding, mean, out_map=smap)
                pm, pmaps = pkg.ssim_pyramid(tx, ty, padding, octs, want_maps=True)
                torch.cuda.synchronize()
            finally:
                lib.gbssim_tune_fwd_split(1)
            label = f"split={split} {shape} {padding}"
            assert np.max(np.abs(mean.cpu().numpy() - ref_mean)) <= MEAN_TOL, label
            assert np.max(np.abs(smap.cpu().numpy() - ref_map)) <= MAP_TOL, label
            assert np.max(np.abs(pm.cpu().numpy() - ref_pm)) <= MEAN_TOL, label
            for o in range(octs):
                tol = MAP_TOL if o == 0 else OCTAVE_MAP_TOL
                assert np.max(np.abs(pmaps[o].cpu().numpy() - ref_pmaps[o])) <= tol, (label, o)


@pytest.mark.parametrize("name", ["tiny64_valid", "splat1080_valid", "splat1080_same",
                                  "batch512_valid", "volume128_valid"])
@pytest.mark.parametrize("path", ["saved", "recompute"])
def test_parity_workloads(dev, oracle_mod, name, path):
    """Every workload at full size: means, gradients and the SSIM map."""
    wl = WORKLOADS[name]
    x, y = make_inputs(name)
    dl = dl_vector(name)
    got = _run(dev, x, y, dl, wl.padding, wl.want_grad2, path, want_map=True)
    ref = _oracle(oracle_mod, x, y, dl, wl.padding, wl.want_grad2, want_map=True)
    _assert_parity(got, ref, wl.want_grad2, f"{name} {path}")


SMALL_3D = [
    ((1, 1, 11, 11, 11), "valid", 1),
    ((1, 1, 12, 12, 12), "valid", 2),
    ((2, 2, 13, 19, 37), "valid", 3),
    ((1, 2, 9, 17, 40), "same", 4),
    ((2, 1, 30, 21, 45), "same", 5),    # several z segments, two tile columns
    ((1, 1, 40, 36, 70), "valid", 6),   # ragged tiles (16 x 32) in both directions
    ((1, 1, 1, 1, 1), "same", 7),
    ((1, 1, 3, 40, 2), "same", 8),
    ((1, 1, 150, 11, 12), "valid", 9),  # one output column block, many z segments
    ((1, 1, 90, 2, 3), "same", 10),     # long thin columns, padding slices at both ends
    ((3, 1, 12, 30, 17), "same", 11),   # several images: per-image means of the z kernel
    ((1, 1, 25, 140, 12), "valid", 12), # more columns than one z-kernel block
]


@pytest.mark.parametrize("path", ["saved", "recompute"])
@pytest.mark.parametrize("shape,padding,seed", SMALL_3D)
def test_parity_small_3d(dev, oracle_mod, shape, padding, seed, path):
    x, y = uniform_pair(shape, 800 + seed, std=0.08)
    dl = np.linspace(-1.0, 0.5, shape[0])
    got = _run(dev, x, y, dl, padding, True, path, want_map=True)
    ref = _oracle(oracle_mod, x, y, dl, padding, True, want_map=True)
    _assert_parity(got, ref, True, f"{shape} {padding} {path}")


def test_autograd_api_3d(dev, oracle_mod):
    import torch

    import differentiable_image_quality_gb300 as pkg

    x, y = uniform_pair((1, 2, 14, 15, 16), 703, std=0.1)
    for padding in ("valid", "same"):
        tx = torch.from_numpy(x).to(dev).requires_grad_(True)
        ty = torch.from_numpy(y).to(dev)
        loss = 1.0 - pkg.fused_ssim3d(tx, ty, padding=padding)
        loss.backward()
        ref_mean = oracle_mod.ssim3d(x, y, padding)
        g1, _ = oracle_mod.ssim3d_grad(x, y, [-1.0], padding, want_grad2=False)
        assert abs(loss.item() - (1 - ref_mean[0])) <= MEAN_TOL
        err = np.max(np.abs(tx.grad.cpu().numpy() - g1)) / np.max(np.abs(g1))
        assert err <= GRAD_RTOL


def test_deterministic_and_paths_agree(dev):
    x, y = make_inputs("batch512_valid")
    dl = dl_vector("batch512_valid")
    a = _run(dev, x, y, dl, "valid", True, "saved")
    b = _run(dev, x, y, dl, "valid", True, "saved")
    c = _run(dev, x, y, dl, "valid", True, "recompute")
    for k in ("mean", "g1", "g2"):
        np.testing.assert_array_equal(a[k], b[k])
    # the two paths differ only by where dL is applied (float32 rounding)
    assert np.max(np.abs(a["g1"] - c["g1"])) <= 1e-6 * np.max(np.abs(a["g1"]))


def test_identical_images(dev):
    x, _ = uniform_pair((1, 3, 70, 90), 700)
    for padding in ("valid", "same"):
        got = _run(dev, x, x, [-1.0], padding, True, "saved", want_map=True)
        assert abs(got["mean"][0] - 1.0) <= MEAN_TOL
        assert np.max(np.abs(got["map"] - 1.0)) <= MAP_TOL
        # the exact gradient is zero; the float32 one is rounding noise far below
        # the typical gradient of a differing pair (~1e-6 per pixel here)
        assert np.max(np.abs(got["g1"])) < 1e-8


def test_outputs_stay_inside_their_buffers(dev):
    """Guard bands around every output stay untouched (NaN sentinels elsewhere)."""
    import torch

    import differentiable_image_quality_gb300 as pkg

    shape = (2, 3, 45, 140)
    x, y = uniform_pair(shape, 701, std=0.1)
    n = int(np.prod(shape))
    guard = 4096
    for padding in ("valid", "same"):
        ho = shape[2] - 10 if padding == "valid" else shape[2]
        wo = shape[3] - 10 if padding == "valid" else shape[3]
        nmap = shape[0] * shape[1] * ho * wo
        sentinel = 12345.0
        tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
        big = torch.full((4 * guard + 2 * nmap + 2 * n + 8,), sentinel, device=dev)
        mean = big[guard: guard + 2]
        smap = big[2 * guard: 2 * guard + nmap].view(shape[0], shape[1], ho, wo)
        saved = big[3 * guard + nmap: 3 * guard + nmap + 2 * n]
        pkg.ssim_fwd(tx, ty, padding, mean, out_map=smap, saved=saved, want_grad2=True)
        g = torch.full((2 * guard + 2 * n,), sentinel, device=dev)
        g1 = g[guard: guard + n].view(shape)
        g2 = g[guard + n: guard + 2 * n].view(shape)
        pkg.ssim_bwd(torch.tensor([-1.0, 2.0], device=dev), tx, ty, padding, g1, g2)
        torch.cuda.synchronize()
        hb = big.cpu().numpy()
        assert np.all(hb[:guard] == sentinel) and np.all(hb[guard + 2: 2 * guard] == sentinel)
        assert np.all(hb[2 * guard + nmap: 3 * guard + nmap] == sentinel)
        assert np.all(hb[3 * guard + nmap + 2 * n:] == sentinel)
        hg = g.cpu().numpy()
        assert np.all(hg[:guard] == sentinel) and np.all(hg[guard + 2 * n:] == sentinel)
        assert np.all(np.isfinite(hb[2 * guard: 2 * guard + nmap]))


def test_autograd_api(dev, oracle_mod):
    import torch

    import differentiable_image_quality_gb300 as pkg

    x, y = uniform_pair((2, 3, 48, 61), 702, std=0.1)
    for padding in ("valid", "same"):
        for train in (True, False):
            tx = torch.from_numpy(x).to(dev).requires_grad_(True)
            ty = torch.from_numpy(y).to(dev).requires_grad_(True)
            loss = 1.0 - pkg.fused_ssim(tx, ty, padding=padding, train=train)
            loss.backward()
            ref_mean = oracle_mod.ssim2d(x, y, padding)
            g1, g2 = oracle_mod.ssim2d_grad(x, y, [-0.5, -0.5], padding)
            assert abs(loss.item() - (1 - ref_mean.mean())) <= MEAN_TOL
            for got, ref in ((tx.grad, g1), (ty.grad, g2)):
                err = np.max(np.abs(got.cpu().numpy() - ref)) / np.max(np.abs(ref))
                assert err <= GRAD_RTOL
    with torch.no_grad():
        tx = torch.from_numpy(x).to(dev)
        m = pkg.fused_ssim(tx, tx, padding="valid", train=False, per_image=True)
    assert m.shape == (2,) and torch.all(torch.abs(m - 1) <= MEAN_TOL)


def test_python_api_errors(dev):
    import torch

    import differentiable_image_quality_gb300 as pkg

    a = torch.rand(1, 1, 32, 32, device=dev)
    with pytest.raises(TypeError):
        pkg.fused_ssim(a.double(), a.double())
    with pytest.raises(ValueError):
        pkg.fused_ssim(a, a[:, :, :31])
    with pytest.raises(ValueError):
        pkg.fused_ssim(a.transpose(2, 3), a)
    with pytest.raises(pkg.GbssimError):
        pkg.fused_ssim(a[:, :, :10], a[:, :, :10].clone(), padding="valid")


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_parity_unaligned_base_pointers(dev, oracle_mod, padding):
    """Images that start 4 bytes past a 16-byte boundary (W % 4 == 0): the
    4-byte staging path instead of the 16-byte one."""
    import torch

    import differentiable_image_quality_gb300 as pkg

    shape = (1, 2, 40, 260)
    x, y = uniform_pair(shape, 704, std=0.1)
    n = int(np.prod(shape))
    bx = torch.empty(n + 1, device=dev)
    by = torch.empty(n + 1, device=dev)
    tx = bx[1:].view(shape)
    ty = by[1:].view(shape)
    tx.copy_(torch.from_numpy(x))
    ty.copy_(torch.from_numpy(y))
    assert tx.data_ptr() % 16 == 4
    mean = torch.empty(1, device=dev)
    saved = torch.empty(pkg.saved_bytes(shape, True) // 4, device=dev)
    pkg.ssim_fwd(tx, ty, padding, mean, saved=saved, want_grad2=True)
    g1, g2 = torch.empty_like(tx), torch.empty_like(ty)
    r1 = torch.empty_like(tx)
    dl = torch.tensor([-1.0], device=dev)
    pkg.ssim_bwd(dl, tx, ty, padding, g1, g2, saved=saved)
    pkg.ssim_bwd(dl, tx, ty, padding, r1)
    torch.cuda.synchronize()
    ref = _oracle(oracle_mod, x, y, [-1.0], padding, True)
    _assert_parity({"mean": mean.cpu().numpy(), "g1": g1.cpu().numpy(), "g2": g2.cpu().numpy()},
                   ref, True, f"unaligned {padding}")
    _assert_parity({"mean": mean.cpu().numpy(), "g1": r1.cpu().numpy()}, ref, False,
                   f"unaligned recompute {padding}")


@pytest.mark.parametrize("name", ["tiny64_valid", "splat1080_same", "batch512_valid",
                                  "volume128_valid"])
def test_single_call_forward_backward(dev, oracle_mod, name):
    """ssim_fwd_bwd / ssim3d_fwd_bwd: means, map and gradients from one call."""
    import torch

    import differentiable_image_quality_gb300 as pkg

    wl = WORKLOADS[name]
    x, y = make_inputs(name)
    dl = dl_vector(name)
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    tdl = torch.from_numpy(dl).to(dev)
    N = x.shape[0]
    mean = torch.full((N,), float("nan"), device=dev)
    g1 = torch.full_like(tx, float("nan"))
    g2 = torch.full_like(ty, float("nan")) if wl.want_grad2 else None
    ext = [s - 10 if wl.padding == "valid" else s for s in x.shape[2:]]
    smap = torch.full((N, x.shape[1], *ext), float("nan"), device=dev)
    call = pkg.ssim3d_fwd_bwd if x.ndim == 5 else pkg.ssim_fwd_bwd
    call(tx, ty, wl.padding, tdl, mean, g1, g2, out_map=smap)
    torch.cuda.synchronize()
    got = {"mean": mean.cpu().numpy(), "g1": g1.cpu().numpy(), "map": smap.cpu().numpy()}
    if wl.want_grad2:
        got["g2"] = g2.cpu().numpy()
    ref = _oracle(oracle_mod, x, y, dl, wl.padding, wl.want_grad2, want_map=True)
    _assert_parity(got, ref, wl.want_grad2, f"single call {name}")


@pytest.mark.parametrize("path", ["saved", "recompute"])
@pytest.mark.parametrize("ndim", [2, 3])
def test_nan_propagates_within_its_reach(dev, oracle_mod, path, ndim):
    """A NaN pixel of one image makes that image's mean NaN and the gradient NaN
    within 20 pixels of it (window, then adjoint); every other image and every
    pixel out of that reach keep the oracle's values."""
    shape = (2, 1, 44, 46) if ndim == 2 else (2, 1, 24, 24, 48)
    x, y = uniform_pair(shape, 4242 + ndim, std=0.08)
    dl = np.array([-1.0, 0.5])
    ref = _oracle(oracle_mod, x, y, dl, "valid", False)  # clean reference
    c = tuple(s // 2 for s in shape[2:])
    x = x.copy()
    x[(0, 0) + c] = np.nan
    got = _run(dev, x, y, dl, "valid", False, path)
    assert np.isnan(got["mean"][0])
    assert abs(got["mean"][1] - ref["mean"][1]) <= MEAN_TOL
    g = got["g1"]
    # image 1: unaffected
    err = np.max(np.abs(g[1] - ref["g1"][1])) / np.max(np.abs(ref["g1"][1]))
    assert err <= GRAD_RTOL
    # image 0: NaN inside the reach, the oracle's values (of the clean pair) far from it
    idx = np.indices(shape[2:])
    dist = np.max(np.abs(idx - np.array(c).reshape((-1,) + (1,) * len(c))), axis=0)
    assert np.isnan(g[0, 0][dist <= 10]).all()
    far = dist > 20
    assert far.any() and np.isfinite(g[0, 0][far]).all()
    scale = np.max(np.abs(ref["g1"][0]))
    assert np.max(np.abs(g[0, 0][far] - ref["g1"][0, 0][far])) / scale <= GRAD_RTOL


@pytest.mark.parametrize("path", ["saved", "recompute"])
@pytest.mark.parametrize("shape,padding", [((1, 3, 140, 300), "valid"), ((1, 3, 140, 300), "same"),
                                           ((1, 1, 30, 34, 41), "valid"), ((1, 1, 30, 34, 41), "same")])
def test_values_outside_the_unit_range(dev, oracle_mod, shape, padding, path):
    """Inputs are not checked against [0, 1] (the constants assume that range,
    the arithmetic does not): images in [-0.25, 1.25], with a block of each at
    a constant beyond the range, match the oracle at the usual bars for the
    mean and the gradients, and for 2D maps.  3D maps: the 3D kernels shift by
    1/2, so shifted values reach 0.75 instead of 0.5 and sigma11 + sigma22
    carries about twice the rounding; measured 7.3e-5 where one image is flat
    beside the other's noise, held to 1.5e-4."""
    rng = np.random.default_rng(41 + len(shape))
    x = rng.uniform(-0.25, 1.25, size=shape)
    y = np.clip(x + rng.normal(0.0, 0.05, size=shape), -0.25, 1.25)
    x[..., :20, :25] = 1.25
    y[..., :20, :25] = 1.2
    x[..., -16:, -30:] = -0.25
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.ascontiguousarray(y, dtype=np.float32)
    want_grad2 = padding == "same"
    dl = [-1.0]
    got = _run(dev, x, y, dl, padding, want_grad2, path, want_map=True)
    ref = _oracle(oracle_mod, x, y, dl, padding, want_grad2, want_map=True)
    if len(shape) == 5:
        dmap = np.max(np.abs(got.pop("map").astype(np.float64) - ref["map"]))
        assert dmap <= 1.5e-4, f"{shape} {padding} {path} map off by {dmap:.3e}"
    _assert_parity(got, ref, want_grad2, f"{shape} {padding} {path}")


@pytest.mark.parametrize("path", ["saved", "recompute"])
@pytest.mark.parametrize("shape,padding", [((1, 3, 140, 300), "valid"), ((1, 2, 140, 300), "same"),
                                           ((1, 1, 30, 34, 41), "valid"), ((1, 1, 30, 34, 41), "same")])
def test_flat_backgrounds(dev, oracle_mod, shape, padding, path):
    """Renders on a white or black background: both images exactly 1 over the
    left three quarters of the columns, exactly 0 over the top fifth of the
    rows, noise elsewhere.  In the flat windows sigma11 + sigma22 + C2 is ~C2,
    so the derivatives of S with respect to the second moments are of order
    1 / C2 there; the mean, the map and the gradients still meet the usual
    bars (the backward multiplies those derivatives by x - y)."""
    rng = np.random.default_rng(77 + len(shape))
    x = rng.random(shape)
    y = np.clip(x + rng.normal(0.0, 0.05, size=shape), 0.0, 1.0)
    W = shape[-1]
    x[..., : int(0.75 * W)] = 1.0
    y[..., : int(0.75 * W)] = 1.0
    H = shape[-2]
    x[..., : H // 5, :] = 0.0
    y[..., : H // 5, :] = 0.0
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.ascontiguousarray(y, dtype=np.float32)
    want_grad2 = padding == "same"
    dl = [-1.0]
    got = _run(dev, x, y, dl, padding, want_grad2, path, want_map=True)
    ref = _oracle(oracle_mod, x, y, dl, padding, want_grad2, want_map=True)
    _assert_parity(got, ref, want_grad2, f"{shape} {padding} {path}")


@pytest.mark.parametrize("path", ["saved", "recompute"])
@pytest.mark.parametrize("shape,padding", [((40, 3, 20, 24), "valid"), ((40, 3, 20, 24), "same"),
                                           ((12, 2, 12, 13, 14), "valid"), ((12, 2, 12, 13, 14), "same")])
def test_many_small_images(dev, oracle_mod, shape, padding, path):
    """A batch of many small images (120 planes in 2D, 24 in 3D): more planes
    than one wave of blocks holds, a per-image mean over blocks of many planes,
    per-image upstream gradients."""
    x, y = uniform_pair(shape, 4100 + len(shape), std=0.1)
    dl = np.linspace(-1.0, 0.5, shape[0])
    want_grad2 = padding == "same"
    got = _run(dev, x, y, dl, padding, want_grad2, path, want_map=True)
    ref = _oracle(oracle_mod, x, y, dl, padding, want_grad2, want_map=True)
    _assert_parity(got, ref, want_grad2, f"{shape} {padding} {path}")
