"""ssim_fwd_noalloc gives the same results as ssim_fwd.

ssim_fwd_noalloc is the forward for callers that may not allocate device memory
themselves -- a plug-in inside an application that owns the GPU's memory, or a
latency-critical caller that must not call cudaMalloc.  Instead of a caller's
workspace it uses a fixed scratch array that the library keeps on each device.
These checks call it through the C ABI (ctypes, raw device pointers) twice in a
row, on two different problems, and compare each result with ssim_fwd's, within
the bars the parity tests use; one problem per padding is also compared with
the oracle directly.  The file is named to be collected last.
"""
import numpy as np
import pytest

from workloads import make_inputs, uniform_pair

pytestmark = pytest.mark.gpu

MEAN_TOL = 1e-5
GRAD_RTOL = 1e-4
MAP_TOL = 5e-6
ETOOLARGE = -6


@pytest.fixture(scope="module")
def env():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    return torch, _abi.load(), torch.device("cuda:0")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _outputs(torch, dev, shape, padding, want_map, want_saved):
    N, C, H, W = shape
    ho, wo = (H - 10, W - 10) if padding == "valid" else (H, W)
    mean = torch.full((N,), float("nan"), device=dev)
    smap = torch.full((N, C, ho, wo), float("nan"), device=dev) if want_map else None
    saved = torch.full((2 * N * C * H * W,), float("nan"), device=dev) if want_saved else None
    return mean, smap, saved


def _case(torch, dev, x, y, padding, want_map, want_saved):
    return {"x": torch.from_numpy(x).to(dev), "y": torch.from_numpy(y).to(dev),
            "padding": padding, "map": want_map, "saved": want_saved}


def _call(torch, lib, dev, case, noalloc):
    """One forward of `case` on the current stream: through ssim_fwd_noalloc, or
    through ssim_fwd (the package's wrapper, a workspace of its own)."""
    import differentiable_image_quality_gb300 as pkg

    tx, ty = case["x"], case["y"]
    N, C, H, W = tx.shape
    mean, smap, saved = _outputs(torch, dev, tuple(tx.shape), case["padding"], case["map"],
                                 case["saved"])
    pad = 0 if case["padding"] == "valid" else 1
    nbytes = 0 if saved is None else saved.numel() * 4
    stream = torch.cuda.current_stream(dev).cuda_stream
    if noalloc:
        st = lib.ssim_fwd_noalloc(_ptr(tx), _ptr(ty), N, C, H, W, pad, _ptr(mean), _ptr(smap),
                                  _ptr(saved), nbytes, int(case["saved"]), stream)
        assert st == 0, lib.gbssim_strerror(st)
    else:
        pkg.ssim_fwd(tx, ty, case["padding"], mean, out_map=smap, saved=saved,
                     want_grad2=case["saved"])
    return mean, smap, saved


def _compare(got, ref):
    gm, gmap, gsaved = (None if t is None else t.cpu().numpy() for t in got)
    rm, rmap, rsaved = (None if t is None else t.cpu().numpy() for t in ref)
    assert np.max(np.abs(gm - rm)) <= MEAN_TOL
    if rmap is not None:
        assert np.all(np.isfinite(gmap)) and np.max(np.abs(gmap - rmap)) <= MAP_TOL
    if rsaved is not None:
        assert np.all(np.isfinite(gsaved))
        assert np.max(np.abs(gsaved - rsaved)) <= GRAD_RTOL * np.max(np.abs(rsaved))


def test_noalloc_forward_matches_ssim_fwd_on_two_calls_in_a_row(env):
    torch, lib, dev = env
    x1, y1 = make_inputs("splat1080_valid")
    x2, y2 = uniform_pair((2, 3, 97, 150), 901, std=0.1)
    cases = [_case(torch, dev, x1, y1, "valid", False, True),
             _case(torch, dev, x2, y2, "same", True, True)]
    refs = [_call(torch, lib, dev, c, noalloc=False) for c in cases]
    got = [_call(torch, lib, dev, c, noalloc=True) for c in cases]  # two calls in a row
    torch.cuda.synchronize()
    for g, r in zip(got, refs):
        _compare(g, r)
    # and the first problem again, after the second left its contents in the scratch
    again = _call(torch, lib, dev, cases[0], noalloc=True)
    torch.cuda.synchronize()
    _compare(again, refs[0])


def test_noalloc_forward_on_a_stream_of_its_own(env):
    """Two calls queued back to back on a stream the test creates (not the
    legacy default stream): the clearing of the array and each kernel stay in
    order on that stream, so both results match ssim_fwd's."""
    torch, lib, dev = env
    x1, y1 = uniform_pair((1, 3, 130, 260), 902, std=0.05)
    x2, y2 = uniform_pair((3, 1, 64, 77), 903, std=0.2)
    cases = [_case(torch, dev, x1, y1, "valid", True, False),
             _case(torch, dev, x2, y2, "same", False, True)]
    refs = [_call(torch, lib, dev, c, noalloc=False) for c in cases]
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        got = [_call(torch, lib, dev, c, noalloc=True) for c in cases]
    side.synchronize()
    for g, r in zip(got, refs):
        _compare(g, r)


def test_noalloc_forward_rejects_problems_beyond_its_scratch(env):
    _, lib, _ = env
    # 64 RGB 1080p images need more than the 1 MiB array: refused by the size
    # check, which comes first; the null pointers are never reached (were the
    # check to break, ssim_fwd's own null-pointer check would refuse them too)
    st = lib.ssim_fwd_noalloc(None, None, 64, 3, 1080, 1920, 0, None, None, None, 0, 0, None)
    assert st == ETOOLARGE
    assert b"ssim_fwd_noalloc" in lib.gbssim_strerror(st)


@pytest.mark.parametrize("padding", ["valid", "same"])
def test_noalloc_forward_matches_the_oracle(env, oracle_mod, padding):
    """The no-allocation forward against the oracle directly: per-image means,
    the map, and the saved fields, which are the gradients of each image's mean
    with respect to both images (dLoss/dmean = 1)."""
    torch, lib, dev = env
    x, y = uniform_pair((2, 3, 57, 141), 904, std=0.1)
    mean, smap, saved = _call(torch, lib, dev, _case(torch, dev, x, y, padding, True, True),
                              noalloc=True)
    torch.cuda.synchronize()
    ref_mean, ref_map = oracle_mod.ssim2d(x, y, padding, want_map=True)
    g1, g2 = oracle_mod.ssim2d_grad(x, y, np.ones(x.shape[0]), padding)
    assert np.max(np.abs(mean.cpu().numpy() - ref_mean)) <= MEAN_TOL
    assert np.max(np.abs(smap.cpu().numpy().astype(np.float64) - ref_map)) <= MAP_TOL
    fields = saved.cpu().numpy().astype(np.float64).reshape((2,) + x.shape)
    for got, ref in ((fields[0], g1), (fields[1], g2)):
        assert np.max(np.abs(got - ref)) <= GRAD_RTOL * np.max(np.abs(ref))
