"""Host-side checks of the C ABI (no GPU needed).

The library must load and export every function include/gbssim.h declares;
argument errors must come back as status codes before any CUDA call; the
float32 taps must be the roundings of the window the oracle computes.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbssim.h")

EINVAL, ESHAPE, EALIGN, EWORKSPACE = -1, -2, -3, -4
FAKE = 0x10000  # an aligned address never dereferenced: every call below fails its checks first


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#.*", "", text)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{}]*\)\s*;", text)))


@pytest.fixture(scope="module")
def lib():
    from differentiable_image_quality_gb300 import _abi, _build

    _build.build()
    return _abi.load()


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("ssim_fwd", "ssim_bwd", "ssim3d_fwd", "ssim3d_bwd", "gbssim_workspace_bytes",
                 "gbssim_saved_bytes", "gbssim_strerror"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from differentiable_image_quality_gb300 import _abi

    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gbssim.h but not exported"
        assert name in _abi.SIGNATURES, f"{name} has no ctypes signature"


def test_product_library_exports_only_the_header(lib):
    """The test hooks live in the test build; the product library's dynamic
    symbols are the header's functions and nothing else."""
    import subprocess

    from differentiable_image_quality_gb300 import _abi, _build

    for hook in _abi.TEST_SIGNATURES:
        assert not hasattr(lib, hook), f"{hook} is exported by the product library"
    test_lib = _abi.load_test()
    for hook in _abi.TEST_SIGNATURES:
        assert hasattr(test_lib, hook), f"{hook} missing from the test build"
    try:
        out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                             text=True, check=True).stdout
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("nm not available")
    exported = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert exported == declared_functions()


def test_abi_version(lib):
    assert lib.gbssim_abi_version() == 1


def test_window_is_float32_rounding_of_oracle_window(lib, oracle_mod):
    w = (ctypes.c_float * 11)()
    lib.gbssim_window(w)
    w32 = np.array(list(w), dtype=np.float32)
    np.testing.assert_array_equal(w32, oracle_mod.gauss_window().astype(np.float32))


def test_buffer_sizes(lib):
    assert lib.gbssim_saved_bytes(2, 3, 40, 50, 0) == 2 * 3 * 40 * 50 * 4
    assert lib.gbssim_saved_bytes(2, 3, 40, 50, 1) == 2 * 2 * 3 * 40 * 50 * 4
    assert lib.gbssim_workspace_bytes(1, 3, 1080, 1920, 0) > 0
    assert lib.gbssim_workspace_bytes(1, 3, 10, 1920, 0) == 0  # valid needs H >= 11
    assert lib.gbssim_workspace_bytes(1, 3, 10, 1920, 1) > 0   # same accepts it
    assert lib.gbssim_workspace_bytes(0, 3, 64, 64, 0) == 0
    assert lib.gbssim_workspace_bytes(1, 1, 64, 64, 7) == 0


def fwd(lib, img1=FAKE, img2=FAKE, N=1, C=3, H=64, W=64, pad=0, mean=FAKE, smap=None,
        saved=None, saved_bytes=0, g2=0, ws=FAKE, ws_bytes=1 << 20):
    return lib.ssim_fwd(img1, img2, N, C, H, W, pad, mean, smap, saved, saved_bytes, g2, ws,
                        ws_bytes, None)


def test_forward_argument_errors(lib):
    assert fwd(lib, img1=None) == EINVAL
    assert fwd(lib, mean=None) == EINVAL
    assert fwd(lib, img2=FAKE + 2) == EALIGN
    assert fwd(lib, pad=3) == EINVAL
    assert fwd(lib, N=0) == ESHAPE
    assert fwd(lib, C=0) == ESHAPE
    assert fwd(lib, H=10) == ESHAPE
    assert fwd(lib, W=10, pad=0) == ESHAPE
    assert fwd(lib, ws=None) == EWORKSPACE
    assert fwd(lib, ws=FAKE + 4) == EWORKSPACE
    nbytes = 1 * 3 * 64 * 64 * 4
    assert fwd(lib, saved=1 << 30, saved_bytes=nbytes - 4) == EWORKSPACE
    assert fwd(lib, saved=1 << 30, saved_bytes=nbytes, g2=1) == EWORKSPACE
    # saved overlapping an input
    assert fwd(lib, img1=1 << 30, saved=(1 << 30) + 64, saved_bytes=nbytes) == EINVAL


def test_backward_argument_errors(lib):
    n = 1 * 3 * 64 * 64 * 4

    def bwd(dL=FAKE, img1=1 << 30, img2=2 << 30, grad1=3 << 30, grad2=None, saved=None,
            saved_bytes=0, pad=0, H=64):
        return lib.ssim_bwd(dL, img1, img2, 1, 3, H, 64, pad, saved, saved_bytes, grad1, grad2,
                            None)

    assert bwd(dL=None) == EINVAL
    assert bwd(grad1=None) == EINVAL
    assert bwd(grad1=(1 << 30) + 8) == EINVAL            # overlaps img1
    assert bwd(grad2=(3 << 30) + n - 4) == EINVAL        # overlaps grad1
    assert bwd(grad1=(3 << 30) + 1) == EALIGN
    assert bwd(pad=-1) == EINVAL
    assert bwd(H=10) == ESHAPE
    assert bwd(saved=4 << 30, saved_bytes=n - 4) == EWORKSPACE
    assert bwd(saved=4 << 30, saved_bytes=n, grad2=5 << 30) == EWORKSPACE
    assert bwd(saved=3 << 30, saved_bytes=n, grad1=(3 << 30) + 4) == EINVAL  # shifted alias


def test_strerror(lib):
    assert lib.gbssim_strerror(0) == b"ok"
    for st in (EINVAL, ESHAPE, EALIGN, EWORKSPACE, -5):
        assert len(lib.gbssim_strerror(st)) > 10
    assert lib.gbssim_strerror(123) == b"unknown status"


def test_python_api_rejects_cpu_tensors():
    import torch

    import differentiable_image_quality_gb300 as pkg

    x = torch.zeros(1, 1, 16, 16)
    with pytest.raises(TypeError):
        pkg.fused_ssim(x, x)


def test_3d_argument_errors(lib):
    n = 1 * 1 * 12 * 12 * 12 * 4
    ws = lib.gbssim3d_workspace_bytes(1, 1, 12, 12, 12, 0)
    assert ws > 2 * 2 * 2 * 16  # derivative fields of the 2x2x2 output domain
    assert lib.gbssim3d_workspace_bytes(1, 1, 10, 12, 12, 0) == 0
    assert lib.gbssim3d_saved_bytes(1, 1, 12, 12, 12, 1) == 2 * n

    def fwd(D=12, pad=0, wsp=FAKE * 256, wsb=ws, saved=None, sb=0):
        return lib.ssim3d_fwd(1 << 30, 2 << 30, 1, 1, D, 12, 12, pad, 3 << 30, None, saved, sb, 0,
                              wsp, wsb, None)

    assert fwd(D=10) == ESHAPE
    assert fwd(pad=2) == EINVAL
    assert fwd(wsb=ws - 1) == EWORKSPACE
    assert fwd(wsp=FAKE * 256 + 16) == EWORKSPACE  # workspace must be 256-byte aligned
    assert fwd(saved=4 << 30, sb=n - 4) == EWORKSPACE

    def bwd(wsp=FAKE * 256, wsb=ws, saved=None, sb=0, g1=5 << 30):
        return lib.ssim3d_bwd(FAKE, 1 << 30, 2 << 30, 1, 1, 12, 12, 12, 0, saved, sb, g1, None,
                              wsp, wsb, None)

    assert bwd(wsp=None) == EWORKSPACE
    assert bwd(wsb=ws - 1) == EWORKSPACE
    assert bwd(g1=(1 << 30) + 4) == EINVAL
    assert bwd(saved=4 << 30, sb=n - 4, wsp=None) == EWORKSPACE


def test_pyramid_sizes_and_argument_errors(lib):
    # 64 x 64 valid: octave extents 64, 32, 16 (outputs 54, 22, 6); a fourth (8) is too small
    per = [54 * 54, 22 * 22, 6 * 6]
    assert lib.gbssim_pyramid_map_floats(1, 3, 64, 64, 0, 3) == 3 * 3 * sum(per)
    assert lib.gbssim_pyramid_map_floats(1, 3, 64, 64, 0, 4) == 0
    assert lib.gbssim_pyramid_workspace_bytes(1, 3, 64, 64, 0, 4) == 0
    assert lib.gbssim_pyramid_workspace_bytes(1, 3, 64, 64, 0, 0) == 0
    assert lib.gbssim_pyramid_workspace_bytes(1, 3, 64, 64, 1, 7) > 0  # same: down to 1 x 1
    ws = lib.gbssim_pyramid_workspace_bytes(1, 3, 64, 64, 0, 3)
    # the downscaled pairs of octaves 1 and 2 live in the workspace
    assert ws >= 2 * 3 * (32 * 32 + 16 * 16) * 4

    def pyr(img1=1 << 30, img2=2 << 30, octaves=3, pad=0, means=3 << 30, maps=None,
            wsp=FAKE * 256, wsb=ws):
        return lib.ssim_pyramid(img1, img2, 1, 3, 64, 64, pad, octaves, means, maps, wsp, wsb,
                                None)

    assert pyr(img1=None) == EINVAL
    assert pyr(means=None) == EINVAL
    assert pyr(means=(3 << 30) + 2) == EALIGN
    assert pyr(pad=4) == EINVAL
    assert pyr(octaves=4) == ESHAPE
    assert pyr(octaves=0) == ESHAPE
    assert pyr(wsb=ws - 1) == EWORKSPACE
    assert pyr(wsp=FAKE * 256 + 16) == EWORKSPACE
    assert pyr(maps=(1 << 30) + 64) == EINVAL  # maps overlapping img1
    assert pyr(wsp=3 << 30) == EINVAL             # workspace overlapping the means
