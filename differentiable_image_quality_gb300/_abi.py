"""ctypes view of the C ABI declared in include/gbssim.h.

Only argument marshalling happens here: tensors become device pointers, the
current CUDA stream becomes the `stream` argument, and a negative status
becomes a Python exception.  Every step of the computation runs in libgbssim.so.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

from . import _build

VALID, SAME = 0, 1
PADDING = {"valid": VALID, "same": SAME}

_lock = threading.Lock()
_lib = None       # the product library
_test_lib = None  # the test build, loaded on request
_active = None    # the library the package's calls go to (None: the product library)

# names the header declares, with (restype, argtypes)
_vp, _sz, _i, _fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "gbssim_abi_version": (_i, []),
    "gbssim_strerror": (ctypes.c_char_p, [_i]),
    "gbssim_device_status": (_i, [ctypes.POINTER(ctypes.c_uint)]),
    "gbssim_window": (None, [ctypes.POINTER(ctypes.c_float)]),
    "gbssim_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "gbssim_saved_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "ssim_fwd": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _fp, _fp, _fp, _sz, _i, _vp, _sz, _vp]),
    "ssim_bwd": (_i, [_fp, _fp, _fp, _i, _i, _i, _i, _i, _fp, _sz, _fp, _fp, _vp]),
    "ssim_fwd_noalloc": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _fp, _fp, _fp, _sz, _i, _vp]),
    "ssim_fwd_bwd": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _fp, _fp, _fp, _fp, _fp, _vp, _sz, _vp]),
    "ssim3d_fwd_bwd": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _i, _fp, _fp, _fp, _fp, _fp, _vp, _sz,
                            _vp]),
    "gbssim_pyramid_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "gbssim_pyramid_map_floats": (_sz, [_i, _i, _i, _i, _i, _i]),
    "ssim_pyramid": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _i, _fp, _fp, _vp, _sz, _vp]),
    "gbssim3d_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "gbssim3d_saved_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "ssim3d_fwd": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _i, _fp, _fp, _fp, _sz, _i, _vp, _sz, _vp]),
    "ssim3d_bwd": (_i, [_fp, _fp, _fp, _i, _i, _i, _i, _i, _i, _fp, _sz, _fp, _fp, _vp, _sz,
                        _vp]),
}
# exported only by the test build (libgbssim_test.so, csrc/gbssim_test_hooks.h):
# forced row segments, the staging modes that drive the tests of the bounded-wait
# failure path, and the per-stage statistics dump
TEST_SIGNATURES = {
    "gbssim_tune_seg_rows": (None, [_i]),
    "gbssim_tune_staging": (None, [_i]),
    "gbssim_tune_fwd_split": (None, [_i]),
    "gbssim_test_stage_dump2d": (_i, [_fp, _fp, _i, _i, _i, _i, _i, _fp, _fp, _fp, _fp, _vp]),
}


class GbssimError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed: status {status}: {message}")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def _open(path: str, signatures: dict):
    lib = ctypes.CDLL(path)
    for name, (res, args) in signatures.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(build_if_missing: bool = False):
    """The library the package's calls go to: libgbssim.so unless a test has
    switched to the test build (using_test_library).  Raises when it has not
    been built (no fallback)."""
    global _lib
    with _lock:
        if _active is not None:
            return _active
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if build_if_missing:
                _build.build()
            else:
                raise RuntimeError(
                    "libgbssim.so is not built: run `python -c \"import __graft_entry__ as g; "
                    "g.build()\"` or differentiable_image_quality_gb300._build.build()")
        _lib = _open(_build.LIB, SIGNATURES)
        return _lib


def load_test():
    """The test build libgbssim_test.so (the product ABI plus TEST_SIGNATURES)."""
    global _test_lib
    with _lock:
        if _test_lib is None:
            if not os.path.exists(_build.TEST_LIB):
                raise RuntimeError("libgbssim_test.so is not built: run _build.build()")
            _test_lib = _open(_build.TEST_LIB, {**SIGNATURES, **TEST_SIGNATURES})
        return _test_lib


@contextlib.contextmanager
def using_test_library():
    """Route the package's calls to the test build inside the block (tests of
    the staging hooks); yields that library."""
    global _active
    lib = load_test()
    with _lock:
        prev, _active = _active, lib
    try:
        yield lib
    finally:
        with _lock:
            _active = prev


def check(fn: str, status: int) -> None:
    if status != 0:
        msg = load().gbssim_strerror(status).decode()
        raise GbssimError(fn, status, msg)


def ptr(t) -> int | None:
    return None if t is None else t.data_ptr()
