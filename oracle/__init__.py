"""The double-precision CPU oracle of the differentiable SSIM loss.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may build, load or call anything here; the CUDA
library never does, and this module never imports it.

The arithmetic lives in ``ssim_oracle.c`` (plain C, double precision, direct
11x11 / 11x11x11 window sums, no separable passes); this file compiles it with
gcc into ``oracle/_build/libssim_oracle.so`` and wraps it with ctypes.  Arrays
go in and come out as float64 numpy arrays; float32 inputs are widened exactly.

Sources followed (see the C file's header for the details):
TriSSIM README "How it works" (the five blurred quantities, the adjoint and the
chain rule), fused-ssim README introduction, "Usage", "Constraints" and
"3D data" (the 11-tap window, padding modes, data range, 3D); the ssimulacra2
hand-off page's per-octave loop (a 2x downscale between octaves, then blur,
sigma maps and error maps per octave), read for SSIM as the maps l, cs and S.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssim_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libssim_oracle.so")

PADDING = {"valid": 0, "same": 1}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP: single thread
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        llp = ctypes.POINTER(ctypes.c_longlong)
        i = ctypes.c_int
        lib.oracle_gauss_window.argtypes = [dp]
        lib.oracle_gauss_window.restype = None
        lib.oracle_out_extent.argtypes = [i, i]
        lib.oracle_out_extent.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        lib.oracle_set_num_threads.argtypes = [i]
        lib.oracle_set_num_threads.restype = None
        lib.oracle_blur2d.argtypes = [dp, i, i, i, dp]
        lib.oracle_blur2d_adjoint.argtypes = [dp, i, i, i, dp]
        lib.oracle_blur3d.argtypes = [dp, i, i, i, i, dp]
        lib.oracle_blur3d_adjoint.argtypes = [dp, i, i, i, i, dp]
        lib.oracle_ssim2d_stats.argtypes = [dp, dp, i, i, i, i, i, dp]
        lib.oracle_ssim2d.argtypes = [dp, dp, i, i, i, i, i, dp, dp]
        lib.oracle_ssim2d_grad.argtypes = [dp, dp, dp, i, i, i, i, i, dp, dp]
        lib.oracle_ssim2d_grad_at.argtypes = [dp, dp, dp, i, i, i, i, i, ctypes.c_longlong,
                                              llp, dp, dp]
        lib.oracle_ssim3d.argtypes = [dp, dp, i, i, i, i, i, i, dp, dp]
        lib.oracle_ssim3d_grad.argtypes = [dp, dp, dp, i, i, i, i, i, i, dp, dp]
        lib.oracle_ssim3d_grad_at.argtypes = [dp, dp, dp, i, i, i, i, i, i, ctypes.c_longlong,
                                              llp, dp, dp]
        lib.oracle_ssim3d_map_at.argtypes = [dp, dp, i, i, i, i, i, i, ctypes.c_longlong,
                                              ctypes.POINTER(ctypes.c_longlong), dp]
        lib.oracle_downscale2x.argtypes = [dp, i, i, dp]
        lib.oracle_ssim2d_components.argtypes = [dp, dp, i, i, i, i, i, dp, dp, dp, dp]
        lib.oracle_ssim_point.argtypes = [ctypes.c_double] * 5 + [dp]
        lib.oracle_ssim_point.restype = ctypes.c_double
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad argument")


def _pad(padding: str) -> int:
    try:
        return PADDING[padding]
    except KeyError:
        raise ValueError(f"padding must be 'valid' or 'same', got {padding!r}") from None


def set_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (independent outputs only)."""
    _load().oracle_set_num_threads(int(n))


def gauss_window() -> np.ndarray:
    w = np.zeros(11, dtype=np.float64)
    _load().oracle_gauss_window(_ptr(w))
    return w


def out_extent(n: int, padding: str) -> int:
    return int(_load().oracle_out_extent(int(n), _pad(padding)))


def blur2d(f, padding: str) -> np.ndarray:
    f = _f64(f)
    H, W = f.shape
    out = np.empty((out_extent(H, padding), out_extent(W, padding)))
    _check(_load().oracle_blur2d(_ptr(f), H, W, _pad(padding), _ptr(out)), "blur2d")
    return out


def blur2d_adjoint(g, H: int, W: int, padding: str) -> np.ndarray:
    g = _f64(g)
    if g.shape != (out_extent(H, padding), out_extent(W, padding)):
        raise ValueError("g must have the output extent of an H x W image")
    out = np.empty((H, W))
    _check(_load().oracle_blur2d_adjoint(_ptr(g), H, W, _pad(padding), _ptr(out)),
           "blur2d_adjoint")
    return out


def blur3d(f, padding: str) -> np.ndarray:
    f = _f64(f)
    D, H, W = f.shape
    out = np.empty(tuple(out_extent(s, padding) for s in (D, H, W)))
    _check(_load().oracle_blur3d(_ptr(f), D, H, W, _pad(padding), _ptr(out)), "blur3d")
    return out


def blur3d_adjoint(g, D: int, H: int, W: int, padding: str) -> np.ndarray:
    g = _f64(g)
    if g.shape != tuple(out_extent(s, padding) for s in (D, H, W)):
        raise ValueError("g must have the output extent of a D x H x W volume")
    out = np.empty((D, H, W))
    _check(_load().oracle_blur3d_adjoint(_ptr(g), D, H, W, _pad(padding), _ptr(out)),
           "blur3d_adjoint")
    return out


def ssim_point(mu1, mu2, e11, e22, e12):
    """(S, [dS/dmu1, dS/dmu2, dS/de11, dS/de22, dS/de12]) at one set of moments."""
    d = np.zeros(5)
    s = _load().oracle_ssim_point(float(mu1), float(mu2), float(e11), float(e22), float(e12),
                                  _ptr(d))
    return float(s), d


def ssim2d_stats(x, y, padding: str) -> np.ndarray:
    """(N, C, 5, Ho, Wo): mu1, mu2, E[x^2], E[y^2], E[xy] under the window."""
    x, y = _f64(x), _f64(y)
    N, C, H, W = x.shape
    out = np.empty((N, C, 5, out_extent(H, padding), out_extent(W, padding)))
    _check(_load().oracle_ssim2d_stats(_ptr(x), _ptr(y), N, C, H, W, _pad(padding), _ptr(out)),
           "ssim2d_stats")
    return out


def ssim2d(x, y, padding: str, want_map: bool = False):
    """Per-image mean SSIM (N,), and the SSIM map (N, C, Ho, Wo) when asked."""
    x, y = _f64(x), _f64(y)
    if x.shape != y.shape or x.ndim != 4:
        raise ValueError("x and y must be NCHW arrays of one shape")
    N, C, H, W = x.shape
    mean = np.empty(N)
    smap = (np.empty((N, C, out_extent(H, padding), out_extent(W, padding)))
            if want_map else None)
    _check(_load().oracle_ssim2d(_ptr(x), _ptr(y), N, C, H, W, _pad(padding), _ptr(mean),
                                 _ptr(smap)), "ssim2d")
    return (mean, smap) if want_map else mean


def ssim2d_grad(x, y, dL, padding: str, want_grad2: bool = True):
    """(grad1, grad2 or None) of sum_n dL[n] * mean[n]."""
    x, y = _f64(x), _f64(y)
    N, C, H, W = x.shape
    dL = _f64(np.broadcast_to(np.asarray(dL, dtype=np.float64), (N,)))
    g1 = np.empty_like(x)
    g2 = np.empty_like(x) if want_grad2 else None
    _check(_load().oracle_ssim2d_grad(_ptr(x), _ptr(y), _ptr(dL), N, C, H, W, _pad(padding),
                                      _ptr(g1), _ptr(g2)), "ssim2d_grad")
    return g1, g2


def ssim2d_grad_at(x, y, dL, padding: str, flat_idx, want_grad2: bool = True):
    """Gradients at the given flat NCHW indices only."""
    x, y = _f64(x), _f64(y)
    N, C, H, W = x.shape
    dL = _f64(np.broadcast_to(np.asarray(dL, dtype=np.float64), (N,)))
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    g1 = np.empty(idx.shape[0])
    g2 = np.empty(idx.shape[0]) if want_grad2 else None
    rc = _load().oracle_ssim2d_grad_at(
        _ptr(x), _ptr(y), _ptr(dL), N, C, H, W, _pad(padding), int(idx.shape[0]),
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)), _ptr(g1), _ptr(g2))
    _check(rc, "ssim2d_grad_at")
    return g1, g2


def ssim3d(x, y, padding: str, want_map: bool = False):
    x, y = _f64(x), _f64(y)
    if x.shape != y.shape or x.ndim != 5:
        raise ValueError("x and y must be NCDHW arrays of one shape")
    N, C, D, H, W = x.shape
    mean = np.empty(N)
    smap = (np.empty((N, C) + tuple(out_extent(s, padding) for s in (D, H, W)))
            if want_map else None)
    _check(_load().oracle_ssim3d(_ptr(x), _ptr(y), N, C, D, H, W, _pad(padding), _ptr(mean),
                                 _ptr(smap)), "ssim3d")
    return (mean, smap) if want_map else mean


def ssim3d_grad(x, y, dL, padding: str, want_grad2: bool = True):
    x, y = _f64(x), _f64(y)
    N, C, D, H, W = x.shape
    dL = _f64(np.broadcast_to(np.asarray(dL, dtype=np.float64), (N,)))
    g1 = np.empty_like(x)
    g2 = np.empty_like(x) if want_grad2 else None
    _check(_load().oracle_ssim3d_grad(_ptr(x), _ptr(y), _ptr(dL), N, C, D, H, W, _pad(padding),
                                      _ptr(g1), _ptr(g2)), "ssim3d_grad")
    return g1, g2


def ssim3d_grad_at(x, y, dL, padding: str, flat_idx, want_grad2: bool = True):
    x, y = _f64(x), _f64(y)
    N, C, D, H, W = x.shape
    dL = _f64(np.broadcast_to(np.asarray(dL, dtype=np.float64), (N,)))
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    g1 = np.empty(idx.shape[0])
    g2 = np.empty(idx.shape[0]) if want_grad2 else None
    rc = _load().oracle_ssim3d_grad_at(
        _ptr(x), _ptr(y), _ptr(dL), N, C, D, H, W, _pad(padding), int(idx.shape[0]),
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)), _ptr(g1), _ptr(g2))
    _check(rc, "ssim3d_grad_at")
    return g1, g2


def ssim3d_map_at(x, y, padding: str, flat_idx) -> np.ndarray:
    """S at the given flat indices of the NCDHW output domain (the map of
    ssim3d(..., want_map=True) at those places, without forming all of it)."""
    x, y = _f64(x), _f64(y)
    N, C, D, H, W = x.shape
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    out = np.empty(idx.shape[0])
    rc = _load().oracle_ssim3d_map_at(
        _ptr(x), _ptr(y), N, C, D, H, W, _pad(padding), int(idx.shape[0]),
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)), _ptr(out))
    _check(rc, "ssim3d_map_at")
    return out


def downscale2x(f) -> np.ndarray:
    """One octave down: means of 2x2 blocks, ragged edges over their in-range pixels."""
    f = _f64(f)
    H, W = f.shape
    out = np.empty(((H + 1) // 2, (W + 1) // 2))
    _check(_load().oracle_downscale2x(_ptr(f), H, W, _ptr(out)), "downscale2x")
    return out


def ssim2d_components(x, y, padding: str, want_maps: bool = False):
    """Per-image means (3, N) of the luminance term l, the contrast-structure term
    cs and S = l * cs; with want_maps also the maps (3, N, C, Ho, Wo)."""
    x, y = _f64(x), _f64(y)
    if x.shape != y.shape or x.ndim != 4:
        raise ValueError("x and y must be NCHW arrays of one shape")
    N, C, H, W = x.shape
    means = np.empty((3, N))
    maps = (np.empty((3, N, C, out_extent(H, padding), out_extent(W, padding)))
            if want_maps else None)
    _check(_load().oracle_ssim2d_components(
        _ptr(x), _ptr(y), N, C, H, W, _pad(padding),
        _ptr(maps[0]) if want_maps else None, _ptr(maps[1]) if want_maps else None,
        _ptr(maps[2]) if want_maps else None, _ptr(means)), "ssim2d_components")
    return (means, maps) if want_maps else means


def downscale_pair(x, y):
    """Both NCHW images one octave down (every plane with downscale2x)."""
    x, y = _f64(x), _f64(y)
    N, C, H, W = x.shape
    ox = np.empty((N, C, (H + 1) // 2, (W + 1) // 2))
    oy = np.empty_like(ox)
    for n in range(N):
        for c in range(C):
            ox[n, c] = downscale2x(x[n, c])
            oy[n, c] = downscale2x(y[n, c])
    return ox, oy


def ssim2d_pyramid(x, y, padding: str, octaves: int, want_maps: bool = False):
    """Per-octave SSIM components: octave 0 is the input pair, octave o + 1 the
    pair of octave o one level down.  Returns means (octaves, 3, N) and, with
    want_maps, the list of per-octave maps (3, N, C, Ho, Wo)."""
    x, y = _f64(x), _f64(y)
    means, maps = [], []
    for o in range(octaves):
        if o:
            x, y = downscale_pair(x, y)
        r = ssim2d_components(x, y, padding, want_maps)
        if want_maps:
            means.append(r[0])
            maps.append(r[1])
        else:
            means.append(r)
    means = np.stack(means)
    return (means, maps) if want_maps else means
