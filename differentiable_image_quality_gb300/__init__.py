"""A fused, differentiable SSIM loss for NVIDIA GB300 (sm_103a).

The computation runs in hand-written CUDA kernels behind the C ABI of
include/gbssim.h (libgbssim.so); this package only marshals torch tensors,
streams and workspace memory to it.  There is no CPU or PyTorch fallback: if
the library is not built, or a tensor is not a contiguous float32 CUDA tensor,
the call raises.

Python API (fused-ssim README, "Usage" and "3D data"; TriSSIM README, "Usage"):

    fused_ssim(img1, img2, padding="same", train=True, per_image=False)
    fused_ssim3d(img1, img2, padding="same", train=True, per_image=False)

img1/img2 are NCHW (NCDHW) float32 tensors in [0, 1].  The result is the mean
SSIM over the batch (a scalar), or the per-image means with per_image=True.
Both images may require gradients; training code uses ``loss = 1 - fused_ssim(...)``.
With train=True and a gradient required, the forward also produces the
gradient fields of the per-image means, so the backward is one scaling pass;
train=False is the inference mode (and a later backward recomputes).  The
choice is per call: a grad-enabled forward that no backward will follow (a
validation loss under autograd) should pass train=False, which skips the
gradient work the stored path does inside the forward.  Calls on different
CUDA streams may run concurrently: each stream gets its own scratch buffer.

The thin wrappers ssim_fwd / ssim_bwd / ssim3d_fwd / ssim3d_bwd expose the C
ABI calls one to one on torch tensors.

    ssim_pyramid(img1, img2, padding, octaves, want_maps=False)

is the forward-only per-octave stage (2x box-downscaled octaves; per octave the
luminance term l, the contrast-structure term cs and S = l * cs, their maps and
per-image means).
"""
from __future__ import annotations

import torch

from . import _abi
from ._abi import SAME, VALID, GbssimError

__all__ = [
    "fused_ssim",
    "fused_ssim3d",
    "ssim_fwd",
    "ssim_bwd",
    "ssim3d_fwd",
    "ssim3d_bwd",
    "ssim_fwd_bwd",
    "ssim3d_fwd_bwd",
    "ssim_pyramid",
    "pyramid_extents",
    "workspace_bytes",
    "saved_bytes",
    "window",
    "GbssimError",
    "VALID",
    "SAME",
]


def _pad(padding) -> int:
    if isinstance(padding, int) and padding in (VALID, SAME):
        return padding
    try:
        return _abi.PADDING[padding]
    except KeyError:
        raise ValueError(f"padding must be 'valid' or 'same', got {padding!r}") from None


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _check_pair(img1: torch.Tensor, img2: torch.Tensor, ndim: int) -> None:
    for name, t in (("img1", img1), ("img2", img2)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32, got {t.dtype}")
        if t.dim() != ndim + 2:
            raise ValueError(f"{name} must have {ndim + 2} dimensions, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if img1.shape != img2.shape or img1.device != img2.device:
        raise ValueError("img1 and img2 must have one shape and one device")


def window() -> list:
    """The eleven float32 taps the kernels use."""
    import ctypes

    w = (ctypes.c_float * 11)()
    _abi.load().gbssim_window(w)
    return list(w)


def workspace_bytes(shape, padding) -> int:
    lib = _abi.load()
    if len(shape) == 4:
        return int(lib.gbssim_workspace_bytes(*shape, _pad(padding)))
    return int(lib.gbssim3d_workspace_bytes(*shape, _pad(padding)))


def saved_bytes(shape, want_grad2: bool) -> int:
    lib = _abi.load()
    if len(shape) == 4:
        return int(lib.gbssim_saved_bytes(*shape, int(want_grad2)))
    return int(lib.gbssim3d_saved_bytes(*shape, int(want_grad2)))


_ws_cache: dict = {}


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """A zero-filled scratch buffer per (device, current stream), grown on
    demand (256-byte aligned, as the caching allocator returns).  The library
    leaves its counter zero after every completed call, and calls on one stream
    run one after another, so a stream's calls can share its buffer; calls on
    different streams get different buffers and may run at the same time."""
    stream = torch.cuda.current_stream(device)
    key = (device.type, device.index, stream.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        # allocated on the stream that will use it: the caching allocator orders
        # its zero-fill before that stream's later work
        buf = torch.zeros(max(nbytes, 4096), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


# ----------------------------------------------------------------- thin wrappers

def ssim_fwd(img1, img2, padding, out_mean, out_map=None, saved=None, want_grad2=False,
             workspace=None):
    _check_pair(img1, img2, 2)
    N, C, H, W = img1.shape
    pad = _pad(padding)
    lib = _abi.load()
    need = int(lib.gbssim_workspace_bytes(N, C, H, W, pad))
    if workspace is None:
        workspace = _workspace(img1.device, need)
    st = lib.ssim_fwd(_abi.ptr(img1), _abi.ptr(img2), N, C, H, W, pad, _abi.ptr(out_mean),
                      _abi.ptr(out_map), _abi.ptr(saved),
                      0 if saved is None else saved.numel() * saved.element_size(),
                      int(bool(want_grad2)), _abi.ptr(workspace),
                      workspace.numel() * workspace.element_size(), _stream(img1))
    _abi.check("ssim_fwd", st)


def ssim_bwd(dL, img1, img2, padding, grad1, grad2=None, saved=None):
    _check_pair(img1, img2, 2)
    N, C, H, W = img1.shape
    lib = _abi.load()
    st = lib.ssim_bwd(_abi.ptr(dL), _abi.ptr(img1), _abi.ptr(img2), N, C, H, W, _pad(padding),
                      _abi.ptr(saved), 0 if saved is None else saved.numel() * saved.element_size(),
                      _abi.ptr(grad1), _abi.ptr(grad2), _stream(img1))
    _abi.check("ssim_bwd", st)


def ssim3d_fwd(img1, img2, padding, out_mean, out_map=None, saved=None, want_grad2=False,
               workspace=None):
    _check_pair(img1, img2, 3)
    N, C, D, H, W = img1.shape
    pad = _pad(padding)
    lib = _abi.load()
    need = int(lib.gbssim3d_workspace_bytes(N, C, D, H, W, pad))
    if workspace is None:
        workspace = _workspace(img1.device, need)
    st = lib.ssim3d_fwd(_abi.ptr(img1), _abi.ptr(img2), N, C, D, H, W, pad, _abi.ptr(out_mean),
                        _abi.ptr(out_map), _abi.ptr(saved),
                        0 if saved is None else saved.numel() * saved.element_size(),
                        int(bool(want_grad2)), _abi.ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(img1))
    _abi.check("ssim3d_fwd", st)


def ssim3d_bwd(dL, img1, img2, padding, grad1, grad2=None, saved=None, workspace=None):
    _check_pair(img1, img2, 3)
    N, C, D, H, W = img1.shape
    pad = _pad(padding)
    lib = _abi.load()
    if saved is None and workspace is None:
        workspace = _workspace(img1.device, int(lib.gbssim3d_workspace_bytes(N, C, D, H, W, pad)))
    st = lib.ssim3d_bwd(_abi.ptr(dL), _abi.ptr(img1), _abi.ptr(img2), N, C, D, H, W, pad,
                        _abi.ptr(saved),
                        0 if saved is None else saved.numel() * saved.element_size(),
                        _abi.ptr(grad1), _abi.ptr(grad2), _abi.ptr(workspace),
                        0 if workspace is None else workspace.numel() * workspace.element_size(),
                        _stream(img1))
    _abi.check("ssim3d_bwd", st)


def ssim_fwd_bwd(img1, img2, padding, dL, out_mean, grad1, grad2=None, out_map=None,
                 workspace=None):
    """Forward and backward in one call (dL = dLoss/dmean[n] known beforehand)."""
    _check_pair(img1, img2, 2)
    N, C, H, W = img1.shape
    pad = _pad(padding)
    lib = _abi.load()
    if workspace is None:
        workspace = _workspace(img1.device, int(lib.gbssim_workspace_bytes(N, C, H, W, pad)))
    st = lib.ssim_fwd_bwd(_abi.ptr(img1), _abi.ptr(img2), N, C, H, W, pad, _abi.ptr(dL),
                          _abi.ptr(out_mean), _abi.ptr(out_map), _abi.ptr(grad1), _abi.ptr(grad2),
                          _abi.ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream(img1))
    _abi.check("ssim_fwd_bwd", st)


def ssim3d_fwd_bwd(img1, img2, padding, dL, out_mean, grad1, grad2=None, out_map=None,
                   workspace=None):
    """ssim_fwd_bwd for NCDHW volumes."""
    _check_pair(img1, img2, 3)
    N, C, D, H, W = img1.shape
    pad = _pad(padding)
    lib = _abi.load()
    if workspace is None:
        workspace = _workspace(img1.device,
                               int(lib.gbssim3d_workspace_bytes(N, C, D, H, W, pad)))
    st = lib.ssim3d_fwd_bwd(_abi.ptr(img1), _abi.ptr(img2), N, C, D, H, W, pad, _abi.ptr(dL),
                            _abi.ptr(out_mean), _abi.ptr(out_map), _abi.ptr(grad1),
                            _abi.ptr(grad2), _abi.ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(img1))
    _abi.check("ssim3d_fwd_bwd", st)


def pyramid_extents(H: int, W: int, octaves: int) -> list:
    """(H_o, W_o) of octaves 0 .. octaves-1: each halves the last, rounding up."""
    out = []
    for _ in range(octaves):
        out.append((H, W))
        H, W = (H + 1) // 2, (W + 1) // 2
    return out


def ssim_pyramid(img1, img2, padding, octaves: int, want_maps: bool = False, out_means=None,
                 maps=None, workspace=None):
    """Per-octave SSIM components of NCHW float32 CUDA images.

    Returns (means, maps): means is a (octaves, 3, N) float32 tensor -- per octave
    the per-image means of l, cs and S -- and maps, with want_maps (or a given
    flat ``maps`` buffer), a list of per-octave (3, N, C, Ho, Wo) views of the
    l, cs and S maps; else None."""
    _check_pair(img1, img2, 2)
    N, C, H, W = img1.shape
    pad = _pad(padding)
    lib = _abi.load()
    need = int(lib.gbssim_pyramid_workspace_bytes(N, C, H, W, pad, int(octaves)))
    if need == 0:
        raise ValueError(f"invalid shape {tuple(img1.shape)} for {octaves} octaves "
                         f"with padding {padding!r}")
    if workspace is None:
        workspace = _workspace(img1.device, need)
    if out_means is None:
        out_means = torch.empty((int(octaves), 3, N), dtype=torch.float32, device=img1.device)
    nf = int(lib.gbssim_pyramid_map_floats(N, C, H, W, pad, int(octaves)))
    if maps is None and want_maps:
        maps = torch.empty(nf, dtype=torch.float32, device=img1.device)
    if maps is not None and (maps.numel() < nf or maps.dtype != torch.float32
                             or not maps.is_contiguous() or maps.device != img1.device):
        raise ValueError(f"maps must be a contiguous float32 tensor of at least {nf} elements "
                         f"on {img1.device}")
    if out_means.shape != (int(octaves), 3, N) or out_means.dtype != torch.float32:
        raise ValueError(f"out_means must be a float32 tensor of shape ({int(octaves)}, 3, {N})")
    st = lib.ssim_pyramid(_abi.ptr(img1), _abi.ptr(img2), N, C, H, W, pad, int(octaves),
                          _abi.ptr(out_means), _abi.ptr(maps), _abi.ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(img1))
    _abi.check("ssim_pyramid", st)
    views = None
    if maps is not None:
        views, pos = [], 0
        for h, w in pyramid_extents(H, W, int(octaves)):
            ho, wo = (h - 10, w - 10) if pad == VALID else (h, w)
            n = 3 * N * C * ho * wo
            views.append(maps[pos:pos + n].view(3, N, C, ho, wo))
            pos += n
    return out_means, views


# ----------------------------------------------------------------- autograd

class _FusedSSIM(torch.autograd.Function):
    @staticmethod
    def forward(ctx, img1, img2, padding, train, ndim):
        _check_pair(img1, img2, ndim)
        fwd = ssim_fwd if ndim == 2 else ssim3d_fwd
        N = img1.shape[0]
        out_mean = torch.empty(N, dtype=torch.float32, device=img1.device)
        want1, want2 = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        saved = None
        if train and (want1 or want2):
            nbytes = saved_bytes(tuple(img1.shape), want2)
            saved = torch.empty(nbytes // 4, dtype=torch.float32, device=img1.device)
        fwd(img1, img2, padding, out_mean, saved=saved, want_grad2=want2)
        ctx.padding, ctx.ndim, ctx.saved_fields = padding, ndim, saved
        ctx.save_for_backward(img1, img2)
        return out_mean

    @staticmethod
    def backward(ctx, g_mean):
        img1, img2 = ctx.saved_tensors
        bwd = ssim_bwd if ctx.ndim == 2 else ssim3d_bwd
        dL = g_mean.detach().to(torch.float32).contiguous()
        want2 = ctx.needs_input_grad[1]
        grad1 = torch.empty_like(img1)
        grad2 = torch.empty_like(img2) if want2 else None
        bwd(dL, img1, img2, ctx.padding, grad1, grad2, saved=ctx.saved_fields)
        return (grad1 if ctx.needs_input_grad[0] else None), grad2, None, None, None


def fused_ssim(img1: torch.Tensor, img2: torch.Tensor, padding: str = "same", train: bool = True,
               per_image: bool = False) -> torch.Tensor:
    """Mean SSIM of NCHW float32 CUDA images in [0, 1] (11x11 Gaussian window,
    sigma 1.5, C1 = 0.01^2, C2 = 0.03^2).  padding: "same" (zero) or "valid"."""
    m = _FusedSSIM.apply(img1, img2, _pad(padding), bool(train), 2)
    return m if per_image else m.mean()


def fused_ssim3d(img1: torch.Tensor, img2: torch.Tensor, padding: str = "same",
                 train: bool = True, per_image: bool = False) -> torch.Tensor:
    """Mean SSIM of NCDHW float32 CUDA volumes with an 11x11x11 window."""
    m = _FusedSSIM.apply(img1, img2, _pad(padding), bool(train), 3)
    return m if per_image else m.mean()
