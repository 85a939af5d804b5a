"""Seeded synthetic inputs for the SSIM loss.

This module is shared by the tests, the benchmark and the smoke check.  It
holds input synthesis only -- random images with the shapes, value ranges and
structure of the workloads the pages describe -- and none of the SSIM
arithmetic.  It imports neither the CUDA package nor the oracle.

Every array is drawn in float64 with numpy's PCG64 generator from a fixed seed
and then rounded to float32; the same float32 arrays feed the GPU and (widened
back to float64) the oracle.

Workloads (pages: TriSSIM README "Performance" for the 1080p fp32 valid
forward+backward step; fused-ssim README "Usage" for NCHW batches in [0, 1],
"3D data" for NCDHW volumes):

=================  =================  =======  ==========  ============
name               shape              padding  grads       dL per image
=================  =================  =======  ==========  ============
tiny64_valid       1x3x64x64          valid    img1, img2  -1
splat1080_valid    1x3x1080x1920      valid    img1        -1
splat1080_same     1x3x1080x1920      same     img1, img2  -1
batch512_valid     8x3x512x512        valid    img1        -1/8
volume128_valid    1x1x128x128x128    valid    img1        -1
volume256_valid    1x1x256x256x256    valid    img1        -1
=================  =================  =======  ==========  ============

volume256_valid is the 128^3 volume's generator at twice the extent: a volume
whose per-slice intermediate fields (the XY-blurred statistics and the Z
adjoint of the derivatives, 248 MB each) no longer fit in the GPU's L2.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "make_inputs",
    "splat_render",
    "trilinear_noise_volume",
    "uniform_pair",
    "noisy_copy",
]


@dataclass(frozen=True)
class Workload:
    name: str
    shape: tuple  # (N, C, H, W) or (N, C, D, H, W)
    padding: str  # "valid" or "same"
    want_grad2: bool
    dl_per_image: float  # dLoss/dmean[n] for loss = 1 - mean over the batch of mean[n]
    seed: int

    @property
    def ndim(self) -> int:
        return len(self.shape) - 2

    @property
    def megapixels(self) -> float:
        """Input pixels (or voxels) per call, channels not counted, in millions."""
        n = self.shape[0]
        for s in self.shape[2:]:
            n *= s
        return n / 1e6


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny64_valid", (1, 3, 64, 64), "valid", True, -1.0, 1001),
        Workload("splat1080_valid", (1, 3, 1080, 1920), "valid", False, -1.0, 1002),
        Workload("splat1080_same", (1, 3, 1080, 1920), "same", True, -1.0, 1003),
        Workload("batch512_valid", (8, 3, 512, 512), "valid", False, -1.0 / 8.0, 1004),
        Workload("volume128_valid", (1, 1, 128, 128, 128), "valid", False, -1.0, 1005),
        Workload("volume256_valid", (1, 1, 256, 256, 256), "valid", False, -1.0, 1006),
    )
}


def noisy_copy(rng: np.random.Generator, img: np.ndarray, std: float, gain: float = 1.0,
               bias: float = 0.0) -> np.ndarray:
    """clamp(gain * img + bias + N(0, std^2), 0, 1), in float64."""
    return np.clip(gain * img + bias + rng.normal(0.0, std, size=img.shape), 0.0, 1.0)


def uniform_pair(shape, seed: int, std: float = 0.05):
    """img1 ~ U[0, 1]; img2 = clamp(img1 + N(0, std^2), 0, 1); both float32."""
    rng = np.random.default_rng(seed)
    a = rng.random(shape)
    b = noisy_copy(rng, a, std)
    return a.astype(np.float32), b.astype(np.float32)


def splat_render(rng: np.random.Generator, n: int, c: int, h: int, w: int,
                 blobs: int = 200, s_lo: float = 10.0, s_hi: float = 60.0) -> np.ndarray:
    """A smooth render: a sum of isotropic 2D Gaussian blobs, clamped to [0, 1].

    Blob k has its centre uniform over the image, a standard deviation
    s_k ~ U[s_lo, s_hi] pixels and a colour ~ U[0, 1]^c.  Each blob's footprint
    is the outer product of two 1D profiles, so an image is one small matrix
    product per channel.  Returns float64 of shape (n, c, h, w).
    """
    out = np.empty((n, c, h, w), dtype=np.float64)
    ii = np.arange(h, dtype=np.float64)
    jj = np.arange(w, dtype=np.float64)
    for b in range(n):
        cy = rng.uniform(0.0, h, size=blobs)
        cx = rng.uniform(0.0, w, size=blobs)
        s = rng.uniform(s_lo, s_hi, size=blobs)
        col = rng.random((blobs, c))
        gy = np.exp(-((ii[None, :] - cy[:, None]) ** 2) / (2.0 * s[:, None] ** 2))  # (K, h)
        gx = np.exp(-((jj[None, :] - cx[:, None]) ** 2) / (2.0 * s[:, None] ** 2))  # (K, w)
        for ch in range(c):
            out[b, ch] = (gy * col[:, ch : ch + 1]).T @ gx
    return np.clip(out, 0.0, 1.0)


def _linear_upsample_matrix(src: int, dst: int) -> np.ndarray:
    """(dst, src) matrix of linear interpolation with aligned corners:
    output i samples the source at u = i * (src - 1) / (dst - 1)."""
    m = np.zeros((dst, src), dtype=np.float64)
    for i in range(dst):
        u = i * (src - 1) / (dst - 1)
        i0 = min(int(np.floor(u)), src - 2)
        t = u - i0
        m[i, i0] += 1.0 - t
        m[i, i0 + 1] += t
    return m


def trilinear_noise_volume(rng: np.random.Generator, n: int, c: int, d: int, h: int, w: int,
                           coarse: int = 16) -> np.ndarray:
    """U[0, 1] noise on a coarse^3 grid, trilinearly upsampled (aligned corners)
    to d x h x w.  Returns float64 of shape (n, c, d, h, w)."""
    base = rng.random((n, c, coarse, coarse, coarse))
    mz = _linear_upsample_matrix(coarse, d)
    my = _linear_upsample_matrix(coarse, h)
    mx = _linear_upsample_matrix(coarse, w)
    return np.einsum("zk,yi,xj,nckij->nczyx", mz, my, mx, base, optimize=True)


def make_inputs(name: str):
    """(img1, img2) float32 arrays for the named workload."""
    wl = WORKLOADS[name]
    rng = np.random.default_rng(wl.seed)
    if name == "tiny64_valid":
        a = rng.random(wl.shape)
        b = noisy_copy(rng, a, 0.05)
    elif name in ("splat1080_valid", "splat1080_same"):
        a = splat_render(rng, *wl.shape)
        b = noisy_copy(rng, a, 0.02)
    elif name == "batch512_valid":
        a = rng.random(wl.shape)
        b = noisy_copy(rng, a, 0.1, gain=0.8, bias=0.1)
    elif name in ("volume128_valid", "volume256_valid"):
        a = trilinear_noise_volume(rng, *wl.shape)
        b = noisy_copy(rng, a, 0.03)
    else:  # pragma: no cover
        raise KeyError(name)
    return (np.ascontiguousarray(a, dtype=np.float32),
            np.ascontiguousarray(b, dtype=np.float32))


def dl_vector(name: str) -> np.ndarray:
    """dLoss/dmean[n] for every image of the named workload (float32)."""
    wl = WORKLOADS[name]
    return np.full((wl.shape[0],), wl.dl_per_image, dtype=np.float32)
