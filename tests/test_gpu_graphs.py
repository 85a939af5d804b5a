"""The C ABI under CUDA graph capture.

A training loop that launches the same loss every step can capture it once
and replay the graph, so the host issues one launch per step instead of the
library's two or three.  Every call here works on a stream being captured:
argument checks and tensor-map encoding run on the host while the call is
recorded, the kernels' parameters (tensor maps included) are fixed at capture,
and each launch leaves the workspace's completion counter at zero, so the
graph can be replayed any number of times.  The test captures the stored
training step (forward with saved gradient fields, then the scaling backward)
on static buffers, copies new images into them before each replay, and checks
every replay against the oracle at the parity bars.
"""
import numpy as np
import pytest

from workloads import uniform_pair

pytestmark = pytest.mark.gpu

MEAN_TOL = 1e-5
GRAD_RTOL = 1e-4


@pytest.fixture(scope="module")
def pkg():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiable_image_quality_gb300 as pkg
    from differentiable_image_quality_gb300 import _build

    _build.build()
    return pkg


def _capture(torch, step):
    """Warm `step` up on a side stream, then capture it into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    return graph


@pytest.mark.parametrize("shape,padding", [((2, 3, 60, 140), "valid"), ((1, 2, 47, 131), "same"),
                                           ((2, 1, 16, 18, 20), "valid")])
def test_training_step_replayed_from_a_graph(pkg, oracle_mod, shape, padding):
    import torch

    dev = torch.device("cuda:0")
    lib = pkg._abi.load()
    is3d = len(shape) == 5
    N = shape[0]
    x0 = torch.zeros(shape, device=dev)
    y0 = torch.zeros(shape, device=dev)
    mean = torch.empty(N, device=dev)
    want2 = padding == "same"
    saved = torch.empty(pkg.saved_bytes(shape, want2) // 4, device=dev)
    pad = 0 if padding == "valid" else 1
    ws_bytes = (lib.gbssim3d_workspace_bytes(*shape, pad) if is3d
                else lib.gbssim_workspace_bytes(*shape, pad))
    ws = torch.zeros(int(ws_bytes), dtype=torch.uint8, device=dev)
    dL = torch.linspace(-1.0, -0.5, N, device=dev)
    g1 = torch.empty_like(x0)
    g2 = torch.empty_like(y0) if want2 else None
    fwd = pkg.ssim3d_fwd if is3d else pkg.ssim_fwd
    bwd = pkg.ssim3d_bwd if is3d else pkg.ssim_bwd

    def step():
        fwd(x0, y0, padding, mean, saved=saved, want_grad2=want2, workspace=ws)
        bwd(dL, x0, y0, padding, g1, g2, saved=saved)

    x, y = uniform_pair(shape, 2300, std=0.1)
    x0.copy_(torch.from_numpy(x))
    y0.copy_(torch.from_numpy(y))
    graph = _capture(torch, step)
    dl = dL.cpu().numpy().astype(np.float64)
    for seed in (2301, 2302, 2303):
        x, y = uniform_pair(shape, seed, std=0.1 if seed % 2 else 0.03)
        x0.copy_(torch.from_numpy(x))
        y0.copy_(torch.from_numpy(y))
        graph.replay()
        torch.cuda.synchronize()
        if is3d:
            ref_mean = oracle_mod.ssim3d(x, y, padding)
            r1, r2 = oracle_mod.ssim3d_grad(x, y, dl, padding, want2)
        else:
            ref_mean = oracle_mod.ssim2d(x, y, padding)
            r1, r2 = oracle_mod.ssim2d_grad(x, y, dl, padding, want2)
        assert np.max(np.abs(mean.cpu().numpy() - ref_mean)) <= MEAN_TOL, seed
        for got, ref in ((g1, r1), (g2, r2)) if want2 else ((g1, r1),):
            err = np.max(np.abs(got.cpu().numpy().astype(np.float64) - ref)) / np.max(np.abs(ref))
            assert err <= GRAD_RTOL, f"{seed}: gradient relative error {err:.3e}"


def test_per_octave_stage_replayed_from_a_graph(pkg, oracle_mod):
    import torch

    dev = torch.device("cuda:0")
    lib = pkg._abi.load()
    shape, octaves = (1, 3, 200, 300), 4
    N, C, H, W = shape
    x0 = torch.zeros(shape, device=dev)
    y0 = torch.zeros(shape, device=dev)
    nbytes = int(lib.gbssim_pyramid_workspace_bytes(N, C, H, W, 0, octaves))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    means = torch.empty(octaves * 3 * N, device=dev)
    stream = lambda: torch.cuda.current_stream(dev).cuda_stream  # noqa: E731

    def step():
        st = lib.ssim_pyramid(x0.data_ptr(), y0.data_ptr(), N, C, H, W, 0, octaves,
                              means.data_ptr(), None, ws.data_ptr(), nbytes, stream())
        assert st == 0, lib.gbssim_strerror(st)

    x, y = uniform_pair(shape, 2400, std=0.1)
    x0.copy_(torch.from_numpy(x))
    y0.copy_(torch.from_numpy(y))
    graph = _capture(torch, step)
    for seed in (2401, 2402):
        x, y = uniform_pair(shape, seed, std=0.05)
        x0.copy_(torch.from_numpy(x))
        y0.copy_(torch.from_numpy(y))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.ssim2d_pyramid(x, y, "valid", octaves)
        got = means.cpu().numpy().reshape(ref.shape)
        assert np.max(np.abs(got - ref)) <= MEAN_TOL, seed
