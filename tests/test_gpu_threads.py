"""Two host threads calling the library at once, each on its own stream with
its own workspace and outputs (the plan cache and per-device set-up are shared
and locked): every call gives the same bits as the same call made alone."""
import threading

import numpy as np
import pytest

from workloads import uniform_pair

pytestmark = pytest.mark.gpu


def test_concurrent_calls_on_two_streams():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiable_image_quality_gb300 as pkg

    dev = torch.device("cuda:0")
    jobs = [((2, 3, 200, 260), "valid", 11), ((1, 2, 150, 333), "same", 12),
            ((1, 1, 20, 21, 22), "valid", 13)]

    def run(shape, padding, seed, stream):
        x, y = uniform_pair(shape, seed, std=0.08)
        with torch.cuda.stream(stream):
            tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
            N = shape[0]
            three = len(shape) == 5
            ws = torch.zeros(pkg.workspace_bytes(shape, padding), dtype=torch.uint8, device=dev)
            mean = torch.empty(N, device=dev)
            saved = torch.empty(pkg.saved_bytes(shape, False) // 4, device=dev)
            fwd = pkg.ssim3d_fwd if three else pkg.ssim_fwd
            bwd = pkg.ssim3d_bwd if three else pkg.ssim_bwd
            fwd(tx, ty, padding, mean, saved=saved, workspace=ws)
            g1 = torch.empty_like(tx)
            dl = torch.full((N,), -1.0, device=dev)
            bwd(dl, tx, ty, padding, g1, saved=saved)
            stream.synchronize()
            return mean.cpu().numpy(), g1.cpu().numpy()

    alone = [run(*j, torch.cuda.Stream(dev)) for j in jobs]
    results = {}
    errors = []

    def worker(t):
        try:
            s = torch.cuda.Stream(dev)
            for it in range(6):
                j = jobs[(t + it) % len(jobs)]
                results[(t, it)] = ((t + it) % len(jobs), run(*j, s))
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert len(results) == 12
    for (t, it), (k, (m, g)) in results.items():
        assert np.array_equal(m, alone[k][0]), (t, it, "mean")
        assert np.array_equal(g, alone[k][1]), (t, it, "grad")


def test_fused_ssim_autograd_on_two_streams_at_once(oracle_mod):
    """The autograd API on two streams whose work overlaps on the GPU: each
    stream gets its own scratch buffer, so both losses and gradients match the
    oracle."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiable_image_quality_gb300 as pkg

    dev = torch.device("cuda:0")
    cases = [((2, 3, 300, 410), "valid", 21), ((1, 3, 257, 380), "same", 22)]
    streams = [torch.cuda.Stream(dev) for _ in cases]
    inputs, outs = [], []
    for (shape, padding, seed), s in zip(cases, streams):
        x, y = uniform_pair(shape, seed, std=0.08)
        with torch.cuda.stream(s):
            t1 = torch.from_numpy(x).to(dev).requires_grad_(True)
            t2 = torch.from_numpy(y).to(dev).requires_grad_(True)
        inputs.append((x, y, t1, t2))
    torch.cuda.synchronize()
    for (shape, padding, _), s, (_, _, t1, t2) in zip(cases, streams, inputs):
        with torch.cuda.stream(s):  # both forwards queued before either backward
            outs.append(1.0 - pkg.fused_ssim(t1, t2, padding))
    for loss, s in zip(outs, streams):
        with torch.cuda.stream(s):
            loss.backward()
    torch.cuda.synchronize()
    for (shape, padding, _), (x, y, t1, t2), loss in zip(cases, inputs, outs):
        N = shape[0]
        ref_mean = oracle_mod.ssim2d(x, y, padding)
        g1, g2 = oracle_mod.ssim2d_grad(x, y, np.full(N, -1.0 / N), padding)
        assert abs(float(loss.item()) - (1.0 - float(np.mean(ref_mean)))) <= 1e-5
        for got, ref in ((t1.grad, g1), (t2.grad, g2)):
            err = np.max(np.abs(got.cpu().numpy() - ref)) / np.max(np.abs(ref))
            assert err <= 1e-4, f"{shape} {padding}: gradient error {err:.2e}"
