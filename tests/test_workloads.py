"""The seeded input generators (CPU only)."""
import numpy as np
import torch

import workloads as wl


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * s for s in (1e-3, 1.0, 1e3)])
    x = np.concatenate([x, np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = wl.bf16_round(x)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    np.testing.assert_array_equal(wl.from_bf16_bits(wl.bf16_bits(got)), got)


def test_normal_deterministic_and_thread_independent(monkeypatch):
    a = wl.normal((9, 1, 2), (3000, 3000), 0.5)
    monkeypatch.setattr(wl, "_THREADS", 1)
    b = wl.normal((9, 1, 2), (3000, 3000), 0.5)
    np.testing.assert_array_equal(a, b)
    assert a.dtype == np.float32 and a.shape == (3000, 3000)
    assert abs(float(a.std()) - 0.5) < 2e-3 and abs(float(a.mean())) < 2e-3
    c = wl.normal((9, 1, 3), (3000, 3000), 0.5)
    assert not np.array_equal(a, c)


def test_orthonormal_columns_and_spectrum():
    v = wl.random_orthonormal_columns((1, 2, 3), 256, 64)
    np.testing.assert_allclose(v.T @ v, np.eye(64), atol=1e-12)
    s = wl.log_uniform_spectrum((1, 2, 4), 1000)
    assert s.min() >= 1e-4 and s.max() <= 1.0
    g = wl.illconditioned(7, 64, 256)
    sv = np.linalg.svd(g.astype(np.float64), compute_uv=False)
    want = np.sort(wl.log_uniform_spectrum((7, 0, 12), 64))[::-1]
    np.testing.assert_allclose(sv, want, rtol=1e-5, atol=1e-6)


def test_spike_dominates_gradient():
    w = wl.small_workload("t", [(384, 96)], kind="step", grad_std=1e-3, spike_rank=4, spike_gain=50.0, seed=11)
    g = wl.gradient(w, 0).astype(np.float64)
    assert np.array_equal(g.astype(np.float32), wl.bf16_round(g.astype(np.float32)))
    s = np.linalg.svd(g, compute_uv=False)
    # four spike directions carry most of the energy
    assert (s[:4] ** 2).sum() / (s ** 2).sum() > 0.9
    assert 40 < g.std() / 1e-3 < 60


def test_workload_table():
    assert wl.GPT2_124M.count == 72 and wl.GPT2_124M.elements() == 84934656
    assert wl.GPT2_350M.count == 144 and wl.GPT2_350M.elements() == 301989888
    assert wl.SQUARE_64x1024.count == 64
    assert wl.ILLCOND_4096x16384.steps == 10
    m = wl.momentum_buffer(wl.SINGLE_128x256, 0)
    assert m.shape == (128, 256) and not m.any()
    p = wl.parameter(wl.SINGLE_128x256, 0)
    assert p.dtype == np.float32 and abs(float(p.std()) - 0.02) < 2e-3
