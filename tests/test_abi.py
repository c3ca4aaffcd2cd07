"""The C ABI without a GPU: exports, host-side argument checks and plan arithmetic."""
import ctypes

import pytest

import muon_newton_schulz_09_b300 as mu
from muon_newton_schulz_09_b300 import MUON_BF16, MUON_ERR_INVALID, MUON_F32, MUON_OK, MuonMatrix


def test_library_exports_every_declared_function():
    lib = mu.load_library()
    names = mu.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_kernel_names():
    assert mu.status_string(MUON_OK) == "MUON_OK"
    assert mu.status_string(5) == "MUON_ERR_TIMEOUT"
    assert mu.status_string(99) == "MUON_ERR_UNKNOWN"
    assert [mu.kernel_name(k) for k in range(mu.KERNEL_KINDS)] == [
        "momentum_norm", "norm", "scale_orient", "gram_xxt", "gram_aa", "combine_ax_bx", "update", "copy_out",
        "newton_schulz"]


def test_default_config():
    cfg = mu.MuonConfig()
    mu.load_library().muon_default_config(ctypes.byref(cfg))
    assert (cfg.steps, cfg.a, cfg.b, cfg.c, cfg.scale_lr_by_shape, cfg.weight_decay, cfg.precise_carry,
            cfg.persistent) == (5, 1.5, -0.5, 0.0, 1, 0.0, 2, 2)
    assert abs(cfg.eps - 1e-7) < 1e-12


def test_null_handle_is_invalid():
    lib = mu.load_library()
    assert lib.muon_orthogonalize(None, None, None, 0, 5, 1.5, -0.5, 0.0, None) == MUON_ERR_INVALID
    assert lib.muon_step(None, None, None, None, 0, 0.02, 0.95, 1, None) == MUON_ERR_INVALID
    assert lib.muon_destroy(None) == MUON_OK
    assert lib.muon_last_error(None) == b"null handle"


def M(ptr, r, c, ld=None, dt=MUON_BF16):
    return MuonMatrix(ctypes.c_void_p(ptr), r, c, c if ld is None else ld, dt)


BASE = 1 << 32


def test_check_orthogonalize():
    ok = [M(BASE, 64, 128)]
    out = [M(BASE + (1 << 24), 64, 128, dt=MUON_F32)]
    assert mu.check_orthogonalize(ok, out, 5)[0] == MUON_OK
    assert mu.check_orthogonalize(ok, ok, 5)[0] == MUON_OK  # in place
    assert mu.check_orthogonalize([], [], 5)[0] == MUON_OK
    bad = [
        ([M(BASE, 64, 128)], [M(BASE + (1 << 24), 64, 127)], 5, "differ in shape"),
        ([M(BASE, 64, 128, ld=100)], out, 5, "ld"),
        ([M(0, 64, 128)], out, 5, "null pointer"),
        ([M(BASE, 64, 128, dt=7)], out, 5, "dtype"),
        (ok, out, -1, "steps"),
        ([M(BASE, -1, 128)], [M(BASE, -1, 128)], 5, "out of range"),
        ([M(BASE, 40000, 40000)], [M(BASE, 40000, 40000)], 5, "too large"),
        ([M(BASE, 8, 8), M(BASE, 8, 8, dt=MUON_F32)], [M(BASE + 4096, 8, 8), M(BASE + 8192, 8, 8)], 1, "dtype"),
        ([M(BASE, 8, 8), M(BASE, 8, 8)], [M(BASE + 4096, 8, 8), M(BASE + 4096 + 64, 8, 8)], 1, "overlap"),
    ]
    for ins, outs, steps, why in bad:
        st, msg = mu.check_orthogonalize(ins, outs, steps)
        assert st == MUON_ERR_INVALID and why in msg, (why, msg)


def test_zero_sized_matrices_accepted():
    assert mu.check_orthogonalize([M(0, 0, 16)], [M(0, 0, 16)], 5)[0] == MUON_OK
    assert mu.check_step([M(0, 16, 0)], [M(0, 16, 0)], [M(0, 16, 0, dt=MUON_F32)])[0] == MUON_OK


def test_check_step():
    p = [M(BASE, 32, 64)]
    g = [M(BASE + (1 << 20), 32, 64)]
    m = [M(BASE + (2 << 20), 32, 64, dt=MUON_F32)]
    assert mu.check_step(p, g, m)[0] == MUON_OK
    st, msg = mu.check_step(p, g, [M(BASE + (2 << 20), 32, 64)])
    assert st == MUON_ERR_INVALID and "F32" in msg
    st, msg = mu.check_step(p, [M(BASE + 64, 32, 64)], m)
    assert st == MUON_ERR_INVALID and "overlap" in msg
    st, msg = mu.check_step(p, [M(BASE + (1 << 20), 32, 65)], m)
    assert st == MUON_ERR_INVALID and "shape" in msg


def test_plan_stats_gpt2_124m():
    shapes = [(768, 768)] * 4 + [(768, 3072), (3072, 768)]
    s = mu.plan_stats(shapes * 12)
    assert s["groups"] == 2
    # 768 = 6 row tiles of 128 and 3 column tiles of 256: 2 + 4 + 6 = 12 Gram tiles reach the upper triangle
    assert s["gram_tiles"] == 72 * 12
    # combine: 6 row tiles x (3 or 12) column tiles of 256
    assert s["combine_tiles"] == 48 * 6 * 3 + 24 * 6 * 12
    n = 768
    want = 48 * (n * (n + 1) * n + 2 * n * n * n) + 24 * (n * (n + 1) * 3072 + 2 * n * n * 3072)
    assert s["flops_per_iter"] == pytest.approx(want, rel=1e-12)
    assert 5 * s["flops_per_iter"] == pytest.approx(9.789e11, rel=1e-3)


def test_plan_stats_ragged_and_c():
    s = mu.plan_stats([(130, 70), (70, 130), (0, 5)], with_c=True)
    assert s["groups"] == 1
    assert s["gram_tiles"] == 2 * 2 * 1  # one tile per matrix, doubled for the A A pass
    # 1024 = 8 row tiles, 4 column tiles: 2 + 4 + 6 + 8; 4096: 32 row tiles, 16 column tiles
    assert mu.plan_stats([(1024, 1024)])["gram_tiles"] == 20
    assert mu.plan_stats([(4096, 16384)])["gram_tiles"] == sum(min(2 * j + 2, 32) for j in range(16))
    assert s["combine_tiles"] == 2
    n, m = 70, 130
    assert s["flops_per_iter"] == pytest.approx(2 * (n * (n + 1) * m + 2 * n * n * m + n * n * (n + 1)))


def test_selftest_wait_rejects_bad_limits_without_a_handle():
    lib = mu.load_library()
    assert lib.muon_selftest_wait(None, 50_000_000, None) == MUON_ERR_INVALID
    assert lib.muon_selftest_persistent(None, 50_000_000, None) == MUON_ERR_INVALID


def test_profiling_calls_reject_a_null_handle():
    lib = mu.load_library()
    mhz = ctypes.c_double(-1.0)
    assert lib.muon_profile_clock(None, ctypes.byref(mhz)) == MUON_ERR_INVALID
    assert lib.muon_profile_enable(None, 1) == MUON_ERR_INVALID
    assert lib.muon_profile_read(None, None, None) == MUON_ERR_INVALID


def test_create_rejects_a_bad_config_before_touching_a_gpu():
    lib = mu.load_library()
    h = ctypes.c_void_p()
    for field, value in [("precise_carry", 3), ("precise_carry", -1), ("steps", -1), ("weight_decay", -0.5), ("eps", float("nan")),
                         ("persistent", 3)]:
        cfg = mu.MuonConfig()
        lib.muon_default_config(ctypes.byref(cfg))
        setattr(cfg, field, value)
        assert lib.muon_create(ctypes.byref(h), 0, ctypes.byref(cfg)) == MUON_ERR_INVALID, field


def test_workspace_limit_calls_reject_a_null_handle():
    lib = mu.load_library()
    v = ctypes.c_int64(-1)
    assert lib.muon_set_workspace_limit(None, 1 << 20) == MUON_ERR_INVALID
    assert lib.muon_workspace_bytes(None, ctypes.byref(v)) == MUON_ERR_INVALID
