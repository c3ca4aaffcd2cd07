"""CUDA path vs the fp64 oracle on small and ragged cases (GPU).

Every comparison runs the library through its C ABI (via the ctypes binding)
and the oracle in fp64 on the same bf16- or fp32-valued inputs drawn from
``workloads.py``. The bar is the relative Frobenius error per matrix, TOL.
Sizes span several 128-wide tiles and ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import TOL, bf16_ulp, dev, host, rel_f

pytestmark = pytest.mark.gpu

CUBIC = (1.5, -0.5, 0.0)
QUINTIC = (15 / 8, -10 / 8, 3 / 8)

RAGGED = [(128, 256), (256, 128), (130, 70), (70, 130), (1, 5), (5, 1), (2, 2), (64, 200), (200, 64),
          (129, 257), (257, 129), (384, 96), (300, 300), (513, 1000)]


@pytest.fixture(scope="module")
def muon():
    from muon_newton_schulz_09_b300 import Muon
    with Muon(0) as m:
        yield m


def inputs_for(shapes, dtype="bf16", seed=101, std=1.0):
    w = wl.small_workload("t", shapes, dtype=dtype, grad_std=std, seed=seed)
    return w, [wl.gradient(w, j) for j in range(w.count)]


def run_orth(muon, xs, in_dtype, out_dtype, steps, coeffs):
    ins = [dev(x, in_dtype) for x in xs]
    outs = [torch.empty(x.shape, dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16, device="cuda")
            for x in xs]
    muon.orthogonalize(ins, outs, steps=steps, coeffs=coeffs)
    torch.cuda.synchronize()
    assert muon.get_error() == 0
    return [host(o) for o in outs]


@pytest.mark.parametrize("in_dtype", ["bf16", "f32"])
def test_steps0_is_frobenius_normalisation(muon, in_dtype):
    _, xs = inputs_for(RAGGED, in_dtype, seed=7)
    got = run_orth(muon, xs, in_dtype, "f32", 0, CUBIC)
    for x, o in zip(xs, got):
        want = oracle.frobenius_normalize(x)
        # X0 is rounded to bf16 once (and u once more for bf16 inputs): 2^-8 relative per element at most.
        assert rel_f(o, want) < 4e-3, x.shape


@pytest.mark.parametrize("coeffs,steps", [(CUBIC, 1), (CUBIC, 5), (QUINTIC, 3)], ids=["cubic1", "cubic5", "quintic3"])
def test_orthogonalize_ragged_batch(muon, coeffs, steps):
    _, xs = inputs_for(RAGGED, "bf16", seed=11)
    got = run_orth(muon, xs, "bf16", "f32", steps, coeffs)
    for x, o in zip(xs, got):
        want = oracle.orthogonalize(x, steps, coeffs)
        assert rel_f(o, want) < TOL, (x.shape, rel_f(o, want))


def test_orthogonalize_bf16_out_and_f32_in(muon):
    _, xs = inputs_for([(256, 640), (640, 256), (100, 100)], "f32", seed=12)
    got = run_orth(muon, xs, "f32", "bf16", 5, CUBIC)
    for x, o in zip(xs, got):
        assert rel_f(o, oracle.orthogonalize(x, 5, CUBIC)) < TOL


def test_in_place_and_strided(muon):
    _, xs = inputs_for([(200, 136), (136, 200)], "bf16", seed=13)
    wants = [oracle.orthogonalize(x, 5, CUBIC) for x in xs]
    # in place on padded (ld > cols) views
    bufs = [torch.zeros(x.shape[0], x.shape[1] + 24, dtype=torch.bfloat16, device="cuda") for x in xs]
    views = [b[:, :x.shape[1]] for b, x in zip(bufs, xs)]
    for v, x in zip(views, xs):
        v.copy_(dev(x))
    muon.orthogonalize(views, views, steps=5, coeffs=CUBIC)
    torch.cuda.synchronize()
    for b, v, w in zip(bufs, views, wants):
        assert rel_f(host(v), w) < TOL
        assert torch.count_nonzero(b[:, v.shape[1]:]) == 0  # padding untouched


def test_zero_matrix_and_empty(muon):
    z = torch.zeros(96, 160, dtype=torch.bfloat16, device="cuda")
    out = torch.full((96, 160), 7.0, device="cuda")
    empty_in = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    empty_out = torch.zeros(0, 64, device="cuda")
    muon.orthogonalize([z, empty_in], [out, empty_out], steps=5)
    muon.orthogonalize([], [], steps=5)
    torch.cuda.synchronize()
    assert muon.get_error() == 0
    assert torch.all(out == 0)


def test_transpose_equivariance(muon):
    _, xs = inputs_for([(192, 448)], "bf16", seed=14)
    x = xs[0]
    a = run_orth(muon, [x, np.ascontiguousarray(x.T)], "bf16", "f32", 5, CUBIC)
    assert rel_f(a[1].T, a[0]) < 1e-2


def test_deterministic(muon):
    _, xs = inputs_for([(300, 700), (700, 300), (1024, 1024)], "bf16", seed=15)
    ins = [dev(x) for x in xs]
    o1 = [torch.empty(x.shape, device="cuda") for x in xs]
    o2 = [torch.empty(x.shape, device="cuda") for x in xs]
    muon.orthogonalize(ins, o1, steps=5)
    muon.orthogonalize(ins, o2, steps=5)
    torch.cuda.synchronize()
    for a, b in zip(o1, o2):
        assert torch.equal(a, b)


# ----------------------------------------------------------------------------- muon_step

def step_case(shapes, grad_dtype, param_dtype, seed, nesterov=True, beta=0.95, zero_momentum=False):
    w = wl.small_workload("s", shapes, kind="step", dtype=grad_dtype, param_dtype=param_dtype, grad_std=1e-3,
                          spike_rank=2, spike_gain=20.0, seed=seed, nesterov=nesterov, beta=beta,
                          zero_momentum=zero_momentum)
    g = [wl.gradient(w, j) for j in range(w.count)]
    m = [wl.momentum_buffer(w, j) for j in range(w.count)]
    p = [wl.parameter(w, j) for j in range(w.count)]
    return w, g, m, p


@pytest.mark.parametrize("nesterov,beta", [(True, 0.95), (False, 0.9), (True, 0.0)])
def test_step_orthogonal_update_f32_params(muon, nesterov, beta):
    """f32 params at zero: W' = -lr*s*O exactly enough to read O back, and the momentum in fp32."""
    shapes = [(256, 768), (768, 256), (130, 70), (384, 384)]
    w, g, m, _ = step_case(shapes, "bf16", "f32", seed=21, nesterov=nesterov, beta=beta)
    lr = 0.02
    P = [torch.zeros(s, device="cuda") for s in shapes]
    G = [dev(x, "bf16") for x in g]
    M = [dev(x, "f32") for x in m]
    muon.step(P, G, M, lr=lr, beta=beta, nesterov=nesterov)
    torch.cuda.synchronize()
    assert muon.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        w_new, buf_new, o = oracle.muon_step(np.zeros((r, c)), g[j], m[j], lr, beta, nesterov, 5, CUBIC)
        s = oracle.lr_scale(r, c)
        assert rel_f(host(M[j]), buf_new) < 1e-6
        assert rel_f(-host(P[j]) / (lr * s), o) < TOL, (r, c)


def test_step_bf16_params(muon):
    """bf16 params: W' is within one bf16 ulp of the oracle's W', plus 5% of the largest update element."""
    shapes = [(512, 1536), (1536, 512), (96, 96)]
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=22)
    lr = 0.02
    P = [dev(x, "bf16") for x in p]
    G = [dev(x, "bf16") for x in g]
    M = [dev(x, "f32") for x in m]
    muon.step(P, G, M, lr=lr, beta=0.95, nesterov=True)
    torch.cuda.synchronize()
    for j, (r, c) in enumerate(shapes):
        w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (r, c, float(err.max()))


@pytest.mark.parametrize("pad", [0, 3], ids=["direct", "fallback"])
def test_step_bf16_params_ragged(muon, pad):
    """Ragged and transposed bf16 params. pad = 0: the last combine writes W directly (16-byte rows);
    pad = 3: ld is not a multiple of 8, so the separate update kernel runs. Both must agree with
    the oracle to one bf16 ulp plus 5% of the largest update element."""
    shapes = [(130, 70), (70, 130), (1, 5), (5, 1), (200, 64), (257, 129)]
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=23)
    lr = 0.02
    bufs = [torch.zeros(r, c + pad, dtype=torch.bfloat16, device="cuda") for r, c in shapes]
    P = [b[:, :c] for b, (r, c) in zip(bufs, shapes)]
    for t, x in zip(P, p):
        t.copy_(dev(x, "bf16"))
    G = [dev(x, "bf16") for x in g]
    M = [dev(x, "f32") for x in m]
    muon.step(P, G, M, lr=lr, beta=0.95, nesterov=True)
    torch.cuda.synchronize()
    assert muon.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (r, c, float(err.max()))
        if pad:
            assert torch.count_nonzero(bufs[j][:, c:]) == 0  # padding untouched


@pytest.mark.parametrize("scale", [1e-13, 1e12], ids=["tiny", "huge"])
def test_step_extreme_gradient_scale(muon, scale):
    """Gradient norms outside [1e-10, 1e10]: u is scaled in place before the first products instead of
    through them, and O is the same as for a gradient of ordinary size (Newton-Schulz is scale invariant)."""
    shapes = [(256, 512), (512, 256), (130, 70)]
    w, g, _, _ = step_case(shapes, "bf16", "f32", seed=24)
    gs = [wl.bf16_round((x.astype(np.float64) * scale).astype(np.float32)) for x in g]
    lr = 0.02
    P = [torch.zeros(sh, device="cuda") for sh in shapes]
    M = [torch.zeros(sh, device="cuda") for sh in shapes]
    muon.step(P, [dev(x, "bf16") for x in gs], M, lr=lr, beta=0.95, nesterov=True)
    torch.cuda.synchronize()
    assert muon.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        _, _, o = oracle.muon_step(np.zeros((r, c)), gs[j], np.zeros((r, c)), lr, 0.95, True, 5, CUBIC)
        got = -host(P[j]) / (lr * oracle.lr_scale(r, c))
        assert np.isfinite(got).all()
        assert rel_f(got, o) < TOL, (r, c, rel_f(got, o))


def test_step_zero_iterations_is_normalised_momentum():
    """steps = 0: O is X0 = u / (||u||_F + eps) itself, in the caller's orientation."""
    from muon_newton_schulz_09_b300 import Muon
    shapes = [(192, 320), (320, 192)]
    w, g, m, _ = step_case(shapes, "bf16", "f32", seed=25)
    P = [torch.zeros(sh, device="cuda") for sh in shapes]
    with Muon(0, steps=0) as m0:
        m0.step(P, [dev(x, "bf16") for x in g], [dev(x, "f32") for x in m], lr=1.0, beta=0.9, nesterov=False)
        torch.cuda.synchronize()
        assert m0.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        _, u = oracle.momentum(g[j], m[j], 0.9, False)
        want = oracle.frobenius_normalize(u)
        assert rel_f(-host(P[j]) / oracle.lr_scale(r, c), want) < 4e-3


@pytest.mark.parametrize("param_dtype", ["bf16", "f32"], ids=["fused", "kernel"])
def test_step_weight_decay(param_dtype):
    """Decoupled weight decay wd = 1.0: W' = W (1 - lr wd) - lr s O. bf16 params take the update fused
    into the last combine, fp32 params the separate update kernel."""
    from muon_newton_schulz_09_b300 import Muon
    shapes = [(256, 640), (640, 256), (130, 70)]
    w, g, m, p = step_case(shapes, "bf16", param_dtype, seed=26)
    lr, wd = 0.02, 1.0
    P = [dev(x, param_dtype) for x in p]
    with Muon(0, weight_decay=wd) as mw:
        mw.step(P, [dev(x, "bf16") for x in g], [dev(x, "f32") for x in m], lr=lr, beta=0.95, nesterov=True)
        torch.cuda.synchronize()
        assert mw.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC, weight_decay=wd)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        ulp = bf16_ulp(w_new) if param_dtype == "bf16" else np.abs(w_new) * 2.0 ** -22
        assert np.all(err <= ulp + 0.05 * upd), (r, c, float(err.max()))


def test_step_f32_grads_config1(muon):
    """One fp32 128x256 gradient N(0,1), zero momentum, beta 0.95, 5 cubic iterations."""
    w = wl.SINGLE_128x256
    g = wl.gradient(w, 0)
    m = wl.momentum_buffer(w, 0)
    P = [torch.zeros(128, 256, device="cuda")]
    muon.step(P, [dev(g, "f32")], [dev(m, "f32")], lr=1.0, beta=w.beta, nesterov=w.nesterov)
    torch.cuda.synchronize()
    _, _, o = oracle.muon_step(np.zeros((128, 256)), g, m, 1.0, w.beta, w.nesterov, 5, CUBIC)
    got = -host(P[0])
    assert rel_f(got, o) < TOL
    # distance to the SVD polar factor is a reported number (about 0.5 after 5 steps), not a pass/fail bound
    u, _, vt = np.linalg.svd(g.astype(np.float64), full_matrices=False)
    assert abs(rel_f(got, u @ vt) - rel_f(o, u @ vt)) < 0.02


def test_bounded_wait_expiry_is_reported_and_recoverable(muon):
    """A device wait that nothing satisfies gives up after its limit and raises MUON_ERR_TIMEOUT, and the
    context keeps working (failure detection without a fault or a hang)."""
    from muon_newton_schulz_09_b300 import MUON_ERR_TIMEOUT, MUON_OK
    assert muon.get_error() == MUON_OK
    muon.selftest_wait(50_000_000)
    assert muon.get_error() == MUON_ERR_TIMEOUT
    assert muon.get_error() == MUON_OK  # reading clears the flag
    _, xs = inputs_for([(256, 384)], "bf16", seed=16)
    got = run_orth(muon, xs, "bf16", "f32", 5, CUBIC)
    assert rel_f(got[0], oracle.orthogonalize(xs[0], 5, CUBIC)) < TOL


def test_persistent_stage_wait_expiry_is_reported_and_recoverable(muon):
    """The persistent launch with a planted work item whose stage count is never reached: every wait
    gives up after 50 ms, the launch ends with MUON_ERR_TIMEOUT instead of hanging or faulting, the
    stage counters are reset, and the same plan then computes the right result."""
    import time
    from muon_newton_schulz_09_b300 import MUON_ERR_TIMEOUT, MUON_OK
    assert muon.get_error() == MUON_OK
    t0 = time.perf_counter()
    muon.selftest_persistent(50_000_000)
    elapsed = time.perf_counter() - t0
    assert muon.get_error() == MUON_ERR_TIMEOUT
    assert elapsed < 5.0, elapsed
    _, xs = inputs_for([(256, 256)], "bf16", seed=48)
    got = run_orth(muon, xs, "bf16", "f32", 5, CUBIC)  # the self-test's plan, counters reset
    assert muon.get_error() == MUON_OK
    assert rel_f(got[0], oracle.orthogonalize(xs[0], 5, CUBIC)) < TOL


def test_profiling_counts_launches_and_reads_the_sm_clock(muon):
    """Profiling brackets each kernel with events and has the GEMM kernels report their own SM clock."""
    _, xs = inputs_for([(256, 384), (384, 256)], "bf16", seed=17)
    muon.profile_read()  # drop anything recorded before
    muon.profile(True)
    got = run_orth(muon, xs, "bf16", "f32", 3, CUBIC)
    muon.profile(False)
    prof = muon.profile_read()
    mhz = muon.profile_clock()
    # every iteration runs in one persistent launch
    assert prof["newton_schulz"][1] == 1 and prof["gram_xxt"][1] == 0 and prof["combine_ax_bx"][1] == 0
    assert prof["norm"][1] == 1 and all(ms > 0 for ms, n in prof.values() if n)
    assert 300.0 < mhz < 3000.0, mhz
    for g, x in zip(got, xs):
        assert rel_f(g, oracle.orthogonalize(x, 3, CUBIC)) < TOL


# ---------------------------------------------------------------- precise carry (X as bf16 hi + lo)

@pytest.fixture(scope="module")
def muon_carry():
    from muon_newton_schulz_09_b300 import Muon
    with Muon(0, precise_carry=True) as m:
        yield m


def spiked_inputs(shapes, seed):
    """N(0, 1e-3) plus a rank-4 spike 50x as strong: the bulk singular values sit far below the spike's."""
    w = wl.small_workload("spk", shapes, dtype="bf16", grad_std=1e-3, spike_rank=4, spike_gain=50.0, seed=seed)
    return [wl.gradient(w, j) for j in range(w.count)]


@pytest.fixture(scope="module")
def muon_rounded():
    from muon_newton_schulz_09_b300 import Muon
    with Muon(0, precise_carry=False) as m:
        yield m


@pytest.mark.parametrize("coeffs,steps,out_dtype", [(CUBIC, 5, "f32"), (QUINTIC, 5, "f32"), (QUINTIC, 3, "bf16")],
                         ids=["cubic5_f32", "quintic5_f32", "quintic3_bf16"])
def test_precise_carry_orthogonalize(muon, muon_carry, muon_rounded, coeffs, steps, out_dtype):
    """With the carry every ragged, transposed and square matrix is within the bar, and for fp32
    outputs at least four times closer to the oracle than with X rounded to bf16 every iteration.
    The default config carries exactly when c != 0: it gives the carried result for the quintic and
    the rounded one for the cubic, bit for bit."""
    shapes = [(128, 256), (256, 128), (130, 70), (70, 130), (384, 96), (300, 300), (513, 1000)]
    xs = spiked_inputs(shapes, seed=41)
    got_c = run_orth(muon_carry, xs, "bf16", out_dtype, steps, coeffs)
    got = run_orth(muon_rounded, xs, "bf16", out_dtype, steps, coeffs)
    got_d = run_orth(muon, xs, "bf16", out_dtype, steps, coeffs)
    for x, gc, g, gd in zip(xs, got_c, got, got_d):
        want = oracle.orthogonalize(x, steps, coeffs)
        ec, e = rel_f(gc, want), rel_f(g, want)
        assert ec < TOL, (x.shape, ec)
        if out_dtype == "f32":
            assert ec < 0.25 * e, (x.shape, ec, e)
        assert np.array_equal(gd, gc if coeffs[2] != 0 else g), x.shape


def test_precise_carry_zero_iterations_keeps_x0():
    """steps = 0 with fp32 output: O = X0 = g/(||g||+eps) through hi + lo, far inside one bf16 rounding."""
    from muon_newton_schulz_09_b300 import Muon
    shapes = [(130, 70), (70, 130), (256, 256)]
    _, xs = inputs_for(shapes, "f32", seed=42)
    with Muon(0, precise_carry=True) as mc:
        got = run_orth(mc, xs, "f32", "f32", 0, CUBIC)
    for x, o in zip(xs, got):
        assert rel_f(o, oracle.frobenius_normalize(x)) < 2e-5


@pytest.mark.parametrize("param_dtype", ["f32", "bf16"], ids=["kernel_update", "fused_update"])
def test_precise_carry_step(muon_carry, param_dtype):
    """muon_step with the carry on spiked gradients: the fused last combine (bf16 params) and the update
    kernel (fp32 params) both use X_k = hi + lo; O read back from fp32 params at zero is within 5e-3."""
    shapes = [(256, 768), (768, 256), (130, 70), (384, 384)]
    g = spiked_inputs(shapes, seed=43)
    w, _, m, p = step_case(shapes, "bf16", param_dtype, seed=43)
    lr = 0.02
    if param_dtype == "f32":
        P = [torch.zeros(s, device="cuda") for s in shapes]
        p = [np.zeros(s) for s in shapes]
    else:
        P = [dev(x, "bf16") for x in p]
    M = [dev(x, "f32") for x in m]
    muon_carry.step(P, [dev(x, "bf16") for x in g], M, lr=lr, beta=0.95, nesterov=True)
    torch.cuda.synchronize()
    assert muon_carry.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        w_new, buf_new, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
        assert rel_f(host(M[j]), buf_new) < 1e-6
        if param_dtype == "f32":
            assert rel_f(-host(P[j]) / (lr * oracle.lr_scale(r, c)), o) < 5e-3, (r, c)
        else:
            upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
            err = np.abs(host(P[j]) - w_new)
            assert np.all(err <= bf16_ulp(w_new) + 0.02 * upd), (r, c, float(err.max()))


def test_precise_carry_extreme_scale(muon_carry):
    """A norm outside the fold range: the momentum kernel rescales hi + lo in place."""
    shapes = [(256, 512), (512, 256)]
    g = [wl.bf16_round((x.astype(np.float64) * 1e12).astype(np.float32)) for x in spiked_inputs(shapes, seed=44)]
    lr = 0.02
    P = [torch.zeros(sh, device="cuda") for sh in shapes]
    M = [torch.zeros(sh, device="cuda") for sh in shapes]
    muon_carry.step(P, [dev(x, "bf16") for x in g], M, lr=lr, beta=0.95, nesterov=True)
    torch.cuda.synchronize()
    assert muon_carry.get_error() == 0
    for j, (r, c) in enumerate(shapes):
        _, _, o = oracle.muon_step(np.zeros((r, c)), g[j], np.zeros((r, c)), lr, 0.95, True, 5, CUBIC)
        assert rel_f(-host(P[j]) / (lr * oracle.lr_scale(r, c)), o) < 5e-3, (r, c)


def test_step_more_matrices_than_one_launch_table(muon):
    """200 bf16 matrices: the elementwise kernels split at 128 matrices per launch, and with more than
    160 matrices in one GEMM batch the update leaves the last combine for the separate update kernel."""
    shapes = [(64, 96)] * 120 + [(96, 64)] * 60 + [(130, 70)] * 20
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=45)
    lr = 0.02
    P = [dev(x, "bf16") for x in p]
    M = [dev(x, "f32") for x in m]
    muon.step(P, [dev(x, "bf16") for x in g], M, lr=lr, beta=0.95, nesterov=True)
    torch.cuda.synchronize()
    assert muon.get_error() == 0
    for j in (0, 119, 120, 150, 179, 180, 199):
        r, c = shapes[j]
        w_new, buf_new, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
        assert rel_f(host(M[j]), buf_new) < 1e-6
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (j, float(err.max()))


def test_many_iterations_reach_the_polar_factor(muon):
    """25 cubic iterations on well-conditioned inputs: the GPU result is within the bar of the fp64 iterate,
    and both are within 2e-2 of the SVD polar factor U V^T."""
    shapes = [(128, 384), (384, 128), (256, 256)]
    _, xs = inputs_for(shapes, "f32", seed=46)
    # a well-conditioned spectrum: sigma in [0.5, 1] (the iteration needs about log(1/sigma_min) steps)
    ys = []
    for x in xs:
        u, s, vt = np.linalg.svd(x.astype(np.float64), full_matrices=False)
        s = np.linspace(0.5, 1.0, s.size)[::-1]
        ys.append(((u * s) @ vt).astype(np.float32))
    got = run_orth(muon, ys, "f32", "f32", 25, CUBIC)
    for y, gk in zip(ys, got):
        want = oracle.orthogonalize(y, 25, CUBIC)
        u, _, vt = np.linalg.svd(y.astype(np.float64), full_matrices=False)
        assert rel_f(gk, want) < TOL
        assert rel_f(gk, u @ vt) < 2e-2


def test_step_without_shape_scaled_lr():
    """scale_lr_by_shape = 0: every matrix takes the plain lr, tall ones included (fused update for the
    bf16 params, the update kernel for the fp32 ones)."""
    from muon_newton_schulz_09_b300 import Muon
    shapes = [(384, 128), (128, 384), (130, 70)]
    lr = 0.02
    for param_dtype in ("bf16", "f32"):
        w, g, m, p = step_case(shapes, "bf16", param_dtype, seed=27)
        P = [dev(x, param_dtype) for x in p]
        with Muon(0, scale_lr_by_shape=False) as m0:
            m0.step(P, [dev(x, "bf16") for x in g], [dev(x, "f32") for x in m], lr=lr, beta=0.95, nesterov=True)
            torch.cuda.synchronize()
            assert m0.get_error() == 0
        for j, (r, c) in enumerate(shapes):
            w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC, scale_lr_by_shape=False)
            upd = lr * np.abs(o).max()
            err = np.abs(host(P[j]) - w_new)
            ulp = bf16_ulp(w_new) if param_dtype == "bf16" else np.abs(w_new) * 2.0 ** -22
            assert np.all(err <= ulp + 0.05 * upd), (param_dtype, r, c, float(err.max()))
            # the shape-scaled update s lr O (s = sqrt(r / c) for tall matrices) is (s - 1) / s away
            if r > c:
                s = oracle.lr_scale(r, c)
                w_scaled, _, _ = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
                assert rel_f(host(P[j]) - p[j], w_scaled - p[j]) > 0.5 * (s - 1.0) / s


def test_workspace_limit_gives_nomem_without_side_effects():
    """A plan that would exceed the handle's device-memory cap fails as an exhausted cudaMalloc does:
    MUON_ERR_NOMEM before any launch, the caller's tensors untouched, plans already built kept, and
    the next call with room builds the plan and computes the right step."""
    from muon_newton_schulz_09_b300 import MUON_ERR_NOMEM, Muon, MuonError
    small = [(128, 256)]
    shapes = [(256, 640), (640, 256), (130, 70)]
    lr = 0.02
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=28)
    P = [dev(x, "bf16") for x in p]
    G = [dev(x, "bf16") for x in g]
    M = [dev(x, "f32") for x in m]
    with Muon(0) as mw:
        # a first plan fits under the cap and stays usable
        xs = [dev(np.ones(s, np.float32), "bf16") for s in small]
        outs = [torch.empty(s, device="cuda") for s in small]
        mw.orthogonalize(xs, outs, steps=1)
        torch.cuda.synchronize()
        held = mw.workspace_bytes()
        assert held > 0
        mw.set_workspace_limit(held + 4096)
        p0 = [t.clone() for t in P]
        m0 = [t.clone() for t in M]
        with pytest.raises(MuonError) as e:
            mw.step(P, G, M, lr=lr, beta=0.95, nesterov=True)
        assert e.value.status == MUON_ERR_NOMEM
        torch.cuda.synchronize()
        assert mw.get_error() == 0 and mw.workspace_bytes() == held
        for a, b in zip(P + M, p0 + m0):
            assert torch.equal(a, b)
        mw.orthogonalize(xs, outs, steps=1)  # the earlier plan still runs
        torch.cuda.synchronize()
        assert rel_f(host(outs[0]), oracle.orthogonalize(np.ones(small[0]), 1, CUBIC)) < TOL
        mw.set_workspace_limit(0)
        mw.step(P, G, M, lr=lr, beta=0.95, nesterov=True)
        torch.cuda.synchronize()
        assert mw.get_error() == 0 and mw.workspace_bytes() > held
    for j, (r, c) in enumerate(shapes):
        w_new, buf_new, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (r, c, float(err.max()))
        assert rel_f(host(M[j]), buf_new) < 1e-6


@pytest.mark.parametrize("coeffs,steps", [(CUBIC, 5), (QUINTIC, 3)], ids=["cubic5", "quintic3"])
def test_per_phase_launches_match_the_oracle(coeffs, steps):
    """persistent = 0: one launch per Gram and combine phase instead of the persistent launch, on the
    ragged batch and on a step whose last combine writes the bf16 parameters."""
    from muon_newton_schulz_09_b300 import Muon
    _, xs = inputs_for(RAGGED, "bf16", seed=12)
    shapes = [(256, 640), (640, 256), (130, 70)]
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=29)
    lr = 0.02
    with Muon(0, persistent=False, a=coeffs[0], b=coeffs[1], c=coeffs[2], steps=steps) as mp:
        got = run_orth(mp, xs, "bf16", "f32", steps, coeffs)
        P = [dev(x, "bf16") for x in p]
        mp.step(P, [dev(x, "bf16") for x in g], [dev(x, "f32") for x in m], lr=lr, beta=0.95, nesterov=True)
        torch.cuda.synchronize()
        assert mp.get_error() == 0
    for x, o in zip(xs, got):
        assert rel_f(o, oracle.orthogonalize(x, steps, coeffs)) < TOL, x.shape
    for j, (r, c) in enumerate(shapes):
        w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, steps, coeffs)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (r, c, float(err.max()))


def test_persistent_and_per_phase_launches_agree_bit_for_bit():
    """The persistent launch and the per-phase launches run the same tiles with the same arithmetic, so
    their outputs are equal bit for bit: orthogonalize (cubic, and the quintic with its default
    carry) on the ragged batch, and a step whose last combine writes bf16 parameters."""
    from muon_newton_schulz_09_b300 import Muon
    _, xs = inputs_for(RAGGED, "bf16", seed=13)
    shapes = [(256, 640), (640, 256), (130, 70), (1, 5)]
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=30)
    outs = {}
    for persistent in (True, False):
        with Muon(0, persistent=persistent) as mu:
            o1 = run_orth(mu, xs, "bf16", "f32", 5, CUBIC)
            o2 = run_orth(mu, xs, "bf16", "bf16", 3, QUINTIC)
            P = [dev(x, "bf16") for x in p]
            M = [dev(x, "f32") for x in m]
            mu.step(P, [dev(x, "bf16") for x in g], M, lr=0.02, beta=0.95, nesterov=True)
            torch.cuda.synchronize()
            assert mu.get_error() == 0
            outs[persistent] = (o1, o2, [host(t) for t in P], [host(t) for t in M])
    for a, b in zip(outs[True], outs[False]):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_default_handle_chooses_the_launches_by_work_per_cluster():
    """The default handle takes the per-phase launches for a 4096 x 16384 matrix (1356 k-blocks per
    cluster per iteration) and the persistent launch for a small set, as launch_choice says."""
    from muon_newton_schulz_09_b300 import Muon, launch_choice
    gen = torch.Generator(device="cuda").manual_seed(5)
    with Muon(0) as mu:
        for shapes, persistent in [([(4096, 16384)], False), ([(256, 768), (768, 256)], True)]:
            assert launch_choice(shapes)[0] is persistent
            x = [torch.randn(s, device="cuda", generator=gen).to(torch.bfloat16) for s in shapes]
            out = [torch.empty(s, device="cuda", dtype=torch.bfloat16) for s in shapes]
            mu.profile_read()
            mu.profile(True)
            mu.orthogonalize(x, out, steps=1)
            torch.cuda.synchronize()
            mu.profile(False)
            prof = mu.profile_read()
            assert mu.get_error() == 0
            assert prof["newton_schulz"][1] == (1 if persistent else 0)
            assert prof["gram_xxt"][1] == (0 if persistent else 1)
            assert prof["combine_ax_bx"][1] == (0 if persistent else 1)


@pytest.mark.parametrize("persistent", [True, False], ids=["persistent", "per_phase"])
def test_step_replays_from_a_cuda_graph(persistent):
    """Once a call has built its plan and schedule, a step on fixed tensors issues kernel launches
    only, so it can be captured in a CUDA graph: each replay is one step, bit for bit what the same
    step does called directly, with momentum and parameters carried from replay to replay."""
    from muon_newton_schulz_09_b300 import Muon
    shapes = [(256, 768), (768, 256), (130, 70), (384, 384)]
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=36)
    lr = 0.02
    with Muon(0, persistent=persistent) as mu:
        G = [dev(x, "bf16") for x in g]
        P, M = [dev(x, "bf16") for x in p], [dev(x, "f32") for x in m]
        Pe, Me = [t.clone() for t in P], [t.clone() for t in M]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):  # direct calls; the first one builds the plan
                mu.step(Pe, G, Me, lr=lr, beta=0.95, nesterov=True, stream=s)
        torch.cuda.synchronize()
        assert mu.get_error() == 0
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            mu.step(P, G, M, lr=lr, beta=0.95, nesterov=True, stream=s)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        assert mu.get_error() == 0
        for a, b in zip(P + M, Pe + Me):
            assert torch.equal(a, b)
        # and the replays moved the parameters: three steps of the oracle
        for j, (r, c) in enumerate(shapes):
            wj, bj = p[j], m[j]
            for _ in range(3):
                wj, bj, o = oracle.muon_step(wj, g[j], bj, lr, 0.95, True, 5, CUBIC)
            upd = 3 * lr * oracle.lr_scale(r, c) * np.abs(o).max()
            assert np.all(np.abs(host(P[j]) - wj) <= 3 * bf16_ulp(wj) + 0.05 * upd), (r, c)


def test_quintic_over_several_persistent_launches():
    """20 quintic iterations take two persistent launches (16 + 4): the second starts from the first's
    X, the folded scale applies only in the first and the update only in the last. The default config
    carries X as hi + lo for c != 0 across both."""
    from muon_newton_schulz_09_b300 import Muon
    shapes = [(256, 640), (640, 256), (130, 70), (384, 384)]
    w, g, m, p = step_case(shapes, "bf16", "bf16", seed=31)
    lr, steps = 0.02, 20
    with Muon(0, steps=steps, a=QUINTIC[0], b=QUINTIC[1], c=QUINTIC[2]) as mq:
        mq.profile_read()
        mq.profile(True)
        P = [dev(x, "bf16") for x in p]
        mq.step(P, [dev(x, "bf16") for x in g], [dev(x, "f32") for x in m], lr=lr, beta=0.95, nesterov=True)
        torch.cuda.synchronize()
        mq.profile(False)
        prof = mq.profile_read()
        assert mq.get_error() == 0
        assert prof["newton_schulz"][1] == 2
    for j, (r, c) in enumerate(shapes):
        w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, steps, QUINTIC)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(P[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (r, c, float(err.max()))


def test_more_shape_groups_than_the_persistent_launch_names():
    """1025 distinct shapes (1 x k rows): the call runs the per-phase launches and is still right."""
    shapes = [(1, k) for k in range(1, 1026)]
    _, xs = inputs_for(shapes, "bf16", seed=47)
    from muon_newton_schulz_09_b300 import Muon
    with Muon(0) as mu:
        got = run_orth(mu, xs, "bf16", "f32", 5, CUBIC)
    for j in (0, 1, 511, 1024):
        assert rel_f(got[j], oracle.orthogonalize(xs[j], 5, CUBIC)) < TOL, shapes[j]
