"""Pins for the fp64 oracle. CPU only.

The oracle is checked against things outside its own code:
  * the SVD closed form U diag(p^k(sigma)) V^T (LAPACK's SVD, not matmul iteration);
  * the polar factor U V^T as the limit of the cubic iteration;
  * hand-worked 2x2 cases (tests/golden/ns_2x2.json) and exact rational
    arithmetic on tiny inputs (brute force with fractions.Fraction);
  * invariants: singular values in [0, 1], transpose / orthogonal / scale
    equivariance, zero input;
  * elementwise closed forms for the momentum and update steps.
The last group plants plausible mistakes in copies of the oracle's steps and
checks that at least one pin catches each of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import muon_oracle as mo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ns_2x2.json")
CUBIC = (1.5, -0.5, 0.0)
QUINTIC = (15 / 8, -10 / 8, 3 / 8)
ODD = (2.0, -1.5, 0.5)


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def F(*args):
    return Fraction(*args)


# ----------------------------------------------------------------------------- brute force

def frac_matmul(a, b):
    return [[sum(a[i][k] * b[k][j] for k in range(len(b))) for j in range(len(b[0]))] for i in range(len(a))]


def frac_T(a):
    return [list(r) for r in zip(*a)]


def frac_ns(x, steps, a, b, c):
    """Newton-Schulz in exact rationals on a tiny matrix that is already normalised."""
    for _ in range(steps):
        g = frac_matmul(x, frac_T(x))
        gg = frac_matmul(g, g)
        n = len(g)
        poly = [[b * g[i][j] + c * gg[i][j] for j in range(n)] for i in range(n)]
        px = frac_matmul(poly, x)
        x = [[a * x[i][j] + px[i][j] for j in range(len(x[0]))] for i in range(len(x))]
    return x


# ----------------------------------------------------------------------------- closed form

def svd_closed_form(g, steps, coeffs, eps=0.0):
    """U diag(p^k(sigma / (||G||_F + eps))) V^T, with ||G||_F = sqrt(sum sigma^2) taken from the SVD."""
    a, b, c = coeffs
    u, s, vt = np.linalg.svd(np.asarray(g, np.float64), full_matrices=False)
    p = s / (math.sqrt(float(np.sum(s * s))) + eps)
    for _ in range(steps):
        p = a * p + b * p ** 3 + c * p ** 5
    return (u * p) @ vt


def closed_form_error(orth, shapes=((6, 10), (10, 6), (7, 7), (1, 5), (5, 1)),
                      coeff_sets=(CUBIC, QUINTIC, ODD), steps_list=(0, 1, 3, 5)):
    rng = np.random.default_rng(12345)
    worst = 0.0
    for shape in shapes:
        g = rng.standard_normal(shape)
        for coeffs in coeff_sets:
            for k in steps_list:
                want = svd_closed_form(g, k, coeffs, eps=1e-7)
                got = orth(g, k, coeffs, 1e-7)
                if np.shape(got) != np.shape(want):
                    return float("inf")
                worst = max(worst, mo.rel_frobenius(got, want))
    return worst


def test_closed_form_any_coefficients():
    assert closed_form_error(oracle.orthogonalize) < 1e-12


def test_closed_form_workload_shape_many_steps():
    rng = np.random.default_rng(7)
    g = rng.standard_normal((128, 256))
    for k in (5, 10):
        assert mo.rel_frobenius(oracle.orthogonalize(g, k, CUBIC, 0.0), svd_closed_form(g, k, CUBIC)) < 1e-12


def test_polar_limit():
    """Enough cubic steps reach U V^T. At 5 steps the iterate is still far from it (about 0.5 in rel-F)."""
    rng = np.random.default_rng(1)
    g = rng.standard_normal((128, 256))
    u, _, vt = np.linalg.svd(g, full_matrices=False)
    polar = u @ vt
    assert mo.rel_frobenius(oracle.orthogonalize(g, 25, CUBIC, 0.0), polar) < 1e-10
    far = mo.rel_frobenius(oracle.orthogonalize(g, 5, CUBIC, 0.0), polar)
    assert 0.2 < far < 0.8


# ----------------------------------------------------------------------------- hand-worked 2x2

@pytest.mark.parametrize("case", golden()["cases"], ids=lambda c: c["name"])
def test_golden_2x2_ns(case):
    g = np.array(case["G"], dtype=np.float64)
    coeffs = tuple(float(F(x)) for x in case["coeffs"])
    scale = 1.0
    if "scale" in case:
        scale = {"1/sqrt(3)": 1 / math.sqrt(3)}[case["scale"]]
    want = scale * np.array([[float(F(x)) for x in row] for row in case["expected"]])
    got = oracle.orthogonalize(g, case["steps"], coeffs, 0.0)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)
    if "polar_factor" in case:
        pf = case["polar_factor"]
        q = np.array([[float(F(x)) for x in row] for row in pf["matrix"]]) / math.sqrt(5)
        np.testing.assert_allclose(oracle.orthogonalize(g, 40, coeffs, 0.0), q, atol=1e-14)


def test_golden_values_match_exact_rationals():
    """The stored fractions equal the brute-force rational iteration (cases with rational norm)."""
    for case in golden()["cases"]:
        if "scale" in case:
            continue
        g = [[F(v) for v in row] for row in case["G"]]
        norm2 = sum(v * v for row in g for v in row)
        norm = Fraction(math.isqrt(norm2.numerator), math.isqrt(norm2.denominator))
        assert norm * norm == norm2
        x0 = [[v / norm for v in row] for row in g]
        a, b, c = (F(x) for x in case["coeffs"])
        tall = len(g) > len(g[0])
        x = frac_T(x0) if tall else x0
        x = frac_ns(x, case["steps"], a, b, c)
        x = frac_T(x) if tall else x
        assert x == [[F(v) for v in row] for row in case["expected"]]


def test_exact_rational_several_steps():
    """Five cubic steps on diag(3,4)/5 in exact arithmetic against the oracle."""
    x = frac_ns([[F(3, 5), F(0)], [F(0), F(4, 5)]], 5, F(3, 2), F(-1, 2), F(0))
    want = np.array([[float(v) for v in row] for row in x])
    got = oracle.orthogonalize(np.diag([3.0, 4.0]), 5, CUBIC, 0.0)
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    # non-diagonal rational input: G = [[3, 4], [0, 0]] has norm 5
    x = frac_ns([[F(3, 5), F(4, 5)], [F(0), F(0)]], 4, F(3, 2), F(-1, 2), F(0))
    got = oracle.orthogonalize(np.array([[3.0, 4.0], [0.0, 0.0]]), 4, CUBIC, 0.0)
    np.testing.assert_allclose(got, np.array([[float(v) for v in r] for r in x]), atol=1e-15)


# ----------------------------------------------------------------------------- invariants

def test_singular_values_in_unit_interval():
    rng = np.random.default_rng(3)
    for shape in ((32, 80), (80, 32), (40, 40)):
        g = rng.standard_normal(shape)
        for k in (1, 5, 12):
            s = np.linalg.svd(oracle.orthogonalize(g, k, CUBIC), compute_uv=False)
            assert s.max() <= 1.0 + 1e-12 and s.min() >= 0.0


def test_transpose_equivariance():
    rng = np.random.default_rng(4)
    g = rng.standard_normal((24, 60))
    for coeffs in (CUBIC, QUINTIC):
        np.testing.assert_allclose(oracle.orthogonalize(g.T, 5, coeffs), oracle.orthogonalize(g, 5, coeffs).T,
                                   atol=1e-13)


def test_orthogonal_equivariance():
    rng = np.random.default_rng(5)
    g = rng.standard_normal((20, 36))
    q, _ = np.linalg.qr(rng.standard_normal((20, 20)))
    r, _ = np.linalg.qr(rng.standard_normal((36, 36)))
    lhs = oracle.orthogonalize(q @ g @ r, 5, CUBIC)
    rhs = q @ oracle.orthogonalize(g, 5, CUBIC) @ r
    assert mo.rel_frobenius(lhs, rhs) < 1e-12


def test_scale_invariance_and_zero():
    rng = np.random.default_rng(6)
    g = rng.standard_normal((16, 48))
    base = oracle.orthogonalize(g, 5, CUBIC, 0.0)
    for s in (1e-3, 7.0, 1e4):
        assert mo.rel_frobenius(oracle.orthogonalize(s * g, 5, CUBIC, 0.0), base) < 1e-13
    z = oracle.orthogonalize(np.zeros((5, 9)), 5, CUBIC, 1e-7)
    assert np.all(z == 0.0)


def test_momentum_convention_proportional():
    """Zero start: the EMA (lerp) convention gives (1-beta) times this u, so O is the same (NS is scale invariant)."""
    rng = np.random.default_rng(8)
    g = rng.standard_normal((12, 30))
    beta = 0.95
    _, u = oracle.momentum(g, np.zeros_like(g), beta, True)
    buf_lerp = (1 - beta) * g
    u_lerp = (1 - beta) * g + beta * buf_lerp
    np.testing.assert_allclose(u_lerp, (1 - beta) * u, rtol=1e-14)
    assert mo.rel_frobenius(oracle.orthogonalize(u_lerp, 5, CUBIC, 0.0),
                            oracle.orthogonalize(u, 5, CUBIC, 0.0)) < 1e-13


# ----------------------------------------------------------------------------- momentum and update

def test_momentum_elementwise():
    g = [[1.0, -2.0, 0.5]]
    buf = [[0.25, 4.0, -1.0]]
    beta = 0.9
    bn, un = mo.momentum(np.array(g), np.array(buf), beta, True)
    bp, up = mo.momentum(np.array(g), np.array(buf), beta, False)
    for j in range(3):
        nb = beta * buf[0][j] + g[0][j]
        assert bn[0, j] == nb and bp[0, j] == nb
        assert un[0, j] == g[0][j] + beta * nb
        assert up[0, j] == nb
    b0, u0 = mo.momentum(np.array(g), np.array(buf), 0.0, True)
    assert np.array_equal(u0, np.array(g)) and np.array_equal(b0, np.array(g))


def test_lr_scale():
    assert oracle.lr_scale(3072, 768) == 2.0
    assert oracle.lr_scale(768, 3072) == 1.0
    assert oracle.lr_scale(1024, 1024) == 1.0
    assert oracle.lr_scale(4096, 1024) == 2.0


def test_lr_scale_via_step():
    """A 3x1 column: O = g/|g| after the transpose rule, update scaled by sqrt(3)."""
    g = np.array([[1.0], [2.0], [2.0]])
    w_new, _, o = mo.muon_step(np.zeros((3, 1)), g, np.zeros((3, 1)), 0.5, 0.0, False, 4, CUBIC, 0.0)
    np.testing.assert_allclose(o, g / 3.0, atol=1e-15)
    np.testing.assert_allclose(w_new, -0.5 * math.sqrt(3.0) * g / 3.0, atol=1e-15)


def test_lr_scale_off_via_step():
    """scale_lr_by_shape = False: the same 3x1 column takes the plain lr, with no sqrt(3) factor."""
    g = np.array([[1.0], [2.0], [2.0]])
    w = np.array([[0.5], [-1.0], [0.25]])
    w_new, _, o = mo.muon_step(w, g, np.zeros((3, 1)), 0.5, 0.0, False, 4, CUBIC, 0.0, False)
    np.testing.assert_allclose(o, g / 3.0, atol=1e-15)
    np.testing.assert_allclose(w_new, w - 0.5 * g / 3.0, atol=1e-15)
    # the wide orientation is unaffected by the switch either way (max(1, r/c) = 1)
    wide = np.array([[3.0, 4.0]])
    a, _, _ = mo.muon_step(np.zeros((1, 2)), wide, np.zeros((1, 2)), 0.1, 0.0, False, 2, CUBIC, 0.0, True)
    b, _, _ = mo.muon_step(np.zeros((1, 2)), wide, np.zeros((1, 2)), 0.1, 0.0, False, 2, CUBIC, 0.0, False)
    np.testing.assert_allclose(a, [[-0.06, -0.08]], atol=1e-15)
    np.testing.assert_allclose(b, a, atol=0)


def test_rel_frobenius_hand_values():
    """||x - ref||_F / ||ref||_F on a 2x2 worked by hand: the difference has norm 1 and ref has norm
    sqrt(1 + 4 + 9 + 25) = sqrt(39). A dropped square root would give 1/39, the wrong denominator
    (||x||_F = sqrt(30)) 1/sqrt(30). A zero reference gives the absolute error."""
    x = np.array([[1.0, 2.0], [3.0, 4.0]])
    ref = np.array([[1.0, 2.0], [3.0, 5.0]])
    assert oracle.rel_frobenius(x, ref) == pytest.approx(1.0 / math.sqrt(39.0), rel=1e-15)
    assert oracle.rel_frobenius(ref, ref) == 0.0
    assert oracle.rel_frobenius(np.array([[3.0, 4.0]]), np.zeros((1, 2))) == pytest.approx(5.0, rel=1e-15)


def test_weight_decay_closed_form():
    """W' = W (1 - lr wd) - lr s O, element by element: a 1x2 row (no transpose, s = 1) whose
    orthogonalised update is g/|g| exactly (a single row is its own polar factor at any step count)."""
    w = np.array([[2.0, -4.0]])
    g = np.array([[3.0, 4.0]])
    lr, wd = 0.1, 1.0
    w_new, _, o = mo.muon_step(w, g, np.zeros((1, 2)), lr, 0.0, False, 3, CUBIC, 0.0, True, wd)
    np.testing.assert_allclose(o, g / 5.0, atol=1e-15)
    np.testing.assert_allclose(w_new, [[2.0 * 0.9 - 0.1 * 0.6, -4.0 * 0.9 - 0.1 * 0.8]], atol=1e-15)
    # wd = 0 leaves the plain update
    w0, _, _ = mo.muon_step(w, g, np.zeros((1, 2)), lr, 0.0, False, 3, CUBIC, 0.0, True, 0.0)
    np.testing.assert_allclose(w0, w - lr * g / 5.0, atol=1e-15)


def test_pins_catch_planted_weight_decay_mistakes(monkeypatch):
    def coupled(w, o, lr, scale_lr_by_shape=True, weight_decay=0.0):  # decay without the lr factor
        s = mo.lr_scale(*np.shape(w)) if scale_lr_by_shape else 1.0
        return np.asarray(w, np.float64) * (1.0 - weight_decay) - lr * s * np.asarray(o, np.float64)

    def on_update(w, o, lr, scale_lr_by_shape=True, weight_decay=0.0):  # decay applied to O, not W
        s = mo.lr_scale(*np.shape(w)) if scale_lr_by_shape else 1.0
        return np.asarray(w, np.float64) - lr * s * (1.0 + weight_decay) * np.asarray(o, np.float64)

    for fn in (coupled, on_update):
        with monkeypatch.context() as m:
            m.setattr(mo, "muon_update", fn)
            with pytest.raises(AssertionError):
                test_weight_decay_closed_form()


@pytest.mark.parametrize("case", golden()["muon_step"], ids=lambda c: c["name"])
def test_golden_muon_step(case):
    w = np.array(case["W"], np.float64)
    g = np.array(case["G"], np.float64)
    buf = np.array(case["buf"], np.float64)
    coeffs = tuple(float(F(x)) for x in case["coeffs"])
    w_new, buf_new, _ = oracle.muon_step(w, g, buf, float(F(case["lr"])), float(F(case["beta"])),
                                         case["nesterov"], case["steps"], coeffs, 0.0)
    scale = 1.0
    if "expected_W_scale" in case:
        scale = {"-1/(10*sqrt(65))": -1 / (10 * math.sqrt(65))}[case["expected_W_scale"]]
    want = scale * np.array([[float(F(x)) for x in r] for r in case["expected_W"]])
    np.testing.assert_allclose(w_new, want, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(buf_new, np.array([[float(F(x)) for x in r] for r in case["expected_buf"]]))


# ----------------------------------------------------------------------------- planted mistakes

def _orth_from(ns=None, normalize=None, restore=True):
    ns = ns or mo.newton_schulz
    normalize = normalize or mo.frobenius_normalize

    def orth(g, steps, coeffs, eps):
        x0 = normalize(g, eps)
        t = x0.shape[0] > x0.shape[1]
        x = ns(x0.T if t else x0, steps, *coeffs)
        return x.T if (t and restore) else x
    return orth


def _ns_wrong_side(x, steps, a, b, c):
    """Gram taken as X^T X and applied from the left; differs from the right answer for square X."""
    for _ in range(steps):
        gram = x.T @ x
        poly = b * gram + c * gram @ gram
        x = a * x + (poly @ x if x.shape[0] == x.shape[1] else x @ poly)
    return x


def _ns_no_b(x, steps, a, b, c):
    return mo.newton_schulz(x, steps, a, 0.0, c)


def _ns_b_sign(x, steps, a, b, c):
    return mo.newton_schulz(x, steps, a, -b, c)


def _ns_c_as_a2(x, steps, a, b, c):
    for _ in range(steps):
        gram = x @ x.T
        x = a * x + (b * gram + c * gram) @ x
    return x


def _ns_one_short(x, steps, a, b, c):
    return mo.newton_schulz(x, max(0, steps - 1), a, b, c)


def _norm_maxabs(u, eps):
    u = np.asarray(u, np.float64)
    return u / (np.abs(u).max() + eps)


def _norm_squared(u, eps):
    u = np.asarray(u, np.float64)
    return u / (np.sum(u * u) + eps)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mutant", [
    _orth_from(ns=_ns_wrong_side), _orth_from(ns=_ns_no_b), _orth_from(ns=_ns_b_sign),
    _orth_from(ns=_ns_c_as_a2), _orth_from(ns=_ns_one_short), _orth_from(normalize=_norm_maxabs),
    _orth_from(normalize=_norm_squared), _orth_from(restore=False)],
    ids=["gram_side", "drop_b", "b_sign", "c_term", "one_step_short", "maxabs_norm", "squared_norm",
         "no_restore"])
def test_pins_catch_planted_ns_mistakes(mutant):
    assert closed_form_error(mutant) > 1e-6


def test_pins_catch_planted_step_mistakes(monkeypatch):
    cases = golden()["muon_step"]

    def fails():
        try:
            test_momentum_elementwise()
            test_lr_scale_via_step()
            for c in cases:
                test_golden_muon_step(c)
        except AssertionError:
            return True
        return False

    assert not fails()

    def mom_old_buf(g, buf, beta, nesterov):
        g = np.asarray(g, np.float64)
        buf = np.asarray(buf, np.float64)
        nb = beta * buf + g
        return nb, (g + beta * buf if nesterov else nb)

    def mom_no_g(g, buf, beta, nesterov):
        g = np.asarray(g, np.float64)
        buf = np.asarray(buf, np.float64)
        nb = beta * buf + g
        return nb, (beta * nb if nesterov else nb)

    def upd_plus(w, o, lr, scale_lr_by_shape=True, weight_decay=0.0):
        s = mo.lr_scale(*np.shape(w)) if scale_lr_by_shape else 1.0
        return np.asarray(w, np.float64) * (1.0 - lr * weight_decay) + lr * s * np.asarray(o, np.float64)

    def scale_inverted(rows, cols):
        return max(1.0, cols / rows) ** 0.5

    for name, fn in (("momentum", mom_old_buf), ("momentum", mom_no_g), ("muon_update", upd_plus),
                     ("lr_scale", scale_inverted)):
        with monkeypatch.context() as m:
            m.setattr(mo, name, fn)
            assert fails(), f"planted mistake in {name} ({fn.__name__}) not caught"
