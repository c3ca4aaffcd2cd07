"""Plain fp64 CPU oracle of the Muon optimizer step. TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may call this module. The CUDA library never calls it, and it shares no code
with the CUDA library. Both are fed from the seeded generators in
``workloads.py``.

What the pages fix
------------------
"How to train a GPT model in 3 minutes: an analysis of modded-nanogpt's
optimizations", section 2 (custom Muon optimizer), says three things. Muon
replaces AdamW for the hidden projection matrices. Its idea comes from
spectral gradient descent, which steps along the orthogonal polar factor
U V^T of the update. It reaches that factor with a Newton-Schulz iteration
in place of an SVD. The record analysis on the mhpq.cn page, section 6.2,
confirms that projection matrices take the Muon path and gates take Adam.

What the pages leave open, and the reading taken here
------------------------------------------------------
The pages print no formula. Each step below is the plainest reading of the
stated configuration:

1. momentum:  buf <- beta*buf + g;  u = g + beta*buf (Nesterov) or u = buf
2. normalise: X0 = u / (||u||_F + eps)
3. orient:    X = X0^T when rows > cols (square matrices are not transposed)
4. iterate k times:  A = X X^T;  B = b*A + c*A*A;  X <- a*X + B X
5. restore:   O = X^T if transposed in step 3
6. update:    W <- W * (1 - lr * wd) - lr * max(1, rows/cols)^0.5 * O

The weight decay wd (0 unless given) follows the energy-efficiency article on
Modded-NanoGPT (hyperparameter paragraph), which reports wd = 1.0 without its
form; the decoupled form above is the plainest reading.

Everything is float64. Matrix products use numpy's matmul, a library
primitive. There is no blocking, fusion or reordering beyond the steps as
written.

Parity pins live in the CPU test suite. They are: the SVD closed form
U diag(p^k(sigma)) V^T for any coefficients; the polar factor U V^T as the
limit; exact rational arithmetic on hand-worked 2x2 cases; invariants
(singular values in [0,1], transpose, orthogonal and scale equivariance,
zero input); and elementwise closed forms for the momentum and update steps.
"""
from __future__ import annotations

import numpy as np

DEFAULT_COEFFS = (1.5, -0.5, 0.0)
DEFAULT_EPS = 1e-7


def momentum(g, buf, beta: float, nesterov: bool):
    """Step 1. Returns (new buffer, Newton-Schulz input u), both float64.

    buf_new = beta*buf + g.  u = g + beta*buf_new with Nesterov, else u = buf_new.
    """
    g = np.asarray(g, dtype=np.float64)
    buf = np.asarray(buf, dtype=np.float64)
    buf_new = beta * buf + g
    u = g + beta * buf_new if nesterov else buf_new
    return buf_new, u


def frobenius_normalize(u, eps: float = DEFAULT_EPS):
    """Step 2. X0 = u / (||u||_F + eps). The eps sits outside the square root; u = 0 gives 0."""
    u = np.asarray(u, dtype=np.float64)
    norm = np.sqrt(np.sum(u * u))
    return u / (norm + eps)


def newton_schulz(x, steps: int, a: float, b: float, c: float):
    """Step 4 on an n x m matrix (n <= m expected, not required).

    Each iteration applies X <- a*X + (b*A + c*A*A) X with A = X X^T, the odd
    matrix polynomial a*X + b*(X X^T) X + c*(X X^T)^2 X.
    """
    x = np.asarray(x, dtype=np.float64)
    for _ in range(steps):
        gram = x @ x.T
        poly = b * gram + c * (gram @ gram)
        x = a * x + poly @ x
    return x


def orthogonalize(g, steps: int = 5, coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS):
    """Steps 2-5: normalise, orient so the Gram side is the short one, iterate, restore orientation."""
    a, b, c = coeffs
    x0 = frobenius_normalize(g, eps)
    transposed = x0.shape[0] > x0.shape[1]
    x = x0.T if transposed else x0
    x = newton_schulz(x, steps, a, b, c)
    return x.T if transposed else x


def lr_scale(rows: int, cols: int) -> float:
    """Step 6 shape factor max(1, rows/cols)^0.5. rows is the stored first dimension."""
    return max(1.0, rows / cols) ** 0.5


def muon_update(w, o, lr: float, scale_lr_by_shape: bool = True, weight_decay: float = 0.0):
    """Step 6. W (1 - lr*wd) - lr * s * O in float64, where s is lr_scale or 1."""
    w = np.asarray(w, dtype=np.float64)
    s = lr_scale(*w.shape) if scale_lr_by_shape else 1.0
    return w * (1.0 - lr * weight_decay) - (lr * s) * np.asarray(o, dtype=np.float64)


def muon_step(w, g, buf, lr: float, beta: float, nesterov: bool, steps: int = 5,
              coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS, scale_lr_by_shape: bool = True,
              weight_decay: float = 0.0):
    """One full Muon step for one matrix. Returns (W_new, buf_new, O), all float64."""
    buf_new, u = momentum(g, buf, beta, nesterov)
    o = orthogonalize(u, steps, coeffs, eps)
    return muon_update(w, o, lr, scale_lr_by_shape, weight_decay), buf_new, o


def rel_frobenius(x, ref) -> float:
    """||x - ref||_F / ||ref||_F in float64 (absolute error when ref is 0)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.linalg.norm(x - ref)
    n = np.linalg.norm(ref)
    return float(d / n) if n > 0 else float(d)
