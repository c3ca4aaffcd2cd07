"""Seeded synthetic workloads for the Muon Newton-Schulz step.

This module draws numbers and fixes shapes. It does none of the Muon
arithmetic (no momentum, norm, iteration or update). Both the fp64 oracle and
the CUDA path are fed from it, and it is the only code they share.

Every matrix of a workload is generated from its own seed tuple
``(workload seed, role, matrix index)``. One matrix of a large batch can
therefore be rebuilt on its own, without generating the rest. That is how the
full-size parity tests take their sampled matrices.

Values are returned as float32 numpy arrays. Tensors that are bf16 on the
device hold only bf16-representable values, rounded to nearest-even by
``bf16_round``.

The shapes follow the GPT-2 hidden-matrix sets that the modded-nanogpt
speedrun trains with Muon ("How to train a GPT model in 3 minutes: an
analysis of modded-nanogpt's optimizations", section 2, custom Muon
optimizer; GPT-2 124M per section 1). The shapes themselves, the
distributions and the Newton-Schulz settings of each workload are not given
on those pages. They are the five stated benchmark configurations.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 22          # elements per independent stream: the result does not depend on thread count
_THREADS = max(1, min(32, os.cpu_count() or 1))

# roles in the seed tuple
ROLE_GRAD, ROLE_SPIKE_P, ROLE_SPIKE_Q, ROLE_MOMENTUM, ROLE_PARAM, ROLE_INPUT = range(6)


def normal(seed: tuple, shape, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) samples.

    The array is cut into fixed 4M-element chunks, and each chunk is drawn
    from its own PCG64 stream, spawned from ``SeedSequence(seed)``. The
    values depend on the seed and the shape only, not on the thread count.
    """
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, np.float32)
    nch = max(1, (n + _CHUNK - 1) // _CHUNK)
    streams = np.random.SeedSequence(list(seed)).spawn(nch)

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        np.random.Generator(np.random.PCG64(streams[i])).standard_normal(
            hi - lo, dtype=np.float32, out=out[lo:hi])

    if nch == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(fill, range(nch)))
    if std != 1.0:
        out *= np.float32(std)
    return out.reshape(shape)


def generator(seed: tuple) -> np.random.Generator:
    """A small single-stream generator for vectors (signs, spectra, permutations)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(seed))))


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> float32 holding the nearest bf16 value (ties to even). Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(np.shape(x))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 encodings of a float32 array whose values are already bf16-representable."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16).reshape(np.shape(x))


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple                 # ((rows, cols), ...) as stored, row-major
    kind: str                     # "step" (momentum + orthogonalize + update) or "orthogonalize"
    dtype: str                    # gradient / input dtype on the device: "bf16" or "f32"
    param_dtype: str = "bf16"
    steps: int = 5
    coeffs: tuple = (1.5, -0.5, 0.0)
    eps: float = 1e-7
    beta: float = 0.95
    nesterov: bool = True
    lr: float = 0.02
    grad_std: float = 1e-3
    spike_rank: int = 0
    spike_gain: float = 0.0
    zero_momentum: bool = False
    param_std: float = 0.02
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def count(self) -> int:
        return len(self.shapes)

    def elements(self) -> int:
        return int(sum(r * c for r, c in self.shapes))


def _gpt2_shapes(layers: int, d: int) -> tuple:
    per_layer = [(d, d)] * 4 + [(d, 4 * d), (4 * d, d)]
    return tuple(per_layer * layers)


SINGLE_128x256 = Workload(
    name="single_128x256_f32", shapes=((128, 256),), kind="step", dtype="f32",
    param_dtype="f32", grad_std=1.0, zero_momentum=True, seed=1,
    notes="one fp32 128x256 gradient N(0,1); zero momentum, beta=0.95; 5 cubic iterations")

GPT2_124M = Workload(
    name="gpt2_124m_hidden", shapes=_gpt2_shapes(12, 768), kind="step", dtype="bf16",
    grad_std=1e-3, spike_rank=4, spike_gain=50.0, seed=2,
    notes="12 x (4x 768x768, 768x3072, 3072x768) bf16, N(0,1e-3) + rank-4 spike x50, Nesterov beta=0.95, 5 iterations")

SQUARE_64x1024 = Workload(
    name="square_64x1024", shapes=((1024, 1024),) * 64, kind="orthogonalize", dtype="bf16",
    grad_std=1.0, seed=3,
    notes="64 bf16 1024x1024 N(0,1), no momentum, 5 cubic iterations")

ILLCOND_4096x16384 = Workload(
    name="illcond_4096x16384", shapes=((4096, 16384),), kind="orthogonalize", dtype="bf16",
    steps=10, seed=4,
    notes="U diag(s) V^T, s log-uniform in [1e-4, 1], 10 iterations")

GPT2_350M = Workload(
    name="gpt2_350m_hidden", shapes=_gpt2_shapes(24, 1024), kind="step", dtype="bf16",
    grad_std=1e-3, seed=5,
    notes="24 x (4x 1024^2, 1024x4096, 4096x1024) bf16, N(0,1e-3), full step incl. update")

# The c != 0 path at benchmark scale: the GPT-2 124M set, its gradients with the rank-4 spike,
# and the second-order Newton-Schulz quintic (15, -10, 3)/8 (the pages give no coefficients; this
# is the textbook polynomial). The spike's bf16 rounding noise lands in the tiny bulk singular
# values and the quintic's slope 15/8 at zero amplifies it every iteration: X rounded to bf16
# every iteration ends about 2.1e-2 from the exact result, so calls with c != 0 carry X as
# bf16 hi + lo by default.
GPT2_124M_QUINTIC = Workload(
    name="gpt2_124m_hidden_quintic", shapes=_gpt2_shapes(12, 768), kind="step", dtype="bf16",
    grad_std=1e-3, spike_rank=4, spike_gain=50.0, seed=2, coeffs=(15 / 8, -10 / 8, 3 / 8),
    notes="GPT-2 124M hidden set, N(0,1e-3) + rank-4 spike x50, quintic (15,-10,3)/8 Newton-Schulz, 5 iterations")

WORKLOADS = {w.name: w for w in (SINGLE_128x256, GPT2_124M, SQUARE_64x1024, ILLCOND_4096x16384, GPT2_350M,
                                 GPT2_124M_QUINTIC)}


# --------------------------------------------------------------------------------------
# per-matrix tensors
# --------------------------------------------------------------------------------------

def _round_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_round(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def gradient(w: Workload, j: int, seed_offset: int = 0) -> np.ndarray:
    """Gradient (or orthogonalize input) of matrix j.

    ``N(0, grad_std^2)`` entries. With ``spike_rank > 0`` a low-rank term is added:
    ``spike_gain * grad_std * (P Q^T) / sqrt(rank)``, where P (rows x rank) and
    Q (cols x rank) have N(0,1) entries. Each entry of the spike then has
    standard deviation ``spike_gain`` times that of the dense part. The result
    is rounded to the device dtype.
    """
    r, c = w.shapes[j]
    if w.name == ILLCOND_4096x16384.name or w.extra.get("illcond"):
        return _round_dtype(illconditioned(w.seed + seed_offset, r, c), w.dtype)
    base = (w.seed + seed_offset, j)
    g = normal(base + (ROLE_GRAD,), (r, c), w.grad_std)
    if w.spike_rank > 0:
        p = normal(base + (ROLE_SPIKE_P,), (r, w.spike_rank))
        q = normal(base + (ROLE_SPIKE_Q,), (c, w.spike_rank))
        g += (p @ q.T) * np.float32(w.spike_gain * w.grad_std / np.sqrt(w.spike_rank))
    return _round_dtype(g, w.dtype)


def momentum_buffer(w: Workload, j: int) -> np.ndarray:
    """fp32 momentum state before the step.

    Zero when the workload says so. Otherwise it is the buffer after one earlier
    step from zero: a gradient drawn with another seed, of the same distribution.
    """
    r, c = w.shapes[j]
    if w.zero_momentum:
        return np.zeros((r, c), np.float32)
    return gradient(w, j, seed_offset=1000).astype(np.float32)


def parameter(w: Workload, j: int) -> np.ndarray:
    """Weight matrix before the step: N(0, param_std^2), random init in the device dtype."""
    r, c = w.shapes[j]
    return _round_dtype(normal((w.seed, j, ROLE_PARAM), (r, c), w.param_std), w.param_dtype)


# --------------------------------------------------------------------------------------
# ill-conditioned matrix U diag(s) V^T
# --------------------------------------------------------------------------------------

def _fwht(a: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along axis 0 (Sylvester order). Length is a power of two."""
    a = np.array(a, dtype=np.float64, copy=True)
    n = a.shape[0]
    h = 1
    while h < n:
        v = a.reshape(n // (2 * h), 2, h, -1)
        x = v[:, 0].copy()
        v[:, 0] += v[:, 1]
        v[:, 1] = x - v[:, 1]
        h *= 2
    return a


def random_orthonormal_columns(seed: tuple, n: int, k: int) -> np.ndarray:
    """n x k matrix with orthonormal columns (k <= n, n a power of two).

    Built as D1 H D2 H E / n. H is the n x n Sylvester-Hadamard matrix, the D
    are random sign diagonals, and E picks k columns in random order. It is a
    dense orthogonal construction that costs O(n k log n), not the O(n^3) of a
    QR factorisation.
    """
    assert n & (n - 1) == 0 and k <= n
    g = generator(seed)
    d1 = g.choice([-1.0, 1.0], n)
    d2 = g.choice([-1.0, 1.0], n)
    perm = g.permutation(n)[:k]
    e = np.zeros((n, k))
    e[perm, np.arange(k)] = 1.0
    m = _fwht(e)
    m *= d2[:, None]
    m = _fwht(m)
    m *= d1[:, None] / n
    return m


def log_uniform_spectrum(seed: tuple, k: int, lo: float = 1e-4, hi: float = 1.0) -> np.ndarray:
    g = generator(seed)
    return np.exp(g.uniform(np.log(lo), np.log(hi), k))


def illconditioned(seed: int, r: int, c: int, lo: float = 1e-4) -> np.ndarray:
    """float32 r x c matrix U diag(s) V^T, with s log-uniform in [lo, 1] and random orthonormal U and V.

    Both r and c must be powers of two.
    """
    k = min(r, c)
    u = random_orthonormal_columns((seed, 0, 10), r, k)
    v = random_orthonormal_columns((seed, 0, 11), c, k)
    s = log_uniform_spectrum((seed, 0, 12), k, lo)
    return ((u * s[None, :]) @ v.T).astype(np.float32)


def small_workload(name: str, shapes, kind: str = "orthogonalize", dtype: str = "bf16", **kw) -> Workload:
    """A test-sized workload with the same recipe as the named ones."""
    return Workload(name=name, shapes=tuple(tuple(s) for s in shapes), kind=kind, dtype=dtype, **kw)
