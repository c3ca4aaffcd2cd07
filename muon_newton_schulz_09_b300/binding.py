"""ctypes binding of libmuon.so (the C ABI in include/muon.h).

Argument marshalling only: every step of the Muon path runs in the library's
CUDA kernels. Torch tensors are accepted for convenience (device memory and
streams); nothing here computes on them. Importing this module does not need a
GPU; creating a ``Muon`` handle does.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libmuon.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "muon.h")

MUON_OK, MUON_ERR_INVALID, MUON_ERR_CUDA, MUON_ERR_NOMEM, MUON_ERR_UNSUPPORTED, MUON_ERR_TIMEOUT = range(6)
MUON_F32, MUON_BF16 = 0, 1
MUON_CARRY_WHEN_C = 2
MUON_PERSISTENT_AUTO = 2
KERNEL_KINDS = 9


class MuonError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class MuonMatrix(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld", ctypes.c_int64), ("dtype", ctypes.c_int32)]


class MuonConfig(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int32), ("a", ctypes.c_float), ("b", ctypes.c_float), ("c", ctypes.c_float),
                ("eps", ctypes.c_float), ("scale_lr_by_shape", ctypes.c_int32), ("weight_decay", ctypes.c_float),
                ("precise_carry", ctypes.c_int32), ("persistent", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None


def header_functions() -> list:
    """Names of the functions include/muon.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_]+)\s*\(", text)))


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmuon.so. Raises if it has not been built: there is no fallback path."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with `python -m muon_newton_schulz_09_b300.build`")
    lib = ctypes.CDLL(path)
    c = ctypes
    P = c.POINTER
    sig = {
        "muon_default_config": (None, [P(MuonConfig)]),
        "muon_create": (c.c_int, [P(c.c_void_p), c.c_int, P(MuonConfig)]),
        "muon_destroy": (c.c_int, [c.c_void_p]),
        "muon_orthogonalize": (c.c_int, [c.c_void_p, P(MuonMatrix), P(MuonMatrix), c.c_int, c.c_int, c.c_float,
                                         c.c_float, c.c_float, c.c_void_p]),
        "muon_step": (c.c_int, [c.c_void_p, P(MuonMatrix), P(MuonMatrix), P(MuonMatrix), c.c_int, c.c_float,
                                c.c_float, c.c_int, c.c_void_p]),
        "muon_get_error": (c.c_int, [c.c_void_p, c.c_void_p]),
        "muon_status_string": (c.c_char_p, [c.c_int]),
        "muon_last_error": (c.c_char_p, [c.c_void_p]),
        "muon_check_orthogonalize": (c.c_int, [P(MuonMatrix), P(MuonMatrix), c.c_int, c.c_int, c.c_char_p, c.c_int]),
        "muon_check_step": (c.c_int, [P(MuonMatrix), P(MuonMatrix), P(MuonMatrix), c.c_int, c.c_char_p, c.c_int]),
        "muon_plan_stats": (c.c_int, [P(c.c_int64), P(c.c_int64), c.c_int, c.c_int, P(c.c_int), P(c.c_int64),
                                      P(c.c_int64), P(c.c_double)]),
        "muon_profile_enable": (c.c_int, [c.c_void_p, c.c_int]),
        "muon_profile_read": (c.c_int, [c.c_void_p, P(c.c_double), P(c.c_int64)]),
        "muon_profile_clock": (c.c_int, [c.c_void_p, P(c.c_double)]),
        "muon_kernel_name": (c.c_char_p, [c.c_int]),
        "muon_selftest_wait": (c.c_int, [c.c_void_p, c.c_int64, c.c_void_p]),
        "muon_selftest_persistent": (c.c_int, [c.c_void_p, c.c_int64, c.c_void_p]),
        "muon_set_workspace_limit": (c.c_int, [c.c_void_p, c.c_int64]),
        "muon_launch_choice": (c.c_int, [P(c.c_int64), P(c.c_int64), c.c_int, c.c_int, c.c_int, c.c_int,
                                         P(c.c_int), P(c.c_double)]),
        "muon_persistent_schedule": (c.c_int, [P(c.c_int64), P(c.c_int64), c.c_int, c.c_int, c.c_int, c.c_int,
                                               P(c.c_int32), c.c_int64, P(c.c_int32), P(c.c_int64)]),
        "muon_shard_layout": (c.c_int, [P(c.c_int64), P(c.c_int64), c.c_int, c.c_int, c.c_int, c.c_int64,
                                        P(c.c_int), P(c.c_int64), P(c.c_int64), P(c.c_double)]),
        "muon_workspace_bytes": (c.c_int, [c.c_void_p, P(c.c_int64)]),
        "muon_normalize_noalloc": (c.c_int, [P(MuonMatrix), P(MuonMatrix), c.c_int, c.c_float, c.c_void_p,
                                             c.c_char_p, c.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().muon_status_string(status).decode()
    except ImportError:
        return f"status {status}"


def kernel_name(kind: int) -> str:
    return load_library().muon_kernel_name(kind).decode()


# ----------------------------------------------------------------------------- descriptors

def describe(t) -> MuonMatrix:
    """muon_matrix for a 2-D CUDA tensor (float32 or bfloat16, unit column stride)."""
    import torch
    if t.dim() != 2:
        raise ValueError(f"expected a 2-D tensor, got shape {tuple(t.shape)}")
    if t.dtype == torch.float32:
        dt = MUON_F32
    elif t.dtype == torch.bfloat16:
        dt = MUON_BF16
    else:
        raise ValueError(f"unsupported dtype {t.dtype}")
    rows, cols = t.shape
    if rows > 0 and cols > 1 and t.stride(1) != 1:
        raise ValueError("the column stride must be 1 (row-major)")
    ld = t.stride(0) if rows > 1 else max(cols, 1)
    return MuonMatrix(ctypes.c_void_p(t.data_ptr()), rows, cols, max(ld, cols), dt)


def matrix_array(items: Sequence) -> ctypes.Array:
    arr = (MuonMatrix * max(1, len(items)))()
    for i, m in enumerate(items):
        arr[i] = m if isinstance(m, MuonMatrix) else describe(m)
    return arr


def check_orthogonalize(inputs: Sequence, outputs: Sequence, steps: int):
    """Host-only argument check (no GPU). Returns (status, message)."""
    lib = load_library()
    msg = ctypes.create_string_buffer(256)
    st = lib.muon_check_orthogonalize(matrix_array(inputs), matrix_array(outputs), len(inputs), steps, msg, 256)
    return st, msg.value.decode()


def check_step(params: Sequence, grads: Sequence, momentum: Sequence):
    lib = load_library()
    msg = ctypes.create_string_buffer(256)
    st = lib.muon_check_step(matrix_array(params), matrix_array(grads), matrix_array(momentum), len(params), msg,
                             256)
    return st, msg.value.decode()


def plan_stats(shapes: Sequence, with_c: bool = False) -> dict:
    """Groups, tile counts and algorithmic flops per Newton-Schulz iteration (host only)."""
    lib = load_library()
    n = len(shapes)
    rows = (ctypes.c_int64 * max(1, n))(*[int(r) for r, _ in shapes])
    cols = (ctypes.c_int64 * max(1, n))(*[int(c) for _, c in shapes])
    g = ctypes.c_int()
    gt = ctypes.c_int64()
    ct = ctypes.c_int64()
    fl = ctypes.c_double()
    st = lib.muon_plan_stats(rows, cols, n, int(with_c), ctypes.byref(g), ctypes.byref(gt), ctypes.byref(ct),
                             ctypes.byref(fl))
    if st != MUON_OK:
        raise MuonError(st, "muon_plan_stats")
    return {"groups": g.value, "gram_tiles": gt.value, "combine_tiles": ct.value, "flops_per_iter": fl.value}


def launch_choice(shapes: Sequence, with_c: bool = False, clusters: int = 74, persistent: Optional[bool] = None):
    """(uses the persistent launch, k-blocks of one iteration per cluster) for a handle whose
    `persistent` option is given (None: the library default, chosen per call). Host only."""
    lib = load_library()
    n = len(shapes)
    rows = (ctypes.c_int64 * max(1, n))(*[int(r) for r, _ in shapes])
    cols = (ctypes.c_int64 * max(1, n))(*[int(c) for _, c in shapes])
    mode = MUON_PERSISTENT_AUTO if persistent is None else int(bool(persistent))
    use, kb = ctypes.c_int(), ctypes.c_double()
    st = lib.muon_launch_choice(rows, cols, n, int(bool(with_c)), int(clusters), mode, ctypes.byref(use),
                                ctypes.byref(kb))
    if st != MUON_OK:
        raise MuonError(st, "muon_launch_choice")
    return bool(use.value), kb.value


def persistent_schedule(shapes: Sequence, steps: int, with_c: bool = False, clusters: int = 74):
    """(items, begin) of the persistent launch's work lists (host only): items as an N x 4 list of
    [kind | group << 2 | flags << 12, matrix in group, row | col << 16, counter target]."""
    lib = load_library()
    n = len(shapes)
    rows = (ctypes.c_int64 * max(1, n))(*[int(r) for r, _ in shapes])
    cols = (ctypes.c_int64 * max(1, n))(*[int(c) for _, c in shapes])
    cnt = ctypes.c_int64()
    st = lib.muon_persistent_schedule(rows, cols, n, int(steps), int(bool(with_c)), int(clusters), None, 0, None,
                                      ctypes.byref(cnt))
    if st != MUON_OK:
        raise MuonError(st, "muon_persistent_schedule")
    items = (ctypes.c_int32 * max(4, 4 * cnt.value))()
    begin = (ctypes.c_int32 * (clusters + 1))()
    st = lib.muon_persistent_schedule(rows, cols, n, int(steps), int(bool(with_c)), int(clusters), items,
                                      cnt.value, begin, ctypes.byref(cnt))
    if st != MUON_OK:
        raise MuonError(st, "muon_persistent_schedule")
    flat = list(items[:4 * cnt.value])
    return [flat[4 * i:4 * i + 4] for i in range(cnt.value)], list(begin)


def _stream_ptr(stream, device) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def normalize_noalloc(inputs: Sequence, outputs: Sequence, eps: float = 1e-7, stream=None):
    """out[j] = in[j] / (||in[j]||_F + eps) without any device allocation (muon_normalize_noalloc).

    For callers that cannot allocate device memory. Runs on the current CUDA
    device; the library keeps its small scratch in a static device array, so
    calls that overlap on the GPU must not be issued.
    """
    import torch
    lib = load_library()
    msg = ctypes.create_string_buffer(256)
    st = lib.muon_normalize_noalloc(matrix_array(inputs), matrix_array(outputs), len(inputs), eps,
                                    _stream_ptr(stream, torch.cuda.current_device()), msg, 256)
    if st != MUON_OK:
        raise MuonError(st, "muon_normalize_noalloc: " + msg.value.decode())
    return outputs


class Muon:
    """A libmuon handle on one CUDA device."""

    def __init__(self, device: int = 0, steps: int = 5, a: float = 1.5, b: float = -0.5, c: float = 0.0,
                 eps: float = 1e-7, scale_lr_by_shape: bool = True, weight_decay: float = 0.0,
                 precise_carry: Optional[bool] = None, persistent: Optional[bool] = None):
        self.lib = load_library()
        self.device = device
        # precise_carry: True always, False never, None (the library default) for calls with c != 0
        carry = MUON_CARRY_WHEN_C if precise_carry is None else int(bool(precise_carry))
        # persistent: True the persistent launch, False one launch per phase, None (the library default)
        # chosen per call by the work per cluster
        mode = MUON_PERSISTENT_AUTO if persistent is None else int(bool(persistent))
        self.config = MuonConfig(steps, a, b, c, eps, int(bool(scale_lr_by_shape)), weight_decay, carry, mode)
        h = ctypes.c_void_p()
        st = self.lib.muon_create(ctypes.byref(h), device, ctypes.byref(self.config))
        if st != MUON_OK:
            raise MuonError(st, f"muon_create(device={device})")
        self.handle = h

    def _check(self, st: int, what: str):
        if st != MUON_OK:
            raise MuonError(st, f"{what}: {self.lib.muon_last_error(self.handle).decode()}")

    def orthogonalize(self, inputs: Sequence, outputs: Sequence, steps: Optional[int] = None,
                      coeffs: Optional[Sequence[float]] = None, stream=None):
        """out[j] = NS_k(in[j]); inputs and outputs are tensors or MuonMatrix descriptors."""
        steps = self.config.steps if steps is None else steps
        a, b, c = (self.config.a, self.config.b, self.config.c) if coeffs is None else coeffs
        st = self.lib.muon_orthogonalize(self.handle, matrix_array(inputs), matrix_array(outputs), len(inputs),
                                         int(steps), a, b, c, _stream_ptr(stream, self.device))
        self._check(st, "muon_orthogonalize")
        return outputs

    def step(self, params: Sequence, grads: Sequence, momentum: Sequence, lr: float, beta: float = 0.95,
             nesterov: bool = True, stream=None):
        """One Muon step: momentum update, Newton-Schulz orthogonalisation and the scaled weight update."""
        st = self.lib.muon_step(self.handle, matrix_array(params), matrix_array(grads), matrix_array(momentum),
                                len(params), lr, beta, int(bool(nesterov)), _stream_ptr(stream, self.device))
        self._check(st, "muon_step")

    def prepare_step(self, params: Sequence, grads: Sequence, momentum: Sequence, lr: float, beta: float = 0.95,
                     nesterov: bool = True, stream=None):
        """Builds the descriptor arrays once and returns a callable that issues this muon_step.

        For loops that step the same tensors every iteration: the per-call cost is
        then one ctypes call. The tensors must stay alive and in place.
        """
        P, G, M = matrix_array(params), matrix_array(grads), matrix_array(momentum)
        n, s = len(params), _stream_ptr(stream, self.device)
        fn, h = self.lib.muon_step, self.handle

        def call():
            st = fn(h, P, G, M, n, lr, beta, int(bool(nesterov)), s)
            if st != MUON_OK:
                self._check(st, "muon_step")
        return call

    def prepare_orthogonalize(self, inputs: Sequence, outputs: Sequence, steps: Optional[int] = None,
                              coeffs: Optional[Sequence[float]] = None, stream=None):
        """Like prepare_step, for muon_orthogonalize."""
        steps = self.config.steps if steps is None else steps
        a, b, c = (self.config.a, self.config.b, self.config.c) if coeffs is None else coeffs
        I, O = matrix_array(inputs), matrix_array(outputs)
        n, s = len(inputs), _stream_ptr(stream, self.device)
        fn, h = self.lib.muon_orthogonalize, self.handle

        def call():
            st = fn(h, I, O, n, int(steps), a, b, c, s)
            if st != MUON_OK:
                self._check(st, "muon_orthogonalize")
        return call

    def selftest_wait(self, limit_ns: int = 50_000_000, stream=None):
        """Queues the failure-detection self-test (a bounded wait that must expire)."""
        self._check(self.lib.muon_selftest_wait(self.handle, int(limit_ns), _stream_ptr(stream, self.device)),
                    "muon_selftest_wait")

    def set_workspace_limit(self, nbytes: int):
        """Caps the device memory of this handle's plans (0: no cap); see muon_set_workspace_limit."""
        self._check(self.lib.muon_set_workspace_limit(self.handle, int(nbytes)), "muon_set_workspace_limit")

    def workspace_bytes(self) -> int:
        """Device memory the handle's plans hold now."""
        v = ctypes.c_int64()
        self._check(self.lib.muon_workspace_bytes(self.handle, ctypes.byref(v)), "muon_workspace_bytes")
        return v.value

    def selftest_persistent(self, limit_ns: int = 50_000_000, stream=None):
        """Runs the persistent launch's failure-detection self-test (a stage wait that must expire)."""
        self._check(self.lib.muon_selftest_persistent(self.handle, int(limit_ns), _stream_ptr(stream, self.device)),
                    "muon_selftest_persistent")

    def get_error(self, stream=None) -> int:
        return self.lib.muon_get_error(self.handle, _stream_ptr(stream, self.device))

    def profile(self, enable: bool = True):
        self._check(self.lib.muon_profile_enable(self.handle, int(enable)), "muon_profile_enable")

    def profile_read(self) -> dict:
        """{kernel name: (total ms, launches)} since the last read."""
        ms = (ctypes.c_double * KERNEL_KINDS)()
        n = (ctypes.c_int64 * KERNEL_KINDS)()
        self._check(self.lib.muon_profile_read(self.handle, ms, n), "muon_profile_read")
        return {kernel_name(k): (ms[k], n[k]) for k in range(KERNEL_KINDS)}

    def profile_clock(self) -> float:
        """MHz of the SM clock under the GEMM kernels profiled since profiling was turned on."""
        v = ctypes.c_double()
        self._check(self.lib.muon_profile_clock(self.handle, ctypes.byref(v)), "muon_profile_clock")
        return v.value

    def close(self):
        if getattr(self, "handle", None):
            self.lib.muon_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
