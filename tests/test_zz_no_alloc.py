"""muon_normalize_noalloc: the normalisation for callers that cannot allocate device memory (GPU).

The entry point keeps its scratch in a static device array inside the library
instead of a workspace it would have to cudaMalloc. Its output is compared on
two calls in a row (the second runs on the scratch the first left behind) with:

  * the existing path that computes the same thing, muon_orthogonalize with
    zero Newton-Schulz steps, X0 = in / (||in||_F + eps). Both reduce the norm
    with the same kernel, so bf16 outputs agree to one bf16 ulp per element.
    For fp32 outputs the existing path holds X0 in its bf16 workspace, so the
    two agree to half a bf16 ulp per element (the existing value is the fp32
    one rounded);
  * the fp64 oracle's normalisation: to fp32 rounding (rel-F 1e-6) for fp32
    outputs and to bf16 rounding (rel-F 4e-3) for bf16 outputs, including an
    input whose row stride is not its width.

This file sorts last so that a stop at the first failure has already run every
other test.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import bf16_ulp, dev, host, rel_f

pytestmark = pytest.mark.gpu

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _batch(shapes, dtype, seed, pad_first=0):
    """Seeded inputs on the GPU; the first one (when pad_first > 0) sits in a wider buffer (ld != cols)."""
    w = wl.small_workload("noalloc", shapes, dtype=dtype, grad_std=1.0, seed=seed)
    xs = [wl.gradient(w, j) for j in range(w.count)]
    ts = [dev(x, dtype) for x in xs]
    if pad_first:
        r, c = shapes[0]
        wide = torch.zeros(r, c + pad_first, dtype=TORCH_DT[dtype], device="cuda")
        wide[:, :c].copy_(ts[0])
        ts[0] = wide[:, :c]
    return xs, ts


def _existing(muon, ins, out_dtype):
    outs = [torch.empty(t.shape, dtype=TORCH_DT[out_dtype], device="cuda") for t in ins]
    muon.orthogonalize(ins, outs, steps=0)
    return outs


CALLS = [
    # (shapes, input dtype, output dtype, seed, padding of the first input's rows)
    ([(130, 70), (128, 256), (256, 128), (1, 5), (513, 1000)], "bf16", "f32", 41, 6),
    ([(768, 3072), (64, 200), (3, 3), (200, 64)], "f32", "bf16", 42, 0),
]


def test_noalloc_matches_existing_entry_point_and_oracle_twice():
    from muon_newton_schulz_09_b300 import Muon, normalize_noalloc
    with Muon(0) as muon:
        for shapes, in_dt, out_dt, seed, pad in CALLS:
            xs, ins = _batch(shapes, in_dt, seed, pad)
            outs = [torch.full(t.shape, 7.0, dtype=TORCH_DT[out_dt], device="cuda") for t in ins]
            normalize_noalloc(ins, outs)
            ref = _existing(muon, ins, out_dt)
            torch.cuda.synchronize()
            assert muon.get_error() == 0
            for x, o, r in zip(xs, outs, ref):
                got, other = host(o), host(r)
                want = oracle.frobenius_normalize(x)
                assert np.isfinite(got).all()
                diff = np.abs(got - other)
                if out_dt == "bf16":
                    assert np.all(diff <= bf16_ulp(other)), (x.shape, float(diff.max()))
                    assert rel_f(got, want) < 4e-3, (x.shape, rel_f(got, want))
                else:
                    assert np.all(diff <= 0.5 * bf16_ulp(got) + 1e-7 * np.abs(got)), (x.shape, float(diff.max()))
                    assert rel_f(got, want) < 1e-6, (x.shape, rel_f(got, want))


def test_noalloc_rejects_sizes_beyond_its_limit():
    from muon_newton_schulz_09_b300 import MUON_ERR_INVALID, MuonError, MuonMatrix, normalize_noalloc
    import muon_newton_schulz_09_b300 as mu
    x = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    too_many = [x] * 129
    with pytest.raises(MuonError) as e:
        normalize_noalloc(too_many, [torch.empty(8, 8, device="cuda") for _ in too_many])
    assert e.value.status == MUON_ERR_INVALID and "MATRICES" in str(e.value)
    # 2^26 + 1 elements: the descriptor is checked on the host before anything touches the pointer
    big = MuonMatrix(x.data_ptr(), 8193, 8192, 8192, mu.MUON_BF16)
    big_out = MuonMatrix(x.data_ptr() + (1 << 30), 8193, 8192, 8192, mu.MUON_F32)
    with pytest.raises(MuonError) as e:
        normalize_noalloc([big], [big_out])
    assert e.value.status == MUON_ERR_INVALID and "MUON_NOALLOC_MAX_ELEMENTS" in str(e.value)
