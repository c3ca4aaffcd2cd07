"""muon_normalize_noalloc: the normalisation for callers that cannot allocate device memory (GPU).

The entry point keeps its scratch in a static device array inside the library
instead of a workspace it would have to cudaMalloc. Its output is compared with
the existing path that computes the same thing, muon_orthogonalize with zero
Newton-Schulz steps (X0 = in / (||in||_F + eps)), on two calls in a row, so the
second call runs on scratch the first one left behind. This file sorts last so
that a stop at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import TOL, dev, host, rel_f

pytestmark = pytest.mark.gpu


def _batch(shapes, dtype, seed):
    w = wl.small_workload("noalloc", shapes, dtype=dtype, grad_std=1.0, seed=seed)
    return [dev(wl.gradient(w, j), dtype) for j in range(w.count)]


def _existing(muon, ins):
    outs = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in ins]
    muon.orthogonalize(ins, outs, steps=0)
    return outs


def test_noalloc_matches_existing_entry_point_twice():
    from muon_newton_schulz_09_b300 import Muon, normalize_noalloc
    calls = [
        (_batch([(128, 256), (256, 128), (130, 70), (1, 5), (513, 1000)], "bf16", seed=41), torch.float32),
        (_batch([(768, 3072), (64, 200), (3, 3)], "f32", seed=42), torch.bfloat16),
    ]
    with Muon(0) as muon:
        for ins, out_dtype in calls:
            outs = [torch.full(t.shape, 7.0, dtype=out_dtype, device="cuda") for t in ins]
            normalize_noalloc(ins, outs)
            ref = _existing(muon, ins)
            torch.cuda.synchronize()
            assert muon.get_error() == 0
            for o, r in zip(outs, ref):
                e = rel_f(host(o), host(r))
                assert e < TOL, (tuple(o.shape), e)
                assert np.isfinite(host(o)).all()


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
