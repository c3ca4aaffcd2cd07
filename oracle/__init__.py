"""fp64 CPU oracle of the Muon step. TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use it. The CUDA library does not.
"""
from .muon_oracle import (DEFAULT_COEFFS, DEFAULT_EPS, frobenius_normalize, lr_scale, momentum,
                          muon_step, muon_update, newton_schulz, orthogonalize, rel_frobenius)

__all__ = ["DEFAULT_COEFFS", "DEFAULT_EPS", "frobenius_normalize", "lr_scale", "momentum", "muon_step",
           "muon_update", "newton_schulz", "orthogonalize", "rel_frobenius"]
