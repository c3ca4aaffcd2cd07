"""Muon optimizer step for one B300 (sm_103a): C-ABI CUDA library + thin binding.

The library (lib/libmuon.so, built from csrc/ by ``build.py``) computes the
Muon step: momentum, Frobenius normalisation, Newton-Schulz orthogonalisation
on the tensor cores (tcgen05/TMEM/TMA) and the scaled weight update. This
package only marshals arguments to it.
"""
from .binding import (KERNEL_KINDS, MUON_BF16, MUON_ERR_CUDA, MUON_ERR_INVALID, MUON_ERR_NOMEM,
                      MUON_ERR_TIMEOUT, MUON_ERR_UNSUPPORTED, MUON_F32, MUON_OK, Muon, MuonConfig, MuonError,
                      MuonMatrix, check_orthogonalize, check_step, describe, header_functions, kernel_name,
                      launch_choice, load_library, normalize_noalloc, persistent_schedule, plan_stats,
                      status_string)
from .sharded import ShardedMuon, ShardLayout, shard_layout, sharded_step

__all__ = ["KERNEL_KINDS", "MUON_BF16", "MUON_ERR_CUDA", "MUON_ERR_INVALID", "MUON_ERR_NOMEM", "MUON_ERR_TIMEOUT",
           "MUON_ERR_UNSUPPORTED", "MUON_F32", "MUON_OK", "Muon", "MuonConfig", "MuonError", "MuonMatrix",
           "check_orthogonalize", "check_step", "describe", "header_functions", "kernel_name", "launch_choice",
           "load_library",
           "normalize_noalloc", "persistent_schedule", "plan_stats", "status_string", "ShardedMuon", "ShardLayout", "shard_layout",
           "sharded_step"]
