"""Bounded-decay chunked linear attention for GB300 (sm_103a).

The compute lives in libbdla.so (C ABI declared in include/bdla.h); this
package holds the CUDA sources (csrc/), their build script, a thin ctypes
binding and the seeded synthetic input generator.
"""
from .bdla import (BOUNDED, CHUNK, SOFTPLUS, BdlaError, Workspace, bwd, bwd_vec, decay,  # noqa: F401
                   bwd_delta, decode, fwd, fwd_delta, fwd_vec, lib, n_slots, tile_states,
                   workspace_bytes)

__all__ = ["BOUNDED", "SOFTPLUS", "CHUNK", "BdlaError", "Workspace", "fwd", "bwd", "fwd_vec", "bwd_vec",
           "fwd_delta", "bwd_delta", "tile_states",
           "decay", "decode", "lib", "n_slots", "workspace_bytes"]
