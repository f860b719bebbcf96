"""GB300-native (sm_103a) gated delta rule: chunkwise forward and backward, KDA, and the decode step.

The computation lives in libgdn_gb300.so (C ABI, include/gdn.h): hand-written
CUDA kernels for sm_103a.  This package is its thin Python binding; torch
supplies device memory and streams.  Build the library with
``gated_delta_rule_gdn_gb300.build.build()``; the calls raise if it is
missing.
"""
from ._binding import (GdnError, bwd_workspace_size, chunk_bwd, chunk_fwd_noalloc, gdn_chunk_bwd, kda_chunk_bwd, chunk_plan, device_status, gdn_chunk_fwd, gdn_recurrent_step, kda_chunk_fwd, kda_recurrent_step, last_error,
                       lib_path, load, workspace_size)

__all__ = ["gdn_chunk_fwd", "kda_chunk_fwd", "gdn_recurrent_step", "kda_recurrent_step", "device_status", "chunk_plan", "last_error", "load",
           "lib_path", "GdnError", "workspace_size", "chunk_fwd_noalloc",
           "chunk_bwd", "gdn_chunk_bwd", "kda_chunk_bwd", "bwd_workspace_size"]
