"""GB300 (sm_103a) chunked Kimi Delta Attention forward and backward.

The compute path is libkda_gb300.so (C ABI in include/kda.h), reached through
``kda_gate``, ``kda_chunk_fwd``, ``kda_chunk_fwd_gated`` and
``kda_recurrent_step`` (``chunk_workspace_size`` sizes the two-phase path's
scratch; ``kda_chunk_fwd_static`` runs it on the library's own scratch),
``kda_gated_rmsnorm`` (the output gate; ``kda_chunk_fwd_gated_norm`` fuses it
into the forward) and ``kda_chunk_bwd`` (the VJP,
scratch sized by ``chunk_bwd_workspace_size``);
``inputs`` holds the seeded synthetic workloads.
"""
from .binding import (KDAError, chunk_bwd_workspace_size, chunk_workspace_size,  # noqa: F401
                      kda_chunk_bwd, kda_chunk_fwd, kda_chunk_fwd_gated, kda_chunk_fwd_gated_norm,
                      kda_chunk_fwd_static,
                      kda_gate, kda_gated_rmsnorm, kda_recurrent_step, library_path, load_library,
                      status_string)
