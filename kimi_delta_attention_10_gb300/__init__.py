"""GB300 (sm_103a) chunked Kimi Delta Attention forward.

The compute path is libkda_gb300.so (C ABI in include/kda.h), reached through
``kda_gate`` and ``kda_chunk_fwd``; ``inputs`` holds the seeded synthetic
workloads.
"""
from .binding import (KDAError, kda_chunk_fwd, kda_gate, library_path,  # noqa: F401
                      load_library, status_string)
