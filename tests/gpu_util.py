"""Helpers for the GPU parity tests: run the library, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kimi_delta_attention_10_gb300 import kda_chunk_fwd, kda_gate
from kimi_delta_attention_10_gb300.inputs import KDAInputs

# Output tolerances (rel-L2 against the FP64 oracle), per mode.
TOL = {"fp32_exact": 1e-5, "bf16_tc": 3e-3}

# The library's chunk paths: (mode, workspace).  With a workspace each mode
# runs in two phases (prepare every chunk, then scan); without one, in its
# single-pass kernel.
PATHS = {"fp32_exact": ("fp32_exact", None), "fp32_exact_2p": ("fp32_exact", "auto"),
         "bf16_tc": ("bf16_tc", "auto"), "bf16_tc_1pass": ("bf16_tc", None)}
OUT_DTYPE = {"fp32_exact": torch.float32, "fp32_exact_2p": torch.float32, "bf16_tc": None,
             "bf16_tc_1pass": None}


def path_kw(path: str) -> dict:
    mode, ws = PATHS[path]
    return dict(mode=mode, workspace=ws)


def tol(path: str) -> float:
    return TOL[PATHS[path][0]]


def device_inputs(x: KDAInputs, device="cuda"):
    return {name: getattr(x, name).to(device) for name in
            ("q", "k", "v", "f", "A_log", "dt_bias", "b", "cu_seqlens")}


def gpu_pipeline(x: KDAInputs, path: str, out_dtype=None, host_mirror=True):
    """kda_gate then kda_chunk_fwd on the GPU; CPU copies of (out, final_state, g, beta)."""
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    out, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           out_dtype=out_dtype,
                           cu_seqlens_host=x.cu_seqlens.tolist() if host_mirror else None,
                           **path_kw(path))
    torch.cuda.synchronize()
    return out.cpu(), S.cpu(), g.cpu(), beta.cpu()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.float().numpy().astype(np.float64)


def oracle_pipeline(x: KDAInputs, heads=None):
    """FP64 gate + recurrence from the raw draws, for all heads or a subset."""
    sel = slice(None) if heads is None else list(heads)
    o, S, g, beta = oracle.reference(
        f64(x.q[:, sel]), f64(x.k[:, sel]), f64(x.v[:, sel]), f64(x.f[:, sel]),
        f64(x.A_log[sel]), f64(x.dt_bias[sel]), f64(x.b[:, sel]), x.cu_seqlens.numpy(),
        x.scale)
    return o, S, g, beta


def rel_l2(x, ref) -> float:
    return oracle.rel_l2(np.asarray(x, np.float64), ref)
