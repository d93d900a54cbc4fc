"""FP64 CPU oracle of the KDA forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library in
``kimi_delta_attention_10_gb300`` and never imports it; the CUDA path never
imports this package.

Contents
  * ``gate`` / ``forward``: the compiled C token-by-token FP64 oracle
    (``kda_oracle.c``), threaded over (sequence, head) units.
  * ``forward_matrix_numpy``: a NumPy restatement of the recurrence in its
    matrix form S_t = (I - beta_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + beta_t
    k_t v_t^T, for tiny shapes.
  * ``chunked`` (submodule): the FP64 chunked (WY) form, a different
    algorithm for the same result.
  * ``exact_scalar`` (submodule): exact rational evaluation of the K = V = 1
    case by its explicit-sum closed form.
  * ``output_gate`` (submodule): the output gate with gated RMSNorm applied to
    the attention output, in float64.
  * ``backward`` (submodule): the vector-Jacobian product of the recurrence
    (dq, dk, dv, dg, dbeta, dS_0 from dO and dS_T), token by token in float64.

Pages followed: XTuner "Add opt-in FP32 KDA chunk computation" (sections
Problem, Change, Validation: an independent FP64 recurrence is the
reference; Q/K are L2-normalised inside the op) and "GLM-5.3-Flash F6.2: KDA
correctness and FLA sequence parallelism" (the fused-gate commit: the gate
-exp(A_log) * softplus(f + dt_bias) with FP32 A_log/dt_bias is computed
outside the kernel; beta is a sigmoid of its logits).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

# Planted-mistake switches understood by kda_oracle.c (tests only).
MUTATIONS = {
    "none": 0, "no_erase": 1, "decay_after": 2, "read_before": 3, "transposed_read": 4,
    "no_l2norm": 5, "beta_on_v_only": 6, "gate_no_alog": 7, "gate_bias_head0": 8,
    "skip_scale": 9, "ignore_init": 10,
}

L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, IEEE arithmetic)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lm", "-lpthread"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            d = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.kda_oracle_gate.argtypes = [d, d, d, d, ctypes.c_int64, ctypes.c_int32,
                                            ctypes.c_int32, d, d, ctypes.c_int32]
            lib.kda_oracle_gate.restype = None
            lib.kda_oracle_forward.argtypes = [
                d, d, d, d, d, i32p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_int32,
                ctypes.c_double, d, d, d, ctypes.c_int32, ctypes.c_int32]
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_default_threads.restype = ctypes.c_int32
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return int(_load().kda_oracle_default_threads())


def gate(f, A_log, dt_bias, b, mutation: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """g = -exp(A_log[h]) * softplus(f + dt_bias[h, c]) and beta = sigmoid(b), FP64.

    f: [T,H,K], A_log: [H], dt_bias: [H,K], b: [T,H]."""
    f = _f64(f); A_log = _f64(A_log); dt_bias = _f64(dt_bias); b = _f64(b)
    T, H, K = f.shape
    assert A_log.shape == (H,) and dt_bias.shape == (H, K) and b.shape == (T, H)
    g = np.empty((T, H, K), np.float64)
    beta = np.empty((T, H), np.float64)
    _load().kda_oracle_gate(_ptr(f), _ptr(A_log), _ptr(dt_bias), _ptr(b), T, H, K,
                            _ptr(g), _ptr(beta), int(mutation))
    return g, beta


def forward(q, k, v, g, beta, cu_seqlens, scale: float, l2norm: bool = True,
            eps: float = L2_EPS, final_state: bool = True, nthreads: int = 0,
            mutation: int = 0, initial_state=None) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """Token-by-token FP64 KDA forward.

    q, k: [T,H,K]; v: [T,H,V]; g: [T,H,K]; beta: [T,H]; cu_seqlens: [N+1];
    initial_state: [N,H,K,V] or None (zero).
    Returns o [T,H,V] and final_state [N,H,K,V] (or None)."""
    q = _f64(q); k = _f64(k); v = _f64(v); g = _f64(g); beta = _f64(beta)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, H, K = q.shape
    V = v.shape[2]
    N = cu.shape[0] - 1
    assert k.shape == (T, H, K) and g.shape == (T, H, K) and v.shape[:2] == (T, H)
    assert beta.shape == (T, H)
    o = np.zeros((T, H, V), np.float64)
    S = np.zeros((N, H, K, V), np.float64) if final_state else None
    init = None
    if initial_state is not None:
        init = _f64(initial_state)
        assert init.shape == (N, H, K, V)
    rc = _load().kda_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), N, T, H, K, V, float(scale),
        1 if l2norm else 0, float(eps),
        _ptr(init) if init is not None else ctypes.POINTER(ctypes.c_double)(), _ptr(o),
        _ptr(S) if S is not None else ctypes.POINTER(ctypes.c_double)(),
        int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError("kda_oracle_forward rejected its arguments")
    return o, S


def reference(q, k, v, f, A_log, dt_bias, b, cu_seqlens, scale: float,
              nthreads: int = 0, mutation: int = 0, initial_state=None):
    """The whole path from raw draws: FP64 gate, then the FP64 forward.

    Returns (o, final_state, g, beta)."""
    g, beta = gate(f, A_log, dt_bias, b, mutation=mutation)
    o, S = forward(q, k, v, g, beta, cu_seqlens, scale, nthreads=nthreads,
                   mutation=mutation, initial_state=initial_state)
    return o, S, g, beta


def forward_matrix_numpy(q, k, v, g, beta, cu_seqlens, scale: float, l2norm: bool = True,
                         eps: float = L2_EPS):
    """The recurrence in its matrix form, one token at a time (tiny shapes only).

    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t, with q, k L2-normalised first."""
    q = _f64(q); k = _f64(k); v = _f64(v); g = _f64(g); beta = _f64(beta)
    T, H, K = q.shape
    V = v.shape[2]
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    o = np.zeros((T, H, V))
    S_all = np.zeros((len(cu) - 1, H, K, V))
    I = np.eye(K)
    for n in range(len(cu) - 1):
        for h in range(H):
            S = np.zeros((K, V))
            for t in range(cu[n], cu[n + 1]):
                qt, kt = q[t, h], k[t, h]
                if l2norm:
                    qt = qt / np.sqrt(qt @ qt + eps)
                    kt = kt / np.sqrt(kt @ kt + eps)
                S = (I - beta[t, h] * np.outer(kt, kt)) @ np.diag(np.exp(g[t, h])) @ S \
                    + beta[t, h] * np.outer(kt, v[t, h])
                o[t, h] = scale * (S.T @ qt)
            S_all[n, h] = S
    return o, S_all


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 in FP64 (0 when both are zero)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    num = float(np.linalg.norm((x - ref).ravel()))
    den = float(np.linalg.norm(ref.ravel()))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
