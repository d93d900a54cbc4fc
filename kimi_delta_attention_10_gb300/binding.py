"""ctypes binding of libkda_gb300.so (include/kda.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; PyTorch provides the
device memory and the stream.  There is no fallback: if the library is
missing, or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

import torch

from . import _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_ALIGNMENT = 3
KDA_ERR_CUDA = 4
KDA_ERR_TIMEOUT = 5
KDA_ERR_DEVICE_ARG = 6
KDA_ERR_TOO_LARGE = 7
KDA_ERR_RANGE = 8

# kda_test_set_fault values (test hook)
KDA_TEST_FAULT_NONE = 0
KDA_TEST_FAULT_SCAN = 1
KDA_TEST_FAULT_PREP = 2
KDA_TEST_FAULT_SINGLE_PASS = 3

KDA_F32 = 0
KDA_BF16 = 1

KDA_MODE_BF16_TC = 0
KDA_MODE_FP32_EXACT = 1

MODES = {"bf16_tc": KDA_MODE_BF16_TC, "fp32_exact": KDA_MODE_FP32_EXACT}

# Every symbol include/kda.h declares.
EXPORTS = ("kda_gate", "kda_chunk_workspace_size", "kda_chunk_fwd", "kda_chunk_fwd_gated",
           "kda_chunk_fwd_gated_norm",
           "kda_chunk_fwd_static", "kda_recurrent_step", "kda_gated_rmsnorm",
           "kda_chunk_bwd_workspace_size", "kda_chunk_bwd", "kda_test_set_fault",
           "kda_status_string", "kda_abi_version")

_lock = threading.Lock()
_lib = None


class KDAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libkda_gb300.so (optionally building it first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"{path} is missing: build it with kimi_delta_attention_10_gb300._build.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.kda_gate.argtypes = [vp, i32, vp, vp, vp, i32, i64, i32, i32, vp, vp, vp]
        lib.kda_gate.restype = i32
        lib.kda_chunk_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32,
                                                 ctypes.POINTER(i64)]
        lib.kda_chunk_workspace_size.restype = i32
        lib.kda_chunk_fwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                      ctypes.c_float, i32, i32, vp, i32, vp, vp, vp, i64, vp, vp]
        lib.kda_chunk_fwd.restype = i32
        lib.kda_chunk_fwd_gated.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, vp, vp,
                                            i32, i64, i32, i32, i32, ctypes.c_float, i32, i32,
                                            vp, i32, vp, vp, vp, i64, vp, vp]
        lib.kda_chunk_fwd_gated.restype = i32
        lib.kda_chunk_fwd_gated_norm.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, vp,
                                                 vp, i32, i64, i32, i32, i32, ctypes.c_float, i32,
                                                 i32, vp, i32, vp, ctypes.c_float, vp, i32, vp, vp,
                                                 vp, i64, vp, vp]
        lib.kda_chunk_fwd_gated_norm.restype = i32
        lib.kda_chunk_fwd_static.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i64, i32, i32,
                                             i32, ctypes.c_float, i32, vp, i32, vp, vp, vp, vp]
        lib.kda_chunk_fwd_static.restype = i32
        lib.kda_recurrent_step.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                           ctypes.c_float, i32, vp, vp, i32, vp]
        lib.kda_recurrent_step.restype = i32
        lib.kda_gated_rmsnorm.argtypes = [vp, i32, vp, i32, vp, i64, i32, ctypes.c_float, vp, i32,
                                          vp]
        lib.kda_gated_rmsnorm.restype = i32
        lib.kda_chunk_bwd_workspace_size.argtypes = [i32, i64, i32, i32, i32, ctypes.POINTER(i64)]
        lib.kda_chunk_bwd_workspace_size.restype = i32
        lib.kda_chunk_bwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                      ctypes.c_float, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                      vp, vp, i64, vp, vp]
        lib.kda_chunk_bwd.restype = i32
        lib.kda_test_set_fault.argtypes = [i32]
        lib.kda_test_set_fault.restype = i32
        lib.kda_status_string.argtypes = [i32]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_abi_version.argtypes = []
        lib.kda_abi_version.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().kda_status_string(int(status)).decode()


def set_test_fault(where: int) -> None:
    """Test hook: make CTA 0 of the named kernel lose one arrival so that its
    bounded wait gives up (KDA_TEST_FAULT_*; KDA_TEST_FAULT_NONE turns it off)."""
    st = load_library().kda_test_set_fault(int(where))
    if st != KDA_OK:
        raise KDAError(st, "kda_test_set_fault")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev_ptr(t: Optional[torch.Tensor], name: str) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise RuntimeError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def kda_gate(f: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor, b: torch.Tensor,
             g_out: Optional[torch.Tensor] = None, beta_out: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """g = -exp(A_log[h]) * softplus(f + dt_bias), beta = sigmoid(b) (FP32 outputs)."""
    lib = load_library()
    T, H, K = f.shape
    if g_out is None:
        g_out = torch.empty((T, H, K), dtype=torch.float32, device=f.device)
    if beta_out is None:
        beta_out = torch.empty((T, H), dtype=torch.float32, device=f.device)
    st = lib.kda_gate(_dev_ptr(f, "f"), _dtype_code(f), _dev_ptr(A_log, "A_log"),
                      _dev_ptr(dt_bias, "dt_bias"), _dev_ptr(b, "b"), _dtype_code(b), T, H, K,
                      _dev_ptr(g_out, "g_out"), _dev_ptr(beta_out, "beta_out"),
                      _stream_handle(stream, f.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_gate")
    return g_out, beta_out


def _chunk_outputs(q, v, cu_seqlens, out, out_dtype, output_final_state, final_state):
    T, H, K = q.shape
    V = v.shape[2]
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, H, V), dtype=out_dtype or v.dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, K, V), dtype=torch.float32, device=q.device)
    return out, final_state


def chunk_workspace_size(N: int, T: int, H: int, K: int = 128, V: int = 128,
                         mode: str = "bf16_tc") -> int:
    """Bytes of workspace the mode's two-phase chunk path needs."""
    out = ctypes.c_int64(0)
    st = load_library().kda_chunk_workspace_size(N, T, H, K, V, MODES[mode], ctypes.byref(out))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_workspace_size")
    return out.value


def _workspace(workspace, mode, N, T, H, K, V, device):
    """(pointer, bytes) for the call: None -> no workspace (single-pass
    kernel); "auto" -> a fresh buffer of the size the mode's two-phase path
    needs; a tensor -> its storage."""
    if workspace is None:
        return None, 0, None
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be None, 'auto' or a CUDA tensor")
        workspace = torch.empty(chunk_workspace_size(N, T, H, K, V, mode), dtype=torch.uint8,
                                device=device)
    ptr = _dev_ptr(workspace, "workspace")
    return ptr, workspace.numel() * workspace.element_size(), workspace


def _host_offsets(cu_seqlens_host):
    if cu_seqlens_host is None:
        return None, None
    arr = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def kda_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                  beta: torch.Tensor, cu_seqlens: torch.Tensor, scale: Optional[float] = None,
                  mode: str = "bf16_tc", out: Optional[torch.Tensor] = None,
                  out_dtype: Optional[torch.dtype] = None, output_final_state: bool = True,
                  final_state: Optional[torch.Tensor] = None,
                  initial_state: Optional[torch.Tensor] = None,
                  cu_seqlens_host: Optional[Sequence[int]] = None, qk_l2norm: bool = True,
                  status: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None, workspace="auto"):
    """Chunked KDA forward.  Returns (out [T,H,V], final_state [N,H,K,V] or None).

    workspace: "auto" (bf16_tc allocates the two-phase path's scratch), a CUDA
    tensor of at least chunk_workspace_size(...) bytes, or None (single-pass
    kernel, no scratch)."""
    lib = load_library()
    T, H, K = q.shape
    V = v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    out, final_state = _chunk_outputs(q, v, cu_seqlens, out, out_dtype, output_final_state,
                                      final_state)
    keep, host = _host_offsets(cu_seqlens_host)
    ws, ws_bytes, ws_keep = _workspace(workspace, mode, N, T, H, K, V, q.device)
    st = lib.kda_chunk_fwd(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(q),
        _dev_ptr(g, "g"), _dev_ptr(beta, "beta"), _dev_ptr(cu_seqlens, "cu_seqlens"), host,
        N, T, H, K, V, float(scale), 1 if qk_l2norm else 0, MODES[mode],
        _dev_ptr(out, "out"), _dtype_code(out), _dev_ptr(initial_state, "initial_state"),
        _dev_ptr(final_state, "final_state"), ws, ws_bytes, _dev_ptr(status, "status"),
        _stream_handle(stream, q.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd")
    return out, final_state


def kda_chunk_fwd_gated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, f: torch.Tensor,
                        A_log: torch.Tensor, dt_bias: torch.Tensor, b: torch.Tensor,
                        cu_seqlens: torch.Tensor, scale: Optional[float] = None,
                        mode: str = "bf16_tc", out: Optional[torch.Tensor] = None,
                        out_dtype: Optional[torch.dtype] = None, output_final_state: bool = True,
                        final_state: Optional[torch.Tensor] = None,
                        initial_state: Optional[torch.Tensor] = None,
                        cu_seqlens_host: Optional[Sequence[int]] = None, qk_l2norm: bool = True,
                        status: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None, workspace="auto"):
    """Chunked KDA forward with the gate (g, beta from f, A_log, dt_bias, b) fused in;
    workspace as kda_chunk_fwd."""
    lib = load_library()
    T, H, K = q.shape
    V = v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    out, final_state = _chunk_outputs(q, v, cu_seqlens, out, out_dtype, output_final_state,
                                      final_state)
    keep, host = _host_offsets(cu_seqlens_host)
    ws, ws_bytes, ws_keep = _workspace(workspace, mode, N, T, H, K, V, q.device)
    st = lib.kda_chunk_fwd_gated(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(q),
        _dev_ptr(f, "f"), _dtype_code(f), _dev_ptr(A_log, "A_log"), _dev_ptr(dt_bias, "dt_bias"),
        _dev_ptr(b, "b"), _dtype_code(b), _dev_ptr(cu_seqlens, "cu_seqlens"), host,
        N, T, H, K, V, float(scale), 1 if qk_l2norm else 0, MODES[mode],
        _dev_ptr(out, "out"), _dtype_code(out), _dev_ptr(initial_state, "initial_state"),
        _dev_ptr(final_state, "final_state"), ws, ws_bytes, _dev_ptr(status, "status"),
        _stream_handle(stream, q.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_gated")
    return out, final_state


def kda_chunk_fwd_gated_norm(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, f: torch.Tensor,
                             A_log: torch.Tensor, dt_bias: torch.Tensor, b: torch.Tensor,
                             cu_seqlens: torch.Tensor, z: torch.Tensor, weight: torch.Tensor,
                             scale: Optional[float] = None, eps: float = 1e-6,
                             mode: str = "bf16_tc", out: Optional[torch.Tensor] = None,
                             out_dtype: Optional[torch.dtype] = None,
                             output_final_state: bool = True,
                             final_state: Optional[torch.Tensor] = None,
                             initial_state: Optional[torch.Tensor] = None,
                             cu_seqlens_host: Optional[Sequence[int]] = None,
                             qk_l2norm: bool = True, status: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None, workspace="auto"):
    """kda_chunk_fwd_gated with the output gate and gated RMSNorm applied to its
    output (z [T,H,V] gate pre-activation, weight [V]); returns (y, final_state)."""
    lib = load_library()
    T, H, K = q.shape
    V = v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    out, final_state = _chunk_outputs(q, v, cu_seqlens, out, out_dtype, output_final_state,
                                      final_state)
    keep, host = _host_offsets(cu_seqlens_host)
    ws, ws_bytes, ws_keep = _workspace(workspace, mode, N, T, H, K, V, q.device)
    st = lib.kda_chunk_fwd_gated_norm(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(q),
        _dev_ptr(f, "f"), _dtype_code(f), _dev_ptr(A_log, "A_log"), _dev_ptr(dt_bias, "dt_bias"),
        _dev_ptr(b, "b"), _dtype_code(b), _dev_ptr(cu_seqlens, "cu_seqlens"), host,
        N, T, H, K, V, float(scale), 1 if qk_l2norm else 0, MODES[mode],
        _dev_ptr(z, "z"), _dtype_code(z), _dev_ptr(weight, "weight"), float(eps),
        _dev_ptr(out, "out"), _dtype_code(out), _dev_ptr(initial_state, "initial_state"),
        _dev_ptr(final_state, "final_state"), ws, ws_bytes, _dev_ptr(status, "status"),
        _stream_handle(stream, q.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_gated_norm")
    return out, final_state


def kda_chunk_fwd_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                         beta: torch.Tensor, cu_seqlens: torch.Tensor, out: torch.Tensor,
                         scale: Optional[float] = None,
                         final_state: Optional[torch.Tensor] = None,
                         initial_state: Optional[torch.Tensor] = None,
                         cu_seqlens_host: Optional[Sequence[int]] = None, qk_l2norm: bool = True,
                         status: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """kda_chunk_fwd (bf16_tc, two-phase) on the library's static scratch: allocates
    nothing, so `out` (and `final_state`, if wanted) are the caller's.  Problems
    beyond the 64 MiB scratch raise KDAError(KDA_ERR_TOO_LARGE)."""
    lib = load_library()
    T, H, K = q.shape
    V = v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    keep, host = _host_offsets(cu_seqlens_host)
    st = lib.kda_chunk_fwd_static(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(q),
        _dev_ptr(g, "g"), _dev_ptr(beta, "beta"), _dev_ptr(cu_seqlens, "cu_seqlens"), host,
        N, T, H, K, V, float(scale), 1 if qk_l2norm else 0,
        _dev_ptr(out, "out"), _dtype_code(out), _dev_ptr(initial_state, "initial_state"),
        _dev_ptr(final_state, "final_state"), _dev_ptr(status, "status"),
        _stream_handle(stream, q.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_fwd_static")


def kda_recurrent_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                       beta: torch.Tensor, state: torch.Tensor, scale: Optional[float] = None,
                       out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
                       qk_l2norm: bool = True, stream: Optional[torch.cuda.Stream] = None):
    """One decode token per sequence: q, k [N,H,K], v [N,H,V], g [N,H,K], beta [N,H];
    state [N,H,K,V] FP32 is updated in place.  Returns out [N,H,V]."""
    lib = load_library()
    N, H, K = q.shape
    V = v.shape[2]
    if scale is None:
        scale = K ** -0.5
    if out is None:
        out = torch.empty((N, H, V), dtype=out_dtype or v.dtype, device=q.device)
    st = lib.kda_recurrent_step(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(q),
        _dev_ptr(g, "g"), _dev_ptr(beta, "beta"), N, H, K, V, float(scale),
        1 if qk_l2norm else 0, _dev_ptr(state, "state"), _dev_ptr(out, "out"),
        _dtype_code(out), _stream_handle(stream, q.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_recurrent_step")
    return out


def kda_gated_rmsnorm(o: torch.Tensor, z: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6,
                      out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """y = o / sqrt(mean(o^2) + eps) * weight * sigmoid(z) over the last dim (V = 128);
    o and z of shape [..., V], weight [V] FP32.  Returns y (out if given)."""
    lib = load_library()
    V = o.shape[-1]
    rows = o.numel() // V if V else 0
    if out is None:
        out = torch.empty(o.shape, dtype=out_dtype or o.dtype, device=o.device)
    st = lib.kda_gated_rmsnorm(_dev_ptr(o, "o"), _dtype_code(o), _dev_ptr(z, "z"), _dtype_code(z),
                               _dev_ptr(weight, "weight"), rows, V, float(eps),
                               _dev_ptr(out, "out"), _dtype_code(out),
                               _stream_handle(stream, o.device))
    if st != KDA_OK:
        raise KDAError(st, "kda_gated_rmsnorm")
    return out


def chunk_bwd_workspace_size(N: int, T: int, H: int, K: int = 128, V: int = 128) -> int:
    """Bytes of workspace kda_chunk_bwd needs."""
    out = ctypes.c_int64(0)
    st = load_library().kda_chunk_bwd_workspace_size(N, T, H, K, V, ctypes.byref(out))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_bwd_workspace_size")
    return out.value


def kda_chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                  beta: torch.Tensor, cu_seqlens: torch.Tensor, dout: torch.Tensor,
                  scale: Optional[float] = None, dfinal_state: Optional[torch.Tensor] = None,
                  initial_state: Optional[torch.Tensor] = None, want_dinitial: bool = True,
                  cu_seqlens_host: Optional[Sequence[int]] = None, qk_l2norm: bool = True,
                  status: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None, workspace=None):
    """Backward of kda_chunk_fwd.  Returns FP32 (dq, dk, dv, dg, dbeta, dinitial_state
    or None).  workspace: None (a fresh buffer) or a CUDA tensor of at least
    chunk_bwd_workspace_size(...) bytes."""
    lib = load_library()
    T, H, K = q.shape
    V = v.shape[2]
    N = cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dg = (torch.empty((T, H, K), **f32) for _ in range(3))
    dv = torch.empty((T, H, V), **f32)
    dbeta = torch.empty((T, H), **f32)
    dinit = torch.empty((N, H, K, V), **f32) if want_dinitial else None
    if workspace is None:
        workspace = torch.empty(chunk_bwd_workspace_size(N, T, H, K, V), dtype=torch.uint8,
                                device=dev)
    keep, host = _host_offsets(cu_seqlens_host)
    st = lib.kda_chunk_bwd(
        _dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dtype_code(q),
        _dev_ptr(g, "g"), _dev_ptr(beta, "beta"), _dev_ptr(cu_seqlens, "cu_seqlens"), host,
        N, T, H, K, V, float(scale), 1 if qk_l2norm else 0,
        _dev_ptr(dout, "dout"), _dtype_code(dout), _dev_ptr(initial_state, "initial_state"),
        _dev_ptr(dfinal_state, "dfinal_state"), _dev_ptr(dq, "dq"), _dev_ptr(dk, "dk"),
        _dev_ptr(dv, "dv"), _dev_ptr(dg, "dg"), _dev_ptr(dbeta, "dbeta"),
        _dev_ptr(dinit, "dinitial_state"), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev_ptr(status, "status"),
        _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KDAError(st, "kda_chunk_bwd")
    return dq, dk, dv, dg, dbeta, dinit
