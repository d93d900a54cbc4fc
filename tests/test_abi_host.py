"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

Every negative case below is rejected by the host validation in kda_api.cu
before any CUDA call, so fake (never dereferenced) pointer values are safe."""
import ctypes
import os
import re

import pytest

from kimi_delta_attention_10_gb300 import _build, binding

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.kda_abi_version() == 3
    assert binding.status_string(0) == "ok"
    for s in range(1, 9):
        assert binding.status_string(s) not in ("ok", "unknown status")
    assert binding.status_string(99) == "unknown status"


# A fake, 16-byte-aligned device address that is never dereferenced.
P = 0x10000
MIS = 0x10004


def chunk(lib, **kw):
    a = dict(q=P, k=P, v=P, qkv=1, g=P, beta=P, cu=P, cu_host=None, N=1, T=10, H=2, K=128,
             V=128, scale=0.1, l2=1, mode=1, out=P, out_dt=1, s0=None, fs=None, ws=None,
             ws_bytes=0, status=None, stream=None)
    a.update(kw)
    host = a["cu_host"]
    if host is not None:
        host = ctypes.cast((ctypes.c_int32 * len(host))(*host), ctypes.c_void_p)
    return lib.kda_chunk_fwd(a["q"], a["k"], a["v"], a["qkv"], a["g"], a["beta"], a["cu"], host,
                             a["N"], a["T"], a["H"], a["K"], a["V"], a["scale"], a["l2"],
                             a["mode"], a["out"], a["out_dt"], a["s0"], a["fs"], a["ws"],
                             a["ws_bytes"], a["status"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(qkv=7), binding.KDA_ERR_INVALID_ARG),
    (dict(out_dt=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(mode=5), binding.KDA_ERR_INVALID_ARG),
    (dict(l2=2), binding.KDA_ERR_INVALID_ARG),
    (dict(K=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(K=16, V=24), binding.KDA_ERR_UNSUPPORTED),     # the pages' rectangular case
    (dict(V=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(N=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(T=-3), binding.KDA_ERR_INVALID_ARG),
    (dict(H=0), binding.KDA_ERR_INVALID_ARG),
    (dict(q=None), binding.KDA_ERR_INVALID_ARG),
    (dict(out=None), binding.KDA_ERR_INVALID_ARG),
    (dict(cu=None), binding.KDA_ERR_INVALID_ARG),
    (dict(q=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(g=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(fs=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(s0=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(status=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(cu_host=[0, 9]), binding.KDA_ERR_INVALID_ARG),           # last != T
    (dict(cu_host=[1, 10]), binding.KDA_ERR_INVALID_ARG),          # first != 0
    (dict(N=2, cu_host=[0, 7, 5]), binding.KDA_ERR_INVALID_ARG),   # decreasing (and last != T)
    (dict(N=3, cu_host=[0, 7, 5, 10]), binding.KDA_ERR_INVALID_ARG),
    (dict(mode=0, ws=MIS, ws_bytes=1 << 40), binding.KDA_ERR_ALIGNMENT),
    (dict(mode=0, ws=P, ws_bytes=1024), binding.KDA_ERR_INVALID_ARG),   # workspace too small
])
def test_chunk_fwd_rejects_bad_arguments(lib, kw, expect):
    assert chunk(lib, **kw) == expect


def workspace_size(lib, N, T, H, K=128, V=128, mode=0):
    out = ctypes.c_int64(-1)
    st = lib.kda_chunk_workspace_size(N, T, H, K, V, mode, ctypes.byref(out))
    return st, out.value


def test_workspace_size_bound():
    """The size covers the worst case of T / 64 + N chunks (every sequence
    adds at most one partial chunk), a 1 KiB-aligned offsets header and the
    FP32 state carried between chunk windows."""
    lib = binding.load_library()
    rec = 74240
    for N, T, H in [(1, 16384, 64), (16, 32768, 64), (3, 65, 4), (0, 0, 1), (5000, 70000, 2)]:
        st, nbytes = workspace_size(lib, N, T, H)
        assert st == binding.KDA_OK
        # flag, N + 1 offsets, N scan order, 3 chunk-window unit counters
        hdr = -(-(4 * (2 * N + 8)) // 1024) * 1024
        assert nbytes == hdr + (T // 64 + N) * H * rec + N * H * 128 * 128 * 4
        # the exact chunk count of any split of T tokens into N sequences is no larger
        lens = [T // max(N, 1)] * N
        if N:
            lens[-1] += T - sum(lens)
        assert sum(-(-L // 64) for L in lens) <= T // 64 + N
    # FP32-exact mode in two phases: the header and one 148224-byte record
    # per (chunk bound, head)
    hdr2 = -(-(4 * (2 * 2 + 9)) // 1024) * 1024
    assert workspace_size(lib, 2, 100, 3, mode=1) == (binding.KDA_OK,
                                                      hdr2 + (100 // 64 + 2) * 3 * 148224)
    assert workspace_size(lib, 2, 100, 3, K=64)[0] == binding.KDA_ERR_UNSUPPORTED
    assert workspace_size(lib, -1, 100, 3)[0] == binding.KDA_ERR_INVALID_ARG
    assert workspace_size(lib, 2, 100, 3, mode=7)[0] == binding.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_workspace_size(1, 10, 1, 128, 128, 0, None) == binding.KDA_ERR_INVALID_ARG
    assert binding.chunk_workspace_size(1, 16384, 64) == workspace_size(lib, 1, 16384, 64)[1]


def gate(lib, **kw):
    a = dict(f=P, fdt=0, A=P, dt=P, b=P, bdt=0, T=10, H=2, K=128, g=P, beta=P, stream=None)
    a.update(kw)
    return lib.kda_gate(a["f"], a["fdt"], a["A"], a["dt"], a["b"], a["bdt"], a["T"], a["H"],
                        a["K"], a["g"], a["beta"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(fdt=3), binding.KDA_ERR_INVALID_ARG),
    (dict(bdt=3), binding.KDA_ERR_INVALID_ARG),
    (dict(K=6), binding.KDA_ERR_UNSUPPORTED),
    (dict(H=0), binding.KDA_ERR_INVALID_ARG),
    (dict(T=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(f=None), binding.KDA_ERR_INVALID_ARG),
    (dict(beta=None), binding.KDA_ERR_INVALID_ARG),
    (dict(g=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(A=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(T=0), binding.KDA_OK),                                    # nothing to do
    (dict(T=0, f=None, b=None, g=None, beta=None), binding.KDA_OK),  # empty tensors
])
def test_gate_rejects_bad_arguments(lib, kw, expect):
    assert gate(lib, **kw) == expect


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 2, 128)
    with pytest.raises(RuntimeError, match="CUDA tensor"):
        binding.kda_gate(x, torch.zeros(2), torch.zeros(2, 128), torch.zeros(4, 2))


def gated(lib, **kw):
    a = dict(q=P, k=P, v=P, qkv=1, f=P, fdt=0, A=P, dt=P, b=P, bdt=0, cu=P, N=1, T=10, H=2,
             K=128, V=128, mode=0, out=P, out_dt=1, s0=None, fs=None)
    a.update(kw)
    return lib.kda_chunk_fwd_gated(a["q"], a["k"], a["v"], a["qkv"], a["f"], a["fdt"], a["A"],
                                   a["dt"], a["b"], a["bdt"], a["cu"], None, a["N"], a["T"],
                                   a["H"], a["K"], a["V"], 0.1, 1, a["mode"], a["out"],
                                   a["out_dt"], a["s0"], a["fs"], a.get("ws"), a.get("ws_bytes", 0),
                                   None, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(fdt=4), binding.KDA_ERR_INVALID_ARG),
    (dict(fdt=1, f=MIS), binding.KDA_ERR_ALIGNMENT),   # BF16 f accepted, checked like F32
    (dict(bdt=4), binding.KDA_ERR_INVALID_ARG),
    (dict(A=None), binding.KDA_ERR_INVALID_ARG),
    (dict(f=None), binding.KDA_ERR_INVALID_ARG),
    (dict(b=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(K=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(mode=3), binding.KDA_ERR_INVALID_ARG),
    (dict(ws=P, ws_bytes=100), binding.KDA_ERR_INVALID_ARG),
])
def test_chunk_fwd_gated_rejects_bad_arguments(lib, kw, expect):
    assert gated(lib, **kw) == expect


def step(lib, **kw):
    a = dict(q=P, k=P, v=P, qkv=1, g=P, beta=P, N=4, H=2, K=128, V=128, state=P, out=P, out_dt=1)
    a.update(kw)
    return lib.kda_recurrent_step(a["q"], a["k"], a["v"], a["qkv"], a["g"], a["beta"], a["N"],
                                  a["H"], a["K"], a["V"], 0.1, 1, a["state"], a["out"],
                                  a["out_dt"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(N=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(N=0, q=None), binding.KDA_OK),               # nothing to do
    (dict(V=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(state=None), binding.KDA_ERR_INVALID_ARG),
    (dict(state=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(qkv=9), binding.KDA_ERR_INVALID_ARG),
])
def test_recurrent_step_rejects_bad_arguments(lib, kw, expect):
    assert step(lib, **kw) == expect


def static(lib, **kw):
    a = dict(q=P, k=P, v=P, qkv=1, g=P, beta=P, cu=P, N=1, T=10, H=2, K=128, V=128, out=P,
             out_dt=1)
    a.update(kw)
    return lib.kda_chunk_fwd_static(a["q"], a["k"], a["v"], a["qkv"], a["g"], a["beta"], a["cu"],
                                    None, a["N"], a["T"], a["H"], a["K"], a["V"], 0.1, 1,
                                    a["out"], a["out_dt"], None, None, None, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(K=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(g=None), binding.KDA_ERR_INVALID_ARG),
    (dict(beta=MIS), binding.KDA_ERR_ALIGNMENT),
    # over the 64 MiB static scratch: (T / 64 + N) * H records of 74240 bytes
    (dict(T=1024, N=1, H=64), binding.KDA_ERR_TOO_LARGE),
    (dict(T=64 * 14, N=1, H=64), binding.KDA_ERR_TOO_LARGE),
])
def test_chunk_fwd_static_rejects_bad_arguments(lib, kw, expect):
    assert static(lib, **kw) == expect


def test_static_scratch_limit_at_64_heads_one_sequence(lib):
    """H = 64, N = 1: T / 64 + N = 13 fits the 64 MiB scratch (12 full chunks,
    768 tokens), 14 does not (the bound adds 64 x 64 KiB of state carry)."""
    assert static(lib, T=64 * 12, N=1, H=64) != binding.KDA_ERR_TOO_LARGE
    assert static(lib, T=64 * 13, N=1, H=64) == binding.KDA_ERR_TOO_LARGE
    assert workspace_size(lib, 1, 64 * 12, 64)[1] <= (64 << 20) < workspace_size(lib, 1, 64 * 13, 64)[1]


def test_test_fault_hook_rejects_unknown_values(lib):
    assert lib.kda_test_set_fault(4) == binding.KDA_ERR_INVALID_ARG
    assert lib.kda_test_set_fault(-1) == binding.KDA_ERR_INVALID_ARG
    assert lib.kda_test_set_fault(binding.KDA_TEST_FAULT_NONE) == binding.KDA_OK


def test_static_scratch_limit_is_the_workspace_bound(lib):
    """The largest problems the static scratch admits are the ones whose
    workspace bound fits in 64 MiB."""
    for H in (1, 8, 64):
        lo, hi = 0, 1 << 20                   # chunk counts: lo fits, hi does not
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if workspace_size(lib, 1, 64 * mid, H)[1] <= (64 << 20):
                lo = mid
            else:
                hi = mid
        assert static(lib, T=64 * hi, N=1, H=H) == binding.KDA_ERR_TOO_LARGE
        # at the limit the call gets past the size check (without a GPU it then
        # fails at the device set-up instead)
        assert static(lib, T=64 * lo, N=1, H=H) != binding.KDA_ERR_TOO_LARGE


def grms(lib, **kw):
    a = dict(o=P, odt=1, z=P, zdt=1, w=P, rows=10, V=128, eps=1e-6, y=P, ydt=1)
    a.update(kw)
    return lib.kda_gated_rmsnorm(a["o"], a["odt"], a["z"], a["zdt"], a["w"], a["rows"], a["V"],
                                 a["eps"], a["y"], a["ydt"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(V=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(rows=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(eps=-1.0), binding.KDA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), binding.KDA_ERR_INVALID_ARG),
    (dict(odt=5), binding.KDA_ERR_INVALID_ARG),
    (dict(z=None), binding.KDA_ERR_INVALID_ARG),
    (dict(w=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(ydt=0), binding.KDA_ERR_INVALID_ARG),          # y aliases o with another dtype
    (dict(rows=0, o=None, z=None, w=None, y=None), binding.KDA_OK),
])
def test_gated_rmsnorm_rejects_bad_arguments(lib, kw, expect):
    assert grms(lib, **kw) == expect


def bwd(lib, **kw):
    ptr = lambda i: P + 0x1000 * i                 # distinct, 16-byte aligned, never dereferenced
    a = dict(q=ptr(0), k=ptr(1), v=ptr(2), qkv=1, g=ptr(3), beta=ptr(4), cu=ptr(5), host=None,
             N=1, T=100, H=2, K=128, V=128, scale=0.1, l2=1, dout=ptr(6), ddt=1, init=None,
             dfin=None, dq=ptr(7), dk=ptr(8), dv=ptr(9), dg=ptr(10), db=ptr(11), dinit=None,
             ws=ptr(12), wsb=1 << 40, status=None)
    a.update(kw)
    host = a["host"]
    hp = None
    if host is not None:
        arr = (ctypes.c_int32 * len(host))(*host)
        hp = ctypes.cast(arr, ctypes.c_void_p)
    return lib.kda_chunk_bwd(a["q"], a["k"], a["v"], a["qkv"], a["g"], a["beta"], a["cu"], hp,
                             a["N"], a["T"], a["H"], a["K"], a["V"], a["scale"], a["l2"],
                             a["dout"], a["ddt"], a["init"], a["dfin"], a["dq"], a["dk"], a["dv"],
                             a["dg"], a["db"], a["dinit"], a["ws"], a["wsb"], a["status"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(K=64), binding.KDA_ERR_UNSUPPORTED),
    (dict(ddt=5), binding.KDA_ERR_INVALID_ARG),
    (dict(dout=None), binding.KDA_ERR_INVALID_ARG),
    (dict(dq=None), binding.KDA_ERR_INVALID_ARG),
    (dict(db=None), binding.KDA_ERR_INVALID_ARG),
    (dict(ws=None), binding.KDA_ERR_INVALID_ARG),
    (dict(ws=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(dg=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(dinit=MIS), binding.KDA_ERR_ALIGNMENT),
    (dict(wsb=1024), binding.KDA_ERR_INVALID_ARG),
    (dict(host=[0, 99]), binding.KDA_ERR_INVALID_ARG),      # cu[N] != T
    (dict(l2=2), binding.KDA_ERR_INVALID_ARG),
    (dict(N=0, T=0, ws=None, q=None, k=None, v=None, dout=None, dq=None, dk=None, dv=None,
          dg=None, db=None), binding.KDA_OK),
    (dict(dq=P), binding.KDA_ERR_INVALID_ARG),                       # output is the q input
    (dict(dg=P + 0x8000), binding.KDA_ERR_INVALID_ARG),              # two outputs (dk, dg) alias
    (dict(dinit=P + 0xC000), binding.KDA_ERR_INVALID_ARG),           # output is the workspace
])
def test_chunk_bwd_rejects_bad_arguments(lib, kw, expect):
    assert bwd(lib, **kw) == expect


def test_bwd_workspace_size(lib):
    def size(N, T, H):
        out = ctypes.c_int64(0)
        assert lib.kda_chunk_bwd_workspace_size(N, T, H, 128, 128, ctypes.byref(out)) == 0
        return out.value

    def expected(N, T, H):
        hdr = -(-(4 * (2 * N + 5)) // 1024) * 1024
        state = 128 * 128 * 4
        ckpt = 4 * (T // 64 + N) * H * state            # one state per 16-token segment (bound)
        part = 3 * (3 * T * H * 128 + T * H) * 4        # partial row sums of column slices 1..3
        part = -(-part // 256) * 256
        scratch = min(4 * N * H, 1024) * 16 * (128 * 32 * 4)   # 16 state slices per CTA
        return hdr + ckpt + part + scratch
    for N, T, H in [(1, 16384, 64), (3, 100, 2), (1, 64, 256), (1, 64, 257), (0, 0, 1), (7, 5, 3)]:
        assert size(N, T, H) == expected(N, T, H), (N, T, H)
    out = ctypes.c_int64(0)
    assert lib.kda_chunk_bwd_workspace_size(1, 64, 1, 64, 128, ctypes.byref(out)) == \
        binding.KDA_ERR_UNSUPPORTED
