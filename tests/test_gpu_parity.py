"""GPU parity: the CUDA path against the FP64 oracle, element by element.

Tolerances: rel-L2 <= 1e-5 for the FP32-exact path with FP32 output,
<= 3e-3 for the BF16 tensor-core path.  The gate is checked elementwise."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_10_gb300 import kda_chunk_fwd, kda_gate
from kimi_delta_attention_10_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

from gpu_util import (OUT_DTYPE, PATHS, device_inputs, f64, gpu_pipeline, oracle_pipeline,
                      path_kw, rel_l2, tol)

pytestmark = pytest.mark.gpu

# Heads compared on the two large workloads (the GPU still runs all 64).
SAMPLED_HEADS = [0, 17, 42, 63]

_cache = {}


def inputs(i):
    if i not in _cache:
        _cache[i] = workload_inputs(i)
    return _cache[i]


@pytest.mark.parametrize("wi", range(len(WORKLOADS)))
def test_gate_matches_oracle(wi):
    x = inputs(wi)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    torch.cuda.synchronize()
    heads = SAMPLED_HEADS if x.T > 4096 else list(range(x.H))
    g_ref, b_ref = oracle.gate(f64(x.f[:, heads]), f64(x.A_log[heads]),
                               f64(x.dt_bias[heads]), f64(x.b[:, heads]))
    g_gpu = g.cpu()[:, heads].double().numpy()
    b_gpu = beta.cpu()[:, heads].double().numpy()
    # FP32 rounding of f + dt_bias moves softplus by up to |x| * 2^-24 relatively.
    assert np.max(np.abs(g_gpu - g_ref) / np.abs(g_ref)) < 2e-6
    assert np.max(np.abs(b_gpu - b_ref) / b_ref) < 1e-6


def test_gate_extremes_and_bf16_inputs():
    T, H, K = 6, 3, 128
    gen = torch.Generator().manual_seed(5)
    dt_bias = torch.randn(H, K, generator=gen) * 0.5
    f = torch.empty(T, H, K)
    f[0], f[1], f[2] = -30.0 - dt_bias, -dt_bias, 30.0 - dt_bias
    f[3:] = torch.randn(3, H, K, generator=gen)
    A_log = torch.tensor([0.0, 1.0, float(np.log(16.0))])
    b = torch.tensor([[-20.0, 0.0, 20.0]] * T)
    for fdt in (torch.float32, torch.bfloat16):
        fx, bx = f.to(fdt), b.to(fdt)
        g, beta = kda_gate(fx.cuda(), A_log.cuda(), dt_bias.cuda(), bx.cuda())
        g_ref, b_ref = oracle.gate(f64(fx), f64(A_log), f64(dt_bias), f64(bx))
        g_gpu = g.cpu().double().numpy()
        assert np.all(g_gpu < 0)
        assert np.max(np.abs(g_gpu - g_ref) / np.abs(g_ref)) < 4e-6
        assert np.max(np.abs(beta.cpu().double().numpy() - b_ref) / b_ref) < 2e-6


MODES = list(PATHS)     # FP32-exact and BF16 tensor-core, each single-pass and two-phase


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("wi", range(len(WORKLOADS)))
def test_chunk_matches_oracle(wi, mode):
    """Full path (gate + chunk) on each workload; all heads on the small ones,
    sampled heads on the 16384-token and packed 32768-token workloads."""
    x = inputs(wi)
    out, S, _, _ = gpu_pipeline(x, mode, out_dtype=OUT_DTYPE[mode])
    heads = SAMPLED_HEADS if x.T > 4096 else None
    o_ref, S_ref, _, _ = oracle_pipeline(x, heads)
    sel = slice(None) if heads is None else heads
    o_gpu = out[:, sel].double().numpy()
    S_gpu = S[:, sel].double().numpy()
    assert np.isfinite(o_gpu).all() and np.isfinite(S_gpu).all()
    e_o, e_S = rel_l2(o_gpu, o_ref), rel_l2(S_gpu, S_ref)
    print(f"{WORKLOADS[wi].name} {mode}: out rel-L2 {e_o:.3e}, final state rel-L2 {e_S:.3e}")
    assert e_o <= tol(mode) and e_S <= tol(mode)


def _small(lens, H=4, seed=0, dtype=torch.bfloat16):
    return make_inputs(lens, H, 128, 128, dtype, seed)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [127, 128], [129, 0, 3], [0], [200, 1, 64]])
def test_chunk_edge_lengths(lens, mode):
    x = _small(lens, seed=sum(lens) + len(lens))
    out, S, _, _ = gpu_pipeline(x, mode, out_dtype=OUT_DTYPE[mode])
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    if x.T:
        assert rel_l2(out.double().numpy(), o_ref) <= tol(mode)
    assert rel_l2(S.double().numpy(), S_ref) <= tol(mode)
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(S[n]) == 0


@pytest.mark.parametrize("mode", MODES)
def test_packing_is_bitwise_per_sequence(mode):
    lens = [70, 5, 129]
    x = _small(lens, seed=3)
    out, S, _, _ = gpu_pipeline(x, mode, out_dtype=OUT_DTYPE[mode])
    cu = x.cu_seqlens.tolist()
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    for n in range(len(lens)):
        a, z = cu[n], cu[n + 1]
        cu1 = torch.tensor([0, z - a], dtype=torch.int32, device="cuda")
        o1, S1 = kda_chunk_fwd(d["q"][a:z].contiguous(), d["k"][a:z].contiguous(),
                               d["v"][a:z].contiguous(), g[a:z].contiguous(),
                               beta[a:z].contiguous(), cu1, x.scale,
                               out_dtype=OUT_DTYPE[mode], **path_kw(mode))
        assert torch.equal(o1.cpu(), out[a:z]) and torch.equal(S1.cpu()[0], S[n])


@pytest.mark.parametrize("mode", MODES)
def test_deterministic_and_head_permutation(mode):
    x = _small([150, 40], H=6, seed=4)
    out1, S1, _, _ = gpu_pipeline(x, mode, out_dtype=OUT_DTYPE[mode])
    out2, S2, _, _ = gpu_pipeline(x, mode, out_dtype=OUT_DTYPE[mode])
    assert torch.equal(out1, out2) and torch.equal(S1, S2)
    perm = torch.tensor([3, 0, 5, 1, 4, 2])
    xp = _small([150, 40], H=6, seed=4)
    for name in ("q", "k", "v", "f", "b"):
        setattr(xp, name, getattr(xp, name)[:, perm].contiguous())
    xp.A_log = xp.A_log[perm].contiguous()
    xp.dt_bias = xp.dt_bias[perm].contiguous()
    outp, Sp, _, _ = gpu_pipeline(xp, mode, out_dtype=OUT_DTYPE[mode])
    assert torch.equal(outp, out1[:, perm]) and torch.equal(Sp, S1[:, perm])


@pytest.mark.parametrize("mode", MODES)
def test_without_l2norm_on_prenormalised_inputs(mode):
    x = _small([90], H=2, seed=6, dtype=torch.float32)
    x.q = x.q / torch.sqrt((x.q * x.q).sum(-1, keepdim=True))
    x.k = x.k / torch.sqrt((x.k * x.k).sum(-1, keepdim=True))
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    out, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           qk_l2norm=False, **path_kw(mode))
    g_ref, b_ref = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    o_ref, S_ref = oracle.forward(f64(x.q), f64(x.k), f64(x.v), g_ref, b_ref,
                                  x.cu_seqlens.numpy(), x.scale, l2norm=False)
    assert rel_l2(out.cpu().double().numpy(), o_ref) <= tol(mode)
    assert rel_l2(S.cpu().double().numpy(), S_ref) <= tol(mode)


def test_bf16_output_in_fp32_mode():
    x = _small([129], H=2, seed=7)
    out, S, _, _ = gpu_pipeline(x, "fp32_exact", out_dtype=torch.bfloat16)
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    assert out.dtype == torch.bfloat16
    assert rel_l2(out.double().numpy(), o_ref) <= 3e-3      # BF16 rounding of the output
    assert rel_l2(S.double().numpy(), S_ref) <= 1e-5


@pytest.mark.parametrize("mode", MODES)
def test_device_detects_bad_offsets_without_host_mirror(mode):
    """Offsets past T with no host mirror: the kernel reports through the status
    word, skips that sequence, and computes the others."""
    x = _small([40, 30], H=2, seed=8)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    bad = torch.tensor([0, 40, 90], dtype=torch.int32, device="cuda")   # 90 > T = 70
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(70, 2, 128, device="cuda")
    kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, bad, x.scale, out=out, status=status,
                  **path_kw(mode))
    torch.cuda.synchronize()
    assert int(status[0]) == 6
    o_ref, _, _, _ = oracle_pipeline(x)
    assert rel_l2(out[:40].cpu().double().numpy(), o_ref[:40]) <= tol(mode)
    assert torch.count_nonzero(out[40:]) == 0


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("host_mirror", [True, False])
def test_many_short_sequences(mode, host_mirror):
    """2600 packed sequences of 0..24 tokens: more than one 1024-wide tile of the
    two-phase path's chunk-offset scan, and a preparation grid sized from the
    offsets bound when no host mirror is given."""
    gen = torch.Generator().manual_seed(61)
    lens = torch.randint(0, 25, (2600,), generator=gen).tolist()
    x = _small(lens, H=2, seed=62)
    out, S, _, _ = gpu_pipeline(x, mode, out_dtype=OUT_DTYPE[mode], host_mirror=host_mirror)
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    assert rel_l2(out.double().numpy(), o_ref) <= tol(mode)
    assert rel_l2(S.double().numpy(), S_ref) <= tol(mode)
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(S[n]) == 0


@pytest.mark.parametrize("mode", MODES)
def test_final_state_may_alias_initial_state(mode):
    lens = [150, 0, 70]
    x = _small(lens, seed=63)
    gen = torch.Generator().manual_seed(63)
    S0 = (torch.randn(len(lens), x.H, 128, 128, generator=gen) * 0.2).cuda()
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    kw = dict(out_dtype=OUT_DTYPE[mode], **path_kw(mode))
    o1, S1 = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           initial_state=S0, **kw)
    S_inout = S0.clone()
    o2, S2 = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           initial_state=S_inout, final_state=S_inout, **kw)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S_inout.data_ptr()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
