"""GPU tests of the fused-gate entry point, the initial state and the decode step."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_10_gb300 import (kda_chunk_fwd, kda_chunk_fwd_gated, kda_gate,
                                           kda_recurrent_step)
from kimi_delta_attention_10_gb300.inputs import make_inputs, workload_inputs

from gpu_util import (OUT_DTYPE, PATHS, device_inputs, f64, oracle_pipeline, path_kw, rel_l2,
                      tol)

pytestmark = pytest.mark.gpu

MODES = list(PATHS)


def _small(lens, H=4, seed=0, dtype=torch.bfloat16):
    return make_inputs(lens, H, 128, 128, dtype, seed)


# Fused against unfused on the tensor-core paths: they differ only by the fused
# prologue's e^g (relative 1e-5 against kda_gate's exp(g)), which flips a few
# FP16 operand and BF16 output roundings; both stay within 3e-3 of the oracle.
FUSED_VS_UNFUSED_TC = 2e-3


def assert_fused_matches_unfused(mode, o1, s1, o2, s2):
    """Bit for bit in FP32-exact mode (the gate's own arithmetic); within
    FUSED_VS_UNFUSED_TC on the tensor-core paths (the fast e^g)."""
    if PATHS[mode][0] == "fp32_exact":
        assert torch.equal(o1, o2) and torch.equal(s1, s2)
    else:
        f = lambda t: t.float().cpu().double().numpy()
        assert rel_l2(f(o2), f(o1)) <= FUSED_VS_UNFUSED_TC
        assert rel_l2(f(s2), f(s1)) <= FUSED_VS_UNFUSED_TC


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", ["packed_37_28_f32", "single_129_bf16", "edges"])
def test_gated_equals_gate_then_chunk(case, mode):
    """FP32-exact: the fused prologue uses the gate's exact FP32 arithmetic."""
    x = _small([1, 64, 0, 130], seed=21) if case == "edges" else workload_inputs(case)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    o1, s1 = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           out_dtype=OUT_DTYPE[mode], **path_kw(mode))
    o2, s2 = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], x.scale, out_dtype=OUT_DTYPE[mode],
                                 **path_kw(mode))
    torch.cuda.synchronize()
    assert_fused_matches_unfused(mode, o1, s1, o2, s2)


@pytest.mark.parametrize("mode", MODES)
def test_gated_matches_oracle(mode):
    x = workload_inputs("single_2048_bf16")
    d = device_inputs(x)
    out, S = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], x.scale, out_dtype=OUT_DTYPE[mode],
                                 cu_seqlens_host=x.cu_seqlens.tolist(), **path_kw(mode))
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    assert rel_l2(out.cpu().double().numpy(), o_ref) <= tol(mode)
    assert rel_l2(S.cpu().double().numpy(), S_ref) <= tol(mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("lens", [[1, 64, 0, 130], [8192]])
def test_gated_bf16_f_equals_gate_then_chunk(lens, mode):
    """f in BF16 (the gate projection's activation dtype): the fused call reads
    it as kda_gate does (FP32-exact: the same bits as kda_gate on the same BF16
    f followed by kda_chunk_fwd); 8192 tokens run the two-phase path in four
    windows."""
    x = _small(lens, H=2, seed=23)
    x.f = x.f.to(torch.bfloat16)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    o1, s1 = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           out_dtype=OUT_DTYPE[mode], **path_kw(mode))
    o2, s2 = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], x.scale, out_dtype=OUT_DTYPE[mode],
                                 **path_kw(mode))
    torch.cuda.synchronize()
    assert_fused_matches_unfused(mode, o1, s1, o2, s2)


@pytest.mark.parametrize("mode", MODES)
def test_gated_bf16_f_matches_oracle(mode):
    """BF16 f against the FP64 oracle fed the same BF16 values, upcast."""
    x = workload_inputs("single_2048_bf16")
    x.f = x.f.to(torch.bfloat16)
    d = device_inputs(x)
    out, S = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], x.scale, out_dtype=OUT_DTYPE[mode],
                                 cu_seqlens_host=x.cu_seqlens.tolist(), **path_kw(mode))
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    assert rel_l2(out.cpu().double().numpy(), o_ref) <= tol(mode)
    assert rel_l2(S.cpu().double().numpy(), S_ref) <= tol(mode)


def test_gated_bf16_beta_logits():
    x = _small([70, 33], seed=22)
    x.b = x.b.to(torch.bfloat16)
    d = device_inputs(x)
    out, S = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], x.scale, mode="fp32_exact",
                                 out_dtype=torch.float32)
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    assert rel_l2(out.cpu().double().numpy(), o_ref) <= 1e-5
    assert rel_l2(S.cpu().double().numpy(), S_ref) <= 1e-5


@pytest.mark.parametrize("mode", MODES)
def test_initial_state_matches_oracle(mode):
    lens = [100, 0, 37]
    x = _small(lens, seed=23)
    gen = torch.Generator().manual_seed(23)
    S0 = torch.randn(len(lens), x.H, 128, 128, generator=gen) * 0.2
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    out, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           out_dtype=OUT_DTYPE[mode], initial_state=S0.cuda(), **path_kw(mode))
    gr, br = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    o_ref, S_ref = oracle.forward(f64(x.q), f64(x.k), f64(x.v), gr, br, x.cu_seqlens.numpy(),
                                  x.scale, initial_state=S0.double().numpy())
    assert rel_l2(out.cpu().double().numpy(), o_ref) <= tol(mode)
    assert rel_l2(S.cpu().double().numpy(), S_ref) <= tol(mode)
    # the empty sequence returns its initial state
    assert torch.equal(S[1].cpu(), S0[1])


@pytest.mark.parametrize("mode", MODES)
def test_split_at_chunk_boundary_is_bitwise(mode):
    """Two calls, the second continuing from the first's final state, reproduce one
    call exactly when the split falls on a chunk boundary."""
    x = _small([200], seed=24)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    kw = dict(out_dtype=OUT_DTYPE[mode], **path_kw(mode))
    o, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale, **kw)
    cut = 128
    c1 = torch.tensor([0, cut], dtype=torch.int32, device="cuda")
    c2 = torch.tensor([0, 200 - cut], dtype=torch.int32, device="cuda")
    sl = lambda t, a, z: t[a:z].contiguous()
    o1, S1 = kda_chunk_fwd(sl(d["q"], 0, cut), sl(d["k"], 0, cut), sl(d["v"], 0, cut),
                           sl(g, 0, cut), sl(beta, 0, cut), c1, x.scale, **kw)
    o2, S2 = kda_chunk_fwd(sl(d["q"], cut, 200), sl(d["k"], cut, 200), sl(d["v"], cut, 200),
                           sl(g, cut, 200), sl(beta, cut, 200), c2, x.scale, initial_state=S1,
                           **kw)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([o1, o2]), o) and torch.equal(S2, S)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_recurrent_step_matches_oracle(dtype):
    N, H = 5, 3
    x = make_inputs([1] * N, H, 128, 128, dtype, seed=25)
    gen = torch.Generator().manual_seed(25)
    S0 = torch.randn(N, H, 128, 128, generator=gen) * 0.3
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    state = S0.cuda().clone()
    out = kda_recurrent_step(d["q"], d["k"], d["v"], g, beta, state, x.scale,
                             out_dtype=torch.float32)
    gr, br = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    o_ref, S_ref = oracle.forward(f64(x.q), f64(x.k), f64(x.v), gr, br, x.cu_seqlens.numpy(),
                                  x.scale, initial_state=S0.double().numpy())
    assert rel_l2(out.cpu().double().numpy(), o_ref) <= 1e-5
    assert rel_l2(state.cpu().double().numpy(), S_ref) <= 1e-5


@pytest.mark.parametrize("mode", MODES)
def test_chunk_prefill_then_decode_matches_oracle(mode):
    """Prefill 97 tokens with the chunk kernel, decode 3 more one at a time: the
    decoded outputs and the final state match one oracle run over all 100."""
    T, H, pre = 100, 2, 97
    x = _small([T], H=H, seed=26)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    c = torch.tensor([0, pre], dtype=torch.int32, device="cuda")
    _, S = kda_chunk_fwd(d["q"][:pre].contiguous(), d["k"][:pre].contiguous(),
                         d["v"][:pre].contiguous(), g[:pre].contiguous(),
                         beta[:pre].contiguous(), c, x.scale, out_dtype=OUT_DTYPE[mode],
                         **path_kw(mode))
    outs = []
    for t in range(pre, T):
        sl = lambda z: z[t:t + 1].clone()           # fresh, 16-byte-aligned storage
        outs.append(kda_recurrent_step(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(g), sl(beta), S,
                                       x.scale, out_dtype=torch.float32))
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    o_dec = torch.cat(outs).cpu().double().numpy()
    assert rel_l2(o_dec, o_ref[pre:]) <= tol(mode)
    assert rel_l2(S.cpu().double().numpy(), S_ref) <= tol(mode)
