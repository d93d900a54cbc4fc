"""One very long sequence (262144 tokens, 4096 chunks, 2 heads): the forward in
both modes and the backward, checked on the last 300 tokens of a head and on
the final state.  The oracle runs the prefix to get the state where the
suffix starts; from that state the suffix's outputs and gradients are exactly
those of the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import backward as oracle_backward
from kimi_delta_attention_10_gb300 import kda_chunk_bwd, kda_chunk_fwd
from kimi_delta_attention_10_gb300.inputs import make_cotangents, make_inputs

from gpu_util import TOL, device_inputs, f64, rel_l2

pytestmark = pytest.mark.gpu

T, H, P = 262144, 2, 300


@pytest.fixture(scope="module")
def case():
    x = make_inputs([T], H, 128, 128, torch.bfloat16, 111)
    g, beta = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    g32, b32 = torch.from_numpy(g).float(), torch.from_numpy(beta).float()
    # the oracle state before the suffix, per head, from the same FP32 g and beta
    sl = lambda t, h, a, b: f64(t[a:b, h:h + 1])
    S_pre = []
    for h in range(H):
        _, S = oracle.forward(sl(x.q, h, 0, T - P), sl(x.k, h, 0, T - P), sl(x.v, h, 0, T - P),
                              sl(g32, h, 0, T - P), sl(b32, h, 0, T - P),
                              np.array([0, T - P], np.int32), x.scale)
        S_pre.append(S)
    return x, g32, b32, S_pre


@pytest.mark.parametrize("mode", ["bf16_tc", "fp32_exact"])
def test_long_forward_suffix_and_final_state(case, mode):
    x, g32, b32, S_pre = case
    d = device_inputs(x)
    out, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g32.cuda(), b32.cuda(), d["cu_seqlens"],
                           x.scale, mode=mode, out_dtype=torch.float32,
                           cu_seqlens_host=x.cu_seqlens.tolist(),
                           workspace="auto" if mode == "bf16_tc" else None)
    torch.cuda.synchronize()
    out, S = out.cpu().double().numpy(), S.cpu().double().numpy()
    sl = lambda t, h: f64(t[T - P:, h:h + 1])
    for h in range(H):
        o_ref, S_ref = oracle.forward(sl(x.q, h), sl(x.k, h), sl(x.v, h), sl(g32, h), sl(b32, h),
                                      np.array([0, P], np.int32), x.scale,
                                      initial_state=S_pre[h])
        assert rel_l2(out[T - P:, h:h + 1], o_ref) <= TOL[mode], (h, "out")
        assert rel_l2(S[:, h:h + 1], S_ref) <= TOL[mode], (h, "state")


def test_long_backward_suffix(case):
    x, g32, b32, S_pre = case
    d = device_inputs(x)
    dO, dfin, _ = make_cotangents(T, 1, H, 128, 128, 112, dout_dtype=torch.bfloat16)
    grads = kda_chunk_bwd(d["q"], d["k"], d["v"], g32.cuda(), b32.cuda(), d["cu_seqlens"],
                          dO.cuda(), x.scale, dfinal_state=dfin.cuda(), want_dinitial=False,
                          cu_seqlens_host=x.cu_seqlens.tolist())
    torch.cuda.synchronize()
    grads = [t.cpu().double().numpy() for t in grads[:5]]
    sl = lambda t, h: f64(t[T - P:, h:h + 1])
    for h in range(H):
        ref = oracle_backward(sl(x.q, h), sl(x.k, h), sl(x.v, h), sl(g32, h), sl(b32, h),
                              np.array([0, P], np.int32), x.scale, sl(dO, h),
                              dS_final=f64(dfin[:, h:h + 1]), initial_state=S_pre[h])
        for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), grads, ref):
            assert rel_l2(a[T - P:, h:h + 1], b) <= 1e-5, (h, name)
