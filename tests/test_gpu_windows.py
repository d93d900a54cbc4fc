"""The two-phase tensor-core path cut into chunk windows (preparation of later
windows beside the scan of earlier ones, by programmatic dependent launch on
the caller's stream) against the same path in one window
(kda_chunk_fwd_static never cuts), bit for bit,
and against the FP64 oracle.  Windows are used when the (sequence, head)
count is at most the SM count and there are at least 64 chunks."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_10_gb300 import (kda_chunk_fwd, kda_chunk_fwd_gated, kda_chunk_fwd_static,
                                           kda_gate)
from kimi_delta_attention_10_gb300.inputs import make_inputs

from gpu_util import device_inputs, f64, rel_l2

pytestmark = pytest.mark.gpu


def _both(lens, H, seed, init, host_mirror):
    x = make_inputs(lens, H, 128, 128, torch.bfloat16, seed)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    S0 = None
    if init:
        gen = torch.Generator().manual_seed(seed + 1)
        S0 = (torch.randn(x.N, H, 128, 128, generator=gen) * 0.1).cuda()
    host = x.cu_seqlens.tolist() if host_mirror else None
    o_w, S_w = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                             mode="bf16_tc", workspace="auto", initial_state=S0,
                             cu_seqlens_host=host)
    o_1 = torch.full_like(o_w, float("nan"))
    S_1 = torch.full_like(S_w, float("nan"))
    kda_chunk_fwd_static(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], o_1, x.scale,
                         final_state=S_1, initial_state=S0, cu_seqlens_host=host)
    torch.cuda.synchronize()
    return x, S0, (o_w, S_w), (o_1, S_1)


@pytest.mark.parametrize("lens,H,init,host_mirror", [
    ([3000, 0, 1200], 2, True, True),       # a sequence across both windows, an empty one
    ([16384], 2, False, True),              # three windows
    ([2100, 2100], 3, True, False),         # windows from the chunk bound (no host mirror)
    ([5000, 1, 6000, 0, 3000], 3, True, True),   # three windows, sequences across several
])
def test_windows_are_bitwise_one_window(lens, H, init, host_mirror):
    _, _, (o_w, S_w), (o_1, S_1) = _both(lens, H, 91 + H, init, host_mirror)
    assert torch.equal(o_w, o_1)
    assert torch.equal(S_w, S_1)


def test_windows_match_oracle():
    x, S0, (o_w, S_w), _ = _both([3000, 0, 1200], 2, 95, True, True)
    o_ref, S_ref, _, _ = oracle.reference(
        f64(x.q), f64(x.k), f64(x.v), f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b),
        x.cu_seqlens.numpy(), x.scale, initial_state=S0.cpu().double().numpy())
    assert rel_l2(o_w.float().cpu().numpy(), o_ref) <= 3e-3
    assert rel_l2(S_w.cpu().numpy(), S_ref) <= 3e-3
    # the empty sequence passes its initial state through unchanged
    assert np.array_equal(S_w[1].cpu().numpy(), S0[1].cpu().numpy())


def test_fused_gate_in_windows_matches_gate_then_chunk():
    """The timed configuration's shape of schedule (three chunk windows) with the
    gate fused into the preparation (its fast e^g), against kda_gate +
    kda_chunk_fwd and against the FP64 oracle."""
    x = make_inputs([16384], 2, 128, 128, torch.bfloat16, 97)
    d = device_inputs(x)
    host = x.cu_seqlens.tolist()
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    o1, s1 = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                           mode="bf16_tc", workspace="auto", cu_seqlens_host=host)
    o2, s2 = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], x.scale, mode="bf16_tc",
                                 workspace="auto", cu_seqlens_host=host)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().double().numpy()
    assert rel_l2(f(o2), f(o1)) <= 2e-3 and rel_l2(f(s2), f(s1)) <= 2e-3
    g_ref, b_ref = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    o_ref, S_ref = oracle.forward(f64(x.q), f64(x.k), f64(x.v), g_ref, b_ref,
                                  x.cu_seqlens.numpy(), x.scale)
    assert rel_l2(f(o2), o_ref) <= 3e-3 and rel_l2(f(s2), S_ref) <= 3e-3
