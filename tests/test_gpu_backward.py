"""GPU parity of kda_chunk_bwd (the VJP of the forward) against the FP64
backward oracle, output by output, on the same seeded inputs.

g and beta come from the FP64 oracle gate rounded to FP32, so both sides
differentiate the same recurrence; the tolerance is the FP32 path's rel-L2
bar.  The full-size case (one 16384-token sequence, 64 heads) is checked on a
suffix of sampled heads: with the oracle state at the suffix start as initial
state, the suffix's gradients are exactly those of the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
from oracle.backward import backward as oracle_backward
from kimi_delta_attention_10_gb300 import (KDAError, chunk_bwd_workspace_size, kda_chunk_bwd)
from kimi_delta_attention_10_gb300.inputs import make_cotangents, make_inputs, workload_inputs

from gpu_util import f64, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-5          # rel-L2 of every gradient against FP64 (FP32 arithmetic)
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dS0")


def _gate32(x):
    g, beta = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    return torch.from_numpy(g).float(), torch.from_numpy(beta).float()


def _run(x, g, beta, dO, dfinal, init, l2norm=True, q=None, k=None, want_dinitial=True):
    q = x.q if q is None else q
    k = x.k if k is None else k
    cu = lambda t: None if t is None else t.cuda()
    res = kda_chunk_bwd(q.cuda(), k.cuda(), x.v.cuda(), g.cuda(), beta.cuda(),
                        x.cu_seqlens.cuda(), dO.cuda(), x.scale, dfinal_state=cu(dfinal),
                        initial_state=cu(init), want_dinitial=want_dinitial,
                        cu_seqlens_host=x.cu_seqlens.tolist(), qk_l2norm=l2norm)
    torch.cuda.synchronize()
    return [None if r is None else r.cpu().double().numpy() for r in res]


def _ref(x, g, beta, dO, dfinal, init, l2norm=True, q=None, k=None):
    q = x.q if q is None else q
    k = x.k if k is None else k
    opt = lambda t: None if t is None else f64(t)
    return oracle_backward(f64(q), f64(k), f64(x.v), f64(g), f64(beta), x.cu_seqlens.numpy(),
                           x.scale, f64(dO), dS_final=opt(dfinal), initial_state=opt(init),
                           l2norm=l2norm)


def _check(got, ref, skip=()):
    for name, a, b in zip(NAMES, got, ref):
        if name in skip:
            continue
        err = rel_l2(a, b)
        assert err <= TOL, f"{name}: rel-L2 {err:.3e}"


def test_fp32_two_sequences_with_states():
    x = make_inputs([100, 37], 2, 128, 128, torch.float32, 81)
    g, beta = _gate32(x)
    dO, dfin, init = make_cotangents(x.T, x.N, 2, 128, 128, 81)
    _check(_run(x, g, beta, dO, dfin, init), _ref(x, g, beta, dO, dfin, init))


def test_bf16_ragged_without_states_no_l2norm():
    """Lengths spanning several chunks, a one-token and an empty sequence; BF16
    q/k/v and dout; no normalisation (q, k scaled by 1/16, exactly, to keep the
    un-normalised recurrence contractive); no initial or final state."""
    x = make_inputs([130, 1, 0, 64], 3, 128, 128, torch.bfloat16, 82)
    g, beta = _gate32(x)
    dO, _, _ = make_cotangents(x.T, x.N, 3, 128, 128, 82, dout_dtype=torch.bfloat16)
    q, k = x.q / 16, x.k / 16
    got = _run(x, g, beta, dO, None, None, l2norm=False, q=q, k=k)
    ref = _ref(x, g, beta, dO, None, None, l2norm=False, q=q, k=k)
    _check(got, ref)


def test_more_units_than_resident_ctas():
    """70 short sequences x 4 heads: each persistent CTA walks several units."""
    gen = torch.Generator().manual_seed(83)
    lens = torch.randint(1, 10, (70,), generator=gen).tolist()
    x = make_inputs(lens, 4, 128, 128, torch.float32, 83)
    g, beta = _gate32(x)
    dO, dfin, init = make_cotangents(x.T, x.N, 4, 128, 128, 83)
    _check(_run(x, g, beta, dO, dfin, init), _ref(x, g, beta, dO, dfin, init))


def test_empty_sequences_pass_the_state_gradient_through():
    x = make_inputs([0, 0, 0], 2, 128, 128, torch.float32, 84)
    g, beta = _gate32(x)
    dO, dfin, _ = make_cotangents(0, 3, 2, 128, 128, 84)
    got = _run(x, g, beta, dO, dfin, None)
    assert np.array_equal(got[5], f64(dfin))
    got = _run(x, g, beta, dO, None, None)
    assert not np.any(got[5])


def test_workspace_too_small_is_rejected():
    x = make_inputs([65], 1, 128, 128, torch.float32, 85)
    g, beta = _gate32(x)
    dO, _, _ = make_cotangents(x.T, 1, 1, 128, 128, 85)
    need = chunk_bwd_workspace_size(1, x.T, 1)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(KDAError):
        kda_chunk_bwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), g.cuda(), beta.cuda(),
                      x.cu_seqlens.cuda(), dO.cuda(), workspace=ws)


def test_full_size_suffix_of_sampled_heads():
    """One 16384-token sequence, 64 heads, BF16 q/k/v (the timed workload):
    the last 200 tokens (three chunk boundaries) of heads 0 and 37."""
    x = workload_inputs("single_16384_bf16")
    T, H, P = x.T, x.H, 200
    g, beta = _gate32(x)
    dO, dfin, _ = make_cotangents(T, 1, H, 128, 128, 86, dout_dtype=torch.bfloat16)
    got = _run(x, g, beta, dO, dfin, None, want_dinitial=False)
    assert got[5] is None
    for h in (0, 37):
        sl = lambda t: t[:, h:h + 1]
        pre = np.array([0, T - P], np.int32)
        _, S = oracle.forward(f64(sl(x.q)[:T - P]), f64(sl(x.k)[:T - P]), f64(sl(x.v)[:T - P]),
                              f64(sl(g)[:T - P]), f64(sl(beta)[:T - P]), pre, x.scale)
        ref = oracle_backward(f64(sl(x.q)[T - P:]), f64(sl(x.k)[T - P:]), f64(sl(x.v)[T - P:]),
                              f64(sl(g)[T - P:]), f64(sl(beta)[T - P:]),
                              np.array([0, P], np.int32), x.scale, f64(sl(dO)[T - P:]),
                              dS_final=f64(dfin[:, h:h + 1]), initial_state=S)
        for name, a, b in zip(NAMES[:5], got[:5], ref[:5]):
            err = rel_l2(a[T - P:, h:h + 1], b)
            assert err <= TOL, f"head {h} {name}: rel-L2 {err:.3e}"
