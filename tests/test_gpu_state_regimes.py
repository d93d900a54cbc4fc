"""GPU parity where the carried state dominates the output.

The five workloads draw exp(A_log) in [1, 16], so every channel forgets within
a few tokens and resetting the state at each chunk start moves their output by
only a few percent.  The regimes here (``inputs.STATE_REGIMES``: slow decay
through the gate, slow or no decay given directly, beta at 0, 1e-3 and 1,
keys along one direction, zero q/k rows, an initial state) make the state
carried across chunks most of the output: with the oracle, resetting it at
every chunk start moves the output by 44-97 % (beta = 1 along one direction,
where each write overwrites the last, by 3.5 %; beta = 0 writes nothing).

Every forward path of the library runs each regime against the FP64 oracle
("Add opt-in FP32 KDA chunk computation", section Validation: an independent
FP64 recurrence as the reference): FP32-exact mode in its single-pass kernel
and in two phases (rel-L2 <= 1e-5, F32 output), and the BF16 tensor-core path
(<= 3e-3, BF16 output) in two phases with a workspace (8192 tokens: three chunk
windows with the FP32 state carry between them), in the single-pass kernel,
and on the static scratch of kda_chunk_fwd_static (one window).  Output and
final state are both checked.
"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_10_gb300 import (kda_chunk_fwd, kda_chunk_fwd_static, kda_gate)
from kimi_delta_attention_10_gb300.binding import KDA_ERR_RANGE
from kimi_delta_attention_10_gb300.inputs import STATE_REGIMES, state_regime_inputs

from gpu_util import f64, rel_l2

pytestmark = pytest.mark.gpu

H = 4
# one sequence of 128 chunks (three windows), and three sequences across windows
LAYOUTS = {"single_8192": [8192], "packed_5000_3000_192": [5000, 3000, 192]}
PATHS = ("fp32_exact", "fp32_two_phase", "two_phase", "single_pass", "static")
TOL = {"fp32_exact": 1e-5, "fp32_two_phase": 1e-5, "two_phase": 3e-3, "single_pass": 3e-3,
       "static": 3e-3}

_inputs, _refs = {}, {}


def regime(name, layout):
    key = (name, layout)
    if key not in _inputs:
        _inputs[key] = state_regime_inputs(name, LAYOUTS[layout], H=H, seed=len(_inputs) + 11)
    return _inputs[key]


def oracle_ref(name, layout):
    """FP64 oracle: gate from the raw draws, or the given g and beta upcast."""
    key = (name, layout)
    if key not in _refs:
        ri = regime(name, layout)
        x = ri.x
        if ri.g is None:
            g, beta = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
        else:
            g, beta = f64(ri.g), f64(ri.beta)
        init = None if ri.initial_state is None else f64(ri.initial_state)
        _refs[key] = oracle.forward(f64(x.q), f64(x.k), f64(x.v), g, beta,
                                    x.cu_seqlens.numpy(), x.scale, initial_state=init)
    return _refs[key]


def run_gpu(ri, path, v_override=None):
    """One forward call of `path`; returns (out, final_state, status) on the CPU."""
    x = ri.x
    dev = "cuda"
    q, k = x.q.to(dev), x.k.to(dev)
    v = (x.v if v_override is None else v_override).to(dev)
    cu = x.cu_seqlens.to(dev)
    if ri.g is None:
        g, beta = kda_gate(x.f.to(dev), x.A_log.to(dev), x.dt_bias.to(dev), x.b.to(dev))
    else:
        g, beta = ri.g.to(dev), ri.beta.to(dev)
    init = None if ri.initial_state is None else ri.initial_state.to(dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    if path == "static":
        out = torch.empty(x.T, H, 128, dtype=v.dtype, device=dev)
        S = torch.empty(x.N, H, 128, 128, device=dev)
        kda_chunk_fwd_static(q, k, v, g, beta, cu, out, x.scale, initial_state=init,
                             final_state=S, status=status)
    else:
        kw = {"fp32_exact": dict(mode="fp32_exact", workspace=None, out_dtype=torch.float32),
              "fp32_two_phase": dict(mode="fp32_exact", workspace="auto", out_dtype=torch.float32),
              "two_phase": dict(mode="bf16_tc", workspace="auto"),
              "single_pass": dict(mode="bf16_tc", workspace=None)}[path]
        out, S = kda_chunk_fwd(q, k, v, g, beta, cu, x.scale, initial_state=init,
                               cu_seqlens_host=x.cu_seqlens.tolist(), status=status, **kw)
    torch.cuda.synchronize()
    return out.cpu(), S.cpu(), int(status[0])


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("name", STATE_REGIMES)
def test_state_regime_matches_oracle(name, layout, path):
    ri = regime(name, layout)
    o_ref, S_ref = oracle_ref(name, layout)
    out, S, status = run_gpu(ri, path)
    assert status == 0
    o_gpu, S_gpu = out.double().numpy(), S.double().numpy()
    assert np.isfinite(o_gpu).all() and np.isfinite(S_gpu).all()
    if name == "beta_zero":
        # nothing is written and the state starts at zero: exactly zero
        assert not np.any(o_ref) and not np.any(S_ref)
        assert not np.any(o_gpu) and not np.any(S_gpu)
        return
    e_o, e_S = rel_l2(o_gpu, o_ref), rel_l2(S_gpu, S_ref)
    print(f"{name} {layout} {path}: out rel-L2 {e_o:.3e}, final state rel-L2 {e_S:.3e}")
    assert e_o <= TOL[path] and e_S <= TOL[path]
    if name == "zero_qk_rows":
        # a zero query reads nothing: those output rows are exactly zero
        assert not np.any(o_gpu[3::7])


@pytest.mark.parametrize("path", PATHS)
def test_values_near_the_fp16_limit_pass_or_are_reported(path):
    """|v| up to 6e4 (just inside FP16): the tensor-core paths either match the
    oracle or report KDA_ERR_RANGE through the status word, never a silent
    infinity; the FP32 path matches."""
    ri = regime("alog_0.05", "single_8192")
    x = ri.x
    v = x.v.float()
    v = (v * (6.0e4 / float(v.abs().max()))).to(x.v.dtype)
    g, beta = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    o_ref, S_ref = oracle.forward(f64(x.q), f64(x.k), f64(v), g, beta, x.cu_seqlens.numpy(),
                                  x.scale)
    out, S, status = run_gpu(ri, path, v_override=v)
    o_gpu, S_gpu = out.double().numpy(), S.double().numpy()
    finite = np.isfinite(o_gpu).all() and np.isfinite(S_gpu).all()
    print(f"{path}: status {status}, finite {finite}")
    if path.startswith("fp32"):
        assert status == 0 and finite
    if status == 0:
        assert finite
        assert rel_l2(o_gpu, o_ref) <= TOL[path] and rel_l2(S_gpu, S_ref) <= TOL[path]
    else:
        assert status == KDA_ERR_RANGE


@pytest.mark.parametrize("path", ["two_phase", "single_pass", "static"])
def test_values_beyond_fp16_are_reported(path):
    """|v| about 1e5 does not fit FP16: the tensor-core paths must say so."""
    ri = regime("alog_0.05", "packed_5000_3000_192")
    v = (ri.x.v.float() * 3.0e4).to(ri.x.v.dtype)
    _, _, status = run_gpu(ri, path, v_override=v)
    assert status == KDA_ERR_RANGE


@pytest.mark.parametrize("path", ["fp32_exact", "fp32_two_phase"])
def test_fp32_paths_keep_fp32_range(path):
    """|v| about 1e5, beyond FP16: the FP32-exact paths still match the oracle.
    The two-phase path's tensor-core scan holds the state and Delta as FP16
    pairs scaled per chunk by a power of two, so FP16's range does not apply."""
    ri = regime("alog_0.05", "packed_5000_3000_192")
    x = ri.x
    v = (x.v.float() * 3.0e4).to(x.v.dtype)
    g, beta = oracle.gate(f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b))
    o_ref, S_ref = oracle.forward(f64(x.q), f64(x.k), f64(v), g, beta, x.cu_seqlens.numpy(),
                                  x.scale)
    out, S, status = run_gpu(ri, path, v_override=v)
    assert status == 0
    e_o, e_S = rel_l2(out.double().numpy(), o_ref), rel_l2(S.double().numpy(), S_ref)
    print(f"{path} |v| ~ 1e5: out rel-L2 {e_o:.3e}, final state rel-L2 {e_S:.3e}")
    assert e_o <= TOL[path] and e_S <= TOL[path]
