"""GPU parity of kda_gated_rmsnorm (output gate with gated RMSNorm) against the
FP64 oracle, elementwise, and of the whole forward followed by the gate."""
import numpy as np
import pytest
import torch

from oracle.output_gate import gated_rmsnorm
from kimi_delta_attention_10_gb300 import kda_chunk_fwd, kda_gate, kda_gated_rmsnorm
from kimi_delta_attention_10_gb300.inputs import make_inputs

from gpu_util import device_inputs, oracle_pipeline, rel_l2

pytestmark = pytest.mark.gpu


def _draw(rows, seed, dtype):
    gen = torch.Generator().manual_seed(seed)
    o = torch.randn(rows, 128, generator=gen).to(dtype)
    z = (torch.randn(rows, 128, generator=gen) * 2).to(dtype)
    w = torch.rand(128, generator=gen) + 0.5
    return o, z, w


def _ref(o, z, w, eps):
    f = lambda t: t.double().numpy()
    return gated_rmsnorm(f(o), f(z), f(w), eps)


@pytest.mark.parametrize("rows", [1, 37, 4096 + 5])
def test_fp32_matches_oracle_elementwise(rows):
    o, z, w = _draw(rows, 71 + rows, torch.float32)
    y = kda_gated_rmsnorm(o.cuda(), z.cuda(), w.cuda(), eps=1e-6)
    ref = _ref(o, z, w, 1e-6)
    err = np.abs(y.cpu().double().numpy() - ref) / np.maximum(np.abs(ref), 1e-30)
    assert err.max() <= 2e-6


@pytest.mark.parametrize("odt,zdt,ydt", [(torch.bfloat16, torch.bfloat16, torch.bfloat16),
                                         (torch.bfloat16, torch.float32, torch.float32),
                                         (torch.float32, torch.bfloat16, torch.bfloat16)])
def test_mixed_dtypes_match_oracle(odt, zdt, ydt):
    o, z, w = _draw(1000, 72, torch.float32)
    o, z = o.to(odt), z.to(zdt)
    y = kda_gated_rmsnorm(o.cuda(), z.cuda(), w.cuda(), eps=1e-5, out_dtype=ydt)
    assert y.dtype == ydt
    ref = _ref(o, z, w, 1e-5)
    err = np.abs(y.cpu().double().numpy() - ref) / np.maximum(np.abs(ref), 1e-30)
    # BF16 output rounding is at most 2^-9 relative; FP32 output as above
    assert err.max() <= (2.0 ** -8 if ydt == torch.bfloat16 else 2e-6)


def test_in_place_and_zero_rows():
    o, z, w = _draw(64, 73, torch.bfloat16)
    o[5] = 0
    od, zd, wd = o.cuda(), z.cuda(), w.cuda()
    y = kda_gated_rmsnorm(od, zd, wd, eps=1e-6)
    kda_gated_rmsnorm(od, zd, wd, eps=1e-6, out=od)
    torch.cuda.synchronize()
    assert torch.equal(od, y)
    assert torch.count_nonzero(y[5]) == 0
    empty = torch.empty(0, 128, device="cuda")
    assert kda_gated_rmsnorm(empty, empty, wd).numel() == 0


@pytest.mark.parametrize("mode", ["bf16_tc", "fp32_exact"])
def test_forward_then_output_gate_matches_oracle(mode):
    """The chunked forward followed by the output gate, against the FP64
    recurrence followed by the FP64 gated RMSNorm."""
    x = make_inputs([100, 37], 4, 128, 128, torch.bfloat16, 74)
    gen = torch.Generator().manual_seed(74)
    zg = torch.randn(x.T, 4, 128, generator=gen).to(torch.bfloat16)
    w = torch.rand(128, generator=gen) + 0.5
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    o, _ = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale, mode=mode,
                         out_dtype=torch.float32 if mode == "fp32_exact" else None)
    y = kda_gated_rmsnorm(o, zg.cuda(), w.cuda(), eps=1e-6, out_dtype=torch.float32)
    o_ref, _, _, _ = oracle_pipeline(x)
    y_ref = gated_rmsnorm(o_ref, zg.double().numpy(), w.double().numpy(), 1e-6)
    assert rel_l2(y.cpu().double().numpy(), y_ref) <= (1e-5 if mode == "fp32_exact" else 3e-3)
