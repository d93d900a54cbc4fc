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


# ---------------------------------------------------------------- fused forward + gate
FUSED_CASES = {"packed_edges": ([1, 64, 0, 130, 77], 4), "single_2048": ([2048], 64),
               "single_8192_windows": ([8192], 2)}


def _fused_case(lens, H, seed, zdt):
    x = make_inputs(lens, H, 128, 128, torch.bfloat16, seed)
    x.f = x.f.to(torch.bfloat16)
    gen = torch.Generator().manual_seed(seed + 500)
    z = (torch.randn(x.T, H, 128, generator=gen) * 2).to(zdt)
    w = torch.rand(128, generator=gen) + 0.5
    return x, z, w


@pytest.mark.parametrize("path", ["two_phase", "single_pass", "fp32_exact", "fp32_two_phase"])
@pytest.mark.parametrize("case", list(FUSED_CASES))
@pytest.mark.parametrize("zdt", [torch.bfloat16, torch.float32])
def test_forward_with_output_gate_matches_oracle(case, path, zdt):
    """kda_chunk_fwd_gated_norm against the FP64 forward followed by the FP64
    gate.  Two-phase with BF16 z is the fused scan epilogue (its o rows never
    reach memory); the other paths run the forward and the gate kernel."""
    from kimi_delta_attention_10_gb300 import kda_chunk_fwd_gated_norm
    lens, H = FUSED_CASES[case]
    x, z, w = _fused_case(lens, H, 31 + len(lens), zdt)
    d = device_inputs(x)
    kw = {"two_phase": dict(mode="bf16_tc", workspace="auto"),
          "single_pass": dict(mode="bf16_tc", workspace=None),
          "fp32_exact": dict(mode="fp32_exact", workspace=None, out_dtype=torch.float32),
          "fp32_two_phase": dict(mode="fp32_exact", workspace="auto",
                                 out_dtype=torch.float32)}[path]
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y, S = kda_chunk_fwd_gated_norm(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                    d["b"], d["cu_seqlens"], z.cuda(), w.cuda(), x.scale,
                                    eps=1e-6, cu_seqlens_host=x.cu_seqlens.tolist(),
                                    status=status, **kw)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    o_ref, S_ref, _, _ = oracle_pipeline(x)
    f = lambda t: t.float().double().numpy()
    y_ref = gated_rmsnorm(o_ref, f(z), f(w), 1e-6)
    tol = 1e-5 if path.startswith("fp32") else 3e-3
    e_y, e_S = rel_l2(y.cpu().float().double().numpy(), y_ref), rel_l2(S.cpu().double().numpy(), S_ref)
    print(f"{case} {path} z={zdt}: y rel-L2 {e_y:.3e}, final state rel-L2 {e_S:.3e}")
    assert np.isfinite(y.cpu().float().numpy()).all()
    assert e_y <= tol and e_S <= tol


def test_fused_output_gate_leaves_the_state_path_unchanged():
    """The fused epilogue changes only what is stored for the output: the final
    state is the bits of kda_chunk_fwd_gated's."""
    from kimi_delta_attention_10_gb300 import kda_chunk_fwd_gated, kda_chunk_fwd_gated_norm
    x, z, w = _fused_case([8192], 2, 41, torch.bfloat16)
    d = device_inputs(x)
    args = (d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"], d["b"], d["cu_seqlens"])
    host = x.cu_seqlens.tolist()
    o1, S1 = kda_chunk_fwd_gated(*args, x.scale, workspace="auto", cu_seqlens_host=host)
    y2, S2 = kda_chunk_fwd_gated_norm(*args, z.cuda(), w.cuda(), x.scale, eps=1e-6,
                                      workspace="auto", cu_seqlens_host=host)
    y3 = kda_gated_rmsnorm(o1, z.cuda(), w.cuda(), eps=1e-6)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2)
    # the unfused gate reads o rounded to BF16, the fused one its FP32 value
    f = lambda t: t.float().cpu().double().numpy()
    assert rel_l2(f(y2), f(y3)) <= 3e-3


def test_fused_output_gate_rejects_z_aliasing_out():
    from kimi_delta_attention_10_gb300 import KDAError, kda_chunk_fwd_gated_norm
    x, z, w = _fused_case([70], 2, 43, torch.bfloat16)
    d = device_inputs(x)
    zc = z.cuda()
    with pytest.raises(KDAError):
        kda_chunk_fwd_gated_norm(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                 d["b"], d["cu_seqlens"], zc, w.cuda(), x.scale, out=zc)
