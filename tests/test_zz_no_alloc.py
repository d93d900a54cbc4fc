"""kda_chunk_fwd_static (the two-phase tensor-core path on the library's own
static scratch, no allocation) against kda_chunk_fwd with a caller workspace.

Collected last (file name) and independent of the other tests: it must pass
alone and after them."""
import pytest
import torch

from kimi_delta_attention_10_gb300 import (KDAError, kda_chunk_fwd, kda_chunk_fwd_static,
                                           kda_gate)
from kimi_delta_attention_10_gb300.binding import KDA_ERR_TOO_LARGE
from kimi_delta_attention_10_gb300.inputs import make_inputs

from gpu_util import device_inputs

pytestmark = pytest.mark.gpu


def _case(lens, H, seed, dtype=torch.bfloat16):
    x = make_inputs(lens, H, 128, 128, dtype, seed)
    d = device_inputs(x)
    g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
    return x, d, g, beta


def test_static_scratch_equals_workspace_path_on_two_calls_in_a_row():
    """Two calls in a row (the second smaller, so stale scratch from the first
    is present): each equals the workspace entry point bit for bit."""
    cases = [([200, 37, 64], 8, 51, torch.bfloat16), ([5, 130], 4, 52, torch.float32)]
    for lens, H, seed, dtype in cases:
        x, d, g, beta = _case(lens, H, seed, dtype)
        o_ref, S_ref = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale,
                                     mode="bf16_tc", workspace="auto",
                                     cu_seqlens_host=x.cu_seqlens.tolist())
        out = torch.full_like(o_ref, float("nan"))
        S = torch.full_like(S_ref, float("nan"))
        kda_chunk_fwd_static(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], out, x.scale,
                             final_state=S)
        torch.cuda.synchronize()
        assert torch.equal(out, o_ref) and torch.equal(S, S_ref), (lens, H)


def test_static_scratch_rejects_problems_over_its_size():
    # H = 64: (T / 64 + N) * H records of 74240 bytes exceed 64 MiB at 1024 tokens
    x, d, g, beta = _case([1024], 64, 53)
    out = torch.zeros(x.T, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KDAError) as e:
        kda_chunk_fwd_static(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], out, x.scale)
    assert e.value.status == KDA_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0          # nothing was launched
