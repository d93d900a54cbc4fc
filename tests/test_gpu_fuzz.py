"""Seeded random configurations across the forward's API surface, each against
the FP64 oracle: packed lengths drawn from a mix of chunk-edge and free
values, 1-6 heads, BF16 or FP32 activations, every chunk path (two-phase and
single-pass, both modes), the gate separate or fused (f and the beta logits
in FP32 or BF16), with or without an initial state, FP32 or BF16 output.  Four
of the cases hold one sequence long enough for the two-phase path to cut it
into chunk windows.  Each call also reports a clean status word."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import OUT_DTYPE, PATHS, device_inputs, f64, path_kw, rel_l2, tol
from kimi_delta_attention_10_gb300 import kda_chunk_fwd, kda_chunk_fwd_gated, kda_gate
from kimi_delta_attention_10_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = (0, 1, 2, 63, 64, 65, 127, 128, 129)
N_CASES = 48
LONG = {3: "bf16_tc", 11: "fp32_exact_2p", 27: "bf16_tc", 40: "fp32_exact_2p"}


def draw_case(seed: int) -> dict:
    gen = torch.Generator().manual_seed(9000 + seed)
    pick = lambda seq: seq[int(torch.randint(0, len(seq), (1,), generator=gen))]
    if seed in LONG:                        # one long sequence: chunk windows
        lens = [int(torch.randint(4100, 6000, (1,), generator=gen))]
        H = 2
    else:
        n = int(torch.randint(1, 25, (1,), generator=gen))
        lens = []
        for _ in range(n):
            if float(torch.rand(1, generator=gen)) < 0.5:
                lens.append(pick(EDGE_LENGTHS))
            else:
                lens.append(int(torch.randint(1, 601, (1,), generator=gen)))
        if sum(lens) == 0:
            lens[0] = 1
        H = pick((1, 2, 3, 4, 6))
    path = LONG.get(seed) or pick(tuple(PATHS))
    fused = pick((False, True))
    return dict(
        lens=lens, H=H, path=path, fused=fused,
        qkv=pick((torch.bfloat16, torch.float32)),
        f_bf16=fused and pick((False, True)),
        b_bf16=fused and pick((False, True)),
        init=pick((False, True)),
        out_bf16=OUT_DTYPE[path] is None and pick((False, True)),
        seed=100 + seed)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration_matches_oracle(seed):
    c = draw_case(seed)
    x = make_inputs(c["lens"], c["H"], 128, 128, c["qkv"], c["seed"])
    N = len(c["lens"])
    # the values the library sees: 16-bit copies of f and b where it reads them so
    if c["f_bf16"]:
        x.f = x.f.to(torch.bfloat16).float()
    if c["b_bf16"]:
        x.b = x.b.to(torch.bfloat16).float()
    S0 = None
    if c["init"]:
        S0 = torch.randn(N, c["H"], 128, 128, generator=torch.Generator().manual_seed(c["seed"])) * 0.3
    d = device_inputs(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_dtype = torch.bfloat16 if c["out_bf16"] else torch.float32
    kw = dict(out_dtype=out_dtype, initial_state=None if S0 is None else S0.cuda(),
              cu_seqlens_host=x.cu_seqlens.tolist(), status=status, **path_kw(c["path"]))
    if c["fused"]:
        f = d["f"].to(torch.bfloat16) if c["f_bf16"] else d["f"]
        b = d["b"].to(torch.bfloat16) if c["b_bf16"] else d["b"]
        out, S = kda_chunk_fwd_gated(d["q"], d["k"], d["v"], f, d["A_log"], d["dt_bias"], b,
                                     d["cu_seqlens"], x.scale, **kw)
    else:
        g, beta = kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"])
        out, S = kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, c
    o_ref, S_ref, _, _ = oracle.reference(
        f64(x.q), f64(x.k), f64(x.v), f64(x.f), f64(x.A_log), f64(x.dt_bias), f64(x.b),
        x.cu_seqlens.numpy(), x.scale, initial_state=None if S0 is None else S0.double().numpy())
    o, Sg = out.float().cpu().numpy(), S.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(Sg).all(), c
    e_o, e_S = rel_l2(o, o_ref), rel_l2(Sg, S_ref)
    assert e_o <= tol(c["path"]) and e_S <= tol(c["path"]), (c, e_o, e_S)
