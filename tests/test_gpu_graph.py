"""The forward (with its chunk windows and programmatic dependent launches)
and the backward captured in CUDA graphs: replays give the bits of eager
calls.  Buffers and workspaces are allocated before capture; the calls
allocate nothing."""
import pytest
import torch

from kimi_delta_attention_10_gb300 import (chunk_bwd_workspace_size, chunk_workspace_size,
                                           kda_chunk_bwd, kda_chunk_fwd_gated)
from kimi_delta_attention_10_gb300.inputs import make_cotangents, make_inputs

from gpu_util import device_inputs

pytestmark = pytest.mark.gpu


def test_fused_forward_in_a_graph_is_bitwise_eager():
    x = make_inputs([16384], 2, 128, 128, torch.bfloat16, 101)    # three chunk windows
    d = device_inputs(x)
    host = x.cu_seqlens.tolist()
    ws = torch.empty(chunk_workspace_size(x.N, x.T, x.H), dtype=torch.uint8, device="cuda")
    out = torch.empty(x.T, x.H, 128, dtype=torch.bfloat16, device="cuda")
    fs = torch.empty(x.N, x.H, 128, 128, device="cuda")

    def call():
        kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"], d["b"],
                            d["cu_seqlens"], x.scale, out=out, final_state=fs,
                            cu_seqlens_host=host, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                                   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref_out, ref_fs = out.clone(), fs.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    out.zero_()
    fs.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fs, ref_fs)


def test_backward_in_a_graph_is_bitwise_eager():
    x = make_inputs([300, 77], 3, 128, 128, torch.float32, 102)
    d = device_inputs(x)
    gen = torch.Generator().manual_seed(102)
    g = (-torch.rand(x.T, x.H, 128, generator=gen) * 0.5).cuda()
    beta = torch.rand(x.T, x.H, generator=gen).cuda()
    dO, dfin, _ = make_cotangents(x.T, x.N, x.H, 128, 128, 102)
    dO, dfin = dO.cuda(), dfin.cuda()
    ws = torch.empty(chunk_bwd_workspace_size(x.N, x.T, x.H), dtype=torch.uint8, device="cuda")
    host = x.cu_seqlens.tolist()
    res = {}

    def call():
        res["g"] = kda_chunk_bwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], dO, x.scale,
                                 dfinal_state=dfin, cu_seqlens_host=host, workspace=ws)

    call()
    torch.cuda.synchronize()
    ref = [t.clone() for t in res["g"]]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()                                   # outputs allocated in the graph's pool
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(res["g"], ref):
        assert torch.equal(a, b)
