"""bench.py host logic on the CPU: the multi-rank reduction (gloo, world size 2),
the whole-job rate, the reference arm's JSON line, the head subset and the traffic lookup."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [12.5, 40.0][rank]
        out[rank] = bench.max_over_ranks(per_rank_ms, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 40.0, 1: 40.0}


def test_max_over_ranks_without_group():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25


def test_whole_job_rate_is_weak_scaling():
    # 2 ranks x 16384 tokens x 10 steps in 1 s
    assert bench.whole_job_rate(2, 16384, 10, 1000.0) == pytest.approx(327680.0)


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_json_line():
    r = _run_bench(["--impl", "reference", "--workload", "packed_37_28_f32", "--steps", "2",
                    "--warmup", "1"], {"RANK": "0"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "packed_37_28_f32"


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--workload", "packed_37_28_f32", "--steps", "1",
                    "--warmup", "0"], {"RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_chunk_windows_rule():
    """Windows only when the scan leaves SMs idle and there are >= 64 chunks."""
    assert bench.chunk_windows(1, 64, 256, 152) == 3          # 16384 tokens x 64 heads
    assert bench.chunk_windows(1, 64, 32, 152) == 1           # 2048 tokens: one window
    assert bench.chunk_windows(16, 64, 520, 152) == 1         # 1024 scan CTAs fill the GPU
    assert bench.chunk_windows(1, 2, 66, 152) == 2


def test_chunk_windows_mirror_matches_the_library_constants():
    """bench.chunk_windows restates the window rule of kda_chunk_split.cu
    (min(kMaxWindows, chunks / kWindowChunks) when N * H <= the SM count)."""
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "kimi_delta_attention_10_gb300", "csrc", "kda_chunk_split.cu")).read()
    max_w = int(re.search(r"constexpr int kMaxWindows = (\d+);", src).group(1))
    per_w = int(re.search(r"constexpr int kWindowChunks = (\d+);", src).group(1))
    assert ("const int64_t W_shape = heads <= sms ? std::min<int64_t>(kMaxWindows, chunks / "
            "kWindowChunks) : 1;") in src
    for chunks in (0, 31, 32, 63, 64, 100, 256, 10000):
        assert bench.chunk_windows(1, 64, chunks, 152) == max(1, min(max_w, chunks // per_w))
    assert bench.chunk_windows(3, 64, 10000, 152) == 1


def test_first_heads_keeps_the_leading_heads():
    from kimi_delta_attention_10_gb300.inputs import make_inputs
    full = make_inputs([70, 5], 6, 128, 128, torch.bfloat16, 3)
    ref = make_inputs([70, 5], 6, 128, 128, torch.bfloat16, 3)
    x = bench.first_heads(full, 4)
    for n in ("q", "k", "v", "f"):
        assert getattr(x, n).shape == (75, 4, 128) and getattr(x, n).is_contiguous()
        assert torch.equal(getattr(x, n), getattr(ref, n)[:, :4])
    assert torch.equal(x.b, ref.b[:, :4]) and x.b.is_contiguous()
    assert torch.equal(x.A_log, ref.A_log[:4]) and torch.equal(x.dt_bias, ref.dt_bias[:4])
    assert torch.equal(x.cu_seqlens, ref.cu_seqlens)


def test_kernel_traffic_only_while_the_sources_match(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1")
    import hashlib
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"key": {"sources": ["k.cu"], "sources_sha256_16": sha, "dram_bytes_per_call": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("key") == 1234
    assert bench.kernel_traffic("other") is None
    src.write_bytes(b"kernel v2")                    # changed since the capture
    assert bench.kernel_traffic("key") is None
