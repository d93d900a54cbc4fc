"""Seeded synthetic inputs for the KDA forward (workload recipes only).

This module draws random tensors and nothing else: it holds none of the
method's arithmetic (no gate, no normalisation, no recurrence), so that the
CUDA path and the FP64 oracle can both consume its output without sharing
any computation.

Workloads follow the geometry the XTuner pages test and time KDA on
("Add opt-in FP32 KDA chunk computation", section Validation: packed
lengths 37/28, a chunk boundary at 129 tokens, 64 heads x 128 dims, and
the 129/2048/16384-token CUDA-graph timings), with a packed 32768-token
batch of random lengths as the varlen stress case.

Draw order, all from one CPU ``torch.Generator`` seeded per workload:
(random sequence lengths, packed workload only) -> q -> k -> v -> f ->
A_log -> dt_bias -> b.  Every tensor is drawn in FP32; q/k/v are then
rounded to the workload's activation dtype.

Distributions: q, k, v, f, b ~ N(0, 1); A_log ~ U(0, ln 16) per head;
dt_bias ~ N(0, 0.5^2) per (head, channel).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

H_DEFAULT = 64
K_DEFAULT = 128
V_DEFAULT = 128


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    qkv_dtype: torch.dtype
    seqlens: Optional[List[int]] = None      # None -> drawn (packed random lengths)
    total_tokens: int = 0                     # used when seqlens is None
    max_len: int = 0                          # used when seqlens is None
    final_state: bool = False
    H: int = H_DEFAULT
    K: int = K_DEFAULT
    V: int = V_DEFAULT


WORKLOADS: List[Workload] = [
    Workload("packed_37_28_f32", seed=0, qkv_dtype=torch.float32, seqlens=[37, 28],
             final_state=True),
    Workload("single_129_bf16", seed=1, qkv_dtype=torch.bfloat16, seqlens=[129],
             final_state=True),
    Workload("single_2048_bf16", seed=2, qkv_dtype=torch.bfloat16, seqlens=[2048],
             final_state=True),
    Workload("single_16384_bf16", seed=3, qkv_dtype=torch.bfloat16, seqlens=[16384],
             final_state=True),
    Workload("packed_32768_bf16", seed=4, qkv_dtype=torch.bfloat16, seqlens=None,
             total_tokens=32768, max_len=4096, final_state=True),
]

WORKLOAD_BY_NAME: Dict[str, Workload] = {w.name: w for w in WORKLOADS}


def draw_packed_lengths(gen: torch.Generator, total: int, max_len: int) -> List[int]:
    """Integers uniform in [1, max_len], drawn one at a time until their sum
    reaches ``total``; the last one is cut so that the sum is exactly ``total``."""
    lens: List[int] = []
    acc = 0
    while acc < total:
        n = int(torch.randint(1, max_len + 1, (1,), generator=gen).item())
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


@dataclass
class KDAInputs:
    """CPU tensors for one forward call, in the library's layout.

    q, k: [T, H, K]; v: [T, H, V] (activation dtype); f: [T, H, K] FP32 gate
    pre-activation; A_log: [H] FP32; dt_bias: [H, K] FP32; b: [T, H] FP32 beta
    logits; cu_seqlens: [N+1] int32 packed offsets.
    """
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    f: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    b: torch.Tensor
    cu_seqlens: torch.Tensor
    scale: float
    seqlens: List[int] = field(default_factory=list)

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.numel() - 1)


def make_inputs(seqlens: List[int], H: int, K: int, V: int, qkv_dtype: torch.dtype,
                seed: int, gen: Optional[torch.Generator] = None) -> KDAInputs:
    """Draw one input set for the given packed lengths (see the module doc)."""
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    T = int(sum(seqlens))
    q = torch.randn(T, H, K, generator=gen, dtype=torch.float32)
    k = torch.randn(T, H, K, generator=gen, dtype=torch.float32)
    v = torch.randn(T, H, V, generator=gen, dtype=torch.float32)
    f = torch.randn(T, H, K, generator=gen, dtype=torch.float32)
    A_log = torch.rand(H, generator=gen, dtype=torch.float32) * math.log(16.0)
    dt_bias = torch.randn(H, K, generator=gen, dtype=torch.float32) * 0.5
    b = torch.randn(T, H, generator=gen, dtype=torch.float32)
    cu = torch.zeros(len(seqlens) + 1, dtype=torch.int32)
    if seqlens:
        cu[1:] = torch.cumsum(torch.tensor(seqlens, dtype=torch.int64), 0).to(torch.int32)
    return KDAInputs(q=q.to(qkv_dtype), k=k.to(qkv_dtype), v=v.to(qkv_dtype), f=f,
                     A_log=A_log, dt_bias=dt_bias, b=b, cu_seqlens=cu,
                     scale=1.0 / math.sqrt(K), seqlens=list(seqlens))


def workload_inputs(w: Workload | str | int) -> KDAInputs:
    """Inputs of one named workload (by object, name or index)."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    elif isinstance(w, str):
        w = WORKLOAD_BY_NAME[w]
    gen = torch.Generator().manual_seed(w.seed)
    seqlens = w.seqlens if w.seqlens is not None else draw_packed_lengths(
        gen, w.total_tokens, w.max_len)
    return make_inputs(seqlens, w.H, w.K, w.V, w.qkv_dtype, w.seed, gen=gen)


def workload_seqlens(w: Workload | str | int) -> List[int]:
    """Sequence lengths of a workload without drawing its tensors."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    elif isinstance(w, str):
        w = WORKLOAD_BY_NAME[w]
    if w.seqlens is not None:
        return list(w.seqlens)
    gen = torch.Generator().manual_seed(w.seed)
    return draw_packed_lengths(gen, w.total_tokens, w.max_len)


def make_cotangents(T: int, N: int, H: int, K: int, V: int, seed: int,
                    dout_dtype: torch.dtype = torch.float32):
    """Seeded draws for a backward call: dout [T,H,V] ~ N(0,1) in ``dout_dtype``,
    dfinal_state [N,H,K,V] ~ N(0,1) and initial_state [N,H,K,V] ~ N(0, 0.5^2),
    both FP32, in that order from one generator."""
    gen = torch.Generator().manual_seed(seed)
    dout = torch.randn(T, H, V, generator=gen, dtype=torch.float32).to(dout_dtype)
    dfinal = torch.randn(N, H, K, V, generator=gen, dtype=torch.float32)
    init = torch.randn(N, H, K, V, generator=gen, dtype=torch.float32) * 0.5
    return dout, dfinal, init
