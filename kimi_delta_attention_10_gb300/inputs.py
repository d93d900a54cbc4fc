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


# Regimes in which the state carried from chunk to chunk dominates the output
# (the workloads above forget within a few tokens: mean g is about -4 per token).
STATE_REGIMES = ("alog_0.01", "alog_0.05", "g_slow", "g_zero_beta_small", "g_zero",
                 "beta_zero", "beta_one_direction", "zero_qk_rows", "initial_state")


@dataclass
class RegimeInputs:
    """One input set of a state regime.

    ``x`` holds q, k, v and the gate pre-activations.  When ``g`` and ``beta``
    are given ([T,H,K] and [T,H] FP32), they are the decay and write strength
    fed to the chunk forward directly, and the pre-activations are unused;
    otherwise both sides form them from the pre-activations.  ``initial_state``
    is [N,H,K,V] FP32 or None (zero)."""
    x: KDAInputs
    g: Optional[torch.Tensor] = None
    beta: Optional[torch.Tensor] = None
    initial_state: Optional[torch.Tensor] = None


def state_regime_inputs(regime: str, seqlens: List[int], H: int = 4,
                        qkv_dtype: torch.dtype = torch.bfloat16, seed: int = 0) -> RegimeInputs:
    """Seeded draws of one state regime (q, k, v, f, b as in ``make_inputs``,
    then the regime's own draws from a second generator seeded 1000 + seed):

    alog_0.01, alog_0.05  exp(A_log) = 0.01 or 0.05 for every head: slow decay
                          through the gate (g about -0.007 or -0.035 per token)
    g_slow                g ~ U(-0.05, 0) per element, beta ~ U(0, 1)
    g_zero_beta_small     g = 0, beta = 1e-3 (the linear-attention limit)
    g_zero                g = 0, beta ~ U(0, 1) (delta rule without decay)
    beta_zero             g ~ U(-0.05, 0), beta = 0 (nothing is ever written)
    beta_one_direction    g ~ U(-0.05, 0), beta = 1, every key of a head along
                          one direction u_h ~ N(0, I) with an N(0, 1) length
                          (the delta rule overwrites)
    zero_qk_rows          exp(A_log) = 0.05, q rows t % 7 == 3 and k rows
                          t % 5 == 1 set to zero
    initial_state         exp(A_log) = 0.05, initial state ~ N(0, 0.3^2)
    """
    K = V = 128
    x = make_inputs(seqlens, H, K, V, qkv_dtype, seed)
    gen = torch.Generator().manual_seed(1000 + seed)
    T, N = x.T, x.N
    r = RegimeInputs(x=x)
    slow_g = lambda: -0.05 * torch.rand(T, H, K, generator=gen, dtype=torch.float32)
    if regime in ("alog_0.01", "alog_0.05"):
        x.A_log = torch.full((H,), math.log(float(regime.split("_")[1])), dtype=torch.float32)
    elif regime == "g_slow":
        r.g = slow_g()
        r.beta = torch.rand(T, H, generator=gen, dtype=torch.float32)
    elif regime == "g_zero_beta_small":
        r.g = torch.zeros(T, H, K)
        r.beta = torch.full((T, H), 1e-3, dtype=torch.float32)
    elif regime == "g_zero":
        r.g = torch.zeros(T, H, K)
        r.beta = torch.rand(T, H, generator=gen, dtype=torch.float32)
    elif regime == "beta_zero":
        r.g = slow_g()
        r.beta = torch.zeros(T, H)
    elif regime == "beta_one_direction":
        r.g = slow_g()
        r.beta = torch.ones(T, H)
        u = torch.randn(H, K, generator=gen, dtype=torch.float32)
        length = torch.randn(T, H, 1, generator=gen, dtype=torch.float32)
        x.k = (length * u).to(qkv_dtype)
    elif regime == "zero_qk_rows":
        x.A_log = torch.full((H,), math.log(0.05), dtype=torch.float32)
        x.q[3::7] = 0
        x.k[1::5] = 0
    elif regime == "initial_state":
        x.A_log = torch.full((H,), math.log(0.05), dtype=torch.float32)
        r.initial_state = 0.3 * torch.randn(N, H, K, V, generator=gen, dtype=torch.float32)
    else:
        raise KeyError(regime)
    return r
