"""FP64 chunked (WY) form of the KDA forward -- TEST INFRASTRUCTURE ONLY.

A second algorithm for the same result as the token loop in ``kda_oracle.c``.
The pages call the training kernel's intermediates "chunk solve/state
intermediates" ("Add opt-in FP32 KDA chunk computation", sections Problem and
Change); this module writes that chunk solve out in plain FP64 NumPy so that
the tests can check the algebra against the token recurrence.

Derivation (per sequence and head; a chunk is C consecutive tokens starting at
a multiple of C from the sequence start, the last one possibly shorter).  With
S0 the state entering the chunk and G_i = sum_{t<=i} g_t the in-chunk inclusive
log-decay prefix (per channel), the delta written by token i is

    delta_i = beta_i (v_i - S'_i^T k_i),  S'_i = Diag(e^{G_i}) S0
              + sum_{j<i} Diag(e^{G_i - G_j}) k_j delta_j^T.

Collecting the j<i terms gives (I + A) Delta = diag(beta) V - diag(beta)
(K o e^G) S0 with A_ij = beta_i sum_c k_ic k_jc e^{G_ic - G_jc} (j < i).  So

    T = (I + A)^-1,  W = T diag(beta) (K o e^G),  U = T diag(beta) V,
    Delta = U - W S0,
    O = scale [ (Q o e^G) S0 + Aqk Delta ],  Aqk_ij = sum_c q_ic k_jc e^{G_ic-G_jc} (j<=i),
    S_C = Diag(e^{G_last}) S0 + (K o e^{G_last - G})^T Delta.

Pairwise exponentials are taken directly as exp(G_i - G_j) (never as a
product of e^{G_i} and e^{-G_j}), so nothing overflows.
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def _norm_rows(x: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def chunk_step(Q, Kk, Vv, g, b, S0, scale):
    """One chunk: Q, Kk [L,K] (already normalised), Vv [L,V], g [L,K], b [L], S0 [K,V].

    Returns (O [L,V], S_end [K,V])."""
    L = Q.shape[0]
    G = np.cumsum(g, axis=0)                                   # [L, K]
    diff = G[:, None, :] - G[None, :, :]                       # [i, j, c] = G_i - G_j
    lower = np.tril(np.ones((L, L), dtype=bool))               # j <= i
    diff = np.where(lower[:, :, None], diff, -np.inf)
    E = np.exp(diff)                                           # e^{G_i - G_j}, 0 above diag
    A = np.einsum("ic,jc,ijc->ij", Kk, Kk, E) * b[:, None]
    A = np.tril(A, -1)
    Aqk = np.einsum("ic,jc,ijc->ij", Q, Kk, E)
    Tm = np.linalg.inv(np.eye(L) + A)
    eG = np.exp(G)
    W = Tm @ (b[:, None] * Kk * eG)
    U = Tm @ (b[:, None] * Vv)
    Delta = U - W @ S0
    O = scale * ((Q * eG) @ S0 + Aqk @ Delta)
    S_end = np.exp(G[-1])[:, None] * S0 + (Kk * np.exp(G[-1][None, :] - G)).T @ Delta
    return O, S_end


def forward_chunked(q, k, v, g, beta, cu_seqlens, scale: float, C: int = 64,
                    l2norm: bool = True, eps: float = L2_EPS, initial_state=None):
    """Chunked FP64 forward over packed sequences.  Shapes as the token oracle;
    initial_state [N,H,K,V] or None (zero)."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64); g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, H, K = q.shape
    V = v.shape[2]
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    o = np.zeros((T, H, V))
    S_all = np.zeros((len(cu) - 1, H, K, V))
    for n in range(len(cu) - 1):
        bos, eos = cu[n], cu[n + 1]
        for h in range(H):
            S = (np.zeros((K, V)) if initial_state is None
                 else np.array(initial_state[n, h], np.float64))
            for c0 in range(bos, eos, C):
                c1 = min(c0 + C, eos)
                Q = q[c0:c1, h]
                Kk = k[c0:c1, h]
                if l2norm:
                    Q = _norm_rows(Q, eps)
                    Kk = _norm_rows(Kk, eps)
                O, S = chunk_step(Q, Kk, v[c0:c1, h], g[c0:c1, h], beta[c0:c1, h], S, scale)
                o[c0:c1, h] = O
            S_all[n, h] = S
    return o, S_all
