"""FP64 oracle of the KDA forward's vector-Jacobian product -- TEST INFRASTRUCTURE ONLY.

The backward of the chunked KDA forward (the pages test it against FP64
budgets: "Add opt-in FP32 KDA chunk computation", section Validation) is the
VJP of the token recurrence that defines the forward, per sequence and head:

    a_t  = exp(g_t)                       q^_t = q_t / sqrt(|q_t|^2 + eps)  (k^ alike)
    S'_t = Diag(a_t) S_{t-1}
    u_t  = S'_t^T k^_t
    d_t  = beta_t (v_t - u_t)
    S_t  = S'_t + k^_t d_t^T
    o_t  = scale S_t^T q^_t

Given dO (the gradient of a scalar loss with respect to every o_t) and dS_T
(with respect to the final state), this walks the tokens backwards, applying
the chain rule to each line above in reverse order, and returns dq, dk, dv,
dg, dbeta and dS_0.  Written from the recurrence by hand, in float64, one
token at a time; ``mutation`` plants one known mistake (tests only).
"""
from __future__ import annotations

import numpy as np

MUTATIONS = ("none", "no_decay_in_dS", "dg_without_a", "sign_du", "no_norm_chain")


def _norm(x, eps, on):
    if not on:
        return x.copy(), 1.0
    n = np.sqrt((x * x).sum() + eps)
    return x / n, n


def _norm_vjp(x, n, dxn, on, mutation):
    """x^ = x / n, n = sqrt(|x|^2 + eps):  dx = dx^ / n - x (x . dx^) / n^3."""
    if not on or mutation == "no_norm_chain":
        return dxn
    return dxn / n - x * (x @ dxn) / n ** 3


def backward(q, k, v, g, beta, cu_seqlens, scale, dO, dS_final=None, initial_state=None,
             l2norm=True, eps=1e-6, mutation="none"):
    """Arrays as the forward: q, k [T, H, K], v [T, H, V], g [T, H, K], beta [T, H],
    dO [T, H, V], dS_final / initial_state [N, H, K, V] or None.
    Returns (dq, dk, dv, dg, dbeta, dS0) in float64."""
    if mutation not in MUTATIONS:
        raise ValueError(mutation)
    f = lambda a: None if a is None else np.asarray(a, np.float64)
    q, k, v, g, beta, dO = map(f, (q, k, v, g, beta, dO))
    dS_final, initial_state = f(dS_final), f(initial_state)
    T, H, K = q.shape
    V = v.shape[2]
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    dq, dk, dv, dg = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dS0 = np.zeros((N, H, K, V))
    for n in range(N):
        for h in range(H):
            S = np.zeros((K, V)) if initial_state is None else initial_state[n, h].copy()
            tape = []
            for t in range(cu[n], cu[n + 1]):
                qn, nq = _norm(q[t, h], eps, l2norm)
                kn, nk = _norm(k[t, h], eps, l2norm)
                a = np.exp(g[t, h])
                Sprev = S
                Sp = a[:, None] * Sprev
                u = Sp.T @ kn
                d = beta[t, h] * (v[t, h] - u)
                S = Sp + np.outer(kn, d)
                tape.append((t, qn, nq, kn, nk, a, Sprev, Sp, u, d, S))
            dS = np.zeros((K, V)) if dS_final is None else dS_final[n, h].copy()
            for (t, qn, nq, kn, nk, a, Sprev, Sp, u, d, S) in reversed(tape):
                # o = scale S^T q^
                dqn = scale * (S @ dO[t, h])
                dS = dS + scale * np.outer(qn, dO[t, h])
                # S = S' + k^ d^T
                dSp = dS.copy()
                dkn = dS @ d
                dd = dS.T @ kn
                # d = beta (v - u)
                dv[t, h] = beta[t, h] * dd
                du = (beta[t, h] if mutation == "sign_du" else -beta[t, h]) * dd
                dbeta[t, h] = dd @ (v[t, h] - u)
                # u = S'^T k^
                dSp = dSp + np.outer(kn, du)
                dkn = dkn + Sp @ du
                # S' = Diag(a) S_prev, a = exp(g)
                da = (dSp * Sprev).sum(1)
                dg[t, h] = da if mutation == "dg_without_a" else a * da
                dS = dSp if mutation == "no_decay_in_dS" else a[:, None] * dSp
                dq[t, h] = _norm_vjp(q[t, h], nq, dqn, l2norm, mutation)
                dk[t, h] = _norm_vjp(k[t, h], nk, dkn, l2norm, mutation)
            dS0[n, h] = dS
    return dq, dk, dv, dg, dbeta, dS0


def forward(q, k, v, g, beta, cu_seqlens, scale, initial_state=None, l2norm=True, eps=1e-6):
    """The same recurrence forward (o, S_T), for the finite-difference pins."""
    f = lambda a: None if a is None else np.asarray(a, np.float64)
    q, k, v, g, beta, initial_state = map(f, (q, k, v, g, beta, initial_state))
    T, H, K = q.shape
    V = v.shape[2]
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    o = np.zeros((T, H, V))
    ST = np.zeros((N, H, K, V))
    for n in range(N):
        for h in range(H):
            S = np.zeros((K, V)) if initial_state is None else initial_state[n, h].copy()
            for t in range(cu[n], cu[n + 1]):
                qn, _ = _norm(q[t, h], eps, l2norm)
                kn, _ = _norm(k[t, h], eps, l2norm)
                Sp = np.exp(g[t, h])[:, None] * S
                d = beta[t, h] * (v[t, h] - Sp.T @ kn)
                S = Sp + np.outer(kn, d)
                o[t, h] = scale * (S.T @ qn)
            ST[n, h] = S
    return o, ST
