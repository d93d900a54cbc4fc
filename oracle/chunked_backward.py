"""FP64 chunked (WY) form of the KDA forward's VJP -- TEST INFRASTRUCTURE ONLY.

A second algorithm for the gradients that ``oracle.backward`` computes token
by token (the pages test the chunked backward against FP64 budgets: "Add
opt-in FP32 KDA chunk computation", section Validation).  Each chunk of C
tokens is written in the WY form of the forward (see ``oracle.chunked``):

    G = cumsum(g) within the chunk,  E_ijc = e^{G_ic - G_jc} (j <= i, else 0)
    P_ij = sum_c k_ic k_jc E_ijc,    A = strict_lower(diag(beta) P)
    M = (I + A)^-1,  T' = M diag(beta),  K~ = K o e^G,  R = V - K~ S0,  D = T' R
    Aqk_ij = sum_c q_ic k_jc E_ijc (j <= i),  Q~ = Q o e^G
    O = scale (Q~ S0 + Aqk D),  S_end = e^{G_last} o S0 + K''^T D,  K'' = K o e^{G_last - G}

and its reverse-mode derivative is taken line by line, chunk by chunk from
the last, the state gradient dS carried backwards.  With the records of the
forward preparation this is what a chunked GPU backward computes: the state
recurrence needs only A_qk, K'', Q~ and W = T' K~ (dS0 = e^{G_last} o dS +
scale Q~^T dO - W^T dD).  The tests require it to equal the token oracle.
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def _chunk_forward(Qh, Kh, V, g, b, S0, scale):
    """Intermediates of one chunk; Qh, Kh are the normalised rows [L,K]."""
    L = Qh.shape[0]
    G = np.cumsum(g, axis=0)                                   # [L, K]
    lower = np.tril(np.ones((L, L), dtype=bool))               # j <= i
    E = np.exp(np.where(lower[:, :, None], G[:, None, :] - G[None, :, :], -np.inf))
    P = np.einsum("ic,jc,ijc->ij", Kh, Kh, E)
    A = np.tril(b[:, None] * P, -1)
    M = np.linalg.inv(np.eye(L) + A)
    Tp = M * b[None, :]
    eG = np.exp(G)
    Kt = Kh * eG
    R = V - Kt @ S0
    D = Tp @ R
    Aqk = np.tril(np.einsum("ic,jc,ijc->ij", Qh, Kh, E))
    Qt = Qh * eG
    eGC = np.exp(G[-1])
    Kpp = Kh * np.exp(G[-1][None, :] - G)
    O = scale * (Qt @ S0 + Aqk @ D)
    S_end = eGC[:, None] * S0 + Kpp.T @ D
    return dict(G=G, E=E, P=P, M=M, Tp=Tp, eG=eG, Kt=Kt, R=R, D=D, Aqk=Aqk, Qt=Qt, eGC=eGC,
                Kpp=Kpp, O=O, S_end=S_end)


def _chunk_backward(Qh, Kh, b, S0, scale, dO, dS, f):
    """Gradients of one chunk with respect to Qh, Kh, V, g, b and S0, given dO
    (of the chunk's outputs) and dS (of its end state)."""
    # O = scale (Q~ S0 + Aqk D);  S_end = e^{G_last} o S0 + K''^T D
    dD = scale * f["Aqk"].T @ dO + f["Kpp"] @ dS
    dAqk = np.tril(scale * dO @ f["D"].T)
    dQt = scale * dO @ S0.T
    dKpp = f["D"] @ dS.T
    dS0 = f["eGC"][:, None] * dS + scale * f["Qt"].T @ dO
    # D = T' R,  R = V - K~ S0
    dR = f["Tp"].T @ dD
    dTp = np.tril(dD @ f["R"].T)
    dV = dR
    dKt = -dR @ S0.T
    dS0 = dS0 - f["Kt"].T @ dR
    # T' = M diag(b);  M = (I + A)^-1;  A = strict_lower(diag(b) P)
    dM = dTp * b[None, :]
    db = np.sum(dTp * f["M"], axis=0)
    dA = np.tril(-f["M"].T @ dM @ f["M"].T, -1)
    db += np.sum(dA * f["P"], axis=1)
    dP = dA * b[:, None]
    dQh = np.zeros_like(Qh)
    dKh = np.zeros_like(Kh)
    dG = np.zeros_like(Kh)
    E = f["E"]
    # P_ij = sum_c k_ic k_jc E_ijc
    t = dP[:, :, None] * E
    dKh += np.einsum("ijc,jc->ic", t, Kh) + np.einsum("ijc,ic->jc", t, Kh)
    w = t * Kh[:, None, :] * Kh[None, :, :]
    dG += w.sum(axis=1) - w.sum(axis=0)
    # Aqk_ij = sum_c q_ic k_jc E_ijc
    t = dAqk[:, :, None] * E
    dQh += np.einsum("ijc,jc->ic", t, Kh)
    dKh += np.einsum("ijc,ic->jc", t, Qh)
    w = t * Qh[:, None, :] * Kh[None, :, :]
    dG += w.sum(axis=1) - w.sum(axis=0)
    # Q~ = Q o e^G,  K~ = K o e^G
    dQh += dQt * f["eG"]
    dG += dQt * f["Qt"]
    dKh += dKt * f["eG"]
    dG += dKt * f["Kt"]
    # K'' = K o e^{G_last - G}
    dKh += dKpp * np.exp(f["G"][-1][None, :] - f["G"])
    w = dKpp * f["Kpp"]
    dG -= w
    dG[-1] += w.sum(axis=0)
    # e^{G_last} o S0
    dG[-1] += f["eGC"] * np.sum(dS * S0, axis=1)
    # G = cumsum(g)
    dg = np.cumsum(dG[::-1], axis=0)[::-1]
    return dQh, dKh, dV, dg, db, dS0


def _norm(x, eps, on):
    if not on:
        return x.copy(), np.ones((x.shape[0], 1))
    n = np.sqrt(np.sum(x * x, axis=1, keepdims=True) + eps)
    return x / n, n


def _norm_vjp(x, n, dxn, on):
    if not on:
        return dxn
    return dxn / n - x * np.sum(x * dxn, axis=1, keepdims=True) / n ** 3


def backward_chunked(q, k, v, g, beta, cu_seqlens, scale, dO, dS_final=None,
                     initial_state=None, l2norm=True, eps=L2_EPS, C=64):
    """Same arguments and results as ``oracle.backward.backward``:
    (dq, dk, dv, dg, dbeta, dS0) in float64, the sequences cut into chunks of C."""
    f64 = lambda a: None if a is None else np.asarray(a, np.float64)
    q, k, v, g, beta, dO = map(f64, (q, k, v, g, beta, dO))
    dS_final, initial_state = f64(dS_final), f64(initial_state)
    T, H, K = q.shape
    V = v.shape[2]
    cu = [int(c) for c in cu_seqlens]
    N = len(cu) - 1
    dq, dk, dv, dg = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dS0_all = np.zeros((N, H, K, V))
    for n in range(N):
        bos, eos = cu[n], cu[n + 1]
        for h in range(H):
            Qh, nq = _norm(q[bos:eos, h], eps, l2norm)
            Kh, nk = _norm(k[bos:eos, h], eps, l2norm)
            starts = list(range(0, eos - bos, C))
            S = np.zeros((K, V)) if initial_state is None else initial_state[n, h].copy()
            S_in = []
            for c0 in starts:                               # the state entering each chunk
                c1 = min(c0 + C, eos - bos)
                S_in.append(S)
                S = _chunk_forward(Qh[c0:c1], Kh[c0:c1], v[bos + c0:bos + c1, h],
                                   g[bos + c0:bos + c1, h], beta[bos + c0:bos + c1, h], S,
                                   scale)["S_end"]
            dS = np.zeros((K, V)) if dS_final is None else dS_final[n, h].copy()
            dQh = np.zeros_like(Qh)
            dKh = np.zeros_like(Kh)
            for c0, S0 in reversed(list(zip(starts, S_in))):
                c1 = min(c0 + C, eos - bos)
                sl = slice(bos + c0, bos + c1)
                fw = _chunk_forward(Qh[c0:c1], Kh[c0:c1], v[sl, h], g[sl, h], beta[sl, h], S0,
                                    scale)
                gq, gk, gv, gg, gb, dS = _chunk_backward(Qh[c0:c1], Kh[c0:c1], beta[sl, h], S0,
                                                         scale, dO[sl, h], dS, fw)
                dQh[c0:c1] = gq
                dKh[c0:c1] = gk
                dv[sl, h] = gv
                dg[sl, h] = gg
                dbeta[sl, h] = gb
            dq[bos:eos, h] = _norm_vjp(q[bos:eos, h], nq, dQh, l2norm)
            dk[bos:eos, h] = _norm_vjp(k[bos:eos, h], nk, dKh, l2norm)
            dS0_all[n, h] = dS
    return dq, dk, dv, dg, dbeta, dS0_all
