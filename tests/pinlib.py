"""Pins of the FP64 oracle: checks against facts that do not come from the oracle.

Each pin takes a planted-mistake switch (``mutation``, 0 = the real oracle)
and returns ``(error, tolerance)``.  ``test_oracle_pins`` requires every pin
to pass for mutation 0; ``test_oracle_mutations`` requires every planted
mistake to fail at least one pin, after the page's own test-of-the-test (a
planted scaling error must fail: "Add opt-in FP32 KDA chunk computation",
section Validation).
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

import oracle
from oracle import chunked, exact_scalar

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _gate_draws(rng, T, H, K):
    """Gate inputs with the workloads' distributions."""
    f = rng.standard_normal((T, H, K))
    A_log = rng.uniform(0.0, math.log(16.0), H)
    dt_bias = 0.5 * rng.standard_normal((H, K))
    b = rng.standard_normal((T, H))
    return f, A_log, dt_bias, b


def _qkv(rng, T, H, K, V):
    return (rng.standard_normal((T, H, K)), rng.standard_normal((T, H, K)),
            rng.standard_normal((T, H, V)))


# --------------------------------------------------------------------------- pins

def pin_scalar_exact(mutation=0):
    """K = V = 1 against exact rationals (tests/golden/scalar_k1v1.json)."""
    d = json.load(open(os.path.join(GOLDEN, "scalar_k1v1.json")))
    F = lambda xs: np.array([float(Fraction(x)) for x in xs])
    T = len(d["q"])
    q = F(d["q"]).reshape(T, 1, 1)
    k = F(d["k"]).reshape(T, 1, 1)
    v = F(d["v"]).reshape(T, 1, 1)
    g = np.log(F(d["a"])).reshape(T, 1, 1)
    beta = F(d["beta"]).reshape(T, 1)
    o, S = oracle.forward(q, k, v, g, beta, d["cu_seqlens"], float(Fraction(d["scale"])),
                          l2norm=True, eps=0.0, mutation=mutation)
    o_ref = F(d["o"])
    S_ref = F(d["final_state"])
    err = max(np.max(np.abs(o.ravel() - o_ref)), np.max(np.abs(S.ravel() - S_ref)))
    return float(err), 1e-13


def pin_beta_zero(mutation=0):
    """beta = 0: nothing is ever written, so o = 0 and S = 0 exactly."""
    rng = _rng(1)
    lens = [5, 0, 9]
    T, H, K, V = sum(lens), 3, 8, 6
    q, k, v = _qkv(rng, T, H, K, V)
    g = -rng.uniform(0.0, 3.0, (T, H, K))
    beta = np.zeros((T, H))
    o, S = oracle.forward(q, k, v, g, beta, _cu(lens), 0.5, mutation=mutation)
    return float(max(np.max(np.abs(o)), np.max(np.abs(S)))), 0.0


def _gla_closed_form(q, k, v, g, cu, scale, eps=oracle.L2_EPS):
    """o_t = scale * sum_{j<=t} ((q^_t o e^{G_t - G_j}) . k^_j) v_j: gated linear
    attention, the first-order term of KDA in a constant small beta."""
    T, H, K = q.shape
    o = np.zeros((T, H, v.shape[2]))
    qn = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + eps)
    kn = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + eps)
    for n in range(len(cu) - 1):
        a, z = cu[n], cu[n + 1]
        for h in range(H):
            G = np.cumsum(g[a:z, h], axis=0)
            for t in range(z - a):
                dec = np.exp(G[t][None, :] - G[: t + 1])            # [j, c]
                w = np.sum(qn[a + t, h][None, :] * dec * kn[a:a + t + 1, h], axis=1)
                o[a + t, h] = scale * (w @ v[a:a + t + 1, h])
    return o


def pin_small_beta_gla(mutation=0):
    """beta = eps -> o / eps approaches gated linear attention (error O(eps))."""
    rng = _rng(2)
    lens = [11, 6]
    T, H, K, V = sum(lens), 2, 8, 8
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, _ = oracle.gate(f, A_log * 0.1, dt_bias, b)     # milder decay keeps long-range terms
    eps = 1e-7
    beta = np.full((T, H), eps)
    cu = _cu(lens)
    o, _ = oracle.forward(q, k, v, g, beta, cu, 0.25, mutation=mutation)
    ref = _gla_closed_form(q, k, v, g, cu, 0.25)
    return oracle.rel_l2(o / eps, ref), 1e-5


def pin_small_beta_linear_attention(mutation=0):
    """beta = eps, g = 0 -> o / eps approaches scale * sum_{j<=t} (q^_t . k^_j) v_j."""
    rng = _rng(3)
    lens = [13]
    T, H, K, V = 13, 2, 6, 4
    q, k, v = _qkv(rng, T, H, K, V)
    eps = 1e-7
    o, _ = oracle.forward(q, k, v, np.zeros((T, H, K)), np.full((T, H), eps), _cu(lens),
                          0.5, mutation=mutation)
    qn = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + oracle.L2_EPS)
    kn = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + oracle.L2_EPS)
    kv = np.cumsum(np.einsum("thc,thm->thcm", kn, v), axis=0)     # running sum of k v^T
    ref = 0.5 * np.einsum("thcm,thc->thm", kv, qn)
    return oracle.rel_l2(o / eps, ref), 1e-5


def pin_delta_overwrite(mutation=0):
    """beta = 1, every key along one direction u, decay uniform over channels:
    each write replaces the previous one, so o_t = scale * (u^ . q^_t) v_t."""
    rng = _rng(4)
    T, H, K, V = 9, 2, 8, 5
    u = rng.standard_normal((H, K))
    alpha = rng.uniform(0.5, 2.0, (T, H, 1))                     # unnormalised magnitudes
    k = alpha * u[None]
    q = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = np.repeat(-rng.uniform(0.0, 2.0, (T, H, 1)), K, axis=2)  # same decay on every channel
    beta = np.ones((T, H))
    scale = 1.0 / math.sqrt(K)
    # eps = 0: the closed form needs exactly unit keys
    o, _ = oracle.forward(q, k, v, g, beta, _cu([T]), scale, eps=0.0, mutation=mutation)
    un = u / np.sqrt(np.sum(u * u, -1, keepdims=True))
    qn = q / np.sqrt(np.sum(q * q, -1, keepdims=True))
    ref = scale * np.einsum("hc,thc->th", un, qn)[:, :, None] * v
    return oracle.rel_l2(o, ref), 1e-9


def pin_packing(mutation=0):
    """Packed output equals per-sequence runs concatenated (final states too)."""
    rng = _rng(5)
    lens = [7, 1, 0, 12]
    T, H, K, V = sum(lens), 2, 8, 6
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b, mutation=mutation)
    o, S = oracle.forward(q, k, v, g, beta, _cu(lens), 0.3, mutation=mutation)
    err = 0.0
    cu = _cu(lens)
    for n, L in enumerate(lens):
        a, z = cu[n], cu[n + 1]
        o1, S1 = oracle.forward(q[a:z], k[a:z], v[a:z], g[a:z], beta[a:z], [0, L], 0.3,
                                mutation=mutation)
        err = max(err, float(np.max(np.abs(o[a:z] - o1), initial=0.0)),
                  float(np.max(np.abs(S[n] - S1[0]))))
    return err, 0.0


def pin_chunked_form(mutation=0, C=64, lens=(37, 28), H=2, K=32, V=32, seed=6):
    """The chunked WY form (a different algorithm) agrees with the token loop."""
    rng = _rng(seed)
    T = sum(lens)
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    cu = _cu(list(lens))
    o, S = oracle.forward(q, k, v, g, beta, cu, 0.2, mutation=mutation)
    oc, Sc = chunked.forward_chunked(q, k, v, g, beta, cu, 0.2, C=C)
    return max(oracle.rel_l2(o, oc), oracle.rel_l2(S, Sc)), 1e-12


def pin_linearity_in_v(mutation=0):
    """o and S are linear in v."""
    rng = _rng(7)
    lens = [10, 5]
    T, H, K, V = sum(lens), 2, 8, 6
    q, k, v1 = _qkv(rng, T, H, K, V)
    v2 = rng.standard_normal((T, H, V))
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    cu = _cu(lens)
    run = lambda vv: oracle.forward(q, k, vv, g, beta, cu, 0.3, mutation=mutation)
    o1, S1 = run(v1); o2, S2 = run(v2); o3, S3 = run(v1 - 2.5 * v2)
    return max(oracle.rel_l2(o3, o1 - 2.5 * o2), oracle.rel_l2(S3, S1 - 2.5 * S2)), 1e-13


def pin_permutations(mutation=0):
    """Permuting V columns permutes o's columns; permuting heads permutes o's heads."""
    rng = _rng(8)
    lens = [9, 4]
    T, H, K, V = sum(lens), 3, 8, 6
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    cu = _cu(lens)
    o, S = oracle.forward(q, k, v, g, beta, cu, 0.3, mutation=mutation)
    pv = rng.permutation(V)
    ov, Sv = oracle.forward(q, k, v[:, :, pv], g, beta, cu, 0.3, mutation=mutation)
    ph = rng.permutation(H)
    oh, Sh = oracle.forward(q[:, ph], k[:, ph], v[:, ph], g[:, ph], beta[:, ph], cu, 0.3,
                            mutation=mutation)
    err = max(float(np.max(np.abs(ov - o[:, :, pv]))), float(np.max(np.abs(Sv - S[..., pv]))),
              float(np.max(np.abs(oh - o[:, ph]))), float(np.max(np.abs(Sh - S[:, ph]))))
    return err, 1e-14


def pin_scale(mutation=0):
    """o is proportional to scale; S does not depend on it."""
    rng = _rng(9)
    T, H, K, V = 8, 2, 8, 6
    q, k, v = _qkv(rng, T, H, K, V)
    g = -rng.uniform(0, 2, (T, H, K))
    beta = rng.uniform(0, 1, (T, H))
    o1, S1 = oracle.forward(q, k, v, g, beta, [0, T], 1.0, mutation=mutation)
    o2, S2 = oracle.forward(q, k, v, g, beta, [0, T], 0.125, mutation=mutation)
    return max(oracle.rel_l2(o2, 0.125 * o1), oracle.rel_l2(S2, S1)), 1e-15


def pin_gate_special_values(mutation=0):
    """softplus(0) = ln 2; exp(A_log = ln 16) = 16; sigmoid(0) = 1/2; softplus(x) -> x."""
    H, K = 3, 4
    A_log = np.array([0.0, math.log(16.0), math.log(4.0)])
    dt_bias = np.arange(H * K, dtype=np.float64).reshape(H, K) * 0.25 - 1.0
    T = 2
    f = np.empty((T, H, K))
    f[0] = -dt_bias                     # f + dt_bias = 0 -> softplus = ln 2
    f[1] = 40.0 - dt_bias               # f + dt_bias = 40 -> softplus = 40 (+ e^-40)
    b = np.array([[0.0, 0.0, 0.0], [math.log(3.0), -math.log(3.0), 0.0]])
    g, beta = oracle.gate(f, A_log, dt_bias, b, mutation=mutation)
    lam = np.array([1.0, 16.0, 4.0])
    g_ref = np.empty_like(g)
    g_ref[0] = -lam[:, None] * math.log(2.0)
    g_ref[1] = -lam[:, None] * 40.0
    beta_ref = np.array([[0.5, 0.5, 0.5], [0.75, 0.25, 0.5]])
    err = max(float(np.max(np.abs(g - g_ref) / np.abs(g_ref))),
              float(np.max(np.abs(beta - beta_ref))))
    return err, 1e-15


def pin_numpy_matrix_form(mutation=0):
    """The C token loop agrees with the NumPy matrix statement of the recurrence."""
    rng = _rng(10)
    lens = [6, 0, 7]
    T, H, K, V = sum(lens), 2, 5, 3
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    cu = _cu(lens)
    o, S = oracle.forward(q, k, v, g, beta, cu, 0.4, mutation=mutation)
    o2, S2 = oracle.forward_matrix_numpy(q, k, v, g, beta, cu, 0.4)
    return max(oracle.rel_l2(o, o2), oracle.rel_l2(S, S2)), 1e-13


def pin_initial_state_decay(mutation=0):
    """beta = 0 from an initial state S0: the state only decays, so
    o_t = scale * sum_c q^_tc e^{G_tc} S0[c, :] and S_T = Diag(e^{G_T}) S0."""
    rng = _rng(12)
    lens = [9, 4]
    T, H, K, V = sum(lens), 2, 6, 5
    q, k, v = _qkv(rng, T, H, K, V)
    g = -rng.uniform(0.0, 1.5, (T, H, K))
    S0 = rng.standard_normal((len(lens), H, K, V))
    cu = _cu(lens)
    o, S = oracle.forward(q, k, v, g, np.zeros((T, H)), cu, 0.7, mutation=mutation,
                          initial_state=S0)
    qn = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + oracle.L2_EPS)
    o_ref = np.zeros_like(o)
    S_ref = np.zeros_like(S)
    for n in range(len(lens)):
        a, z = cu[n], cu[n + 1]
        G = np.cumsum(g[a:z], axis=0)                                  # [t, h, c]
        o_ref[a:z] = 0.7 * np.einsum("thc,thc,hcm->thm", qn[a:z], np.exp(G), S0[n])
        S_ref[n] = np.exp(G[-1])[:, :, None] * S0[n]
    return max(oracle.rel_l2(o, o_ref), oracle.rel_l2(S, S_ref)), 1e-13


def pin_split_sequence(mutation=0):
    """Running a sequence in two pieces, the second from the first's final state
    (chunked WY form), equals one run of the whole (token loop)."""
    rng = _rng(13)
    T, H, K, V = 70, 2, 16, 16
    cut = 29
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    o, S = oracle.forward(q, k, v, g, beta, [0, T], 0.3, mutation=mutation)
    o1, S1 = oracle.forward(q[:cut], k[:cut], v[:cut], g[:cut], beta[:cut], [0, cut], 0.3,
                            mutation=mutation)
    o2, S2 = chunked.forward_chunked(q[cut:], k[cut:], v[cut:], g[cut:], beta[cut:],
                                     [0, T - cut], 0.3, C=16, initial_state=S1)
    err = max(oracle.rel_l2(np.concatenate([o1, o2]), o), oracle.rel_l2(S2, S))
    return err, 1e-12


def pin_chunked_with_initial_state(mutation=0):
    """The chunked WY form from an initial state agrees with the token loop."""
    rng = _rng(14)
    lens = [37, 28]
    T, H, K, V = sum(lens), 2, 16, 16
    q, k, v = _qkv(rng, T, H, K, V)
    f, A_log, dt_bias, b = _gate_draws(rng, T, H, K)
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    S0 = 0.3 * rng.standard_normal((len(lens), H, K, V))
    cu = _cu(lens)
    o, S = oracle.forward(q, k, v, g, beta, cu, 0.2, mutation=mutation, initial_state=S0)
    oc, Sc = chunked.forward_chunked(q, k, v, g, beta, cu, 0.2, C=64, initial_state=S0)
    return max(oracle.rel_l2(o, oc), oracle.rel_l2(S, Sc)), 1e-12


PINS = {
    "scalar_exact": pin_scalar_exact,
    "beta_zero": pin_beta_zero,
    "small_beta_gla": pin_small_beta_gla,
    "small_beta_linear_attention": pin_small_beta_linear_attention,
    "delta_overwrite": pin_delta_overwrite,
    "packing": pin_packing,
    "chunked_form": pin_chunked_form,
    "linearity_in_v": pin_linearity_in_v,
    "permutations": pin_permutations,
    "scale": pin_scale,
    "gate_special_values": pin_gate_special_values,
    "numpy_matrix_form": pin_numpy_matrix_form,
    "initial_state_decay": pin_initial_state_decay,
    "split_sequence": pin_split_sequence,
    "chunked_with_initial_state": pin_chunked_with_initial_state,
}


def failing_pins(mutation: int):
    out = []
    for name, fn in PINS.items():
        err, tol = fn(mutation)
        if not (err <= tol) or not np.isfinite(err):
            out.append(name)
    return out
