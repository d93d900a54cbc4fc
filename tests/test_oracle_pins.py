"""The FP64 oracle against facts that do not come from it (CPU only)."""
import json
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import chunked, exact_scalar
import pinlib


@pytest.mark.parametrize("name", list(pinlib.PINS))
def test_pin(name):
    err, tol = pinlib.PINS[name](0)
    assert np.isfinite(err) and err <= tol, f"{name}: error {err:.3e} > {tol:.0e}"


@pytest.mark.parametrize("C", [1, 16, 64, 128])
@pytest.mark.parametrize("case", ["packed_37_28", "boundary_129"])
def test_chunked_form_matches_token_loop(C, case, golden_dir):
    """The chunk solve agrees with the recurrence at the page's own test lengths
    (packed 37/28 and a 129-token sequence that crosses two chunk boundaries)."""
    cases = {c["name"]: c for c in
             json.load(open(os.path.join(golden_dir, "page_cases.json")))["recurrence_test_cases"]}
    lens = tuple(cases[case]["seqlens"])
    err, tol = pinlib.pin_chunked_form(0, C=C, lens=lens, H=2, K=32, V=32, seed=11 + C)
    assert err <= tol, err


def test_chunked_form_full_head_dim():
    """K = V = 128 (the production head geometry) on one head."""
    err, tol = pinlib.pin_chunked_form(0, C=64, lens=(65,), H=1, K=128, V=128, seed=3)
    assert err <= tol, err


def test_scalar_exact_random():
    """K = V = 1 on fresh random rationals, several packings, exact reference."""
    rng = random.Random(7)
    for trial in range(5):
        lens = [rng.randint(0, 9) for _ in range(rng.randint(1, 3))]
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        T = cu[-1]
        if T == 0:
            continue
        pick = [Fraction(-3), Fraction(-1), Fraction(2), Fraction(5)]
        q = [rng.choice(pick) for _ in range(T)]
        k = [rng.choice(pick) for _ in range(T)]
        v = [Fraction(rng.randint(-20, 20), 4) for _ in range(T)]
        a = [Fraction(rng.randint(1, 32), 32) for _ in range(T)]
        beta = [Fraction(rng.randint(0, 16), 16) for _ in range(T)]
        o_ref, S_ref = exact_scalar.explicit_sum(q, k, v, a, beta, cu, Fraction(1, 2))
        arr = lambda xs: np.array([float(x) for x in xs]).reshape(T, 1, 1)
        o, S = oracle.forward(arr(q), arr(k), arr(v), np.log(arr(a)),
                              arr(beta).reshape(T, 1), cu, 0.5, eps=0.0)
        assert np.max(np.abs(o.ravel() - [float(x) for x in o_ref])) < 1e-13
        assert np.max(np.abs(S.ravel() - [float(x) for x in S_ref])) < 1e-13


def test_gate_ranges():
    """g < 0 and 0 < beta < 1 over the workloads' distributions, including the
    extremes f + dt_bias in {-30, 0, 30}."""
    rng = np.random.default_rng(0)
    T, H, K = 50, 4, 16
    f = rng.standard_normal((T, H, K))
    f[0] = -30.0
    f[1] = 0.0
    f[2] = 30.0
    A_log = rng.uniform(0, np.log(16), H)
    dt_bias = np.zeros((H, K))
    b = rng.standard_normal((T, H))
    g, beta = oracle.gate(f, A_log, dt_bias, b)
    assert np.all(g < 0) and np.all((beta > 0) & (beta < 1))
    lam = np.exp(A_log)[:, None]
    assert np.allclose(g[1], -lam * np.log(2.0), rtol=1e-15, atol=0)
    assert np.allclose(g[2], -lam * (30.0 + np.log1p(np.exp(-30.0))), rtol=1e-15, atol=0)
    assert np.allclose(g[0], -lam * np.exp(-30.0), rtol=1e-13, atol=0)


def test_oracle_rejects_bad_offsets():
    z = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.forward(z, z, z, z, np.zeros((4, 1)), [0, 3], 1.0)       # last != T
    with pytest.raises(ValueError):
        oracle.forward(z, z, z, z, np.zeros((4, 1)), [0, 3, 2, 4], 1.0)  # decreasing
