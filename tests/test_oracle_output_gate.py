"""Pins of the FP64 gated-RMSNorm oracle (oracle/output_gate.py), and proof that
each planted mistake in it fails at least one pin.

Pins come from the definition's closed forms and invariants, not from a
restatement of the code:
  * a worked example with exact values (V = 2, o = (3, 4), w = (1, 2),
    z = (0, ln 3)): y = (3 sqrt 2 / 10, 6 sqrt 2 / 5)
  * unit RMS of y when w = 1, the gate is open and eps = 0
  * invariance under o -> c o (c > 0, eps = 0) and oddness in o
  * the gate's symmetry sigmoid(z) + sigmoid(-z) = 1 and sigmoid(0) = 1/2
  * the eps regime: for |o| << sqrt(eps), y -> o w sigmoid(z) / sqrt(eps)
  * rows are independent (a permutation of rows permutes the output)
"""
import math

import numpy as np
import pytest

from oracle.output_gate import MUTATIONS, gated_rmsnorm


def pin_worked_example(fn):
    y = fn(np.array([3.0, 4.0]), np.array([0.0, math.log(3.0)]), np.array([1.0, 2.0]), 0.0)
    ref = np.array([3 * math.sqrt(2) / 10, 6 * math.sqrt(2) / 5])
    return np.allclose(y, ref, rtol=1e-14, atol=0)


def pin_unit_rms(fn):
    rng = np.random.default_rng(1)
    o = rng.standard_normal((7, 3, 128))
    y = fn(o, np.full_like(o, 60.0), np.ones(128), 0.0)   # sigmoid(60) = 1 in float64
    return np.allclose(np.sqrt((y * y).mean(-1)), 1.0, rtol=1e-13)


def pin_scale_and_sign(fn):
    rng = np.random.default_rng(2)
    o = rng.standard_normal((5, 64))
    z = rng.standard_normal((5, 64))
    w = rng.uniform(0.5, 1.5, 64)
    y = fn(o, z, w, 0.0)
    return (np.allclose(fn(7.5 * o, z, w, 0.0), y, rtol=1e-13)
            and np.array_equal(fn(-o, z, w, 0.0), -y))


def pin_gate_symmetry(fn):
    rng = np.random.default_rng(3)
    o = rng.standard_normal((4, 32))
    z = rng.standard_normal((4, 32)) * 3
    w = rng.uniform(0.5, 1.5, 32)
    open_ = fn(o, np.full_like(z, 60.0), w, 1e-6)
    half = fn(o, np.zeros_like(z), w, 1e-6)
    return (np.allclose(fn(o, z, w, 1e-6) + fn(o, -z, w, 1e-6), open_, rtol=1e-13)
            and np.allclose(half, 0.5 * open_, rtol=1e-15))


def pin_eps_regime(fn):
    rng = np.random.default_rng(4)
    o = rng.standard_normal((3, 16)) * 1e-9
    z = rng.standard_normal((3, 16))
    w = rng.uniform(0.5, 1.5, 16)
    eps = 1e-6
    ref = o * w / (1.0 + np.exp(-z)) / math.sqrt(eps)
    return np.allclose(fn(o, z, w, eps), ref, rtol=1e-9)


def pin_rows_independent(fn):
    rng = np.random.default_rng(5)
    o = rng.standard_normal((6, 8))
    z = rng.standard_normal((6, 8))
    w = rng.uniform(0.5, 1.5, 8)
    perm = rng.permutation(6)
    return np.array_equal(fn(o[perm], z[perm], w, 1e-6), fn(o, z, w, 1e-6)[perm])


PINS = [pin_worked_example, pin_unit_rms, pin_scale_and_sign, pin_gate_symmetry,
        pin_eps_regime, pin_rows_independent]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_meets_pin(pin):
    assert pin(gated_rmsnorm)


@pytest.mark.parametrize("mutation", [m for m in MUTATIONS if m != "none"])
def test_each_planted_mistake_fails_a_pin(mutation):
    fn = lambda o, z, w, eps: gated_rmsnorm(o, z, w, eps, mutation=mutation)
    failed = [p.__name__ for p in PINS if not p(fn)]
    assert failed, f"mutation {mutation} passes every pin"
