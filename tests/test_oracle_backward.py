"""Pins of the FP64 backward oracle (oracle/backward.py).

The VJP is checked against central finite differences of the scalar
L = sum(dO * o) + sum(dS_T * S_T), in float64, on tiny shapes that still
cover packing, both normalisations and an initial state; each planted mistake
in the VJP must fail that check.  Its forward is also tied to the pinned C
oracle, so the function differentiated is the one every other test uses."""
import numpy as np
import pytest

import oracle
from oracle.backward import MUTATIONS, backward, forward


def _case(seed, lens=(3, 2), H=2, K=3, V=2, init=True):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    c = dict(q=rng.standard_normal((T, H, K)), k=rng.standard_normal((T, H, K)),
             v=rng.standard_normal((T, H, V)), g=-rng.uniform(0.05, 1.5, (T, H, K)),
             beta=rng.uniform(0.1, 0.9, (T, H)),
             S0=rng.standard_normal((len(lens), H, K, V)) * 0.5 if init else None)
    dO = rng.standard_normal((T, H, V))
    dST = rng.standard_normal((len(lens), H, K, V))
    return c, cu, dO, dST


def _loss(c, cu, dO, dST, l2norm):
    o, ST = forward(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, 0.7,
                    initial_state=c["S0"], l2norm=l2norm)
    return (dO * o).sum() + (dST * ST).sum()


def _fd_check(c, cu, dO, dST, l2norm, mutation="none", h=1e-6):
    dq, dk, dv, dg, db, dS0 = backward(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, 0.7, dO,
                                       dS_final=dST, initial_state=c["S0"], l2norm=l2norm,
                                       mutation=mutation)
    ana = dict(q=dq, k=dk, v=dv, g=dg, beta=db, S0=dS0)
    for name in ("q", "k", "v", "g", "beta", "S0"):
        if c[name] is None:
            continue
        x = c[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(c, cu, dO, dST, l2norm)
            x[idx] = old - h
            lm = _loss(c, cu, dO, dST, l2norm)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        if not np.allclose(ana[name], num, rtol=1e-6, atol=1e-8):
            return False, name
    return True, None


@pytest.mark.parametrize("l2norm", [True, False])
@pytest.mark.parametrize("init", [True, False])
def test_vjp_matches_finite_differences(l2norm, init):
    c, cu, dO, dST = _case(11 + 2 * l2norm + init, init=init)
    ok, name = _fd_check(c, cu, dO, dST, l2norm)
    assert ok, f"d{name} disagrees with central differences"


def test_forward_is_the_pinned_oracle():
    c, cu, dO, dST = _case(12, lens=(5, 0, 4), H=3, K=4, V=4)
    o, ST = forward(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, 0.7, initial_state=c["S0"])
    o_c, S_c = oracle.forward(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, 0.7,
                              initial_state=c["S0"])
    assert np.allclose(o, o_c, rtol=1e-12, atol=1e-14) and np.allclose(ST, S_c, rtol=1e-12)


@pytest.mark.parametrize("mutation", [m for m in MUTATIONS if m != "none"])
def test_each_planted_mistake_fails_finite_differences(mutation):
    c, cu, dO, dST = _case(13)
    ok, _ = _fd_check(c, cu, dO, dST, True, mutation=mutation)
    assert not ok


# ---- a second algorithm: the chunked (WY) VJP must equal the token VJP

from oracle.chunked_backward import backward_chunked  # noqa: E402


def _both(c, cu, dO, dST, l2norm, C, mutation="none"):
    a = backward(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, 0.7, dO, dS_final=dST,
                 initial_state=c["S0"], l2norm=l2norm, mutation=mutation)
    b = backward_chunked(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, 0.7, dO, dS_final=dST,
                         initial_state=c["S0"], l2norm=l2norm, C=C)
    return [np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300) for x, y in zip(a, b)]


@pytest.mark.parametrize("C", [1, 3, 16, 64])
@pytest.mark.parametrize("l2norm,init", [(True, True), (False, False)])
def test_chunked_vjp_equals_token_vjp(C, l2norm, init):
    c, cu, dO, dST = _case(21 + C, lens=(9, 0, 17, 40), H=2, K=6, V=5, init=init)
    assert max(_both(c, cu, dO, dST, l2norm, C)) < 1e-12


def test_chunked_vjp_equals_token_vjp_full_width():
    """K = V = 128 (the library's shape), two packed sequences across chunk edges."""
    c, cu, dO, dST = _case(22, lens=(130, 37), H=1, K=128, V=128)
    assert max(_both(c, cu, dO, dST, True, 64)) < 1e-12


@pytest.mark.parametrize("mutation", [m for m in MUTATIONS if m != "none"])
def test_each_planted_mistake_disagrees_with_the_chunked_vjp(mutation):
    c, cu, dO, dST = _case(23, lens=(9, 17), H=2, K=6, V=5)
    assert max(_both(c, cu, dO, dST, True, 4, mutation=mutation)) > 1e-6
