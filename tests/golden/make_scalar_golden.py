"""Writes scalar_k1v1.json: the K = V = 1 KDA case evaluated exactly.

The expected values come from ``oracle.exact_scalar.explicit_sum`` (exact
rational arithmetic on the explicit-sum solution of the scalar recurrence);
nothing here touches the CUDA library.  Run from the repository root:

    python tests/golden/make_scalar_golden.py
"""
import json
import os
import random
import sys
from fractions import Fraction

sys.path.insert(0, os.path.abspath(os.path.join(os.path.dirname(__file__), "..", "..")))
from oracle.exact_scalar import explicit_sum  # noqa: E402


def main():
    rng = random.Random(20261111)
    seqlens = [7, 0, 12]                      # includes an empty sequence
    cu = [0]
    for n in seqlens:
        cu.append(cu[-1] + n)
    T = cu[-1]
    pick = [Fraction(-2), Fraction(-1), Fraction(1), Fraction(3)]
    q = [rng.choice(pick) for _ in range(T)]
    k = [rng.choice(pick) for _ in range(T)]
    v = [Fraction(rng.randint(-16, 16), 8) for _ in range(T)]
    a = [Fraction(rng.randint(1, 64), 64) for _ in range(T)]        # decay factor e^{g}
    beta = [Fraction(rng.randint(0, 32), 32) for _ in range(T)]
    scale = Fraction(1, 3)
    o, finals = explicit_sum(q, k, v, a, beta, cu, scale)
    s = lambda xs: [str(x) for x in xs]
    doc = {
        "what": "KDA with K = V = 1: S_t = (1 - beta_t) a_t S_{t-1} + beta_t sign(k_t) v_t, "
                "o_t = scale * S_t * sign(q_t); exact rationals from the explicit-sum "
                "solution. The oracle gets g_t = ln(a_t), L2 normalisation with eps = 0.",
        "cite": "Add opt-in FP32 KDA chunk computation (XTuner PR #2301), section Validation: "
                "packed multi-sequence cases checked against an independent FP64 recurrence",
        "cu_seqlens": cu, "scale": str(scale),
        "q": s(q), "k": s(k), "v": s(v), "a": s(a), "beta": s(beta),
        "o": s(o), "final_state": s(finals),
    }
    out = os.path.join(os.path.dirname(__file__), "scalar_k1v1.json")
    with open(out, "w") as fh:
        json.dump(doc, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
