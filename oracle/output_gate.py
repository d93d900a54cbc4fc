"""FP64 oracle of the KDA output gate with gated RMSNorm -- TEST INFRASTRUCTURE ONLY.

The pages name this step but print no formula: the KDA module ends in a
low-rank output gate (g_a_proj -> g_b_proj) and a "gated-norm" wrapper
(XTuner "GLM-5.3-Flash F6.2: KDA correctness and FLA sequence parallelism",
module commit and the FLA sequence-SP commit).  The plain reading taken here:
for each token t and head h, with o the attention output row, z the output
gate's pre-activation row (both of length V) and w a per-channel weight shared
by all heads,

    y[t,h,v] = o[t,h,v] / sqrt(mean_v' o[t,h,v']^2 + eps) * w[v] * sigmoid(z[t,h,v])

evaluated here in float64 exactly as written.  ``mutation`` plants one known
mistake (tests only) so that the pins can be shown to catch it.
"""
from __future__ import annotations

import numpy as np

MUTATIONS = ("none", "sum_not_mean", "no_weight", "silu_gate", "eps_outside_sqrt")


def gated_rmsnorm(o, z, w, eps: float, mutation: str = "none") -> np.ndarray:
    """o, z: [..., V]; w: [V].  Returns y of the same shape (float64)."""
    o = np.asarray(o, np.float64)
    z = np.asarray(z, np.float64)
    w = np.asarray(w, np.float64)
    if mutation not in MUTATIONS:
        raise ValueError(mutation)
    sq = o * o
    ms = sq.sum(-1, keepdims=True) if mutation == "sum_not_mean" else sq.mean(-1, keepdims=True)
    if mutation == "eps_outside_sqrt":
        inv = 1.0 / (np.sqrt(ms) + eps)
    else:
        inv = 1.0 / np.sqrt(ms + eps)
    gate = z / (1.0 + np.exp(-z)) if mutation == "silu_gate" else 1.0 / (1.0 + np.exp(-z))
    scale = np.ones_like(w) if mutation == "no_weight" else w
    return o * inv * scale * gate
