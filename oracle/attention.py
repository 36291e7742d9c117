"""Decode-step attention over a tiered KV cache, and the score update.  Test infrastructure.

Source: gist.science summary of "Not All Thoughts Need HBM":
  * "Zero-approximation-error offloading": a T1 token is prefetched to the GPU
    at full precision before the attention step, so it contributes exactly the
    term it would have contributed had it never left HBM.  Proposition 1: the
    approximation error depends only on the evicted set T3, not on the T0/T1
    split.
  * "Importance scoring": at each decode step t,
        s_i(t) = s_i(t-1) + (1/|L|) sum_{l in L} (1/H) sum_{h=1..H} alpha_{l,h}(t)[i]
ARKV summary, "Tri-state cache assignment": quantised tokens are dequantised on
the fly and concatenated with the others in their original order before
attention.

Readings where the pages are silent: softmax scale 1/sqrt(d); evicted tokens are
excluded from both numerator and denominator; under GQA query head h reads KV
head floor(h / G), G = Hq / Hkv; H in the score equation is the number of query
heads; the token being decoded is appended before attention and attends to
itself.

All arithmetic is fp64 on bf16-exact inputs.
"""

import numpy as np


def attend(q, K, V, G: int):
    """Attention of every query head over a list of retained rows.

    q  -- [Hq, d]       query of the decoded token, fp64
    K  -- [R, Hkv, d]   keys of the retained tokens, in logical (position) order
    V  -- [R, Hkv, d]   values, same order
    G  -- query heads per KV head

    Returns (o [Hq, d], alpha [Hq, R]).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, d = q.shape
    R = K.shape[0]
    o = np.zeros((Hq, d))
    alpha = np.zeros((Hq, R))
    for h in range(Hq):
        g = h // G
        z = K[:, g, :] @ q[h] / np.sqrt(d)
        z = z - z.max()
        e = np.exp(z)
        a = e / e.sum()
        alpha[h] = a
        o[h] = a @ V[:, g, :]
    return o, alpha


def score_increment(alpha_per_layer, num_layers: int) -> np.ndarray:
    """(1/|L|) sum_l (1/H) sum_h alpha_{l,h}[i] for one decode step.

    alpha_per_layer -- list over layers of [Hq, R] arrays (same retained order).
    """
    inc = None
    for a in alpha_per_layer:
        H = a.shape[0]
        term = a.sum(axis=0) / H
        inc = term if inc is None else inc + term
    return inc / num_layers
