"""Pins for the oracle's decode attention and score increment: torch's
scaled_dot_product_attention in fp64 (a library routine), closed forms, and the
invariant that each step adds exactly 1 to the sum of scores."""
import math

import numpy as np
import pytest
import torch

from oracle import attention


def sdpa_gqa(q, K, V, G, keep=None):
    """Library attention for one decode query per head: q [Hq,d], K/V [N,Hkv,d]."""
    qt = torch.from_numpy(q)[:, None, :]                       # [Hq, 1, d]
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq, N, d]
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    mask = None
    if keep is not None:
        mask = torch.from_numpy(keep)[None, None, :].expand(qt.shape[0], 1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("Hq,Hkv,d,N", [(4, 2, 64, 37), (8, 1, 16, 5), (6, 3, 8, 200), (5, 5, 32, 1)])
def test_matches_library_attention(Hq, Hkv, d, N):
    rng = np.random.default_rng(Hq * 1000 + N)
    q = rng.standard_normal((Hq, d))
    K = rng.standard_normal((N, Hkv, d)) * 2
    V = rng.standard_normal((N, Hkv, d))
    G = Hq // Hkv
    o, a = attention.attend(q, K, V, G)
    np.testing.assert_allclose(o, sdpa_gqa(q, K, V, G), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a.sum(axis=1), 1.0, rtol=0, atol=1e-14)


def test_masked_equals_attention_over_retained_subset():
    rng = np.random.default_rng(7)
    Hq, Hkv, d, N = 4, 2, 32, 50
    q = rng.standard_normal((Hq, d))
    K = rng.standard_normal((N, Hkv, d))
    V = rng.standard_normal((N, Hkv, d))
    keep = rng.random(N) > 0.3
    keep[-1] = True
    R = np.nonzero(keep)[0]
    o, _ = attention.attend(q, K[R], V[R], 2)
    np.testing.assert_allclose(o, sdpa_gqa(q, K, V, 2, keep), rtol=1e-12, atol=1e-13)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((1, 2, 16))
    V = rng.standard_normal((1, 2, 16))
    o, a = attention.attend(q, K, V, 2)
    assert np.array_equal(a, np.ones((4, 1)))
    assert np.array_equal(o, np.repeat(V[0], 2, axis=0))


def test_equal_keys_give_the_mean_value():
    rng = np.random.default_rng(4)
    N = 9
    K = np.repeat(rng.standard_normal((1, 1, 8)), N, axis=0)
    V = rng.standard_normal((N, 1, 8))
    o, a = attention.attend(rng.standard_normal((3, 8)), K, V, 3)
    np.testing.assert_allclose(a, 1.0 / N, rtol=1e-15)
    np.testing.assert_allclose(o, np.repeat(V.mean(axis=0), 3, axis=0), rtol=1e-13)


def test_closed_form_logits():
    # d = 4 so the scale is 1/2; q = (2,0,0,0) against keys with first entry 0, 1, -1
    # gives logits 0, 1, -1: alpha_1/alpha_0 = alpha_0/alpha_2 = e.
    q = np.array([[2.0, 0, 0, 0]])
    K = np.array([[[0.0, 0, 0, 0]], [[1.0, 0, 0, 0]], [[-1.0, 0, 0, 0]]])
    V = np.eye(4)[[0, 1, 2]][:, None, :]
    o, a = attention.attend(q, K, V, 1)
    assert math.isclose(a[0, 1] / a[0, 0], math.e, rel_tol=1e-15)
    assert math.isclose(a[0, 0] / a[0, 2], math.e, rel_tol=1e-15)
    assert math.isclose(a[0, 0], 1.0 / (1.0 + math.e + 1.0 / math.e), rel_tol=1e-15)
    np.testing.assert_allclose(o[0, :3], a[0], rtol=1e-15)


def test_score_increment_sums_to_one_and_weights_layers_and_heads_equally():
    rng = np.random.default_rng(5)
    L, Hq, R = 3, 4, 11
    alphas = []
    for _ in range(L):
        x = rng.random((Hq, R))
        alphas.append(x / x.sum(axis=1, keepdims=True))
    inc = attention.score_increment(alphas, L)
    assert math.isclose(inc.sum(), 1.0, rel_tol=1e-14)
    # one-hot attention: layer l, head h looks only at token (l*Hq + h) % R;
    # each such (l, h) pair contributes 1/(L*Hq) to that token.
    one_hot = []
    for l in range(L):
        a = np.zeros((Hq, R))
        for h in range(Hq):
            a[h, (l * Hq + h) % R] = 1.0
        one_hot.append(a)
    inc = attention.score_increment(one_hot, L)
    counts = np.bincount([(l * Hq + h) % R for l in range(L) for h in range(Hq)], minlength=R)
    np.testing.assert_allclose(inc, counts / (L * Hq), rtol=1e-15)
