"""Pins for the oracle's decode session: Proposition 1 (output independent of the
T0/T1 split at a fixed evicted set) as an exact equality, equivalence with library
attention masked over the evicted set, the per-step invariant sum_i delta s_i = 1,
and the re-tier cadence (every Delta steps) and rules."""
import numpy as np
import pytest
import torch

from oracle import fp8, session, tiering
from tiered_kv_cache_gqa_gb300 import synth


def tiny(**kw):
    wl = synth.WORKLOADS["tiny"]
    return wl.with_(**kw)


def make_session(wl):
    return session.Session(wl.num_layers, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                           wl.batch, wl.prompt_len, wl.num_sinks, wl.window, wl.delta, wl.ratios)


def as_np(t):
    return t.float().numpy()


def run(wl, steps, sess=None):
    gen = synth.Generator(wl)
    sess = sess or make_session(wl)
    K, V = gen.prefill()
    sess.prefill(as_np(K), as_np(V))
    outs = []
    for t in range(1, steps + 1):
        q, k, v = gen.decode_step(t)
        outs.append(sess.step(as_np(q), as_np(k), as_np(v)))
    return sess, outs


def dense_attention(q, K, V, G, keep):
    qt = torch.from_numpy(q)[:, None, :]
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    m = torch.from_numpy(keep)[None, None, :].expand(qt.shape[0], 1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=m)[:, 0].numpy()


def test_score_sum_grows_by_one_per_step_and_retier_every_delta():
    wl = tiny(prefill_len=160, prompt_len=16, decode_steps=40, delta=16, window=8)
    gen = synth.Generator(wl)
    sess = make_session(wl)
    K, V = gen.prefill()
    sess.prefill(as_np(K), as_np(V))
    changes = []
    for t in range(1, 41):
        before = sess.tier_map().copy()
        q, k, v = gen.decode_step(t)
        sess.step(as_np(q), as_np(k), as_np(v))
        assert abs(sess.scores().sum() - t) < 1e-12 * t
        after = sess.tier_map()
        changes.append(not np.array_equal(after[:, :before.shape[1]], before))
    assert [i + 1 for i, c in enumerate(changes) if c] == [16, 32]
    tiers = sess.tier_map()[0]
    N = sess.N
    assert int((tiers == 3).sum()) == tiering.count_of(tiering.ratio_ppm(wl.ratios[3]), 32 + 160)
    assert np.all(tiers[:wl.prompt_len] == 0)


def test_matches_library_attention_masked_by_evicted_set():
    wl = tiny(prefill_len=200, decode_steps=24, delta=8, window=16,
              ratios=(0.3, 0.5, 0.0, 0.2))
    gen = synth.Generator(wl)
    sess = make_session(wl)
    K, V = gen.prefill()
    sess.prefill(as_np(K), as_np(V))
    allK = [as_np(K)[0, 0]]
    allV = [as_np(V)[0, 0]]
    for t in range(1, 25):
        q, k, v = gen.decode_step(t)
        tiers_before = sess.tier_map()[0]
        out = sess.step(as_np(q), as_np(k), as_np(v))
        allK.append(as_np(k)[0, 0][None])
        allV.append(as_np(v)[0, 0][None])
        Kd = np.concatenate(allK).astype(np.float64)
        Vd = np.concatenate(allV).astype(np.float64)
        keep = np.concatenate([tiers_before, [0]]) != 3
        ref = dense_attention(as_np(q)[0, 0].astype(np.float64), Kd, Vd, wl.group, keep)
        np.testing.assert_allclose(out[0, 0], ref, rtol=1e-11, atol=1e-12)
    assert int((sess.tier_map()[0] == 3).sum()) > 0


def test_proposition_1_output_independent_of_hbm_split():
    """Same evicted set, T0 share 30/50/70 %: outputs must be identical, bit for bit."""
    base = tiny(prefill_len=300, decode_steps=12, delta=1000)
    gen = synth.Generator(base)
    K, V = gen.prefill()
    steps = [gen.decode_step(t) for t in range(1, 13)]
    rng = np.random.default_rng(0)
    N0 = base.prefill_len
    prot = tiering.protected_mask(N0, base.prompt_len, base.num_sinks, base.window)
    cand = np.nonzero(~prot)[0]
    evicted = rng.choice(cand, size=9, replace=False)
    rest = np.setdiff1d(cand, evicted)
    results = []
    for share in (0.3, 0.5, 0.7):
        sess = make_session(base)
        sess.prefill(as_np(K), as_np(V))
        tiers = np.zeros((1, N0), dtype=np.uint8)
        tiers[0, evicted] = 3
        n_t1 = int(round((1 - share) * len(rest)))
        tiers[0, rng.permutation(rest)[:n_t1]] = 1
        sess.apply_tiers(tiers)
        outs = [sess.step(as_np(q), as_np(k), as_np(v)) for q, k, v in steps]
        results.append((np.stack(outs), sess.scores()))
    for o, s in results[1:]:
        assert np.array_equal(o, results[0][0])
        assert np.array_equal(s, results[0][1])


def test_t2_rows_are_dequantised_and_t2_promotion_restores_full_precision():
    wl = tiny(prefill_len=120, decode_steps=4, delta=1000, outlier_rate=0.05)
    gen = synth.Generator(wl)
    sess = make_session(wl)
    K, V = gen.prefill()
    sess.prefill(as_np(K), as_np(V))
    tiers = np.zeros((1, 120), dtype=np.uint8)
    tiers[0, 70:90] = 2
    sess.apply_tiers(tiers)
    # T2 rows are the codec's dequantised rows (codec pinned in test_oracle_fp8)
    Kf = as_np(K)[0, 0]
    for i in (70, 80, 89):
        for g in range(wl.num_kv_heads):
            codes, scale = fp8.quantise_row(Kf[i, g])
            assert np.array_equal(sess._row(0, i)[0][0, g], fp8.dequantise_row(codes, scale))
            assert not np.array_equal(sess._row(0, i)[0][0, g], Kf[i, g].astype(np.float64))
    q, k, v = gen.decode_step(1)
    out = sess.step(as_np(q), as_np(k), as_np(v), auto_retier=False)
    Kd = np.concatenate([Kf, as_np(k)[0, 0][None]]).astype(np.float64)
    Vd = np.concatenate([as_np(V)[0, 0], as_np(v)[0, 0][None]]).astype(np.float64)
    for i in range(70, 90):
        Kd[i] = sess._row(0, i)[0][0]
        Vd[i] = sess._row(0, i)[1][0]
    ref = dense_attention(as_np(q)[0, 0].astype(np.float64), Kd, Vd, wl.group,
                          np.ones(121, dtype=bool))
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-11, atol=1e-12)
    # promote back: exact bf16 values again
    tiers = sess.tier_map().copy()
    tiers[0, 70:90] = 1
    sess.apply_tiers(tiers)
    assert np.array_equal(sess._row(0, 75)[0][0], Kf[75])


def test_evicted_position_cannot_return():
    wl = tiny(prefill_len=100, decode_steps=1)
    sess = make_session(wl)
    gen = synth.Generator(wl)
    K, V = gen.prefill()
    sess.prefill(as_np(K), as_np(V))
    t = np.zeros((1, 100), dtype=np.uint8)
    t[0, 80] = 3
    sess.apply_tiers(t)
    t[0, 80] = 0
    with pytest.raises(ValueError):
        sess.apply_tiers(t)
