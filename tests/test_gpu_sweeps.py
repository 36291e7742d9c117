"""The configuration sweeps at full size: the 7B-shaped stack at HBM (T0) shares of
30 / 50 / 70 % with 3 % evicted, and the 14B-shaped stack on the 3 x 3 grid of HBM
shares 30 / 50 / 70 % x eviction 0 / 3 / 10 % ("Not All Thoughts Need HBM", fugumt.com
abstract: the controlled grid of HBM ratio x eviction; gist.science summary, results on
accuracy vs eviction).

Per grid point, at the configuration's full shape and token count, through the C ABI:
  1. fed fp32 scores (random, with ties) -> tkv_retier: tiers bit-exact against the
     oracle's assignment;
  2. one decode step (the T1 rows cross the host link; s cleared first, so s after the
     step is the step's increment): sampled (layer, sequence, KV head) groups of the
     output within 2e-3 of the oracle, and the increment of s of one sequence, summed by
     the oracle over every layer and query head, within 1e-4 relative;
  3. new scores -> a second re-tier (tiers bit-exact; rows are promoted back) -> a
     decode step that carries the delta prefetch, checked as in 2.
At each eviction level the outputs and increments of the three HBM shares are bitwise
identical (Proposition 1: same evicted set, different T0/T1 split)."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from oracle import attention, tiering
from tiered_kv_cache_gqa_gb300 import synth

from harness import ATOL_OUT, check_scores, gpu_step

pytestmark = pytest.mark.gpu

GRID = {
    # name: (workload, pre-filled positions, evictions, samples (layer, sequence, kv head))
    "7b": ("7b", 2511, (0.03,), [(0, 0, 0), (27, 0, 3), (13, 0, 1)]),
    "14b": ("14b", 4095, (0.0, 0.03, 0.10), [(0, 0, 0), (47, 7, 7), (20, 3, 4)]),
}
T0_SHARES = (0.3, 0.5, 0.7)


def _scores(rng, B, N):
    s = rng.random((B, N)).astype(np.float32)
    s[:, ::5] = np.round(s[:, ::5] * 16) / 16          # ties
    return s


def _oracle_layer(gen, N, tiers_b, q, k, v, layer, b):
    """fp64 output [Hq, d] and attention weights [Hq, R] of one layer of sequence b."""
    kk, vv = gen.kv_rows(b, layer, 0, N)                          # [Hkv][N][d]
    K = torch.cat([kk, k[layer, b][:, None]], dim=1).transpose(0, 1).float().cpu().numpy()
    V = torch.cat([vv, v[layer, b][:, None]], dim=1).transpose(0, 1).float().cpu().numpy()
    keep = np.append(tiers_b, 0) != 3
    return attention.attend(q[layer, b].float().cpu().numpy().astype(np.float64), K[keep], V[keep],
                            gen.wl.group)


def _check_step(WL, gen, N, tiers, q, k, v, out, s_gpu, samples):
    L, G = WL.num_layers, WL.group
    for layer, b, kvh in samples:
        o, _ = _oracle_layer(gen, N, tiers[b], q, k, v, layer, b)
        err = np.abs(out[layer, b].numpy() - o).max()
        assert err <= ATOL_OUT, ((layer, b, kvh), err)
    # s increment of sequence 0 over every layer and query head
    alphas = [_oracle_layer(gen, N, tiers[0], q, k, v, l, 0)[1] for l in range(L)]
    inc = attention.score_increment(alphas, L)
    keep = np.append(tiers[0], 0) != 3
    want = np.zeros(N + 1)
    want[keep] = inc
    check_scores(s_gpu[0], want)


@pytest.mark.parametrize("case", sorted(GRID))
def test_sweep_grid_parity_and_proposition_1(case):
    name, N, evictions, samples = GRID[case]
    base = synth.WORKLOADS[name].with_(prefill_len=N, decode_steps=2, seed=91)
    gen = synth.Generator(base, device="cuda")
    prefill = [gen.prefill_layer(l) for l in range(base.num_layers)]
    steps = [gen.decode_step(t) for t in (1, 2)]
    rng = np.random.default_rng(5)
    fed = [_scores(rng, base.batch, N), _scores(rng, base.batch, N + 1)]
    for t3 in evictions:
        results = []
        for t0 in T0_SHARES:
            WL = base.with_(ratios=(t0, 1.0 - t0 - t3, 0.0, t3))
            ppm = tuple(tiering.ratio_ppm(r) for r in WL.ratios)
            ctx = tkv.TieredKV.for_workload(WL)
            for l in range(WL.num_layers):
                ctx.append(l, prefill[l][0], prefill[l][1], N)
            old = np.zeros((WL.batch, N), np.uint8)
            res = []
            for i, (q, k, v) in enumerate(steps):
                n = N + i
                ctx.set_scores(fed[i][:, :n])
                ctx.retier()
                tiers = ctx.tiers()
                for b in range(WL.batch):
                    want = tiering.assign_tiers(fed[i][b, :n].astype(np.float64), old[b], n, WL.prompt_len,
                                                WL.num_sinks, WL.window, ppm)
                    assert np.array_equal(tiers[b], want), (t0, t3, i, b)
                old = np.concatenate([tiers, np.zeros((WL.batch, 1), np.uint8)], axis=1)
                ctx.set_scores(np.zeros((WL.batch, n), np.float32))
                out = torch.empty(WL.num_layers, WL.batch, WL.num_q_heads, WL.head_dim, device="cuda")
                gpu_step(ctx, q, k, v, out)
                res.append((out.cpu(), ctx.scores(), tiers))
            st = ctx.stats()
            assert st["h2d_bytes_t1_stream"] > 0 and st["last_promoted"] > 0
            ctx.close()
            results.append(res)
        # Proposition 1: the same outputs and increments at every HBM share
        for res in results[1:]:
            for (o, s, t), (o0, s0, t0_) in zip(res, results[0]):
                assert torch.equal(o, o0) and np.array_equal(s, s0)
                assert np.array_equal(t == 3, t0_ == 3)
        # and they are the oracle's
        for i, (o, s, t) in enumerate(results[0]):
            q, k, v = steps[i]
            _check_step(base, gen, N + i, t, q, k, v, o, s, samples)
