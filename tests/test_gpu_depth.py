"""GPU parity at real stack depth and at the largest re-tier size.

* The 7B-shaped stack at its full depth (28 layers, 28/4 heads, d 128, batch 1)
  over about a thousand positions, 70 decode steps across a re-tier, in
  lockstep with the fp64 oracle: attention output (max-abs 2e-3) and the
  cumulative score s (1e-4 relative) every step -- s sums the attention weights
  over all 28 layers and 28 query heads ("Importance scoring") -- and the tiers
  bit-exact at the re-tier.
* The re-tier at the 70B-shaped size (batch 8, 16,384 positions per sequence):
  tiers from fed fp32 scores, random and tie-heavy, bit-exact against the
  oracle's assignment, over two rounds (the second starts from the first's
  tiers, so it promotes, demotes and evicts)."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from oracle import tiering
from tiered_kv_cache_gqa_gb300 import synth

from harness import lockstep

pytestmark = pytest.mark.gpu


def test_7b_stack_depth_lockstep_across_a_retier():
    wl = synth.WORKLOADS["7b"].with_(prefill_len=960, decode_steps=70, seed=31)
    retiers = []
    ctx, sess, worst = lockstep(wl, 70, on_retier=lambda t, c: retiers.append(c.stats()["tier_count"]))
    assert len(retiers) == 1 and retiers[0][1] > 0 and retiers[0][3] > 0
    # steps 65..70 read T1 rows from the staging ring and skip the evicted rows
    assert ctx.stats()["h2d_bytes_t1_stream"] > 0


def test_retier_bit_exact_at_the_70b_size():
    WL = synth.WORKLOADS["70b"]
    B, N = WL.batch, 16384
    ctx = tkv.TieredKV(num_layers=1, num_q_heads=WL.num_q_heads, num_kv_heads=WL.num_kv_heads,
                       head_dim=WL.head_dim, batch=B, max_tokens=N, prompt_len=WL.prompt_len,
                       num_sinks=WL.num_sinks, recent_window=WL.window,
                       ratios=(0.28, 0.6, 0.09, 0.03))
    k = torch.randn(B, N, WL.num_kv_heads, WL.head_dim, generator=torch.Generator().manual_seed(0))
    k = k.to(torch.bfloat16).cuda()
    ctx.append(0, k, k, N)
    del k
    ppm = tuple(tiering.ratio_ppm(r) for r in (0.28, 0.6, 0.09, 0.03))
    old = np.zeros((B, N), dtype=np.uint8)
    rng = np.random.default_rng(7)
    for rnd in range(2):
        s = rng.random((B, N)).astype(np.float32)
        s[1] = np.round(s[1] * 8) / 8                    # heavy ties
        s[2] = 0.5                                       # all equal
        i3 = np.arange(0, N - 1, 3)
        s[3, i3] = s[3, i3 + 1]                          # pairs of equal scores
        s[4] = np.float32(1e-7) * rng.integers(0, 4, N)  # tiny values, many ties
        ctx.set_scores(s)
        ctx.retier()
        got = ctx.tiers()
        for b in range(B):
            want = tiering.assign_tiers(s[b].astype(np.float64), old[b], N, WL.prompt_len,
                                        WL.num_sinks, WL.window, ppm)
            assert np.array_equal(got[b], want), (rnd, b, np.argwhere(got[b] != want)[:10].tolist())
        counts = [(got == t).sum() for t in range(4)]
        assert all(c > 0 for c in counts)
        old = got
    assert ctx.stats()["status"] == tkv.TKV_OK
