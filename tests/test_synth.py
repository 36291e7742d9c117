"""The synthetic input recipe (CPU): every slice regenerates alone, and the
generator has the stated structure -- 1 % heavy hitters shared by layers and
heads with K += 4u, queries boosted by sqrt(d)/2 along u, u drifting by 30
degrees per epoch, 0.1 % outlier channels scaled x20."""
import math

import numpy as np
import pytest
import torch

from tiered_kv_cache_gqa_gb300 import synth

WL = synth.Workload("synth", 3, 8, 2, 64, 2, prompt_len=16, prefill_len=3000, decode_steps=600,
                    window=16, drift_every=256, seed=5)


def test_slices_regenerate_alone():
    g1, g2 = synth.Generator(WL), synth.Generator(WL)
    k_all, v_all = g1.kv_rows(1, 2, 0, 700)
    k_mid, v_mid = g2.kv_rows(1, 2, 333, 200)           # starts and ends inside 64-row blocks
    assert torch.equal(k_all[:, 333:533], k_mid) and torch.equal(v_all[:, 333:533], v_mid)
    q1, k1, v1 = g1.decode_step(7)
    q2, k2, v2 = synth.Generator(WL).decode_step(7)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    assert not torch.equal(q1, g1.decode_step(8)[0])
    assert not torch.equal(synth.Generator(WL.with_(seed=6)).kv_rows(0, 0, 0, 64)[0], g1.kv_rows(0, 0, 0, 64)[0])


def test_heavy_hitters_shared_and_boosted():
    g = synth.Generator(WL)
    hh = g.heavy_hitters(0, 0, WL.prefill_len).numpy()
    assert 0.005 < hh.mean() < 0.02                      # 1 % of positions
    assert np.array_equal(hh, synth.Generator(WL).heavy_hitters(0, 0, WL.prefill_len).numpy())
    # K of a heavy hitter carries +4u: its projection on u averages 4, other rows 0
    for layer in range(WL.num_layers):
        k, _ = g.kv_rows(0, layer, 0, WL.prefill_len)   # [Hkv][N][d]
        u = g.u_at(0)[layer]                             # [Hkv][d]
        proj = torch.einsum("hnd,hd->hn", k.float(), u).numpy()
        assert abs(proj[:, hh].mean() - WL.hh_gain) < 0.3
        assert abs(proj[:, ~hh].mean()) < 0.1


def test_query_boost_along_u():
    g = synth.Generator(WL)
    beta = math.sqrt(WL.head_dim) / 2
    proj = []
    for t in range(1, 40):
        q, _, _ = g.decode_step(t)                       # [L][B][Hq][d]
        u = g.u_at(g.epoch_of_step(t)).repeat_interleave(WL.group, dim=1)   # [L][Hq][d]
        proj.append(torch.einsum("lbhd,lhd->lbh", q.float(), u).flatten())
    assert abs(torch.cat(proj).mean().item() - beta) < 0.2


def test_drift_turns_u_by_30_degrees_per_epoch():
    g = synth.Generator(WL)
    assert g.epoch_of_step(256) == 0 and g.epoch_of_step(257) == 1
    for e in range(1, 4):
        a, b = g.u_at(e - 1), g.u_at(e)
        assert torch.allclose(b.norm(dim=-1), torch.ones(b.shape[:-1]), atol=1e-5)
        cos = (a * b).sum(-1)
        assert torch.allclose(cos, torch.full_like(cos, math.cos(math.pi / 6)), atol=1e-5)


def test_outlier_channels():
    wl = WL.with_(outlier_rate=0.02, num_kv_heads=2, num_q_heads=8)
    g = synth.Generator(wl)
    gain = g.channel_gain                                # [2][L][Hkv][d]
    frac = (gain > 1).float().mean().item()
    assert 0.005 < frac < 0.04
    assert set(np.unique(gain.numpy()).tolist()) == {1.0, wl.outlier_gain}
    k, v = g.kv_rows(1, 0, 0, 2000)                      # [Hkv][N][d]
    sd = k.float().std(dim=1)                            # per (head, channel)
    big = gain[0, 0] > 1
    if bool(big.any()):
        assert sd[big].min().item() > 10 * sd[~big].max().item() / 2
    assert synth.Generator(WL).channel_gain is None
