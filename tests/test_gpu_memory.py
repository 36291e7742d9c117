"""The HBM-footprint calculator against the library's own accounting on the GPU:
tkv_stats.hbm_bytes_kv_resident and kv_bytes_full_cache equal the calculator's
numbers for the tiers the context holds, for each T1 transport and T2 placement."""
import numpy as np
import pytest

import tiered_kv_cache_gqa_gb300 as tkv
from oracle import tiering
from tiered_kv_cache_gqa_gb300 import memory, synth

from harness import prefill_both

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("t1,t2", [(tkv.TKV_T1_COPY_ENGINE, tkv.TKV_T2_HBM),
                                   (tkv.TKV_T1_COPY_ENGINE, tkv.TKV_T2_HOST),
                                   (tkv.TKV_T1_RESIDENT, tkv.TKV_T2_HBM)])
def test_calculator_matches_the_library_accounting(t1, t2):
    wl = synth.Workload("mem", 3, 16, 4, 128, 3, prompt_len=32, prefill_len=1500, decode_steps=1,
                        window=32, ratios=(0.3, 0.5, 0.15, 0.05), seed=18)
    ctx = tkv.TieredKV.for_workload(wl, t1_transport=t1, t2_placement=t2)
    prefill_both(ctx, None, synth.Generator(wl))
    N = wl.prefill_len
    ppm = tuple(tiering.ratio_ppm(r) for r in wl.ratios)
    rng = np.random.default_rng(1)
    tiers = np.stack([tiering.assign_tiers(rng.random(N), np.zeros(N, np.uint8), N, wl.prompt_len,
                                           wl.num_sinks, wl.window, ppm) for _ in range(wl.batch)])
    ctx.set_tiers(tiers)
    st = ctx.stats()
    counts = [tuple(int((tiers[b] == k).sum()) for k in range(4)) for b in range(wl.batch)]
    # steady-state counts of the calculator equal those of the assignment
    assert all(c == memory.tier_counts(N, wl.ratios, wl.prompt_len, wl.num_sinks, wl.window) for c in counts)
    hw2 = int(max(np.nonzero(tiers[b] == 2)[0].size for b in range(wl.batch)))
    f = memory.footprint(wl.num_layers, wl.batch, wl.num_kv_heads, wl.head_dim, counts,
                         t1_rows_staged=st["t1_rows_streamed"], t1_resident=t1 == tkv.TKV_T1_RESIDENT,
                         t2_on_host=t2 == tkv.TKV_T2_HOST, t2_rows_staged=hw2)
    assert st["kv_bytes_full_cache"] == f.full_bytes
    assert st["hbm_bytes_kv_resident"] == f.resident_bytes
    # the re-tier hands out dense T1 slots: one staged layer holds exactly the T1 rows
    assert st["t1_rows_streamed"] == max(c[1] for c in counts)


def test_host_link_probe_reports_the_three_paths():
    rc, link = tkv.tkv_measure_host_link(0, 64 << 20)
    assert rc == tkv.TKV_OK
    for k in ("h2d_ce_gbs", "h2d_sm_gbs", "d2h_ce_gbs"):
        assert 1.0 < link[k] < 2000.0, (k, link[k])
