"""The HBM-footprint calculator (CPU): closed forms, hand-worked tier counts, agreement
with the oracle's tier assignment, and the pages' projection range.

"Not All Thoughts Need HBM" (fugumt.com abstract; gist.science summary, results on
system overhead) projects 2-48 GB of HBM saved at production batch sizes."""
import numpy as np
import pytest

from oracle import tiering
from tiered_kv_cache_gqa_gb300 import memory


def test_full_cache_of_the_70b_shaped_batch():
    # 80 layers x 8 sequences x 16,384 positions x (K + V) x 8 KV heads x 128 x 2 bytes
    f = memory.projection(80, 8, 8, 128, 16384, (1.0, 0.0, 0.0, 0.0))
    assert f.full_bytes == 42_949_672_960
    assert f.resident_bytes == f.full_bytes and f.saved_bytes == 0


def test_tier_counts_hand_worked():
    # P = prompt 50 + window 64 = 114; n0 = max(114, 300); n2 = n3 = 50; T1 takes the rest
    assert memory.tier_counts(1000, (0.3, 0.6, 0.05, 0.05), 50, 4, 64) == (300, 600, 50, 50)
    # the protected set covers every position: nothing leaves T0, nothing is evicted
    assert memory.tier_counts(100, (0.2, 0.5, 0.1, 0.2), 90, 4, 20) == (100, 0, 0, 0)
    # T1 shrinks first, then T2, when the protected set is large
    assert memory.tier_counts(100, (0.1, 0.1, 0.2, 0.1), 60, 4, 20) == (80, 0, 10, 10)


@pytest.mark.parametrize("seed", range(6))
def test_tier_counts_equal_the_oracle_assignment(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(50, 3000))
    prompt, sinks, window = int(rng.integers(0, 200)), int(rng.integers(0, 8)), int(rng.integers(0, 200))
    r = rng.dirichlet(np.ones(4))
    ppm = tuple(tiering.ratio_ppm(x) for x in r)
    ratios = tuple(x / 1e6 for x in ppm[:3]) + (1.0 - sum(ppm[:3]) / 1e6,)
    ppm = tuple(tiering.ratio_ppm(x) for x in ratios)
    t = tiering.assign_tiers(rng.random(N), np.zeros(N, np.uint8), N, prompt, sinks, window, ppm)
    want = tuple(int((t == k).sum()) for k in range(4))
    assert memory.tier_counts(N, ratios, prompt, sinks, window) == want


def test_footprint_hand_worked():
    # 2 layers, 1 sequence, 1 KV head, d 64: row = 256 B, T2 row = 2 * 80 = 160 B
    f = memory.footprint(2, 1, 1, 64, (10, 20, 5, 3))
    assert f.full_bytes == 38 * 2 * 256
    # T0 all layers + T2 all layers + two staged layers of T1
    assert f.resident_bytes == 10 * 2 * 256 + 5 * 2 * 160 + 2 * 20 * 256
    f = memory.footprint(2, 1, 1, 64, (10, 20, 5, 3), t1_resident=True, t2_on_host=True)
    assert f.resident_bytes == 10 * 2 * 256 + 2 * 5 * 160 + 2 * 20 * 256


def test_70b_batch_8_savings_fall_in_the_pages_projection():
    # the pages project 2-48 GB saved at production batch sizes (70B-class, batch 8)
    for r0 in (0.3, 0.5, 0.7):
        f = memory.projection(80, 8, 8, 128, 16384, (r0, 0.97 - r0, 0.0, 0.03), prompt_len=1024)
        assert 2e9 <= f.saved_bytes <= 48e9, (r0, f.saved_bytes)
