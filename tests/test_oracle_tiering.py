"""Pins for the oracle's tier assignment: hand-worked cases (tests/golden/tiering_cases.txt)
and a brute-force pairwise check of the ranking rule on random and tie-heavy inputs."""
import os

import numpy as np
import pytest

from oracle import tiering

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiering_cases.txt")


def load_cases():
    lines = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    cases, i = [], 0
    while i < len(lines):
        assert lines[i][0] == "case"
        N, prompt, sinks, window = map(int, lines[i + 1])
        ratios = tuple(float(x) for x in lines[i + 2])
        old = np.array([int(x) for x in lines[i + 3][1:]], dtype=np.uint8)
        s = np.array([0.0 if x == "-" else float(x) for x in lines[i + 4][1:]])
        new = np.array([int(x) for x in lines[i + 5][1:]], dtype=np.uint8)
        assert len(old) == len(s) == len(new) == N
        cases.append((lines[i][1], N, prompt, sinks, window, ratios, old, s, new))
        i += 6
    return cases


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c[0])
def test_golden(case):
    name, N, prompt, sinks, window, ratios, old, s, want = case
    ppm = tuple(tiering.ratio_ppm(r) for r in ratios)
    got = tiering.assign_tiers(s, old, N, prompt, sinks, window, ppm)
    assert got.tolist() == want.tolist()


def check_rules(s, old, new, N, prompt, sinks, window, ppm):
    prot = np.zeros(N, bool)
    prot[:sinks] = True
    prot[:prompt] = True
    prot[max(N - window, 0):] = True
    assert np.all(new[prot] == 0)
    assert np.all(new[old == 3] == 3)
    cand = np.nonzero(~prot & (old != 3))[0]
    # brute force over pairs: a candidate placed in a better tier outranks one in a worse tier
    rank_tier = {0: 0, 1: 1, 2: 2, 3: 3}
    for i in cand:
        for j in cand:
            if rank_tier[int(new[i])] < rank_tier[int(new[j])]:
                assert (s[i] > s[j]) or (s[i] == s[j] and i < j), (i, j)
    # counts
    n_prot = int(prot.sum())
    n0 = max(n_prot, ppm[0] * N // 10**6)
    n2 = ppm[2] * N // 10**6
    n3 = ppm[3] * N // 10**6
    e_old = int((old == 3).sum())
    n_ev = min(max(n3 - e_old, 0), len(cand))
    m = len(cand) - n_ev
    c0 = min(n0 - n_prot, m)
    c2 = min(n2, m - c0)
    assert int((new == 3).sum()) == e_old + n_ev
    assert int((new[cand] == 0).sum()) == c0
    assert int((new == 2).sum()) == c2
    assert int((new == 1).sum()) == m - c0 - c2


@pytest.mark.parametrize("seed", range(12))
def test_random_and_tie_heavy_inputs(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 90))
    prompt, sinks, window = int(rng.integers(0, 8)), int(rng.integers(0, 5)), int(rng.integers(0, 12))
    raw = rng.dirichlet(np.ones(4))
    ppm = tuple(int(x) for x in np.round(raw * 1e6))
    if seed % 2:
        s = rng.integers(0, 3, N).astype(np.float64) / 4.0      # many exact ties
    else:
        s = rng.random(N)
    old = np.zeros(N, dtype=np.uint8)
    prot = tiering.protected_mask(N, prompt, sinks, window)
    ev = (rng.random(N) < 0.1) & ~prot
    old[ev] = 3
    new = tiering.assign_tiers(s, old, N, prompt, sinks, window, ppm)
    check_rules(s, old, new, N, prompt, sinks, window, ppm)


def test_ratio_counts_are_exact_integers():
    # floor(ppm * N / 1e6) in integer arithmetic: 0.29 * 100 is 29, not 28
    assert tiering.count_of(tiering.ratio_ppm(0.29), 100) == 29
    assert tiering.count_of(tiering.ratio_ppm(0.03), 576) == 17
    assert tiering.count_of(tiering.ratio_ppm(0.5), 576) == 288


def test_protected_mask():
    p = tiering.protected_mask(20, 3, 4, 5)
    assert np.nonzero(p)[0].tolist() == [0, 1, 2, 3, 15, 16, 17, 18, 19]
