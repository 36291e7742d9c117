"""Tier assignment by cumulative attention score.  Test infrastructure.

Source: gist.science summary of "Not All Thoughts Need HBM":
  * "Four-tier classification": T0 (HBM) holds the protected tokens -- the
    prompt, the attention sinks and the recent window -- and the most important
    reasoning tokens; T1 (DDR) medium-importance tokens at full precision;
    T2 low-importance tokens at 8-bit; T3 only the least important tail,
    discarded permanently.
  * "System implementation": tiers are re-assigned every Delta = 64 decode
    steps (which amortises the sort).

Readings taken where the pages are silent:
  * the ranking key is (s descending, position ascending): on an exact tie in
    s the lower position ranks higher, so the higher position is evicted
    first;
  * tier sizes are fractions of N, the number of positions so far (evicted
    ones included), rounded down; a ratio is held as an integer number of
    parts per million, so  n_k = floor(ppm_k * N / 10^6)  exactly;
  * T3 only grows: its target n3 is cumulative and evicted tokens never come
    back; protected tokens are never evicted, so T3 may fall short;
  * T0's target n0 = max(|P|, n0) includes the protected set P;
  * after the evictions, the remaining m unprotected tokens are handed out
    from the top: T0 gets min(n0 - |P|, m), T2 gets min(n2, rest), T1 gets what
    is left -- so when P is too large, T1 shrinks first, then T2;
  * ranks [0, c0) -> T0, [c0, c0+c1) -> T1, [c0+c1, m) -> T2, the tail -> T3.
"""

import numpy as np

PPM = 1_000_000


def ratio_ppm(r: float) -> int:
    """A tier ratio as integer parts per million (round to nearest)."""
    return int(round(float(r) * PPM))


def count_of(ppm: int, n: int) -> int:
    """floor(ppm * n / 10^6) in exact integer arithmetic."""
    return (int(ppm) * int(n)) // PPM


def protected_mask(N: int, prompt_len: int, num_sinks: int, window: int) -> np.ndarray:
    """P = sinks [0, num_sinks)  U  prompt [0, prompt_len)  U  recent window [N-W, N)."""
    p = np.zeros(N, dtype=bool)
    p[: min(num_sinks, N)] = True
    p[: min(prompt_len, N)] = True
    p[max(N - window, 0):N] = True
    return p


def tier_targets(N: int, ppm: tuple, n_protected: int):
    """Targets (n0, n2, n3) for N positions; n1 is whatever remains."""
    n0 = max(n_protected, count_of(ppm[0], N))
    n2 = count_of(ppm[2], N)
    n3 = count_of(ppm[3], N)
    return n0, n2, n3


def rank_order(candidates: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Candidates sorted best-first by (s descending, position ascending)."""
    cand = [int(i) for i in candidates]
    cand.sort(key=lambda i: (-float(s[i]), i))
    return np.array(cand, dtype=np.int64)


def assign_tiers(s, old_tiers, N: int, prompt_len: int, num_sinks: int, window: int,
                 ratios_ppm: tuple) -> np.ndarray:
    """New tier (0..3) of each of the N positions.

    s          -- cumulative scores, length >= N (compared as given: feed fp32
                  values to compare with an fp32 implementation)
    old_tiers  -- current tiers, length >= N; positions appended since the last
                  re-tier are in T0; T3 entries stay T3
    ratios_ppm -- (T0, T1, T2, T3) ratios in parts per million
    """
    s = np.asarray(s)[:N]
    old = np.asarray(old_tiers)[:N].astype(np.int64)
    prot = protected_mask(N, prompt_len, num_sinks, window)
    evicted_old = old == 3
    if np.any(prot & evicted_old):
        raise ValueError("a protected position is already evicted")
    n0, n2, n3 = tier_targets(N, ratios_ppm, int(prot.sum()))

    new = np.full(N, -1, dtype=np.int64)
    new[prot] = 0
    new[evicted_old] = 3

    cand = np.nonzero(~prot & ~evicted_old)[0]
    order = rank_order(cand, s)
    n_cand = len(order)

    n_evict = min(max(n3 - int(evicted_old.sum()), 0), n_cand)
    m = n_cand - n_evict
    c0 = min(n0 - int(prot.sum()), m)
    c2 = min(n2, m - c0)
    c1 = m - c0 - c2

    new[order[:c0]] = 0
    new[order[c0:c0 + c1]] = 1
    new[order[c0 + c1:m]] = 2
    new[order[m:]] = 3
    assert np.all(new >= 0)
    return new.astype(np.uint8)
