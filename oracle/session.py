"""A decode session over the four-tier KV cache.  Test infrastructure.

Source: gist.science summary of "Not All Thoughts Need HBM" -- "Four-tier
classification" (T0 HBM, T1 DDR at full precision, T2 8-bit, T3 evicted),
"Importance scoring" (the s_i update), "Zero-approximation-error offloading"
(T1 rows are fetched back at full precision before attention) and "System
implementation" (re-tier every Delta = 64 decode steps); fugumt.com abstract of
the same paper (tokens are moved to CPU memory rather than destroyed).

Each tier is its own container, and attention reads every token through the
tier map from the container it sits in, so that tests exercise Proposition 1
rather than assume it:

  hbm[b]    T0: position -> (K [L,Hkv,d], V [L,Hkv,d]) bf16-exact values
  ddr[b]    T1: position -> (K, V) at full precision
  t2[b]     T2: position -> dequantised (K, V) computed from the E4M3 codes
  master[b] full-precision copy of every T2 token (kept on the host), so a
            token promoted out of T2 gets its exact values back
  (T3 tokens are dropped from every container.)

Step semantics (readings where the pages are silent):
  * decode steps are numbered from 1; in step t every sequence appends one new
    position N (into T0: it is inside the recent window) before attention, and
    the new position starts with s = 0;
  * pre-filled positions are not scored (s starts at 0 for them too);
  * before the first re-tier every position is in T0;
  * the re-tier runs after the score update of every step t with t % Delta == 0.
"""

import numpy as np

from . import attention, fp8, tiering


class Session:
    def __init__(self, num_layers, num_q_heads, num_kv_heads, head_dim, batch,
                 prompt_len, num_sinks, window, delta, ratios):
        assert num_q_heads % num_kv_heads == 0
        self.L, self.Hq, self.Hkv, self.d, self.B = (num_layers, num_q_heads, num_kv_heads,
                                                     head_dim, batch)
        self.G = num_q_heads // num_kv_heads
        self.prompt_len, self.num_sinks, self.window, self.delta = (prompt_len, num_sinks,
                                                                    window, delta)
        self.ratios_ppm = tuple(tiering.ratio_ppm(r) for r in ratios)
        self.N = 0
        self.step_index = 0
        self.tiers = [[] for _ in range(batch)]
        self.s = [[] for _ in range(batch)]
        self.hbm = [dict() for _ in range(batch)]
        self.ddr = [dict() for _ in range(batch)]
        self.t2 = [dict() for _ in range(batch)]
        self.master = [dict() for _ in range(batch)]

    # ------------------------------------------------------------------ rows
    def _row(self, b, i):
        """Full-precision or dequantised (K, V) of position i, read through its tier."""
        t = self.tiers[b][i]
        if t == 0:
            return self.hbm[b][i]
        if t == 1:
            return self.ddr[b][i]
        if t == 2:
            return self.t2[b][i]
        raise KeyError("position %d of sequence %d is evicted" % (i, b))

    def retained(self, b):
        return [i for i in range(self.N) if self.tiers[b][i] != 3]

    def _append(self, k, v):
        """k, v: [L][B][Hkv][d] arrays of one new position."""
        i = self.N
        for b in range(self.B):
            self.hbm[b][i] = (np.array(k[:, b], dtype=np.float32),
                              np.array(v[:, b], dtype=np.float32))
            self.tiers[b].append(0)
            self.s[b].append(0.0)
        self.N += 1

    # --------------------------------------------------------------- prefill
    def prefill(self, k, v):
        """k, v: [L][B][n][Hkv][d]; positions enter T0 unscored."""
        k = np.asarray(k, dtype=np.float32)
        v = np.asarray(v, dtype=np.float32)
        for j in range(k.shape[2]):
            self._append(k[:, :, j], v[:, :, j])

    # ------------------------------------------------------------------ step
    def attend_layer(self, layer, b, q):
        """o [Hq,d] and alpha [Hq,R] of one layer for sequence b (no state change)."""
        R = self.retained(b)
        K = np.stack([self._row(b, i)[0][layer] for i in R])
        V = np.stack([self._row(b, i)[1][layer] for i in R])
        o, a = attention.attend(q, K, V, self.G)
        return o, a, R

    def step(self, q, k, v, rank_scores=None, auto_retier=True):
        """One decode step for all sequences.

        q: [L][B][Hq][d]; k, v: [L][B][Hkv][d].  Returns out [L][B][Hq][d] (fp64).
        rank_scores, if given, is what a re-tier in this step ranks by
        (a [B][N] array; default: this session's own fp64 scores).
        """
        self._append(np.asarray(k), np.asarray(v))
        out = np.zeros((self.L, self.B, self.Hq, self.d))
        for b in range(self.B):
            alphas = []
            R = None
            for l in range(self.L):
                o, a, R = self.attend_layer(l, b, np.asarray(q[l][b], dtype=np.float64))
                out[l, b] = o
                alphas.append(a)
            inc = attention.score_increment(alphas, self.L)
            for j, i in enumerate(R):
                self.s[b][i] += inc[j]
        self.step_index += 1
        if auto_retier and self.step_index % self.delta == 0:
            self.retier(rank_scores)
        return out

    # ---------------------------------------------------------------- tiers
    def assign(self, rank_scores=None):
        """New tiers [B][N] that a re-tier now would produce (no state change)."""
        new = []
        for b in range(self.B):
            s = np.asarray(self.s[b] if rank_scores is None else rank_scores[b])
            new.append(tiering.assign_tiers(s, np.array(self.tiers[b], dtype=np.uint8), self.N,
                                            self.prompt_len, self.num_sinks, self.window,
                                            self.ratios_ppm))
        return np.stack(new) if new else np.zeros((0, self.N), np.uint8)

    def retier(self, rank_scores=None):
        self.apply_tiers(self.assign(rank_scores))

    def apply_tiers(self, new_tiers):
        """Move every position to the tier given in new_tiers [B][N]."""
        for b in range(self.B):
            for i in range(self.N):
                old, new = self.tiers[b][i], int(new_tiers[b][i])
                if old == new:
                    continue
                if old == 3:
                    raise ValueError("an evicted position cannot come back")
                full = self._full_precision(b, i, old)
                for store in (self.hbm[b], self.ddr[b], self.t2[b], self.master[b]):
                    store.pop(i, None)
                if new == 0:
                    self.hbm[b][i] = full
                elif new == 1:
                    self.ddr[b][i] = full
                elif new == 2:
                    self.master[b][i] = full
                    self.t2[b][i] = self._quantised(full)
                self.tiers[b][i] = new

    def _full_precision(self, b, i, tier):
        if tier == 0:
            return self.hbm[b][i]
        if tier == 1:
            return self.ddr[b][i]
        return self.master[b][i]

    def _quantised(self, full):
        """Dequantised (K, V): one E4M3 row + fp32 scale per (layer, KV head)."""
        out = []
        for x in full:
            deq = np.zeros(x.shape, dtype=np.float64)
            for l in range(x.shape[0]):
                for g in range(x.shape[1]):
                    codes, scale = fp8.quantise_row(x[l, g])
                    deq[l, g] = fp8.dequantise_row(codes, scale)
            out.append(deq)
        return tuple(out)

    # --------------------------------------------------------------- access
    def scores(self):
        return np.array([self.s[b] for b in range(self.B)], dtype=np.float64)

    def tier_map(self):
        return np.array([self.tiers[b] for b in range(self.B)], dtype=np.uint8)
