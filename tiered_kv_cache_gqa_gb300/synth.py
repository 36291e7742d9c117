"""Seeded synthetic workloads for tiered decode attention.

This module only draws inputs (queries, keys, values) and describes workload
shapes.  It holds none of the method's arithmetic, imports neither the CUDA
binding nor the oracle, and is the one piece both of them are fed from.

Workload shapes follow the attention stacks the pages evaluate on ("Not All
Thoughts Need HBM": 7B, 14B and 32B models; a 70B batch-8 projection for the
HBM savings).  There is no public dataset behind them here: the long reasoning
chains of the pages' benchmarks are stood in for by this recipe.

Recipe (all draws fp32, then rounded to bf16 with round-to-nearest-even):
  * K, V, Q entries ~ N(0, 1);
  * per (layer, KV head) a random unit vector u;
  * heavy hitters: each position is one with probability 0.01, the same set
    for every layer and head; a heavy hitter's key gets K += 4 u;
  * every decode query of the group that reads KV head g gets q += beta u,
    beta = sqrt(d) / 2 (so a heavy hitter's logit is raised by about 2);
  * optional drift: every `drift_every` decode steps u <- cos(theta) u +
    sin(theta) w, w a fresh unit vector orthogonal to u, theta = pi / 6;
  * optional outlier channels: each (layer, KV head, channel) is, with
    probability `outlier_rate`, scaled by `outlier_gain` at every position,
    independently for K and V.
Every draw is keyed by (seed, sequence, layer, kind, position or step) so any
slice can be regenerated on its own.
"""

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    batch: int
    prompt_len: int
    prefill_len: int          # positions present before the first decode step (prompt included)
    decode_steps: int
    num_sinks: int = 4
    window: int = 64
    delta: int = 64
    ratios: tuple = (1.0, 0.0, 0.0, 0.0)   # (T0, T1, T2, T3)
    hh_rate: float = 0.01
    hh_gain: float = 4.0
    drift_every: int = 0
    drift_theta: float = math.pi / 6
    outlier_rate: float = 0.0
    outlier_gain: float = 20.0
    seed: int = 0

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_tokens(self):
        return self.prefill_len + self.decode_steps

    def with_(self, **kw):
        return replace(self, **kw)


# Shapes of the configurations the pages' experiments use.  Where a sequence
# length is long, `prefill_len` fast-forwards to the end state (filled
# positions are drawn exactly like decoded ones), then a short decode runs.
WORKLOADS = {
    # 1 layer, 4/2 heads, d 64: 64-token prompt + 448 pre-filled, 128 decode
    # steps (re-tier after step 64, then 64 steps that read T1 and skip T3).
    "tiny": Workload("tiny", 1, 4, 2, 64, 1, prompt_len=64, prefill_len=512,
                     decode_steps=128, window=64, ratios=(0.50, 0.47, 0.0, 0.03)),
    # 7B-shaped: 28 layers, 28/4 heads, d 128, batch 1; 512-token prompt and
    # 2000 decode steps with drift every 256 steps.  HBM ratio 30/50/70 %.
    "7b": Workload("7b", 28, 28, 4, 128, 1, prompt_len=512, prefill_len=512,
                   decode_steps=2000, window=64, ratios=(0.50, 0.47, 0.0, 0.03),
                   drift_every=256),
    # 14B-shaped: 48 layers, 40/8 heads, batch 8; 1024 prompt + 3072 decode.
    "14b": Workload("14b", 48, 40, 8, 128, 8, prompt_len=1024, prefill_len=1024,
                    decode_steps=3072, window=128, ratios=(0.50, 0.47, 0.0, 0.03)),
    # 32B-shaped: 64 layers, 40/8 heads, batch 4, 8192 tokens; T2 15 % fp8,
    # 0.1 % outlier channels x20.
    "32b": Workload("32b", 64, 40, 8, 128, 4, prompt_len=512, prefill_len=8064,
                    decode_steps=128, window=64, ratios=(0.40, 0.40, 0.15, 0.05),
                    outlier_rate=0.001),
    # 70B-shaped: 80 layers, 64/8 heads, batch 8, 16384 tokens per sequence.
    "70b": Workload("70b", 80, 64, 8, 128, 8, prompt_len=1024, prefill_len=16256,
                    decode_steps=128, window=64, ratios=(0.30, 0.67, 0.0, 0.03)),
}


def _gen(device, *key):
    g = torch.Generator(device=device)
    h = 0
    for k in key:
        h = (h * 1_000_003 + int(k)) % (2 ** 62)
    g.manual_seed(h)
    return g


def _stable_str_key(s: str) -> int:
    # Python's str hash is salted per process; use a fixed polynomial instead.
    h = 0
    for ch in s.encode():
        h = (h * 131 + ch) % (2 ** 61)
    return h


def _key(*parts):
    return tuple(_stable_str_key(p) if isinstance(p, str) else int(p) for p in parts)


class Generator:
    """Draws the inputs of one workload on a given torch device."""

    def __init__(self, wl: Workload, device="cpu"):
        self.wl = wl
        self.device = torch.device(device)
        L, Hkv, d = wl.num_layers, wl.num_kv_heads, wl.head_dim
        g = _gen(self.device, *_key(wl.seed, "u"))
        u = torch.randn(L, Hkv, d, generator=g, device=self.device)
        self.u0 = u / u.norm(dim=-1, keepdim=True)
        self._u_cache = {0: self.u0}
        if wl.outlier_rate > 0:
            g = _gen(self.device, *_key(wl.seed, "outliers"))
            r = torch.rand(2, L, Hkv, d, generator=g, device=self.device)
            self.channel_gain = torch.where(r < wl.outlier_rate,
                                            torch.tensor(wl.outlier_gain, device=self.device),
                                            torch.tensor(1.0, device=self.device))
        else:
            self.channel_gain = None
        # Caches of values already drawn (pure memoisation: a value never depends on whether it
        # came from a cache): heavy-hitter offsets per (sequence, block), and the last K/V block
        # drawn per (sequence, layer), which successive decode positions share.
        self._hh_cache = {}
        self._blk_cache = {}

    # ----------------------------------------------------------- direction u
    def u_at(self, epoch: int):
        """u for drift epoch `epoch` ([L, Hkv, d], unit rows)."""
        if epoch in self._u_cache:
            return self._u_cache[epoch]
        prev = self.u_at(epoch - 1)
        g = _gen(self.device, *_key(self.wl.seed, "drift", epoch))
        w = torch.randn(prev.shape, generator=g, device=self.device)
        w = w - (w * prev).sum(-1, keepdim=True) * prev
        w = w / w.norm(dim=-1, keepdim=True)
        th = self.wl.drift_theta
        u = math.cos(th) * prev + math.sin(th) * w
        u = u / u.norm(dim=-1, keepdim=True)
        self._u_cache[epoch] = u
        return u

    def epoch_of_step(self, step: int):
        """Drift epoch of decode step `step` (steps count from 1)."""
        if self.wl.drift_every <= 0:
            return 0
        return (step - 1) // self.wl.drift_every

    def epoch_of_position(self, pos: int):
        """Drift epoch in force when position `pos` was produced."""
        step = pos - self.wl.prefill_len + 1
        return self.epoch_of_step(step) if step >= 1 else 0

    # ------------------------------------------------------- heavy hitters
    def heavy_hitters(self, b: int, start: int, n: int):
        """bool[n]: which of positions [start, start+n) of sequence b are heavy hitters."""
        g = _gen(self.device, *_key(self.wl.seed, "hh", b))
        total = start + n
        r = torch.rand(total, generator=g, device=self.device)
        return r[start:total] < self.wl.hh_rate

    # ----------------------------------------------------------- K / V rows
    BLOCK = 64   # positions drawn together; a row's value does not depend on the slice asked for

    def _hh_offsets(self, b: int, blk: int):
        """Offsets within block `blk` of sequence b that are heavy hitters (a list)."""
        key = (b, blk)
        if key not in self._hh_cache:
            hh = self.heavy_hitters(b, blk * self.BLOCK, self.BLOCK)
            self._hh_cache[key] = torch.nonzero(hh).flatten().tolist()
        return self._hh_cache[key]

    def _kv_block(self, b: int, layer: int, blk: int):
        key = (b, layer)
        hit = self._blk_cache.get(key)
        if hit is not None and hit[0] == blk:
            return hit[1]
        wl = self.wl
        Hkv, d, n = wl.num_kv_heads, wl.head_dim, self.BLOCK
        start = blk * n
        g = _gen(self.device, *_key(wl.seed, "kv", b, layer, blk))
        kv = torch.randn(2, Hkv, n, d, generator=g, device=self.device)
        for j in self._hh_offsets(b, blk):
            u = self.u_at(self.epoch_of_position(start + j))[layer]   # [Hkv, d]
            kv[0, :, j, :] += wl.hh_gain * u
        if self.channel_gain is not None:
            kv = kv * self.channel_gain[:, layer][:, :, None, :]
        kv = kv.to(torch.bfloat16)
        self._blk_cache[key] = (blk, kv)
        return kv

    def kv_rows(self, b: int, layer: int, start: int, n: int):
        """K, V of positions [start, start+n) of (sequence b, layer): [Hkv, n, d] bf16."""
        first, last = start // self.BLOCK, (start + n - 1) // self.BLOCK
        blocks = torch.cat([self._kv_block(b, layer, k) for k in range(first, last + 1)], dim=2)
        off = start - first * self.BLOCK
        kv = blocks[:, :, off:off + n, :]
        return kv[0], kv[1]

    def prefill_layer(self, layer: int, n: int = None):
        """K, V of the first n positions of one layer: [B][n][Hkv][d] bf16 each."""
        wl = self.wl
        n = wl.prefill_len if n is None else n
        K = torch.empty(wl.batch, n, wl.num_kv_heads, wl.head_dim, dtype=torch.bfloat16,
                        device=self.device)
        V = torch.empty_like(K)
        for b in range(wl.batch):
            k, v = self.kv_rows(b, layer, 0, n)
            K[b] = k.transpose(0, 1)
            V[b] = v.transpose(0, 1)
        return K, V

    def prefill(self, n: int = None):
        """K, V of the first n positions: [L][B][n][Hkv][d] bf16 each."""
        wl = self.wl
        n = wl.prefill_len if n is None else n
        K = torch.empty(wl.num_layers, wl.batch, n, wl.num_kv_heads, wl.head_dim,
                        dtype=torch.bfloat16, device=self.device)
        V = torch.empty_like(K)
        for l in range(wl.num_layers):
            K[l], V[l] = self.prefill_layer(l, n)
        return K, V

    def decode_step(self, step: int):
        """Inputs of decode step `step` (from 1): q [L][B][Hq][d], k, v [L][B][Hkv][d], bf16."""
        wl = self.wl
        L, B, Hq, Hkv, d = wl.num_layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
        pos = wl.prefill_len + step - 1
        u = self.u_at(self.epoch_of_step(step))               # [L, Hkv, d]
        q = torch.empty(L, B, Hq, d, dtype=torch.bfloat16, device=self.device)
        k = torch.empty(L, B, Hkv, d, dtype=torch.bfloat16, device=self.device)
        v = torch.empty_like(k)
        beta = math.sqrt(d) / 2.0
        for b in range(B):
            g = _gen(self.device, *_key(wl.seed, "q", b, step))
            qq = torch.randn(L, Hq, d, generator=g, device=self.device)
            qq = qq + beta * u.repeat_interleave(wl.group, dim=1)
            q[:, b] = qq.to(torch.bfloat16)
            for l in range(L):
                kk, vv = self.kv_rows(b, l, pos, 1)
                k[l, b] = kk[:, 0]
                v[l, b] = vv[:, 0]
        return q, k, v
