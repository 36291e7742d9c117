"""HBM footprint of the tiered KV cache: what stays resident in HBM and what tiering saves.

"Not All Thoughts Need HBM" (fugumt.com abstract; gist.science summary, results on
system overhead) projects 2-48 GB of HBM saved at production batch sizes.  This module
computes the same quantity for a given shape, batch, sequence length, tier ratios, T1
transport, T2 placement and staging depth, with the library's own accounting
(tkv_stats.hbm_bytes_kv_resident), so a projection can be set next to a measurement.

Byte counts (Hkv KV heads, head dim d, L layers, B sequences):
  * a full-precision row (K and V of one token, one layer): 2 * Hkv * d * 2 bytes;
  * a T2 row: K and V as d E4M3 codes plus a 16-byte slot for the fp32 scale each:
    2 * Hkv * (d + 16) bytes;
  * resident in HBM: every T0 row of every layer; T2 rows of every layer (or, with T2 in
    host memory, the staged layers' T2 rows); the T1 rows of the staged layers (the
    staging ring holds `staging_layers` layers; with the resident-T1 transport all L);
  * the full cache: every position of every layer at full precision.
Tier counts per sequence follow the re-tier's rule: n_k = floor(ratio_k * N) (ratios in
parts per million), T0 at least the protected set, T1 the remainder.
"""
from dataclasses import dataclass

PPM = 1_000_000


def _ppm(r):
    return int(round(float(r) * PPM))


def row_bytes(num_kv_heads, head_dim):
    """K and V of one token in one layer, bf16."""
    return 2 * num_kv_heads * head_dim * 2


def t2_row_bytes(num_kv_heads, head_dim):
    """K and V of one token in one layer as E4M3 codes with their scale slots."""
    return 2 * num_kv_heads * (head_dim + 16)


def protected_count(N, prompt_len, num_sinks, window):
    """|sinks U prompt U last `window` positions| for N positions."""
    a = min(N, max(prompt_len, num_sinks))
    return a + (N - max(a, max(0, N - window)))


def tier_counts(N, ratios, prompt_len=0, num_sinks=0, window=0):
    """Tokens per tier (T0, T1, T2, T3) of one sequence of N positions at steady state
    (T3 at its target: every eviction already made)."""
    P = protected_count(N, prompt_len, num_sinks, window)
    n0 = max(P, _ppm(ratios[0]) * N // PPM)
    n2 = _ppm(ratios[2]) * N // PPM
    n3 = min(_ppm(ratios[3]) * N // PPM, N - P)
    m = N - P - n3
    c0 = min(n0 - P, m)
    c2 = min(n2, m - c0)
    return (P + c0, m - c0 - c2, c2, n3)


@dataclass
class Footprint:
    full_bytes: int          # the whole cache at full precision, in HBM
    resident_bytes: int      # what tiering keeps in HBM
    host_bytes: int          # what lives in pinned host memory (T1 rows, T2 masters / records)

    @property
    def saved_bytes(self):
        return self.full_bytes - self.resident_bytes


def footprint(num_layers, batch, num_kv_heads, head_dim, counts, t1_rows_staged=None,
              staging_layers=2, t1_resident=False, t2_on_host=False, t2_rows_staged=None):
    """HBM footprint for per-sequence tier counts `counts` = (T0, T1, T2, T3) (or a list of
    such tuples, one per sequence).  `t1_rows_staged` / `t2_rows_staged`: rows per sequence
    that one staged layer holds (default: the T1 / T2 count of the largest sequence)."""
    per_seq = [tuple(counts)] * batch if isinstance(counts[0], int) else [tuple(c) for c in counts]
    L = num_layers
    rb, r2 = row_bytes(num_kv_heads, head_dim), t2_row_bytes(num_kv_heads, head_dim)
    n0 = sum(c[0] for c in per_seq)
    n1 = sum(c[1] for c in per_seq)
    n2 = sum(c[2] for c in per_seq)
    N = sum(per_seq[0])
    hw1 = max(c[1] for c in per_seq) if t1_rows_staged is None else t1_rows_staged
    hw2 = max(c[2] for c in per_seq) if t2_rows_staged is None else t2_rows_staged
    t1_layers = L if t1_resident else staging_layers
    t2_hbm = (staging_layers * batch * hw2 * r2) if t2_on_host else n2 * L * r2
    resident = n0 * L * rb + t2_hbm + t1_layers * batch * hw1 * rb
    host = n1 * L * rb + n2 * L * rb + (n2 * L * r2 if t2_on_host else 0)
    return Footprint(full_bytes=batch * N * L * rb, resident_bytes=resident, host_bytes=host)


def projection(num_layers, batch, num_kv_heads, head_dim, N, ratios, prompt_len=0, num_sinks=4,
               window=64, **kw):
    """Footprint of B sequences of N positions at the tier ratios (steady state)."""
    c = tier_counts(N, ratios, prompt_len, num_sinks, window)
    return footprint(num_layers, batch, num_kv_heads, head_dim, c, **kw)


# Shapes of the attention stacks the pages evaluate (L, Hkv, d).
SHAPES = {"7B": (28, 4, 128), "14B": (48, 8, 128), "32B": (64, 8, 128), "70B": (80, 8, 128)}


def table(batches=(1, 8), lengths=(4096, 16384), t0=(0.3, 0.5, 0.7), t3=0.03):
    """Rows (shape, batch, N, T0 ratio, full GB, resident GB, saved GB)."""
    rows = []
    for name, (L, Hkv, d) in SHAPES.items():
        for B in batches:
            for N in lengths:
                for r0 in t0:
                    f = projection(L, B, Hkv, d, N, (r0, 1.0 - r0 - t3, 0.0, t3), prompt_len=1024)
                    rows.append((name, B, N, r0, f.full_bytes / 1e9, f.resident_bytes / 1e9,
                                 f.saved_bytes / 1e9))
    return rows


if __name__ == "__main__":
    print("%-4s %5s %6s %5s %9s %12s %9s" % ("", "batch", "N", "T0", "full GB", "resident GB", "saved GB"))
    for r in table():
        print("%-4s %5d %6d %5.2f %9.2f %12.2f %9.2f" % r)
