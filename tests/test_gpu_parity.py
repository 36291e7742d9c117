"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances: attention output max-abs 2e-3 (bf16 inputs, fp32 accumulate);
s within 1e-4 relative (+1e-7 absolute floor for s near 0); tiers and every
stored byte bit-exact; outputs bitwise identical across T0/T1 splits."""
import math

import numpy as np
import pytest
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from oracle import fp8, tiering
from tiered_kv_cache_gqa_gb300 import synth

from harness import ATOL_OUT, check_scores, f64, gpu_step, lockstep, make_session, prefill_both

pytestmark = pytest.mark.gpu


def test_tiny_workload_lockstep():
    """The Tiny configuration: 1 layer, 4/2 heads, d 64, 512 positions, 128 decode steps with
    re-tiers after steps 64 and 128 (steps 65..128 read T1 from the staging ring and skip T3)."""
    wl = synth.WORKLOADS["tiny"]
    ctx, sess, worst = lockstep(wl, wl.decode_steps)
    st = ctx.stats()
    assert st["retiers"] == 2
    assert st["tier_count"][1] > 0 and st["tier_count"][3] == math.floor(0.03 * 640)
    assert st["h2d_bytes_t1_stream"] > 0


SHAPES = {
    # name: (L, Hq, Hkv, d, B, prefill, steps, ratios, outliers)
    "g4_d128_b2_t2": (2, 16, 4, 128, 2, 900, 70, (0.40, 0.35, 0.15, 0.10), 0.01),
    "g5_d128": (1, 40, 8, 128, 1, 700, 66, (0.50, 0.47, 0.0, 0.03), 0.0),
    "g7_d128": (2, 28, 4, 128, 1, 1100, 66, (0.30, 0.67, 0.0, 0.03), 0.0),
    "g8_d128_long": (1, 64, 8, 128, 1, 2100, 65, (0.30, 0.60, 0.05, 0.05), 0.001),
    "g1_d64": (1, 3, 3, 64, 3, 300, 66, (0.5, 0.3, 0.1, 0.1), 0.0),
    # odd and even half-warp head splits: G = 3 (2 + 1 heads), G = 6 (3 + 3), G = 8 at d 64
    "g3_d64_b2": (2, 6, 2, 64, 2, 500, 66, (0.4, 0.4, 0.1, 0.1), 0.005),
    "g6_d128": (1, 24, 4, 128, 1, 800, 66, (0.3, 0.6, 0.05, 0.05), 0.0),
    "g8_d64_b2": (1, 16, 2, 64, 2, 700, 66, (0.3, 0.5, 0.15, 0.05), 0.01),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_shapes_lockstep(name):
    L, Hq, Hkv, d, B, pre, steps, ratios, orate = SHAPES[name]
    wl = synth.Workload(name, L, Hq, Hkv, d, B, prompt_len=32, prefill_len=pre, decode_steps=steps,
                        window=32, ratios=ratios, outlier_rate=orate, seed=hash(name) % 1000)
    ctx, sess, worst = lockstep(wl, steps)
    tiers = ctx.tiers()
    if ratios[2] > 0:
        assert (tiers == 2).any()
    assert (tiers == 1).any() and (tiers == 3).any()


def _split_tiers(N, wl, evicted, t1_share, rng):
    prot = tiering.protected_mask(N, wl.prompt_len, wl.num_sinks, wl.window)
    t = np.zeros(N, dtype=np.uint8)
    t[evicted] = 3
    free = np.nonzero(~prot & (t != 3))[0]
    t[rng.permutation(free)[: int(round(t1_share * len(free)))]] = 1
    return t


def test_proposition_1_bitwise_across_hbm_split():
    """Same evicted set, T0 share 30 / 50 / 70 %: outputs and scores must be bit-identical."""
    wl = synth.Workload("prop1", 2, 16, 4, 128, 2, prompt_len=16, prefill_len=1500, decode_steps=3,
                        window=16, ratios=(0.3, 0.67, 0.0, 0.03), seed=11)
    gen = synth.Generator(wl)
    K, V = gen.prefill()
    steps = [gen.decode_step(t) for t in range(1, 4)]
    rng = np.random.default_rng(3)
    N = wl.prefill_len
    prot = tiering.protected_mask(N, wl.prompt_len, wl.num_sinks, wl.window)
    evicted = [rng.choice(np.nonzero(~prot)[0], size=60, replace=False) for _ in range(wl.batch)]
    results = []
    for t0_share in (0.3, 0.5, 0.7):
        ctx = tkv.TieredKV.for_workload(wl)
        for l in range(wl.num_layers):
            ctx.append(l, K[l].contiguous().cuda(), V[l].contiguous().cuda(), N)
        tiers = np.stack([_split_tiers(N, wl, evicted[b], 1 - t0_share, np.random.default_rng(b))
                          for b in range(wl.batch)])
        ctx.set_tiers(tiers)
        assert np.array_equal(ctx.tiers(), tiers)
        out = torch.empty(len(steps), wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim,
                          device="cuda")
        for i, (q, k, v) in enumerate(steps):
            gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out[i])
        results.append((out.cpu(), ctx.scores(), ctx.stats()))
    for o, s, st in results[1:]:
        assert torch.equal(o, results[0][0])
        assert np.array_equal(s, results[0][1])
    assert results[0][2]["tier_count"][1] > results[2][2]["tier_count"][1]
    # and the common result is the oracle's
    sess = make_session(wl)
    sess.prefill(K.float().numpy(), V.float().numpy())
    t = np.zeros((wl.batch, N), dtype=np.uint8)
    for b in range(wl.batch):
        t[b, evicted[b]] = 3
    sess.apply_tiers(t)
    for i, (q, k, v) in enumerate(steps):
        ref = sess.step(q.float().numpy(), k.float().numpy(), v.float().numpy(), auto_retier=False)
        assert np.abs(results[0][0][i].numpy() - ref).max() <= ATOL_OUT
    check_scores(results[0][1], sess.scores())


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_retier_bit_exact_on_fed_scores(seed):
    """Tiers from fed fp32 scores (random, and with many exact ties) equal the oracle's."""
    rng = np.random.default_rng(seed)
    wl = synth.Workload("fed", 1, 8, 2, 64, 4, prompt_len=20, prefill_len=3000, decode_steps=1,
                        window=50, ratios=(0.25, 0.45, 0.2, 0.1), seed=seed)
    gen = synth.Generator(wl)
    ctx = tkv.TieredKV.for_workload(wl)
    prefill_both(ctx, None, gen)
    old = np.zeros((wl.batch, wl.prefill_len), dtype=np.uint8)
    ppm = tuple(tiering.ratio_ppm(r) for r in wl.ratios)
    for rnd in range(3):
        s = rng.random((wl.batch, wl.prefill_len)).astype(np.float32)
        s[1] = np.round(s[1] * 4) / 4                 # heavy ties
        s[2] = 0.0                                    # all equal
        s[3, ::7] = s[3, 1::7][: len(s[3, ::7])] if rnd else s[3, ::7]
        ctx.set_scores(s)
        ctx.retier()
        got = ctx.tiers()
        for b in range(wl.batch):
            want = tiering.assign_tiers(s[b].astype(np.float64), old[b], wl.prefill_len, wl.prompt_len,
                                        wl.num_sinks, wl.window, ppm)
            assert np.array_equal(got[b], want), (rnd, b, np.argwhere(got[b] != want)[:10].tolist())
        old = got


def test_stored_rows_byte_exact_through_every_move():
    """T1 writeback, E4M3 codes and scales, delta prefetch back into T0 (from T1 and from T2):
    every stored byte equals the original bf16 row or the oracle's quantisation of it."""
    wl = synth.Workload("rows", 2, 8, 2, 128, 2, prompt_len=8, prefill_len=400, decode_steps=2,
                        window=8, ratios=(0.5, 0.3, 0.15, 0.05), outlier_rate=0.02, seed=5)
    gen = synth.Generator(wl)
    ctx = tkv.TieredKV.for_workload(wl)
    K, V = prefill_both(ctx, None, gen)
    Kb = K.view(torch.int16).numpy().view(np.uint16)      # [L][B][n][Hkv][d] bf16 bits
    Vb = V.view(torch.int16).numpy().view(np.uint16)
    rng = np.random.default_rng(0)
    N = wl.prefill_len
    tiers = np.zeros((wl.batch, N), dtype=np.uint8)
    for b in range(wl.batch):
        tiers[b, 8 + rng.permutation(N - 16)[:150]] = 1
        idx2 = np.nonzero(tiers[b] == 0)[0]
        idx2 = idx2[(idx2 >= 8) & (idx2 < N - 8)]
        tiers[b, rng.permutation(idx2)[:60]] = 2
    ctx.set_tiers(tiers)

    def original(l, b, i):
        return np.stack([Kb[l, b, i], Vb[l, b, i]])       # [2][Hkv][d]

    for b in range(wl.batch):
        for l in range(wl.num_layers):
            for i in np.nonzero(tiers[b] == 1)[0][:40]:
                t, data, _ = ctx.row(l, b, int(i))
                assert t == 1 and np.array_equal(data, original(l, b, i))
            for i in np.nonzero(tiers[b] == 2)[0][:40]:
                t, codes, scales = ctx.row(l, b, int(i))
                assert t == 2
                orig = np.stack([K[l, b, i].float().numpy(), V[l, b, i].float().numpy()])
                for kv in range(2):
                    for h in range(wl.num_kv_heads):
                        c_ref, s_ref = fp8.quantise_row(orig[kv, h])
                        assert scales[kv, h] == s_ref
                        assert np.array_equal(codes[kv, h], c_ref)
    # promote everything back to T0: rows come back through the delta prefetch of the next step
    back = np.zeros_like(tiers)
    ctx.set_tiers(back)
    q, k, v = gen.decode_step(1)
    out = torch.empty(wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim, device="cuda")
    gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out)
    for b in range(wl.batch):
        for l in range(wl.num_layers):
            for i in list(np.nonzero(tiers[b] == 1)[0][:30]) + list(np.nonzero(tiers[b] == 2)[0][:30]):
                t, data, _ = ctx.row(l, b, int(i))
                assert t == 0 and np.array_equal(data, original(l, b, i)), (l, b, i)
    st = ctx.stats()
    assert st["last_promoted"] == int((tiers != 0).sum())


def test_first_token_attends_to_itself():
    """N = 1: alpha = 1 and o = v (closed form); s of that token becomes 1."""
    ctx = tkv.TieredKV(num_layers=2, num_q_heads=8, num_kv_heads=2, head_dim=128, batch=2,
                       max_tokens=8, prompt_len=0, num_sinks=0, recent_window=0,
                       ratios=(1.0, 0.0, 0.0, 0.0))
    g = torch.Generator().manual_seed(0)
    q = torch.randn(2, 2, 8, 128, generator=g).bfloat16().cuda()
    k = torch.randn(2, 2, 2, 128, generator=g).bfloat16().cuda()
    v = torch.randn(2, 2, 2, 128, generator=g).bfloat16().cuda()
    out = torch.empty(2, 2, 8, 128, device="cuda")
    gpu_step(ctx, q, k, v, out)
    want = v.float().repeat_interleave(4, dim=2)
    assert torch.equal(out, want)
    assert np.array_equal(ctx.scores(), np.ones((2, 1), dtype=np.float32))


def test_everything_protected_and_empty_tiers():
    """Prompt covers every position: a re-tier keeps all in T0, T1 is empty, no copies run."""
    wl = synth.Workload("prot", 1, 4, 2, 64, 1, prompt_len=200, prefill_len=150, decode_steps=64,
                        window=64, ratios=(0.2, 0.5, 0.0, 0.3), seed=2)
    ctx, sess, worst = lockstep(wl, 64)
    assert (ctx.tiers() == 0).all()
    assert ctx.stats()["h2d_bytes_t1_stream"] == 0


def test_call_order_and_capacity_errors_leave_context_usable():
    ctx = tkv.TieredKV(num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=64, batch=1,
                       max_tokens=10, prompt_len=2, num_sinks=1, recent_window=2,
                       ratios=(0.5, 0.5, 0.0, 0.0))
    k = torch.zeros(1, 12, 2, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, 4, 64, device="cuda")
    lib = tkv.load()
    assert tkv.tkv_append(ctx.ctx, 1, k, k, 1) == tkv.TKV_EINVAL          # layer 0 first
    kflat = k.view(-1)
    assert tkv.tkv_append(ctx.ctx, 0, kflat[1:].data_ptr(), k, 1) == tkv.TKV_EINVAL   # k not 16-byte aligned
    assert tkv.tkv_append(ctx.ctx, 0, k, kflat[4:].data_ptr(), 1) == tkv.TKV_EINVAL   # v not 16-byte aligned
    assert tkv.tkv_append(ctx.ctx, 0, k, k, 11) == tkv.TKV_ECAPACITY       # beyond max_tokens
    assert tkv.tkv_decode_step(ctx.ctx, 0, q, out) == tkv.TKV_EINVAL       # nothing open
    assert tkv.tkv_retier(ctx.ctx) == tkv.TKV_OK
    ctx.append(0, k, k, 10)
    assert tkv.tkv_retier(ctx.ctx) == tkv.TKV_EINVAL                       # prefill group open
    ctx.append(1, k, k, 10)
    assert tkv.tkv_append(ctx.ctx, 0, k, k, 1) == tkv.TKV_ECAPACITY        # full
    assert ctx.stats()["status"] == tkv.TKV_OK
    assert ctx.tiers().shape == (1, 10)
    bad = np.zeros((1, 10), dtype=np.uint8)
    bad[0, 5] = 3
    ctx.set_tiers(bad)
    bad[0, 5] = 0
    assert tkv.tkv_set_tiers(ctx.ctx, bad) == tkv.TKV_EINVAL               # no coming back from T3
    ctx.sync()


def test_prefetch_ahead_of_layer_0_applies_every_layers_delta():
    """Layers prefetched out of order -- prefetch(1) before decode_step(0), layer 0 never
    prefetched explicitly -- across re-tiers that promote rows: every layer still reads its
    promoted rows from T0 (lockstep with the oracle on out, s and tiers every step)."""
    wl = synth.Workload("ahead", 3, 16, 4, 128, 2, prompt_len=16, prefill_len=600, decode_steps=48,
                        window=16, delta=16, ratios=(0.3, 0.6, 0.05, 0.05), seed=12)
    promoted = []
    ctx, sess, worst = lockstep(wl, 48, order="ahead",
                                on_retier=lambda t, c: promoted.append(c.stats()["last_promoted"]))
    assert len(promoted) == 3 and sum(promoted[1:]) > 0


def test_contexts_of_different_capacities_coexist():
    """A context created after another, with smaller tier stores, must not break the first's
    re-tiers (kernel launch limits are shared by every context of the process)."""
    big = synth.Workload("big", 1, 8, 2, 128, 2, prompt_len=16, prefill_len=6000, decode_steps=64,
                         window=16, ratios=(0.3, 0.6, 0.05, 0.05), seed=15)
    small = big.with_(name="small", prefill_len=300, seed=16)
    ctx_big, sess, worst = lockstep(big, 1)
    ctx_small, _, _ = lockstep(small, 64)          # creates, steps and re-tiers the small one
    gen = synth.Generator(big)
    out = torch.empty(1, big.batch, big.num_q_heads, big.head_dim, device="cuda")
    for t in range(2, 65):
        q, k, v = gen.decode_step(t)
        gpu_step(ctx_big, q.cuda(), k.cuda(), v.cuda(), out)
        sess.step(q.float().numpy(), k.float().numpy(), v.float().numpy(), auto_retier=False)
    ctx_big.retier()
    s_gpu = ctx_big.scores()
    assert np.array_equal(ctx_big.tiers(), sess.assign(rank_scores=s_gpu.astype(np.float64)))
    ctx_small.retier()
    assert ctx_big.stats()["status"] == ctx_small.stats()["status"] == tkv.TKV_OK


def test_set_tiers_refuses_to_evict_a_protected_position():
    """Sinks, prompt and recent window are never evicted: tkv_set_tiers returns EINVAL and
    changes nothing; an unprotected position can be evicted."""
    ctx = tkv.TieredKV(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=64, batch=1,
                       max_tokens=32, prompt_len=6, num_sinks=2, recent_window=4,
                       ratios=(0.5, 0.5, 0.0, 0.0))
    k = torch.zeros(1, 20, 2, 64, dtype=torch.bfloat16, device="cuda")
    ctx.append(0, k, k, 20)
    for pos in (0, 5, 16, 19):                      # sink, prompt, window (N - W = 16), last
        bad = np.zeros((1, 20), dtype=np.uint8)
        bad[0, pos] = 3
        assert tkv.tkv_set_tiers(ctx.ctx, bad) == tkv.TKV_EINVAL, pos
        assert (ctx.tiers() == 0).all()
    ok = np.zeros((1, 20), dtype=np.uint8)
    ok[0, 10] = 3
    ctx.set_tiers(ok)
    assert np.array_equal(ctx.tiers(), ok)
    assert ctx.stats()["status"] == tkv.TKV_OK


def test_t1_transports_are_bitwise_identical():
    """Copy engine, SM copy kernel, the split of both, four copy streams and the HBM-resident
    copy kept by the re-tier put the same bytes in the rows the kernel reads: outputs and scores
    are bit-identical across the five transports (the copy-engine transport is the one the
    lockstep tests compare with the oracle; the resident copy has its own lockstep test below).
    The resident copy streams nothing per step."""
    wl = synth.Workload("t1x", 3, 16, 4, 128, 2, prompt_len=16, prefill_len=900, decode_steps=70,
                        window=16, ratios=(0.3, 0.6, 0.05, 0.05), seed=8)
    outs = []
    for mode in (tkv.TKV_T1_COPY_ENGINE, tkv.TKV_T1_SM_COPY, tkv.TKV_T1_SPLIT, tkv.TKV_T1_MULTI_CE,
                 tkv.TKV_T1_RESIDENT):
        gen = synth.Generator(wl)
        ctx = tkv.TieredKV.for_workload(wl, t1_transport=mode)
        prefill_both(ctx, None, gen)
        res = []
        out = torch.empty(wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim, device="cuda")
        for t in range(1, 71):
            q, k, v = gen.decode_step(t)
            gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out)
            if t % 64 == 0:
                ctx.retier()
            if t > 64:
                res.append(out.cpu().clone())
        outs.append((torch.stack(res), ctx.scores(), ctx.stats()["h2d_bytes_t1_stream"]))
    assert outs[0][2] > 0 and outs[-1][2] == 0
    for o, s, _ in outs[1:]:
        assert torch.equal(o, outs[0][0])
        assert np.array_equal(s, outs[0][1])


def test_host_store_allocations_are_bitwise_identical():
    """The host stores as huge-page arenas assembled from measured units and registered with
    CUDA, or as cudaHostAlloc blocks: the same bytes reach the kernel, so outputs, scores and
    tiers are bit-identical across re-tiers that write back, quantise and promote through those
    stores.  The T1 store here spans several arena units (32 layers x 16,384 slots, 2 GiB)."""
    wl = synth.Workload("hostalloc", 32, 16, 4, 128, 2, prompt_len=16, prefill_len=900, decode_steps=70,
                        window=16, delta=32, ratios=(0.3, 0.5, 0.15, 0.05), seed=14)
    runs = []
    for mode in (tkv.TKV_HOST_HUGE_ARENA, tkv.TKV_HOST_PINNED_ALLOC):
        for t2 in (tkv.TKV_T2_HBM, tkv.TKV_T2_HOST):
            gen = synth.Generator(wl)
            ctx = tkv.TieredKV.for_workload(wl, host_alloc=mode, t2_placement=t2, max_tokens=16384)
            prefill_both(ctx, None, gen)
            out = torch.empty(wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim, device="cuda")
            res = []
            for t in range(1, 71):
                q, k, v = gen.decode_step(t)
                gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out)
                if t % wl.delta == 0:
                    ctx.retier()
                if t > 32:
                    res.append(out.cpu().clone())
            st = ctx.stats()
            runs.append((torch.stack(res), ctx.scores(), ctx.tiers(), st))
            ctx.close()
    for o, s, t, st in runs[1:]:
        assert torch.equal(o, runs[0][0])
        assert np.array_equal(s, runs[0][1]) and np.array_equal(t, runs[0][2])
    assert runs[2][3]["host_huge_bytes"] == 0 and runs[0][3]["host_huge_bytes"] >= 0


def test_resident_t1_lockstep_with_the_oracle():
    """TKV_T1_RESIDENT (the HBM copy of T1 kept by the re-tier's moves) in lockstep with the
    fp64 oracle: out, s and tiers every step, across two re-tiers that demote, promote,
    quantise and evict."""
    wl = synth.Workload("t1res", 3, 16, 4, 128, 2, prompt_len=16, prefill_len=900, decode_steps=70,
                        window=16, delta=32, ratios=(0.3, 0.55, 0.1, 0.05), outlier_rate=0.01, seed=13)
    promoted = []
    ctx, sess, worst = lockstep(wl, 70, t1_transport=tkv.TKV_T1_RESIDENT,
                                on_retier=lambda t, c: promoted.append(c.stats()["last_promoted"]))
    st = ctx.stats()
    assert st["h2d_bytes_t1_stream"] == 0 and st["retiers"] == 2 and promoted[1] > 0
    assert st["tier_count"][1] > 0 and st["tier_count"][2] > 0 and st["tier_count"][3] > 0


def test_t2_on_host_matches_t2_in_hbm_bitwise_and_the_oracle():
    """T2 records in pinned host memory, staged per layer with the T1 rows, against the HBM
    pool: the kernel reads the same bytes, so outputs, scores, tiers and stored records are
    identical; the host placement also runs in lockstep with the oracle."""
    wl = synth.Workload("t2host", 3, 16, 4, 128, 2, prompt_len=16, prefill_len=900, decode_steps=70,
                        window=16, ratios=(0.3, 0.4, 0.25, 0.05), outlier_rate=0.01, seed=9)
    runs = []
    for place in (tkv.TKV_T2_HBM, tkv.TKV_T2_HOST):
        gen = synth.Generator(wl)
        ctx = tkv.TieredKV.for_workload(wl, t2_placement=place)
        prefill_both(ctx, None, gen)
        out = torch.empty(wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim, device="cuda")
        res = []
        for t in range(1, 71):
            q, k, v = gen.decode_step(t)
            gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out)
            if t % 64 == 0:
                ctx.retier()
            if t > 64:
                res.append(out.cpu().clone())
        tiers = ctx.tiers()
        recs = [ctx.row(l, b, int(i)) for l in range(wl.num_layers) for b in range(wl.batch)
                for i in np.nonzero(tiers[b] == 2)[0][:20]]
        runs.append((torch.stack(res), ctx.scores(), tiers, ctx.stats(), recs))
    (o0, s0, t0, st0, r0), (o1, s1, t1, st1, r1) = runs
    assert (t0 == 2).sum() > 100
    assert torch.equal(o0, o1)
    assert np.array_equal(s0, s1) and np.array_equal(t0, t1)
    assert st0["h2d_bytes_t2_stream"] == 0 < st1["h2d_bytes_t2_stream"]
    assert st1["hbm_bytes_kv_resident"] < st0["hbm_bytes_kv_resident"]
    for (ta, ca, sa), (tb, cb, sb) in zip(r0, r1):
        assert ta == tb == 2 and np.array_equal(ca, cb) and np.array_equal(sa, sb)
    _, _, worst = lockstep(wl, 70, t2_placement=tkv.TKV_T2_HOST)
    assert worst <= ATOL_OUT
