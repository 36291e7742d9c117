"""CUDA-graph decode steps (tkv_capture_begin / tkv_capture_end / tkv_replay)
against eager steps.

A replayed step runs the kernels and copies of the calls it was captured from,
so outputs, scores and tiers must be bit-identical to an eager run of the same
steps.  A captured step is valid only while its launch geometry covers the
retained counts (the run crosses such a boundary and re-captures), and a
re-tier discards it (the step after a re-tier carries the delta prefetch and
runs eagerly)."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from tiered_kv_cache_gqa_gb300 import synth

from harness import gpu_step, prefill_both

pytestmark = pytest.mark.gpu

WL = synth.Workload("graph", 3, 16, 4, 128, 2, prompt_len=16, prefill_len=600, decode_steps=140,
                    window=16, ratios=(0.4, 0.5, 0.05, 0.05), seed=31)
STEPS = 140


def run(use_graph, t1_mode, t2_place=tkv.TKV_T2_HBM):
    gen = synth.Generator(WL)
    ctx = tkv.TieredKV.for_workload(WL, t1_transport=t1_mode, t2_placement=t2_place)
    prefill_both(ctx, None, gen)
    L, B, Hq, Hkv, d = WL.num_layers, WL.batch, WL.num_q_heads, WL.num_kv_heads, WL.head_dim
    out = torch.empty(L, B, Hq, d, device="cuda")
    # a captured step reads the buffers it was captured with: inputs go through fixed ones
    sq = torch.empty(L, B, Hq, d, dtype=torch.bfloat16, device="cuda")
    sk = torch.empty(L, B, Hkv, d, dtype=torch.bfloat16, device="cuda")
    sv = torch.empty_like(sk)
    outs, left, replays, captures = [], 0, 0, 0
    for t in range(1, STEPS + 1):
        q, k, v = gen.decode_step(t)
        sq.copy_(q)
        sk.copy_(k)
        sv.copy_(v)
        if use_graph and left == 0 and (t == 1 or (t - 1) % WL.delta != 0):
            ctx.capture_begin()
            gpu_step(ctx, sq, sk, sv, out)      # recorded, not run
            left = ctx.capture_end()
            captures += 1
        if use_graph and left > 0:
            ctx.replay()
            left -= 1
            replays += 1
        else:
            gpu_step(ctx, sq, sk, sv, out)
        outs.append(out.cpu().clone())
        if t % WL.delta == 0:
            ctx.retier()
            left = 0
    st = ctx.stats()
    res = (torch.stack(outs), ctx.scores(), ctx.tiers(), st["step"], st["num_tokens"])
    return res, replays, captures, ctx


@pytest.mark.parametrize("t1_mode,t2_place", [(tkv.TKV_T1_COPY_ENGINE, tkv.TKV_T2_HBM),
                                              (tkv.TKV_T1_SM_COPY, tkv.TKV_T2_HBM),
                                              (tkv.TKV_T1_RESIDENT, tkv.TKV_T2_HBM),
                                              (tkv.TKV_T1_MULTI_CE, tkv.TKV_T2_HBM),
                                              (tkv.TKV_T1_COPY_ENGINE, tkv.TKV_T2_HOST)])
def test_replayed_steps_match_eager_steps_bitwise(t1_mode, t2_place):
    ref, _, _, _ = run(False, tkv.TKV_T1_COPY_ENGINE)
    got, replays, captures, ctx = run(True, t1_mode, t2_place)
    assert replays > 100 and captures >= 4          # geometry boundaries and re-tiers re-capture
    assert torch.equal(got[0], ref[0])
    assert np.array_equal(got[1], ref[1])
    assert np.array_equal(got[2], ref[2])
    assert got[3] == ref[3] == STEPS
    assert got[4] == ref[4] == WL.prefill_len + STEPS
    # a re-tier discards the graph
    ctx.retier()
    with pytest.raises(tkv.TkvError):
        ctx.replay()


def test_capture_of_a_partial_step_is_refused_and_leaves_the_context_usable():
    gen = synth.Generator(WL)
    ctx = tkv.TieredKV.for_workload(WL)
    prefill_both(ctx, None, gen)
    L, B, Hq, d = WL.num_layers, WL.batch, WL.num_q_heads, WL.head_dim
    out = torch.empty(L, B, Hq, d, device="cuda")
    q, k, v = (x.cuda() for x in gen.decode_step(1))
    ctx.capture_begin()
    ctx.append(0, k[0], v[0], 1)                    # not a whole step
    with pytest.raises(tkv.TkvError):
        ctx.capture_end()
    with pytest.raises(tkv.TkvError):
        ctx.replay()
    gpu_step(ctx, q, k, v, out)                     # the same step, eagerly
    assert ctx.stats()["num_tokens"] == WL.prefill_len + 1
    ref_ctx = tkv.TieredKV.for_workload(WL)
    prefill_both(ref_ctx, None, synth.Generator(WL))
    ref = torch.empty_like(out)
    gpu_step(ref_ctx, q, k, v, ref)
    assert torch.equal(out, ref)
    assert np.array_equal(ctx.scores(), ref_ctx.scores())
