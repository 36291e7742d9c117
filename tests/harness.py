"""Shared helpers for the GPU parity tests: drive the CUDA path and the oracle in lockstep."""
import numpy as np
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from oracle import session
from tiered_kv_cache_gqa_gb300 import synth

ATOL_OUT = 2e-3           # attention output, max-abs (bf16 inputs, fp32 accumulate)
S_RTOL, S_ATOL = 1e-4, 1e-7


def make_session(wl):
    return session.Session(wl.num_layers, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.batch,
                           wl.prompt_len, wl.num_sinks, wl.window, wl.delta, wl.ratios)


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def prefill_both(ctx, sess, gen, n=None):
    wl = gen.wl
    n = wl.prefill_len if n is None else n
    K, V = gen.prefill(n)
    for l in range(wl.num_layers):
        ctx.append(l, K[l].contiguous().cuda(), V[l].contiguous().cuda(), n)
    if sess is not None:
        sess.prefill(K.float().numpy(), V.float().numpy())
    return K, V


def gpu_step(ctx, q, k, v, out, order="canonical"):
    """One decode step through the C ABI.

    order="canonical": append(l); prefetch(0) when l == 0; prefetch(l+1); decode_step(l).
    order="ahead": layer 0 is never prefetched explicitly (decode_step(0) issues it, after
    prefetch(1) has run): append(l); prefetch(l+1); decode_step(l)."""
    L = q.shape[0]
    for l in range(L):
        ctx.append(l, k[l], v[l], 1)
        if l == 0 and order == "canonical":
            ctx.prefetch(0)
        if l + 1 < L:
            ctx.prefetch(l + 1)
        ctx.decode_step(l, q[l], out[l])


def check_scores(s_gpu, s_ref):
    err = np.abs(s_gpu.astype(np.float64) - s_ref)
    bound = S_RTOL * np.abs(s_ref) + S_ATOL
    assert np.all(err <= bound), "s mismatch: worst %g (bound %g)" % (
        float(err.max()), float(bound[np.argmax(err - bound)]))


def lockstep(wl, steps, device="cpu", check_out=True, order="canonical", on_retier=None, **ctx_kw):
    """Runs `steps` decode steps on both sides; re-tier every wl.delta steps.

    The re-tier is checked bit-exactly by feeding the GPU's fp32 scores to the
    oracle's tier assignment; both sides then continue from the same tiers.
    `on_retier(t, ctx)` is called after each re-tier.
    Returns (ctx, sess, worst output error)."""
    gen = synth.Generator(wl, device=device)
    ctx = tkv.TieredKV.for_workload(wl, **ctx_kw)
    sess = make_session(wl)
    prefill_both(ctx, sess, gen)
    L, B, Hq, d = wl.num_layers, wl.batch, wl.num_q_heads, wl.head_dim
    out = torch.empty(L, B, Hq, d, dtype=torch.float32, device="cuda")
    worst = 0.0
    for t in range(1, steps + 1):
        q, k, v = gen.decode_step(t)
        gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out, order=order)
        ref = sess.step(q.float().numpy(), k.float().numpy(), v.float().numpy(), auto_retier=False)
        if check_out:
            err = float(np.abs(out.cpu().numpy().astype(np.float64) - ref).max())
            worst = max(worst, err)
            assert err <= ATOL_OUT, "step %d: max |out - oracle| = %g" % (t, err)
        s_gpu = ctx.scores()
        check_scores(s_gpu, sess.scores())
        if t % wl.delta == 0:
            ctx.retier()
            t_gpu = ctx.tiers()
            want = sess.assign(rank_scores=s_gpu.astype(np.float64))
            assert np.array_equal(t_gpu, want), "step %d: tiers differ at %s" % (
                t, np.argwhere(t_gpu != want)[:10].tolist())
            sess.apply_tiers(want)
            if on_retier is not None:
                on_retier(t, ctx)
    return ctx, sess, worst
