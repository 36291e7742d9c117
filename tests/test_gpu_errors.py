"""Error paths, with the failures made on the host (no device fault is ever caused).

The library's fault-injection hook (TKV_FAULT_INJECT, read by tkv_create):
  * "hostalloc": the pinned host allocations fail -> tkv_create returns
    TKV_ENOMEM and leaves nothing behind;
  * "call:N": the N-th checked CUDA call of the context reports failure after it
    ran -> that call returns TKV_ECUDA, and every later call on the context
    returns TKV_ESTATE (the context is poisoned), while tkv_get_stats and
    tkv_destroy keep working.
A fresh context without the hook then runs a decode step in lockstep with the
oracle: the device was never touched by the injected failures."""
import ctypes
import numpy as np
import pytest
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from tiered_kv_cache_gqa_gb300 import synth

from harness import lockstep

pytestmark = pytest.mark.gpu

WL = synth.Workload("errors", 2, 8, 2, 64, 2, prompt_len=8, prefill_len=200, decode_steps=8,
                    window=8, delta=4, ratios=(0.4, 0.4, 0.1, 0.1), seed=17)


def _config():
    cfg = tkv.Config()
    cfg.num_layers, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim = 2, 8, 2, 64
    cfg.batch, cfg.max_tokens, cfg.prompt_len, cfg.num_sinks, cfg.recent_window = 2, 256, 8, 4, 8
    cfg.retier_interval = 4
    cfg.ratio_t0, cfg.ratio_t1, cfg.ratio_t2, cfg.ratio_t3 = 0.4, 0.4, 0.1, 0.1
    cfg.compute_stream = tkv.torch_stream_handle()
    return cfg


def test_pinned_host_allocation_failure_returns_enomem(monkeypatch):
    lib = tkv.load()
    monkeypatch.setenv("TKV_FAULT_INJECT", "hostalloc")
    ctx = ctypes.c_void_p()
    assert lib.tkv_create(ctypes.byref(_config()), ctypes.byref(ctx)) == tkv.TKV_ENOMEM
    assert not ctx.value
    monkeypatch.delenv("TKV_FAULT_INJECT")
    assert lib.tkv_create(ctypes.byref(_config()), ctypes.byref(ctx)) == tkv.TKV_OK
    lib.tkv_destroy(ctx)


def _drive(ctx, gen, out, steps):
    """Prefill, decode steps and re-tiers through the raw C calls; returns the statuses seen."""
    seen = []
    L = WL.num_layers
    K, V = gen.prefill()
    for l in range(L):
        seen.append(tkv.tkv_append(ctx, l, K[l].contiguous().cuda(), V[l].contiguous().cuda(), WL.prefill_len))
    for t in range(1, steps + 1):
        q, k, v = (x.cuda() for x in gen.decode_step(t))
        for l in range(L):
            seen.append(tkv.tkv_append(ctx, l, k[l], v[l], 1))
            if l + 1 < L:
                seen.append(tkv.tkv_prefetch(ctx, l + 1))
            seen.append(tkv.tkv_decode_step(ctx, l, q[l], out[l]))
        if t % WL.delta == 0:
            seen.append(tkv.tkv_retier(ctx))
    seen.append(tkv.tkv_sync(ctx))
    return seen


@pytest.mark.parametrize("n", [1, 5, 23, 60])
def test_failed_enqueue_poisons_the_context(monkeypatch, n):
    monkeypatch.setenv("TKV_FAULT_INJECT", "call:%d" % n)
    ctx = tkv.tkv_create(_config())
    monkeypatch.delenv("TKV_FAULT_INJECT")
    out = torch.empty(WL.num_layers, WL.batch, WL.num_q_heads, WL.head_dim, device="cuda")
    seen = _drive(ctx, synth.Generator(WL), out, WL.decode_steps)
    bad = [s for s in seen if s != tkv.TKV_OK]
    assert bad and bad[0] == tkv.TKV_ECUDA, seen
    # everything after the failure is refused, and reports the poisoned state
    assert all(s == tkv.TKV_ESTATE for s in bad[1:]), bad
    assert tkv.tkv_retier(ctx) == tkv.TKV_ESTATE
    assert tkv.tkv_get_scores(ctx, np.zeros((2, 1), np.float32)) == tkv.TKV_ESTATE
    st = tkv.tkv_get_stats(ctx)
    assert st.status == tkv.TKV_ECUDA and st.cuda_error == 999 and st.cuda_error_line > 0
    tkv.tkv_destroy(ctx)
    torch.cuda.synchronize()


def test_device_is_healthy_after_injected_failures():
    ctx, sess, worst = lockstep(WL, WL.decode_steps)
    assert ctx.stats()["status"] == tkv.TKV_OK and ctx.stats()["retiers"] == 2
