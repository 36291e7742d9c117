"""The allocation-free entry point against the context path.

tkv_decode_dense_noalloc serves callers that cannot let a library allocate
device memory (a runtime whose caching allocator owns the memory budget, or a
decode loop that cannot take the device-wide stall of cudaMalloc).  It runs on
fixed scratch arrays, so this test checks it against tkv_decode_step on two
decode steps in a row, bitwise (both run the same kernels in the same launch
plan): the second call must not see anything left behind by the first.  The file is named to be collected last."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gqa_gb300 as tkv
from tiered_kv_cache_gqa_gb300 import synth

from harness import gpu_step

pytestmark = pytest.mark.gpu


def dense_kv(K, V):
    """[L][B][n][Hkv][d] K and V -> [L][2][B][Hkv][n][d]."""
    return torch.stack([K.permute(0, 1, 3, 2, 4), V.permute(0, 1, 3, 2, 4)], dim=1).contiguous()


def test_noalloc_matches_context_path_on_two_calls():
    wl = synth.Workload("noalloc", 2, 16, 4, 128, 2, prompt_len=16, prefill_len=700, decode_steps=2,
                        window=16, ratios=(1.0, 0.0, 0.0, 0.0), seed=21)
    gen = synth.Generator(wl)
    K, V = gen.prefill()
    L, B, Hq, Hkv, d = wl.num_layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim

    ctx = tkv.TieredKV.for_workload(wl)
    for l in range(L):
        ctx.append(l, K[l].contiguous().cuda(), V[l].contiguous().cuda(), wl.prefill_len)

    s_dense = torch.zeros(B, wl.prefill_len, device="cuda")
    Kall, Vall = K, V
    for t in (1, 2):
        q, k, v = gen.decode_step(t)
        out_ctx = torch.empty(L, B, Hq, d, device="cuda")
        gpu_step(ctx, q.cuda(), k.cuda(), v.cuda(), out_ctx)

        Kall = torch.cat([Kall, k[:, :, None]], dim=2)
        Vall = torch.cat([Vall, v[:, :, None]], dim=2)
        R = Kall.shape[2]
        kv = dense_kv(Kall, Vall).cuda()
        s_dense = torch.cat([s_dense, torch.zeros(B, 1, device="cuda")], dim=1).contiguous()
        out_na = torch.full((L, B, Hq, d), float("nan"), device="cuda")
        rc = tkv.tkv_decode_dense_noalloc(q.cuda().contiguous(), kv, out_na, s_dense, L, B, Hq, Hkv, d, R)
        assert rc == tkv.TKV_OK, tkv.status_string(rc)
        torch.cuda.synchronize()
        # the same kernels in the same launch plan, over the same rows in the same order:
        # outputs and scores are bitwise equal
        assert torch.equal(out_na, out_ctx), "call %d: max |noalloc - context| = %g" % (
            t, (out_na - out_ctx).abs().max().item())
        assert np.array_equal(s_dense.cpu().numpy(), ctx.scores()), "call %d: s differs" % t


def test_noalloc_rejects_sizes_beyond_its_scratch():
    q = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, device="cuda")
    # 16 sequences * 16 KV heads * 1024 positions > 131,072 retained (sequence, KV head, row) triples
    rc = tkv.tkv_decode_dense_noalloc(q, q, out, out, 1, 16, 128, 16, 128, 1024)
    assert rc == tkv.TKV_ECAPACITY
    rc = tkv.tkv_decode_dense_noalloc(q, q, out, out, 1, 1, 64, 8, 96, 16)
    assert rc == tkv.TKV_EINVAL
