"""The layer-step kernels driven by the host row builder through whole
decodes under each KV-cache refresh policy (full recompute, Fast-dLLM
PrefixCache and DualCache, FreeCache, the Flash-dLLM draft forward), against
the float64 oracle step by step.

The oracle keeps its own cache, updated only at the rows each policy
chooses, so stale cached K/V are exercised exactly as the policy leaves them.
Each stage gets identical inputs on both sides: before a step the GPU cache
is set to the oracle's (stored bf16 values, exact), the projection is
compared, then the attention runs on the oracle's Q and cache."""
import numpy as np
import pytest

import oracle
from oracle import refresh as rf
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy", [rf.FULL, rf.PREFIX, rf.DUAL, rf.FREECACHE, rf.FLASH_DRAFT])
def test_decode_trace_under_refresh_policy(policy):
    import torch
    import kv_cache_attention_gb300 as fdl
    wl = synth.refresh_trace()
    s, g, e = wl.shape, wl.geom, wl.extra
    Hh, hd, d, dt, B, N = s.n_heads, s.head_dim, s.d_model, s.dtype, wl.batch, wl.max_seq
    prompts, lengths, block = e["prompts"], wl.seq_len, e["block"]
    max_rows = int(lengths.sum())
    ctx = fdl.fdl_create(d, Hh, hd, s.rope_theta, B, N, 0, g.page_size, g.n_pages, max_rows, 16, dt)
    assert ctx.tile_m == 128                         # the tensor-core attention
    w_dev, bt, kv_len = H.dev(e["w"]), H.ints(g.block_table), H.ints(lengths)
    w = e["w"].values()
    n_slots = g.n_pages * g.page_size
    kc_o, vc_o = np.zeros((n_slots, d)), np.zeros((n_slots, d))
    masked = np.zeros((B, N), np.uint8)
    for b in range(B):
        masked[b, prompts[b]:lengths[b]] = 1
    state = np.full(B, -1, np.int32)
    st_o = state.copy()
    rng = np.random.default_rng([e["seed"], 3, policy])
    total_rows = 0
    for step in range(200):
        tracked = n_tracked = tr_list = None
        if policy == rf.FLASH_DRAFT:
            tracked = np.full((B, 8), -1, np.int32)
            n_tracked = np.zeros(B, np.int32)
            tr_list = []
            for b in range(B):
                pick = rng.permutation(np.nonzero(masked[b, :lengths[b]] == 0)[0])[:8]
                tracked[b, :len(pick)], n_tracked[b] = pick, len(pick)
                tr_list.append(pick.tolist())
        rows = fdl.fdl_refresh_rows(policy, prompts, lengths, masked, block, state, tracked, n_tracked)
        for b in range(B):
            want, st_o[b] = rf.refresh_rows(policy, masked[b], int(prompts[b]), int(lengths[b]), block,
                                            int(st_o[b]), () if tr_list is None else tr_list[b])
            lo, hi = rows.cu_seqlens[b], rows.cu_seqlens[b + 1]
            assert list(zip(rows.row_rope_pos[lo:hi].tolist(), rows.row_kind[lo:hi].tolist())) == want
        R = rows.n_rows
        if R == 0:
            break
        total_rows += R
        x = synth.trace_hidden(e["seed"], step, R, d)
        kc = H.dev(synth.make_tensor(kc_o, dt))
        vc = H.dev(synth.make_tensor(vc_o, dt))
        q = H.empty((R, Hh, hd), dt)
        rs, rp, rk, cu = H.ints(rows.row_seq), H.ints(rows.row_rope_pos), H.ints(rows.row_kind), H.ints(rows.cu_seqlens)
        ctx.qkv_rope_cache_write(H.dev(x), w_dev, rs, rp, H.ints(rows.row_cache_pos), bt, kc, vc, q)
        ctx.sync_status()
        q_o, kc_o, vc_o = oracle.qkv_rope_cache_write(
            x.values(), w, Hh, hd, s.rope_theta, rows.row_rope_pos, rows.row_seq, rows.row_cache_pos,
            g.block_table, g.page_size, kc_o, vc_o, dt)
        H.assert_close(H.host(q), q_o, dt, f"q, step {step}")
        H.assert_close(H.host(kc), kc_o, dt, f"k cache, step {step}")
        H.assert_close(H.host(vc), vc_o, dt, f"v cache, step {step}")
        q = H.dev(synth.make_tensor(q_o, dt))
        kc = H.dev(synth.make_tensor(kc_o, dt))
        vc = H.dev(synth.make_tensor(vc_o, dt))
        o = H.empty((R, Hh, hd), dt)
        lse = torch.empty((R, Hh), dtype=torch.float32, device="cuda")
        tr = torch.zeros((B, N), dtype=torch.float32, device="cuda")
        ctx.sched_attn(q, kc, vc, bt, cu, kv_len, rk, o, lse_out=lse, track_scores=tr)
        ctx.sync_status()
        o_o, lse_o, tr_o = oracle.sched_attn(q_o, kc_o, vc_o, g.block_table, g.page_size, rows.cu_seqlens,
                                             lengths, rows.row_kind, max_seq=N, dtype=dt)
        H.assert_close(H.host(o), o_o, dt, f"O, step {step}")
        H.assert_close(H.host(lse), lse_o, "f32", f"LSE, step {step}")
        H.assert_close(H.host(tr), tr_o, "f32", f"tracker, step {step}")
        for b in range(B):
            lo, hi = rows.cu_seqlens[b], rows.cu_seqlens[b + 1]
            dec = rows.row_rope_pos[lo:hi][rows.row_kind[lo:hi] == 1]
            masked[b, synth.trace_unmask(rng, dec)] = 0
    else:
        pytest.fail("decode did not finish")
    assert not masked.any() and total_rows > 0
    ctx.close()
