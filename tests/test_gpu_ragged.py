"""Ragged batch of 16 (bf16, LLaDA layer shape, paged cache of 64-slot pages
randomly permuted in one pool): even sequences in cache phase (32 window +
32 tracked rows), odd sequences in full refresh (every position a query
row). Fused projection, scheduled attention with the tracker, work list and
top-32, each stage against the float64 oracle on identical inputs."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def test_ragged_batch_layer_step():
    import torch
    import kv_cache_attention_gb300 as fdl
    wl = synth.ragged_batch()
    e, s, g = wl.extra, wl.shape, wl.geom
    Hh, hd, dt, B = s.n_heads, s.head_dim, s.dtype, wl.batch
    rows = e["rows"]
    R = rows.n_rows
    ctx = fdl.fdl_create(s.d_model, Hh, hd, s.rope_theta, B, wl.max_seq, 0, g.page_size, g.n_pages, R, 16, dt)
    bt = H.ints(g.block_table)
    kc, vc = H.dev(e["k_cache"]), H.dev(e["v_cache"])
    q = H.empty((R, Hh, hd), dt)
    ctx.qkv_rope_cache_write(H.dev(e["x"]), H.dev(e["w"]), H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                             H.ints(rows.row_cache_pos), bt, kc, vc, q)
    ctx.sync_status()
    q_o, kc_o, vc_o = oracle.qkv_rope_cache_write(
        e["x"].values(), e["w"].values(), Hh, hd, s.rope_theta, rows.row_rope_pos, rows.row_seq,
        rows.row_cache_pos, g.block_table, g.page_size, e["k_cache"].values(), e["v_cache"].values(), dt)
    H.assert_close(H.host(q), q_o, dt, "q_out")
    H.assert_close(H.host(kc), kc_o, dt, "k_cache")
    H.assert_close(H.host(vc), vc_o, dt, "v_cache")
    del kc, vc, q
    q = H.dev(synth.make_tensor(q_o, dt))
    kc, vc = H.dev(synth.make_tensor(kc_o, dt)), H.dev(synth.make_tensor(vc_o, dt))
    o = H.empty((R, Hh, hd), dt)
    lse = torch.empty((R, Hh), dtype=torch.float32, device="cuda")
    tr = torch.zeros((B, wl.max_seq), dtype=torch.float32, device="cuda")
    wlo = torch.full((ctx.worklist_capacity(R, B),), -7, dtype=torch.int32, device="cuda")
    kv_len = wl.seq_len
    ctx.sched_attn(q, kc, vc, bt, H.ints(rows.cu_seqlens), H.ints(kv_len), H.ints(rows.row_kind), o,
                   lse_out=lse, track_scores=tr, worklist_out=wlo)
    ctx.sync_status()
    o_o, lse_o, tr_o = oracle.sched_attn(q_o, kc_o, vc_o, g.block_table, g.page_size, rows.cu_seqlens, kv_len,
                                         rows.row_kind, max_seq=wl.max_seq, dtype=dt)
    H.assert_close(H.host(o), o_o, dt, "attention O")
    H.assert_close(H.host(lse), lse_o, "f32", "LSE")
    H.assert_close(H.host(tr), tr_o, "f32", "tracker scores")
    np.testing.assert_allclose(tr_o.sum(1), 1.0, atol=1e-9)
    w = H.host(wlo)
    want = oracle.work_list(rows.cu_seqlens, kv_len, ctx.tile_m)
    assert np.array_equal(w[1:1 + 4 * int(w[0])].reshape(-1, 4), want)
    k = e["topk"]
    sc32 = tr_o.astype(np.float32)
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.track_topk(H.dev(sc32), H.u8(e["eligible"]), H.ints(kv_len), k, idx, cnt)
    ctx.sync_status()
    idx_o, cnt_o = oracle.track_topk(sc32, e["eligible"], kv_len, k)
    assert H.host(idx).tolist() == idx_o.tolist()
    assert H.host(cnt).tolist() == cnt_o.tolist()
    ctx.close()
