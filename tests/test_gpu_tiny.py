"""Tiny fp32 single layer, batch 1 (d_model 256, 4 x 64 heads, theta 1e4):
the whole Algorithm 2 step on the GPU through the C ABI, each stage
compared with the float64 oracle running its own chain on the same inputs.

Stages: init full forward (all 112 positions) -> tracker top-8 -> draft
step (16 window + 8 tracked rows) -> eps unmasking with forced progress ->
verify forward (T_v + draft views + mask views) -> prefix acceptance.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _ctx(wl, max_rows):
    import kv_cache_attention_gb300 as fdl
    s = wl.shape
    return fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, wl.batch, wl.max_seq,
                          wl.max_views, wl.geom.page_size, wl.geom.n_pages, max_rows,
                          wl.extra["vocab"], s.dtype)


def test_tiny_fp32_algorithm_step():
    import torch
    wl = synth.tiny_fp32()
    e, s, g = wl.extra, wl.shape, wl.geom
    d, Hh, hd, N = s.d_model, s.n_heads, s.head_dim, wl.max_seq
    ctx = _ctx(wl, max_rows=N)
    W = H.dev(e["w"])
    bt = H.ints(g.block_table)
    kc, vc = H.dev(e["k_cache"]), H.dev(e["v_cache"])
    kc_o, vc_o = e["k_cache"].values(), e["v_cache"].values()
    Wv = e["w"].values()
    kv_len = np.array([N], np.int32)

    def forward(rows, X, search_pos=None, n_search=None, track=True):
        nonlocal kc_o, vc_o
        R = rows.n_rows
        q = H.empty((R, Hh, hd), "f32")
        ctx.qkv_rope_cache_write(H.dev(X), W, H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                                 H.ints(rows.row_cache_pos), bt, kc, vc, q)
        q_o, kc_o, vc_o = oracle.qkv_rope_cache_write(
            X.values(), Wv, Hh, hd, s.rope_theta, rows.row_rope_pos, rows.row_seq, rows.row_cache_pos,
            g.block_table, g.page_size, kc_o, vc_o, "f32")
        ctx.sync_status()
        H.assert_close(H.host(q), q_o, "f32", "q_out")
        H.assert_close(H.host(kc), kc_o, "f32", "k_cache")
        H.assert_close(H.host(vc), vc_o, "f32", "v_cache")
        # attention consumes the oracle's stored Q and cache (identical inputs)
        q = H.dev(q_o.astype(np.float32))
        kc.copy_(H.dev(kc_o.astype(np.float32)))
        vc.copy_(H.dev(vc_o.astype(np.float32)))
        o = H.empty((R, Hh, hd), "f32")
        lse = torch.empty((R, Hh), dtype=torch.float32, device="cuda")
        tr = torch.zeros((1, N), dtype=torch.float32, device="cuda") if track else None
        wlo = torch.full((ctx.worklist_capacity(R, 1),), -7, dtype=torch.int32, device="cuda")
        sp = None if search_pos is None else H.ints(np.asarray(search_pos, np.int32).reshape(1, -1))
        ns = None if n_search is None else H.ints([n_search])
        ctx.sched_attn(q, kc, vc, bt, H.ints(rows.cu_seqlens), H.ints(kv_len), H.ints(rows.row_kind), o,
                       lse_out=lse, track_scores=tr, search_pos=sp, n_search=ns, worklist_out=wlo)
        ctx.sync_status()
        o_o, lse_o, tr_o = oracle.sched_attn(
            q_o, kc_o, vc_o, g.block_table, g.page_size, rows.cu_seqlens, kv_len, rows.row_kind,
            search_pos=None if search_pos is None else [list(search_pos)],
            n_search=None if n_search is None else [n_search], max_seq=N, dtype="f32")
        H.assert_close(H.host(o), o_o, "f32", "attention O")
        H.assert_close(H.host(lse), lse_o, "f32", "LSE")
        wl_gpu = H.host(wlo)
        n_items = int(wl_gpu[0])
        nk = kv_len + (2 * n_search if n_search else 0)
        want = oracle.work_list(rows.cu_seqlens, nk, ctx.tile_m)
        assert np.array_equal(wl_gpu[1:1 + 4 * n_items].reshape(-1, 4), want)
        if track:
            H.assert_close(H.host(tr), tr_o, "f32", "tracker scores")
            np.testing.assert_allclose(tr_o.sum(), 1.0, atol=1e-12)
            return tr_o
        return None

    # Algorithm 2 step 1: init full forward over all positions
    rows0 = synth.build_rows([synth.full_rows(N, e["window_pos"])])
    tr_o = forward(rows0, e["x_init"])
    # tracked set = top-8 of the init scores among decoded positions
    k = e["topk"]
    idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1,), dtype=torch.int32, device="cuda")
    sc32 = tr_o.astype(np.float32)
    ctx.track_topk(H.dev(sc32), H.u8(e["eligible"]), H.ints([N]), k, idx, cnt)
    idx_o, cnt_o = oracle.track_topk(sc32, e["eligible"], [N], k)
    assert H.host(idx).tolist() == idx_o.tolist() and H.host(cnt).tolist() == cnt_o.tolist()
    tracked = idx_o[0, :cnt_o[0]]

    # step 2: draft forward over the window + tracked rows
    rows1 = synth.build_rows([synth.draft_rows(e["window_pos"], tracked)])
    forward(rows1, e["x_step"])

    # eps unmasking of the window rows (force progress on)
    logits = H.guard_logits(e["logits"], np.zeros(16, np.int32), e["eps"])
    Rw, ms = logits.shape[0], e["max_search"]
    row_seq, row_pos = np.zeros(Rw, np.int32), e["window_pos"]
    conf = torch.empty(Rw, dtype=torch.float32, device="cuda")
    arg = torch.empty(Rw, dtype=torch.int32, device="cuda")
    com = torch.empty(Rw, dtype=torch.uint8, device="cuda")
    srows = torch.empty((1, ms), dtype=torch.int32, device="cuda")
    nsr = torch.empty((1,), dtype=torch.int32, device="cuda")
    ctx.unmask_verify(1, ms, logits=H.dev(logits), row_seq=H.ints(row_seq), row_pos=H.ints(row_pos),
                      eps=e["eps"], force_progress=True, conf=conf, argmax=arg, commit=com,
                      search_rows=srows, n_search=nsr)
    ctx.sync_status()
    u = oracle.unmask(logits.values(), row_seq, row_pos, 1, e["eps"], True, ms)
    H.assert_close(H.host(conf), u["conf"], "f32", "confidence")
    assert H.host(arg).tolist() == u["argmax"].tolist()
    assert H.host(com).tolist() == u["commit"].tolist()
    assert H.host(srows).tolist() == u["search_rows"].tolist()
    assert H.host(nsr).tolist() == u["n_search"].tolist()
    n_s = int(u["n_search"][0])
    assert n_s > 0

    # step 3: verify forward (T_v shrink: beta_t + beta_m - 2|S| rows of T)
    srow = u["search_rows"][0, :n_s]
    search_pos = row_pos[srow]
    n_tv = max(0, len(tracked) + Rw - 2 * n_s)
    rows2 = synth.build_rows([synth.verify_rows(tracked[:n_tv], search_pos, N)])
    Xv = synth.Tensor(e["x_verify"].data[:rows2.n_rows], "f32")
    forward(rows2, Xv, search_pos=search_pos, n_search=n_s, track=False)

    # prefix acceptance on the mask views
    ml = np.zeros((ms, logits.shape[1]), np.float32)
    ml[:n_s] = e["mask_logits"].data[srow]
    ml = H.guard_mask_logits(synth.Tensor(ml, "f32"), e["gamma"])
    draft = np.full(ms, -1, np.int32)
    draft[:n_s] = u["argmax"][srow]
    acc = torch.empty(ms, dtype=torch.uint8, device="cuda")
    nacc = torch.empty(1, dtype=torch.int32, device="cuda")
    mconf = torch.empty(ms, dtype=torch.float32, device="cuda")
    marg = torch.empty(ms, dtype=torch.int32, device="cuda")
    ctx.unmask_verify(1, ms, mask_logits=H.dev(ml), draft_tok=H.ints(draft), gamma=e["gamma"], n_search=nsr,
                      accept=acc, n_accept=nacc, mask_conf=mconf, mask_argmax=marg)
    ctx.sync_status()
    v = oracle.verify(ml.values(), draft, u["n_search"], e["gamma"], 1, ms)
    H.assert_close(H.host(mconf)[:n_s], v["mask_conf"][:n_s], "f32", "mask confidence")
    assert H.host(marg)[:n_s].tolist() == v["mask_argmax"][:n_s].tolist()
    assert H.host(acc).tolist() == v["accept"].tolist()
    assert H.host(nacc).tolist() == v["n_accept"].tolist()
    ctx.close()
