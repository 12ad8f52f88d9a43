"""Flash-Verify stress (bf16, batch 32, prompt 512 + gen 1024, window 32,
32 tracked): draft forward, eps unmasking over vocab 126464 (about 30% of
rows above eps), verify forward with 32 T_v + 16 draft-view + 16 mask-view
rows per sequence under the self-view-blocking mask, and prefix acceptance
(draft/mask argmax agreement ~0.7, gamma 0.8). Every stage against the
float64 oracle on identical inputs."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def test_flash_verify_step():
    import torch
    import kv_cache_attention_gb300 as fdl
    wl = synth.flash_verify()
    e, s, g = wl.extra, wl.shape, wl.geom
    Hh, hd, dt, B, N = s.n_heads, s.head_dim, s.dtype, wl.batch, wl.max_seq
    ms, V = e["max_search"], e["vocab"]
    rows = e["rows"]
    R = rows.n_rows
    ctx = fdl.fdl_create(s.d_model, Hh, hd, s.rope_theta, B, N, wl.max_views, g.page_size, g.n_pages, R, V, dt)
    bt = H.ints(g.block_table)
    W = H.dev(e["w"])
    kv_len = wl.seq_len

    # draft forward: projection + attention on identical inputs
    kc, vc = H.dev(e["k_cache"]), H.dev(e["v_cache"])
    q = H.empty((R, Hh, hd), dt)
    ctx.qkv_rope_cache_write(H.dev(e["x"]), W, H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                             H.ints(rows.row_cache_pos), bt, kc, vc, q)
    ctx.sync_status()
    q_o, kc_o, vc_o = oracle.qkv_rope_cache_write(
        e["x"].values(), e["w"].values(), Hh, hd, s.rope_theta, rows.row_rope_pos, rows.row_seq,
        rows.row_cache_pos, g.block_table, g.page_size, e["k_cache"].values(), e["v_cache"].values(), dt)
    H.assert_close(H.host(q), q_o, dt, "draft q_out")
    written = oracle.slot_map(rows.row_seq, rows.row_cache_pos, g.block_table, g.page_size)
    H.assert_close(H.host(kc)[written], kc_o[written], dt, "draft k_cache rows")
    H.assert_close(H.host(vc)[written], vc_o[written], dt, "draft v_cache rows")
    q = H.dev(synth.make_tensor(q_o, dt))
    kc, vc = H.dev(synth.make_tensor(kc_o, dt)), H.dev(synth.make_tensor(vc_o, dt))
    o = H.empty((R, Hh, hd), dt)
    lse = torch.empty((R, Hh), dtype=torch.float32, device="cuda")
    tr = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    ctx.sched_attn(q, kc, vc, bt, H.ints(rows.cu_seqlens), H.ints(kv_len), H.ints(rows.row_kind), o,
                   lse_out=lse, track_scores=tr)
    ctx.sync_status()
    o_o, lse_o, tr_o = oracle.sched_attn(q_o, kc_o, vc_o, g.block_table, g.page_size, rows.cu_seqlens, kv_len,
                                         rows.row_kind, max_seq=N, dtype=dt)
    H.assert_close(H.host(o), o_o, dt, "draft attention O")
    H.assert_close(H.host(lse), lse_o, "f32", "draft LSE")
    H.assert_close(H.host(tr), tr_o, "f32", "tracker scores")

    # eps unmasking of the 32 x 32 window rows
    wseq, wpos = e["window_row_seq"], e["window_row_pos"]
    logits = H.guard_logits(e["logits"], wseq, e["eps"])
    Rw = logits.shape[0]
    conf = torch.empty(Rw, dtype=torch.float32, device="cuda")
    arg = torch.empty(Rw, dtype=torch.int32, device="cuda")
    com = torch.empty(Rw, dtype=torch.uint8, device="cuda")
    srows = torch.empty((B, ms), dtype=torch.int32, device="cuda")
    nsr = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.unmask_verify(B, ms, logits=H.dev(logits), row_seq=H.ints(wseq), row_pos=H.ints(wpos), eps=e["eps"],
                      force_progress=False, conf=conf, argmax=arg, commit=com, search_rows=srows, n_search=nsr)
    ctx.sync_status()
    u = oracle.unmask(logits.values(), wseq, wpos, B, e["eps"], False, ms)
    H.assert_close(H.host(conf), u["conf"], "f32", "confidence")
    assert H.host(arg).tolist() == u["argmax"].tolist()
    assert H.host(com).tolist() == u["commit"].tolist()
    assert H.host(srows).tolist() == u["search_rows"].tolist()
    assert H.host(nsr).tolist() == u["n_search"].tolist()
    frac = float(u["commit"].mean())
    assert 0.2 < frac < 0.4

    # verify forward: T_v (A11: beta_t + beta_m - 2|S| of the tracked set) + views
    per_seq, search_pos = [], np.zeros((B, ms), np.int32)
    for b in range(B):
        m = int(u["n_search"][b])
        sp = wpos[u["search_rows"][b, :m]]
        search_pos[b, :m] = sp
        n_tv = max(0, 32 + 32 - 2 * m)
        per_seq.append(synth.verify_rows(e["tracked"][b][:n_tv], sp, int(kv_len[b])))
    vrows = synth.build_rows(per_seq)
    Rv = vrows.n_rows
    Xv = synth.Tensor(e["x_verify"].data[:Rv], dt)
    qv = H.empty((Rv, Hh, hd), dt)
    kc2, vc2 = H.dev(synth.make_tensor(kc_o, dt)), H.dev(synth.make_tensor(vc_o, dt))
    ctx.qkv_rope_cache_write(H.dev(Xv), W, H.ints(vrows.row_seq), H.ints(vrows.row_rope_pos),
                             H.ints(vrows.row_cache_pos), bt, kc2, vc2, qv)
    ctx.sync_status()
    qv_o, kc2_o, vc2_o = oracle.qkv_rope_cache_write(
        Xv.values(), e["w"].values(), Hh, hd, s.rope_theta, vrows.row_rope_pos, vrows.row_seq,
        vrows.row_cache_pos, g.block_table, g.page_size, kc_o, vc_o, dt)
    H.assert_close(H.host(qv), qv_o, dt, "verify q_out")
    written = oracle.slot_map(vrows.row_seq, vrows.row_cache_pos, g.block_table, g.page_size)
    H.assert_close(H.host(kc2)[written], kc2_o[written], dt, "view k_cache rows")
    qv = H.dev(synth.make_tensor(qv_o, dt))
    kc2, vc2 = H.dev(synth.make_tensor(kc2_o, dt)), H.dev(synth.make_tensor(vc2_o, dt))
    ov = H.empty((Rv, Hh, hd), dt)
    lsev = torch.empty((Rv, Hh), dtype=torch.float32, device="cuda")
    ctx.sched_attn(qv, kc2, vc2, bt, H.ints(vrows.cu_seqlens), H.ints(kv_len), H.ints(vrows.row_kind), ov,
                   lse_out=lsev, search_pos=H.ints(search_pos), n_search=nsr)
    ctx.sync_status()
    ov_o, lsev_o, _ = oracle.sched_attn(qv_o, kc2_o, vc2_o, g.block_table, g.page_size, vrows.cu_seqlens, kv_len,
                                        vrows.row_kind, search_pos=search_pos, n_search=u["n_search"], max_seq=N,
                                        dtype=dt)
    H.assert_close(H.host(ov), ov_o, dt, "verify attention O")
    H.assert_close(H.host(lsev), lsev_o, "f32", "verify LSE")

    # prefix acceptance on the mask views, in search order
    ml = np.zeros((B * ms, V), np.uint16)
    draft = np.full(B * ms, -1, np.int32)
    for b in range(B):
        m = int(u["n_search"][b])
        r = u["search_rows"][b, :m]
        ml[b * ms:b * ms + m] = e["mask_logits_by_window_row"].data[r]
        draft[b * ms:b * ms + m] = u["argmax"][r]
    mlt = H.guard_mask_logits(synth.Tensor(ml, dt), e["gamma"])
    acc = torch.empty(B * ms, dtype=torch.uint8, device="cuda")
    nacc = torch.empty(B, dtype=torch.int32, device="cuda")
    mconf = torch.empty(B * ms, dtype=torch.float32, device="cuda")
    marg = torch.empty(B * ms, dtype=torch.int32, device="cuda")
    ctx.unmask_verify(B, ms, mask_logits=H.dev(mlt), draft_tok=H.ints(draft), gamma=e["gamma"], n_search=nsr,
                      accept=acc, n_accept=nacc, mask_conf=mconf, mask_argmax=marg)
    ctx.sync_status()
    v = oracle.verify(mlt.values(), draft, u["n_search"], e["gamma"], B, ms)
    valid = np.concatenate([np.arange(b * ms, b * ms + int(u["n_search"][b])) for b in range(B)])
    H.assert_close(H.host(mconf)[valid], v["mask_conf"][valid], "f32", "mask confidence")
    assert H.host(marg)[valid].tolist() == v["mask_argmax"][valid].tolist()
    assert H.host(acc).tolist() == v["accept"].tolist()
    assert H.host(nacc).tolist() == v["n_accept"].tolist()
    assert v["n_accept"].sum() > 0
    ctx.close()
