"""Edge cases through the C ABI: empty and ragged inputs, the limits, and
device-side index errors that must be reported (never trapped)."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _tiny_ctx(dtype="f32", max_rows=64, n_pages=4, page_size=32, max_batch=4, max_seq=96, max_views=8, vocab=64):
    import kv_cache_attention_gb300 as fdl
    return fdl.fdl_create(256, 4, 64, 1e4, max_batch, max_seq, max_views, page_size, n_pages, max_rows, vocab,
                          dtype)


def test_host_validation_rejects_bad_calls():
    import torch
    import kv_cache_attention_gb300 as fdl
    ctx = _tiny_ctx()
    x = torch.zeros((65, 256), device="cuda")
    with pytest.raises(fdl.FdlError) as ei:
        ctx.qkv_rope_cache_write(x, x, x, x, x, torch.zeros((1, 1), dtype=torch.int32, device="cuda"), x, x, x)
    assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
    sc = torch.zeros((1, 96), device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in (0, 1025):
        with pytest.raises(fdl.FdlError):
            ctx.track_topk(sc, torch.ones((1, 96), dtype=torch.uint8, device="cuda"), z, k, z, z)
    ctx.close()


def test_empty_calls_are_no_ops():
    import torch
    ctx = _tiny_ctx()
    e = torch.zeros((0, 256), device="cuda")
    ei = torch.zeros(0, dtype=torch.int32, device="cuda")
    bt = torch.zeros((1, 3), dtype=torch.int32, device="cuda")
    kc = torch.full((128, 256), 3.0, device="cuda")
    ctx.qkv_rope_cache_write(e, e, ei, ei, ei, bt, kc, kc, e)
    o = torch.full((0, 4, 64), 1.0, device="cuda")
    ctx.sched_attn(e.view(0, 4, 64), kc, kc, bt, H.ints([0]), ei, ei, o)
    ctx.sync_status()
    assert (H.host(kc) == 3.0).all()
    ctx.close()


def test_out_of_pool_page_is_reported_and_skipped():
    import kv_cache_attention_gb300 as fdl
    import torch
    ctx = _tiny_ctx()
    rng = np.random.default_rng(0)
    x = torch.as_tensor(rng.standard_normal((3, 256), dtype=np.float32)).cuda()
    w = torch.as_tensor(rng.standard_normal((768, 256), dtype=np.float32) * 0.02).cuda()
    bt = H.ints([[0, 9, 1]])          # page 9 is outside the 4-page pool
    kc = torch.zeros((128, 256), device="cuda")
    vc = torch.zeros((128, 256), device="cuda")
    q = torch.zeros((3, 4, 64), device="cuda")
    ctx.qkv_rope_cache_write(x, w, H.ints([0, 0, 0]), H.ints([1, 40, 70]), H.ints([1, 40, 70]), bt, kc, vc, q)
    with pytest.raises(fdl.FdlError) as ei:
        ctx.sync_status()
    assert ei.value.status == fdl.FDL_ERR_DEVICE_INDEX
    k = H.host(kc)
    assert np.abs(k[1]).sum() > 0 and np.abs(k[32 + 6]).sum() > 0   # rows 0 and 2 written
    assert np.count_nonzero(np.abs(k).sum(1)) == 2                    # row 1 skipped
    ctx.sync_status()  # the word was cleared
    ctx.close()


def test_inconsistent_cu_seqlens_is_reported():
    import kv_cache_attention_gb300 as fdl
    import torch
    ctx = _tiny_ctx()
    q = torch.zeros((8, 4, 64), device="cuda")
    kc = torch.zeros((128, 256), device="cuda")
    o = torch.full((8, 4, 64), 5.0, device="cuda")
    ctx.sched_attn(q, kc, kc, H.ints([[0, 1, 2]]), H.ints([0, 9]), H.ints([10]), H.ints(np.zeros(8)), o)
    with pytest.raises(fdl.FdlError) as ei:
        ctx.sync_status()
    assert ei.value.status == fdl.FDL_ERR_DEVICE_INDEX
    assert (H.host(o) == 5.0).all()   # nothing scheduled
    ctx.close()


def test_attention_empty_sequences_and_zero_keys():
    import torch
    ctx = _tiny_ctx()
    rng = np.random.default_rng(1)
    B = 3
    cu = np.array([0, 5, 5, 9], np.int32)         # sequence 1 has no rows
    kv_len = np.array([7, 30, 0], np.int32)       # sequence 2 has no keys
    geom = synth.paged_geometry(rng, [96, 96, 96], 32)
    nslot = geom.n_pages * 32
    K = rng.standard_normal((nslot, 256)).astype(np.float32)
    V = rng.standard_normal((nslot, 256)).astype(np.float32)
    q = rng.standard_normal((9, 4, 64)).astype(np.float32)
    kinds = np.array([1, 1, 0, 1, 0, 1, 0, 0, 1], np.int32)
    ctx2 = _tiny_ctx(n_pages=geom.n_pages)
    o = torch.zeros((9, 4, 64), device="cuda")
    lse = torch.zeros((9, 4), device="cuda")
    tr = torch.zeros((B, 96), device="cuda")
    ctx2.sched_attn(H.dev(q), H.dev(K), H.dev(V), H.ints(geom.block_table), H.ints(cu), H.ints(kv_len),
                    H.ints(kinds), o, lse_out=lse, track_scores=tr)
    ctx2.sync_status()
    o_o, lse_o, tr_o = oracle.sched_attn(q.astype(np.float64), K.astype(np.float64), V.astype(np.float64),
                                         geom.block_table, 32, cu, kv_len, kinds, max_seq=96, dtype="f32")
    H.assert_close(H.host(o), o_o, "f32", "O")
    assert np.array_equal(np.isinf(H.host(lse)), np.isinf(lse_o))
    fin = np.isfinite(lse_o)
    H.assert_close(H.host(lse)[fin], lse_o[fin], "f32", "LSE")
    H.assert_close(H.host(tr), tr_o, "f32", "tracker")
    ctx.close()
    ctx2.close()


def test_topk_ties_signed_zero_and_short_sequences():
    import torch
    ctx = _tiny_ctx(max_batch=4)
    sc = np.zeros((4, 96), np.float32)
    sc[0, :] = 0.5                                   # all equal: lowest positions win
    sc[1, ::2] = -0.0                                # -0.0 equals +0.0
    sc[1, 5] = 1.0
    sc[2] = np.random.default_rng(2).integers(0, 3, 96).astype(np.float32)
    el = np.ones((4, 96), np.uint8)
    el[3, :] = 0
    el[3, [4, 9]] = 1                                # fewer eligible than k
    seq_len = np.array([96, 96, 50, 96], np.int32)
    for k in (1, 7, 64):
        idx = torch.empty((4, k), dtype=torch.int32, device="cuda")
        cnt = torch.empty((4,), dtype=torch.int32, device="cuda")
        ctx.track_topk(H.dev(sc), H.u8(el), H.ints(seq_len), k, idx, cnt)
        ctx.sync_status()
        want, wc = oracle.track_topk(sc, el, seq_len, k)
        assert H.host(idx).tolist() == want.tolist(), k
        assert H.host(cnt).tolist() == wc.tolist()
    ctx.close()


def test_topk_every_selection_path():
    """Rows that take each way through the selection: spread scores (the
    threshold bin is found within one digit), dense ties at the full key with
    at most 1024 candidates, more than 1024 keys tied at the threshold (cut
    by position), all keys equal, and rows longer than the shared-memory
    stage (read from global memory)."""
    import torch
    rng = np.random.default_rng(11)
    for ld in (4000, 9000):
        ctx = _tiny_ctx(max_batch=5)
        sc = np.zeros((5, ld), np.float32)
        sc[0] = (32 * np.exp(1.5 * rng.standard_normal(ld)) / ld).astype(np.float32)
        sc[1] = rng.integers(0, 40, ld).astype(np.float32) / 8            # ~100 copies of each value
        sc[2] = np.where(rng.random(ld) < 0.6, 1.0, rng.random(ld)).astype(np.float32)  # >1024 tied at the top
        sc[3] = 0.25
        sc[4] = rng.standard_normal(ld).astype(np.float32)
        el = (rng.random((5, ld)) < 0.8).astype(np.uint8)
        seq_len = np.array([ld, ld - 7, ld, ld - 100, ld // 3], np.int32)
        for k in (32, 1024):
            idx = torch.empty((5, k), dtype=torch.int32, device="cuda")
            cnt = torch.empty((5,), dtype=torch.int32, device="cuda")
            ctx.track_topk(H.dev(sc), H.u8(el), H.ints(seq_len), k, idx, cnt)
            ctx.sync_status()
            want, wc = oracle.track_topk(sc, el, seq_len, k)
            assert H.host(idx).tolist() == want.tolist(), (ld, k)
            assert H.host(cnt).tolist() == wc.tolist()
        ctx.close()


def test_unmask_ties_and_forced_progress_per_sequence():
    import torch
    ctx = _tiny_ctx(max_batch=4, vocab=64)
    rng = np.random.default_rng(3)
    L = rng.standard_normal((10, 64)).astype(np.float32)
    L[3] = L[2]                                      # identical rows: order by position
    L[7, 5] = 40.0                                   # one certain row in sequence 2
    seq = np.array([0, 0, 0, 0, 2, 2, 2, 2, 3, 3], np.int32)   # sequence 1 has no rows
    pos = np.array([9, 4, 6, 5, 1, 2, 3, 0, 8, 7], np.int32)
    for force in (False, True):
        conf = torch.empty(10, device="cuda")
        arg = torch.empty(10, dtype=torch.int32, device="cuda")
        com = torch.empty(10, dtype=torch.uint8, device="cuda")
        sr = torch.empty((4, 3), dtype=torch.int32, device="cuda")
        ns = torch.empty(4, dtype=torch.int32, device="cuda")
        ctx.unmask_verify(4, 3, logits=H.dev(L), row_seq=H.ints(seq), row_pos=H.ints(pos), eps=0.9,
                          force_progress=force, conf=conf, argmax=arg, commit=com, search_rows=sr, n_search=ns)
        ctx.sync_status()
        u = oracle.unmask(L.astype(np.float64), seq, pos, 4, 0.9, force, 3)
        assert H.host(com).tolist() == u["commit"].tolist()
        assert H.host(sr).tolist() == u["search_rows"].tolist()
        assert H.host(ns).tolist() == u["n_search"].tolist()
    ctx.close()


def _projection(ctx, wl):
    e, s, g = wl.extra, wl.shape, wl.geom
    rows = e["rows"]
    kc, vc = H.dev(e["k_cache"]), H.dev(e["v_cache"])
    q = H.empty((rows.n_rows, s.n_heads, s.head_dim), s.dtype)
    ctx.qkv_rope_cache_write(H.dev(e["x"]), H.dev(e["w"]), H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                             H.ints(rows.row_cache_pos), H.ints(g.block_table), kc, vc, q)
    return q, kc, vc


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """A main-loop wait budget of 300 cycles is far shorter than a DRAM load,
    so the tensor-core projection's first wait gives up: the kernel drains
    its loads, writes nothing and reports FDL_ERR_TIMEOUT through the error
    word. With the default budget restored, the next call on the same
    context (same split-K counters) matches the oracle."""
    import kv_cache_attention_gb300 as fdl
    wl = synth.projection_case(seed=7301, d_model=512, n_heads=4, n_rows=64)
    e, s, g = wl.extra, wl.shape, wl.geom
    rows = e["rows"]
    ctx = fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, wl.batch, wl.max_seq, 0,
                         g.page_size, g.n_pages, rows.n_rows, 16, s.dtype)
    with pytest.raises(fdl.FdlError) as ei:
        ctx.set_wait_budget(-1)
    assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
    ctx.set_wait_budget(300)
    _projection(ctx, wl)
    with pytest.raises(fdl.FdlError) as ei:
        ctx.sync_status()
    assert ei.value.status == fdl.FDL_ERR_TIMEOUT
    ctx.set_wait_budget(0)
    for _ in range(2):
        q, kc, vc = _projection(ctx, wl)
        ctx.sync_status()
        q_o, kc_o, vc_o = oracle.qkv_rope_cache_write(
            e["x"].values(), e["w"].values(), s.n_heads, s.head_dim, s.rope_theta, rows.row_rope_pos,
            rows.row_seq, rows.row_cache_pos, g.block_table, g.page_size, e["k_cache"].values(),
            e["v_cache"].values(), s.dtype)
        H.assert_close(H.host(q), q_o, s.dtype, "q_out after a timed-out call")
        H.assert_close(H.host(kc), kc_o, s.dtype, "k_cache after a timed-out call")
        H.assert_close(H.host(vc), vc_o, s.dtype, "v_cache after a timed-out call")
    ctx.close()
