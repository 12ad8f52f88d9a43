"""The allocation-free scheduled attention (fdl_sched_attn_noalloc).

It serves callers that cannot call cudaMalloc (an external allocator owns
the device heap, or an allocation's implicit synchronisation is not
affordable): the same attention kernels run with their scratch in a static
device array instead of a context workspace. Here it is called twice in a
row through the C ABI, on two different workloads, and each result must
match the context-based fdl_sched_attn within the parity tolerances (bf16 O
2e-2 / one ulp, fp32 LSE and tracker scores 1e-4). The second call also
shows that what the first call left in the shared array does not leak into
the next. This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _inputs(wl, R):
    import torch
    rng = np.random.default_rng(77)
    s, g = wl.shape, wl.geom
    q = H.dev(synth.make_tensor(rng.standard_normal((R, s.n_heads, s.head_dim)).astype(np.float32) * 1.3, "bf16"))
    return q


def _run_both(wl, rows, kv_len):
    import torch
    import kv_cache_attention_gb300 as fdl
    s, g, e = wl.shape, wl.geom, wl.extra
    R, B = rows.n_rows, wl.batch
    N = wl.max_seq
    ctx = fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, B, N, wl.max_views, g.page_size,
                         g.n_pages, R, 16, s.dtype)
    q = _inputs(wl, R)
    kc, vc = H.dev(e["k_cache"]), H.dev(e["v_cache"])
    args = (H.ints(g.block_table), H.ints(rows.cu_seqlens), H.ints(kv_len), H.ints(rows.row_kind))
    o_ref = H.empty((R, s.n_heads, s.head_dim), s.dtype)
    lse_ref = torch.empty((R, s.n_heads), dtype=torch.float32, device="cuda")
    tr_ref = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    ctx.sched_attn(q, kc, vc, args[0], args[1], args[2], args[3], o_ref, lse_out=lse_ref, track_scores=tr_ref)
    ctx.sync_status()
    o = torch.full((R, s.n_heads, s.head_dim), 7.0, dtype=o_ref.dtype, device="cuda")
    lse = torch.full((R, s.n_heads), 7.0, dtype=torch.float32, device="cuda")
    tr = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fdl.fdl_sched_attn_noalloc(ctx.cfg, q, kc, vc, args[0], args[1], args[2], args[3], o, lse_out=lse,
                               track_scores=tr, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.host(o), H.host(o_ref), s.dtype, "no-alloc attention O")
    H.assert_close(H.host(lse), H.host(lse_ref), "f32", "no-alloc LSE")
    H.assert_close(H.host(tr), H.host(tr_ref), "f32", "no-alloc tracker scores")
    ctx.close()


def test_noalloc_attention_matches_context_attention_twice():
    # call 1: the LLaDA-shaped single layer (one sequence, 64 rows, flat cache)
    wl = synth.llada_layer()
    _run_both(wl, wl.extra["rows"], wl.seq_len)
    # call 2: a ragged batch over a permuted paged cache, with more work items
    wl2 = synth.ragged_batch(batch=6)
    _run_both(wl2, wl2.extra["rows"], wl2.seq_len)


def test_noalloc_rejects_calls_beyond_the_static_scratch():
    import torch
    import kv_cache_attention_gb300 as fdl
    cfg = fdl.fdl_config(4096, 32, 128, 5e5, 2048, 768, 0, 800, 2048, 1 << 20, 16, fdl.FDL_BF16)
    z = torch.zeros(8, dtype=torch.int32, device="cuda")
    q = torch.zeros((8, 32, 128), dtype=torch.bfloat16, device="cuda")
    kv_len = torch.zeros(1025, dtype=torch.int32, device="cuda")     # B = 1025 > 1024
    with pytest.raises(fdl.FdlError) as ei:
        fdl.fdl_sched_attn_noalloc(cfg, q, q, q, z.view(1, 8), z, kv_len, z, q)
    assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
