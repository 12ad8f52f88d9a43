"""The allocation-free scheduled attention (fdl_sched_attn_noalloc).

Some callers of this library cannot call cudaMalloc: code running under an
external memory manager that owns the whole device heap, or code on a
latency-critical path where an allocation (which may synchronise the device)
is not acceptable. For them the attention runs with its scratch (the
device-built work list and the per-sequence masked-row counts) in one static
device array of the library instead of a context workspace.

Only the CUDA-core attention (fp32, or head_dim 64) reads that array; the
tensor-core attention finds its own work items. So the calls here are mostly
CUDA-core ones, made back to back through the C ABI with the largest call
first: a later, smaller call would read the earlier call's items and counts
if it did not rewrite every word it reads. Each call is checked against the
float64 oracle (bf16 O 2e-2 / one ulp, fp32 1e-4) and against the context
entry point fdl_sched_attn on the same inputs, and its device error word
must stay zero. This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _simt_case(seed: int, dtype: str, lengths, page_size: int, n_heads: int = 4, head_dim: int = 64):
    """Paged ragged batch: even sequences take 16 window + 8 tracked rows,
    odd ones refresh every position (window rows among them)."""
    rng = np.random.default_rng(seed)
    d = n_heads * head_dim
    lengths = np.asarray(lengths, np.int32)
    geom = synth.paged_geometry(rng, lengths, page_size)
    per_seq = []
    for b, n in enumerate(lengths):
        n = int(n)
        wpos = np.arange(n // 2, n // 2 + 16)
        if b % 2 == 0:
            per_seq.append(synth.draft_rows(wpos, np.sort(rng.choice(n // 2, size=8, replace=False))))
        else:
            per_seq.append(synth.full_rows(n, wpos))
    rows = synth.build_rows(per_seq)
    q = synth.make_tensor(synth.normal(rng, (rows.n_rows, n_heads, head_dim), 1.3), dtype)
    slots = geom.n_pages * geom.page_size
    kc = synth.make_tensor(synth.normal(rng, (slots, d), 1.0), dtype)
    vc = synth.make_tensor(synth.normal(rng, (slots, d), 1.0), dtype)
    shape = synth.LayerShape(d, n_heads, head_dim, 1.0e4, dtype)
    return shape, geom, rows, q, kc, vc, lengths


def _run(shape, geom, rows, q_t, kc_t, vc_t, kv_len, max_seq, with_oracle: bool):
    import torch
    import kv_cache_attention_gb300 as fdl
    s, g = shape, geom
    R, B = rows.n_rows, len(kv_len)
    ctx = fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, B, max_seq, 0, g.page_size,
                         g.n_pages, R, 16, s.dtype)
    q, kc, vc = H.dev(q_t), H.dev(kc_t), H.dev(vc_t)
    bt, cu, kl, kinds = H.ints(g.block_table), H.ints(rows.cu_seqlens), H.ints(kv_len), H.ints(rows.row_kind)
    o_ref = H.empty((R, s.n_heads, s.head_dim), s.dtype)
    lse_ref = torch.empty((R, s.n_heads), dtype=torch.float32, device="cuda")
    tr_ref = torch.zeros((B, max_seq), dtype=torch.float32, device="cuda")
    ctx.sched_attn(q, kc, vc, bt, cu, kl, kinds, o_ref, lse_out=lse_ref, track_scores=tr_ref)
    ctx.sync_status()
    o = torch.full((R, s.n_heads, s.head_dim), 7.0, dtype=o_ref.dtype, device="cuda")
    lse = torch.full((R, s.n_heads), 7.0, dtype=torch.float32, device="cuda")
    tr = torch.zeros((B, max_seq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fdl.fdl_sched_attn_noalloc(ctx.cfg, q, kc, vc, bt, cu, kl, kinds, o, lse_out=lse, track_scores=tr,
                               device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H.assert_close(H.host(o), H.host(o_ref), s.dtype, "no-alloc O vs fdl_sched_attn")
    H.assert_close(H.host(lse), H.host(lse_ref), "f32", "no-alloc LSE vs fdl_sched_attn")
    H.assert_close(H.host(tr), H.host(tr_ref), "f32", "no-alloc tracker vs fdl_sched_attn")
    if with_oracle:
        o_o, lse_o, tr_o = oracle.sched_attn(q_t.values(), kc_t.values(), vc_t.values(), g.block_table,
                                             g.page_size, rows.cu_seqlens, kv_len, rows.row_kind,
                                             max_seq=max_seq, dtype=s.dtype)
        H.assert_close(H.host(o), o_o, s.dtype, "no-alloc O vs oracle")
        H.assert_close(H.host(lse), lse_o, "f32", "no-alloc LSE vs oracle")
        H.assert_close(H.host(tr), tr_o, "f32", "no-alloc tracker vs oracle")
    ctx.close()


def test_noalloc_scratch_path_largest_call_first():
    # call 1: fp32, six sequences over 16-slot pages, three of them full
    # refreshes: the largest work list of the three calls (about 60 items)
    sh, g, rows, q, kc, vc, L = _simt_case(2101, "f32", [150, 203, 97, 181, 66, 240], page_size=16)
    assert rows.n_rows > 400
    _run(sh, g, rows, q, kc, vc, L, int(L.max()), True)
    # call 2: bf16 with head_dim 64 (also the CUDA-core kernel), two sequences
    sh, g, rows, q, kc, vc, L = _simt_case(2102, "bf16", [77, 130], page_size=32)
    _run(sh, g, rows, q, kc, vc, L, int(L.max()), True)
    # call 3: the tiny fp32 layer, one sequence of 24 rows on a flat cache
    wl = synth.tiny_fp32()
    e = wl.extra
    rows = synth.build_rows([synth.draft_rows(e["window_pos"], np.arange(8, dtype=np.int32) * 5)])
    rng = np.random.default_rng(2103)
    q = synth.make_tensor(synth.normal(rng, (rows.n_rows, wl.shape.n_heads, wl.shape.head_dim), 1.3), "f32")
    _run(wl.shape, wl.geom, rows, q, e["k_cache"], e["v_cache"], wl.seq_len, wl.max_seq, True)


def test_noalloc_tensor_core_path_twice():
    # bf16, head_dim 128: the tensor-core attention (it does not use the
    # static array); the ragged call comes first, then the single sequence
    wl2 = synth.ragged_batch(batch=6)
    rng = np.random.default_rng(77)
    s = wl2.shape
    rows = wl2.extra["rows"]
    q = synth.make_tensor(synth.normal(rng, (rows.n_rows, s.n_heads, s.head_dim), 1.3), "bf16")
    _run(s, wl2.geom, rows, q, wl2.extra["k_cache"], wl2.extra["v_cache"], wl2.seq_len, wl2.max_seq, False)
    wl = synth.llada_layer()
    rows = wl.extra["rows"]
    q = synth.make_tensor(synth.normal(rng, (rows.n_rows, s.n_heads, s.head_dim), 1.3), "bf16")
    _run(wl.shape, wl.geom, rows, q, wl.extra["k_cache"], wl.extra["v_cache"], wl.seq_len, wl.max_seq, True)


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
    # the CUDA-core attention takes 16 rows per work item: 65536 rows of one
    # sequence need 4096 + 1 items, one more than the array holds
    cfg = fdl.fdl_config(64, 1, 64, 1e4, 1, 65536, 0, 65536, 1, 65536, 16, fdl.FDL_F32)
    q = torch.zeros((65536, 1, 64), dtype=torch.float32, device="cuda")
    one = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(fdl.FdlError) as ei:
        fdl.fdl_sched_attn_noalloc(cfg, q, q, q, z.view(1, 8), z, one, z, q)
    assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
    # a config that fdl_create rejects is rejected here too (theta <= 1)
    cfg = fdl.fdl_config(64, 1, 64, 1.0, 1, 64, 0, 64, 1, 64, 16, fdl.FDL_F32)
    with pytest.raises(fdl.FdlError) as ei:
        fdl.fdl_sched_attn_noalloc(cfg, q[:8], q, q, z.view(1, 8), z, one, z, q[:8])
    assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
