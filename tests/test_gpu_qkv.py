"""Fused QKV + RoPE + cache scatter (tensor-core path for bf16 contexts)
against the float64 oracle, over shapes that exercise every tile width
(up to 64 query rows: the weight stream and its merge; 64/128/256-row tiles
of the split-K kernels above), ragged row tails, paged caches,
rows without a cache write, and head_dim 64 and 128."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu

CASES = [
    # (d_model, n_heads, n_rows)
    (1024, 8, 1),
    (1024, 8, 24),
    (1024, 8, 64),
    (1024, 8, 100),
    (1024, 8, 300),
    (1024, 16, 37),   # head_dim 64 through the weight stream (up to 64 rows)
    (1024, 16, 777),
    (4096, 32, 64),
    (4096, 32, 520),
]


@pytest.mark.parametrize("d_model,n_heads,n_rows", CASES)
def test_projection_matches_oracle(d_model, n_heads, n_rows):
    import kv_cache_attention_gb300 as fdl
    wl = synth.projection_case(seed=7000 + n_rows + d_model, d_model=d_model, n_heads=n_heads, n_rows=n_rows)
    e, s, g = wl.extra, wl.shape, wl.geom
    rows = e["rows"]
    ctx = fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, wl.batch, wl.max_seq, 0,
                         g.page_size, g.n_pages, n_rows, 16, s.dtype)
    kc, vc = H.dev(e["k_cache"]), H.dev(e["v_cache"])
    q = H.empty((n_rows, s.n_heads, s.head_dim), s.dtype)
    ctx.qkv_rope_cache_write(H.dev(e["x"]), H.dev(e["w"]), H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                             H.ints(rows.row_cache_pos), H.ints(g.block_table), kc, vc, q)
    ctx.sync_status()
    q_o, kc_o, vc_o = oracle.qkv_rope_cache_write(
        e["x"].values(), e["w"].values(), s.n_heads, s.head_dim, s.rope_theta, rows.row_rope_pos, rows.row_seq,
        rows.row_cache_pos, g.block_table, g.page_size, e["k_cache"].values(), e["v_cache"].values(), s.dtype)
    H.assert_close(H.host(q), q_o, s.dtype, "q_out")
    # every cache row: written rows match the oracle, the rest are untouched (bit-exact)
    H.assert_close(H.host(kc), kc_o, s.dtype, "k_cache")
    H.assert_close(H.host(vc), vc_o, s.dtype, "v_cache")
    written = oracle.slot_map(rows.row_seq, rows.row_cache_pos, g.block_table, g.page_size)
    keep = np.setdiff1d(np.arange(kc_o.shape[0]), written[written >= 0])
    assert np.array_equal(H.host(kc)[keep], e["k_cache"].values()[keep])
    assert np.array_equal(H.host(vc)[keep], e["v_cache"].values()[keep])
    ctx.close()
