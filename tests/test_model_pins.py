"""Pins of the whole-model oracle (oracle/model.py), on the CPU.

RMSNorm and SiLU against hand values and a library routine; a full-refresh
forward through the cache machinery (paged, permuted pages) against a plain
dense transformer computed without any cache; the exactness of a selective
refresh whose tokens did not change; a network whose blocks add nothing; and,
for one layer, the verify forward's extreme views against plain forwards
with the search positions all drafted or all masked.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import model as om
import synth


def test_rmsnorm_hand_values_and_invariances():
    x = np.array([[3.0, 4.0]])
    np.testing.assert_allclose(om.rmsnorm(x, [1.0, 1.0], 0.0), [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]],
                               rtol=1e-15)
    np.testing.assert_allclose(om.rmsnorm(x, [2.0, -1.0], 0.0), [[6 / math.sqrt(12.5), -4 / math.sqrt(12.5)]],
                               rtol=1e-15)
    rng = np.random.default_rng(0)
    y = rng.standard_normal((4, 16))
    g = rng.uniform(0.5, 1.5, 16)
    np.testing.assert_allclose(om.rmsnorm(7.5 * y, g, 0.0), om.rmsnorm(y, g, 0.0), rtol=1e-13)
    c = np.full((1, 8), -0.25)
    np.testing.assert_allclose(om.rmsnorm(c, np.ones(8), 0.0), -np.ones((1, 8)), rtol=1e-15)
    # eps only matters for small rows: a zero row stays zero
    assert (om.rmsnorm(np.zeros((1, 8)), np.ones(8), 1e-5) == 0).all()


def test_silu_against_the_logistic_function():
    from scipy.special import expit
    x = np.concatenate([np.linspace(-40, 40, 801), [-700.0, 700.0, 0.0]])
    np.testing.assert_allclose(om.silu(x), x * expit(x), rtol=1e-13, atol=1e-300)
    assert om.silu(np.array([0.0]))[0] == 0.0
    assert om.silu(np.array([700.0]))[0] == 700.0


def _full_rows(n):
    return synth.build_rows([[(p, p, 0) for p in range(n)]])


def _forward(m, tokens, rows, geom, kcs, vcs, dtype="f32", n=None):
    return om.model_forward(m, tokens, rows.row_seq, rows.row_rope_pos, rows.row_cache_pos, rows.row_kind,
                            rows.cu_seqlens, np.array([n if n is not None else len(tokens)]), geom.block_table,
                            geom.page_size, kcs, vcs, dtype)


@pytest.mark.parametrize("page_size", [16, 64])
def test_full_refresh_equals_a_plain_dense_transformer(page_size):
    m = synth.model_values(synth.model_case(seed=3, d=64, n_heads=2, n_layers=2, ffn=96, vocab=50))
    n = 40
    tokens = np.random.default_rng(1).integers(0, 50, size=n)
    rng = np.random.default_rng(2)
    geom = synth.paged_geometry(rng, [n], page_size)          # permuted pages
    slots = geom.n_pages * geom.page_size
    z = [np.zeros((slots, 64)) for _ in range(2)]
    got, _, _, _ = _forward(m, tokens, _full_rows(n), geom, z, [a.copy() for a in z])
    want = om.dense_forward(m, tokens)
    # model_forward stores its intermediates in fp32; the dense one keeps float64
    np.testing.assert_allclose(got, want, atol=2e-5, rtol=0)


def test_selective_refresh_of_unchanged_tokens_is_exact():
    m = synth.model_values(synth.model_case(seed=4, d=64, n_heads=2, n_layers=3, ffn=128, vocab=60))
    n = 48
    tokens = np.random.default_rng(5).integers(0, 60, size=n)
    geom = synth.flat_geometry(1, n)
    z = [np.zeros((n, 64)) for _ in range(3)]
    full, kcs, vcs, _ = _forward(m, tokens, _full_rows(n), geom, z, [a.copy() for a in z], dtype="bf16")
    # refresh 11 positions only, against the caches the full forward left
    pick = np.sort(np.random.default_rng(6).choice(n, 11, replace=False))
    rows = synth.build_rows([[(int(p), int(p), 0) for p in pick]])
    part, kcs2, vcs2, _ = _forward(m, tokens[pick], rows, geom, kcs, vcs, dtype="bf16", n=n)
    np.testing.assert_allclose(part, full[pick], atol=1e-12, rtol=0)
    for a, b in zip(kcs + vcs, kcs2 + vcs2):
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)
    # a changed token at a refreshed position changes its own row
    t2 = tokens.copy()
    t2[pick[0]] = (t2[pick[0]] + 1) % 60
    part2, _, _, _ = _forward(m, t2[pick], rows, geom, kcs, vcs, dtype="bf16", n=n)
    assert np.abs(part2[0] - full[pick[0]]).max() > 1e-3


def test_blocks_that_add_nothing_leave_the_embedding():
    mc = synth.model_case(seed=7, d=64, n_heads=2, n_layers=2, ffn=64, vocab=30)
    m = synth.model_values(mc)
    for w in m["layers"]:
        w["w_o"] = np.zeros_like(w["w_o"])
        w["w_down"] = np.zeros_like(w["w_down"])
    tokens = np.arange(20) % 30
    geom = synth.flat_geometry(1, 20)
    z = [np.zeros((20, 64)) for _ in range(2)]
    got, _, _, _ = _forward(m, tokens, _full_rows(20), geom, z, [a.copy() for a in z], dtype="f32")
    want = om.rmsnorm(m["embed"][tokens], m["g_final"], m["eps"])
    np.testing.assert_allclose(got, oracle.store_round(want, "f32"), rtol=0, atol=0)


def test_model_case_recipe():
    mc = synth.model_case(seed=8)
    assert mc["mask_id"] == mc["vocab"] - 1
    m = synth.model_values(mc)
    assert m["embed"].shape == (2088, 512) and len(m["layers"]) == 2
    assert m["layers"][0]["w_gu"].shape == (2048, 512) and m["layers"][0]["w_down"].shape == (512, 1024)
    assert abs(m["layers"][0]["w_qkv"].std() - 0.02) < 1e-3
    g = m["layers"][1]["g_mlp"]
    assert g.min() >= 0.79 and g.max() <= 1.21


def test_verify_views_equal_plain_forwards_for_one_layer():
    # With one layer, a key depends only on its own token, so the verify
    # forward's views reduce to plain bidirectional forwards: the last draft
    # view sees every search position's draft (and no mask view), the first
    # mask view sees every search position masked.
    from oracle import refresh as rf
    m = synth.model_values(synth.model_case(seed=9, d=64, n_heads=2, n_layers=1, ffn=64, vocab=40,
                                            out_std=0.5, lm_std=0.2))
    mask_id = 39
    n, prompt = 30, 12
    rng = np.random.default_rng(10)
    tokens = np.full(n, mask_id)
    tokens[:prompt] = rng.integers(0, mask_id, prompt)
    tokens[[14, 20]] = [5, 7]                                # two decoded generated positions
    search = [17, 13, 25]                                    # in acceptance order
    drafts = [3, 11, 29]
    views = 2 * len(search)
    geom = synth.flat_geometry(1, n + views)
    z = [np.zeros((n + views, 64))]
    # the draft forward over every position fills the cache
    full, kc, vc, _ = _forward(m, tokens, _full_rows(n), geom, z, [z[0].copy()], dtype="f32")
    # verify forward: two tracked rows, then the views
    vrows = rf.verify_rows([14, 3], search, n, query_budget=8)
    v_seq = np.zeros(len(vrows), np.int32)
    v_rope = np.array([r[0] for r in vrows], np.int32)
    v_cache = np.array([r[1] for r in vrows], np.int32)
    v_kind = np.array([r[2] for r in vrows], np.int32)
    v_tok = np.array([tokens[p] if k < 2 else (drafts[(k - 2) // 2] if k % 2 == 0 else mask_id)
                      for p, _, k in vrows])
    out, _, _, _ = om.model_forward(m, v_tok, v_seq, v_rope, v_cache, v_kind, np.array([0, len(vrows)], np.int32),
                                    np.array([n]), geom.block_table, geom.page_size, kc, vc, "f32",
                                    search_pos=np.array([search]), n_search=np.array([len(search)]))
    filled = tokens.copy()
    filled[search] = drafts
    last_draft = [i for i, (_, _, k) in enumerate(vrows) if k == 2 + 2 * (len(search) - 1)][0]
    first_mask = [i for i, (_, _, k) in enumerate(vrows) if k == 3][0]
    np.testing.assert_allclose(out[last_draft], om.dense_forward(m, filled)[search[-1]], atol=2e-5, rtol=0)
    np.testing.assert_allclose(out[first_mask], om.dense_forward(m, tokens)[search[0]], atol=2e-5, rtol=0)
    # the tracked rows are the plain forward's too (they see base keys only)
    np.testing.assert_allclose(out[0], om.dense_forward(m, tokens)[14], atol=2e-5, rtol=0)
    # and a middle draft view differs from both extremes (it sees a mix)
    mid = [i for i, (_, _, k) in enumerate(vrows) if k == 4][0]
    assert np.abs(out[mid] - om.dense_forward(m, tokens)[search[1]]).max() > 1e-3
