"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU. Each test ties one oracle function to something other than itself:
a hand-worked golden fixture (tests/golden/, each with its citation), a
closed form, an invariant, or brute force on tiny inputs. The cases are
chosen so that a dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- storage
def test_bf16_store_round_ties_to_even():
    one = 1.0
    assert oracle.store_round(np.array([one + 2 ** -8]), "bf16")[0] == 1.0
    assert oracle.store_round(np.array([one + 3 * 2 ** -8]), "bf16")[0] == 1.0 + 2 ** -6
    assert oracle.store_round(np.array([-(one + 3 * 2 ** -8)]), "bf16")[0] == -(1.0 + 2 ** -6)
    assert oracle.store_round(np.array([0.0]), "bf16")[0] == 0.0


def test_bf16_store_round_matches_library_on_float32_inputs():
    # special case that reduces to a library routine: float32 inputs have no
    # double-rounding hazard, so torch's float32 -> bfloat16 cast must agree
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-8, 8, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.store_round(x.astype(np.float64), "bf16"), ref)


# --------------------------------------------------------------------------- slots / work list
def test_slot_golden():
    g = golden("slot_hand.json")
    bt = np.array(g["block_table"], np.int32)
    for (b, c), s in zip(g["queries"], g["slots"]):
        assert oracle.slot_of(bt, g["page_size"], b, c) == s


def test_flat_identity_table_is_flat_layout():
    # closed form: one page of N_max slots per sequence -> slot = b * N_max + c
    B, n_max = 5, 37
    geom = synth.flat_geometry(B, n_max)
    for b in range(B):
        for c in range(n_max):
            assert oracle.slot_of(geom.block_table, geom.page_size, b, c) == b * n_max + c


def test_paged_slots_are_a_bijection():
    rng = np.random.default_rng(3)
    lengths = [130, 64, 1, 200, 77]
    geom = synth.paged_geometry(rng, lengths, 16)
    seen = {}
    for b, n in enumerate(lengths):
        for c in range(n):
            s = oracle.slot_of(geom.block_table, geom.page_size, b, c)
            assert 0 <= s < geom.n_pages * geom.page_size
            assert s not in seen
            seen[s] = (b, c)
    assert len(seen) == sum(lengths)


def test_slot_map_skips_unwritten_rows():
    bt = np.array([[2, 0, 1]], np.int32)
    s = oracle.slot_map([0, 0, 0], [-1, 5, 9], bt, 4)
    assert list(s) == [-1, 1, 5]


def test_work_list_covers_every_row_once():
    rng = np.random.default_rng(5)
    for tile in (1, 16, 64, 128):
        lens = rng.integers(0, 300, size=9)
        lens[3] = 0
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        nk = rng.integers(1, 2000, size=9)
        wl = oracle.work_list(cu, nk, tile)
        owner = np.full(cu[-1], -1)
        prev = (-1, -1)
        for (b, q0, ql, k) in wl:
            assert 1 <= ql <= tile
            assert k == nk[b]
            assert cu[b] <= q0 and q0 + ql <= cu[b + 1]
            assert (b, q0) > prev          # sequences in order, tiles in order
            prev = (b, q0)
            assert np.all(owner[q0:q0 + ql] == -1)
            owner[q0:q0 + ql] = b
        for b in range(9):
            assert np.all(owner[cu[b]:cu[b + 1]] == b)
        # brute-force count: ceil(len / tile) items per sequence
        assert len(wl) == sum(int(math.ceil(l / tile)) for l in lens)


# --------------------------------------------------------------------------- QKV + RoPE
def test_qkv_rope_golden():
    g = golden("qkv_rope_hand.json")
    w = np.array(g["w"], float)
    x = np.array(g["x"], float)
    pos = np.array(g["pos"])
    y = oracle.project_qkv(x, w)
    d, H, hd = g["d_model"], g["n_heads"], g["head_dim"]
    q = oracle.rope(y[:, :d].reshape(-1, H, hd), pos, g["theta"]).reshape(-1, d)
    k = oracle.rope(y[:, d:2 * d].reshape(-1, H, hd), pos, g["theta"]).reshape(-1, d)
    np.testing.assert_allclose(q, g["q"], atol=1e-14)
    np.testing.assert_allclose(k, g["k"], atol=1e-14)
    np.testing.assert_allclose(y[:, 2 * d:], g["v"], atol=1e-14)


def test_qkv_rope_cache_write_golden_slots():
    g = golden("qkv_rope_hand.json")
    w = np.array(g["w"], float)
    x = np.array(g["x"], float)
    bt = np.array([[1, 0]], np.int32)       # page size 2: positions 0,1 -> page 1
    kc = np.full((4, 4), 7.0)
    vc = np.full((4, 4), 7.0)
    q, kc2, vc2 = oracle.qkv_rope_cache_write(
        x, w, 1, 4, g["theta"], g["pos"], [0, 0, 0], [1, -1, 2], bt, 2, kc, vc, "f32")
    # row 0 -> position 1 -> page bt[0][0]=1 -> slot 3; row 2 -> position 2 -> page 0 -> slot 0
    np.testing.assert_allclose(kc2[3], g["k"][0], atol=1e-6)
    np.testing.assert_allclose(vc2[3], g["v"][0], atol=1e-6)
    np.testing.assert_allclose(kc2[0], g["k"][2], atol=1e-6)
    np.testing.assert_allclose(vc2[0], g["v"][2], atol=1e-6)
    assert np.all(kc2[1:3] == 7.0) and np.all(vc2[1:3] == 7.0)
    np.testing.assert_allclose(q.reshape(3, 4), g["q"], atol=1e-6)


def test_rope_invariants():
    rng = np.random.default_rng(7)
    R, H, hd, theta = 20, 3, 64, 5e5
    x = rng.standard_normal((R, H, hd))
    pos = rng.integers(0, 4000, R)
    y = oracle.rope(x, pos, theta)
    half = hd // 2
    n0 = x[..., :half] ** 2 + x[..., half:] ** 2
    n1 = y[..., :half] ** 2 + y[..., half:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(R, int), theta), x)
    # relative position: <R(q,m), R(k,n)> depends on m - n only
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))
    dots = []
    for shift in (0, 17, 1234):
        a = oracle.rope(q, np.array([50 + shift]), theta)
        b = oracle.rope(k, np.array([9 + shift]), theta)
        dots.append(float((a * b).sum()))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# --------------------------------------------------------------------------- attention
def _one_seq_attn(q, K, V, kinds=None, dtype="f32"):
    n, hd = K.shape
    bt = np.zeros((1, 1), np.int32)
    qq = np.asarray(q, float).reshape(-1, 1, hd)
    R = qq.shape[0]
    kinds = [0] * R if kinds is None else kinds
    return oracle.sched_attn(qq, K, V, bt, n, np.array([0, R]), np.array([n]),
                             np.array(kinds), max_seq=n, dtype=dtype)


def test_attention_golden():
    g = golden("attention_hand.json")
    o, lse, _ = _one_seq_attn(np.array([g["q"]]), np.array(g["k"]), np.array(g["v"]))
    np.testing.assert_allclose(o[0, 0], g["o"], atol=1e-6)
    np.testing.assert_allclose(lse[0, 0], g["lse"], atol=1e-12)


def test_attention_equal_keys_give_mean_value():
    rng = np.random.default_rng(11)
    K = np.tile(rng.standard_normal(8), (5, 1))
    V = rng.standard_normal((5, 8))
    q = rng.standard_normal((3, 8))
    o, lse, _ = _one_seq_attn(q, K, V)
    np.testing.assert_allclose(o[:, 0], np.tile(V.mean(0), (3, 1)), atol=1e-6)
    s = q @ K[0] / math.sqrt(8)
    np.testing.assert_allclose(lse[:, 0], s + math.log(5), atol=1e-12)


def test_attention_probabilities_sum_to_one_and_track_mass():
    # every masked row's softmax row sums to 1, so one layer adds exactly 1
    # to sum_i a_b[i] (Eq. 2 averages over heads and masked rows)
    rng = np.random.default_rng(13)
    B, H, hd = 3, 4, 16
    lens = [9, 40, 23]
    geom = synth.paged_geometry(rng, lens, 8)
    nslots = geom.n_pages * geom.page_size
    K = rng.standard_normal((nslots, H * hd)) * 2
    V = rng.standard_normal((nslots, H * hd))
    per_seq = [synth.draft_rows(np.arange(3), np.arange(3, 5)), synth.draft_rows([], [1, 2]),
               synth.full_rows(23, [4, 5, 6])]
    rows = synth.build_rows(per_seq)
    q = rng.standard_normal((rows.n_rows, H, hd))
    total = np.zeros((B, 40))
    for layer in range(3):
        _, lse, tr = oracle.sched_attn(q, K, V, geom.block_table, geom.page_size, rows.cu_seqlens,
                                       np.array(lens), rows.row_kind, max_seq=40)
        total += tr
    np.testing.assert_allclose(total.sum(1), [3.0, 0.0, 3.0], atol=1e-12)
    assert np.all(total >= 0)
    assert np.all(total[0, 9:] == 0) and np.all(total[2, 23:] == 0)


def test_attention_is_layout_independent():
    # the same logical cache through a flat table and a permuted paged table
    rng = np.random.default_rng(17)
    H, hd, n = 2, 8, 50
    Kl = rng.standard_normal((n, H * hd))
    Vl = rng.standard_normal((n, H * hd))
    geom = synth.paged_geometry(rng, [n], 4)
    Kp = np.zeros((geom.n_pages * 4, H * hd))
    Vp = np.zeros_like(Kp)
    for c in range(n):
        s = oracle.slot_of(geom.block_table, 4, 0, c)
        Kp[s], Vp[s] = Kl[c], Vl[c]
    q = rng.standard_normal((6, H, hd))
    kinds = np.array([1, 1, 0, 0, 1, 0])
    cu = np.array([0, 6])
    a = oracle.sched_attn(q, Kl, Vl, np.zeros((1, 1), np.int32), n, cu, [n], kinds, max_seq=n)
    b = oracle.sched_attn(q, Kp, Vp, geom.block_table, 4, cu, [n], kinds, max_seq=n)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_view_rule_every_view_sees_each_position_once():
    kv_len, search = 12, [7, 2, 9, 4]
    m = len(search)
    for j in range(m):
        for kind in (synth.kind_draft_view(j), synth.kind_mask_view(j)):
            vis = oracle.visible_positions(kind, kv_len, search)
            positions = sorted(p for _, p in vis)
            assert positions == list(range(kv_len))
    # extreme cases: the last draft view sees every draft, the first mask view every mask
    last = oracle.visible_positions(synth.kind_draft_view(m - 1), kv_len, search)
    assert sorted(l[1] for l, _ in last if l != "base" and l[0] == "draft") == list(range(m))
    first = oracle.visible_positions(synth.kind_mask_view(0), kv_len, search)
    assert sorted(l[1] for l, _ in first if l != "base" and l[0] == "mask") == list(range(m))
    # a mask view never sees the draft at its own position; a draft view always does
    for j in range(m):
        mv = oracle.visible_positions(synth.kind_mask_view(j), kv_len, search)
        dv = oracle.visible_positions(synth.kind_draft_view(j), kv_len, search)
        assert ("draft", j) not in [l for l, _ in mv] and ("mask", j) in [l for l, _ in mv]
        assert ("draft", j) in [l for l, _ in dv]
        # draft view j sees what mask view j+1 sees (one more accepted draft)
        if j + 1 < m:
            nxt = oracle.visible_positions(synth.kind_mask_view(j + 1), kv_len, search)
            assert sorted(map(str, dv)) == sorted(map(str, nxt))


def test_view_rule_with_drafts_filled_in_reduces_to_plain_forward():
    # D_m (all drafts visible) over a cache whose draft keys equal the base keys
    # at the search positions gives exactly the plain bidirectional forward
    rng = np.random.default_rng(19)
    H, hd, kv_len = 2, 8, 15
    search = [3, 11, 6]
    m = len(search)
    K = rng.standard_normal((kv_len + 2 * m, H * hd))
    V = rng.standard_normal((kv_len + 2 * m, H * hd))
    for j, s in enumerate(search):
        K[kv_len + j], V[kv_len + j] = K[s], V[s]
    q = rng.standard_normal((2, H, hd))
    bt = np.zeros((1, 1), np.int32)
    kinds = np.array([0, synth.kind_draft_view(m - 1)])
    o, lse, _ = oracle.sched_attn(q[[0, 0]], K, V, bt, kv_len + 2 * m, np.array([0, 2]), [kv_len], kinds,
                                  search_pos=[search], n_search=[m], max_seq=kv_len)
    np.testing.assert_allclose(o[1], o[0], atol=1e-6)
    np.testing.assert_allclose(lse[1], lse[0], atol=1e-12)


def test_view_rule_without_search_is_plain_attention():
    rng = np.random.default_rng(23)
    H, hd, n = 2, 4, 10
    K = rng.standard_normal((n, H * hd))
    V = rng.standard_normal((n, H * hd))
    q = rng.standard_normal((3, H, hd))
    bt = np.zeros((1, 1), np.int32)
    a = oracle.sched_attn(q, K, V, bt, n, np.array([0, 3]), [n], np.array([0, 1, 0]), max_seq=n)
    b = oracle.sched_attn(q, K, V, bt, n, np.array([0, 3]), [n], np.array([0, 1, 0]),
                          search_pos=[[]], n_search=[0], max_seq=n)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_tracker_single_row_equals_probabilities():
    g = golden("attention_hand.json")
    _, _, tr = _one_seq_attn(np.array([g["q"]]), np.array(g["k"]), np.array(g["v"]), kinds=[1])
    np.testing.assert_allclose(tr[0], g["p"], atol=1e-12)


# --------------------------------------------------------------------------- top-k
def test_topk_golden():
    g = golden("topk_hand.json")
    idx, cnt = oracle.track_topk(np.array(g["scores"]), np.array(g["eligible"]), g["seq_len"], g["k"])
    assert idx.tolist() == g["idx"] and cnt.tolist() == g["cnt"]


def test_topk_matches_full_sort_with_ties():
    rng = np.random.default_rng(29)
    B, N = 6, 300
    scores = rng.integers(0, 40, size=(B, N)).astype(np.float32) / 7   # many ties
    elig = (rng.uniform(size=(B, N)) < 0.6).astype(np.uint8)
    seq_len = rng.integers(0, N + 1, size=B)
    for k in (1, 8, 32, 400):
        idx, cnt = oracle.track_topk(scores, elig, seq_len, k)
        for b in range(B):
            pos = np.nonzero(elig[b, :seq_len[b]])[0]
            order = pos[np.lexsort((pos, -scores[b, pos].astype(np.float64)))]
            want = order[:k]
            assert cnt[b] == len(want)
            assert idx[b, :cnt[b]].tolist() == want.tolist()
            assert np.all(idx[b, cnt[b]:] == -1)


# --------------------------------------------------------------------------- unmask / verify
def test_unmask_golden():
    g = golden("unmask_hand.json")
    r = oracle.unmask(np.array(g["logits"]), g["row_seq"], g["row_pos"], 2, g["eps"], False, g["max_search"])
    np.testing.assert_allclose(r["conf"], g["conf"], rtol=1e-14)
    assert r["argmax"].tolist() == g["argmax"]
    assert r["commit"].tolist() == g["commit"]
    assert r["n_search"].tolist() == [0, 0]


def test_unmask_order_golden():
    g = golden("unmask_order_hand.json")
    L = np.array(g["logits"])
    r = oracle.unmask(L, g["row_seq"], g["row_pos"], 1, g["eps"], False, g["max_search"])
    assert r["search_rows"][0].tolist() == g["search_plain"]
    f = oracle.unmask(L, g["row_seq"], g["row_pos"], 1, g["eps"], True, g["max_search"])
    assert f["search_rows"][0].tolist() == g["search_forced"]
    assert f["commit"].tolist() == g["commit_forced"]


def test_confidence_closed_forms():
    V = 1000
    # uniform row: c = 1/V; single spike of height s over zeros: e^s / (e^s + V - 1)
    L = np.zeros((3, V))
    L[1, 17] = 4.0
    L[2, 999] = 30.0
    c, a = oracle.row_confidence(L)
    np.testing.assert_allclose(c[0], 1.0 / V, rtol=1e-14)
    np.testing.assert_allclose(c[1], math.exp(4) / (math.exp(4) + V - 1), rtol=1e-14)
    np.testing.assert_allclose(c[2], math.exp(30) / (math.exp(30) + V - 1), rtol=1e-14)
    assert a.tolist() == [0, 17, 999]
    # c invariant under adding a constant to a row; bounded in [1/V, 1]
    rng = np.random.default_rng(31)
    L = rng.standard_normal((50, V)) * 4
    c1, a1 = oracle.row_confidence(L)
    c2, a2 = oracle.row_confidence(L + 123.0)
    np.testing.assert_allclose(c1, c2, rtol=1e-12)
    assert np.all(a1 == a2)
    assert np.all(c1 >= 1.0 / V) and np.all(c1 <= 1.0)
    # the max probability equals the softmax value at the argmax
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    np.testing.assert_allclose(c1, p[np.arange(50), a1], rtol=1e-12)


def test_unmask_commit_is_exactly_threshold_set():
    rng = np.random.default_rng(37)
    V, R, B = 64, 60, 4
    L = rng.standard_normal((R, V)) * 2
    L[np.arange(R), rng.integers(0, V, R)] += rng.uniform(0, 12, R)
    seq = np.sort(rng.integers(0, B, R))
    pos = np.arange(R)
    for eps in (0.3, 0.9):
        r = oracle.unmask(L, seq, pos, B, eps, False, 5)
        c = r["conf"]
        assert set(np.nonzero(r["commit"])[0]) == set(np.nonzero(c >= eps)[0])
        for b in range(B):
            unc = [i for i in range(R) if seq[i] == b and c[i] < eps]
            unc.sort(key=lambda i: -c[i])
            assert r["search_rows"][b, :r["n_search"][b]].tolist() == unc[:5]
        f = oracle.unmask(L, seq, pos, B, eps, True, 5)
        for b in range(B):
            rows = [i for i in range(R) if seq[i] == b]
            if rows and not any(c[i] >= eps for i in rows):
                assert [i for i in rows if f["commit"][i]] == [max(rows, key=lambda i: c[i])]


def test_verify_golden():
    g = golden("verify_hand.json")
    r = oracle.verify(np.array(g["mask_logits"]), g["draft_tok"], g["n_search"], g["gamma"], 2, g["max_search"])
    assert r["accept"].tolist() == g["accept"]
    assert r["n_accept"].tolist() == g["n_accept"]


def test_verify_accepts_a_prefix_brute_force():
    rng = np.random.default_rng(41)
    B, S, V, gamma = 20, 6, 5, 0.8
    L = rng.standard_normal((B * S, V))
    L[np.arange(B * S), rng.integers(0, V, B * S)] += rng.uniform(0, 6, B * S)
    draft = rng.integers(0, V, B * S)
    ns = rng.integers(0, S + 1, B)
    r = oracle.verify(L, draft, ns, gamma, B, S)
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    for b in range(B):
        ok = [bool(draft[b * S + j] == np.argmax(p[b * S + j]) and p[b * S + j].max() >= gamma)
              for j in range(ns[b])]
        stop = ok.index(False) if False in ok else len(ok)
        assert r["n_accept"][b] == stop
        assert r["accept"][b * S:(b + 1) * S].tolist() == [1] * stop + [0] * (S - stop)


def test_theorem1_bias_bound():
    # TV(delta_{x~}, p~) = 1 - c~ <= 1 - gamma per accepted token and
    # 1 - prod c~ <= 1 - gamma^m over an accepted block of m tokens
    rng = np.random.default_rng(43)
    B, S, V, gamma = 30, 8, 16, 0.8
    L = rng.standard_normal((B * S, V))
    L[np.arange(B * S), rng.integers(0, V, B * S)] += rng.uniform(2, 9, B * S)
    _, arg = oracle.row_confidence(L)
    r = oracle.verify(L, arg, np.full(B, S), gamma, B, S)
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    for b in range(B):
        m = int(r["n_accept"][b])
        prod = 1.0
        for j in range(m):
            i = b * S + j
            tv = oracle.tv_point_mass(p[i], int(r["mask_argmax"][i]))
            np.testing.assert_allclose(tv, 1.0 - r["mask_conf"][i], atol=1e-12)
            assert tv <= 1 - gamma + 1e-12
            prod *= r["mask_conf"][i]
        assert 1 - prod <= 1 - gamma ** m + 1e-12


# --------------------------------------------------------------------------- generator recipes
def test_flash_verify_recipe_rates():
    wl = synth.flash_verify(batch=4)
    e = wl.extra
    c, a = oracle.row_confidence(e["logits"].values())
    frac_hi = float(np.mean(c >= e["eps"]))
    assert 0.25 <= frac_hi <= 0.35
    cm, am = oracle.row_confidence(e["mask_logits_by_window_row"].values())
    agree = float(np.mean(am == a))
    assert 0.55 <= agree <= 0.85
    assert 0.35 <= float(np.mean(cm >= e["gamma"])) <= 0.65


# --------------------------------------------------------------------------- LM head (next-row f1)
def test_lm_head_logits_brute_force_and_unit_rows():
    # brute force: every logit as an explicit sum over the hidden dimension
    rng = np.random.default_rng(21)
    h = rng.standard_normal((3, 5))
    w = rng.standard_normal((7, 5))
    L = oracle.lm_head_logits(h, w, chunk=3)
    for r in range(3):
        for v in range(7):
            assert abs(L[r, v] - sum(h[r, k] * w[v, k] for k in range(5))) < 1e-12
    # unit vocabulary rows pick hidden components: W = I gives l = h exactly,
    # a permutation of I permutes them (a transposed operand fails this)
    assert np.array_equal(oracle.lm_head_logits(h, np.eye(5)), h)
    perm = np.array([3, 0, 4, 1, 2])
    assert np.array_equal(oracle.lm_head_logits(h, np.eye(5)[perm]), h[:, perm])
    # chunking only bounds memory (the library product may reassociate)
    np.testing.assert_allclose(oracle.lm_head_logits(h, w, chunk=1), oracle.lm_head_logits(h, w, chunk=100),
                               rtol=1e-14, atol=1e-14)


def test_lm_head_unmask_closed_form_and_composition():
    # one vocabulary row aligned with the hidden state, all others zero: the
    # logits are (a, 0, ..., 0) with a = 6 |h|^2, so c = e^a / (e^a + V - 1)
    V, d = 50, 8
    h = np.zeros((2, d))
    h[0, :4] = 0.5
    h[1, 6] = 1.0  # orthogonal to h[0]: all of row 1's logits are 0
    w = np.zeros((V, d))
    w[17] = 6.0 * h[0]
    out = oracle.lm_head_unmask(h, w, np.array([0, 0]), np.array([10, 11]), 1, 0.5, False, 4)
    a = 6.0 * float(h[0] @ h[0])
    assert abs(out["conf"][0] - math.exp(a) / (math.exp(a) + V - 1)) < 1e-12
    assert out["argmax"][0] == 17
    assert abs(out["conf"][1] - 1.0 / V) < 1e-12 and out["argmax"][1] == 0  # all-zero row: lowest id
    assert out["commit"].tolist() == [1, 0] and out["n_search"].tolist() == [1]
    # the composition with explicit logits
    hidden, wl, _ = synth.lm_head_case(seed=5, vocab=300, d=32, rows=6)
    want = oracle.unmask(hidden.values() @ wl.values().T, np.zeros(6, np.int32), np.arange(6), 1, 0.9, True, 4)
    got = oracle.lm_head_unmask(hidden.values(), wl.values(), np.zeros(6, np.int32), np.arange(6), 1, 0.9, True, 4)
    for key in ("commit", "search_rows", "n_search", "argmax"):
        assert np.array_equal(got[key], want[key])
    np.testing.assert_allclose(got["conf"], want["conf"], rtol=1e-12)


def test_lm_head_verify_closed_form_walk():
    # two sequences, three mask views each, orthogonal unit hidden rows: row r's
    # logits are 0 except a_r at its aligned vocabulary row, so its confidence
    # is e^a / (e^a + V - 1) and its argmax that row (or 0 when a_r = 0)
    V, d, gamma = 40, 8, 0.8
    h = np.eye(d)[:6]
    a_r = [9.0, 9.0, 2.0, 9.0, 0.0, 9.0]            # e^9/(e^9+39) = 0.9952, e^2/(e^2+39) = 0.159
    w = np.zeros((V, d))
    ids = [5, 11, 23, 7, 0, 30]
    for r, (a, v) in enumerate(zip(a_r, ids)):
        w[v] += a * h[r]
    conf = [math.exp(a) / (math.exp(a) + V - 1) for a in a_r]
    # sequence 0: both confident rows agree, then row 2 is below gamma -> 2
    # sequence 1 (two search tokens): row 3 agrees, row 4 is flat (conf 1/V) -> 1
    draft = np.array([5, 11, 23, 7, 0, 30])
    out = oracle.lm_head_verify(h, w, draft, np.array([3, 2]), gamma, 2, 3)
    assert out["n_accept"].tolist() == [2, 1]
    assert out["accept"].tolist() == [1, 1, 0, 1, 0, 0]
    np.testing.assert_allclose(out["mask_conf"][:4], conf[:4], rtol=1e-12)
    assert abs(out["mask_conf"][4] - 1.0 / V) < 1e-12
    assert out["mask_argmax"].tolist()[:5] == ids[:5]
    # a draft mismatch at the first token stops the walk at once
    draft[0] = 6
    assert oracle.lm_head_verify(h, w, draft, np.array([3, 2]), gamma, 2, 3)["n_accept"].tolist() == [0, 1]
    # views past n_search never count: row 1 would be accepted, but sequence 0
    # has one search token
    draft[0] = 5
    assert oracle.lm_head_verify(h, w, draft, np.array([1, 1]), gamma, 2, 3)["n_accept"].tolist() == [1, 1]
    # composition with explicit logits
    hidden, wl, _ = synth.lm_head_case(seed=6, vocab=300, d=32, rows=6, planted=1.0)
    logits = hidden.values() @ wl.values().T
    tok = np.argmax(logits, axis=1)
    want = oracle.verify(logits, tok, np.array([3, 3]), 0.6, 2, 3)
    got = oracle.lm_head_verify(hidden.values(), wl.values(), tok, np.array([3, 3]), 0.6, 2, 3)
    for key in ("accept", "n_accept", "mask_argmax"):
        assert np.array_equal(got[key], want[key])


def test_lm_head_case_plants_confident_rows():
    # the generator's recipe: planted rows are confident in their planted id
    hidden, w, ids = synth.lm_head_case(seed=3, vocab=2048, d=128, rows=20)
    c, a = oracle.row_confidence(oracle.lm_head_logits(hidden.values(), w.values()))
    planted = ids >= 0
    assert planted.sum() == 6
    assert np.array_equal(a[planted], ids[planted])
    assert (c[planted] > 0.3).all() and (c[~planted] < 0.05).all()
