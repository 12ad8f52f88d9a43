"""Fused LM head + unmasking (the next step after the layers): the window
rows' hidden states times the LM-head weight, reduced straight to the eps
rule's decisions without storing the logits. Against the float64 oracle
(``lm_head_unmask``) on identical bf16 inputs.

Confidences within the fp32 tolerance; argmax, commit mask and search list
bit-exact wherever the oracle's decision is not a near-tie (top-2 logits
within 1e-3, a confidence within 1e-3 of eps, or two ranked confidences within
1e-6 relative of each other); everywhere, the decisions must be exactly the
oracle's decision rule applied to the kernel's own confidences."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _run(ctx, hidden, w, row_seq, row_pos, B, eps, force, ms):
    torch = H.torch_mod()
    R = hidden.shape[0]
    conf = torch.empty(R, dtype=torch.float32, device="cuda")
    arg = torch.empty(R, dtype=torch.int32, device="cuda")
    com = torch.empty(R, dtype=torch.uint8, device="cuda")
    srows = torch.full((B, ms), -7, dtype=torch.int32, device="cuda")
    nsr = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.lm_head_unmask(hidden, w, B, ms, row_seq=H.ints(row_seq), row_pos=H.ints(row_pos), eps=eps,
                       force_progress=force, conf=conf, argmax=arg, commit=com, search_rows=srows, n_search=nsr)
    ctx.sync_status()
    return H.host(conf), H.host(arg), H.host(com), H.host(srows), H.host(nsr)


def _check(got, logits, row_seq, row_pos, B, eps, force, ms, rows=None):
    """rows: the window rows whose oracle logits are given (all when None)."""
    conf, arg, com, srows, nsr = got
    R = len(conf)
    rows = np.arange(R) if rows is None else np.asarray(rows)
    c_o, a_o = oracle.row_confidence(logits)
    np.testing.assert_allclose(conf[rows], c_o, atol=H.F32_TOL, rtol=0)
    top2 = np.sort(logits, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 1e-3
    assert np.array_equal(arg[rows][clear], a_o[clear])
    # the decisions are exactly the rule applied to the kernel's confidences
    want = _decide(conf, row_seq, row_pos, B, eps, force, ms)
    assert com.tolist() == want["commit"].tolist()
    assert nsr.tolist() == want["n_search"].tolist()
    assert srows.tolist() == want["search_rows"].tolist()
    return c_o, clear


def _decide(conf, row_seq, row_pos, B, eps, force, ms):
    """The oracle's unmask decision rule on given confidences (float32 values
    compared as float64, the same numbers the kernel compared)."""
    conf = np.asarray(conf, np.float64)
    commit = (conf >= np.float64(np.float32(eps))).astype(np.uint8)
    search = np.full((B, ms), -1, dtype=np.int64)
    n_search = np.zeros(B, dtype=np.int64)
    for b in range(B):
        rows = [r for r in range(len(conf)) if int(row_seq[r]) == b]
        if force and rows and not any(commit[r] for r in rows):
            commit[min(rows, key=lambda r: (-conf[r], int(row_pos[r])))] = 1
        unc = sorted((r for r in rows if not commit[r]), key=lambda r: (-conf[r], int(row_pos[r])))[:ms]
        search[b, :len(unc)] = unc
        n_search[b] = len(unc)
    return dict(commit=commit, search_rows=search, n_search=n_search)


def _ctx(d, V, B, R):
    import kv_cache_attention_gb300 as fdl
    return fdl.fdl_create(d, d // 128, 128, 5e5, B, 64, 0, 64, 1, max(R, 64), V, "bf16")


def test_lm_head_unmask_ragged_vocab_two_sequences():
    # vocab 16384 + 77: 129 vocabulary tiles with a ragged last one
    d, V, R, B, ms = 4096, 16384 + 77, 32, 2, 16
    hidden, w, ids = synth.lm_head_case(seed=1007, vocab=V, d=d, rows=R)
    row_seq = np.repeat(np.arange(B), R // B).astype(np.int32)
    row_pos = (512 + np.arange(R)).astype(np.int32)
    ctx = _ctx(d, V, B, R)
    for eps, force in ((0.9, False), (0.6, True)):
        got = _run(ctx, H.dev(hidden), H.dev(w), row_seq, row_pos, B, eps, force, ms)
        logits = oracle.lm_head_logits(hidden.values(), synth.bf16_bits_to_f32(w.data))
        c_o, _ = _check(got, logits, row_seq, row_pos, B, eps, force, ms)
        # the oracle's own decisions wherever none is a near-tie
        ref = oracle.unmask(logits, row_seq, row_pos, B, eps, force, ms)
        if not np.any(np.abs(c_o - eps) < 1e-3):
            assert got[2].tolist() == ref["commit"].tolist()
        planted = ids >= 0
        assert np.array_equal(got[1][planted], ids[planted])
    ctx.close()


def test_lm_head_unmask_full_vocab_sampled():
    # the LLaDA vocabulary and width, 32 window rows of one sequence; the
    # oracle computes a sample of rows one by one
    d, V, R, B, ms = 4096, 126464, 32, 1, 16
    hidden, w, ids = synth.lm_head_case(seed=1008, vocab=V, d=d, rows=R)
    row_seq = np.zeros(R, np.int32)
    row_pos = (512 + np.arange(R)).astype(np.int32)
    ctx = _ctx(d, V, B, R)
    got = _run(ctx, H.dev(hidden), H.dev(w), row_seq, row_pos, B, 0.9, True, ms)
    pick = np.random.default_rng(0).choice(R, size=6, replace=False)
    w32 = synth.bf16_bits_to_f32(w.data)
    logits = oracle.lm_head_logits(hidden.values()[pick], w32)
    _check(got, logits, row_seq, row_pos, B, 0.9, True, ms, rows=pick)
    planted = ids >= 0
    assert np.array_equal(got[1][planted], ids[planted])
    # repeat: the fixed-order reductions give the same bits
    again = _run(ctx, H.dev(hidden), H.dev(w), row_seq, row_pos, B, 0.9, True, ms)
    for x, y in zip(got, again):
        assert np.array_equal(x, y)
    ctx.close()


def test_lm_head_unmask_limits():
    import kv_cache_attention_gb300 as fdl
    torch = H.torch_mod()
    d, V = 256, 1000
    ctx = fdl.fdl_create(d, 2, 128, 5e5, 2, 64, 0, 64, 1, 128, V, "bf16")
    w = torch.zeros((V, d), dtype=torch.bfloat16, device="cuda")
    for R in (129, 0):            # max_rows is 128
        h = torch.zeros((max(R, 1), d), dtype=torch.bfloat16, device="cuda")
        hh = h if R else h[:0]
        with pytest.raises(fdl.FdlError):
            _run(ctx, hh, w, np.zeros(max(R, 1), np.int32), np.zeros(max(R, 1), np.int32), 1, 0.9, False, 4)
    # 64 rows (the limit), all logits zero: every confidence is 1 / V, argmax 0
    h = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
    got = _run(ctx, h, w, np.zeros(64, np.int32), np.arange(64, dtype=np.int32), 1, 0.9, False, 8)
    np.testing.assert_allclose(got[0], 1.0 / V, rtol=1e-5)
    assert got[1].tolist() == [0] * 64
    assert got[4].tolist() == [8] and got[3][0].tolist() == list(range(8))
    # 100 rows take the many-row kernel (128-row tiles): the same closed form
    h = torch.zeros((100, d), dtype=torch.bfloat16, device="cuda")
    got = _run(ctx, h, w, np.zeros(100, np.int32), np.arange(100, dtype=np.int32), 1, 0.9, False, 8)
    np.testing.assert_allclose(got[0], 1.0 / V, rtol=1e-5)
    assert got[1].tolist() == [0] * 100
    assert got[4].tolist() == [8] and got[3][0].tolist() == list(range(8))
    ctx.close()


def _verify_rule(mask_conf, mask_arg, draft, n_search, gamma, B, ms):
    """The verify rule on given (c~, x~): float32 confidences compared as
    float64 against float32(gamma), the comparison the kernel makes."""
    accept = np.zeros(B * ms, np.uint8)
    n_accept = np.zeros(B, np.int64)
    g = np.float64(np.float32(gamma))
    for b in range(B):
        for j in range(int(n_search[b])):
            r = b * ms + j
            if int(draft[r]) != int(mask_arg[r]) or np.float64(mask_conf[r]) < g:
                break
            accept[r] = 1
            n_accept[b] += 1
    return accept, n_accept


def test_lm_head_verify_ragged_vocab():
    torch = H.torch_mod()
    d, V, B, ms, gamma = 4096, 16384 + 77, 3, 5, 0.8
    R = B * ms
    hidden, w, _ = synth.lm_head_case(seed=1012, vocab=V, d=d, rows=R, planted=1.0)
    c0, _ = oracle.row_confidence(oracle.lm_head_logits(hidden.values(), w.values()))
    # the most confident mask views first, so sequence 0's walk runs several tokens
    hidden = synth.make_tensor(hidden.values()[np.argsort(-c0, kind="stable")], "bf16")
    logits = oracle.lm_head_logits(hidden.values(), w.values())
    n_search = np.array([5, 2, 0], np.int32)
    _, a_o = oracle.row_confidence(logits)
    draft = a_o.astype(np.int32).copy()                 # drafts agree with the mask views' argmax,
    draft[3] = (draft[3] + 1) % V                       # except one inside sequence 0's walk
    want = oracle.verify(logits, draft, n_search, gamma, B, ms)
    ctx = _ctx(d, V, B, R)
    mc = torch.full((R,), -5.0, dtype=torch.float32, device="cuda")
    ma = torch.full((R,), -5, dtype=torch.int32, device="cuda")
    acc = torch.full((R,), 7, dtype=torch.uint8, device="cuda")
    nacc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    ctx.lm_head_verify(H.dev(hidden), H.dev(w), B, ms, n_search=H.ints(n_search), draft_tok=H.ints(draft),
                       gamma=gamma, accept=acc, n_accept=nacc, mask_conf=mc, mask_argmax=ma)
    ctx.sync_status()
    mc, ma, acc, nacc = H.host(mc), H.host(ma), H.host(acc), H.host(nacc)
    valid = np.array([b * ms + j for b in range(B) for j in range(n_search[b])])
    rest = np.setdiff1d(np.arange(R), valid)
    assert (mc[rest] == -5.0).all() and (ma[rest] == -5).all()      # views past n_search are not written
    np.testing.assert_allclose(mc[valid], want["mask_conf"][valid], atol=H.F32_TOL, rtol=0)
    top2 = np.sort(logits[valid], axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 1e-3
    assert np.array_equal(ma[valid][clear], want["mask_argmax"][valid][clear])
    # the decisions are exactly the rule applied to the kernel's own values ...
    rule_acc, rule_n = _verify_rule(mc, ma, draft, n_search, gamma, B, ms)
    assert acc.tolist() == rule_acc.tolist() and nacc.tolist() == rule_n.tolist()
    # ... and the oracle's wherever no walked confidence sits within 1e-3 of gamma
    for b in range(B):
        rows = valid[valid // ms == b]
        if not (np.abs(want["mask_conf"][rows] - gamma) < 1e-3).any():
            assert nacc[b] == want["n_accept"][b]
            assert acc[b * ms:(b + 1) * ms].tolist() == want["accept"][b * ms:(b + 1) * ms].tolist()
    assert nacc[0] == 3 and nacc[2] == 0
    ctx.close()


def test_lm_head_verify_limits():
    import kv_cache_attention_gb300 as fdl
    torch = H.torch_mod()
    d, V = 4096, 1024
    ctx = _ctx(d, V, 16, 64)
    w = torch.zeros((V, d), dtype=torch.bfloat16, device="cuda")
    h = torch.zeros((80, d), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(80, dtype=torch.int32, device="cuda")
    f = torch.zeros(80, dtype=torch.float32, device="cuda")
    u = torch.zeros(80, dtype=torch.uint8, device="cuda")
    for B, ms, status in ((13, 5, fdl.FDL_ERR_INVALID_ARG), (1, 0, fdl.FDL_ERR_INVALID_ARG)):
        with pytest.raises(fdl.FdlError) as ei:
            ctx.lm_head_verify(h, w, B, ms, n_search=z, draft_tok=z, gamma=0.8, accept=u, n_accept=z,
                               mask_conf=f, mask_argmax=z)
        assert ei.value.status == status
    # 64 mask views of zero logits: c~ = 1/V < gamma, so nothing is accepted
    ns = torch.full((16,), 4, dtype=torch.int32, device="cuda")
    nacc = torch.full((16,), -1, dtype=torch.int32, device="cuda")
    ctx.lm_head_verify(h[:64], w, 16, 4, n_search=ns, draft_tok=z[:64], gamma=0.8, accept=u[:64], n_accept=nacc,
                       mask_conf=f[:64], mask_argmax=z[:64])
    ctx.sync_status()
    assert (H.host(nacc) == 0).all() and (H.host(u[:64]) == 0).all()
    np.testing.assert_allclose(H.host(f[:64]), 1.0 / V, rtol=1e-6)
    ctx.close()


def _clear_sequences(conf, logits, row_seq, B, threshold):
    """Sequences whose float64 values hold no near-tie that fp32 could decide
    the other way: a top-2 logit gap below 1e-3, a confidence within 1e-5 of
    the (float32) threshold, or two confidences of the sequence within 1e-6
    relative of each other."""
    conf = np.asarray(conf, np.float64)
    top2 = np.sort(logits, axis=1)[:, -2:]
    gap_ok = (top2[:, 1] - top2[:, 0]) >= 1e-3
    thr_ok = np.abs(conf - np.float64(np.float32(threshold))) >= 1e-5
    out = []
    for b in range(B):
        rows = np.nonzero(np.asarray(row_seq) == b)[0]
        c = np.sort(conf[rows])
        ties = len(c) > 1 and (np.diff(c) < 1e-6 * c[1:]).any()
        out.append(bool(gap_ok[rows].all() and thr_ok[rows].all() and not ties))
    return np.array(out)


@pytest.mark.slow
def test_lm_head_unmask_flash_verify_scale():
    """The Flash-Verify stress scale: 32 sequences x 32 window rows (1024
    rows, the many-row kernel) over the LLaDA vocabulary and width, every
    row's confidence against the float64 oracle, the decisions exactly the
    oracle's for every sequence clear of a near-tie (and the rule on the
    kernel's confidences for the others)."""
    d, V, B, W, ms, eps = 4096, 126464, 32, 32, 16, 0.9
    R = B * W
    hidden, w, ids = synth.lm_head_case(seed=1031, vocab=V, d=d, rows=R, planted=0.6)
    row_seq = np.repeat(np.arange(B), W).astype(np.int32)
    row_pos = np.tile(512 + np.arange(W), B).astype(np.int32)
    ctx = _ctx(d, V, B, R)
    got = _run(ctx, H.dev(hidden), H.dev(w), row_seq, row_pos, B, eps, True, ms)
    logits = oracle.lm_head_logits(hidden.values(), synth.bf16_bits_to_f32(w.data))
    ref = oracle.unmask(logits, row_seq, row_pos, B, eps, True, ms)
    conf, arg, com, srows, nsr = got
    H.assert_close(conf, ref["conf"], "f32", "confidences at 1024 rows")
    top2 = np.sort(logits, axis=1)[:, -2:]
    clear_rows = (top2[:, 1] - top2[:, 0]) > 1e-3
    assert np.array_equal(arg[clear_rows], ref["argmax"][clear_rows])
    want = _decide(conf, row_seq, row_pos, B, eps, True, ms)
    assert com.tolist() == want["commit"].tolist() and srows.tolist() == want["search_rows"].tolist()
    clear = _clear_sequences(ref["conf"], logits, row_seq, B, eps)
    assert clear.sum() >= B // 2, clear.sum()
    for b in np.nonzero(clear)[0]:
        rows = np.nonzero(row_seq == b)[0]
        assert com[rows].tolist() == ref["commit"][rows].tolist(), b
        assert srows[b].tolist() == ref["search_rows"][b].tolist(), b
        assert nsr[b] == ref["n_search"][b], b
    assert np.array_equal(arg[ids >= 0], ids[ids >= 0])
    # the fixed-order reductions repeat bit for bit
    again = _run(ctx, H.dev(hidden), H.dev(w), row_seq, row_pos, B, eps, True, ms)
    for x, y in zip(got, again):
        assert np.array_equal(x, y)
    ctx.close()


@pytest.mark.slow
def test_lm_head_verify_flash_verify_scale():
    """32 sequences x 16 mask views (512 rows) over the LLaDA vocabulary:
    the verify-side fused LM head against the float64 oracle's acceptance."""
    torch = H.torch_mod()
    d, V, B, ms, gamma = 4096, 126464, 32, 16, 0.8
    R = B * ms
    hidden, w, _ = synth.lm_head_case(seed=1032, vocab=V, d=d, rows=R, planted=1.0)
    logits = oracle.lm_head_logits(hidden.values(), synth.bf16_bits_to_f32(w.data))
    rng = np.random.default_rng(1033)
    n_search = rng.integers(0, ms + 1, B).astype(np.int32)
    _, a_o = oracle.row_confidence(logits)
    draft = a_o.astype(np.int32).copy()
    flip = rng.random(R) < 0.15                         # some drafts disagree with the mask view
    draft[flip] = (draft[flip] + 1) % V
    want = oracle.verify(logits, draft, n_search, gamma, B, ms)
    ctx = _ctx(d, V, B, R)
    mc = torch.full((R,), -5.0, dtype=torch.float32, device="cuda")
    ma = torch.full((R,), -5, dtype=torch.int32, device="cuda")
    acc = torch.full((R,), 7, dtype=torch.uint8, device="cuda")
    nacc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    ctx.lm_head_verify(H.dev(hidden), H.dev(w), B, ms, n_search=H.ints(n_search), draft_tok=H.ints(draft),
                       gamma=gamma, accept=acc, n_accept=nacc, mask_conf=mc, mask_argmax=ma)
    ctx.sync_status()
    mc, ma, acc, nacc = H.host(mc), H.host(ma), H.host(acc), H.host(nacc)
    valid = np.array([b * ms + j for b in range(B) for j in range(n_search[b])])
    rest = np.setdiff1d(np.arange(R), valid)
    assert (mc[rest] == -5.0).all() and (ma[rest] == -5).all()
    H.assert_close(mc[valid], want["mask_conf"][valid], "f32", "mask-view confidences at 512 rows")
    top2 = np.sort(logits[valid], axis=1)[:, -2:]
    assert ((top2[:, 1] - top2[:, 0]) > 1e-3).all()     # planted rows: clear argmaxes
    assert np.array_equal(ma[valid], want["mask_argmax"][valid])
    near = np.abs(want["mask_conf"] - np.float64(np.float32(gamma))) < 1e-5
    for b in range(B):
        rows = np.arange(b * ms, b * ms + n_search[b])
        if not near[rows].any():
            assert nacc[b] == want["n_accept"][b], b
            assert acc[b * ms:(b + 1) * ms].tolist() == want["accept"][b * ms:(b + 1) * ms].tolist(), b
    assert want["n_accept"].sum() > 0 and (want["n_accept"] < n_search).any()
    ctx.close()
