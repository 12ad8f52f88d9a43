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
    for R in (65, 0):
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
    for B, ms, status in ((13, 5, fdl.FDL_ERR_UNSUPPORTED), (1, 0, fdl.FDL_ERR_INVALID_ARG)):
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
