"""Whole Flash-dLLM denoising steps on the GPU (fdl_flash_step: the draft
forward through every layer, the fused LM-head unmasking, the verify forward
with its two views per search token, the acceptance walk, the next tracked
set) against the float64 step oracle, by teacher forcing.

Each step starts the oracle from the GPU's own state (tokens, masks, tracked
set and the caches, downloaded before the step) and forces it to follow the
GPU's decisions. Compared:
  * the row sets, exactly;
  * the final rows of both forwards, element by element (two bf16 ulps where
    an ulp exceeds the bf16 tolerance, as for the whole-model forward);
  * each stage boundary on identical inputs: the fused LM head run on the
    oracle's own final window rows must give the oracle's confidences (fp32
    tolerance) and exactly its argmax, commit mask and search lists; the
    verify-side LM head run on the oracle's own mask-view rows must give its
    mask confidences and exactly its predictions and acceptance (a step whose
    oracle values hold a near-tie, where fp32 and float64 may decide
    differently, is checked by the rule instead, and most steps must be
    clear of one);
  * the tracker scores and the caches after the step;
  * the GPU's own decisions, which must be the decision rules applied to its
    own confidences, and its next state, which must be exactly what those
    decisions give."""
import numpy as np
import pytest

import oracle
from oracle import flash_loop as fl
import synth
from tests import _harness as H
from tests.test_gpu_lm_head import _decide, _verify_rule

pytestmark = pytest.mark.gpu


# (prompt lengths, generation lengths): two sequences (32 window rows, the
# one-tile LM head), then five (80 window rows and up to 40 mask views: the
# many-row LM head on the unmask side)
CASES = [([20, 27], [32, 24]), ([20, 27, 9, 33, 14], [32, 24, 40, 16, 29])]


@pytest.mark.parametrize("prompts,gens", CASES)
def test_flash_steps_teacher_forced(prompts, gens):
    torch = H.torch_mod()
    import kv_cache_attention_gb300 as fdl
    mc = synth.model_case(seed=1015, d=512, n_heads=4, n_layers=2, ffn=1024, vocab=2088, out_std=0.5, lm_std=0.2)
    m = synth.model_values(mc)
    w_lm = m["w_lm"]
    L, d, V = len(mc["layers"]), mc["d_model"], mc["vocab"]
    B = len(prompts)
    lengths = (np.array(prompts) + np.array(gens)).astype(np.int32)
    N = int(lengths.max())
    params = dict(window=16, track_budget=16, max_search=8, eps=0.5, gamma=0.2, force_progress=True,
                  mask_id=mc["mask_id"], max_views=16)
    W, MS, BT = params["window"], params["max_search"], params["track_budget"]
    rng = np.random.default_rng(1016)
    geom = synth.paged_geometry(rng, lengths + 2 * MS, 64)      # room for the view keys
    n_slots = geom.n_pages * geom.page_size
    tokens = np.full((B, N), mc["mask_id"], np.int32)
    masked = np.zeros((B, N), np.uint8)
    for b in range(B):
        tokens[b, :prompts[b]] = rng.integers(0, V - 1, prompts[b])
        masked[b, prompts[b]:lengths[b]] = 1
    seqs = dict(prompt_len=np.array(prompts, np.int32), seq_len=lengths, tokens=tokens, masked=masked,
                tracked=np.full((B, BT), -1, np.int32), n_tracked=np.zeros(B, np.int32),
                state=np.full(B, -1, np.int32))
    ctx = fdl.fdl_create(d, mc["n_heads"], mc["head_dim"], mc["theta"], B, N, params["max_views"], geom.page_size,
                         geom.n_pages, int(lengths.sum()), V, "bf16")
    dm = dict(ffn=mc["ffn"], eps=mc["eps"], embed=H.dev(mc["embed"]), g_final=H.dev(mc["g_final"]),
              layers=[{k: H.dev(v) for k, v in w.items()} for w in mc["layers"]])
    wl = H.dev(mc["w_lm"])
    kcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    vcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    bt = H.ints(geom.block_table)
    ws = torch.empty(ctx.flash_workspace_bytes(mc["ffn"], params, B, N), dtype=torch.uint8, device="cuda")
    saw = dict(commit=0, search=0, accept=0, verify_steps=0, max_rw=0)
    checked_steps = exact_steps = exact_verify = 0
    for step in range(64):
        if not seqs["masked"].any():
            break
        snap = {k: v.copy() for k, v in seqs.items()}
        snap_tracked = [snap["tracked"][b, :snap["n_tracked"][b]].tolist() for b in range(B)]
        caches = ([H.host(t).astype(np.float64) for t in kcs], [H.host(t).astype(np.float64) for t in vcs])
        rec = ctx.flash_step(dm, wl, kcs, vcs, bt, params, seqs, ws)
        RW = int(rec["n_window"][0])
        saw["max_rw"] = max(saw["max_rw"], RW)
        force = dict(argmax=rec["argmax"][:RW], commit=rec["commit"][:RW],
                     search_rows=rec["search_rows"].reshape(B, MS), n_search=rec["n_search"],
                     n_accept=rec["n_accept"])
        o_seqs, (okc, ovc), tr = fl.flash_step(
            m, w_lm, dict(prompt_len=snap["prompt_len"], seq_len=snap["seq_len"], tokens=snap["tokens"],
                          masked=snap["masked"], tracked=snap_tracked, state=snap["state"]),
            params, caches, geom, dtype="bf16", force=force)
        # rows
        assert int(rec["n_rows"][0]) == len(tr["draft_pos"]), step
        assert rec["window_pos"][:RW].tolist() == tr["window_pos"].tolist()
        assert rec["window_seq"][:RW].tolist() == tr["window_seq"].tolist()
        # the draft forward's final rows
        _rows_close(rec["draft_final"], tr["draft_final"], f"draft rows, step {step}")
        dec = tr["unmask"]
        # stage boundary: the LM head and the eps decisions on the oracle's rows
        exact_steps += _lm_unmask_stage(ctx, wl, tr, dec, B, params, f"step {step}")
        checked_steps += 1
        # the GPU's decisions are the rule applied to its own confidences
        want = _decide(rec["conf"][:RW], tr["window_seq"], tr["window_pos"], B, params["eps"], True, MS)
        assert rec["commit"][:RW].tolist() == want["commit"].tolist()
        assert rec["n_search"].tolist() == want["n_search"].tolist()
        assert rec["search_rows"].reshape(B, MS).tolist() == want["search_rows"].tolist()
        saw["commit"] += int(rec["commit"][:RW].sum())
        saw["search"] += int(rec["n_search"].sum())
        # verify: the mask views and the acceptance walk
        if tr["verify"] is not None:
            saw["verify_steps"] += 1
            assert int(rec["n_rows"][1]) == len(tr["verify"]["final"])
            ver = tr["verify"]
            _rows_close(rec["verify_final"], ver["final"], f"verify rows, step {step}")
            exact_verify += _lm_verify_stage(ctx, wl, ver, rec["n_search"], B, params, f"step {step}")
            acc, n_acc = _verify_rule(rec["mask_conf"], rec["mask_argmax"], ver["draft_tok"], rec["n_search"],
                                      params["gamma"], B, MS)
            assert rec["n_accept"].tolist() == n_acc.tolist()
            saw["accept"] += int(n_acc.sum())
        # the tracker and the caches after the step
        np.testing.assert_allclose(rec["track"].reshape(B, N), tr["track"], atol=5e-4, rtol=0)
        for l in range(L):
            H.assert_close(H.host(kcs[l]), okc[l], "bf16", f"k cache layer {l}, step {step}")
            H.assert_close(H.host(vcs[l]), ovc[l], "bf16", f"v cache layer {l}, step {step}")
        # the next state: tokens and masks exactly as the forced oracle's; the
        # tracked set = new positions, then the rule on the GPU's own scores
        assert np.array_equal(seqs["tokens"], o_seqs["tokens"]) and np.array_equal(seqs["masked"], o_seqs["masked"])
        assert seqs["state"].tolist() == o_seqs["state"].tolist()
        elig = tr["eligible"]
        idx, cnt = oracle.track_topk(rec["track"].reshape(B, N), elig, lengths, BT)
        for b in range(B):
            new = tr["new"][b][:BT]
            keep = max(0, BT - len(new))
            want_t = new + idx[b, :min(keep, int(cnt[b]))].tolist()
            assert seqs["tracked"][b, :seqs["n_tracked"][b]].tolist() == want_t, (step, b)
    else:
        pytest.fail("decode did not finish")
    assert not seqs["masked"].any()
    assert saw["commit"] > 0 and saw["search"] > 0 and saw["accept"] > 0 and saw["verify_steps"] > 0
    if B * W > 64:
        assert saw["max_rw"] > 64   # the many-row LM head ran inside the step
    # the identical-input stage checks were exact on most steps
    assert exact_steps >= 0.8 * checked_steps, (exact_steps, checked_steps)
    assert exact_verify >= 0.8 * saw["verify_steps"], (exact_verify, saw["verify_steps"])
    ctx.close()


def _near_ties(conf, logits, row_seq, threshold):
    """True where float64 and fp32 may decide differently: the top two logits
    within 1e-3, a confidence within 1e-5 of the (float32) threshold, or two
    confidences of one sequence within 1e-6 relative of each other."""
    conf = np.asarray(conf, np.float64)
    if len(conf) == 0:
        return False
    if (_top2_gap(logits) < 1e-3).any():
        return True
    if (np.abs(conf - np.float64(np.float32(threshold))) < 1e-5).any():
        return True
    for b in np.unique(row_seq):
        c = np.sort(conf[np.asarray(row_seq) == b])
        if len(c) > 1 and (np.diff(c) < 1e-6 * c[1:]).any():
            return True
    return False


def _lm_unmask_stage(ctx, wl, tr, dec, B, params, what):
    """The fused LM head + eps decisions on the oracle's own final window rows
    against the oracle's decisions from the same rows. Returns 1 when the
    decisions were compared exactly (0 when a near-tie left them to the rule)."""
    torch = H.torch_mod()
    MS = params["max_search"]
    hid = H.dev(synth.make_tensor(tr["draft_final"][tr["window_rows"]], "bf16"))
    RW = hid.shape[0]
    conf = torch.empty(RW, dtype=torch.float32, device="cuda")
    arg = torch.empty(RW, dtype=torch.int32, device="cuda")
    com = torch.empty(RW, dtype=torch.uint8, device="cuda")
    srows = torch.full((B, MS), -7, dtype=torch.int32, device="cuda")
    nsr = torch.empty((B,), dtype=torch.int32, device="cuda")
    ctx.lm_head_unmask(hid, wl, B, MS, row_seq=H.ints(tr["window_seq"]), row_pos=H.ints(tr["window_pos"]),
                       eps=params["eps"], force_progress=True, conf=conf, argmax=arg, commit=com,
                       search_rows=srows, n_search=nsr)
    ctx.sync_status()
    conf, arg, com, srows, nsr = H.host(conf), H.host(arg), H.host(com), H.host(srows), H.host(nsr)
    H.assert_close(conf, dec["conf"], "f32", f"LM-head confidences on the oracle's rows, {what}")
    if _near_ties(dec["conf"], tr["window_logits"], tr["window_seq"], params["eps"]):
        want = _decide(conf, tr["window_seq"], tr["window_pos"], B, params["eps"], True, MS)
        assert com.tolist() == want["commit"].tolist(), what
        assert srows.tolist() == want["search_rows"].tolist(), what
        return 0
    assert arg.tolist() == dec["argmax"].tolist(), what
    assert com.tolist() == dec["commit"].tolist(), what
    assert nsr.tolist() == dec["n_search"].tolist(), what
    assert srows.tolist() == dec["search_rows"].tolist(), what
    return 1


def _lm_verify_stage(ctx, wl, ver, n_search, B, params, what):
    """The verify-side LM head on the oracle's own mask-view rows (the
    verify forward's layout) against the oracle's acceptance from them."""
    torch = H.torch_mod()
    MS = params["max_search"]
    mr = ver["mask_rows"]
    hv = np.zeros((B * MS, ver["final"].shape[1]))
    hv[mr >= 0] = ver["final"][mr[mr >= 0]]
    dtok = np.where(ver["draft_tok"] >= 0, ver["draft_tok"], 0)
    acc = torch.empty(B * MS, dtype=torch.uint8, device="cuda")
    nacc = torch.empty(B, dtype=torch.int32, device="cuda")
    mconf = torch.empty(B * MS, dtype=torch.float32, device="cuda")
    marg = torch.empty(B * MS, dtype=torch.int32, device="cuda")
    ctx.lm_head_verify(H.dev(synth.make_tensor(hv, "bf16")), wl, B, MS, n_search=H.ints(n_search),
                       draft_tok=H.ints(dtok), gamma=params["gamma"], accept=acc, n_accept=nacc, mask_conf=mconf,
                       mask_argmax=marg)
    ctx.sync_status()
    mconf, marg, acc, nacc = H.host(mconf), H.host(marg), H.host(acc), H.host(nacc)
    valid = np.array([b * MS + j for b in range(B) for j in range(int(n_search[b]))])
    H.assert_close(mconf[valid], ver["mask_conf"][valid], "f32", f"mask-view confidences on the oracle's rows, {what}")
    gap = _top2_gap(ver["mask_logits"][valid])
    if (gap < 1e-3).any() or (np.abs(ver["mask_conf"][valid] - np.float64(np.float32(params["gamma"]))) < 1e-5).any():
        a, n = _verify_rule(mconf, marg, ver["draft_tok"], n_search, params["gamma"], B, MS)
        assert nacc.tolist() == n.tolist(), what
        return 0
    assert marg[valid].tolist() == ver["mask_argmax"][valid].tolist(), what
    assert nacc.tolist() == ver["n_accept"].tolist(), what
    assert acc[valid].tolist() == ver["accept"][valid].tolist(), what
    return 1


def _top2_gap(logits):
    """Gap between the two largest float64 logits of each row."""
    top = np.sort(logits, axis=1)[:, -2:]
    return top[:, 1] - top[:, 0]


def _rows_close(gpu, ref, what):
    """The final rows element by element, with the whole-model forward's
    rule: bf16 of unit-RMS values that passed through every layer, so where
    an fp32 and a float64 rounding upstream put a value across a rounding
    boundary two bf16 ulps are allowed where an ulp exceeds the bf16
    tolerance."""
    gpu = np.asarray(gpu, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    allowed = np.maximum(H.BF16_TOL, 2.0 * H.bf16_ulp(ref))
    bad = err > allowed
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} elements out of tolerance, worst error "
                           f"{err.max():.3e} ({(err / np.maximum(H.bf16_ulp(ref), 1e-30)).max():.1f} ulps)")

