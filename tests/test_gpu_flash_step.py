"""Whole Flash-dLLM denoising steps on the GPU (fdl_flash_step: the draft
forward through every layer, the fused LM-head unmasking, the verify forward
with its two views per search token, the acceptance walk, the next tracked
set) against the float64 step oracle, by teacher forcing.

Each step starts the oracle from the GPU's own state (tokens, masks, tracked
set and the caches, downloaded before the step) and forces it to follow the
GPU's decisions. Compared: the row sets (exact), the window rows' and mask
views' confidences and predictions (tolerance, and exact argmax where the
top two logits are apart), the tracker scores, the caches after the step;
the GPU's decisions must be exactly the decision rules applied to its own
confidences, and its next state exactly what those decisions give."""
import numpy as np
import pytest

import oracle
from oracle import flash_loop as fl
import synth
from tests import _harness as H
from tests.test_gpu_lm_head import _decide, _verify_rule

pytestmark = pytest.mark.gpu


def test_flash_steps_teacher_forced():
    torch = H.torch_mod()
    import kv_cache_attention_gb300 as fdl
    mc = synth.model_case(seed=1015, d=512, n_heads=4, n_layers=2, ffn=1024, vocab=2088, out_std=0.5, lm_std=0.2)
    m = synth.model_values(mc)
    w_lm = m["w_lm"]
    L, d, V = len(mc["layers"]), mc["d_model"], mc["vocab"]
    prompts, gens = [20, 27], [32, 24]
    B = 2
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
    saw = dict(commit=0, search=0, accept=0, verify_steps=0)
    for step in range(40):
        if not seqs["masked"].any():
            break
        snap = {k: v.copy() for k, v in seqs.items()}
        snap_tracked = [snap["tracked"][b, :snap["n_tracked"][b]].tolist() for b in range(B)]
        caches = ([H.host(t).astype(np.float64) for t in kcs], [H.host(t).astype(np.float64) for t in vcs])
        rec = ctx.flash_step(dm, wl, kcs, vcs, bt, params, seqs, ws)
        RW = int(rec["n_window"][0])
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
        # the draft forward's final rows, then the window rows' confidences and
        # predictions (the logits have a standard deviation near 4.5 here, so a
        # relative difference r in a hidden row moves a logit by about 4.5 r)
        _rows_close(rec["draft_final"], tr["draft_final"], f"draft rows, step {step}")
        dec = tr["unmask"]
        np.testing.assert_allclose(rec["conf"][:RW], dec["conf"], atol=1e-2, rtol=5e-2)
        clear = _top2_gap(tr["window_logits"]) > 0.2
        assert np.array_equal(rec["argmax"][:RW][clear], dec["argmax"][clear])
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
            valid = np.array([b * MS + j for b in range(B) for j in range(int(rec["n_search"][b]))])
            np.testing.assert_allclose(rec["mask_conf"][valid], ver["mask_conf"][valid], atol=1e-2, rtol=5e-2)
            mgap = _top2_gap(ver["mask_logits"])[valid]
            assert np.array_equal(rec["mask_argmax"][valid][mgap > 0.2], ver["mask_argmax"][valid][mgap > 0.2])
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
    ctx.close()


def _top2_gap(logits):
    """Gap between the two largest float64 logits of each row."""
    top = np.sort(logits, axis=1)[:, -2:]
    return top[:, 1] - top[:, 0]


def _rows_close(gpu, ref, what):
    """Each final row (unit RMS times the gains) within 1e-2 relative RMS of
    the oracle's: bf16 roundings of the intermediates on both sides, carried
    through two layers whose W_o and W_down are large. A row taken from the
    wrong position or sequence would be off by about sqrt(2)."""
    gpu = np.asarray(gpu, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    rel = np.sqrt(((gpu - ref) ** 2).mean(1) / (ref ** 2).mean(1))
    assert (rel < 1e-2).all(), f"{what}: worst row relative RMS difference {rel.max():.3e}"

