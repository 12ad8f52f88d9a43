"""Pins of the Flash-dLLM step oracle (oracle/flash_loop.py), on the CPU, with
a tiny random-weight model: closed-form step counts of whole decodes at the
two extremes of eps, and the invariants every step must keep."""
import math

import numpy as np
import pytest

from oracle import flash_loop as fl
import synth

D, H, V = 64, 2, 50


def _setup(prompts, gens, window=4, budget=4, max_search=2, eps=0.9, gamma=0.5, force=True, seed=11):
    # W_o, W_down and the LM head scaled up so that the window rows' confidences
    # spread over (0.1, 0.9): some commit, some are searched, some verified
    mc = synth.model_case(seed=seed, d=D, n_heads=H, n_layers=2, ffn=96, vocab=V, out_std=1.0, lm_std=0.5)
    m = synth.model_values(mc)
    w_lm = m["w_lm"]
    B = len(prompts)
    lengths = np.array(prompts) + np.array(gens)
    max_seq, max_views = int(lengths.max()), 2 * max_search
    geom = synth.flat_geometry(B, max_seq + max_views)
    rng = np.random.default_rng(seed)
    tokens = np.full((B, max_seq), mc["mask_id"], np.int64)
    masked = np.zeros((B, max_seq), np.uint8)
    for b in range(B):
        tokens[b, :prompts[b]] = rng.integers(0, V - 1, prompts[b])
        masked[b, prompts[b]:lengths[b]] = 1
    seqs = dict(prompt_len=np.array(prompts, np.int32), seq_len=lengths.astype(np.int32), tokens=tokens,
                masked=masked, tracked=[[] for _ in range(B)], state=np.full(B, -1, np.int32))
    n_slots = geom.n_pages * geom.page_size
    caches = ([np.zeros((n_slots, D)) for _ in range(2)], [np.zeros((n_slots, D)) for _ in range(2)])
    params = dict(window=window, track_budget=budget, max_search=max_search, eps=eps, gamma=gamma,
                  force_progress=force, mask_id=mc["mask_id"], max_views=max_views)
    return m, w_lm, seqs, params, caches, geom


def _decode(prompts, gens, **kw):
    m, w_lm, seqs, params, caches, geom = _setup(prompts, gens, **kw)
    steps, traces = 0, []
    while seqs["masked"].any():
        seqs, caches, tr = fl.flash_step(m, w_lm, seqs, params, caches, geom, dtype="f32")
        traces.append((tr, seqs))
        steps += 1
        assert steps <= 200
    return steps, seqs, traces, params


def test_eps_zero_decodes_a_whole_window_per_step():
    # every window row commits: ceil(gen / window) steps, no search, no verify
    steps, seqs, traces, _ = _decode([5, 8], [12, 21], eps=0.0)
    assert steps == max(math.ceil(12 / 4), math.ceil(21 / 4))
    for tr, _ in traces:
        assert tr["verify"] is None
    assert not seqs["masked"].any() and (seqs["tokens"][0, :17] != V - 1).all()


def test_eps_one_with_forced_progress_decodes_one_token_per_step():
    # nothing reaches eps = 1 and there is no search list: one forced token per step
    steps, seqs, traces, _ = _decode([5, 8], [7, 10], eps=1.0, max_search=0)
    assert steps == 10
    for t, (tr, _) in enumerate(traces):
        assert [len(n) for n in tr["new"]] == [1 if t < 7 else 0, 1]


def test_every_step_keeps_its_invariants():
    steps, seqs, traces, params = _decode([6, 9], [16, 12], eps=0.5, gamma=0.2, seed=12)
    first = traces[0][0]
    assert first["draft_pos"].tolist() == list(range(22)) + list(range(21))   # the full first forward
    saw_accept = False
    for tr, after in traces:
        dec = tr["unmask"]
        for b in range(2):
            w = tr["window_pos"][tr["window_seq"] == b]
            new = tr["new"][b]
            assert set(new) <= set(w.tolist())                  # only window positions are decoded
            assert len(new) == len(set(new))
            assert 1 <= len(new) or len(w) == 0                   # forced progress
            if tr["verify"] is not None:
                n_acc = int(tr["verify"]["n_accept"][b])
                saw_accept |= n_acc > 0
                acc = tr["verify"]["accept"][b * 2:(b + 1) * 2].tolist()
                assert acc == [1] * n_acc + [0] * (2 - n_acc)     # a prefix
            tracked = after["tracked"][b]
            assert len(tracked) <= params["track_budget"]
            assert tracked[:len(new)] == new[:params["track_budget"]]   # new ones first
            assert not after["masked"][b, tracked].any()
            assert len(set(tracked)) == len(tracked)
            # the rest: the best decoded positions by tracker score (brute-force sort)
            n = int(after["seq_len"][b])
            elig = [p for p in range(n) if not after["masked"][b, p] and p not in new]
            order = sorted(elig, key=lambda p: (-float(np.float32(tr["track"][b, p])), p))
            rest = tracked[len(new):]
            assert rest == order[:len(rest)]
            assert len(rest) == min(max(0, params["track_budget"] - len(new)), len(elig))
    assert saw_accept
    assert steps < 28
