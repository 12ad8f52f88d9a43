"""float64 reference of one Flash-dLLM denoising step (Algorithm 2 steps 2-4)
of a whole model, on the host state of a batch of sequences.

Test infrastructure only (see the package docstring).

Paper digest, "Method steps in detail", Algorithm 2:
  step 1  the prompt followed by masks gets one full forward that fills every
          layer's cache;
  step 2  each step's query is the tracked set T^t plus the sliding masked
          window; for each window position c_i = max_x p(x_i | x^t); positions
          with c_i >= eps are decoded (D^t), the rest form the search set S^t;
  step 3  the verify forward runs the shrunk tracked set T_v and, for each
          search token, a draft view (holding its draft prediction) and a mask
          view (holding [MASK]) under the view mask; walking S^t in order,
          a token is accepted while its draft equals the mask view's argmax and
          the mask view's confidence is >= gamma; the walk stops at the first
          failure;
  step 4  the tracker scores of the draft forward (Eq. (2), summed over the
          layers) pick the top-k decoded tokens, which with the newly decoded
          ones form T^{t+1}.

Readings: the step-1 full forward is the first step's draft forward (its rows
are every position, the window rows among them are decided like any other
step's); the Fast-dLLM fallback commits a sequence's most confident window
row when none reaches eps (force_progress); the verify forward runs only when
some sequence has a search token, and writes nothing but its rows' K/V;
|T_v| = max(0, beta_t + beta_m - 2|S|) taken from the front of the tracked
set; the newly decoded tokens (committed, then accepted, in position order)
come first in T^{t+1}, then the top-(beta_t - |new|) of the other decoded
positions (the prompt included) by tracker score.

Parity: pinned by tests/test_flash_loop_pins.py (closed-form step counts of
whole decodes at the two extremes of eps, invariants of every step).
"""
from __future__ import annotations

import numpy as np

from . import refresh as rf
from .flash_dllm import KIND_WINDOW, lm_head_logits, track_topk, unmask, verify
from .model import model_forward


def flash_step(model: dict, w_lm, seqs: dict, params: dict, caches, geom, dtype: str = "bf16", force=None):
    """One step on ``seqs`` (dict: prompt_len, seq_len, tokens [B, max_seq],
    masked [B, max_seq], tracked (list of lists), state [B]); ``caches`` is
    (k_caches, v_caches) per layer. ``params``: window, track_budget,
    max_search, eps, gamma, force_progress, mask_id, max_views.

    ``force`` (optional) replaces this oracle's own decisions with given ones
    so that a step can follow another implementation's path: keys 'argmax'
    (the draft tokens) and 'commit' [R_w], 'search_rows' [B, max_search],
    'n_search' [B], 'n_accept' [B].

    Returns (new seqs, new caches, trace dict).
    """
    B = len(seqs["prompt_len"])
    max_seq = seqs["tokens"].shape[1]
    tokens, masked = seqs["tokens"].copy(), seqs["masked"].copy()
    state = np.asarray(seqs["state"]).copy()
    kcs, vcs = caches
    ms, win, budget = params["max_search"], params["window"], params["track_budget"]
    trace = {}

    # ---- step 2: the draft forward over the tracked set and the window
    per_seq = []
    for b in range(B):
        rows_b, state[b] = rf.refresh_rows(rf.FLASH_DRAFT, masked[b], int(seqs["prompt_len"][b]),
                                           int(seqs["seq_len"][b]), win, int(state[b]), seqs["tracked"][b])
        per_seq.append(rows_b)
    row_seq = np.array([b for b in range(B) for _ in per_seq[b]], np.int32)
    row_pos = np.array([p for rb in per_seq for p, _ in rb], np.int32)
    row_kind = np.array([k for rb in per_seq for _, k in rb], np.int32)
    cu = np.concatenate([[0], np.cumsum([len(rb) for rb in per_seq])]).astype(np.int32)
    trace["draft_pos"], trace["draft_cu"] = row_pos, cu
    if len(row_pos) == 0:
        return dict(seqs, state=state), caches, trace
    row_tok = tokens[row_seq, row_pos]
    final, kcs, vcs, track = model_forward(model, row_tok, row_seq, row_pos, row_pos, row_kind, cu,
                                           seqs["seq_len"], geom.block_table, geom.page_size, kcs, vcs, dtype,
                                           max_seq=max_seq, track=True)
    trace["draft_final"], trace["track"] = final, track
    wsel = np.nonzero(row_kind == KIND_WINDOW)[0]
    w_seq, w_pos = row_seq[wsel], row_pos[wsel]
    logits = lm_head_logits(final[wsel], w_lm)
    dec = unmask(logits, w_seq, w_pos, B, params["eps"], bool(params["force_progress"]), ms)
    trace["window_pos"], trace["window_seq"], trace["unmask"] = w_pos, w_seq, dec
    trace["window_rows"], trace["window_logits"] = wsel, logits
    commit = dec["commit"] if force is None else np.asarray(force["commit"])
    search_rows = dec["search_rows"] if force is None else np.asarray(force["search_rows"])
    n_search = dec["n_search"] if force is None else np.asarray(force["n_search"])
    draft_tok = np.asarray(dec["argmax"] if force is None else force["argmax"], np.int64)

    committed = [[] for _ in range(B)]
    for r in np.nonzero(commit)[0]:
        committed[int(w_seq[r])].append((int(w_pos[r]), int(draft_tok[r])))
    search = [[int(search_rows[b, j]) for j in range(int(n_search[b]))] for b in range(B)]

    # ---- step 3: the verify forward and the acceptance walk
    accepted = [[] for _ in range(B)]
    trace["verify"] = None
    if any(len(s) for s in search):
        per_seq = []
        s_pos = np.full((B, ms), -1, np.int32)
        for b in range(B):
            sp = [int(w_pos[r]) for r in search[b]]
            s_pos[b, :len(sp)] = sp
            per_seq.append(rf.verify_rows(seqs["tracked"][b], sp, int(seqs["seq_len"][b]), budget + win))
        v_seq = np.array([b for b in range(B) for _ in per_seq[b]], np.int32)
        v_rope = np.array([r[0] for rb in per_seq for r in rb], np.int32)
        v_cache = np.array([r[1] for rb in per_seq for r in rb], np.int32)
        v_kind = np.array([r[2] for rb in per_seq for r in rb], np.int32)
        v_cu = np.concatenate([[0], np.cumsum([len(rb) for rb in per_seq])]).astype(np.int32)
        v_tok = np.empty(len(v_seq), np.int64)
        mask_rows = np.full(B * ms, -1, np.int64)
        for i in range(len(v_seq)):
            b, k = int(v_seq[i]), int(v_kind[i])
            if k < 2:
                v_tok[i] = tokens[b, v_rope[i]]
            elif k % 2 == 0:                         # draft view j: its draft prediction
                v_tok[i] = draft_tok[search[b][(k - 2) // 2]]
            else:                                    # mask view j: [MASK]
                v_tok[i] = params["mask_id"]
                mask_rows[b * ms + (k - 3) // 2] = i
        final_v, kcs, vcs, _ = model_forward(model, v_tok, v_seq, v_rope, v_cache, v_kind, v_cu,
                                             seqs["seq_len"], geom.block_table, geom.page_size, kcs, vcs, dtype,
                                             search_pos=s_pos, n_search=np.array([len(s) for s in search]),
                                             max_seq=max_seq + params["max_views"])
        hv = np.zeros((B * ms, final_v.shape[1]))
        ok = mask_rows >= 0
        hv[ok] = final_v[mask_rows[ok]]
        dtok = np.full(B * ms, -1, np.int64)
        for b in range(B):
            for j, r in enumerate(search[b]):
                dtok[b * ms + j] = draft_tok[r]
        mask_logits = lm_head_logits(hv, w_lm)
        ver = verify(mask_logits, dtok, np.array([len(s) for s in search]), params["gamma"], B, ms)
        trace["verify"] = dict(ver, s_pos=s_pos, draft_tok=dtok, final=final_v, mask_rows=mask_rows,
                               mask_logits=mask_logits)
        n_acc = ver["n_accept"] if force is None else np.asarray(force["n_accept"])
        for b in range(B):
            accepted[b] = [(int(w_pos[r]), int(draft_tok[r])) for r in search[b][:int(n_acc[b])]]

    # ---- step 4: decode, then the next tracked set
    new = []
    for b in range(B):
        nb = sorted(committed[b]) + sorted(accepted[b])
        for p, t in nb:
            tokens[b, p] = t
            masked[b, p] = 0
        new.append([p for p, _ in nb])
    eligible = np.zeros((B, max_seq), np.uint8)
    for b in range(B):
        n = int(seqs["seq_len"][b])
        eligible[b, :n] = 1 - masked[b, :n]
        eligible[b, new[b]] = 0
    idx, cnt = track_topk(track.astype(np.float32), eligible, seqs["seq_len"], budget)
    tracked = []
    for b in range(B):
        keep = max(0, budget - len(new[b]))
        tracked.append(new[b][:budget] + [int(i) for i in idx[b, :min(keep, int(cnt[b]))]])
    trace["new"], trace["eligible"], trace["topk"] = new, eligible, (idx, cnt)
    return dict(seqs, tokens=tokens, masked=masked, state=state, tracked=tracked), (kcs, vcs), trace
