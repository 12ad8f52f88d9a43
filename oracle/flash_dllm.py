"""float64 reference of every step of the Flash-dLLM layer-step hot path.

Test infrastructure only (see the package docstring). Plain definitions,
written for a reader to check against the pages by eye; no blocking, fusion
or reordering beyond what each definition states.
"""
from __future__ import annotations

import math

import numpy as np

KIND_NORMAL = 0
KIND_WINDOW = 1


# ---------------------------------------------------------------------------
# Storage rounding
# ---------------------------------------------------------------------------
def store_round(x: np.ndarray, dtype: str) -> np.ndarray:
    """Value a float64 result takes once stored in ``dtype`` (as float64).

    'bf16': round to nearest, ties to even, at 8 significant bits (directly
    from float64, no intermediate float32). 'f32': IEEE single rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype != "bf16":
        raise ValueError(dtype)
    m, e = np.frexp(x)                 # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


# ---------------------------------------------------------------------------
# Step a1: cache slots and the scheduled work list
# ---------------------------------------------------------------------------
def slot_of(block_table: np.ndarray, page_size: int, b: int, c: int) -> int:
    """Cache slot of sequence b's position c.

    [FD "Core method"]: Flash-Cache writes K/V into a preallocated flat cache
    and block-table scheduling aligns query blocks with their KV blocks. The
    flat per-layer cache of [FD "Method steps", Algorithm 2 step 1] is
    (B * N_max) x d_model; with one page per sequence of N_max slots and an
    identity table, slot = b * N_max + c.
    """
    page = int(block_table[b, c // page_size])
    if page < 0:
        raise IndexError(f"unmapped page for b={b} c={c}")
    return page * page_size + c % page_size


def slot_map(row_seq, row_cache_pos, block_table, page_size) -> np.ndarray:
    """Slot each query row's K/V is written to (-1 where cache_pos < 0)."""
    out = np.full(len(row_seq), -1, dtype=np.int64)
    for r, (b, c) in enumerate(zip(row_seq, row_cache_pos)):
        if c >= 0:
            out[r] = slot_of(block_table, page_size, int(b), int(c))
    return out


def work_list(cu_seqlens, n_keys, tile_m: int) -> np.ndarray:
    """Scheduled attention work items (b, q_start, q_len, n_keys_b).

    [FD "Core method"]: ragged query blocks of every sequence (a small window
    in cache phase, the whole sequence in refresh phase) are laid out as
    blocks with no padding. Items run over sequences in order and, within a
    sequence, over consecutive tiles of at most ``tile_m`` query rows.
    """
    items = []
    for b in range(len(cu_seqlens) - 1):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        start = lo
        while start < hi:
            q_len = min(tile_m, hi - start)
            items.append((b, start, q_len, int(n_keys[b])))
            start += q_len
    return np.asarray(items, dtype=np.int32).reshape(-1, 4)


# ---------------------------------------------------------------------------
# Step a2: fused QKV projection + RoPE + cache write
# ---------------------------------------------------------------------------
def project_qkv(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """[q | k | v] = X W^T, W stored [3 d_model, d_model] (Q rows, K rows, V rows).

    [FD "Core method"]: the QKV projection of the refresh rows, with no bias
    (LLaDA is a LLaMA-style model).
    """
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing, per head.

    x: [R, H, hd]; pos: [R] absolute positions. For i < hd/2 the pair
    (x_i, x_{i+hd/2}) is rotated by angle pos * theta^(-2i/hd):
        x_i'        = x_i cos(a) - x_{i+hd/2} sin(a)
        x_{i+hd/2}' = x_i sin(a) + x_{i+hd/2} cos(a)
    The pages name RoPE without fixing a convention ([FD "Background"],
    [FD "Core method"]); this is the LLaMA/LLaDA convention.
    """
    x = np.asarray(x, np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, np.float64)[:, None] * inv_freq[None, :]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * cos - b * sin, a * sin + b * cos], axis=-1)


def qkv_rope_cache_write(x, w, n_heads, head_dim, theta, row_rope_pos,
                         row_seq, row_cache_pos, block_table, page_size,
                         k_cache, v_cache, dtype):
    """Flash-Cache fused step for one layer.

    [FD "Core method"], [FA "Flash-Cache"]: project the refresh rows to
    Q, K, V, apply RoPE to Q and K, and write K and V straight into their
    cache slots; Q is returned for the attention that follows. Stored
    tensors (Q buffer, cache) take ``dtype``'s rounding.

    Returns (q [R, H, hd], k_cache', v_cache') as float64 arrays (copies).
    """
    d = n_heads * head_dim
    y = project_qkv(x, w)
    R = y.shape[0]
    q = rope(y[:, :d].reshape(R, n_heads, head_dim), row_rope_pos, theta)
    k = rope(y[:, d:2 * d].reshape(R, n_heads, head_dim), row_rope_pos, theta)
    v = y[:, 2 * d:].reshape(R, n_heads, head_dim)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    slots = slot_map(row_seq, row_cache_pos, block_table, page_size)
    for r in range(R):
        if slots[r] >= 0:
            kc[slots[r]] = store_round(k[r].reshape(d), dtype)
            vc[slots[r]] = store_round(v[r].reshape(d), dtype)
    return store_round(q, dtype), kc, vc


# ---------------------------------------------------------------------------
# Steps a3 + a8: scheduled attention with the two-view visibility rule
# ---------------------------------------------------------------------------
def visible_positions(kind: int, kv_len: int, search_pos) -> list:
    """Key list a query row of ``kind`` sees, as (label, position) pairs.

    Labels: 'base' for cache positions 0..kv_len-1, ('draft', j) / ('mask', j)
    for the two view keys of the j-th search token (0-based).

    [FD "Core method"] and [FD "Method steps", step 3]: each search query is
    duplicated into a draft view (holding the draft token) and a mask view
    (holding [MASK]); the two are isolated by a causal mask and share the
    tracked context. [FA "Flash-Verify"]: the mask view must not see the
    draft at its own position but may use earlier drafts. Reading (search
    tokens s_1..s_m in acceptance order, 0-based j here):
      * normal and masked-window rows see all base keys;
      * view rows do not see the base keys at search positions; instead
        draft view k sees draft keys j <= k and mask keys j > k,
        mask view k sees draft keys j < k and mask keys j >= k,
      so each view row sees every position exactly once.
    """
    search_pos = [int(s) for s in search_pos]
    if kind in (KIND_NORMAL, KIND_WINDOW):
        return [("base", c) for c in range(kv_len)]
    k = (kind - 2) // 2
    is_mask_view = (kind - 2) % 2 == 1
    m = len(search_pos)
    if k >= m:
        raise ValueError("view row for a search token that does not exist")
    hidden = set(search_pos)
    keys = [("base", c) for c in range(kv_len) if c not in hidden]
    for j in range(m):
        sees_draft = (j < k) or (j == k and not is_mask_view)
        keys.append((("draft", j) if sees_draft else ("mask", j), search_pos[j]))
    return keys


def visible_keys(kind: int, kv_len: int, search_pos) -> np.ndarray:
    """Cache positions of the keys ``visible_positions`` lists.

    Base key c sits at cache position c; the j-th draft-view key at
    kv_len + j and the j-th mask-view key at kv_len + m + j.
    """
    m = len(search_pos)
    out = []
    for label, c in visible_positions(kind, kv_len, search_pos):
        if label == "base":
            out.append(c)
        elif label[0] == "draft":
            out.append(kv_len + label[1])
        else:
            out.append(kv_len + m + label[1])
    return np.asarray(out, dtype=np.int64)


def sched_attn(q, k_cache, v_cache, block_table, page_size, cu_seqlens, kv_len,
               row_kind, search_pos=None, n_search=None, max_seq=None, dtype="f32"):
    """Exact attention of every query row over its visible cached keys.

    [FD "Background"] Flash Attention computes exact softmax(Q K^T / sqrt(d)) V
    without materialising the score matrix; [FD "Core method"] the scheduled
    kernel attends each sequence's ragged query block to its full cache.
    Per row r and head h: s = q . k / sqrt(hd) over the visible keys,
    p = softmax(s), o = sum p v, LSE = log sum exp(s).

    Tracker increment, [FD "Method steps", step 4, Eq. (2)]:
        a_b[i] += (1/H) sum_h (1/|M_b|) sum_{j in M_b} p_{h,j,i}
    over the masked-window rows j (kind 1) of sequence b, for base keys i.
    The caller sums the returned increments over layers.

    Returns (o [R,H,hd] rounded to ``dtype``, lse [R,H] float64,
    track [B, max_seq] float64).
    """
    q = np.asarray(q, np.float64)
    R, H, hd = q.shape
    B = len(cu_seqlens) - 1
    scale = 1.0 / math.sqrt(hd)
    o = np.zeros((R, H, hd))
    lse = np.full((R, H), -np.inf)
    if max_seq is None:
        max_seq = int(max(kv_len)) if B else 0
    track = np.zeros((B, max_seq))
    for b in range(B):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        n_kv = int(kv_len[b])
        m_b = int(n_search[b]) if search_pos is not None else 0
        sp = [] if search_pos is None else [int(s) for s in search_pos[b][:m_b]]
        kinds = [int(row_kind[r]) for r in range(lo, hi)]
        n_masked = sum(1 for k in kinds if k == KIND_WINDOW)
        groups: dict = {}
        for r, kind in zip(range(lo, hi), kinds):
            key = "plain" if kind in (KIND_NORMAL, KIND_WINDOW) else kind
            groups.setdefault(key, []).append(r)
        for key, rows in groups.items():
            kind = KIND_NORMAL if key == "plain" else key
            pos = visible_keys(kind, n_kv, sp)
            if len(pos) == 0:
                continue
            slots = np.array([slot_of(block_table, page_size, b, int(c)) for c in pos])
            K = np.asarray(k_cache, np.float64)[slots].reshape(len(pos), H, hd)
            V = np.asarray(v_cache, np.float64)[slots].reshape(len(pos), H, hd)
            rows = np.asarray(rows)
            # s[h, r, n] = q[r, h, :] . K[n, h, :] / sqrt(hd)
            s = np.matmul(q[rows].transpose(1, 0, 2), K.transpose(1, 2, 0)) * scale
            mx = s.max(axis=-1, keepdims=True)
            e = np.exp(s - mx)
            l = e.sum(axis=-1, keepdims=True)
            p = e / l
            # o[r, h, :] = sum_n p[h, r, n] V[n, h, :]
            o[rows] = np.matmul(p, V.transpose(1, 0, 2)).transpose(1, 0, 2)
            lse[rows] = (mx + np.log(l))[..., 0].T
            if key == "plain" and n_masked:
                sel = np.array([kinds[r - lo] == KIND_WINDOW for r in rows])
                contrib = p[:, sel, :].sum(axis=(0, 1)) / (H * n_masked)
                track[b, pos] += contrib
    return store_round(o, dtype), lse, track


# ---------------------------------------------------------------------------
# Step a5: top-k of the tracker scores
# ---------------------------------------------------------------------------
def track_topk(scores, eligible, seq_len, k: int):
    """Next step's tracked set from the attention-mass scores.

    [FD "Method steps", step 4]: take the top-k decoded tokens by a_i (the
    newly decoded ones join separately). Candidates are the positions the
    ``eligible`` mask allows among 0..seq_len-1; order is score descending,
    then position ascending.

    Returns (idx [B, k] with -1 padding, cnt [B]).
    """
    scores = np.asarray(scores)
    B = scores.shape[0]
    idx = np.full((B, k), -1, dtype=np.int32)
    cnt = np.zeros(B, dtype=np.int32)
    for b in range(B):
        cand = [i for i in range(int(seq_len[b])) if eligible[b][i]]
        cand.sort(key=lambda i: (-float(scores[b][i]), i))
        top = cand[:k]
        idx[b, :len(top)] = top
        cnt[b] = len(top)
    return idx, cnt


# ---------------------------------------------------------------------------
# Steps a6 + a7: confidence-aware unmasking and Flash-Verify acceptance
# ---------------------------------------------------------------------------
def row_confidence(logits: np.ndarray):
    """Per row: c = max_x p(x) = 1 / sum_v exp(l_v - max l), and the argmax.

    [FD "Background"] (confidence-aware parallel decoding) and [FD "Method
    steps", step 2]: c_i = max_x p(x_i | x^t). The argmax is the lowest
    vocabulary id attaining the maximum logit.
    """
    l = np.asarray(logits, np.float64)
    mx = l.max(axis=1)
    arg = np.argmax(l, axis=1).astype(np.int32)   # first occurrence
    z = np.exp(l - mx[:, None]).sum(axis=1)
    return 1.0 / z, arg


def unmask(logits, row_seq, row_pos, B: int, eps: float, force_progress: bool,
           max_search: int):
    """Draft-step decisions for the masked-window rows.

    [FD "Method steps", step 2]: positions with c_i >= eps are decoded
    (D^t); the others form the search set S^t. [FAST "Confidence-aware
    parallel decoding"]: if no position reaches the threshold, the single
    most confident one is decoded (``force_progress``). The search list of
    each sequence is its uncommitted rows ordered by confidence descending
    (position ascending on ties), capped at ``max_search``; this order is
    also the verify forward's acceptance order ([FA "Flash-Verify"]).

    Returns dict(conf, argmax, commit, search_rows [B, max_search] (-1
    padded, indices into the window rows), n_search [B]).
    """
    conf, arg = row_confidence(logits)
    Rw = len(conf)
    commit = (conf >= eps).astype(np.uint8)
    search = np.full((B, max_search), -1, dtype=np.int32)
    n_search = np.zeros(B, dtype=np.int32)
    for b in range(B):
        rows = [r for r in range(Rw) if int(row_seq[r]) == b]
        if force_progress and rows and not any(commit[r] for r in rows):
            best = min(rows, key=lambda r: (-conf[r], int(row_pos[r])))
            commit[best] = 1
        unc = [r for r in rows if not commit[r]]
        unc.sort(key=lambda r: (-conf[r], int(row_pos[r])))
        unc = unc[:max_search]
        search[b, :len(unc)] = unc
        n_search[b] = len(unc)
    return dict(conf=conf, argmax=arg, commit=commit, search_rows=search, n_search=n_search)


def lm_head_logits(hidden, w_lm, chunk: int = 4096) -> np.ndarray:
    """Window rows' logits over the vocabulary: l = h W_lm^T.

    [FD "Method steps", step 2] takes c_i = max_x p(x_i | x^t) from the
    model's output distribution over the vocabulary; p is the softmax of the
    language-model head applied to the final hidden state of each masked
    position. Reading: the head is a plain linear map [vocab, d_model] with
    no bias (the LLaMA-style output layer of LLaDA), applied to the
    already-normalised hidden state. float64 from the exactly widened
    inputs, computed in vocabulary chunks only to bound memory.
    """
    h = np.asarray(hidden, np.float64)
    V = w_lm.shape[0]
    out = np.empty((h.shape[0], V))
    for v0 in range(0, V, chunk):
        out[:, v0:v0 + chunk] = h @ np.asarray(w_lm[v0:v0 + chunk], np.float64).T
    return out


def lm_head_unmask(hidden, w_lm, row_seq, row_pos, B: int, eps: float, force_progress: bool,
                   max_search: int):
    """Draft-step decisions straight from the hidden states: ``unmask`` of
    ``lm_head_logits``, the composition the fused kernel computes without
    storing the logits ([FD "Method steps", step 2])."""
    return unmask(lm_head_logits(hidden, w_lm), row_seq, row_pos, B, eps, force_progress, max_search)


def lm_head_verify(mask_hidden, w_lm, draft_tok, n_search, gamma: float, B: int, max_search: int):
    """Verify-step acceptance straight from the mask views' hidden states:
    ``verify`` of ``lm_head_logits`` ([FD "Method steps", step 3]: the mask
    view's x_tilde and c_tilde come from the model's output distribution at
    that view, the softmax of the same linear head as in step 2)."""
    return verify(lm_head_logits(mask_hidden, w_lm), draft_tok, n_search, gamma, B, max_search)


def verify(mask_logits, draft_tok, n_search, gamma: float, B: int, max_search: int):
    """Flash-Verify prefix acceptance.

    [FD "Method steps", step 3]: walking the search tokens in order, accept
    token k while its draft x_hat equals the mask view's argmax x_tilde and
    the mask view's confidence c_tilde >= gamma; stop at the first token
    that fails. Row b*max_search + j of ``mask_logits`` / ``draft_tok`` is
    sequence b's j-th search token; rows j >= n_search[b] are ignored.

    Returns dict(mask_conf, mask_argmax, accept [B*max_search], n_accept [B]).
    """
    conf, arg = row_confidence(mask_logits)
    accept = np.zeros(B * max_search, dtype=np.uint8)
    n_accept = np.zeros(B, dtype=np.int32)
    for b in range(B):
        for j in range(int(n_search[b])):
            r = b * max_search + j
            if int(draft_tok[r]) == int(arg[r]) and conf[r] >= gamma:
                accept[r] = 1
                n_accept[b] += 1
            else:
                break
    return dict(mask_conf=conf, mask_argmax=arg, accept=accept, n_accept=n_accept)


def tv_point_mass(p: np.ndarray, x: int) -> float:
    """Total-variation distance between the point mass on x and distribution p.

    TV(delta_x, p) = 1/2 sum_y |delta_x(y) - p(y)|. [FD "Core method"],
    Theorem 1: for an accepted token this equals 1 - c_tilde <= 1 - gamma.
    """
    p = np.asarray(p, np.float64)
    d = -p.copy()
    d[x] += 1.0
    return 0.5 * float(np.abs(d).sum())
