"""Seeded synthetic inputs for the Flash-dLLM per-layer denoising-step hot path.

This module is shared by the tests, the benchmark and the oracle's checks. It
holds none of the method's arithmetic: only random draws, the bf16 storage
rounding of those draws, and the layout of the inputs the method consumes
(row descriptors, block tables, eligibility masks). Every array it returns is
a pure function of the seed.

Shapes and value distributions follow the workloads the Flash-dLLM pages
describe (Flash-dLLM digest, "Method steps" paragraph and the reproduction
paragraph: LLaDA-8B layer shape d_model 4096 with 32 heads of 128, block 16-64
masked window, top-32 tracking, vocab 126464, prompts of a few hundred tokens
and generation lengths 256-1024, batch up to 32).

Row kinds (the ``row_kind`` array):
  0            normal query row (tracked / T_v / full-refresh row)
  1            masked-window row (feeds the attention-mass tracker)
  2 + 2*j      draft view of the j-th search token (0-based)
  3 + 2*j      mask view of the j-th search token (0-based)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

KIND_NORMAL = 0
KIND_WINDOW = 1


def kind_draft_view(j: int) -> int:
    return 2 + 2 * j


def kind_mask_view(j: int) -> int:
    return 3 + 2 * j


LLADA_D_MODEL = 4096
LLADA_HEADS = 32
LLADA_HEAD_DIM = 128
LLADA_THETA = 5.0e5
LLADA_VOCAB = 126464


# --------------------------------------------------------------------------
# bf16 storage format (round-to-nearest-even from float32)
# --------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (RNE via float32) and return the uint16 bits."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32)
    # finite inputs only: u + 0x8000 stays below 2^32 for every finite float32
    u = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Tensor:
    """A host array plus its storage dtype ('f32' or 'bf16').

    ``data`` holds float32 values for 'f32' and uint16 bit patterns for 'bf16'.
    ``values()`` returns the exactly-widened float64 view the oracle consumes.
    """

    data: np.ndarray
    dtype: str

    def values(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.data).astype(np.float64)
        return self.data.astype(np.float64)

    @property
    def shape(self):
        return self.data.shape


def make_tensor(x: np.ndarray, dtype: str) -> Tensor:
    if dtype == "bf16":
        return Tensor(to_bf16_bits(x), "bf16")
    return Tensor(np.ascontiguousarray(np.asarray(x, dtype=np.float32)), "f32")


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


# --------------------------------------------------------------------------
# Layer shape and cache geometry
# --------------------------------------------------------------------------
@dataclass
class LayerShape:
    d_model: int
    n_heads: int
    head_dim: int
    rope_theta: float
    dtype: str  # 'f32' or 'bf16'


@dataclass
class CacheGeometry:
    """Paged (or flat) KV-cache layout shared by all layers of a workload.

    Sequence b's cache position c lives in slot
    ``block_table[b, c // page_size] * page_size + c % page_size``.
    With one page per sequence and an identity table this is the flat
    (B * N_max) x d_model layout of the Flash-Cache design.
    """

    page_size: int
    n_pages: int
    block_table: np.ndarray  # int32 [B, pages_per_seq], -1 = unmapped

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])


def flat_geometry(batch: int, slots_per_seq: int) -> CacheGeometry:
    bt = np.arange(batch, dtype=np.int32).reshape(batch, 1)
    return CacheGeometry(page_size=slots_per_seq, n_pages=batch, block_table=bt)


def paged_geometry(rng: np.random.Generator, lengths, page_size: int) -> CacheGeometry:
    """Pages of all sequences randomly permuted in one pool."""
    need = [int(math.ceil(n / page_size)) for n in lengths]
    total = int(sum(need))
    perm = rng.permutation(total).astype(np.int32)
    width = max(need)
    bt = np.full((len(lengths), width), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k:k + n]
        k += n
    return CacheGeometry(page_size=page_size, n_pages=total, block_table=bt)


# --------------------------------------------------------------------------
# Row descriptors
# --------------------------------------------------------------------------
@dataclass
class RowSet:
    """Query rows of one fused-kernel call, grouped by sequence.

    ``cache_pos == -1`` means the row's K/V are not written to the cache.
    """

    row_seq: np.ndarray
    row_rope_pos: np.ndarray
    row_cache_pos: np.ndarray
    row_kind: np.ndarray
    cu_seqlens: np.ndarray  # int32 [B+1]

    @property
    def n_rows(self) -> int:
        return int(self.row_seq.shape[0])


def build_rows(per_seq) -> RowSet:
    """``per_seq[b]`` is a list of (rope_pos, cache_pos, kind) tuples."""
    seq, rp, cp, kd = [], [], [], []
    cu = [0]
    for b, rows in enumerate(per_seq):
        for (p, c, k) in rows:
            seq.append(b)
            rp.append(p)
            cp.append(c)
            kd.append(k)
        cu.append(len(seq))
    a = lambda v: np.asarray(v, dtype=np.int32)
    return RowSet(a(seq), a(rp), a(cp), a(kd), a(cu))


def draft_rows(window_pos, tracked_pos):
    """Draft-forward rows of one sequence: masked window first, then tracked."""
    rows = [(int(p), int(p), KIND_WINDOW) for p in window_pos]
    rows += [(int(p), int(p), KIND_NORMAL) for p in tracked_pos]
    return rows


def verify_rows(tv_pos, search_pos, kv_len):
    """Verify-forward rows of one sequence: T_v, then draft views, then mask views.

    The j-th search token's draft-view key goes to cache position kv_len + j
    and its mask-view key to kv_len + m + j (m = number of search tokens);
    both are rotated at the search token's own position.
    """
    m = len(search_pos)
    rows = [(int(p), int(p), KIND_NORMAL) for p in tv_pos]
    rows += [(int(s), kv_len + j, kind_draft_view(j)) for j, s in enumerate(search_pos)]
    rows += [(int(s), kv_len + m + j, kind_mask_view(j)) for j, s in enumerate(search_pos)]
    return rows


def full_rows(n, window_pos):
    win = set(int(p) for p in window_pos)
    return [(p, p, KIND_WINDOW if p in win else KIND_NORMAL) for p in range(n)]


# --------------------------------------------------------------------------
# Logits recipes
# --------------------------------------------------------------------------
def spiked_logits(rng, rows: int, vocab: int, noise_std: float, spike_lo: float,
                  spike_hi: float) -> tuple[np.ndarray, np.ndarray]:
    """N(0, noise_std^2) logits with one +U(spike_lo, spike_hi) spike per row."""
    x = normal(rng, (rows, vocab), noise_std)
    idx = rng.integers(0, vocab, size=rows)
    x[np.arange(rows), idx] += rng.uniform(spike_lo, spike_hi, size=rows).astype(np.float32)
    return x, idx


def targeted_logits(rng, spike_idx: np.ndarray, target: np.ndarray, vocab: int):
    """N(0,1) logits whose spike height places the max-probability near ``target``.

    For N(0,1) noise the expected partition sum of the non-spike entries is
    vocab * e^{1/2}; a spike of height log(t/(1-t) * vocab * e^{1/2}) makes the
    spike's probability close to t. This is a property of the noise
    distribution, not a computation on the drawn values, so realised
    confidences scatter around the target by a fraction of a percent.
    """
    rows = spike_idx.shape[0]
    x = normal(rng, (rows, vocab), 1.0)
    t = np.asarray(target, dtype=np.float64)
    h = np.log(t / (1.0 - t) * vocab * math.exp(0.5))
    x[np.arange(rows), spike_idx] = h.astype(np.float32)
    return x


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    shape: LayerShape
    batch: int
    seq_len: np.ndarray        # int32 [B]  base positions per sequence (N_b)
    max_seq: int               # N_max
    max_views: int             # view slots per sequence past N_b
    geom: CacheGeometry
    extra: dict = field(default_factory=dict)


def _cache_fill(rng, n_slots: int, d: int, dtype: str) -> tuple[Tensor, Tensor]:
    """Prefilled cache: K/V of a projection of N(0,1) hidden by N(0,0.02) weights."""
    std = 0.02 * math.sqrt(d)
    return (make_tensor(normal(rng, (n_slots, d), std), dtype),
            make_tensor(normal(rng, (n_slots, d), std), dtype))


def tiny_fp32(seed: int = 1001) -> Workload:
    """Tiny single layer, fp32, batch 1 (d_model 256, 4 heads x 64, theta 1e4).

    Prompt 48 + gen 64 tokens, block/window 16 masked positions (48..63),
    8 tracked rows, vocab 1024 logits N(0,3) with one +U(0,8) spike per row.
    Positions 0..47 plus a seeded half of 64..111 count as decoded (eligible
    for the tracker). Also carries a verify phase: mask-view logits are the
    draft logits plus N(0, 0.5^2) noise, so the two views often agree.
    """
    rng = np.random.default_rng(seed)
    shape = LayerShape(256, 4, 64, 1.0e4, "f32")
    d = shape.d_model
    prompt, gen, window, tracked, vocab, max_search = 48, 64, 16, 8, 1024, 8
    n = prompt + gen
    max_views = 2 * max_search
    geom = flat_geometry(1, n + max_views)
    w = make_tensor(normal(rng, (3 * d, d), 0.02), "f32")
    x_init = make_tensor(normal(rng, (n, d)), "f32")
    x_step = make_tensor(normal(rng, (window + tracked, d)), "f32")
    x_verify = make_tensor(normal(rng, (tracked + 2 * max_search, d)), "f32")
    logits, _ = spiked_logits(rng, window, vocab, 3.0, 0.0, 8.0)
    mask_logits = logits + normal(rng, logits.shape, 0.5)
    eligible = np.zeros((1, n), dtype=np.uint8)
    eligible[0, :prompt] = 1
    later = np.arange(prompt + window, n)
    eligible[0, rng.choice(later, size=len(later) // 2, replace=False)] = 1
    kc, vc = _cache_fill(rng, geom.n_pages * geom.page_size, d, "f32")
    return Workload("tiny_fp32", shape, 1, np.array([n], np.int32), n, max_views, geom, dict(
        w=w, x_init=x_init, x_step=x_step, x_verify=x_verify,
        logits=make_tensor(logits, "f32"), mask_logits=make_tensor(mask_logits, "f32"),
        window_pos=np.arange(prompt, prompt + window, dtype=np.int32),
        eligible=eligible, k_cache=kc, v_cache=vc, topk=tracked, vocab=vocab,
        eps=0.9, gamma=0.8, max_search=max_search, force_progress=True,
        prompt=prompt, gen=gen))


def llada_layer(seed: int = 1002) -> Workload:
    """Single LLaDA-8B-shaped layer, bf16, batch 1 (prompt 512 + gen 256).

    Rows: masked window of 32 (positions 512..543) plus 32 tracked positions
    drawn from the prompt. Hidden ~N(0,1), W ~N(0,0.02); 32 logits rows over
    vocab 126464 ~N(0,3) with one +U(0,10) spike.
    """
    rng = np.random.default_rng(seed)
    shape = LayerShape(LLADA_D_MODEL, LLADA_HEADS, LLADA_HEAD_DIM, LLADA_THETA, "bf16")
    d = shape.d_model
    prompt, gen, window, tracked, max_search = 512, 256, 32, 32, 16
    n = prompt + gen
    max_views = 2 * max_search
    geom = flat_geometry(1, n + max_views)
    w = make_tensor(normal(rng, (3 * d, d), 0.02), "bf16")
    window_pos = np.arange(prompt, prompt + window, dtype=np.int32)
    tracked_pos = np.sort(rng.choice(prompt, size=tracked, replace=False)).astype(np.int32)
    rows = build_rows([draft_rows(window_pos, tracked_pos)])
    x = make_tensor(normal(rng, (rows.n_rows, d)), "bf16")
    logits, _ = spiked_logits(rng, window, LLADA_VOCAB, 3.0, 0.0, 10.0)
    kc, vc = _cache_fill(rng, geom.n_pages * geom.page_size, d, "bf16")
    eligible = np.zeros((1, n), dtype=np.uint8)
    eligible[0, :prompt] = 1
    return Workload("llada_layer", shape, 1, np.array([n], np.int32), n, max_views, geom, dict(
        w=w, x=x, rows=rows, logits=make_tensor(logits, "bf16"),
        window_rows=np.arange(window, dtype=np.int32), window_pos=window_pos,
        eligible=eligible, k_cache=kc, v_cache=vc, topk=32, vocab=LLADA_VOCAB,
        eps=0.9, gamma=0.8, max_search=max_search, force_progress=False))


def ragged_batch(seed: int = 1003, batch: int = 16, page_size: int = 64) -> Workload:
    """Ragged batch of 16, bf16, LLaDA layer shape, paged cache (page 64).

    Prompt lengths ~U{128..1024}, gen 512. Even sequences are in cache phase
    (32 window + 32 tracked rows); odd sequences do a full refresh (every
    position is a query row). Pages of all sequences are randomly permuted
    in one pool.
    """
    rng = np.random.default_rng(seed)
    shape = LayerShape(LLADA_D_MODEL, LLADA_HEADS, LLADA_HEAD_DIM, LLADA_THETA, "bf16")
    d = shape.d_model
    gen, window, tracked = 512, 32, 32
    prompts = rng.integers(128, 1025, size=batch)
    lengths = (prompts + gen).astype(np.int32)
    geom = paged_geometry(rng, lengths, page_size)
    w = make_tensor(normal(rng, (3 * d, d), 0.02), "bf16")
    per_seq = []
    for b in range(batch):
        p = int(prompts[b])
        wpos = np.arange(p, p + window)
        if b % 2 == 0:
            tpos = np.sort(rng.choice(p, size=tracked, replace=False))
            per_seq.append(draft_rows(wpos, tpos))
        else:
            per_seq.append(full_rows(int(lengths[b]), wpos))
    rows = build_rows(per_seq)
    x = make_tensor(normal(rng, (rows.n_rows, d)), "bf16")
    kc, vc = _cache_fill(rng, geom.n_pages * geom.page_size, d, "bf16")
    max_seq = int(lengths.max())
    eligible = np.zeros((batch, max_seq), dtype=np.uint8)
    for b in range(batch):
        eligible[b, :int(prompts[b])] = 1
    return Workload("ragged_batch", shape, batch, lengths, max_seq, 0, geom, dict(
        w=w, x=x, rows=rows, k_cache=kc, v_cache=vc, eligible=eligible, topk=32,
        prompts=prompts.astype(np.int32)))


def layer_chain(seed: int = 1004, batch: int = 8, n_layers: int = 32, n_steps: int = 16) -> Workload:
    """32-layer attention path, bf16, batch 8, prompt 256 + gen 512, window 32.

    Per-layer weights and per-(step, layer) hidden inputs are drawn lazily
    from seeds derived from ``seed`` (see ``weight`` / ``hidden``), so a
    caller can materialise only the layers it needs. Step 0 is the full
    init forward over all 768 positions.
    """
    shape = LayerShape(LLADA_D_MODEL, LLADA_HEADS, LLADA_HEAD_DIM, LLADA_THETA, "bf16")
    prompt, gen, window = 256, 512, 32
    n = prompt + gen
    geom = flat_geometry(batch, n)
    eligible = np.zeros((batch, n), dtype=np.uint8)
    eligible[:, :prompt] = 1
    return Workload("layer_chain", shape, batch, np.full(batch, n, np.int32), n, 0, geom, dict(
        seed=seed, n_layers=n_layers, n_steps=n_steps, prompt=prompt, window=window,
        window_pos=np.arange(prompt, prompt + window, dtype=np.int32),
        eligible=eligible, topk=32))


def chain_weight(seed: int, layer: int, d: int) -> Tensor:
    rng = np.random.default_rng([seed, 1, layer])
    return make_tensor(normal(rng, (3 * d, d), 0.02), "bf16")


def chain_hidden(seed: int, step: int, layer: int, rows: int, d: int) -> Tensor:
    rng = np.random.default_rng([seed, 2, step, layer])
    return make_tensor(normal(rng, (rows, d)), "bf16")


def flash_verify(seed: int = 1005, batch: int = 32) -> Workload:
    """Flash-Verify stress, bf16, batch 32, prompt 512 + gen 1024, window 32, 32 tracked.

    Draft logits (N(0,1) noise, vocab 126464): in every sequence exactly 10 of
    the 32 window rows target a confidence in U(0.901, 0.999) and 22 target
    U(0.05, 0.899) (about 30% above eps=0.9). Mask-view logits are drawn per
    window row: their spike sits on the draft spike with probability 0.7 and
    on a different uniform id otherwise, with confidence targets half in
    U(0.801, 0.999) and half in U(0.05, 0.799) around gamma=0.8. Up to 16
    search tokens per sequence.
    """
    rng = np.random.default_rng(seed)
    shape = LayerShape(LLADA_D_MODEL, LLADA_HEADS, LLADA_HEAD_DIM, LLADA_THETA, "bf16")
    d = shape.d_model
    prompt, gen, window, tracked, max_search = 512, 1024, 32, 32, 16
    n = prompt + gen
    max_views = 2 * max_search
    geom = flat_geometry(batch, n + max_views)
    w = make_tensor(normal(rng, (3 * d, d), 0.02), "bf16")
    window_pos = np.arange(prompt, prompt + window, dtype=np.int32)
    tracked = np.stack([np.sort(rng.choice(prompt, size=32, replace=False)) for _ in range(batch)]).astype(np.int32)
    rows = build_rows([draft_rows(window_pos, tracked[b]) for b in range(batch)])
    x_draft = make_tensor(normal(rng, (rows.n_rows, d)), "bf16")
    x_verify = make_tensor(normal(rng, (batch * (32 + 2 * max_search), d)), "bf16")
    n_w = batch * window
    target = np.empty(n_w)
    for b in range(batch):
        hi = rng.permutation(window) < 10
        t = np.where(hi, rng.uniform(0.901, 0.999, window), rng.uniform(0.05, 0.899, window))
        target[b * window:(b + 1) * window] = t
    draft_idx = rng.integers(0, LLADA_VOCAB, size=n_w)
    logits = targeted_logits(rng, draft_idx, target, LLADA_VOCAB)
    agree = rng.uniform(size=n_w) < 0.7
    other = (draft_idx + rng.integers(1, LLADA_VOCAB, size=n_w)) % LLADA_VOCAB
    mask_idx = np.where(agree, draft_idx, other)
    high = rng.uniform(size=n_w) < 0.5
    mtarget = np.where(high, rng.uniform(0.801, 0.999, n_w), rng.uniform(0.05, 0.799, n_w))
    mask_logits = targeted_logits(rng, mask_idx, mtarget, LLADA_VOCAB)
    kc, vc = _cache_fill(rng, geom.n_pages * geom.page_size, d, "bf16")
    eligible = np.zeros((batch, n), dtype=np.uint8)
    eligible[:, :prompt] = 1
    return Workload("flash_verify", shape, batch, np.full(batch, n, np.int32), n, max_views, geom, dict(
        w=w, x=x_draft, x_verify=x_verify, rows=rows, tracked=tracked, window_pos=window_pos,
        logits=make_tensor(logits, "bf16"), mask_logits_by_window_row=make_tensor(mask_logits, "bf16"),
        k_cache=kc, v_cache=vc, eligible=eligible, topk=32, vocab=LLADA_VOCAB,
        eps=0.9, gamma=0.8, max_search=max_search, force_progress=False,
        window_rows=np.arange(n_w, dtype=np.int32),
        window_row_seq=np.repeat(np.arange(batch, dtype=np.int32), window),
        window_row_pos=np.tile(window_pos, batch).astype(np.int32)))


def projection_case(seed: int, d_model: int, n_heads: int, n_rows: int, batch: int = 3,
                    seq_len: int = 300, page_size: int = 64, theta: float = LLADA_THETA,
                    dtype: str = "bf16") -> Workload:
    """Generic fused-projection case: random rows over a paged cache.

    Rows belong to ``batch`` sequences (sorted by sequence), sit at random
    positions below ``seq_len``, and one row in seven is not written to the
    cache (cache_pos -1) as for rows that only need their query.
    """
    rng = np.random.default_rng(seed)
    hd = d_model // n_heads
    shape = LayerShape(d_model, n_heads, hd, theta, dtype)
    geom = paged_geometry(rng, [seq_len] * batch, page_size)
    w = make_tensor(normal(rng, (3 * d_model, d_model), 0.02), dtype)
    x = make_tensor(normal(rng, (n_rows, d_model)), dtype)
    seq = np.sort(rng.integers(0, batch, n_rows)).astype(np.int32)
    per_seq = []
    for b in range(batch):
        n_b = int(np.sum(seq == b))
        pos = rng.choice(seq_len, size=n_b, replace=False)
        per_seq.append([(int(p), int(p) if rng.uniform() > 1 / 7 else -1, KIND_NORMAL) for p in pos])
    rows = build_rows(per_seq)
    kc, vc = _cache_fill(rng, geom.n_pages * geom.page_size, d_model, dtype)
    return Workload("projection_case", shape, batch, np.full(batch, seq_len, np.int32), seq_len, 0, geom,
                    dict(w=w, x=x, rows=rows, k_cache=kc, v_cache=vc))


# --------------------------------------------------------------------------
# Decode traces for the KV-cache refresh policies
# --------------------------------------------------------------------------
def refresh_trace(seed: int = 1010) -> Workload:
    """Small multi-step decode for the refresh policies: bf16, d_model 512,
    4 heads of 128, theta 1e4; 3 sequences with prompts 37, 64, 5 and gen 70,
    48, 90 (ragged last blocks), block 16; paged cache of 64-slot pages
    randomly permuted in one pool, zero-filled. W ~ N(0, 0.02^2)."""
    rng = np.random.default_rng(seed)
    shape = LayerShape(512, 4, 128, 1.0e4, "bf16")
    prompts = np.array([37, 64, 5], np.int32)
    lengths = (prompts + np.array([70, 48, 90])).astype(np.int32)
    geom = paged_geometry(rng, lengths, 64)
    w = make_tensor(normal(rng, (3 * shape.d_model, shape.d_model), 0.02), "bf16")
    return Workload("refresh_trace", shape, 3, lengths, int(lengths.max()), 0, geom,
                    dict(w=w, prompts=prompts, block=16, seed=seed))


def trace_hidden(seed: int, step: int, rows: int, d: int, dtype: str = "bf16") -> Tensor:
    """Hidden inputs of one step's rows, N(0, 1)."""
    rng = np.random.default_rng([seed, 2, step])
    return make_tensor(normal(rng, (rows, d)), dtype)


def trace_unmask(rng: np.random.Generator, decoded_pos, lo: int = 1, hi: int = 4):
    """Positions a scripted step unmasks: lo..hi of the decoded rows, at random."""
    decoded_pos = np.asarray(decoded_pos)
    if decoded_pos.size == 0:
        return decoded_pos
    return rng.permutation(decoded_pos)[:int(rng.integers(lo, hi + 1))]


# --------------------------------------------------------------------------
# A whole masked-diffusion transformer with random weights
# --------------------------------------------------------------------------
def model_case(seed: int = 1013, d: int = 512, n_heads: int = 4, n_layers: int = 2, ffn: int = 1024,
               vocab: int = 2048 + 40, theta: float = 1.0e4, dtype: str = "bf16", out_std: float = 0.02,
               lm_std: float = 0.02) -> dict:
    """LLaMA-style weights (no biases), bf16: embedding ~ N(0, 1); W_qkv and
    W_gate/W_up (stacked: gate rows, then up rows) ~ N(0, 0.02^2); W_o and
    W_down ~ N(0, out_std^2) (larger values let attention and the FFN move
    the residual stream further from the embeddings); RMSNorm gains
    1 + U(-0.2, 0.2); LM head ~ N(0, lm_std^2). The last vocabulary id is the
    [MASK] token. Returns a dict of Tensors and sizes."""
    rng = np.random.default_rng(seed)
    hd = d // n_heads

    def gain():
        return make_tensor(1.0 + rng.uniform(-0.2, 0.2, size=d), dtype)

    layers = []
    for _ in range(n_layers):
        layers.append(dict(g_attn=gain(), w_qkv=make_tensor(normal(rng, (3 * d, d), 0.02), dtype),
                           w_o=make_tensor(normal(rng, (d, d), out_std), dtype), g_mlp=gain(),
                           w_gu=make_tensor(normal(rng, (2 * ffn, d), 0.02), dtype),
                           w_down=make_tensor(normal(rng, (d, ffn), out_std), dtype)))
    return dict(n_heads=n_heads, head_dim=hd, d_model=d, ffn=ffn, vocab=vocab, theta=theta, eps=1e-5,
                mask_id=vocab - 1, embed=make_tensor(normal(rng, (vocab, d)), dtype), layers=layers,
                g_final=gain(), w_lm=make_tensor(normal(rng, (vocab, d), lm_std), dtype))


def model_values(m: dict) -> dict:
    """The same dict with every Tensor replaced by its float64 values."""
    out = {}
    for k, v in m.items():
        if isinstance(v, Tensor):
            out[k] = v.values()
        elif k == "layers":
            out[k] = [{kk: vv.values() for kk, vv in layer.items()} for layer in v]
        else:
            out[k] = v
    return out


# --------------------------------------------------------------------------
# Language-model head (the step after the path: hidden states -> decisions)
# --------------------------------------------------------------------------
def lm_head_case(seed: int = 1006, vocab: int = 126464, d: int = 4096, rows: int = 32,
                 planted: float = 0.3, w_std: float = 0.02):
    """Window rows' hidden states and an LM-head weight, bf16.

    Hidden ~ N(0, 1), W_lm ~ N(0, w_std^2). For a seeded fraction ``planted``
    of the rows, one vocabulary row of W_lm is replaced by a multiple of that
    hidden row, so its logit stands far above the others and the row's
    confidence lands between 0.5 and 0.999 (the multiple is solved from the
    expected partition sum of the N(0, (w_std |h|)^2) logits, as in
    ``targeted_logits``); the other rows keep confidences near 1 / vocab.
    Returns (hidden Tensor [rows, d], W_lm Tensor [vocab, d], planted ids).
    """
    rng = np.random.default_rng(seed)
    h = normal(rng, (rows, d))
    w = normal(rng, (vocab, d), w_std)
    n_plant = int(round(planted * rows))
    plant_rows = np.sort(rng.choice(rows, size=n_plant, replace=False)) if n_plant else np.zeros(0, np.int64)
    ids = np.full(rows, -1, dtype=np.int64)
    free = rng.permutation(vocab)
    for j, r in enumerate(plant_rows):
        v = int(free[j])
        hn = float(np.linalg.norm(h[r]))
        sigma = w_std * hn
        z_rest = (vocab - 1) * math.exp(sigma * sigma / 2)
        target = float(rng.uniform(0.5, 0.999))
        logit = math.log(target / (1 - target) * z_rest)
        w[v] = (h[r] * (logit / (hn * hn))).astype(np.float32)
        ids[r] = v
    return make_tensor(h, "bf16"), make_tensor(w, "bf16"), ids
