"""Which positions one denoising step recomputes, under each KV-cache refresh
policy the layer-step kernels serve.

Test infrastructure only (see the package docstring). A refresh policy only
chooses the query rows of a step: every chosen row is projected, its K/V
overwrite the cache at its own position, and it attends over the whole
cache. The positions not chosen keep the K/V they were last given. So each
function here returns, per sequence, the list of (position, kind) rows of
one step, plus the sequence's updated policy state, and nothing else.

Pages followed:
  [FAST] Fast-dLLM news piece, section on the key-value cache for block-wise
         decoding: the prompt's KV is computed when inference starts and is
         reused for every step of a block; once a block has been decoded, the
         cache of ALL tokens is recomputed, not only the new ones. DualCache
         caches the suffix too (in block-wise decoding the suffix is all
         masked), so a step only recomputes the current block.
  [FREE] FlashDLM note, key design 1 (FreeCache): the generated part is cut
         into fixed blocks B_1..B_N; the first forward computes the KV of the
         whole sequence; while B_i is generated the active window is B_i and
         every block after it, and the prompt and the frozen blocks only give
         KV; when B_i is fully unmasked its KV is frozen and the window shrinks.
  [FD]   Flash-dLLM paper digest, Algorithm 2: step 1 (one full forward at
         initialisation), step 2 (each step's query is the tracked set plus
         the sliding masked window) and step 3 (the verify forward: the
         tracked set shrunk to free query slots, then the draft view and the
         mask view of each search token).

Readings (where the pages leave a step open):
  * Blocks start at the end of the prompt: block i covers positions
    [P + i*beta, min(P + (i+1)*beta, N)). The current block is the first one
    that still holds a masked position; a sequence with none left takes no
    rows.
  * Fast-dLLM's "update the cache of all tokens after a block" is the first
    forward of the next block: it recomputes every position (and gives that
    step's logits). The very first step of a sequence is such a full forward
    too (the prompt's KV is computed when inference starts).
  * PrefixCache recomputes the current block and everything after it;
    DualCache only the current block. FreeCache recomputes the current block
    and everything after it, with a full forward only at the first step.
  * Kind 1 (masked-window: the rows whose predictions are decoded) marks the
    still-masked positions of the current block; every other row is kind 0.
    Rows of a sequence come in ascending position order.
  * Flash-dLLM's draft forward: the window is the first beta_m still-masked
    positions in generation order (kind 1), then the tracked set (kind 0) in
    the order given; the first step is a full forward.

Parity: pinned by tests/test_refresh_pins.py (closed-form row totals over
scripted decodes, coverage invariants, reductions between policies, the
shapes of the Flash-dLLM forwards).
"""
from __future__ import annotations

FULL = 0          # no cache reuse: every position, every step
PREFIX = 1        # Fast-dLLM PrefixCache
DUAL = 2          # Fast-dLLM DualCache
FREECACHE = 3     # FlashDLM FreeCache
FLASH_DRAFT = 4   # Flash-dLLM draft forward

NO_STEP_YET = -1


def blocks(prompt: int, n: int, beta: int):
    """[FREE] fixed blocks of the generated part, as (start, end) pairs."""
    return [(s, min(s + beta, n)) for s in range(prompt, n, beta)]


def current_block(masked_b, prompt: int, n: int, beta: int):
    """Index of the first block still holding a masked position, or None."""
    for i, (s, e) in enumerate(blocks(prompt, n, beta)):
        if any(int(masked_b[p]) for p in range(s, e)):
            return i
    return None


def refresh_rows(policy: int, masked_b, prompt: int, n: int, beta: int, state: int, tracked=()):
    """Rows of one step of one sequence: ([(position, kind)], new_state).

    ``masked_b[p]`` is 1 while position p is masked; ``state`` is the policy
    state carried between steps (NO_STEP_YET before the first one). For
    FLASH_DRAFT, ``beta`` is the window size beta_m and ``tracked`` the
    tracked positions.
    """
    if policy == FLASH_DRAFT:
        masked_pos = [p for p in range(prompt, n) if int(masked_b[p])]
        if not masked_pos:
            return [], state
        window = masked_pos[:beta]
        if state == NO_STEP_YET:
            win = set(window)
            return [(p, 1 if p in win else 0) for p in range(n)], 0
        return [(p, 1) for p in window] + [(int(p), 0) for p in tracked], state

    cur = current_block(masked_b, prompt, n, beta)
    if cur is None:
        return [], state
    s, e = blocks(prompt, n, beta)[cur]

    def kind(p):
        return 1 if (s <= p < e and int(masked_b[p])) else 0

    if policy == FULL:
        chosen, new_state = range(0, n), cur
    elif policy in (PREFIX, DUAL):
        if state != cur:                       # first forward of this block
            chosen = range(0, n)
        else:
            chosen = range(s, n) if policy == PREFIX else range(s, e)
        new_state = cur
    elif policy == FREECACHE:
        chosen = range(0, n) if state == NO_STEP_YET else range(s, n)
        new_state = cur
    else:
        raise ValueError(policy)
    return [(p, kind(p)) for p in chosen], new_state


def verify_rows(tracked, search_pos, n: int, query_budget: int):
    """[FD] rows of one sequence's verify forward, as (rope_pos, cache_pos, kind).

    The tracked rows kept are the first max(0, budget - 2m) of the tracked set
    (which comes ordered by score); then search token j's draft view
    (kind 2 + 2j, K/V at cache position n + j) and its mask view (kind 3 + 2j,
    at n + m + j), both rotated at the token's own position.
    """
    m = len(search_pos)
    keep = max(0, query_budget - 2 * m)
    rows = [(int(p), int(p), 0) for p in list(tracked)[:keep]]
    rows += [(int(s), n + j, 2 + 2 * j) for j, s in enumerate(search_pos)]
    rows += [(int(s), n + m + j, 3 + 2 * j) for j, s in enumerate(search_pos)]
    return rows
