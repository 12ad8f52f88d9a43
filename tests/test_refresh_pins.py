"""Pins of the refresh-policy oracle (oracle/refresh.py), on the CPU.

The row sets are checked against what the pages fix, computed here without
the oracle: closed-form row totals of a scripted decode (which unmasks the u
leftmost masked positions of the current block per step), coverage
invariants at every step, the freshness of every cached position that each
page states, and reductions between policies (DualCache with one block is
PrefixCache; FreeCache with one block is PrefixCache).
"""
import math

import numpy as np
import pytest

from oracle import refresh as rf

POLICIES = (rf.FULL, rf.PREFIX, rf.DUAL, rf.FREECACHE)


def _block_of(masked, prompt, beta):
    """Current block by hand: the block of the leftmost masked generated position."""
    pos = [p for p in range(prompt, len(masked)) if masked[p]]
    return None if not pos else (pos[0] - prompt) // beta


def _scripted(policy, prompt, gen, beta, u):
    """Runs a decode that unmasks the u leftmost masked positions of the
    current block per step; yields (step, rows, masked-before, block) per step."""
    n = prompt + gen
    masked = np.zeros(n, np.uint8)
    masked[prompt:] = 1
    state, step = rf.NO_STEP_YET, 0
    while masked.any():
        cur = _block_of(masked, prompt, beta)
        rows, state = rf.refresh_rows(policy, masked, prompt, n, beta, state)
        yield step, rows, masked.copy(), cur
        s, e = prompt + cur * beta, min(prompt + (cur + 1) * beta, n)
        left = [p for p in range(s, e) if masked[p]][:u]
        masked[left] = 0
        step += 1
    rows, state = rf.refresh_rows(policy, masked, prompt, n, beta, state)
    assert rows == []


def _closed_form(policy, prompt, gen, beta, u):
    n = prompt + gen
    starts = list(range(prompt, n, beta))
    lens = [min(beta, n - s) for s in starts]
    steps = [math.ceil(L / u) for L in lens]
    if policy == rf.FULL:
        return n * sum(steps)
    if policy == rf.PREFIX:
        return sum(n + (S - 1) * (n - s) for s, S in zip(starts, steps))
    if policy == rf.DUAL:
        return sum(n + (S - 1) * L for L, S in zip(lens, steps))
    if policy == rf.FREECACHE:
        return n + (steps[0] - 1) * (n - starts[0]) + sum(
            S * (n - s) for s, S in zip(starts[1:], steps[1:]))
    raise ValueError(policy)


SHAPES = [(7, 50, 16, 3), (0, 32, 8, 1), (13, 64, 16, 16), (5, 40, 64, 4), (1, 9, 4, 2), (24, 256, 32, 2)]


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("prompt,gen,beta,u", SHAPES)
def test_row_totals_match_the_closed_form(policy, prompt, gen, beta, u):
    total = sum(len(rows) for _, rows, _, _ in _scripted(policy, prompt, gen, beta, u))
    assert total == _closed_form(policy, prompt, gen, beta, u)


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("prompt,gen,beta,u", SHAPES)
def test_every_step_covers_what_its_page_says(policy, prompt, gen, beta, u):
    n = prompt + gen
    prev_block = None
    for step, rows, masked, cur in _scripted(policy, prompt, gen, beta, u):
        pos = [p for p, _ in rows]
        assert pos == sorted(set(pos))                       # distinct, ascending
        s, e = prompt + cur * beta, min(prompt + (cur + 1) * beta, n)
        # decoded rows: exactly the masked positions of the current block
        assert {p for p, k in rows if k == 1} == {p for p in range(s, e) if masked[p]}
        assert all(k in (0, 1) for _, k in rows)
        if policy == rf.FULL:
            expect = range(n)
        elif policy in (rf.PREFIX, rf.DUAL):
            # a full forward exactly at the first step of every block
            expect = range(n) if cur != prev_block else (range(s, n) if policy == rf.PREFIX else range(s, e))
        else:
            expect = range(n) if step == 0 else range(s, n)
        assert pos == list(expect)
        if policy in (rf.FULL, rf.PREFIX, rf.FREECACHE):
            assert {p for p in range(n) if masked[p]} <= set(pos)   # all masks recomputed
        prev_block = cur


@pytest.mark.parametrize("prompt,gen,beta,u", SHAPES)
def test_cached_positions_age_as_each_page_states(prompt, gen, beta, u):
    n = prompt + gen
    for policy in (rf.PREFIX, rf.DUAL, rf.FREECACHE):
        version = np.full(n, -1)
        done_at = {}
        prev = None
        for step, rows, masked, cur in _scripted(policy, prompt, gen, beta, u):
            for p, _ in rows:
                version[p] = step
            for j in range(cur):
                done_at.setdefault(j, step)
            if policy in (rf.PREFIX, rf.DUAL) and cur != prev:
                # Fast-dLLM: once a block is decoded, the whole cache is recomputed,
                # so every position's K/V is from this step and every earlier
                # block is fully decoded.
                assert version.min() == step
                assert not masked[prompt:prompt + cur * beta].any()
            if policy == rf.FREECACHE and step > 0:
                # FreeCache: the prompt keeps the first forward's K/V, and a block
                # is never recomputed after the step it finished unmasking.
                assert (version[:prompt] == 0).all()
                for j, t in done_at.items():
                    s = prompt + j * beta
                    assert (version[s:min(s + beta, n)] < t).all()
            if policy == rf.DUAL and cur == prev:
                # DualCache: the cached suffix is not recomputed inside a block
                e = min(prompt + (cur + 1) * beta, n)
                assert (version[e:] < step).all()
            prev = cur


@pytest.mark.parametrize("prompt,gen,u", [(7, 50, 3), (0, 16, 1), (30, 33, 5)])
def test_one_block_reductions(prompt, gen, u):
    beta = gen  # a single block
    runs = {p: [rows for _, rows, _, _ in _scripted(p, prompt, gen, beta, u)] for p in POLICIES}
    assert runs[rf.DUAL] == runs[rf.PREFIX]
    assert runs[rf.FREECACHE] == runs[rf.PREFIX]
    big = [rows for _, rows, _, _ in _scripted(rf.DUAL, prompt, gen, 4 * gen, u)]
    assert big == runs[rf.PREFIX]


def test_finished_sequence_takes_no_rows():
    masked = np.zeros(40, np.uint8)
    for policy in POLICIES + (rf.FLASH_DRAFT,):
        for state in (rf.NO_STEP_YET, 0, 3):
            assert rf.refresh_rows(policy, masked, 8, 40, 16, state, tracked=(1, 2)) == ([], state)


def test_flash_draft_rows():
    # the llada-layer shape: prompt 512 + gen 256, window 32, 32 tracked
    prompt, n, bm = 512, 768, 32
    rng = np.random.default_rng(5)
    masked = np.zeros(n, np.uint8)
    masked[prompt:] = 1
    rows, st = rf.refresh_rows(rf.FLASH_DRAFT, masked, prompt, n, bm, rf.NO_STEP_YET)
    assert st == 0 and [p for p, _ in rows] == list(range(n))
    assert [p for p, k in rows if k == 1] == list(range(512, 544))
    tracked = rng.choice(prompt, size=32, replace=False)
    rows, st = rf.refresh_rows(rf.FLASH_DRAFT, masked, prompt, n, bm, 0, tracked)
    assert rows == [(p, 1) for p in range(512, 544)] + [(int(p), 0) for p in tracked]
    # a scattered mask: the window is the first 32 masked positions in order
    masked[prompt:] = rng.integers(0, 2, size=n - prompt)
    order = np.nonzero(masked)[0]
    rows, _ = rf.refresh_rows(rf.FLASH_DRAFT, masked, prompt, n, bm, 0, tracked[:5])
    assert [p for p, k in rows if k == 1] == order[:32].tolist()
    assert len(rows) == 37
    # fewer masked positions than the window: all of them
    masked[:] = 0
    masked[[600, 700, 701]] = 1
    rows, _ = rf.refresh_rows(rf.FLASH_DRAFT, masked, prompt, n, bm, 0, ())
    assert rows == [(600, 1), (700, 1), (701, 1)]


def test_verify_rows_shrink_the_tracked_set():
    tracked = list(range(100, 132))
    search = [530 + 2 * j for j in range(16)]
    rows = rf.verify_rows(tracked, search, 1536, 64)      # the stress case: 32 + 16 + 16
    assert len(rows) == 64
    assert rows[:32] == [(p, p, 0) for p in tracked]
    for j, s in enumerate(search):
        assert rows[32 + j] == (s, 1536 + j, 2 + 2 * j)
        assert rows[48 + j] == (s, 1536 + 16 + j, 3 + 2 * j)
    rows = rf.verify_rows(tracked, list(range(600, 640)), 768, 64)   # 2m > budget: no tracked rows
    assert len(rows) == 80 and all(k >= 2 for _, _, k in rows)
    assert rf.verify_rows(tracked, [], 768, 64) == [(p, p, 0) for p in tracked]
