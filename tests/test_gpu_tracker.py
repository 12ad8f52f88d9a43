"""The Eq. (2) attention-mass tracker on the tensor-core attention (bf16,
head_dim 128) against the oracle, and its reproducibility.

Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...",
section "Method steps in detail", step 4, Eq. (2): the scores are the
masked-window rows' attention probabilities averaged over heads and rows.
The kernels add each head's column sums through per-(sequence, slot, head)
partials, one slot per 128-row query tile holding WINDOW rows (up to two per
sequence), which the sequence's last CTA adds in a fixed order; a sequence
whose WINDOW rows span more tiles falls back to atomic adds. Cases:

  decode   rows [64, 150, 40]: one query tile per CTA with two KV splits,
           the middle sequence's WINDOW rows spanning two tiles (two slots);
  refresh  rows [600, 300]: two query tiles per CTA, the first sequence's
           WINDOW rows spanning a pair's two tiles, the second sequence's
           three tiles (the atomic fallback).

Every case: scores within the fp32 tolerance of the oracle, repeated calls
bit-identical for the sequences with at most two WINDOW tiles, and a second
call into the same scores adds the same contribution again."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu

D, HEADS, HD, PAGE = 2048, 16, 128, 64


def _run_case(rows, windows, kv_len, max_seq, seed):
    import torch
    import kv_cache_attention_gb300 as fdl
    rng = np.random.default_rng(seed)
    B = len(rows)
    cu = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(cu[-1])
    kinds = np.zeros(R, np.int32)
    for b, (a, z) in enumerate(windows):
        kinds[cu[b] + a:cu[b] + z] = 1  # FDL_KIND_WINDOW
    geom = synth.paged_geometry(rng, [max_seq] * B, PAGE)
    nslot = geom.n_pages * PAGE
    K = synth.make_tensor(rng.standard_normal((nslot, D)), "bf16")
    V = synth.make_tensor(rng.standard_normal((nslot, D)), "bf16")
    q = synth.make_tensor(rng.standard_normal((R, HEADS, HD)) * 0.5, "bf16")
    kv = np.asarray(kv_len, np.int32)
    ctx = fdl.fdl_create(D, HEADS, HD, 1e4, B, max_seq, 0, PAGE, geom.n_pages, R, 16, "bf16")
    args = (H.dev(q), H.dev(K), H.dev(V), H.ints(geom.block_table), H.ints(cu), H.ints(kv), H.ints(kinds))
    o = H.empty((R, HEADS, HD), "bf16")
    runs = []
    for _ in range(3):
        tr = torch.zeros((B, max_seq), dtype=torch.float32, device="cuda")
        ctx.sched_attn(*args, o, track_scores=tr)
        ctx.sync_status()
        runs.append(H.host(tr))
    # a second call into the same scores adds the same contribution again
    ctx.sched_attn(*args, o, track_scores=tr)
    ctx.sync_status()
    twice = H.host(tr)
    ctx.close()
    _, _, tr_o = oracle.sched_attn(q.values(), K.values(), V.values(), geom.block_table, PAGE, cu, kv, kinds,
                                   max_seq=max_seq, dtype="bf16")
    return runs, twice, tr_o


def _tiles(a, z):
    return len(range(a // 128, (z - 1) // 128 + 1))


@pytest.mark.parametrize("case", ["decode", "refresh"])
def test_tracker_slots_are_exact_and_reproducible(case):
    if case == "decode":
        rows, windows, kv_len, max_seq = [64, 150, 40], [(10, 42), (100, 142), (0, 40)], [300, 380, 200], 384
    else:
        rows, windows, kv_len, max_seq = [600, 300], [(120, 140), (100, 300)], [700, 500], 768
    runs, twice, tr_o = _run_case(rows, windows, kv_len, max_seq, seed=11 if case == "decode" else 12)
    for r in runs:
        H.assert_close(r, tr_o, "f32", f"{case} tracker scores")
    H.assert_close(twice, 2.0 * tr_o, "f32", f"{case} tracker scores after two calls")
    det = [b for b, (a, z) in enumerate(windows) if _tiles(a, z) <= 2]
    assert det, "every case has sequences on the fixed-order path"
    for r in runs[1:]:
        assert np.array_equal(r[det], runs[0][det]), f"{case}: repeated calls differ"
    # the sums really are the (rows x heads)-averaged probabilities: each
    # sequence's scores add up to one
    np.testing.assert_allclose(runs[0].sum(1), 1.0, rtol=1e-4)
