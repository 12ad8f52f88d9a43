"""The library's host row builders (fdl_refresh_rows, fdl_verify_rows) against
the refresh oracle, bit-exact, on seeded random decode traces; and their
argument checks. CPU only: the builders are host code."""
import numpy as np
import pytest

from oracle import refresh as rf


@pytest.fixture(scope="module")
def fdl():
    from kv_cache_attention_gb300 import build
    import kv_cache_attention_gb300 as fdl
    build.build()
    fdl.load_library()
    return fdl


def _oracle_step(policy, masked, prompts, lengths, block, state, tracked=None):
    rows, new_state = [], state.copy()
    for b in range(len(prompts)):
        tr = () if tracked is None else tracked[b]
        r, new_state[b] = rf.refresh_rows(policy, masked[b], int(prompts[b]), int(lengths[b]), block,
                                          int(state[b]), tr)
        rows.append(r)
    return rows, new_state


def _compare(rows_c, rows_o):
    cu = [0]
    for b, r in enumerate(rows_o):
        cu.append(cu[-1] + len(r))
        lo, hi = int(rows_c.cu_seqlens[b]), int(rows_c.cu_seqlens[b + 1])
        got = list(zip(rows_c.row_rope_pos[lo:hi].tolist(), rows_c.row_kind[lo:hi].tolist()))
        assert got == [(p, k) for p, k in r], b
        assert (rows_c.row_seq[lo:hi] == b).all()
    assert rows_c.cu_seqlens.tolist() == cu
    assert (rows_c.row_cache_pos == rows_c.row_rope_pos).all()


@pytest.mark.parametrize("policy", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_builder_matches_oracle_on_random_traces(fdl, policy, seed):
    rng = np.random.default_rng(100 * policy + seed)
    B = int(rng.integers(1, 6))
    block = int(rng.choice([4, 8, 16, 32]))
    prompts = rng.integers(0, 40, size=B).astype(np.int32)
    lengths = (prompts + rng.integers(1, 70, size=B)).astype(np.int32)
    max_seq = int(lengths.max()) + int(rng.integers(0, 5))
    masked = np.zeros((B, max_seq), np.uint8)
    for b in range(B):
        masked[b, prompts[b]:lengths[b]] = 1
    # a few generated positions already known (not masked) at the start
    masked[rng.random(masked.shape) < 0.05] = 0
    st_c = np.full(B, -1, np.int32)
    st_o = st_c.copy()
    for step in range(400):
        tracked = n_tracked = tr_list = None
        if policy == rf.FLASH_DRAFT:
            k = 6
            tracked = np.full((B, k), -1, np.int32)
            n_tracked = np.zeros(B, np.int32)
            tr_list = []
            for b in range(B):
                free = np.nonzero(masked[b, :lengths[b]] == 0)[0]
                pick = rng.permutation(free)[:int(rng.integers(0, k + 1))]
                tracked[b, :len(pick)] = pick
                n_tracked[b] = len(pick)
                tr_list.append(pick.tolist())
        rows_c = fdl.fdl_refresh_rows(policy, prompts, lengths, masked, block, st_c, tracked, n_tracked)
        rows_o, st_o = _oracle_step(policy, masked, prompts, lengths, block, st_o, tr_list)
        _compare(rows_c, rows_o)
        assert st_c.tolist() == st_o.tolist()
        if not masked.any():
            assert rows_c.n_rows == 0
            break
        # unmask a random non-empty part of each sequence's decoded rows
        for b in range(B):
            lo, hi = int(rows_c.cu_seqlens[b]), int(rows_c.cu_seqlens[b + 1])
            dec = rows_c.row_rope_pos[lo:hi][rows_c.row_kind[lo:hi] == 1]
            if len(dec):
                masked[b, rng.permutation(dec)[:int(rng.integers(1, 4))]] = 0
    else:
        pytest.fail("decode did not finish")


def test_verify_builder_matches_oracle(fdl):
    rng = np.random.default_rng(7)
    for _ in range(20):
        B = int(rng.integers(1, 5))
        lengths = rng.integers(20, 90, size=B).astype(np.int32)
        ld_t, ld_s = 12, 10
        tracked = np.full((B, ld_t), -1, np.int32)
        search = np.full((B, ld_s), -1, np.int32)
        nt = rng.integers(0, ld_t + 1, size=B).astype(np.int32)
        ns = rng.integers(0, ld_s + 1, size=B).astype(np.int32)
        for b in range(B):
            tracked[b, :nt[b]] = rng.choice(lengths[b], size=nt[b], replace=False)
            search[b, :ns[b]] = rng.choice(lengths[b], size=ns[b], replace=False)
        budget = int(rng.integers(0, 24))
        rows = fdl.fdl_verify_rows(lengths, tracked, nt, search, ns, budget)
        k = 0
        for b in range(B):
            want = rf.verify_rows(tracked[b, :nt[b]], search[b, :ns[b]].tolist(), int(lengths[b]), budget)
            got = list(zip(rows.row_rope_pos[k:k + len(want)].tolist(), rows.row_cache_pos[k:k + len(want)].tolist(),
                           rows.row_kind[k:k + len(want)].tolist()))
            assert got == want
            assert (rows.row_seq[k:k + len(want)] == b).all()
            k += len(want)
            assert rows.cu_seqlens[b + 1] == k
        assert rows.n_rows == k


def test_builder_rejects_bad_arguments_and_leaves_state(fdl):
    prompts = np.array([4, 3], np.int32)
    lengths = np.array([12, 20], np.int32)
    masked = np.zeros((2, 20), np.uint8)
    masked[0, 5:12] = 1
    masked[1, 3:20] = 1
    st = np.full(2, -1, np.int32)
    bad = [
        dict(max_rows=31),                                  # the first step needs 12 + 20 rows
        dict(block=0),
        dict(policy=5),
        dict(prompt_len=np.array([13, 3], np.int32)),       # prompt past the sequence
        dict(seq_len=np.array([12, 21], np.int32)),         # sequence past max_seq
    ]
    base = dict(policy=1, prompt_len=prompts, seq_len=lengths, masked=masked, block=4, state=st)
    for kw in bad:
        with pytest.raises(fdl.FdlError) as ei:
            fdl.fdl_refresh_rows(**{**base, **kw})
        assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
        assert st.tolist() == [-1, -1]
    with pytest.raises(fdl.FdlError):
        fdl.fdl_refresh_rows(**{**base, "state": np.array([-2, -1], np.int32)})
    rows = fdl.fdl_refresh_rows(**{**base, "max_rows": 32})
    assert rows.n_rows == 32 and st.tolist() == [0, 0]
    # tracked positions must be decoded, inside the sequence and distinct
    fl = {**base, "policy": 4, "state": np.zeros(2, np.int32)}
    for tr in ([[5, -1], [0, -1]], [[0, 0], [0, -1]], [[12, -1], [0, -1]]):
        with pytest.raises(fdl.FdlError):
            fdl.fdl_refresh_rows(**fl, tracked=np.array(tr, np.int32), n_tracked=np.array([2 if tr[0][1] >= 0 else 1, 1],
                                                                                           np.int32))
    with pytest.raises(fdl.FdlError):       # a FLASH_DRAFT call needs its tracked set
        fdl.fdl_refresh_rows(**fl)
    rows = fdl.fdl_refresh_rows(**fl, tracked=np.array([[0, 3], [2, -1]], np.int32),
                                n_tracked=np.array([2, 1], np.int32))
    assert rows.row_rope_pos.tolist() == [5, 6, 7, 8, 0, 3] + [3, 4, 5, 6, 2]
    # verify rows: repeated or out-of-range search positions
    for sp in ([[3, 3]], [[3, 12]]):
        with pytest.raises(fdl.FdlError):
            fdl.fdl_verify_rows(np.array([12], np.int32), np.array([[0]], np.int32), np.array([1], np.int32),
                                np.array(sp, np.int32), np.array([2], np.int32), 8)
    with pytest.raises(fdl.FdlError):
        fdl.fdl_verify_rows(np.array([12], np.int32), np.array([[0]], np.int32), np.array([1], np.int32),
                            np.array([[3, 4]], np.int32), np.array([2], np.int32), 8, max_rows=4)
