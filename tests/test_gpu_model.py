"""The whole-model forward (fdl_model_forward: embedding, per layer RMSNorm,
fused projection, scheduled attention with the tracker, W_o and the SwiGLU
FFN through the dense tensor-core GEMM, then the final norm) against the
float64 oracle on identical bf16 weights and tokens.

A full forward over two ragged sequences on permuted pages; then a selective
refresh of some rows with changed tokens against the caches the oracle
left; then the argument checks."""
import numpy as np
import pytest

import oracle
from oracle import model as om
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _close_rows(gpu, ref, what):
    """The final rows are bf16 of unit-RMS values that passed through every
    layer: a difference of fp32 and float64 rounding upstream may move a value
    across a rounding boundary, so two ulps are allowed where an ulp exceeds
    the bf16 tolerance."""
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    allowed = np.maximum(H.BF16_TOL, 2.0 * H.bf16_ulp(ref))
    bad = err > allowed
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, worst err {err.max():.3e}"


def _dev_model(mc):
    return dict(ffn=mc["ffn"], eps=mc["eps"], embed=H.dev(mc["embed"]), g_final=H.dev(mc["g_final"]),
                layers=[{k: H.dev(v) for k, v in w.items()} for w in mc["layers"]])


def _setup(n_layers=2):
    import kv_cache_attention_gb300 as fdl
    mc = synth.model_case(seed=1013, n_layers=n_layers)
    m = synth.model_values(mc)
    rng = np.random.default_rng(1014)
    lengths = np.array([40, 57], np.int32)
    geom = synth.paged_geometry(rng, lengths, 64)
    n_slots = geom.n_pages * geom.page_size
    d = mc["d_model"]
    ctx = fdl.fdl_create(d, mc["n_heads"], mc["head_dim"], mc["theta"], 2, int(lengths.max()), 0, geom.page_size,
                         geom.n_pages, int(lengths.sum()), mc["vocab"], "bf16")
    return fdl, mc, m, rng, lengths, geom, n_slots, ctx


def _run(ctx, dm, mc, tokens, rows, lengths, geom, kcs, vcs, track=None):
    torch = H.torch_mod()
    R = rows.n_rows
    ws = torch.empty(ctx.model_workspace_bytes(mc["ffn"], R), dtype=torch.uint8, device="cuda")
    out = torch.empty((R, mc["d_model"]), dtype=torch.bfloat16, device="cuda")
    ctx.model_forward(dm, H.ints(tokens), H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                      H.ints(rows.row_cache_pos), H.ints(rows.row_kind), H.ints(rows.cu_seqlens), H.ints(lengths),
                      H.ints(geom.block_table), kcs, vcs, ws, out, track_scores=track)
    ctx.sync_status()
    return H.host(out)


def test_model_forward_full_then_selective_refresh():
    torch = H.torch_mod()
    fdl, mc, m, rng, lengths, geom, n_slots, ctx = _setup()
    d, L, V = mc["d_model"], len(mc["layers"]), mc["vocab"]
    dm = _dev_model(mc)
    # full forward: prompt tokens, then masked positions (the [MASK] id)
    prompts = [24, 31]
    tokens, per_seq = [], []
    for b, n in enumerate(lengths):
        t = rng.integers(0, V - 1, size=n)
        t[prompts[b]:] = mc["mask_id"]
        tokens.append(t)
        per_seq.append(synth.full_rows(int(n), range(prompts[b], prompts[b] + 16)))
    rows = synth.build_rows(per_seq)
    tok = np.concatenate(tokens).astype(np.int32)
    kcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    vcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    track = torch.zeros((2, int(lengths.max())), dtype=torch.float32, device="cuda")
    out = _run(ctx, dm, mc, tok, rows, lengths, geom, kcs, vcs, track)
    z = [np.zeros((n_slots, d)) for _ in range(L)]
    want, kco, vco, tro = om.model_forward(m, tok, rows.row_seq, rows.row_rope_pos, rows.row_cache_pos,
                                           rows.row_kind, rows.cu_seqlens, lengths, geom.block_table,
                                           geom.page_size, z, [a.copy() for a in z], "bf16",
                                           max_seq=int(lengths.max()), track=True)
    _close_rows(out, want, "final rows, full forward")
    for l in range(L):
        H.assert_close(H.host(kcs[l]), kco[l], "bf16", f"k cache layer {l}")
        H.assert_close(H.host(vcs[l]), vco[l], "bf16", f"v cache layer {l}")
    np.testing.assert_allclose(H.host(track), tro, atol=5e-4, rtol=0)
    np.testing.assert_allclose(tro.sum(1), L, atol=1e-9)          # Eq. (2): mass L per sequence
    np.testing.assert_allclose(H.host(track).sum(1), L, rtol=1e-4)
    # selective refresh: unmask some window tokens and refresh them with some
    # tracked ones, against the oracle's caches (uploaded, exact in bf16)
    per_seq, tok2 = [], []
    for b in range(2):
        p = prompts[b]
        win = list(range(p, p + 16))
        new = {p: 17, p + 3: 99}                                  # decoded this step
        tr = sorted(rng.choice(p, 8, replace=False).tolist())
        per_seq.append([(q, q, 1) for q in win] + [(q, q, 0) for q in tr])
        tok2 += [new.get(q, mc["mask_id"]) for q in win] + [int(tokens[b][q]) for q in tr]
    rows2 = synth.build_rows(per_seq)
    tok2 = np.array(tok2, np.int32)
    kcs = [H.dev(synth.make_tensor(a, "bf16")) for a in kco]
    vcs = [H.dev(synth.make_tensor(a, "bf16")) for a in vco]
    track.zero_()
    out2 = _run(ctx, dm, mc, tok2, rows2, lengths, geom, kcs, vcs, track)
    want2, kco2, vco2, tro2 = om.model_forward(m, tok2, rows2.row_seq, rows2.row_rope_pos, rows2.row_cache_pos,
                                               rows2.row_kind, rows2.cu_seqlens, lengths, geom.block_table,
                                               geom.page_size, kco, vco, "bf16", max_seq=int(lengths.max()),
                                               track=True)
    _close_rows(out2, want2, "final rows, selective refresh")
    for l in range(L):
        H.assert_close(H.host(kcs[l]), kco2[l], "bf16", f"k cache layer {l}, refresh")
    np.testing.assert_allclose(H.host(track), tro2, atol=5e-4, rtol=0)
    ctx.close()


def test_model_forward_wide_ffn_takes_the_persistent_gemm():
    """A full forward of 1050 rows through a layer with a 8192-wide FFN: the
    SwiGLU gate/up product has 128 feature tiles x 5 row tiles of 256, four
    waves of the GPU, so it runs on the persistent GEMM (whole-tile waves,
    then stream-K shares merged in CTA order); the other products stay on the
    split-K kernels. Final rows and caches against the oracle."""
    torch = H.torch_mod()
    import kv_cache_attention_gb300 as fdl
    mc = synth.model_case(seed=1015, n_layers=1, ffn=8192)
    m = synth.model_values(mc)
    rng = np.random.default_rng(1016)
    lengths = np.array([520, 530], np.int32)
    geom = synth.paged_geometry(rng, lengths, 64)
    n_slots = geom.n_pages * geom.page_size
    d, V = mc["d_model"], mc["vocab"]
    ctx = fdl.fdl_create(d, mc["n_heads"], mc["head_dim"], mc["theta"], 2, int(lengths.max()), 0, geom.page_size,
                         geom.n_pages, int(lengths.sum()), V, "bf16")
    dm = _dev_model(mc)
    prompts = [300, 310]
    tokens, per_seq = [], []
    for b, n in enumerate(lengths):
        t = rng.integers(0, V - 1, size=n)
        t[prompts[b]:] = mc["mask_id"]
        tokens.append(t)
        per_seq.append(synth.full_rows(int(n), range(prompts[b], prompts[b] + 32)))
    rows = synth.build_rows(per_seq)
    tok = np.concatenate(tokens).astype(np.int32)
    kcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda")]
    vcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda")]
    out = _run(ctx, dm, mc, tok, rows, lengths, geom, kcs, vcs)
    z = [np.zeros((n_slots, d))]
    want, kco, vco, _ = om.model_forward(m, tok, rows.row_seq, rows.row_rope_pos, rows.row_cache_pos,
                                         rows.row_kind, rows.cu_seqlens, lengths, geom.block_table,
                                         geom.page_size, z, [a.copy() for a in z], "bf16",
                                         max_seq=int(lengths.max()), track=False)
    _close_rows(out, want, "final rows, wide-FFN full forward")
    H.assert_close(H.host(kcs[0]), kco[0], "bf16", "k cache, wide-FFN full forward")
    H.assert_close(H.host(vcs[0]), vco[0], "bf16", "v cache, wide-FFN full forward")
    ctx.close()


def test_model_forward_checks_and_edges():
    torch = H.torch_mod()
    fdl, mc, m, rng, lengths, geom, n_slots, ctx = _setup(n_layers=1)
    d = mc["d_model"]
    dm = _dev_model(mc)
    kcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda")]
    vcs = [torch.zeros((n_slots, d), dtype=torch.bfloat16, device="cuda")]
    rows = synth.build_rows([[(0, 0, 0), (5, 5, 0)], [(3, 3, 0)]])
    # a token outside the vocabulary is reported (and gives a zero input row)
    with pytest.raises(fdl.FdlError) as ei:
        _run(ctx, dm, mc, np.array([1, mc["vocab"], 2], np.int32), rows, lengths, geom, kcs, vcs)
    assert ei.value.status == fdl.FDL_ERR_DEVICE_INDEX
    ctx.sync_status()
    bad = dict(dm, ffn=1000)
    with pytest.raises(fdl.FdlError) as ei:
        _run(ctx, bad, mc, np.array([1, 2, 3], np.int32), rows, lengths, geom, kcs, vcs)
    assert ei.value.status == fdl.FDL_ERR_UNSUPPORTED
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty((3, d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fdl.FdlError) as ei:                 # workspace too small
        ctx.model_forward(dm, H.ints([1, 2, 3]), H.ints(rows.row_seq), H.ints(rows.row_rope_pos),
                          H.ints(rows.row_cache_pos), H.ints(rows.row_kind), H.ints(rows.cu_seqlens),
                          H.ints(lengths), H.ints(geom.block_table), kcs, vcs, ws, out)
    assert ei.value.status == fdl.FDL_ERR_INVALID_ARG
    ctx.close()
