"""float64 reference of a whole masked-diffusion transformer forward over the
refresh rows of one step, layer by layer through the KV cache.

Test infrastructure only (see the package docstring).

Pages: the Flash-dLLM paper digest describes dLLMs (LLaDA, Dream) as
bidirectional transformers that predict every masked position in parallel
("Background"), whose every denoising step runs multi-head attention and the
FFN over the query rows ("Method steps in detail", Algorithm 2 step 2: the
step's query Q^t goes through the fused kernel against the full cache); the
FlashDLM note's motivation names the same per-step MHA + FFN cost. Beyond
that the pages are silent on the block's internals.

Reading (the plainest the rest supports, since the model is LLaDA, a
LLaMA-style network): a pre-norm block with RMSNorm,
    a   = RMSNorm(h) * g_attn
    h  += Attn(a) W_o^T
    m   = RMSNorm(h) * g_mlp
    h  += (SiLU(m W_gate^T) * (m W_up^T)) W_down^T
no biases anywhere, then a final RMSNorm before the LM head. RMSNorm(x) =
x / sqrt(mean(x^2) + eps). The input of a row is the embedding of its token
(the [MASK] id for a masked position). Stored intermediates take the storage
dtype's rounding at the points where a kernel writes them to memory: the
normed rows, Q/K/V (in ``qkv_rope_cache_write``), the attention output, the
gate/up products, the SwiGLU product and the final normed rows; the residual
stream h stays in float64 here (fp32 on the GPU).

Parity: pinned by tests/test_model_pins.py (RMSNorm and SiLU special cases,
a full-refresh forward against a plain dense transformer computed without the
cache, and the exactness of a selective refresh whose tokens did not change).
"""
from __future__ import annotations

import math

import numpy as np

from .flash_dllm import qkv_rope_cache_write, sched_attn, store_round


def rmsnorm(x, g, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g, row-wise."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(g, np.float64)


def silu(x) -> np.ndarray:
    """x * sigmoid(x), written for large |x| without overflow."""
    x = np.asarray(x, np.float64)
    return np.where(x >= 0, x / (1.0 + np.exp(-np.abs(x))), x * np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))


def layer_mlp(h, g_mlp, w_gu, w_down, ffn: int, eps: float, dtype: str) -> np.ndarray:
    """The FFN half of a block: returns the residual increment."""
    m = store_round(rmsnorm(h, g_mlp, eps), dtype)
    gu = store_round(m @ np.asarray(w_gu, np.float64).T, dtype)
    u = store_round(silu(gu[:, :ffn]) * gu[:, ffn:], dtype)
    return u @ np.asarray(w_down, np.float64).T


def model_forward(model: dict, tokens, row_seq, row_rope_pos, row_cache_pos, row_kind, cu_seqlens, kv_len,
                  block_table, page_size: int, k_caches, v_caches, dtype: str, search_pos=None,
                  n_search=None, max_seq=None, track: bool = False):
    """Forward of the refresh rows through every layer.

    ``model``: dict with n_heads, head_dim, theta, ffn, eps and the weights
    embed [V, d], layers = [dict(g_attn, w_qkv, w_o, g_mlp, w_gu, w_down)],
    g_final; w_gu holds the gate rows, then the up rows. ``k_caches`` and
    ``v_caches`` are per-layer cache arrays (float64 copies are returned).
    Returns (final normed rows [R, d] rounded to ``dtype``, k caches, v
    caches, tracker increments summed over the layers [B, max_seq] or None).
    """
    H, hd, ffn, eps = model["n_heads"], model["head_dim"], model["ffn"], model["eps"]
    d = H * hd
    R = len(tokens)
    h = np.asarray(model["embed"], np.float64)[np.asarray(tokens, np.int64)]
    kcs, vcs = [], []
    tr_sum = None
    for l, w in enumerate(model["layers"]):
        a = store_round(rmsnorm(h, w["g_attn"], eps), dtype)
        q, kc, vc = qkv_rope_cache_write(a, w["w_qkv"], H, hd, model["theta"], row_rope_pos, row_seq,
                                         row_cache_pos, block_table, page_size, k_caches[l], v_caches[l], dtype)
        o, _, tr = sched_attn(q, kc, vc, block_table, page_size, cu_seqlens, kv_len, row_kind, search_pos,
                              n_search, max_seq=max_seq, dtype=dtype)
        kcs.append(kc)
        vcs.append(vc)
        if track:
            tr_sum = tr if tr_sum is None else tr_sum + tr
        h = h + o.reshape(R, d) @ np.asarray(w["w_o"], np.float64).T
        h = h + layer_mlp(h, w["g_mlp"], w["w_gu"], w["w_down"], ffn, eps, dtype)
    return store_round(rmsnorm(h, model["g_final"], eps), dtype), kcs, vcs, tr_sum


def dense_forward(model: dict, tokens, theta_pos=None):
    """A plain bidirectional transformer over ONE whole sequence, with no cache,
    no block table and no rounding: every position attends to every position.
    Used only to pin ``model_forward`` (a full refresh must equal it up to the
    storage rounding). Returns the final normed rows in float64."""
    H, hd, ffn, eps = model["n_heads"], model["head_dim"], model["ffn"], model["eps"]
    d = H * hd
    n = len(tokens)
    pos = np.arange(n) if theta_pos is None else np.asarray(theta_pos)
    h = np.asarray(model["embed"], np.float64)[np.asarray(tokens, np.int64)]
    half = hd // 2
    inv = model["theta"] ** (-np.arange(half) * 2.0 / hd)
    ang = pos[:, None] * inv[None, :]
    cos, sin = np.cos(ang), np.sin(ang)

    def rot(x):  # x [n, H, hd]
        lo, hi = x[..., :half], x[..., half:]
        c, s = cos[:, None, :], sin[:, None, :]
        return np.concatenate([lo * c - hi * s, lo * s + hi * c], axis=-1)

    for w in model["layers"]:
        a = rmsnorm(h, w["g_attn"], eps)
        y = a @ np.asarray(w["w_qkv"], np.float64).T
        q = rot(y[:, :d].reshape(n, H, hd))
        k = rot(y[:, d:2 * d].reshape(n, H, hd))
        v = y[:, 2 * d:].reshape(n, H, hd)
        s = np.einsum("ihc,jhc->hij", q, k) / math.sqrt(hd)
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o = np.einsum("hij,jhc->ihc", p, v).reshape(n, d)
        h = h + o @ np.asarray(w["w_o"], np.float64).T
        m = rmsnorm(h, w["g_mlp"], eps)
        gu = m @ np.asarray(w["w_gu"], np.float64).T
        h = h + (silu(gu[:, :ffn]) * gu[:, ffn:]) @ np.asarray(w["w_down"], np.float64).T
    return rmsnorm(h, model["g_final"], eps)
