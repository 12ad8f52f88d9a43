"""Python binding of libfdl, the GB300 Flash-dLLM layer-step hot path.

Argument marshalling only: every function forwards torch device tensors as
raw pointers to the C ABI declared in ``include/fdl.h``; all computation
happens in the library's CUDA kernels. The names mirror the C entry points.
Importing this module does not load the library; the first call does, and it
raises ``FdlError`` if ``libfdl.so`` has not been built (there is no other
implementation to fall back on).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfdl.so")

FDL_OK = 0
FDL_ERR_INVALID_ARG = 1
FDL_ERR_UNSUPPORTED = 2
FDL_ERR_OOM = 3
FDL_ERR_CUDA = 4
FDL_ERR_DEVICE_INDEX = 5
FDL_ERR_TIMEOUT = 6

FDL_F32 = 0
FDL_BF16 = 1

FDL_KIND_NORMAL = 0
FDL_KIND_WINDOW = 1


def FDL_KIND_DRAFT_VIEW(j: int) -> int:
    return 2 + 2 * j


def FDL_KIND_MASK_VIEW(j: int) -> int:
    return 3 + 2 * j


# Every symbol include/fdl.h declares.
EXPORTS = (
    "fdl_create", "fdl_destroy", "fdl_set_stream", "fdl_set_wait_budget", "fdl_last_error", "fdl_sync_status",
    "fdl_tile_m", "fdl_worklist_capacity", "fdl_qkv_rope_cache_write", "fdl_sched_attn",
    "fdl_track_topk", "fdl_unmask_verify", "fdl_sched_attn_noalloc", "fdl_lm_head_unmask",
    "fdl_refresh_rows", "fdl_verify_rows", "fdl_lm_head_verify", "fdl_model_workspace_bytes",
    "fdl_model_forward", "fdl_flash_workspace_bytes", "fdl_flash_step",
)

FDL_REFRESH_FULL = 0
FDL_REFRESH_PREFIX = 1
FDL_REFRESH_DUAL = 2
FDL_REFRESH_FREECACHE = 3
FDL_REFRESH_FLASH_DRAFT = 4


class FdlError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"fdl status {status}: {msg}")
        self.status = status


class fdl_config(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("rope_theta", ctypes.c_double), ("max_batch", ctypes.c_int), ("max_seq", ctypes.c_int),
        ("max_views", ctypes.c_int), ("page_size", ctypes.c_int), ("n_pages", ctypes.c_int),
        ("max_rows", ctypes.c_int), ("vocab", ctypes.c_int), ("dtype", ctypes.c_int),
    ]


_P = ctypes.c_void_p


class fdl_unmask_args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("max_search", ctypes.c_int),
        ("logits", _P), ("R_w", ctypes.c_int), ("row_seq", _P), ("row_pos", _P),
        ("eps", ctypes.c_float), ("force_progress", ctypes.c_int),
        ("conf", _P), ("argmax", _P), ("commit", _P), ("search_rows", _P), ("n_search", _P),
        ("mask_logits", _P), ("draft_tok", _P), ("gamma", ctypes.c_float),
        ("accept", _P), ("n_accept", _P), ("mask_conf", _P), ("mask_argmax", _P),
    ]


_PP = ctypes.POINTER(ctypes.c_void_p)


class fdl_model(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("ffn", ctypes.c_int), ("rms_eps", ctypes.c_float), ("embed", _P),
        ("g_attn", _PP), ("w_qkv", _PP), ("w_o", _PP), ("g_mlp", _PP), ("w_gu", _PP), ("w_down", _PP),
        ("g_final", _P),
    ]


class fdl_flash_params(ctypes.Structure):
    _fields_ = [
        ("window", ctypes.c_int), ("track_budget", ctypes.c_int), ("max_search", ctypes.c_int),
        ("eps", ctypes.c_float), ("gamma", ctypes.c_float), ("force_progress", ctypes.c_int),
        ("mask_token", ctypes.c_int),
    ]


class fdl_flash_seqs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("max_seq", ctypes.c_int), ("prompt_len", _P), ("seq_len", _P), ("tokens", _P),
        ("masked", _P), ("tracked", _P), ("n_tracked", _P), ("state", _P),
    ]


class fdl_flash_trace(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("n_rows", "n_window", "window_seq", "window_pos", "conf", "argmax", "commit",
                                  "search_rows", "n_search", "mask_conf", "mask_argmax", "n_accept", "track",
                                  "draft_final", "verify_final")]


class fdl_refresh_args(ctypes.Structure):
    _fields_ = [
        ("policy", ctypes.c_int), ("B", ctypes.c_int), ("max_seq", ctypes.c_int), ("block", ctypes.c_int),
        ("prompt_len", _P), ("seq_len", _P), ("masked", _P), ("state", _P),
        ("tracked", _P), ("tracked_ld", ctypes.c_int), ("n_tracked", _P), ("max_rows", ctypes.c_int),
        ("row_seq", _P), ("row_rope_pos", _P), ("row_cache_pos", _P), ("row_kind", _P),
        ("cu_seqlens", _P), ("n_rows", _P),
    ]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libfdl.so and declares its C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FdlError(FDL_ERR_UNSUPPORTED, f"{path} is not built; run kv_cache_attention_gb300.build.build()")
    L = ctypes.CDLL(path)
    i, p, f, d = ctypes.c_int, _P, ctypes.c_float, ctypes.c_double
    L.fdl_create.argtypes = [ctypes.POINTER(fdl_config), p, ctypes.POINTER(p)]
    L.fdl_create.restype = i
    L.fdl_destroy.argtypes = [p]
    L.fdl_destroy.restype = None
    L.fdl_set_stream.argtypes = [p, p]
    L.fdl_set_stream.restype = i
    L.fdl_set_wait_budget.argtypes = [p, ctypes.c_longlong]
    L.fdl_set_wait_budget.restype = i
    L.fdl_last_error.argtypes = [p]
    L.fdl_last_error.restype = ctypes.c_char_p
    L.fdl_sync_status.argtypes = [p]
    L.fdl_sync_status.restype = i
    L.fdl_tile_m.argtypes = [p]
    L.fdl_tile_m.restype = i
    L.fdl_worklist_capacity.argtypes = [p, i, i]
    L.fdl_worklist_capacity.restype = i
    L.fdl_qkv_rope_cache_write.argtypes = [p, p, p, i, p, p, p, p, i, p, p, p]
    L.fdl_qkv_rope_cache_write.restype = i
    L.fdl_sched_attn.argtypes = [p, p, p, p, p, i, p, p, i, i, p, p, i, p, p, p, p, i, p]
    L.fdl_sched_attn.restype = i
    L.fdl_track_topk.argtypes = [p, p, p, i, p, i, i, p, p]
    L.fdl_track_topk.restype = i
    L.fdl_unmask_verify.argtypes = [p, ctypes.POINTER(fdl_unmask_args)]
    L.fdl_unmask_verify.restype = i
    L.fdl_lm_head_unmask.argtypes = [p, p, p, ctypes.POINTER(fdl_unmask_args)]
    L.fdl_lm_head_unmask.restype = i
    L.fdl_lm_head_verify.argtypes = [p, p, p, ctypes.POINTER(fdl_unmask_args)]
    L.fdl_lm_head_verify.restype = i
    L.fdl_sched_attn_noalloc.argtypes = [ctypes.POINTER(fdl_config), p, p, p, p, p, i, p, p, i, i, p, p, i, p, p,
                                         p, p, i, p]
    L.fdl_sched_attn_noalloc.restype = i
    L.fdl_model_workspace_bytes.argtypes = [p, i, i]
    L.fdl_model_workspace_bytes.restype = ctypes.c_size_t
    L.fdl_model_forward.argtypes = [p, ctypes.POINTER(fdl_model), p, i, p, p, p, p, p, p, i, p, i, _PP, _PP, p, i, p,
                                    p, i, p, ctypes.c_size_t, p]
    L.fdl_model_forward.restype = i
    L.fdl_flash_workspace_bytes.argtypes = [p, i, ctypes.POINTER(fdl_flash_params), i, i]
    L.fdl_flash_workspace_bytes.restype = ctypes.c_size_t
    L.fdl_flash_step.argtypes = [p, ctypes.POINTER(fdl_model), p, _PP, _PP, p, i, ctypes.POINTER(fdl_flash_params),
                                 ctypes.POINTER(fdl_flash_seqs), ctypes.POINTER(fdl_flash_trace), p, ctypes.c_size_t]
    L.fdl_flash_step.restype = i
    L.fdl_refresh_rows.argtypes = [ctypes.POINTER(fdl_refresh_args)]
    L.fdl_refresh_rows.restype = i
    L.fdl_verify_rows.argtypes = [i, p, p, i, p, p, i, p, i, i, p, p, p, p, p, p]
    L.fdl_verify_rows.restype = i
    _lib = L
    return L


def _ptr(t) -> int | None:
    """Device pointer of a tensor (None stays NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise FdlError(FDL_ERR_INVALID_ARG, "tensor arguments must live on the GPU")
    if not t.is_contiguous():
        raise FdlError(FDL_ERR_INVALID_ARG, "tensor arguments must be contiguous")
    return t.data_ptr()


class Context:
    """Owns one ``fdl_ctx``. Methods mirror the C entry points."""

    def __init__(self, handle: int, cfg: fdl_config):
        self.handle = ctypes.c_void_p(handle)
        self.cfg = cfg

    def _check(self, st: int, what: str):
        if st != FDL_OK:
            msg = load_library().fdl_last_error(self.handle)
            raise FdlError(st, f"{what}: {msg.decode() if msg else ''}")

    def close(self):
        if self.handle:
            load_library().fdl_destroy(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def tile_m(self) -> int:
        return load_library().fdl_tile_m(self.handle)

    def worklist_capacity(self, R: int, B: int) -> int:
        return load_library().fdl_worklist_capacity(self.handle, R, B)

    def set_stream(self, stream) -> None:
        self._check(load_library().fdl_set_stream(self.handle, _stream_handle(stream)), "fdl_set_stream")

    def sync_status(self) -> None:
        self._check(load_library().fdl_sync_status(self.handle), "fdl_sync_status")

    def set_wait_budget(self, cycles: int) -> None:
        self._check(load_library().fdl_set_wait_budget(self.handle, int(cycles)), "fdl_set_wait_budget")

    def qkv_rope_cache_write(self, X, Wqkv, row_seq, row_rope_pos, row_cache_pos, block_table,
                             k_cache, v_cache, q_out) -> None:
        R = int(X.shape[0])
        st = load_library().fdl_qkv_rope_cache_write(
            self.handle, _ptr(X), _ptr(Wqkv), R, _ptr(row_seq), _ptr(row_rope_pos), _ptr(row_cache_pos),
            _ptr(block_table), int(block_table.shape[-1]), _ptr(k_cache), _ptr(v_cache), _ptr(q_out))
        self._check(st, "fdl_qkv_rope_cache_write")

    def sched_attn(self, q, k_cache, v_cache, block_table, cu_seqlens_q, kv_len, row_kind, o_out,
                   lse_out=None, track_scores=None, search_pos=None, n_search=None,
                   worklist_out=None) -> None:
        B = int(kv_len.shape[0])
        R = int(q.shape[0])
        search_ld = int(search_pos.shape[-1]) if search_pos is not None else 0
        track_ld = int(track_scores.shape[-1]) if track_scores is not None else 0
        st = load_library().fdl_sched_attn(
            self.handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), int(block_table.shape[-1]),
            _ptr(cu_seqlens_q), _ptr(kv_len), B, R, _ptr(row_kind), _ptr(search_pos), search_ld,
            _ptr(n_search), _ptr(o_out), _ptr(lse_out), _ptr(track_scores), track_ld, _ptr(worklist_out))
        self._check(st, "fdl_sched_attn")

    def track_topk(self, scores, eligible, seq_len, k: int, idx_out, cnt_out) -> None:
        B = int(seq_len.shape[0])
        st = load_library().fdl_track_topk(self.handle, _ptr(scores), _ptr(eligible), int(scores.shape[-1]),
                                           _ptr(seq_len), B, int(k), _ptr(idx_out), _ptr(cnt_out))
        self._check(st, "fdl_track_topk")

    def unmask_verify(self, B: int, max_search: int, *, logits=None, row_seq=None, row_pos=None,
                      eps: float = 0.9, force_progress: bool = False, conf=None, argmax=None, commit=None,
                      search_rows=None, n_search=None, mask_logits=None, draft_tok=None, gamma: float = 0.8,
                      accept=None, n_accept=None, mask_conf=None, mask_argmax=None) -> None:
        a = fdl_unmask_args()
        a.B, a.max_search = int(B), int(max_search)
        a.logits = _ptr(logits)
        a.R_w = int(logits.shape[0]) if logits is not None else 0
        a.row_seq, a.row_pos = _ptr(row_seq), _ptr(row_pos)
        a.eps, a.force_progress = float(eps), int(bool(force_progress))
        a.conf, a.argmax, a.commit = _ptr(conf), _ptr(argmax), _ptr(commit)
        a.search_rows, a.n_search = _ptr(search_rows), _ptr(n_search)
        a.mask_logits, a.draft_tok, a.gamma = _ptr(mask_logits), _ptr(draft_tok), float(gamma)
        a.accept, a.n_accept = _ptr(accept), _ptr(n_accept)
        a.mask_conf, a.mask_argmax = _ptr(mask_conf), _ptr(mask_argmax)
        self._check(load_library().fdl_unmask_verify(self.handle, ctypes.byref(a)), "fdl_unmask_verify")

    def lm_head_unmask(self, hidden, w_lm, B: int, max_search: int, *, row_seq, row_pos, eps: float = 0.9,
                       force_progress: bool = False, conf, argmax, commit, search_rows, n_search) -> None:
        """Unmask-phase decisions straight from the window rows' hidden states
        (hidden [R_w, d_model], w_lm [vocab, d_model], both bf16)."""
        a = fdl_unmask_args()
        a.B, a.max_search = int(B), int(max_search)
        a.R_w = int(hidden.shape[0])
        a.row_seq, a.row_pos = _ptr(row_seq), _ptr(row_pos)
        a.eps, a.force_progress = float(eps), int(bool(force_progress))
        a.conf, a.argmax, a.commit = _ptr(conf), _ptr(argmax), _ptr(commit)
        a.search_rows, a.n_search = _ptr(search_rows), _ptr(n_search)
        self._check(load_library().fdl_lm_head_unmask(self.handle, _ptr(hidden), _ptr(w_lm), ctypes.byref(a)),
                    "fdl_lm_head_unmask")

    def model_workspace_bytes(self, ffn: int, R: int) -> int:
        return int(load_library().fdl_model_workspace_bytes(self.handle, int(ffn), int(R)))

    def flash_workspace_bytes(self, ffn: int, params: dict, B: int, max_seq: int) -> int:
        return int(load_library().fdl_flash_workspace_bytes(self.handle, int(ffn), ctypes.byref(_flash_params(params)),
                                                            int(B), int(max_seq)))

    def flash_step(self, model: dict, w_lm, k_caches, v_caches, block_table, params: dict, seqs: dict, workspace,
                   trace: bool = True):
        """One denoising step (see include/fdl.h). ``seqs``: dict of host numpy
        arrays prompt_len, seq_len (int32 [B]), tokens (int32 [B, max_seq]),
        masked (uint8 [B, max_seq]), tracked (int32 [B, track_budget]),
        n_tracked and state (int32 [B]); the last five are updated in place.
        Returns the step's record as a dict of numpy arrays (or None)."""
        import numpy as np
        m, keep = _model_struct(model)
        kc, vc = _ptr_array(k_caches), _ptr_array(v_caches)
        pr = _flash_params(params)
        B, N = int(seqs["tokens"].shape[0]), int(seqs["tokens"].shape[1])
        sq = fdl_flash_seqs()
        sq.B, sq.max_seq = B, N
        for name, dt in (("prompt_len", np.int32), ("seq_len", np.int32), ("tokens", np.int32), ("masked", np.uint8),
                         ("tracked", np.int32), ("n_tracked", np.int32), ("state", np.int32)):
            _, ptr = _host(seqs[name], dt, name, writable=True)
            setattr(sq, name, ptr)
        rec, tr = None, None
        if trace:
            W, MS = int(params["window"]), max(1, int(params["max_search"]))
            rec = dict(n_rows=np.zeros(2, np.int32), n_window=np.zeros(1, np.int32),
                       window_seq=np.zeros(B * W, np.int32), window_pos=np.zeros(B * W, np.int32),
                       conf=np.zeros(B * W, np.float32), argmax=np.zeros(B * W, np.int32),
                       commit=np.zeros(B * W, np.uint8), search_rows=np.full(B * MS, -1, np.int32),
                       n_search=np.zeros(B, np.int32), mask_conf=np.zeros(B * MS, np.float32),
                       mask_argmax=np.zeros(B * MS, np.int32), n_accept=np.zeros(B, np.int32),
                       track=np.zeros(B * N, np.float32))
            tr = fdl_flash_trace(**{k: v.ctypes.data for k, v in rec.items()})
            import torch
            finals = [torch.empty((self.cfg.max_rows, self.cfg.d_model), dtype=torch.bfloat16, device="cuda")
                      for _ in range(2)]
            tr.draft_final, tr.verify_final = finals[0].data_ptr(), finals[1].data_ptr()
        st = load_library().fdl_flash_step(
            self.handle, ctypes.byref(m), _ptr(w_lm), kc, vc, _ptr(block_table), int(block_table.shape[-1]),
            ctypes.byref(pr), ctypes.byref(sq), ctypes.byref(tr) if tr is not None else None, _ptr(workspace),
            int(workspace.numel() * workspace.element_size()))
        del keep
        self._check(st, "fdl_flash_step")
        if rec is not None:
            n0, n1 = int(rec["n_rows"][0]), int(rec["n_rows"][1])
            rec["draft_final"] = finals[0][:n0].float().cpu().numpy()
            rec["verify_final"] = finals[1][:n1].float().cpu().numpy()
        return rec

    def model_forward(self, model: dict, tokens, row_seq, row_rope_pos, row_cache_pos, row_kind, cu_seqlens_q,
                      kv_len, block_table, k_caches, v_caches, workspace, final_out, search_pos=None,
                      n_search=None, track_scores=None) -> None:
        """Whole-model forward over the rows. ``model``: dict with ffn, eps,
        embed, g_final and layers (dicts with g_attn, w_qkv, w_o, g_mlp, w_gu,
        w_down), all bf16 device tensors; k_caches / v_caches: one tensor per
        layer; workspace: a uint8 device tensor of model_workspace_bytes."""
        m, keep = _model_struct(model)
        kc, vc = _ptr_array(k_caches), _ptr_array(v_caches)
        B = int(kv_len.shape[0])
        R = int(tokens.shape[0])
        search_ld = int(search_pos.shape[-1]) if search_pos is not None else 0
        track_ld = int(track_scores.shape[-1]) if track_scores is not None else 0
        st = load_library().fdl_model_forward(
            self.handle, ctypes.byref(m), _ptr(tokens), R, _ptr(row_seq), _ptr(row_rope_pos), _ptr(row_cache_pos),
            _ptr(row_kind), _ptr(cu_seqlens_q), _ptr(kv_len), B, _ptr(block_table), int(block_table.shape[-1]),
            kc, vc, _ptr(search_pos), search_ld, _ptr(n_search),
            _ptr(track_scores), track_ld, _ptr(workspace), int(workspace.numel() * workspace.element_size()),
            _ptr(final_out))
        self._check(st, "fdl_model_forward")

    def lm_head_verify(self, mask_hidden, w_lm, B: int, max_search: int, *, n_search, draft_tok,
                       gamma: float = 0.8, accept, n_accept, mask_conf, mask_argmax) -> None:
        """Verify acceptance straight from the mask views' hidden states
        (mask_hidden [B*max_search, d_model], w_lm [vocab, d_model], both bf16)."""
        a = fdl_unmask_args()
        a.B, a.max_search = int(B), int(max_search)
        a.n_search, a.draft_tok, a.gamma = _ptr(n_search), _ptr(draft_tok), float(gamma)
        a.accept, a.n_accept = _ptr(accept), _ptr(n_accept)
        a.mask_conf, a.mask_argmax = _ptr(mask_conf), _ptr(mask_argmax)
        self._check(load_library().fdl_lm_head_verify(self.handle, _ptr(mask_hidden), _ptr(w_lm), ctypes.byref(a)),
                    "fdl_lm_head_verify")


def _ptr_array(tensors):
    """Host array of device pointers (kept alive by the caller)."""
    arr = (ctypes.c_void_p * len(tensors))(*[_ptr(t) for t in tensors])
    return ctypes.cast(arr, _PP)


def _model_struct(model: dict):
    """fdl_model for a dict of device tensors, and the pointer arrays it references."""
    layers = model["layers"]
    keep = {k: (ctypes.c_void_p * len(layers))(*[_ptr(w[k]) for w in layers])
            for k in ("g_attn", "w_qkv", "w_o", "g_mlp", "w_gu", "w_down")}
    m = fdl_model()
    m.n_layers, m.ffn, m.rms_eps = len(layers), int(model["ffn"]), float(model["eps"])
    m.embed, m.g_final = _ptr(model["embed"]), _ptr(model["g_final"])
    for k, a in keep.items():
        setattr(m, k, ctypes.cast(a, _PP))
    return m, keep


def _flash_params(params: dict) -> fdl_flash_params:
    pr = fdl_flash_params()
    pr.window, pr.track_budget, pr.max_search = int(params["window"]), int(params["track_budget"]), \
        int(params["max_search"])
    pr.eps, pr.gamma = float(params["eps"]), float(params["gamma"])
    pr.force_progress, pr.mask_token = int(bool(params["force_progress"])), int(params["mask_id"])
    return pr


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def fdl_create(d_model: int, n_heads: int, head_dim: int, rope_theta: float, max_batch: int, max_seq: int,
               max_views: int, page_size: int, n_pages: int, max_rows: int, vocab: int, dtype: str,
               stream=None) -> Context:
    """Creates a context on the current device (dtype 'f32' or 'bf16')."""
    L = load_library()
    cfg = fdl_config(d_model, n_heads, head_dim, float(rope_theta), max_batch, max_seq, max_views,
                     page_size, n_pages, max_rows, vocab, FDL_BF16 if dtype == "bf16" else FDL_F32)
    h = ctypes.c_void_p()
    st = L.fdl_create(ctypes.byref(cfg), _stream_handle(stream), ctypes.byref(h))
    if st != FDL_OK:
        raise FdlError(st, "fdl_create failed (see stderr for the rejected limit)")
    return Context(h.value, cfg)


# C-named module functions over a Context.
def fdl_destroy(ctx: Context) -> None:
    ctx.close()


def fdl_sync_status(ctx: Context) -> None:
    ctx.sync_status()


def fdl_qkv_rope_cache_write(ctx: Context, *a, **k) -> None:
    ctx.qkv_rope_cache_write(*a, **k)


def fdl_sched_attn(ctx: Context, *a, **k) -> None:
    ctx.sched_attn(*a, **k)


def fdl_track_topk(ctx: Context, *a, **k) -> None:
    ctx.track_topk(*a, **k)


def fdl_unmask_verify(ctx: Context, *a, **k) -> None:
    ctx.unmask_verify(*a, **k)


def fdl_lm_head_unmask(ctx: Context, *a, **k) -> None:
    ctx.lm_head_unmask(*a, **k)


def fdl_lm_head_verify(ctx: Context, *a, **k) -> None:
    ctx.lm_head_verify(*a, **k)


def fdl_model_workspace_bytes(ctx: Context, ffn: int, R: int) -> int:
    return ctx.model_workspace_bytes(ffn, R)


def fdl_model_forward(ctx: Context, *a, **k) -> None:
    ctx.model_forward(*a, **k)


def fdl_flash_workspace_bytes(ctx: Context, *a, **k) -> int:
    return ctx.flash_workspace_bytes(*a, **k)


def fdl_flash_step(ctx: Context, *a, **k):
    return ctx.flash_step(*a, **k)


def fdl_sched_attn_noalloc(cfg: fdl_config, q, k_cache, v_cache, block_table, cu_seqlens_q, kv_len, row_kind,
                           o_out, lse_out=None, track_scores=None, search_pos=None, n_search=None,
                           device_error=None, stream=None) -> None:
    """Scheduled attention with no device allocation (no context needed).

    For callers that cannot allocate device memory; see include/fdl.h for
    the static-scratch limits and the serialisation rule.
    """
    B = int(kv_len.shape[0])
    R = int(q.shape[0])
    search_ld = int(search_pos.shape[-1]) if search_pos is not None else 0
    track_ld = int(track_scores.shape[-1]) if track_scores is not None else 0
    st = load_library().fdl_sched_attn_noalloc(
        ctypes.byref(cfg), _stream_handle(stream), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        int(block_table.shape[-1]), _ptr(cu_seqlens_q), _ptr(kv_len), B, R, _ptr(row_kind), _ptr(search_pos),
        search_ld, _ptr(n_search), _ptr(o_out), _ptr(lse_out), _ptr(track_scores), track_ld, _ptr(device_error))
    if st != FDL_OK:
        raise FdlError(st, "fdl_sched_attn_noalloc (reason on stderr)")


# Host row builders (numpy arrays in and out; no GPU involved).
class Rows:
    """Row descriptors of one call (int32 numpy arrays)."""

    def __init__(self, row_seq, row_rope_pos, row_cache_pos, row_kind, cu_seqlens):
        self.row_seq, self.row_rope_pos, self.row_cache_pos = row_seq, row_rope_pos, row_cache_pos
        self.row_kind, self.cu_seqlens = row_kind, cu_seqlens

    @property
    def n_rows(self) -> int:
        return int(self.row_seq.shape[0])


def _host(a, dtype, name: str, writable: bool = False):
    """Contiguous host array of ``dtype`` and its address (None stays NULL)."""
    import numpy as np
    if a is None:
        return None, None
    if writable:
        if not (isinstance(a, np.ndarray) and a.dtype == dtype and a.flags.c_contiguous):
            raise FdlError(FDL_ERR_INVALID_ARG, f"{name} must be a contiguous {np.dtype(dtype).name} numpy array")
        arr = a
    else:
        arr = np.ascontiguousarray(a, dtype=dtype)
    return arr, arr.ctypes.data


def fdl_refresh_rows(policy: int, prompt_len, seq_len, masked, block: int, state, tracked=None,
                     n_tracked=None, max_rows: int | None = None) -> Rows:
    """Rows of one step under a refresh policy (see include/fdl.h).

    ``masked`` is uint8 [B, max_seq]; ``state`` an int32 numpy array [B]
    (-1 before the first step) that the call updates in place; ``tracked``
    int32 [B, ld] and ``n_tracked`` [B] for FDL_REFRESH_FLASH_DRAFT.
    """
    import numpy as np
    m, mp = _host(masked, np.uint8, "masked")
    pl, plp = _host(prompt_len, np.int32, "prompt_len")
    sl, slp = _host(seq_len, np.int32, "seq_len")
    _, stp = _host(state, np.int32, "state", writable=True)
    tr, trp = _host(tracked, np.int32, "tracked")
    _, ntp = _host(n_tracked, np.int32, "n_tracked")
    B, max_seq = int(m.shape[0]), int(m.shape[1])
    if max_rows is None:
        max_rows = int(sl.sum()) + (int(tr.size) if tr is not None else 0)
    out = [np.empty(max(max_rows, 1), np.int32) for _ in range(4)]
    cu = np.empty(B + 1, np.int32)
    n = np.zeros(1, np.int32)
    a = fdl_refresh_args()
    a.policy, a.B, a.max_seq, a.block = int(policy), B, max_seq, int(block)
    a.prompt_len, a.seq_len, a.masked, a.state = plp, slp, mp, stp
    a.tracked, a.tracked_ld = trp, int(tr.shape[-1]) if tr is not None else 0
    a.n_tracked, a.max_rows = ntp, int(max_rows)
    a.row_seq, a.row_rope_pos, a.row_cache_pos, a.row_kind = (o.ctypes.data for o in out)
    a.cu_seqlens, a.n_rows = cu.ctypes.data, n.ctypes.data
    st = load_library().fdl_refresh_rows(ctypes.byref(a))
    if st != FDL_OK:
        raise FdlError(st, "fdl_refresh_rows rejected its arguments")
    r = int(n[0])
    return Rows(*(o[:r] for o in out), cu)


def fdl_verify_rows(seq_len, tracked, n_tracked, search_pos, n_search, query_budget: int,
                    max_rows: int | None = None) -> Rows:
    """Rows of a Flash-Verify forward (see include/fdl.h); int32 host arrays."""
    import numpy as np
    sl, slp = _host(seq_len, np.int32, "seq_len")
    tr, trp = _host(tracked, np.int32, "tracked")
    _, ntp = _host(n_tracked, np.int32, "n_tracked")
    sp, spp = _host(search_pos, np.int32, "search_pos")
    _, nsp = _host(n_search, np.int32, "n_search")
    B = int(sl.shape[0])
    if max_rows is None:
        max_rows = int(tr.size) + 2 * int(sp.size)
    out = [np.empty(max(max_rows, 1), np.int32) for _ in range(4)]
    cu = np.empty(B + 1, np.int32)
    n = np.zeros(1, np.int32)
    st = load_library().fdl_verify_rows(B, slp, trp, int(tr.shape[-1]), ntp, spp, int(sp.shape[-1]), nsp,
                                        int(query_budget), int(max_rows), *(o.ctypes.data for o in out),
                                        cu.ctypes.data, n.ctypes.data)
    if st != FDL_OK:
        raise FdlError(st, "fdl_verify_rows rejected its arguments")
    r = int(n[0])
    return Rows(*(o[:r] for o in out), cu)
