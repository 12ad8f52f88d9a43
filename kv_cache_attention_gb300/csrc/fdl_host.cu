// C-ABI surface of libfdl: context lifetime, host-side validation, status.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "fdl_internal.cuh"

bool fdl_attn_tc_supported(const fdl_config& c);

namespace {

fdl_status fail(fdl_ctx* ctx, fdl_status st, const char* fmt, ...) {
  if (ctx) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(ctx->last_error, sizeof(ctx->last_error), fmt, ap);
    va_end(ap);
  }
  return st;
}

fdl_status cuda_fail(fdl_ctx* ctx, cudaError_t e, const char* what) {
  return fail(ctx, FDL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

fdl_status launched(fdl_ctx* ctx, cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
  ctx->last_error[0] = 0;
  return FDL_OK;
}

}  // namespace

bool fdl_config_ok(const fdl_config* c, char* why, size_t n) {
#define FDL_REQ(cond, msg)          \
  if (!(cond)) {                    \
    snprintf(why, n, "%s", msg);    \
    return false;                   \
  }
  FDL_REQ(c->n_heads > 0 && c->head_dim > 0, "n_heads and head_dim must be positive");
  FDL_REQ(c->d_model == c->n_heads * c->head_dim, "d_model must equal n_heads * head_dim");
  FDL_REQ(c->head_dim == 64 || c->head_dim == 128, "head_dim must be 64 or 128");
  FDL_REQ(c->d_model % 8 == 0, "d_model must be a multiple of 8");
  FDL_REQ(c->rope_theta > 1.0, "rope_theta must exceed 1");
  FDL_REQ(c->max_batch > 0 && c->max_seq > 0 && c->max_rows > 0, "max_batch, max_seq, max_rows must be positive");
  FDL_REQ(c->max_views >= 0 && c->max_views % 2 == 0 && c->max_views <= 512,
          "max_views must be even and in [0, 512]");
  FDL_REQ(c->page_size > 0 && c->n_pages > 0, "page_size and n_pages must be positive");
  FDL_REQ(c->vocab > 0, "vocab must be positive");
  FDL_REQ(c->dtype == FDL_F32 || c->dtype == FDL_BF16, "dtype must be FDL_F32 or FDL_BF16");
  FDL_REQ((long long)c->max_seq + c->max_views < (1LL << 30), "max_seq + max_views too large");
#undef FDL_REQ
  return true;
}

bool fdl_pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("FDL_DISABLE_PDL");
    return !(v && v[0] && v[0] != '0');
  }();
  return on;
}

extern "C" {

fdl_status fdl_create(const fdl_config* cfg, void* cuda_stream, fdl_ctx** out) {
  if (!cfg || !out) return FDL_ERR_INVALID_ARG;
  *out = nullptr;
  char why[256];
  if (!fdl_config_ok(cfg, why, sizeof(why))) {
    fprintf(stderr, "fdl_create: %s\n", why);
    return FDL_ERR_INVALID_ARG;
  }
  fdl_ctx* ctx = (fdl_ctx*)calloc(1, sizeof(fdl_ctx));
  if (!ctx) return FDL_ERR_OOM;
  ctx->cfg = *cfg;
  ctx->stream = (cudaStream_t)cuda_stream;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    free(ctx);
    return FDL_ERR_CUDA;
  }
  // RoPE table in double on the host: angle(p, i) = p * theta^(-2i/hd).
  const int half = cfg->head_dim / 2;
  ctx->rope_positions = cfg->max_seq + cfg->max_views;
  size_t n_tab = (size_t)ctx->rope_positions * half;
  std::vector<float> hc(n_tab), hs(n_tab);
  for (int i = 0; i < half; ++i) {
    double inv = pow(cfg->rope_theta, -2.0 * i / cfg->head_dim);
    for (int p = 0; p < ctx->rope_positions; ++p) {
      double a = (double)p * inv;
      hc[(size_t)p * half + i] = (float)cos(a);
      hs[(size_t)p * half + i] = (float)sin(a);
    }
  }
  ctx->attn_tile_m = fdl_attn_tc_supported(*cfg) ? FDL_TILE_M_TC : FDL_TILE_M_SIMT;
  ctx->worklist_items = (cfg->max_rows + ctx->attn_tile_m - 1) / ctx->attn_tile_m + cfg->max_batch;
  cudaError_t e = cudaSuccess;
  e = e ? e : cudaMalloc(&ctx->rope_cos, n_tab * sizeof(float));
  e = e ? e : cudaMalloc(&ctx->rope_sin, n_tab * sizeof(float));
  e = e ? e : cudaMalloc(&ctx->err_word, sizeof(unsigned));
  e = e ? e : cudaMalloc(&ctx->worklist, (1 + 4 * (size_t)ctx->worklist_items) * sizeof(int));
  e = e ? e : cudaMalloc(&ctx->n_masked, cfg->max_batch * sizeof(int));
  e = e ? e : cudaMalloc(&ctx->tickets, 8 * sizeof(unsigned));
  if (cfg->dtype == FDL_BF16) {
    ctx->qkv_partial_floats = fdl_qkv_partial_floats(ctx->num_sms, cfg->max_rows);
    ctx->qkv_tickets = 4 * ctx->num_sms;
    e = e ? e : cudaMalloc(&ctx->qkv_partials, ctx->qkv_partial_floats * sizeof(float));
    e = e ? e : cudaMalloc(&ctx->qkv_ticket_buf, ctx->qkv_tickets * sizeof(unsigned));
    e = e ? e : cudaMemset(ctx->qkv_ticket_buf, 0, ctx->qkv_tickets * sizeof(unsigned));
    ctx->lm_part_floats = fdl_lm_partial_floats(ctx->num_sms, cfg->max_rows);
    e = e ? e : cudaMalloc(&ctx->lm_part, ctx->lm_part_floats * sizeof(float));
    ctx->lm_rt_ticket_count = fdl_lm_row_tiles(cfg->max_rows);
    e = e ? e : cudaMalloc(&ctx->lm_rt_tickets, ctx->lm_rt_ticket_count * sizeof(unsigned));
    e = e ? e : cudaMemset(ctx->lm_rt_tickets, 0, ctx->lm_rt_ticket_count * sizeof(unsigned));
  }
  if (ctx->attn_tile_m == FDL_TILE_M_TC) {
    // the deterministic tracker's partial column sums and tickets
    ctx->trk_ld = (cfg->max_seq + 3) / 4 * 4;
    const size_t trk = (size_t)cfg->max_batch * FDL_TRK_SLOTS * cfg->n_heads * ctx->trk_ld;
    e = e ? e : cudaMalloc(&ctx->trk_part, trk * sizeof(float));
    e = e ? e : cudaMalloc(&ctx->trk_nslots, (size_t)cfg->max_batch * sizeof(int));
  }
  e = e ? e : cudaMemcpy(ctx->rope_cos, hc.data(), n_tab * sizeof(float), cudaMemcpyHostToDevice);
  e = e ? e : cudaMemcpy(ctx->rope_sin, hs.data(), n_tab * sizeof(float), cudaMemcpyHostToDevice);
  e = e ? e : cudaMemset(ctx->err_word, 0, sizeof(unsigned));
  e = e ? e : cudaMemset(ctx->tickets, 0, 8 * sizeof(unsigned));
  if (e != cudaSuccess) {
    fdl_destroy(ctx);
    return e == cudaErrorMemoryAllocation ? FDL_ERR_OOM : FDL_ERR_CUDA;
  }
  *out = ctx;
  return FDL_OK;
}

void fdl_destroy(fdl_ctx* ctx) {
  if (!ctx) return;
  cudaFree(ctx->rope_cos);
  cudaFree(ctx->rope_sin);
  cudaFree(ctx->err_word);
  cudaFree(ctx->worklist);
  cudaFree(ctx->n_masked);
  cudaFree(ctx->tickets);
  cudaFree(ctx->qkv_partials);
  cudaFree(ctx->qkv_ticket_buf);
  cudaFree(ctx->lm_part);
  cudaFree(ctx->lm_rt_tickets);
  cudaFree(ctx->trk_part);
  cudaFree(ctx->trk_nslots);
  free(ctx);
}

fdl_status fdl_set_stream(fdl_ctx* ctx, void* cuda_stream) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  ctx->stream = (cudaStream_t)cuda_stream;
  return FDL_OK;
}

fdl_status fdl_set_wait_budget(fdl_ctx* ctx, long long cycles) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (cycles < 0) return fail(ctx, FDL_ERR_INVALID_ARG, "wait budget must be >= 0");
  ctx->wait_budget = cycles;
  return FDL_OK;
}

const char* fdl_last_error(const fdl_ctx* ctx) { return ctx ? ctx->last_error : "null context"; }

fdl_status fdl_sync_status(fdl_ctx* ctx) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  unsigned w = 0;
  e = cudaMemcpy(&w, ctx->err_word, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "read error word");
  if (w) {
    e = cudaMemset(ctx->err_word, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(ctx, e, "clear error word");
  }
  if (w & FDL_DEVERR_TIMEOUT) return fail(ctx, FDL_ERR_TIMEOUT, "a bounded device wait gave up (word 0x%x)", w);
  if (w) return fail(ctx, FDL_ERR_DEVICE_INDEX, "device index/shape error (word 0x%x)", w);
  return FDL_OK;
}

int fdl_tile_m(const fdl_ctx* ctx) {
  if (!ctx) return 0;
  return ctx->attn_tile_m;
}

int fdl_worklist_capacity(const fdl_ctx* ctx, int R, int B) {
  if (!ctx || R < 0 || B < 0) return 0;
  int t = fdl_tile_m(ctx);
  return 1 + 4 * ((R + t - 1) / t + B);
}

fdl_status fdl_qkv_rope_cache_write(fdl_ctx* ctx, const void* X, const void* Wqkv, int R,
                                    const int* row_seq, const int* row_rope_pos,
                                    const int* row_cache_pos, const int* block_table, int bt_stride,
                                    void* k_cache, void* v_cache, void* q_out) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (R < 0 || R > ctx->cfg.max_rows)
    return fail(ctx, FDL_ERR_INVALID_ARG, "R=%d outside [0, max_rows=%d]", R, ctx->cfg.max_rows);
  if (R == 0) return FDL_OK;
  if (!X || !Wqkv || !row_seq || !row_rope_pos || !row_cache_pos || !block_table || !k_cache ||
      !v_cache || !q_out)
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_qkv_rope_cache_write: NULL pointer argument");
  if (bt_stride <= 0) return fail(ctx, FDL_ERR_INVALID_ARG, "bt_stride must be positive");
  return launched(ctx, fdl_launch_qkv(ctx, X, Wqkv, R, row_seq, row_rope_pos, row_cache_pos,
                                      block_table, bt_stride, k_cache, v_cache, q_out),
                  "qkv launch");
}

fdl_status fdl_sched_attn(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                          const int* block_table, int bt_stride, const int* cu_seqlens_q,
                          const int* kv_len, int B, int R, const int* row_kind,
                          const int* search_pos, int search_ld, const int* n_search, void* o_out,
                          float* lse_out, float* track_scores, int track_ld, int* worklist_out) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (B < 0 || B > ctx->cfg.max_batch)
    return fail(ctx, FDL_ERR_INVALID_ARG, "B=%d outside [0, max_batch=%d]", B, ctx->cfg.max_batch);
  if (R < 0 || R > ctx->cfg.max_rows)
    return fail(ctx, FDL_ERR_INVALID_ARG, "R=%d outside [0, max_rows=%d]", R, ctx->cfg.max_rows);
  if (B == 0 || R == 0) return FDL_OK;
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !kv_len || !row_kind || !o_out)
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_sched_attn: NULL pointer argument");
  if (bt_stride <= 0) return fail(ctx, FDL_ERR_INVALID_ARG, "bt_stride must be positive");
  if (search_pos && (!n_search || search_ld <= 0))
    return fail(ctx, FDL_ERR_INVALID_ARG, "search_pos needs n_search and search_ld > 0");
  if (search_pos && ctx->cfg.max_views == 0)
    return fail(ctx, FDL_ERR_INVALID_ARG, "search_pos given but the context has max_views = 0");
  if (track_scores && track_ld < ctx->cfg.max_seq)
    return fail(ctx, FDL_ERR_INVALID_ARG, "track_ld=%d below max_seq=%d", track_ld, ctx->cfg.max_seq);
  return launched(ctx, fdl_launch_attn(ctx, q, k_cache, v_cache, block_table, bt_stride, cu_seqlens_q,
                                       kv_len, B, R, row_kind, search_pos, search_ld, n_search, o_out,
                                       lse_out, track_scores, track_ld, worklist_out),
                  "attention launch");
}

fdl_status fdl_track_topk(fdl_ctx* ctx, const float* scores, const unsigned char* eligible, int ld,
                          const int* seq_len, int B, int k, int* idx_out, int* cnt_out) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (B < 0 || B > ctx->cfg.max_batch)
    return fail(ctx, FDL_ERR_INVALID_ARG, "B=%d outside [0, max_batch=%d]", B, ctx->cfg.max_batch);
  if (k < 1 || k > 1024) return fail(ctx, FDL_ERR_INVALID_ARG, "k=%d outside [1, 1024]", k);
  if (ld <= 0) return fail(ctx, FDL_ERR_INVALID_ARG, "ld must be positive");
  if (!scores || !eligible || !seq_len || !idx_out || !cnt_out)
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_track_topk: NULL pointer argument");
  if (B == 0) return FDL_OK;
  return launched(ctx, fdl_launch_topk(ctx, scores, eligible, ld, seq_len, B, k, idx_out, cnt_out),
                  "top-k launch");
}

fdl_status fdl_unmask_verify(fdl_ctx* ctx, const fdl_unmask_args* a) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (!a) return fail(ctx, FDL_ERR_INVALID_ARG, "NULL args");
  if (a->B < 1 || a->B > ctx->cfg.max_batch)
    return fail(ctx, FDL_ERR_INVALID_ARG, "B=%d outside [1, max_batch=%d]", a->B, ctx->cfg.max_batch);
  if (a->max_search < 0 || a->max_search > 1024)
    return fail(ctx, FDL_ERR_INVALID_ARG, "max_search=%d outside [0, 1024]", a->max_search);
  if (a->logits) {
    if (a->R_w < 0 || a->R_w > ctx->cfg.max_rows)
      return fail(ctx, FDL_ERR_INVALID_ARG, "R_w=%d outside [0, max_rows=%d]", a->R_w, ctx->cfg.max_rows);
    if (!a->row_seq || !a->row_pos || !a->conf || !a->argmax || !a->commit || !a->n_search ||
        (a->max_search > 0 && !a->search_rows))
      return fail(ctx, FDL_ERR_INVALID_ARG, "unmask phase: NULL pointer argument");
    if (!(a->eps >= 0.f && a->eps <= 1.f)) return fail(ctx, FDL_ERR_INVALID_ARG, "eps outside [0,1]");
  }
  if (a->mask_logits) {
    if (!a->draft_tok || !a->accept || !a->n_accept || !a->n_search || !a->mask_conf || !a->mask_argmax)
      return fail(ctx, FDL_ERR_INVALID_ARG, "verify phase: NULL pointer argument");
    if (!(a->gamma >= 0.f && a->gamma <= 1.f)) return fail(ctx, FDL_ERR_INVALID_ARG, "gamma outside [0,1]");
    if (a->max_search == 0) return fail(ctx, FDL_ERR_INVALID_ARG, "verify phase needs max_search > 0");
  }
  if (!a->logits && !a->mask_logits) return FDL_OK;
  return launched(ctx, fdl_launch_unmask_verify(ctx, a), "unmask/verify launch");
}

fdl_status fdl_lm_head_unmask(fdl_ctx* ctx, const void* hidden, const void* w_lm, const fdl_unmask_args* a) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (!a || !hidden || !w_lm) return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_lm_head_unmask: NULL argument");
  if (a->logits || a->mask_logits)
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_lm_head_unmask: logits and mask_logits must be NULL");
  if (ctx->cfg.dtype != FDL_BF16)
    return fail(ctx, FDL_ERR_UNSUPPORTED, "fdl_lm_head_unmask: bf16 contexts only");
  if (a->B < 1 || a->B > ctx->cfg.max_batch)
    return fail(ctx, FDL_ERR_INVALID_ARG, "B=%d outside [1, max_batch=%d]", a->B, ctx->cfg.max_batch);
  if (a->R_w < 1 || a->R_w > ctx->cfg.max_rows)
    return fail(ctx, FDL_ERR_INVALID_ARG, "R_w=%d outside [1, max_rows=%d]", a->R_w, ctx->cfg.max_rows);
  if (a->max_search < 0 || a->max_search > 1024)
    return fail(ctx, FDL_ERR_INVALID_ARG, "max_search=%d outside [0, 1024]", a->max_search);
  if (!a->row_seq || !a->row_pos || !a->conf || !a->argmax || !a->commit || !a->n_search ||
      (a->max_search > 0 && !a->search_rows))
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_lm_head_unmask: NULL output or row argument");
  if (!(a->eps >= 0.f && a->eps <= 1.f)) return fail(ctx, FDL_ERR_INVALID_ARG, "eps outside [0,1]");
  if (ctx->cfg.d_model % 64 != 0)
    return fail(ctx, FDL_ERR_UNSUPPORTED, "fdl_lm_head_unmask: d_model must be a multiple of 64");
  return launched(ctx, fdl_launch_lm_head(ctx, hidden, w_lm, a, false), "LM-head unmask launch");
}

fdl_status fdl_lm_head_verify(fdl_ctx* ctx, const void* mask_hidden, const void* w_lm, const fdl_unmask_args* a) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (!a || !mask_hidden || !w_lm) return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_lm_head_verify: NULL argument");
  if (a->logits || a->mask_logits)
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_lm_head_verify: logits and mask_logits must be NULL");
  if (ctx->cfg.dtype != FDL_BF16)
    return fail(ctx, FDL_ERR_UNSUPPORTED, "fdl_lm_head_verify: bf16 contexts only");
  if (a->B < 1 || a->B > ctx->cfg.max_batch)
    return fail(ctx, FDL_ERR_INVALID_ARG, "B=%d outside [1, max_batch=%d]", a->B, ctx->cfg.max_batch);
  if (a->max_search < 1 || a->max_search > 1024)
    return fail(ctx, FDL_ERR_INVALID_ARG, "max_search=%d outside [1, 1024]", a->max_search);
  if ((long long)a->B * a->max_search > ctx->cfg.max_rows)
    return fail(ctx, FDL_ERR_INVALID_ARG, "B*max_search=%lld above max_rows=%d mask-view rows",
                (long long)a->B * a->max_search, ctx->cfg.max_rows);
  if (!a->n_search || !a->draft_tok || !a->accept || !a->n_accept || !a->mask_conf || !a->mask_argmax)
    return fail(ctx, FDL_ERR_INVALID_ARG, "fdl_lm_head_verify: NULL output or input argument");
  if (!(a->gamma >= 0.f && a->gamma <= 1.f)) return fail(ctx, FDL_ERR_INVALID_ARG, "gamma outside [0,1]");
  if (ctx->cfg.d_model % 64 != 0)
    return fail(ctx, FDL_ERR_UNSUPPORTED, "fdl_lm_head_verify: d_model must be a multiple of 64");
  return launched(ctx, fdl_launch_lm_head(ctx, mask_hidden, w_lm, a, true), "LM-head verify launch");
}

}  // extern "C"
