// One Flash-dLLM denoising step of a whole model on a batch of sequences:
// paper digest, "Method steps in detail", Algorithm 2 steps 2-4.
//
//   draft forward   the tracked set T^t and the masked window (the first
//                   step: every position, which fills the caches as step 1
//                   does) through every layer, with the Eq. (2) tracker;
//   unmask          the window rows' confidences and predictions from the
//                   fused LM head; c >= eps is decoded (D^t), the rest,
//                   most confident first, is the search set S^t;
//   verify forward  the shrunk tracked set T_v and a draft view and a mask
//                   view per search token; the fused LM head takes the
//                   acceptance walk on the mask views;
//   update          committed and accepted tokens are written into the
//                   sequences; T^{t+1} = the newly decoded tokens, then the
//                   top-k of the other decoded positions by tracker score.
//
// The host code here only sequences the library's own entry points and
// keeps the per-sequence bookkeeping (the row sets come from the host row
// builders); every arithmetic step runs in the kernels. It synchronises the
// stream three times per step, to read the decisions that shape the next
// part of the step.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "fdl_model.cuh"

namespace {

constexpr int kGatherThreads = 256;

// dst[i, :] = src[idx[i], :] (bf16 rows of d elements); idx < 0 gives zeros
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                                     const int* __restrict__ idx, int d,
                                                                     __nv_bfloat16* __restrict__ dst) {
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int i = blockIdx.x;
  const int r = idx[i];
  for (int c = threadIdx.x; c < d; c += kGatherThreads)
    dst[(size_t)i * d + c] = r >= 0 ? src[(size_t)r * d + c] : __float2bfloat16_rn(0.f);
}

fdl_status loop_fail(fdl_ctx* ctx, fdl_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(ctx->last_error, sizeof(ctx->last_error), fmt, ap);
  va_end(ap);
  return st;
}

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

// Device scratch of one step, carved from the caller's workspace.
struct Scratch {
  int *seq, *rope, *cache, *kind, *tok, *cu, *kv_len, *spos, *nsearch, *gidx, *wseq, *wpos, *draft, *tk_idx,
      *tk_cnt, *argmax, *srows, *m_arg, *n_acc;
  float *track, *conf, *m_conf;
  unsigned char *commit, *accept, *elig;
  __nv_bfloat16 *final_rows, *gathered;
  void* model_ws;
  size_t model_ws_bytes;
  size_t bytes;
};

Scratch carve(char* base, const fdl_ctx* ctx, int ffn, const fdl_flash_params* p, int B, int max_seq) {
  Scratch s{};
  size_t off = 0;
  auto take = [&](size_t n) {
    char* q = base ? base + off : nullptr;
    off += al(n);
    return q;
  };
  const int R = ctx->cfg.max_rows, d = ctx->cfg.d_model;
  const int nw = B * p->window, ns = B * p->max_search, nt = B * p->track_budget;
  auto I = [&](size_t n) { return reinterpret_cast<int*>(take(n * 4)); };
  s.seq = I(R), s.rope = I(R), s.cache = I(R), s.kind = I(R), s.tok = I(R);
  s.cu = I(B + 1), s.kv_len = I(B), s.spos = I(ns > 0 ? ns : 1), s.nsearch = I(B);
  s.gidx = I(nw > ns ? nw : ns), s.wseq = I(nw), s.wpos = I(nw), s.draft = I(ns > 0 ? ns : 1);
  s.tk_idx = I(nt > 0 ? nt : 1), s.tk_cnt = I(B), s.argmax = I(nw), s.srows = I(ns > 0 ? ns : 1);
  s.m_arg = I(ns > 0 ? ns : 1), s.n_acc = I(B);
  s.track = reinterpret_cast<float*>(take((size_t)B * max_seq * 4));
  s.conf = reinterpret_cast<float*>(take((size_t)nw * 4));
  s.m_conf = reinterpret_cast<float*>(take((size_t)(ns > 0 ? ns : 1) * 4));
  s.commit = reinterpret_cast<unsigned char*>(take(nw));
  s.accept = reinterpret_cast<unsigned char*>(take(ns > 0 ? ns : 1));
  s.elig = reinterpret_cast<unsigned char*>(take((size_t)B * max_seq));
  s.final_rows = reinterpret_cast<__nv_bfloat16*>(take((size_t)R * d * 2));
  s.gathered = reinterpret_cast<__nv_bfloat16*>(take((size_t)(nw > ns ? nw : ns) * d * 2));
  s.model_ws_bytes = fdl_model_workspace_bytes(ctx, ffn, R);
  s.model_ws = take(s.model_ws_bytes);
  s.bytes = off;
  return s;
}

// Puts the sequences' refresh state back on every return before the step
// has decoded anything, so a failed call leaves the host state as it was.
struct StateGuard {
  int* state;
  std::vector<int> saved;
  bool done = false;
  StateGuard(int* st, int n) : state(st), saved(st, st + n) {}
  ~StateGuard() {
    if (!done) std::copy(saved.begin(), saved.end(), state);
  }
};

struct Rows {
  std::vector<int> seq, rope, cache, kind, tok, cu;
  int n = 0;
  void resize(int cap, int B) {
    seq.assign(cap, 0), rope.assign(cap, 0), cache.assign(cap, 0), kind.assign(cap, 0), tok.assign(cap, 0);
    cu.assign(B + 1, 0);
  }
};

}  // namespace

extern "C" size_t fdl_flash_workspace_bytes(const fdl_ctx* ctx, int ffn, const fdl_flash_params* p, int B,
                                           int max_seq) {
  if (!ctx || !p || ffn <= 0 || B < 1 || max_seq < 1 || p->window < 1 || p->max_search < 0 ||
      p->track_budget < 0)
    return 0;
  return carve(nullptr, ctx, ffn, p, B, max_seq).bytes;
}

extern "C" fdl_status fdl_flash_step(fdl_ctx* ctx, const fdl_model* m, const void* w_lm, void* const* k_caches,
                                     void* const* v_caches, const int* block_table, int bt_stride,
                                     const fdl_flash_params* p, fdl_flash_seqs* s, fdl_flash_trace* trace,
                                     void* workspace, size_t workspace_bytes) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (!m || !w_lm || !k_caches || !v_caches || !block_table || !p || !s || !workspace || !s->prompt_len ||
      !s->seq_len || !s->tokens || !s->masked || !s->tracked || !s->n_tracked || !s->state)
    return loop_fail(ctx, FDL_ERR_INVALID_ARG, "fdl_flash_step: NULL argument");
  const fdl_config& c = ctx->cfg;
  const int B = s->B, W = p->window, MS = p->max_search, BT = p->track_budget, N = s->max_seq;
  if (B < 1 || B > c.max_batch || N < 1 || W < 1 || MS < 0 || BT < 0 || BT > 1024)
    return loop_fail(ctx, FDL_ERR_INVALID_ARG, "fdl_flash_step: bad sizes (B=%d window=%d max_search=%d)", B, W, MS);
  if (B * W > ctx->cfg.max_rows || B * MS > ctx->cfg.max_rows)
    return loop_fail(ctx, FDL_ERR_UNSUPPORTED, "B*window and B*max_search must be <= max_rows=%d", ctx->cfg.max_rows);
  if (2 * MS > c.max_views) return loop_fail(ctx, FDL_ERR_INVALID_ARG, "2*max_search > max_views");
  if (p->mask_token < 0 || p->mask_token >= c.vocab) return loop_fail(ctx, FDL_ERR_INVALID_ARG, "bad mask_token");
  Scratch d = carve(reinterpret_cast<char*>(workspace), ctx, m->ffn, p, B, N);
  if (workspace_bytes < d.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return loop_fail(ctx, FDL_ERR_INVALID_ARG, "workspace of %zu bytes (256-byte aligned), %zu needed",
                     workspace_bytes, d.bytes);
  const cudaStream_t st = ctx->stream;
  const int dm = c.d_model, R_max = c.max_rows;
  fdl_status rc;
  cudaError_t e = cudaSuccess;
#define FDL_TRY(x)             \
  do {                         \
    rc = (x);                  \
    if (rc != FDL_OK) return rc; \
  } while (0)
#define FDL_CU(x)                                                                            \
  do {                                                                                       \
    e = (x);                                                                                 \
    if (e != cudaSuccess) return loop_fail(ctx, FDL_ERR_CUDA, "fdl_flash_step: %s", cudaGetErrorString(e)); \
  } while (0)
  auto h2d = [&](void* dst, const void* src, size_t n) { return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st); };
  auto d2h = [&](void* dst, const void* src, size_t n) { return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st); };

  // ---- the draft forward's rows (the host row builder)
  Rows rw;
  rw.resize(R_max, B);
  fdl_refresh_args ra = {};
  ra.policy = FDL_REFRESH_FLASH_DRAFT;
  ra.B = B, ra.max_seq = N, ra.block = W;
  ra.prompt_len = s->prompt_len, ra.seq_len = s->seq_len, ra.masked = s->masked, ra.state = s->state;
  ra.tracked = s->tracked, ra.tracked_ld = BT, ra.n_tracked = s->n_tracked;
  ra.max_rows = R_max;
  ra.row_seq = rw.seq.data(), ra.row_rope_pos = rw.rope.data(), ra.row_cache_pos = rw.cache.data();
  ra.row_kind = rw.kind.data(), ra.cu_seqlens = rw.cu.data(), ra.n_rows = &rw.n;
  StateGuard guard(s->state, B);
  rc = fdl_refresh_rows(&ra);
  if (rc != FDL_OK) return loop_fail(ctx, rc, "fdl_flash_step: draft rows rejected (max_rows %d)", R_max);
  if (trace && trace->n_rows) trace->n_rows[0] = rw.n, trace->n_rows[1] = 0;
  if (rw.n == 0) return FDL_OK;  // every sequence is fully decoded
  std::vector<int> win_idx, win_seq, win_pos;
  for (int r = 0; r < rw.n; ++r) {
    rw.tok[r] = s->tokens[(size_t)rw.seq[r] * N + rw.rope[r]];
    if (rw.kind[r] == FDL_KIND_WINDOW) {
      win_idx.push_back(r);
      win_seq.push_back(rw.seq[r]);
      win_pos.push_back(rw.rope[r]);
    }
  }
  const int RW = (int)win_idx.size();
  if (RW < 1 || RW > B * W) return loop_fail(ctx, FDL_ERR_INVALID_ARG, "fdl_flash_step: %d window rows", RW);
  FDL_CU(h2d(d.seq, rw.seq.data(), rw.n * 4));
  FDL_CU(h2d(d.rope, rw.rope.data(), rw.n * 4));
  FDL_CU(h2d(d.kind, rw.kind.data(), rw.n * 4));
  FDL_CU(h2d(d.tok, rw.tok.data(), rw.n * 4));
  FDL_CU(h2d(d.cu, rw.cu.data(), (B + 1) * 4));
  FDL_CU(h2d(d.kv_len, s->seq_len, B * 4));
  FDL_CU(h2d(d.gidx, win_idx.data(), RW * 4));
  FDL_CU(h2d(d.wseq, win_seq.data(), RW * 4));
  FDL_CU(h2d(d.wpos, win_pos.data(), RW * 4));
  FDL_CU(cudaMemsetAsync(d.track, 0, (size_t)B * N * 4, st));
  FDL_TRY(fdl_model_forward(ctx, m, d.tok, rw.n, d.seq, d.rope, d.rope, d.kind, d.cu, d.kv_len, B, block_table,
                            bt_stride, k_caches, v_caches, nullptr, 0, nullptr, d.track, N, d.model_ws,
                            d.model_ws_bytes, d.final_rows));
  if (trace && trace->draft_final)
    FDL_CU(cudaMemcpyAsync(trace->draft_final, d.final_rows, (size_t)rw.n * dm * 2, cudaMemcpyDeviceToDevice, st));
  FDL_CU(fdl_launch_pdl(gather_rows_kernel, dim3(RW), dim3(kGatherThreads), 0, st, 1,
                        (const __nv_bfloat16*)d.final_rows, (const int*)d.gidx, dm, d.gathered));

  // ---- unmask: decisions of the window rows straight from their hidden states
  fdl_unmask_args ua = {};
  ua.B = B, ua.max_search = MS, ua.R_w = RW, ua.row_seq = d.wseq, ua.row_pos = d.wpos;
  ua.eps = p->eps, ua.force_progress = p->force_progress;
  ua.conf = d.conf, ua.argmax = d.argmax, ua.commit = d.commit, ua.search_rows = d.srows, ua.n_search = d.nsearch;
  FDL_TRY(fdl_lm_head_unmask(ctx, d.gathered, w_lm, &ua));
  std::vector<float> conf(RW), track((size_t)B * N);
  std::vector<int> argmax(RW), srows((size_t)B * (MS > 0 ? MS : 1)), nsearch(B);
  std::vector<unsigned char> commit(RW);
  FDL_CU(d2h(conf.data(), d.conf, RW * 4));
  FDL_CU(d2h(argmax.data(), d.argmax, RW * 4));
  FDL_CU(d2h(commit.data(), d.commit, RW));
  if (MS > 0) FDL_CU(d2h(srows.data(), d.srows, (size_t)B * MS * 4));
  FDL_CU(d2h(nsearch.data(), d.nsearch, B * 4));
  FDL_CU(d2h(track.data(), d.track, (size_t)B * N * 4));
  FDL_CU(cudaStreamSynchronize(st));
  FDL_TRY(fdl_sync_status(ctx));

  std::vector<std::vector<int>> committed(B), accepted(B), search(B);
  for (int r = 0; r < RW; ++r)
    if (commit[r]) committed[win_seq[r]].push_back(r);
  bool any_search = false;
  for (int b = 0; b < B; ++b) {
    const int nb = std::max(0, std::min(nsearch[b], MS));
    for (int j = 0; j < nb; ++j) {
      const int r = srows[(size_t)b * MS + j];
      if (r < 0 || r >= RW || win_seq[r] != b) return loop_fail(ctx, FDL_ERR_DEVICE_INDEX, "bad search row");
      search[b].push_back(r);
    }
    any_search |= nb > 0;
  }

  // ---- verify forward and the acceptance walk
  std::vector<int> n_acc(B, 0), spos((size_t)B * (MS > 0 ? MS : 1), -1), ns_host(B), dtok((size_t)B * (MS > 0 ? MS : 1), -1);
  std::vector<float> m_conf((size_t)B * (MS > 0 ? MS : 1), 0.f);
  std::vector<int> m_arg((size_t)B * (MS > 0 ? MS : 1), -1);
  if (any_search) {
    for (int b = 0; b < B; ++b) {
      ns_host[b] = (int)search[b].size();
      for (int j = 0; j < ns_host[b]; ++j) {
        spos[(size_t)b * MS + j] = win_pos[search[b][j]];
        dtok[(size_t)b * MS + j] = argmax[search[b][j]];
      }
    }
    Rows vr;
    vr.resize(R_max, B);
    rc = fdl_verify_rows(B, s->seq_len, s->tracked, BT, s->n_tracked, spos.data(), MS, ns_host.data(), BT + W,
                         R_max, vr.seq.data(), vr.rope.data(), vr.cache.data(), vr.kind.data(), vr.cu.data(), &vr.n);
    if (rc != FDL_OK) return loop_fail(ctx, rc, "fdl_flash_step: verify rows rejected (max_rows %d)", R_max);
    std::vector<int> gidx((size_t)B * MS, -1);
    for (int r = 0; r < vr.n; ++r) {
      const int b = vr.seq[r], k = vr.kind[r];
      if (k < 2) {
        vr.tok[r] = s->tokens[(size_t)b * N + vr.rope[r]];
      } else if (k % 2 == 0) {
        vr.tok[r] = argmax[search[b][(k - 2) / 2]];
      } else {
        vr.tok[r] = p->mask_token;
        gidx[(size_t)b * MS + (k - 3) / 2] = r;
      }
    }
    if (trace && trace->n_rows) trace->n_rows[1] = vr.n;
    FDL_CU(h2d(d.seq, vr.seq.data(), vr.n * 4));
    FDL_CU(h2d(d.rope, vr.rope.data(), vr.n * 4));
    FDL_CU(h2d(d.cache, vr.cache.data(), vr.n * 4));
    FDL_CU(h2d(d.kind, vr.kind.data(), vr.n * 4));
    FDL_CU(h2d(d.tok, vr.tok.data(), vr.n * 4));
    FDL_CU(h2d(d.cu, vr.cu.data(), (B + 1) * 4));
    FDL_CU(h2d(d.spos, spos.data(), (size_t)B * MS * 4));
    FDL_CU(h2d(d.nsearch, ns_host.data(), B * 4));
    FDL_CU(h2d(d.gidx, gidx.data(), (size_t)B * MS * 4));
    FDL_CU(h2d(d.draft, dtok.data(), (size_t)B * MS * 4));
    FDL_TRY(fdl_model_forward(ctx, m, d.tok, vr.n, d.seq, d.rope, d.cache, d.kind, d.cu, d.kv_len, B, block_table,
                              bt_stride, k_caches, v_caches, d.spos, MS, d.nsearch, nullptr, 0, d.model_ws,
                              d.model_ws_bytes, d.final_rows));
    if (trace && trace->verify_final)
      FDL_CU(cudaMemcpyAsync(trace->verify_final, d.final_rows, (size_t)vr.n * dm * 2, cudaMemcpyDeviceToDevice, st));
    FDL_CU(fdl_launch_pdl(gather_rows_kernel, dim3(B * MS), dim3(kGatherThreads), 0, st, 1,
                          (const __nv_bfloat16*)d.final_rows, (const int*)d.gidx, dm, d.gathered));
    fdl_unmask_args va = {};
    va.B = B, va.max_search = MS, va.n_search = d.nsearch, va.draft_tok = d.draft, va.gamma = p->gamma;
    va.accept = d.accept, va.n_accept = d.n_acc, va.mask_conf = d.m_conf, va.mask_argmax = d.m_arg;
    FDL_TRY(fdl_lm_head_verify(ctx, d.gathered, w_lm, &va));
    FDL_CU(d2h(n_acc.data(), d.n_acc, B * 4));
    FDL_CU(d2h(m_conf.data(), d.m_conf, (size_t)B * MS * 4));
    FDL_CU(d2h(m_arg.data(), d.m_arg, (size_t)B * MS * 4));
    FDL_CU(cudaStreamSynchronize(st));
    FDL_TRY(fdl_sync_status(ctx));
    for (int b = 0; b < B; ++b) {
      const int na = std::max(0, std::min(n_acc[b], ns_host[b]));
      for (int j = 0; j < na; ++j) accepted[b].push_back(search[b][j]);
    }
  }

  // ---- decode, then the next tracked set from the draft forward's tracker
  guard.done = true;  // from here on the step updates the sequences
  std::vector<std::vector<int>> fresh(B);
  for (int b = 0; b < B; ++b) {
    std::vector<std::pair<int, int>> c, a;
    for (int r : committed[b]) c.push_back({win_pos[r], argmax[r]});
    for (int r : accepted[b]) a.push_back({win_pos[r], argmax[r]});
    std::sort(c.begin(), c.end());
    std::sort(a.begin(), a.end());
    for (auto* v : {&c, &a})
      for (auto& pt : *v) {
        s->tokens[(size_t)b * N + pt.first] = pt.second;
        s->masked[(size_t)b * N + pt.first] = 0;
        fresh[b].push_back(pt.first);
      }
  }
  std::vector<unsigned char> elig((size_t)B * N, 0);
  for (int b = 0; b < B; ++b) {
    for (int q = 0; q < s->seq_len[b]; ++q) elig[(size_t)b * N + q] = s->masked[(size_t)b * N + q] ? 0 : 1;
    for (int q : fresh[b]) elig[(size_t)b * N + q] = 0;
  }
  std::vector<int> tk_idx((size_t)B * (BT > 0 ? BT : 1), -1), tk_cnt(B, 0);
  if (BT > 0) {
    FDL_CU(h2d(d.elig, elig.data(), (size_t)B * N));
    FDL_TRY(fdl_track_topk(ctx, d.track, d.elig, N, d.kv_len, B, BT, d.tk_idx, d.tk_cnt));
    FDL_CU(d2h(tk_idx.data(), d.tk_idx, (size_t)B * BT * 4));
    FDL_CU(d2h(tk_cnt.data(), d.tk_cnt, B * 4));
    FDL_CU(cudaStreamSynchronize(st));
    FDL_TRY(fdl_sync_status(ctx));
  }
  for (int b = 0; b < B; ++b) {
    int n = 0;
    for (int q : fresh[b])
      if (n < BT) s->tracked[(size_t)b * BT + n++] = q;
    const int keep = BT - n;
    for (int j = 0; j < keep && j < tk_cnt[b]; ++j) s->tracked[(size_t)b * BT + n++] = tk_idx[(size_t)b * BT + j];
    s->n_tracked[b] = n;
  }

  if (trace) {
    if (trace->n_window) *trace->n_window = RW;
    for (int r = 0; r < RW; ++r) {
      if (trace->window_pos) trace->window_pos[r] = win_pos[r];
      if (trace->window_seq) trace->window_seq[r] = win_seq[r];
      if (trace->conf) trace->conf[r] = conf[r];
      if (trace->argmax) trace->argmax[r] = argmax[r];
      if (trace->commit) trace->commit[r] = commit[r];
    }
    for (int b = 0; b < B; ++b) {
      if (trace->n_search) trace->n_search[b] = (int)search[b].size();
      if (trace->n_accept) trace->n_accept[b] = (int)accepted[b].size();
      for (int j = 0; j < MS; ++j) {
        const size_t o = (size_t)b * MS + j;
        if (trace->search_rows) trace->search_rows[o] = j < (int)search[b].size() ? search[b][j] : -1;
        if (trace->mask_conf) trace->mask_conf[o] = m_conf[o];
        if (trace->mask_argmax) trace->mask_argmax[o] = m_arg[o];
      }
    }
    if (trace->track) memcpy(trace->track, track.data(), (size_t)B * N * 4);
  }
#undef FDL_TRY
#undef FDL_CU
  return FDL_OK;
}
