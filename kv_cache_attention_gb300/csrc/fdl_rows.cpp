// Host-side row builders: the query rows of one denoising step under a
// KV-cache refresh policy, and the rows of a Flash-Verify forward.
//
// A refresh policy only decides which positions a step recomputes; the
// layer-step kernels then project those rows, write their K/V into the cache
// at their own positions and attend over the whole cache. Sources:
//   - Fast-dLLM news piece, the key-value cache for block-wise decoding
//     (PrefixCache: the prompt's KV reused within a block and the whole cache
//     recomputed once a block is decoded; DualCache: the masked suffix cached
//     as well, so a step recomputes only its block);
//   - FlashDLM note, key design 1 (FreeCache: a full forward first, then the
//     active window is the current block and every later one, and finished
//     blocks are frozen);
//   - Flash-dLLM paper digest, Algorithm 2 steps 1-3 (initial full forward;
//     the tracked set plus the sliding masked window; the verify forward's
//     shrunk tracked set and two views per search token).
//
// Both builders validate everything first and write nothing (state included)
// unless the whole call is valid.
#include <cstring>
#include <vector>

#include "fdl.h"

namespace {

struct Seq {
  int prompt, n;
  const unsigned char* masked;
};

// First block still holding a masked position (blocks start at the prompt's
// end), or -1 when the sequence is fully decoded.
int current_block(const Seq& s, int block) {
  for (int p = s.prompt; p < s.n; ++p)
    if (s.masked[p]) return (p - s.prompt) / block;
  return -1;
}

// The half-open position range [lo, hi) a step recomputes, for the block
// policies, and the state after the step. Returns false when no row is taken.
bool block_policy_range(int policy, const Seq& s, int block, int state, int* lo, int* hi, int* cur_out,
                        int* new_state) {
  const int cur = current_block(s, block);
  if (cur < 0) return false;
  const int bs = s.prompt + cur * block;
  const int be = bs + block < s.n ? bs + block : s.n;
  *cur_out = cur;
  *new_state = cur;
  *lo = 0;
  *hi = s.n;
  switch (policy) {
    case FDL_REFRESH_FULL:
      break;
    case FDL_REFRESH_PREFIX:
      if (state == cur) *lo = bs;
      break;
    case FDL_REFRESH_DUAL:
      if (state == cur) {
        *lo = bs;
        *hi = be;
      }
      break;
    case FDL_REFRESH_FREECACHE:
      if (state != -1) *lo = bs;
      break;
  }
  return true;
}

}  // namespace

extern "C" fdl_status fdl_refresh_rows(const fdl_refresh_args* a) {
  if (!a) return FDL_ERR_INVALID_ARG;
  const int pol = a->policy;
  if (pol < FDL_REFRESH_FULL || pol > FDL_REFRESH_FLASH_DRAFT) return FDL_ERR_INVALID_ARG;
  if (a->B < 1 || a->block < 1 || a->max_seq < 1 || a->max_rows < 0) return FDL_ERR_INVALID_ARG;
  if (!a->prompt_len || !a->seq_len || !a->masked || !a->state || !a->row_seq || !a->row_rope_pos ||
      !a->row_cache_pos || !a->row_kind || !a->cu_seqlens || !a->n_rows)
    return FDL_ERR_INVALID_ARG;
  const bool flash = pol == FDL_REFRESH_FLASH_DRAFT;
  if (flash && (!a->tracked || !a->n_tracked || a->tracked_ld < 0)) return FDL_ERR_INVALID_ARG;

  // Pass 1: validate and count.
  std::vector<unsigned char> seen;
  long long total = 0;
  for (int b = 0; b < a->B; ++b) {
    const int P = a->prompt_len[b], N = a->seq_len[b];
    if (P < 0 || P > N || N > a->max_seq || a->state[b] < -1) return FDL_ERR_INVALID_ARG;
    const Seq s{P, N, a->masked + (size_t)b * a->max_seq};
    if (flash) {
      const int nt = a->n_tracked[b];
      if (nt < 0 || nt > a->tracked_ld) return FDL_ERR_INVALID_ARG;
      seen.assign((size_t)N, 0);
      const int* tr = a->tracked + (size_t)b * a->tracked_ld;
      for (int t = 0; t < nt; ++t) {
        const int p = tr[t];
        if (p < 0 || p >= N || s.masked[p] || seen[p]) return FDL_ERR_INVALID_ARG;
        seen[p] = 1;
      }
      int n_masked = 0;
      for (int p = P; p < N; ++p) n_masked += s.masked[p] ? 1 : 0;
      if (n_masked == 0) continue;
      total += a->state[b] == -1 ? N : (n_masked < a->block ? n_masked : a->block) + nt;
    } else {
      int lo, hi, cur, ns;
      if (block_policy_range(pol, s, a->block, a->state[b], &lo, &hi, &cur, &ns)) total += hi - lo;
    }
  }
  if (total > a->max_rows) return FDL_ERR_INVALID_ARG;

  // Pass 2: write the rows and update the state.
  int r = 0;
  a->cu_seqlens[0] = 0;
  auto put = [&](int b, int pos, int kind) {
    a->row_seq[r] = b;
    a->row_rope_pos[r] = pos;
    a->row_cache_pos[r] = pos;
    a->row_kind[r] = kind;
    ++r;
  };
  for (int b = 0; b < a->B; ++b) {
    const Seq s{a->prompt_len[b], a->seq_len[b], a->masked + (size_t)b * a->max_seq};
    if (flash) {
      int taken = 0, first_after_window = s.n;
      for (int p = s.prompt; p < s.n; ++p)
        if (s.masked[p] && ++taken == a->block) {
          first_after_window = p + 1;
          break;
        }
      if (taken > 0) {
        if (a->state[b] == -1) {
          for (int p = 0; p < s.n; ++p)
            put(b, p, (p >= s.prompt && p < first_after_window && s.masked[p]) ? FDL_KIND_WINDOW
                                                                                  : FDL_KIND_NORMAL);
          a->state[b] = 0;
        } else {
          for (int p = s.prompt; p < first_after_window; ++p)
            if (s.masked[p]) put(b, p, FDL_KIND_WINDOW);
          const int* tr = a->tracked + (size_t)b * a->tracked_ld;
          for (int t = 0; t < a->n_tracked[b]; ++t) put(b, tr[t], FDL_KIND_NORMAL);
        }
      }
    } else {
      int lo, hi, cur, ns;
      if (block_policy_range(pol, s, a->block, a->state[b], &lo, &hi, &cur, &ns)) {
        const int bs = s.prompt + cur * a->block;
        const int be = bs + a->block < s.n ? bs + a->block : s.n;
        for (int p = lo; p < hi; ++p)
          put(b, p, (p >= bs && p < be && s.masked[p]) ? FDL_KIND_WINDOW : FDL_KIND_NORMAL);
        a->state[b] = ns;
      }
    }
    a->cu_seqlens[b + 1] = r;
  }
  *a->n_rows = r;
  return FDL_OK;
}

extern "C" fdl_status fdl_verify_rows(int B, const int* seq_len, const int* tracked, int tracked_ld,
                                      const int* n_tracked, const int* search_pos, int search_ld,
                                      const int* n_search, int query_budget, int max_rows, int* row_seq,
                                      int* row_rope_pos, int* row_cache_pos, int* row_kind, int* cu_seqlens,
                                      int* n_rows) {
  if (B < 1 || query_budget < 0 || max_rows < 0 || tracked_ld < 0 || search_ld < 0) return FDL_ERR_INVALID_ARG;
  if (!seq_len || !tracked || !n_tracked || !search_pos || !n_search || !row_seq || !row_rope_pos ||
      !row_cache_pos || !row_kind || !cu_seqlens || !n_rows)
    return FDL_ERR_INVALID_ARG;
  std::vector<unsigned char> seen;
  long long total = 0;
  for (int b = 0; b < B; ++b) {
    const int N = seq_len[b], nt = n_tracked[b], m = n_search[b];
    if (N < 0 || nt < 0 || nt > tracked_ld || m < 0 || m > search_ld) return FDL_ERR_INVALID_ARG;
    const int* tr = tracked + (size_t)b * tracked_ld;
    const int* sp = search_pos + (size_t)b * search_ld;
    for (int t = 0; t < nt; ++t)
      if (tr[t] < 0 || tr[t] >= N) return FDL_ERR_INVALID_ARG;
    seen.assign((size_t)N, 0);
    for (int j = 0; j < m; ++j) {
      if (sp[j] < 0 || sp[j] >= N || seen[sp[j]]) return FDL_ERR_INVALID_ARG;
      seen[sp[j]] = 1;
    }
    const int keep = query_budget - 2 * m > 0 ? query_budget - 2 * m : 0;
    total += (keep < nt ? keep : nt) + 2 * m;
  }
  if (total > max_rows) return FDL_ERR_INVALID_ARG;

  int r = 0;
  cu_seqlens[0] = 0;
  for (int b = 0; b < B; ++b) {
    const int N = seq_len[b], nt = n_tracked[b], m = n_search[b];
    const int* tr = tracked + (size_t)b * tracked_ld;
    const int* sp = search_pos + (size_t)b * search_ld;
    const int keep = query_budget - 2 * m > 0 ? query_budget - 2 * m : 0;
    for (int t = 0; t < nt && t < keep; ++t, ++r) {
      row_seq[r] = b;
      row_rope_pos[r] = tr[t];
      row_cache_pos[r] = tr[t];
      row_kind[r] = FDL_KIND_NORMAL;
    }
    for (int v = 0; v < 2; ++v)          // draft views, then mask views
      for (int j = 0; j < m; ++j, ++r) {
        row_seq[r] = b;
        row_rope_pos[r] = sp[j];
        row_cache_pos[r] = N + v * m + j;
        row_kind[r] = v == 0 ? FDL_KIND_DRAFT_VIEW(j) : FDL_KIND_MASK_VIEW(j);
      }
    cu_seqlens[b + 1] = r;
  }
  *n_rows = r;
  return FDL_OK;
}
