// Block-table scheduled attention with the Flash-Verify two-view mask and
// the Eq. (2) attention-mass tracker: work-list builder and the exact-fp32
// CUDA-core kernel.
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...":
//   "Background"  Flash Attention: exact softmax(QK^T/sqrt(d))V, tiled so the
//                 score matrix never reaches HBM;
//   "Core method" block-table scheduled attention aligns every sequence's
//                 ragged query block with its KV blocks, no padding; verify
//                 queries are duplicated into draft and mask views isolated
//                 by a causal mask and sharing the tracked context;
//   "Method steps in detail", step 4, Eq. (2): a_i accumulates, over layers,
//                 the head- and row-averaged attention that masked-window
//                 queries pay to key i.
// aiposthub article, Flash-Verify section: the mask view must not see the
// draft at its own position but may use earlier drafts.
//
// The work list (b, q_start, q_len, n_keys) is built on the device from
// cu_seqlens_q so the whole call stays asynchronous. One CTA handles one
// (work item, head): an online-softmax pass over the visible keys, then, for
// items holding masked-window rows, a second pass that re-forms the final
// probabilities exp(s - lse) and adds their column sums to the tracker.
#include <math.h>

#include "fdl_internal.cuh"

namespace {

constexpr int kBuildThreads = 1024;

__global__ void __launch_bounds__(kBuildThreads)
build_worklist_kernel(const int* __restrict__ cu, const int* __restrict__ kv_len,
                      const int* __restrict__ n_search, int B, int R, int tile_m,
                      const int* __restrict__ row_kind, int max_seq, int max_search_tokens,
                      int* __restrict__ wl, int cap, int* __restrict__ n_masked, unsigned* err) {
  extern __shared__ int offs[];  // [B + 1]
  __shared__ int ok;
  const int tid = threadIdx.x;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  if (tid == 0) {
    int good = (cu[0] == 0) && (cu[B] == R);
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      int rows = cu[b + 1] - cu[b];
      if (rows < 0) good = 0;
      offs[b] = acc;
      acc += rows > 0 ? (rows + tile_m - 1) / tile_m : 0;
    }
    offs[B] = acc;
    if (acc > cap) good = 0;
    ok = good;
    if (!good) fdl::raise_error(err, FDL_DEVERR_SHAPE);
  }
  __syncthreads();
  if (!ok) {
    if (tid == 0) wl[0] = 0;
    for (int b = tid; b < B; b += blockDim.x) n_masked[b] = 0;
    return;
  }
  for (int b = tid; b < B; b += blockDim.x) {
    int kvl = kv_len[b];
    if (kvl < 0 || kvl > max_seq) {
      fdl::raise_error(err, FDL_DEVERR_INDEX);
      kvl = max(0, min(kvl, max_seq));
    }
    int m = 0;
    if (n_search) {
      m = n_search[b];
      if (m < 0 || m > max_search_tokens) {
        fdl::raise_error(err, FDL_DEVERR_INDEX);
        m = max(0, min(m, max_search_tokens));
      }
    }
    const int lo = cu[b], hi = cu[b + 1];
    int item = offs[b];
    for (int q0 = lo; q0 < hi; q0 += tile_m, ++item) {
      int* it = wl + 1 + 4 * item;
      it[0] = b;
      it[1] = q0;
      it[2] = min(tile_m, hi - q0);
      it[3] = kvl + 2 * m;
    }
  }
  const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int b = warp; b < B; b += nw) {
    int c = 0;
    for (int r = cu[b] + lane; r < cu[b + 1]; r += 32) c += (row_kind[r] == FDL_KIND_WINDOW) ? 1 : 0;
    for (int off = 16; off; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if (lane == 0) n_masked[b] = c;
  }
  if (tid == 0) wl[0] = offs[B];
}

struct AttnParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* block_table;
  int bt_stride, page_size, n_pages;
  const int* kv_len;
  const int* row_kind;
  const int* search_pos;
  int search_ld;
  const int* n_search;
  int max_search_tokens;
  void* o;
  float* lse;
  float* track;
  int track_ld;
  const int* wl;
  const int* n_masked;
  int H, d;
  float scale;
  unsigned* err;
};

// Visibility of cache position c to a row of `kind` in a sequence with kvl
// base keys and m search tokens (is_search: c is a search position).
__device__ __forceinline__ bool key_visible(int kind, int c, int kvl, int m, bool is_search) {
  if (kind < 2) return c < kvl;
  if (c < kvl) return !is_search;
  const int v = c - kvl;
  if (v >= 2 * m) return false;
  const int k = (kind - 2) >> 1;
  const bool mask_view = (kind - 2) & 1;
  if (v < m) return mask_view ? (v < k) : (v <= k);  // draft key v
  const int j = v - m;                                // mask key j
  return mask_view ? (j >= k) : (j > k);
}

constexpr int kBM = FDL_TILE_M_SIMT;  // rows per work item
constexpr int kKT = 32;               // keys per tile (one per lane)
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kBM / kWarps;
constexpr int kMaxSearchSmem = 256;

template <typename T, int HD>
__global__ void __launch_bounds__(kWarps * 32) attn_simt_kernel(AttnParams p) {
  constexpr int DPL = HD / 32;  // output dims per lane
  __shared__ float qs[kBM][HD];
  __shared__ float ks[kKT][HD + 1];
  __shared__ float vs[kKT][HD];
  __shared__ unsigned char key_ok[kKT], key_search[kKT];
  __shared__ int spos[kMaxSearchSmem];
  __shared__ float colacc[kKT];

  const int item = blockIdx.x;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  if (item >= p.wl[0]) return;
  const int h = blockIdx.y;
  const int* it = p.wl + 1 + 4 * item;
  const int b = it[0], q0 = it[1], qlen = it[2], nkeys = it[3];
  const int kvl = min(p.kv_len[b], nkeys);
  int m = 0;
  if (p.search_pos) m = (nkeys - kvl) / 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int j = tid; j < m && j < kMaxSearchSmem; j += blockDim.x) spos[j] = p.search_pos[(size_t)b * p.search_ld + j];
  for (int e = tid; e < kBM * HD; e += blockDim.x) {
    int r = e / HD, dd = e % HD;
    qs[r][dd] = r < qlen ? fdl::io<T>::load(reinterpret_cast<const T*>(p.q) + (size_t)(q0 + r) * p.d + h * HD + dd) : 0.f;
  }
  int kind[kRowsPerWarp];
  float mrow[kRowsPerWarp], lrow[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
  for (int t = 0; t < kRowsPerWarp; ++t) {
    int lr = warp * kRowsPerWarp + t;
    kind[t] = lr < qlen ? p.row_kind[q0 + lr] : -1;
    if (kind[t] >= 2 && ((kind[t] - 2) >> 1) >= m) {
      if (lane == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
      kind[t] = -2;  // sees nothing
    }
    mrow[t] = -INFINITY;
    lrow[t] = 0.f;
#pragma unroll
    for (int u = 0; u < DPL; ++u) acc[t][u] = 0.f;
  }
  const T* kc = reinterpret_cast<const T*>(p.k_cache);
  const T* vc = reinterpret_cast<const T*>(p.v_cache);
  for (int kt = 0; kt < nkeys; kt += kKT) {
    __syncthreads();
    // stage the key tile (a warp per key row, coalesced across head dims)
    for (int j = warp; j < kKT; j += kWarps) {
      const int c = kt + j;
      long long slot = -1;
      if (c < nkeys) slot = fdl::cache_slot(p.block_table, p.bt_stride, p.page_size, p.n_pages, b, c, lane == 0 ? p.err : nullptr);
      for (int dd = lane; dd < HD; dd += 32) {
        ks[j][dd] = slot >= 0 ? fdl::io<T>::load(kc + slot * p.d + h * HD + dd) : 0.f;
        vs[j][dd] = slot >= 0 ? fdl::io<T>::load(vc + slot * p.d + h * HD + dd) : 0.f;
      }
      if (lane == 0) {
        key_ok[j] = slot >= 0;
        bool s = false;
        if (c < kvl)
          for (int t = 0; t < m && t < kMaxSearchSmem; ++t) s |= (spos[t] == c);
        key_search[j] = s;
      }
    }
    __syncthreads();
    const int c = kt + lane;
#pragma unroll
    for (int t = 0; t < kRowsPerWarp; ++t) {
      if (kind[t] == -1) continue;
      const int lr = warp * kRowsPerWarp + t;
      float s = 0.f;
#pragma unroll 8
      for (int dd = 0; dd < HD; ++dd) s = fmaf(qs[lr][dd], ks[lane][dd], s);
      s *= p.scale;
      const bool vis = kind[t] >= 0 && key_ok[lane] && key_visible(kind[t], c, kvl, m, key_search[lane]);
      s = vis ? s : -INFINITY;
      float tmax = s;
      for (int off = 16; off; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float mnew = fmaxf(mrow[t], tmax);
      if (mnew == -INFINITY) continue;
      const float pr = vis ? expf(s - mnew) : 0.f;
      const float corr = mrow[t] == -INFINITY ? 0.f : expf(mrow[t] - mnew);
      float psum = pr;
      for (int off = 16; off; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      lrow[t] = lrow[t] * corr + psum;
#pragma unroll
      for (int u = 0; u < DPL; ++u) acc[t][u] *= corr;
      for (int j = 0; j < kKT; ++j) {
        const float pj = __shfl_sync(0xffffffffu, pr, j);
#pragma unroll
        for (int u = 0; u < DPL; ++u) acc[t][u] = fmaf(pj, vs[j][lane + 32 * u], acc[t][u]);
      }
      mrow[t] = mnew;
    }
  }
  float lse_row[kRowsPerWarp];
  bool any_window = false;
#pragma unroll
  for (int t = 0; t < kRowsPerWarp; ++t) {
    const int lr = warp * kRowsPerWarp + t;
    lse_row[t] = lrow[t] > 0.f ? mrow[t] + logf(lrow[t]) : -INFINITY;
    if (lr >= qlen) continue;
    const float inv = lrow[t] > 0.f ? 1.f / lrow[t] : 0.f;
    T* o = reinterpret_cast<T*>(p.o) + (size_t)(q0 + lr) * p.d + h * HD;
#pragma unroll
    for (int u = 0; u < DPL; ++u) fdl::io<T>::store(o + lane + 32 * u, acc[t][u] * inv);
    if (p.lse && lane == 0) p.lse[(size_t)(q0 + lr) * p.H + h] = lse_row[t];
    any_window |= kind[t] == FDL_KIND_WINDOW;
  }
  // Tracker pass over base keys with the final normaliser.
  if (!p.track) return;
  __shared__ int blk_window;
  if (tid == 0) blk_window = 0;
  __syncthreads();
  if (any_window && lane == 0) blk_window = 1;
  __syncthreads();
  const int nm = p.n_masked[b];
  if (!blk_window || nm <= 0) return;
  const float wscale = 1.f / ((float)p.H * (float)nm);
  for (int kt = 0; kt < kvl; kt += kKT) {
    __syncthreads();
    for (int j = warp; j < kKT; j += kWarps) {
      const int c = kt + j;
      long long slot = -1;
      if (c < kvl) slot = fdl::cache_slot(p.block_table, p.bt_stride, p.page_size, p.n_pages, b, c, nullptr);
      for (int dd = lane; dd < HD; dd += 32)
        ks[j][dd] = slot >= 0 ? fdl::io<T>::load(kc + slot * p.d + h * HD + dd) : 0.f;
      if (lane == 0) key_ok[j] = slot >= 0;
    }
    if (tid < kKT) colacc[tid] = 0.f;
    __syncthreads();
    float col = 0.f;
#pragma unroll
    for (int t = 0; t < kRowsPerWarp; ++t) {
      if (kind[t] != FDL_KIND_WINDOW) continue;
      const int lr = warp * kRowsPerWarp + t;
      float s = 0.f;
#pragma unroll 8
      for (int dd = 0; dd < HD; ++dd) s = fmaf(qs[lr][dd], ks[lane][dd], s);
      s *= p.scale;
      if (kt + lane < kvl && key_ok[lane]) col += expf(s - lse_row[t]);
    }
    if (col != 0.f) atomicAdd(&colacc[lane], col);
    __syncthreads();
    if (tid < kKT && kt + tid < kvl && colacc[tid] != 0.f)
      atomicAdd(p.track + (size_t)b * p.track_ld + kt + tid, colacc[tid] * wscale);
  }
}

}  // namespace

bool fdl_attn_tc_supported(const fdl_config& c);
cudaError_t fdl_launch_attn_tc(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                               const int* block_table, int bt_stride, const int* cu_seqlens_q, const int* kv_len,
                               int B, int R, const int* row_kind, const int* search_pos, int search_ld,
                               const int* n_search, int max_search_tokens, void* o_out, float* lse_out, float* track,
                               int track_ld, int cap, bool decode, int* worklist_out);
int fdl_attn_tc_decode_max_batch();

cudaError_t fdl_launch_attn(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                            const int* block_table, int bt_stride, const int* cu_seqlens_q,
                            const int* kv_len, int B, int R, const int* row_kind,
                            const int* search_pos, int search_ld, const int* n_search, void* o_out,
                            float* lse_out, float* track, int track_ld, int* worklist_out) {
  const fdl_config& c = ctx->cfg;
  const int tile = ctx->attn_tile_m;
  const int cap = (R + tile - 1) / tile + B;
  const int max_search_tokens = min(c.max_views / 2, search_pos ? search_ld : 0);
  // The tensor-core kernel finds its own work item from cu_seqlens_q (up to
  // a batch it can stage in shared memory): no separate work-list launch.
  if (tile == FDL_TILE_M_TC && B <= fdl_attn_tc_decode_max_batch())
    return fdl_launch_attn_tc(ctx, q, k_cache, v_cache, block_table, bt_stride, cu_seqlens_q, kv_len, B, R, row_kind,
                              search_pos, search_ld, n_search, max_search_tokens, o_out, lse_out, track, track_ld,
                              cap, true, worklist_out);
  cudaError_t e = fdl_launch_pdl(build_worklist_kernel, dim3(1), dim3(kBuildThreads), (B + 1) * sizeof(int),
                                 ctx->stream, 1, cu_seqlens_q, kv_len, search_pos ? n_search : nullptr, B, R,
                                 tile, row_kind, c.max_seq, max_search_tokens, ctx->worklist,
                                 ctx->worklist_items, ctx->n_masked, ctx->err_word);
  if (e != cudaSuccess) return e;
  if (worklist_out) {
    e = cudaMemcpyAsync(worklist_out, ctx->worklist, (1 + 4 * (size_t)cap) * sizeof(int),
                        cudaMemcpyDeviceToDevice, ctx->stream);
    if (e != cudaSuccess) return e;
  }
  if (ctx->attn_tile_m == FDL_TILE_M_TC)
    return fdl_launch_attn_tc(ctx, q, k_cache, v_cache, block_table, bt_stride, cu_seqlens_q, kv_len, B, R, row_kind,
                              search_pos, search_ld, n_search, max_search_tokens, o_out, lse_out, track, track_ld,
                              cap, false, nullptr);
  AttnParams p;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.page_size = c.page_size;
  p.n_pages = c.n_pages;
  p.kv_len = kv_len;
  p.row_kind = row_kind;
  p.search_pos = search_pos;
  p.search_ld = search_ld;
  p.n_search = n_search;
  p.max_search_tokens = max_search_tokens;
  p.o = o_out;
  p.lse = lse_out;
  p.track = track;
  p.track_ld = track_ld;
  p.wl = ctx->worklist;
  p.n_masked = ctx->n_masked;
  p.H = c.n_heads;
  p.d = c.d_model;
  p.scale = (float)(1.0 / sqrt((double)c.head_dim));
  p.err = ctx->err_word;
  const dim3 grid(cap, c.n_heads), block(kWarps * 32);
  if (c.dtype == FDL_BF16) {
    if (c.head_dim == 128) return fdl_launch_pdl(attn_simt_kernel<__nv_bfloat16, 128>, grid, block, 0, ctx->stream, 1, p);
    return fdl_launch_pdl(attn_simt_kernel<__nv_bfloat16, 64>, grid, block, 0, ctx->stream, 1, p);
  }
  if (c.head_dim == 128) return fdl_launch_pdl(attn_simt_kernel<float, 128>, grid, block, 0, ctx->stream, 1, p);
  return fdl_launch_pdl(attn_simt_kernel<float, 64>, grid, block, 0, ctx->stream, 1, p);
}
