// Confidence unmasking (eps rule + ordered search list) and Flash-Verify
// prefix acceptance.
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...",
// section "Method steps in detail", Algorithm 2 step 2 (c_i = max softmax,
// commit c_i >= eps, the rest form the search set) and step 3 (accept while
// the draft and mask views agree and the mask view's confidence >= gamma,
// stop at the first failure). Fast-dLLM news piece, "confidence-aware
// parallel decoding": commit the most confident token when none passes.
//
// Both phases are HBM-bound reductions over vocab-wide logits rows. Each row
// is split across the CTAs of one thread-block cluster; every CTA streams its
// slice with 128-bit loads and keeps a running (max, sum exp, argmax); warps
// merge with shuffles, CTAs through distributed shared memory. The last
// cluster to finish (a ticket counter that it resets) takes the per-sequence
// decisions, so one launch covers one phase.
#include "fdl_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSplit = 8;

struct Stat {
  float m;  // running max
  float s;  // sum of exp(x - m)
  int i;    // lowest index attaining m
};

__device__ __forceinline__ Stat merge(Stat a, Stat b) {
  Stat r;
  r.m = fmaxf(a.m, b.m);
  float sa = (a.s == 0.f) ? 0.f : a.s * __expf(a.m - r.m);
  float sb = (b.s == 0.f) ? 0.f : b.s * __expf(b.m - r.m);
  r.s = sa + sb;
  if (a.m > b.m) r.i = a.i;
  else if (b.m > a.m) r.i = b.i;
  else r.i = min(a.i, b.i);
  return r;
}

__device__ __forceinline__ Stat shfl_merge(Stat a, int off) {
  Stat b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, off);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, off);
  b.i = __shfl_xor_sync(0xffffffffu, a.i, off);
  return merge(a, b);
}

// Folds 8 (bf16) or 4 (fp32) consecutive values starting at index base.
template <int N>
__device__ __forceinline__ void fold(Stat& st, const float (&v)[N], int base) {
  float vm = v[0];
  int vi = 0;
#pragma unroll
  for (int t = 1; t < N; ++t)
    if (v[t] > vm) {
      vm = v[t];
      vi = t;
    }
  if (vm > st.m) {
    st.s = (st.s == 0.f) ? 0.f : st.s * __expf(st.m - vm);
    st.m = vm;
    st.i = base + vi;
  }
#pragma unroll
  for (int t = 0; t < N; ++t) st.s += __expf(v[t] - st.m);
}

__device__ __forceinline__ void unpack(const int4& q, float (&v)[8]) {
  const unsigned w[4] = {(unsigned)q.x, (unsigned)q.y, (unsigned)q.z, (unsigned)q.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    v[2 * t] = __uint_as_float(w[t] << 16);
    v[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
  }
}

__device__ __forceinline__ void unpack(const int4& q, float (&v)[4]) {
  v[0] = __int_as_float(q.x);
  v[1] = __int_as_float(q.y);
  v[2] = __int_as_float(q.z);
  v[3] = __int_as_float(q.w);
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Reduces elements [lo, hi) of one row (this CTA's slice).
template <typename T>
__device__ Stat slice_stat(const T* row, int lo, int hi, bool vec_ok) {
  constexpr int N = 16 / sizeof(T);
  Stat st{-INFINITY, 0.f, 0x7fffffff};
  const int tid = threadIdx.x;
  int i = lo;
  if (vec_ok) {
    // lo is a multiple of N; stream full vectors, 4 in flight per thread.
    const int n_vec = (hi - lo) / N;
    const int4* vp = reinterpret_cast<const int4*>(row + lo);
    int v = tid;
    for (; v + 3 * kThreads < n_vec; v += 4 * kThreads) {
      int4 q0 = __ldcs(vp + v), q1 = __ldcs(vp + v + kThreads);
      int4 q2 = __ldcs(vp + v + 2 * kThreads), q3 = __ldcs(vp + v + 3 * kThreads);
      float f[N];
      unpack(q0, f); fold(st, f, lo + v * N);
      unpack(q1, f); fold(st, f, lo + (v + kThreads) * N);
      unpack(q2, f); fold(st, f, lo + (v + 2 * kThreads) * N);
      unpack(q3, f); fold(st, f, lo + (v + 3 * kThreads) * N);
    }
    for (; v < n_vec; v += kThreads) {
      float f[N];
      unpack(__ldcs(vp + v), f);
      fold(st, f, lo + v * N);
    }
    i = lo + n_vec * N;
  }
  for (int j = i + tid; j < hi; j += kThreads) {
    float x = to_f<T>(row[j]);
    if (x > st.m) {
      st.s = (st.s == 0.f) ? 0.f : st.s * __expf(st.m - x);
      st.m = x;
      st.i = j;
    }
    st.s += __expf(x - st.m);
  }
  return st;
}

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float ld_dsmem_f32(unsigned addr, unsigned rank) {
  unsigned remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ int ld_dsmem_s32(unsigned addr, unsigned rank) {
  unsigned remote;
  int v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

struct RowParams {
  const void* logits;
  int vocab;
  int n_rows;        // rows with a ticket (all of them, valid or not)
  int split;         // CTAs per row (cluster size)
  int chunk;         // elements per CTA slice (multiple of 8)
  bool vec_ok;
  // verify phase: row r = b*max_search + j is valid only when j < n_search[b]
  const int* n_search;
  int max_search;
  float* out_conf;
  int* out_arg;
  unsigned* ticket;
  unsigned* err;
  // unmask decisions
  int phase;         // 0 = unmask, 1 = verify
  int B;
  const int* row_seq;
  const int* row_pos;
  float eps;
  int force_progress;
  unsigned char* commit;
  int* search_rows;
  int* n_search_out;
  // verify decisions
  const int* draft_tok;
  float gamma;
  unsigned char* accept;
  int* n_accept;
};

// Per-sequence decisions of the unmask phase; one warp per sequence.
__device__ void decide_unmask(const RowParams& p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int R = p.n_rows;
  // row_seq must be non-decreasing and inside [0, B)
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    int s = p.row_seq[r];
    if (s < 0 || s >= p.B || (r + 1 < R && p.row_seq[r + 1] < s)) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
    return;
  }
  for (int b = warp; b < p.B; b += nw) {
    // rows of b: [lo, hi) by binary search on the sorted row_seq
    int lo = 0, hi = R;
    {
      int a = 0, z = R;
      while (a < z) { int m = (a + z) >> 1; if (p.row_seq[m] < b) a = m + 1; else z = m; }
      lo = a;
      z = R;
      while (a < z) { int m = (a + z) >> 1; if (p.row_seq[m] <= b) a = m + 1; else z = m; }
      hi = a;
    }
    // eps rule
    bool any = false;
    for (int r = lo + lane; r < hi; r += 32) any |= __ldcg(p.out_conf + r) >= p.eps;
    any = __any_sync(0xffffffffu, any);
    int forced = -1;
    if (p.force_progress && !any && hi > lo) {
      // most confident row, lowest position on ties
      float bc = -1.f;
      int bp = 0x7fffffff, br = -1;
      for (int r = lo + lane; r < hi; r += 32) {
        float c = __ldcg(p.out_conf + r);
        int ps = p.row_pos[r];
        if (c > bc || (c == bc && ps < bp)) { bc = c; bp = ps; br = r; }
      }
      for (int off = 16; off; off >>= 1) {
        float oc = __shfl_xor_sync(0xffffffffu, bc, off);
        int op = __shfl_xor_sync(0xffffffffu, bp, off);
        int orr = __shfl_xor_sync(0xffffffffu, br, off);
        if (oc > bc || (oc == bc && op < bp)) { bc = oc; bp = op; br = orr; }
      }
      forced = br;
    }
    for (int r = lo + lane; r < hi; r += 32)
      p.commit[r] = (__ldcg(p.out_conf + r) >= p.eps || r == forced) ? 1 : 0;
    // rank the uncommitted rows by (conf desc, pos asc)
    int n_unc = 0;
    for (int r = lo + lane; r < hi; r += 32) {
      float c = __ldcg(p.out_conf + r);
      bool unc = !(c >= p.eps) && r != forced;
      n_unc += unc ? 1 : 0;
      if (!unc) continue;
      int ps = p.row_pos[r];
      int rank = 0;
      for (int o = lo; o < hi; ++o) {
        float co = __ldcg(p.out_conf + o);
        if (co >= p.eps || o == forced) continue;
        int po = p.row_pos[o];
        rank += (co > c || (co == c && po < ps)) ? 1 : 0;
      }
      if (rank < p.max_search) p.search_rows[b * p.max_search + rank] = r;
    }
    for (int off = 16; off; off >>= 1) n_unc += __shfl_xor_sync(0xffffffffu, n_unc, off);
    int ns = min(n_unc, p.max_search);
    for (int j = ns + lane; j < p.max_search; j += 32) p.search_rows[b * p.max_search + j] = -1;
    if (lane == 0) p.n_search_out[b] = ns;
  }
}

// Per-sequence prefix walk of the verify phase; one warp per sequence.
__device__ void decide_verify(const RowParams& p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int b = warp; b < p.B; b += nw) {
    int n = p.n_search[b];
    if (n < 0 || n > p.max_search) {
      if (lane == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
      n = max(0, min(n, p.max_search));
    }
    int stop = n;
    for (int j0 = 0; j0 < n && stop == n; j0 += 32) {
      int j = j0 + lane;
      bool ok = true;
      if (j < n) {
        int r = b * p.max_search + j;
        ok = (p.draft_tok[r] == __ldcg(p.out_arg + r)) && (__ldcg(p.out_conf + r) >= p.gamma);
      }
      unsigned fails = __ballot_sync(0xffffffffu, !ok);
      if (fails) stop = j0 + __ffs(fails) - 1;
    }
    for (int j = lane; j < p.max_search; j += 32) p.accept[b * p.max_search + j] = (j < stop) ? 1 : 0;
    if (lane == 0) p.n_accept[b] = stop;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) row_reduce_kernel(RowParams p) {
  __shared__ Stat warp_stat[kThreads / 32];
  __shared__ float cta_m, cta_s;
  __shared__ int cta_i;
  __shared__ unsigned last;
  const int row = blockIdx.x / p.split;
  const unsigned rank = p.split > 1 ? cluster_rank() : 0u;
  bool valid = row < p.n_rows;
  if (valid && p.phase == 1) {
    int b = row / p.max_search, j = row % p.max_search;
    valid = j < p.n_search[b];
  }
  Stat st{-INFINITY, 0.f, 0x7fffffff};
  if (valid) {
    const T* base = reinterpret_cast<const T*>(p.logits) + (size_t)row * p.vocab;
    int lo = (int)rank * p.chunk;
    int hi = min(p.vocab, lo + p.chunk);
    if (lo < hi) st = slice_stat<T>(base, lo, hi, p.vec_ok);
  }
  for (int off = 16; off; off >>= 1) st = shfl_merge(st, off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_stat[warp] = st;
  __syncthreads();
  if (warp == 0) {
    st = lane < kThreads / 32 ? warp_stat[lane] : Stat{-INFINITY, 0.f, 0x7fffffff};
    for (int off = 16; off; off >>= 1) st = shfl_merge(st, off);
    if (lane == 0) { cta_m = st.m; cta_s = st.s; cta_i = st.i; }
  }
  if (p.split > 1) {
    cluster_sync_all();  // every slice result is in its CTA's shared memory
    if (rank == 0 && threadIdx.x == 0) {
      Stat acc{cta_m, cta_s, cta_i};
      for (int r = 1; r < p.split; ++r) {
        Stat o{ld_dsmem_f32(smem_u32(&cta_m), r), ld_dsmem_f32(smem_u32(&cta_s), r),
               ld_dsmem_s32(smem_u32(&cta_i), r)};
        acc = merge(acc, o);
      }
      cta_m = acc.m; cta_s = acc.s; cta_i = acc.i;
    }
    cluster_sync_all();  // peers stay resident until rank 0 has read them
  } else {
    __syncthreads();
  }
  if (rank != 0) return;
  if (threadIdx.x == 0) {
    if (valid) {
      p.out_conf[row] = 1.f / cta_s;  // cta_s = sum exp(x - max) >= 1
      p.out_arg[row] = cta_i;
    }
    __threadfence();
    unsigned t = atomicAdd(p.ticket, 1u);
    last = (t == (unsigned)p.n_rows - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (p.phase == 0) decide_unmask(p);
  else decide_verify(p);
  if (threadIdx.x == 0) *p.ticket = 0u;  // ready for the next call
}

template <typename T>
cudaError_t launch_phase(fdl_ctx* ctx, RowParams p) {
  if (p.n_rows == 0) return cudaSuccess;
  const int V = p.vocab;
  int split = (2 * ctx->num_sms + p.n_rows - 1) / p.n_rows;
  split = max(1, min(split, kMaxSplit));
  split = min(split, max(1, V / 4096));
  int chunk = (V + split - 1) / split;
  chunk = (chunk + 7) / 8 * 8;
  split = (V + chunk - 1) / chunk;
  p.split = split;
  p.chunk = chunk;
  p.vec_ok = ((reinterpret_cast<uintptr_t>(p.logits) & 15) == 0) && ((size_t)V * sizeof(T)) % 16 == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.n_rows * split), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, row_reduce_kernel<T>, p);
}

}  // namespace

cudaError_t fdl_launch_unmask_verify(fdl_ctx* ctx, const fdl_unmask_args* a) {
  const bool bf16 = ctx->cfg.dtype == FDL_BF16;
  cudaError_t e = cudaSuccess;
  if (a->logits && a->R_w > 0) {
    RowParams p = {};
    p.logits = a->logits;
    p.vocab = ctx->cfg.vocab;
    p.n_rows = a->R_w;
    p.out_conf = a->conf;
    p.out_arg = a->argmax;
    p.ticket = ctx->tickets + 0;
    p.err = ctx->err_word;
    p.phase = 0;
    p.B = a->B;
    p.row_seq = a->row_seq;
    p.row_pos = a->row_pos;
    p.eps = a->eps;
    p.force_progress = a->force_progress;
    p.commit = a->commit;
    p.search_rows = a->search_rows;
    p.n_search_out = a->n_search;
    p.max_search = a->max_search;
    e = bf16 ? launch_phase<__nv_bfloat16>(ctx, p) : launch_phase<float>(ctx, p);
    if (e != cudaSuccess) return e;
  } else if (a->logits && a->R_w == 0) {
    // no window rows: every sequence has an empty search list
    e = cudaMemsetAsync(a->n_search, 0, a->B * sizeof(int), ctx->stream);
    if (e == cudaSuccess && a->max_search > 0)
      e = cudaMemsetAsync(a->search_rows, 0xff, (size_t)a->B * a->max_search * sizeof(int), ctx->stream);
    if (e != cudaSuccess) return e;
  }
  if (a->mask_logits) {
    RowParams p = {};
    p.logits = a->mask_logits;
    p.vocab = ctx->cfg.vocab;
    p.n_rows = a->B * a->max_search;
    p.n_search = a->n_search;
    p.max_search = a->max_search;
    p.out_conf = a->mask_conf;
    p.out_arg = a->mask_argmax;
    p.ticket = ctx->tickets + 1;
    p.err = ctx->err_word;
    p.phase = 1;
    p.B = a->B;
    p.draft_tok = a->draft_tok;
    p.gamma = a->gamma;
    p.accept = a->accept;
    p.n_accept = a->n_accept;
    e = bf16 ? launch_phase<__nv_bfloat16>(ctx, p) : launch_phase<float>(ctx, p);
  }
  return e;
}
