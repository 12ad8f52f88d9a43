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
// Both phases are HBM-bound reductions over vocab-wide logits rows. A row is
// split across the CTAs of one thread-block cluster (up to 8); every CTA
// streams its slice with 128-bit loads, keeps (max, sum exp, argmax) per
// thread over register blocks (tree max, then the sum of exponentials with
// four accumulators), and merges with warp shuffles. The slices' statistics
// meet in the row leader's (cluster rank 0) shared memory through
// distributed shared memory and are merged there in rank order, so the
// result does not depend on timing; the leader writes the row's confidence
// and argmax and takes one ticket per row. The leader that arrives last
// takes the per-sequence decisions: one launch per phase, and the only wait
// on another CTA is the cluster barrier of co-scheduled CTAs.
#include <cudaTypedefs.h>

#include "fdl_internal.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSplit = 8;  // CTAs per row: one (portable) thread-block cluster

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

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// Reduces elements [lo, hi) of one row (this CTA's slice). Each thread takes
// blocks of kVB 128-bit vectors: the block maximum (first index on ties) is
// found before any exponential, then the block's exp(x - max) are summed with
// four accumulators; blocks merge into the running statistic.
template <typename T>
__device__ Stat slice_stat(const T* row, int lo, int hi, bool vec_ok) {
  constexpr int N = 16 / sizeof(T);
  constexpr int kVB = 8;
  Stat st{-INFINITY, 0.f, 0x7fffffff};
  const int tid = threadIdx.x;
  int i = lo;
  if (vec_ok) {
    // lo is a multiple of N
    const int n_vec = (hi - lo) / N;
    const int4* vp = reinterpret_cast<const int4*>(row + lo);
    for (int v0 = 0; v0 < n_vec; v0 += kVB * kThreads) {
      float f[kVB][N];
      bool have[kVB];
#pragma unroll
      for (int u = 0; u < kVB; ++u) {
        const int idx = v0 + u * kThreads + tid;
        have[u] = idx < n_vec;
        const int4 q = have[u] ? __ldcs(vp + idx) : make_int4(0, 0, 0, 0);
        unpack(q, f[u]);
      }
      float bm = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int u = 0; u < kVB; ++u)
#pragma unroll
        for (int t = 0; t < N; ++t)
          if (have[u] && f[u][t] > bm) {
            bm = f[u][t];
            bi = lo + (v0 + u * kThreads + tid) * N + t;
          }
      if (bm == -INFINITY) continue;
      if (bm > st.m) {
        st.s = (st.s == 0.f) ? 0.f : st.s * ex2((st.m - bm) * kLog2e);
        st.m = bm;
        st.i = bi;
      }
      const float mb = st.m * kLog2e;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int u = 0; u < kVB; ++u)
#pragma unroll
        for (int t = 0; t < N; t += 4) {
          if (!have[u]) continue;
          a0 += ex2(fmaf(f[u][t], kLog2e, -mb));
          a1 += ex2(fmaf(f[u][t + 1], kLog2e, -mb));
          a2 += ex2(fmaf(f[u][t + 2], kLog2e, -mb));
          a3 += ex2(fmaf(f[u][t + 3], kLog2e, -mb));
        }
      st.s += (a0 + a1) + (a2 + a3);
    }
    i = lo + n_vec * N;
  }
  for (int j = i + tid; j < hi; j += kThreads) {
    float x = to_f<T>(row[j]);
    if (x > st.m) {
      st.s = (st.s == 0.f) ? 0.f : st.s * ex2((st.m - x) * kLog2e);
      st.m = x;
      st.i = j;
    }
    st.s += ex2((x - st.m) * kLog2e);
  }
  return st;
}

struct RowParams {
  const void* logits;
  int vocab;
  int n_rows;        // rows with a ticket (all of them, valid or not)
  int split;         // CTAs per row (the row's cluster)
  int chunk;         // elements per CTA slice (multiple of 8)
  bool vec_ok;
  // verify phase: row r = b*max_search + j is valid only when j < n_search[b]
  const int* n_search;
  int max_search;
  float* out_conf;
  int* out_arg;
  float* part;                 // fused LM head: per-CTA statistics [CTA][row][3] (max, sum, argmax bits)
  unsigned* ticket;            // arrival counter of the rows, zero between calls
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

// Per-sequence decisions of the unmask phase; one warp per sequence. The
// rows' confidences and positions are first staged in shared memory (up to
// kStageRows rows), together with each sequence's row range (up to
// kStageSeqs sequences), so no step waits on a chain of memory loads: the
// ranking compares a sequence's rows in registers through warp shuffles.
// (kStageRows and kStageSeqs are template arguments: the vocab reduction
// stages up to 2048 rows of up to 1024 sequences, the fused LM head up to 64.)
template <int kStageRows, int kStageSeqs>
__device__ void decide_unmask(const RowParams& p, const int* st_seq, const int* st_pos, const float* st_conf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // parameters used inside loops, read once into registers
  const int R = p.n_rows, B = p.B, max_search = p.max_search;
  const float eps = p.eps;
  const bool force_progress = p.force_progress != 0;
  const int* __restrict__ row_seq = p.row_seq;
  const int* __restrict__ row_pos = p.row_pos;
  const float* out_conf = p.out_conf;
  unsigned char* __restrict__ commit = p.commit;
  int* __restrict__ search_rows = p.search_rows;
  __shared__ float s_conf[kStageRows];
  __shared__ int s_pos[kStageRows];
  __shared__ int s_lo[kStageSeqs], s_hi[kStageSeqs];
  __shared__ int bad;
  const bool staged = R <= kStageRows;
  const bool ranged = staged && B <= kStageSeqs;
  if (threadIdx.x == 0) bad = 0;
  if (ranged)
    for (int b = threadIdx.x; b < B; b += blockDim.x) s_lo[b] = s_hi[b] = 0;
  __syncthreads();
  // rows' sequences, positions and confidences: from the caller's shared
  // copies when given (no global round trip), else from global memory
  const int* seq_src = st_seq ? st_seq : row_seq;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    const int sq = seq_src[r];
    const int prev = r > 0 ? seq_src[r - 1] : -1;
    const int next = r + 1 < R ? seq_src[r + 1] : B;
    if (sq < 0 || sq >= B || next < sq) bad = 1;
    if (staged) {
      s_conf[r] = st_conf ? st_conf[r] : __ldcg(out_conf + r);
      s_pos[r] = st_pos ? st_pos[r] : row_pos[r];
    }
    if (ranged && sq >= 0 && sq < B) {  // rows are sorted by sequence (checked)
      if (prev != sq) s_lo[sq] = r;
      if (next != sq) s_hi[sq] = r + 1;
    }
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
    return;
  }
  auto conf = [&](int r) { return staged ? s_conf[r] : __ldcg(out_conf + r); };
  auto pos = [&](int r) { return staged ? s_pos[r] : row_pos[r]; };
  for (int b = warp; b < B; b += nw) {
    int lo, hi;
    if (ranged) {
      lo = s_lo[b];
      hi = s_hi[b];
    } else {  // rows of b: [lo, hi) by binary search on the sorted row_seq
      int a = 0, z = R;
      while (a < z) { int m = (a + z) >> 1; if (row_seq[m] < b) a = m + 1; else z = m; }
      lo = a;
      z = R;
      while (a < z) { int m = (a + z) >> 1; if (row_seq[m] <= b) a = m + 1; else z = m; }
      hi = a;
    }
    // eps rule
    bool any = false;
    for (int r = lo + lane; r < hi; r += 32) any |= conf(r) >= eps;
    any = __any_sync(0xffffffffu, any);
    int forced = -1;
    if (force_progress && !any && hi > lo) {
      // most confident row, lowest position on ties
      float bc = -1.f;
      int bp = 0x7fffffff, br = -1;
      for (int r = lo + lane; r < hi; r += 32) {
        const float c = conf(r);
        const int ps = pos(r);
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
    for (int r = lo + lane; r < hi; r += 32) commit[r] = (conf(r) >= eps || r == forced) ? 1 : 0;
    // rank the uncommitted rows by (conf desc, pos asc): lane l holds row
    // a0 + l and compares it with every row of the sequence, 32 at a time,
    // through shuffles
    int n_unc = 0;
    for (int a0 = lo; a0 < hi; a0 += 32) {
      const int ra = a0 + lane;
      const bool va = ra < hi;
      const float ca = va ? conf(ra) : 0.f;
      const int pa = va ? pos(ra) : 0;
      const bool ua = va && !(ca >= eps) && ra != forced;
      int rank = 0;
      for (int b0 = lo; b0 < hi; b0 += 32) {
        const int rb = b0 + lane;
        const bool vb = rb < hi;
        const float cb = vb ? conf(rb) : 0.f;
        const int pb = vb ? pos(rb) : 0;
        // an uncommitted row's key for the comparison; committed and absent
        // rows take -1 (below every confidence) so they never outrank
        const float kb = (vb && !(cb >= eps) && rb != forced) ? cb : -1.f;
        // every lane's (key, position) in turn, fully unrolled (shuffles from
        // constant lanes; a rolled loop over dynamic source lanes measured
        // three times slower on this one-warp path)
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float co = __shfl_sync(0xffffffffu, kb, k);
          const int po = __shfl_sync(0xffffffffu, pb, k);
          rank += (co > ca || (co == ca && po < pa)) ? 1 : 0;
        }
      }
      n_unc += ua ? 1 : 0;
      if (ua && rank < max_search) search_rows[b * max_search + rank] = ra;
    }
    for (int off = 16; off; off >>= 1) n_unc += __shfl_xor_sync(0xffffffffu, n_unc, off);
    const int ns = min(n_unc, max_search);
    for (int j = ns + lane; j < max_search; j += 32) search_rows[b * max_search + j] = -1;
    if (lane == 0) p.n_search_out[b] = ns;
  }
}

// Per-sequence prefix walk of the verify phase; one warp per sequence.
__device__ void decide_verify(const RowParams& p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // parameters used inside loops, read once into registers
  const int B = p.B, max_search = p.max_search;
  const float gamma = p.gamma;
  const int* __restrict__ n_search = p.n_search;
  const int* __restrict__ draft_tok = p.draft_tok;
  const int* out_arg = p.out_arg;
  const float* out_conf = p.out_conf;
  unsigned char* __restrict__ accept = p.accept;
  int* __restrict__ n_accept = p.n_accept;
  for (int b = warp; b < B; b += nw) {
    int n = n_search[b];
    if (n < 0 || n > max_search) {
      if (lane == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
      n = max(0, min(n, max_search));
    }
    int stop = n;
    for (int j0 = 0; j0 < n && stop == n; j0 += 32) {
      int j = j0 + lane;
      bool ok = true;
      if (j < n) {
        int r = b * max_search + j;
        ok = (draft_tok[r] == __ldcg(out_arg + r)) && (__ldcg(out_conf + r) >= gamma);
      }
      unsigned fails = __ballot_sync(0xffffffffu, !ok);
      if (fails) stop = j0 + __ffs(fails) - 1;
    }
    for (int j = lane; j < max_search; j += 32) accept[b * max_search + j] = (j < stop) ? 1 : 0;
    if (lane == 0) n_accept[b] = stop;
  }
}

// Calls with at most kThreads rows stage their decision inputs (rows'
// sequences and positions, and the merged confidences) in shared memory of
// the CTA that takes the decisions; every CTA loads the first two at its
// start, since any of them may be the last to arrive.
constexpr int kPreRows = kThreads;

template <typename T>
__global__ void __launch_bounds__(kThreads) row_reduce_kernel(RowParams p) {
  __shared__ Stat warp_stat[kThreads / 32];
  __shared__ float4 cl_stat[kMaxSplit];  // row leader: every slice's (max, sum, argmax bits)
  __shared__ unsigned go;
  __shared__ int pre_seq[kPreRows], pre_pos[kPreRows];
  __shared__ float pre_conf[kPreRows];
  const int row = blockIdx.x / p.split;
  const int sp = blockIdx.x % p.split;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  // verify phase: row r = b*max_search + j is valid only when j < n_search[b]
  const int n_rows_all = p.n_rows, phase = p.phase, ms_all = p.max_search;
  const int* n_search_in = p.n_search;
  auto row_valid = [=](int r) {
    if (r >= n_rows_all) return false;
    if (phase == 1) return r % ms_all < n_search_in[r / ms_all];
    return true;
  };
  const bool valid = row_valid(row);
  const Stat none{-INFINITY, 0.f, 0x7fffffff};
  const bool pre = phase == 0 && n_rows_all <= kPreRows;
  if (pre && (int)threadIdx.x < n_rows_all) {
    pre_seq[threadIdx.x] = p.row_seq[threadIdx.x];
    pre_pos[threadIdx.x] = p.row_pos[threadIdx.x];
  }
  Stat st = none;
  if (valid) {
    const T* base = reinterpret_cast<const T*>(p.logits) + (size_t)row * p.vocab;
    const int lo = sp * p.chunk;
    const int hi = min(p.vocab, lo + p.chunk);
    if (lo < hi) st = slice_stat<T>(base, lo, hi, p.vec_ok);
  }
  for (int off = 16; off; off >>= 1) st = shfl_merge(st, off);
  if (lane == 0) warp_stat[warp] = st;
  __syncthreads();
  if (warp == 0) {
    // block statistic: lanes 0..7 hold the warps' statistics, merged by a
    // fixed xor tree (lane 0 ends with the result)
    Stat acc = lane < kThreads / 32 ? warp_stat[lane] : none;
    for (int off = kThreads / 64; off; off >>= 1) acc = shfl_merge(acc, off);
    if (lane == 0 && p.split > 1) {
      // into slot sp of the row leader's (cluster rank 0) shared memory
      const uint32_t dst = tc::map_cluster(tc::smem_addr(&cl_stat[sp]), 0u);
      asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(acc.m), "f"(acc.s),
                   "f"(__int_as_float(acc.i)), "f"(0.f)
                   : "memory");
    }
    if (lane == 0) warp_stat[0] = acc;
  }
  if (p.split > 1) {
    // The CTAs of a row form a cluster: after the barrier (release /
    // acquire at cluster scope) the leader holds every slice's statistic.
    tc::cluster_sync();
    if (sp != 0) return;
  } else {
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (valid) {
      Stat acc = warp_stat[0];
      if (p.split > 1) {
        // the slices in rank order
        auto slot = [&](int k) { return Stat{cl_stat[k].x, cl_stat[k].y, __float_as_int(cl_stat[k].z)}; };
        acc = slot(0);
        for (int k = 1; k < p.split; ++k) acc = merge(acc, slot(k));
      }
      p.out_conf[row] = 1.f / acc.s;  // acc.s = sum exp(x - max) >= 1
      p.out_arg[row] = acc.i;
    }
    // one ticket per row for the whole grid: the row leader that arrives
    // last takes the decisions. The add releases this row's result and,
    // for the last arrival, acquires every other row's (passed on to the
    // CTA's threads by the barrier)
    unsigned t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(p.ticket) : "memory");
    go = t == (unsigned)(gridDim.x / p.split) - 1u ? 1u : 0u;
  }
  __syncthreads();
  if (!go) return;
  if (p.phase == 0) {
    if (pre) {
      // every row leader wrote its row's confidence to global memory
      for (int r = threadIdx.x; r < n_rows_all; r += kThreads) pre_conf[r] = __ldcg(p.out_conf + r);
    }
    __syncthreads();
    decide_unmask<2048, 1024>(p, pre ? pre_seq : nullptr, pre ? pre_pos : nullptr, pre ? pre_conf : nullptr);
  } else {
    decide_verify(p);
  }
  if (threadIdx.x == 0) *p.ticket = 0u;  // ready for the next call
}

template <typename T>
cudaError_t launch_phase(fdl_ctx* ctx, RowParams p) {
  if (p.n_rows == 0) return cudaSuccess;
  const int V = p.vocab;
  // about four CTAs per SM in total; slices of at least 2048 elements
  int split = (4 * ctx->num_sms + p.n_rows - 1) / p.n_rows;
  split = max(1, min(split, kMaxSplit));
  split = min(split, max(1, V / 2048));
  int chunk = (V + split - 1) / split;
  chunk = (chunk + 7) / 8 * 8;
  split = (V + chunk - 1) / chunk;
  p.split = split;
  p.chunk = chunk;
  p.vec_ok = ((reinterpret_cast<uintptr_t>(p.logits) & 15) == 0) && ((size_t)V * sizeof(T)) % 16 == 0;
  return fdl_launch_pdl(row_reduce_kernel<T>, dim3((unsigned)(p.n_rows * split)), dim3(kThreads), 0, ctx->stream,
                        split, p);
}


// ---------------------------------------------------------------------------
// Fused LM head + unmasking: logits = hidden . W_lm^T are reduced to each
// window row's (max, argmax, sum of exponentials) tile by tile and never
// stored. Same orientation as the projection ("swap AB"): a vocabulary tile
// of 128 rows (TMEM lanes) against all window rows (<= 64, TMEM columns),
// bf16 in, fp32 accumulate (tcgen05.mma). The kernel is persistent: one CTA
// per SM loops over the tiles t = blockIdx.x + k * gridDim.x, its TMA ring
// streams the weight across tile boundaries, and two TMEM accumulators let
// the epilogue of tile k overlap the products of tile k + 1. The epilogue
// stages each fp32 tile in shared memory, reduces every column (window row)
// over the tile's vocabulary rows and merges it into the CTA's running
// statistics in tile order; the CTA publishes them, and the last CTA to take
// the grid ticket merges the CTAs' statistics in CTA order and takes the
// unmask decisions (decide_unmask above). Every merge is in a fixed order.
// ---------------------------------------------------------------------------
constexpr int kLmBM = 128;  // vocabulary rows per tile
constexpr int kLmBN = 64;   // window rows (the whole call)
constexpr int kLmBK = 64;
constexpr int kLmStages = 6;
constexpr int kLmThreads = 192;
constexpr int kLmA = kLmBM * kLmBK * 2;
constexpr int kLmB = kLmBN * kLmBK * 2;
constexpr int kLmStage = kLmA + kLmB;
constexpr int kLmPipe = kLmStages * kLmStage;
constexpr int kLmXs = kLmBM + 1;  // padded row of the fp32 tile: column-wise reads are conflict-free
constexpr int kLmXsBytes = kLmBN * kLmXs * 4;
constexpr int kLmSmem = 1024 + kLmPipe + kLmXsBytes + 256;
static_assert(kLmSmem <= 227 * 1024, "shared memory budget");

struct LmParams {
  RowParams rp;  // decisions of the unmask phase; rp.part holds the CTAs' statistics
  int vocab, nkb, n_tiles;
};

__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                   const LmParams p) {
  extern __shared__ uint8_t lm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(lm_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pipe = smem;
  float* xs = reinterpret_cast<float*>(smem + kLmPipe);  // [window row][vocab row], padded
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLmPipe + kLmXsBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kLmStages;
  uint64_t* tmem_full = bars + 2 * kLmStages;   // [2]
  uint64_t* tmem_empty = tmem_full + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ Stat half_stat[kLmBN];
  __shared__ unsigned go;
  __shared__ int pre_seq[kLmBN], pre_pos[kLmBN];
  __shared__ float pre_conf[kLmBN];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.rp.n_rows;
  const int n_mine = (p.n_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // tiles of this CTA
  const int n_it = n_mine * p.nkb;                                                          // k-blocks of this CTA
  auto tile_of = [&](int j) { return (int)blockIdx.x + j * (int)gridDim.x; };
  const int pre = min(n_it, kLmStages);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&tmem_full[s], 1);
      tc::mbar_init(&tmem_empty[s], 4);  // the four epilogue warps
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tm_w);
    tc::prefetch_tensormap(&tm_h);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 2 * kLmBN);
    tc::tmem_relinquish();
  }
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  auto issue = [&](int it, int s) {
    const int j = it / p.nkb, kb = it % p.nkb;
    uint8_t* a = pipe + s * kLmStage;
    tc::mbar_arrive_expect_tx(&full[s], kLmStage);
    tc::tma_load_2d(a, &tm_w, kb * kLmBK, tile_of(j) * kLmBM, &full[s]);
    tc::tma_load_2d(a + kLmA, &tm_h, kb * kLmBK, 0, &full[s]);
  };
  if (threadIdx.x == 0)
    for (int it = 0; it < pre; ++it) issue(it, it);
  // every CTA may be the last: it stages the unmask decisions' inputs at its start
  if (p.rp.phase == 0 && (int)threadIdx.x < R) {
    pre_seq[threadIdx.x] = p.rp.row_seq[threadIdx.x];
    pre_pos[threadIdx.x] = p.rp.row_pos[threadIdx.x];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int it = pre; it < n_it; ++it) {
        const int s = it % kLmStages;
        if (!tc::mbar_wait(&empty[s], ((uint32_t)(it / kLmStages) & 1u) ^ 1u, abort_flag)) break;
        issue(it, s);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kLmBM, kLmBN);
      int it = 0;
      bool ok = true;
      for (int j = 0; ok && j < n_mine; ++j) {
        const int buf = j & 1;
        // the epilogue has read this accumulator's previous tile (j - 2)
        if (j >= 2 && !tc::mbar_wait(&tmem_empty[buf], (uint32_t)((j - 2) >> 1) & 1u, abort_flag)) break;
        tc::fence_after_sync();
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const int s = it % kLmStages;
          if (!tc::mbar_wait(&full[s], (uint32_t)(it / kLmStages) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a = tc::smem_addr(pipe + s * kLmStage);
          const uint64_t ad = tc::desc_kmajor_sw128(a);
          const uint64_t bd = tc::desc_kmajor_sw128(a + kLmA);
#pragma unroll
          for (int k = 0; k < kLmBK / 16; ++k)
            tc::mma_bf16_ss(tmem + buf * kLmBN, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        if (ok) tc::mma_commit(&tmem_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int t = threadIdx.x - 64;  // 0..127
    const int q = warp & 3;
    const int tq = q * 32 + lane;    // TMEM lane = vocabulary row tile * 128 + tq
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    const int c = t & (kLmBN - 1), half = t >> 6;
    Stat run{-INFINITY, 0.f, 0x7fffffff};  // half 0: column c's statistics over this CTA's tiles so far
    for (int j = 0; j < n_mine; ++j) {
      const int buf = j & 1;
      const int f0 = tile_of(j) * kLmBM;
      const bool got = __all_sync(0xffffffffu, tc::mbar_wait(&tmem_full[buf], (uint32_t)(j >> 1) & 1u, abort_flag));
      tc::fence_after_sync();
      tc::named_bar(1, 128);  // the previous tile's column reads of xs are done
      const bool live = f0 + tq < p.vocab;
#pragma unroll 1
      for (int c0 = 0; c0 < kLmBN; c0 += 16) {
        float v[16];
        if (got) tc::tmem_ld_32x32b_x16(t_lane + buf * kLmBN + c0, v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) xs[(c0 + jj) * kLmXs + tq] = (got && live) ? v[jj] : -INFINITY;
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tmem_empty[buf]);  // the accumulator may take tile j + 2
      tc::named_bar(1, 128);
      // column c over the tile's 128 vocabulary rows: two threads per column,
      // 64 rows each, the maximum (first on ties) before any exponential
      Stat st{-INFINITY, 0.f, 0x7fffffff};
      if (c < R) {
        const float* col = xs + c * kLmXs + half * 64;
        float m = -INFINITY;
        int mi = 0;
        for (int r = 0; r < 64; ++r)
          if (col[r] > m) {
            m = col[r];
            mi = r;
          }
        if (m != -INFINITY) {
          const float mb = m * kLog2e;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          for (int r = 0; r < 64; r += 4) {
            a0 += ex2(fmaf(col[r], kLog2e, -mb));
            a1 += ex2(fmaf(col[r + 1], kLog2e, -mb));
            a2 += ex2(fmaf(col[r + 2], kLog2e, -mb));
            a3 += ex2(fmaf(col[r + 3], kLog2e, -mb));
          }
          st = Stat{m, (a0 + a1) + (a2 + a3), f0 + half * 64 + mi};
        }
      }
      if (half == 1) half_stat[c] = st;
      tc::named_bar(1, 128);
      if (half == 0 && c < R) run = merge(run, merge(st, half_stat[c]));  // tile order; lower rows first
    }
    if (half == 0 && c < R) {
      float* slot = p.rp.part + ((size_t)blockIdx.x * R + c) * 3;
      __stcg(slot, run.m);
      __stcg(slot + 1, run.s);
      __stcg(slot + 2, __int_as_float(run.i));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * kLmBN);
  if (threadIdx.x == 0) {
    if (*abort_flag) fdl::raise_error(p.rp.err, FDL_DEVERR_TIMEOUT);
    // every CTA's statistics are released by its own add; the last arrival
    // acquires all of them (and passes them on with the barrier below)
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(p.rp.ticket) : "memory");
    go = tk == gridDim.x - 1u ? 1u : 0u;
  }
  __syncthreads();
  if (!go) return;
  // ---- last CTA: each window row's statistics over all CTAs, merged in a
  // fixed order (lane l takes CTAs l, l + 32, ... in order, then a fixed xor
  // tree), then the decisions
  const Stat none{-INFINITY, 0.f, 0x7fffffff};
  for (int c = warp; c < R; c += kLmThreads / 32) {
    Stat acc = none;
    for (int cta = lane; cta < (int)gridDim.x; cta += 32) {
      const float* o = p.rp.part + ((size_t)cta * R + c) * 3;
      acc = merge(acc, Stat{__ldcg(o), __ldcg(o + 1), __float_as_int(__ldcg(o + 2))});
    }
    for (int off = 16; off; off >>= 1) acc = shfl_merge(acc, off);
    if (lane == 0) {
      const float conf = acc.s > 0.f ? 1.f / acc.s : 0.f;
      // verify: row b*max_search + j holds a mask view only for j < n_search[b]
      const bool real = p.rp.phase == 0 || c % p.rp.max_search < __ldg(p.rp.n_search + c / p.rp.max_search);
      if (real) {
        p.rp.out_conf[c] = conf;
        p.rp.out_arg[c] = acc.i;
      }
      pre_conf[c] = conf;
    }
  }
  __syncthreads();
  if (p.rp.phase == 0)
    decide_unmask<kLmBN, kLmBN>(p.rp, pre_seq, pre_pos, pre_conf);
  else
    decide_verify(p.rp);
  if (threadIdx.x == 0) *p.rp.ticket = 0u;  // ready for the next call
}

// ---------------------------------------------------------------------------
// Fused LM head for more than 64 rows. With that many rows the window rows
// fill the M = 128 datapath themselves, so a tile takes the plain
// orientation: 128 window rows (TMEM lanes) x 256 vocabulary entries (TMEM
// columns), D = H_tile . W_tile^T, bf16 in, fp32 accumulate (tcgen05.mma).
// Every epilogue thread then reduces its own window row along the
// vocabulary, with no cross-thread reduction. The grid is n_rt row tiles x g
// CTAs; CTA (rt, i) takes the contiguous vocabulary tiles [i n_vt / g,
// (i + 1) n_vt / g) of row tile rt, so the n_rt CTAs of one vocabulary range
// stream the same weight tiles at about the same time and the weight is read
// from DRAM about once. A 4-stage TMA ring feeds the MMA; two TMEM
// accumulators (2 x 256 columns) let the epilogue of one tile overlap the
// products of the next. Each row's (max, sum, argmax) runs over the CTA's
// tiles in order in registers; the CTA publishes them, the last CTA of the
// row tile (one ticket per row tile) merges the g CTAs' statistics in CTA
// order and writes the rows' confidences and argmaxes, and the row tile that
// finishes last (a second ticket) takes the unmask or verify decisions.
// Every merge is in a fixed order.
// ---------------------------------------------------------------------------
constexpr int kRM = 128;  // window rows per row tile
constexpr int kRN = 256;  // vocabulary entries per tile
constexpr int kRK = 64;
constexpr int kRStages = 4;
constexpr int kRA = kRM * kRK * 2;
constexpr int kRB = kRN * kRK * 2;
constexpr int kRStage = kRA + kRB;
constexpr int kRPipe = kRStages * kRStage;
constexpr int kRSmem = 1024 + kRPipe + 256;
static_assert(kRSmem + 8 * 2048 + 8 * 1024 + 64 <= 227 * 1024, "shared memory budget (with the decision staging)");

struct LmRowsParams {
  RowParams rp;           // decisions; rp.part holds the CTAs' per-row statistics [CTA][128][3]
  int vocab, nkb, n_vt, g, n_rt;
  unsigned* rt_tickets;   // [n_rt] arrival counters of the row tiles, zero between calls
};

__global__ void __launch_bounds__(kLmThreads, 1)
    lm_rows_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                   const LmRowsParams p) {
  extern __shared__ uint8_t lr_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(lr_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pipe = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRPipe);
  uint64_t* full = bars;
  uint64_t* empty = bars + kRStages;
  uint64_t* tmem_full = bars + 2 * kRStages;  // [2]
  uint64_t* tmem_empty = tmem_full + 2;       // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ unsigned go;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = p.rp.n_rows;
  const int rt = (int)blockIdx.x / p.g, gi = (int)blockIdx.x % p.g;
  const int vt0 = (int)((long long)gi * p.n_vt / p.g), vt1 = (int)((long long)(gi + 1) * p.n_vt / p.g);
  const int n_mine = vt1 - vt0;
  const int n_it = n_mine * p.nkb;
  const int pre = min(n_it, kRStages);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&tmem_full[s], 1);
      tc::mbar_init(&tmem_empty[s], 4);  // the four epilogue warps
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tm_w);
    tc::prefetch_tensormap(&tm_h);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 2 * kRN);
    tc::tmem_relinquish();
  }
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  auto issue = [&](int it, int s) {
    const int j = it / p.nkb, kb = it % p.nkb;
    uint8_t* a = pipe + s * kRStage;
    tc::mbar_arrive_expect_tx(&full[s], kRStage);
    tc::tma_load_2d(a, &tm_h, kb * kRK, rt * kRM, &full[s]);
    tc::tma_load_2d(a + kRA, &tm_w, kb * kRK, (vt0 + j) * kRN, &full[s]);
  };
  if (threadIdx.x == 0)
    for (int it = 0; it < pre; ++it) issue(it, it);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int it = pre; it < n_it; ++it) {
        const int s = it % kRStages;
        if (!tc::mbar_wait(&empty[s], ((uint32_t)(it / kRStages) & 1u) ^ 1u, abort_flag)) break;
        issue(it, s);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kRM, kRN);
      int it = 0;
      bool ok = true;
      for (int j = 0; ok && j < n_mine; ++j) {
        const int buf = j & 1;
        // the epilogue has read this accumulator's previous tile (j - 2)
        if (j >= 2 && !tc::mbar_wait(&tmem_empty[buf], (uint32_t)((j - 2) >> 1) & 1u, abort_flag)) break;
        tc::fence_after_sync();
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const int s = it % kRStages;
          if (!tc::mbar_wait(&full[s], (uint32_t)(it / kRStages) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a = tc::smem_addr(pipe + s * kRStage);
          const uint64_t ad = tc::desc_kmajor_sw128(a);
          const uint64_t bd = tc::desc_kmajor_sw128(a + kRA);
#pragma unroll
          for (int k = 0; k < kRK / 16; ++k)
            tc::mma_bf16_ss(tmem + buf * kRN, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        if (ok) tc::mma_commit(&tmem_full[buf]);
      }
      // every product issued has finished before the TMEM is freed
      const int last = ok ? n_mine - 1 : -1;
      if (last >= 0) {
        long long t0 = clock64();
        while (!tc::mbar_try_wait(&tmem_full[last & 1], (uint32_t)(last >> 1) & 1u) &&
               clock64() - t0 < tc::kWaitBudgetCycles) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // thread = window row rt * 128 + row (its TMEM lane); the row's running
    // statistics over this CTA's vocabulary tiles, in tile order
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    Stat run{-INFINITY, 0.f, 0x7fffffff};
    for (int j = 0; j < n_mine; ++j) {
      const int buf = j & 1;
      const bool got = __all_sync(0xffffffffu, tc::mbar_wait(&tmem_full[buf], (uint32_t)(j >> 1) & 1u, abort_flag));
      tc::fence_after_sync();
      const int v0 = (vt0 + j) * kRN;
#pragma unroll 1
      for (int c0 = 0; c0 < kRN; c0 += 64) {
        float v[64];
        if (!got) break;
        tc::tmem_ld_32x32b_x64(t_lane + buf * kRN + c0, v);
        const int nvalid = min(64, p.vocab - (v0 + c0));
        // the chunk's maximum (first index on ties) before any exponential
        float m = -INFINITY;
        int mi = 0;
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e < nvalid && v[e] > m) {
            m = v[e];
            mi = e;
          }
        if (m == -INFINITY) continue;
        const float mb = m * kLog2e;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          a0 += e < nvalid ? ex2(fmaf(v[e], kLog2e, -mb)) : 0.f;
          a1 += e + 1 < nvalid ? ex2(fmaf(v[e + 1], kLog2e, -mb)) : 0.f;
          a2 += e + 2 < nvalid ? ex2(fmaf(v[e + 2], kLog2e, -mb)) : 0.f;
          a3 += e + 3 < nvalid ? ex2(fmaf(v[e + 3], kLog2e, -mb)) : 0.f;
        }
        run = merge(run, Stat{m, (a0 + a1) + (a2 + a3), v0 + c0 + mi});
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tmem_empty[buf]);  // the accumulator may take tile j + 2
    }
    if (rt * kRM + row < R) {
      float* slot = p.rp.part + ((size_t)blockIdx.x * kRM + row) * 3;
      __stcg(slot, run.m);
      __stcg(slot + 1, run.s);
      __stcg(slot + 2, __int_as_float(run.i));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * kRN);
  if (threadIdx.x == 0) {
    if (*abort_flag) fdl::raise_error(p.rp.err, FDL_DEVERR_TIMEOUT);
    // this CTA's statistics are released by its add; the row tile's last
    // arrival acquires the others' (passed on by the barrier below)
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(p.rt_tickets + rt) : "memory");
    go = tk == (unsigned)p.g - 1u ? 1u : 0u;
  }
  __syncthreads();
  if (!go) return;
  // ---- last CTA of the row tile: each row's statistics over the g CTAs in
  // CTA order (= vocabulary order), then the row's confidence and argmax
  if (threadIdx.x < kRM) {
    const int r = rt * kRM + (int)threadIdx.x;
    if (r < R) {
      Stat acc{-INFINITY, 0.f, 0x7fffffff};
      for (int i = 0; i < p.g; ++i) {
        const float* o = p.rp.part + ((size_t)(rt * p.g + i) * kRM + threadIdx.x) * 3;
        acc = merge(acc, Stat{__ldcg(o), __ldcg(o + 1), __float_as_int(__ldcg(o + 2))});
      }
      // verify: row b*max_search + j holds a mask view only for j < n_search[b]
      const bool real = p.rp.phase == 0 || r % p.rp.max_search < __ldg(p.rp.n_search + r / p.rp.max_search);
      if (real) {
        p.rp.out_conf[r] = acc.s > 0.f ? 1.f / acc.s : 0.f;
        p.rp.out_arg[r] = acc.i;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.rt_tickets[rt] = 0u;  // every CTA of the row tile has arrived: ready for the next call
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(p.rp.ticket) : "memory");
    go = tk == (unsigned)p.n_rt - 1u ? 1u : 0u;
  }
  __syncthreads();
  if (!go) return;
  // ---- the row tile that finished last: the decisions over every row
  if (p.rp.phase == 0)
    decide_unmask<2048, 1024>(p.rp, nullptr, nullptr, nullptr);
  else
    decide_verify(p.rp);
  if (threadIdx.x == 0) *p.rp.ticket = 0u;  // ready for the next call
}

PFN_cuTensorMapEncodeTiled_v12000 lm_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// bf16 row-major [rows, cols], box kLmBK columns x box_rows rows, 128-byte swizzle
bool lm_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = lm_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kLmBK, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Decision parameters shared by both LM-head kernels.
void lm_decision_params(RowParams& rp, fdl_ctx* ctx, const fdl_unmask_args* a, bool verify, int R) {
  rp.n_rows = R;
  rp.part = ctx->lm_part;
  rp.ticket = ctx->tickets + 2;
  rp.err = ctx->err_word;
  rp.B = a->B;
  rp.max_search = a->max_search;
  if (!verify) {
    rp.phase = 0;
    rp.out_conf = a->conf;
    rp.out_arg = a->argmax;
    rp.row_seq = a->row_seq;
    rp.row_pos = a->row_pos;
    rp.eps = a->eps;
    rp.force_progress = a->force_progress;
    rp.commit = a->commit;
    rp.search_rows = a->search_rows;
    rp.n_search_out = a->n_search;
  } else {
    rp.phase = 1;
    rp.out_conf = a->mask_conf;
    rp.out_arg = a->mask_argmax;
    rp.n_search = a->n_search;
    rp.draft_tok = a->draft_tok;
    rp.gamma = a->gamma;
    rp.accept = a->accept;
    rp.n_accept = a->n_accept;
  }
}

cudaError_t launch_lm_rows(fdl_ctx* ctx, const void* hidden, const void* w_lm, const fdl_unmask_args* a, bool verify,
                           int R) {
  const fdl_config& c = ctx->cfg;
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)lm_rows_kernel, ctx->device, kRSmem)) return e;
  CUtensorMap mw, mh;
  if (!lm_map(&mw, w_lm, (uint64_t)c.vocab, c.d_model, kRN) || !lm_map(&mh, hidden, R, c.d_model, kRM))
    return cudaErrorInvalidValue;
  LmRowsParams p = {};
  lm_decision_params(p.rp, ctx, a, verify, R);
  p.vocab = c.vocab;
  p.nkb = c.d_model / kRK;
  p.n_vt = (c.vocab + kRN - 1) / kRN;
  p.n_rt = (R + kRM - 1) / kRM;
  // CTAs per row tile: the row tiles together fill the SMs, each CTA with at
  // least one vocabulary tile
  p.g = max(1, min(ctx->num_sms / p.n_rt, p.n_vt));
  p.rt_tickets = ctx->lm_rt_tickets;
  if (p.n_rt > ctx->lm_rt_ticket_count || (size_t)p.n_rt * p.g * kRM * 3 > ctx->lm_part_floats)
    return cudaErrorInvalidValue;
  return fdl_launch_pdl(lm_rows_kernel, dim3((unsigned)(p.n_rt * p.g)), dim3(kLmThreads), kRSmem, ctx->stream, 1, mw,
                        mh, p);
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

int fdl_lm_head_max_rows() { return kLmBN; }

size_t fdl_lm_partial_floats(int num_sms, int max_rows) {
  // the small kernel: one set of <= 64 rows' statistics per CTA; the many-row
  // kernel: 128 rows per CTA over n_rt x g <= max(SMs, row tiles) CTAs
  const size_t n_rt = (size_t)(max_rows + kRM - 1) / kRM;
  const size_t small = (size_t)num_sms * kLmBN * 3;
  const size_t rows = (n_rt > (size_t)num_sms ? n_rt : (size_t)num_sms) * kRM * 3;
  return small > rows ? small : rows;
}

int fdl_lm_row_tiles(int max_rows) { return (max_rows + kRM - 1) / kRM; }

cudaError_t fdl_launch_lm_head(fdl_ctx* ctx, const void* hidden, const void* w_lm, const fdl_unmask_args* a,
                               bool verify) {
  const fdl_config& c = ctx->cfg;
  const int R = verify ? a->B * a->max_search : a->R_w;
  if (c.dtype != FDL_BF16 || R < 1 || R > c.max_rows || c.d_model % kLmBK != 0 || !ctx->lm_part)
    return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w_lm)) & 15) return cudaErrorMisalignedAddress;
  if (R > kLmBN) return launch_lm_rows(ctx, hidden, w_lm, a, verify, R);
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)lm_head_kernel, ctx->device, kLmSmem)) return e;
  CUtensorMap mw, mh;
  if (!lm_map(&mw, w_lm, (uint64_t)c.vocab, c.d_model, kLmBM) || !lm_map(&mh, hidden, R, c.d_model, kLmBN))
    return cudaErrorInvalidValue;
  LmParams p = {};
  lm_decision_params(p.rp, ctx, a, verify, R);
  p.vocab = c.vocab;
  p.nkb = c.d_model / kLmBK;
  p.n_tiles = (c.vocab + kLmBM - 1) / kLmBM;
  // persistent: one CTA per SM (or per tile when there are fewer tiles)
  const int grid = min(p.n_tiles, ctx->num_sms);
  return fdl_launch_pdl(lm_head_kernel, dim3((unsigned)grid), dim3(kLmThreads), kLmSmem, ctx->stream, 1, mw, mh, p);
}
