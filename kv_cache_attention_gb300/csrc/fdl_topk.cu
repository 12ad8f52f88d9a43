// Top-k of the attention-mass tracker scores (next step's tracked set).
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...",
// section "Method steps in detail", Algorithm 2 step 4: the k decoded
// tokens with the largest a_i (Eq. (2)) are refreshed next step.
//
// One CTA per sequence; scores map to order-preserving 32-bit keys (0 marks
// an ineligible position). The k-th largest key is found exactly by radix
// select over 8-bit digits; ties at that threshold go to the lowest
// positions; the <= k survivors are ranked by (score desc, position asc).
//
// topk_kernel (rows of up to kStage positions, the common case) is built
// for latency: each thread keeps its contiguous run of keys in registers;
// the digits start at the highest bit where the eligible keys differ (their
// AND/OR, reduced while staging); every warp finds the threshold bin itself
// (no broadcast barrier); histograms rotate over three buffers so clearing
// the next one needs no barrier of its own; and refinement stops as soon as
// at most 256 keys lie at or above the current bin, which then rank among
// themselves by counting (one pass on spread-out scores). Only when more
// keys than fit tie at the full threshold key are the ties cut by position
// with a block prefix count. topk_large_kernel handles longer rows from
// global memory.
#include "fdl_internal.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kMaxK = 1024;
constexpr int kStage = 8192;

__global__ void __launch_bounds__(kThreads)
topk_large_kernel(const float* __restrict__ scores, const unsigned char* __restrict__ eligible, int ld,
            const int* __restrict__ seq_len, int k, int* __restrict__ idx_out, int* __restrict__ cnt_out,
            unsigned* err) {
  __shared__ unsigned hist[256];
  __shared__ unsigned s_prefix, s_remaining, s_count;
  __shared__ unsigned warp_sum[kThreads / 32];
  __shared__ unsigned sel_key[kMaxK];
  __shared__ int sel_pos[kMaxK];
  __shared__ unsigned n_sel;
  __shared__ unsigned skey[kStage];  // order key of eligible positions, 0 = not eligible

  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  int n = seq_len[b];
  if (n < 0 || n > ld) {
    if (tid == 0) fdl::raise_error(err, FDL_DEVERR_INDEX);
    n = max(0, min(n, ld));
  }
  const float* sc = scores + (size_t)b * ld;
  const unsigned char* el = eligible + (size_t)b * ld;
  const bool staged = n <= kStage;
  // order key of position i (0 for an ineligible position; real scores map
  // to keys >= 1 because NaN is excluded)
  auto key_of = [&](int i) -> unsigned {
    if (staged) return skey[i];
    return el[i] ? fdl::float_order_key(sc[i]) : 0u;
  };

  // stage keys and count eligible positions
  unsigned cnt = 0;
  for (int i = tid; i < n; i += kThreads) {
    const bool e = el[i] != 0;
    cnt += e ? 1u : 0u;
    if (staged) skey[i] = e ? fdl::float_order_key(sc[i]) : 0u;
  }
  for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  if (lane == 0) warp_sum[warp] = cnt;
  __syncthreads();
  if (tid == 0) {
    unsigned t = 0;
    for (int w = 0; w < kThreads / 32; ++w) t += warp_sum[w];
    s_count = t;
    s_prefix = 0u;
    s_remaining = min((unsigned)k, t);
    n_sel = 0u;
  }
  __syncthreads();
  const unsigned total = s_count;
  const unsigned kk = min((unsigned)k, total);
  // threshold key T: the kk-th largest order key
  bool take_all = (kk == total);
  unsigned mask = 0u;
  if (!take_all) {
    for (int digit = 3; digit >= 0; --digit) {
      for (int i = tid; i < 256; i += kThreads) hist[i] = 0u;
      __syncthreads();
      const unsigned prefix = s_prefix;
      const int shift = 8 * digit;
      for (int i = tid; i < n; i += kThreads) {
        const unsigned key = key_of(i);
        if (key != 0u && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l down to 248-8l; an exclusive scan from the
        // top bin finds the bin where the running count reaches `remaining`
        const unsigned rem = s_remaining;
        unsigned own = 0u;
#pragma unroll
        for (int t = 0; t < 8; ++t) own += hist[255 - 8 * lane - t];
        unsigned incl = own;
        for (int off = 1; off < 32; off <<= 1) {
          const unsigned v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        const unsigned before = incl - own;
        const bool mine = before < rem && rem <= incl;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        if (mine && lane == __ffs(who) - 1) {
          unsigned acc = before;
          int bin = 255 - 8 * lane;
          for (int t = 0; t < 7; ++t, --bin) {
            if (acc + hist[bin] >= rem) break;
            acc += hist[bin];
          }
          s_remaining = rem - acc;
          s_prefix = prefix | ((unsigned)bin << shift);
        }
      }
      mask |= 255u << shift;
      __syncthreads();
    }
  }
  const unsigned T = s_prefix;
  const unsigned need = s_remaining;  // how many keys equal to T to take
  // Select: every key > T, plus the first `need` keys == T in position order.
  // Each thread owns a contiguous run of positions for the tie prefix count.
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  unsigned ties = 0;
  if (!take_all)
    for (int i = lo; i < hi; ++i)
      if (key_of(i) == T) ++ties;
  // exclusive scan of ties over threads
  unsigned incl = ties;
  for (int off = 1; off < 32; off <<= 1) {
    unsigned v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  __syncthreads();
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned v = lane < kThreads / 32 ? warp_sum[lane] : 0u;
    unsigned x = v;
    for (int off = 1; off < 32; off <<= 1) {
      unsigned y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane < kThreads / 32) warp_sum[lane] = x - v;  // exclusive warp offsets
  }
  __syncthreads();
  unsigned tie_rank = warp_sum[warp] + incl - ties;
  for (int i = lo; i < hi; ++i) {
    const unsigned key = key_of(i);
    if (key == 0u) continue;
    bool take;
    if (take_all) take = true;
    else if (key > T) take = true;
    else if (key == T) take = (tie_rank++ < need);
    else take = false;
    if (take) {
      unsigned slot = atomicAdd(&n_sel, 1u);
      if (slot < (unsigned)kMaxK) {
        sel_key[slot] = key;
        sel_pos[slot] = i;
      }
    }
  }
  __syncthreads();
  const int m = (int)min(n_sel, (unsigned)kMaxK);
  if (tid == 0 && n_sel != kk) fdl::raise_error(err, FDL_DEVERR_SHAPE);
  // rank by (key desc, position asc) and scatter
  for (int s = tid; s < m; s += kThreads) {
    unsigned key = sel_key[s];
    int pos = sel_pos[s];
    int rank = 0;
    for (int o = 0; o < m; ++o) {
      unsigned ko = sel_key[o];
      rank += (ko > key || (ko == key && sel_pos[o] < pos)) ? 1 : 0;
    }
    if (rank < k) idx_out[(size_t)b * k + rank] = pos;
  }
  for (int t = m + tid; t < k; t += kThreads) idx_out[(size_t)b * k + t] = -1;
  if (tid == 0) cnt_out[b] = m;
}


constexpr int kPer = kStage / kThreads;  // keys per thread held in registers
constexpr unsigned kCandStop = 256;      // stop refining once this few candidates remain

__device__ __forceinline__ unsigned warp_incl_scan(unsigned v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += y;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads)
topk_kernel(const float* __restrict__ scores, const unsigned char* __restrict__ eligible, int ld,
            const int* __restrict__ seq_len, int k, int* __restrict__ idx_out, int* __restrict__ cnt_out,
            unsigned* err) {
  constexpr int kWarps = kThreads / 32;
  __shared__ unsigned skey[kStage];
  __shared__ __align__(16) unsigned hist[3][256];
  __shared__ unsigned w_cnt[kWarps], w_or[kWarps], w_and[kWarps], w_tie[kWarps], w_cand[kWarps];
  // candidate (key, position) packed as key << 32 | ~position: a larger
  // value ranks first, so ties on the key go to the lower position
  __shared__ __align__(16) unsigned long long cand[kMaxK];

  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  int n = seq_len[b];
  if (n < 0 || n > ld) {
    if (tid == 0) fdl::raise_error(err, FDL_DEVERR_INDEX);
    n = max(0, min(n, ld));
  }
  const float* sc = scores + (size_t)b * ld;
  const unsigned char* el = eligible + (size_t)b * ld;

  // stage keys (both loads in flight together), count the eligible ones and
  // reduce the AND / OR of their keys
  unsigned cnt = 0u, kor = 0u, kand = 0xffffffffu;
  for (int i = tid; i < n; i += kThreads) {
    const unsigned char e = el[i];
    const float x = sc[i];
    const unsigned key = e ? fdl::float_order_key(x) : 0u;
    skey[i] = key;
    if (key) {
      ++cnt;
      kor |= key;
      kand &= key;
    }
  }
  for (int off = 16; off; off >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    kor |= __shfl_xor_sync(0xffffffffu, kor, off);
    kand &= __shfl_xor_sync(0xffffffffu, kand, off);
  }
  if (lane == 0) {
    w_cnt[warp] = cnt;
    w_or[warp] = kor;
    w_and[warp] = kand;
  }
  if (tid < 256) hist[0][tid] = 0u;
  __syncthreads();
  // every lane of every warp forms the block totals (lanes past the warp
  // count contribute the identity; the xor tree spans all 32 lanes, so every
  // lane ends with the same values)
  unsigned total = lane < kWarps ? w_cnt[lane] : 0u;
  kor = lane < kWarps ? w_or[lane] : 0u;
  kand = lane < kWarps ? w_and[lane] : 0xffffffffu;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    total += __shfl_xor_sync(0xffffffffu, total, off);
    kor |= __shfl_xor_sync(0xffffffffu, kor, off);
    kand &= __shfl_xor_sync(0xffffffffu, kand, off);
  }
  const unsigned kk = min((unsigned)k, total);
  const bool take_all = kk == total;

  // this thread's contiguous run of positions [lo, lo + per)
  const int per = (n + kThreads - 1) / kThreads;  // <= kPer
  const int lo = tid * per;
  unsigned r[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) r[j] = (j < per && lo + j < n) ? skey[lo + j] : 0u;

  // Refine a lower bound `low` on the kk-th largest key with 8-bit digits,
  // starting at the highest bit where the eligible keys differ, until at
  // most kCandStop keys are >= low (every one of the top kk is). If even the
  // full key leaves more (many keys equal to the threshold T), the ties are
  // cut by position instead.
  unsigned low = 1u;            // take_all: every eligible key
  unsigned T = kand, need = kk;
  bool cut_ties = false;
  const unsigned diff = kor ^ kand;
  if (!take_all) {
    if (diff == 0u) {
      cut_ties = true;  // all eligible keys are equal
    } else {
      const int top = ((31 - __clz((int)diff)) >> 3) << 3;  // digit holding the highest differing bit
      unsigned mask = top + 8 >= 32 ? 0u : ~((1u << (top + 8)) - 1u);
      unsigned prefix = kand & mask;
      unsigned rem = kk;
      int buf = 0;
      for (int s = top;; s -= 8, buf = buf == 2 ? 0 : buf + 1) {
        unsigned* h = hist[buf];
        // the next pass's buffer was last read two passes ago, before the
        // previous pass's barrier: clear it now
        if (tid < 256) hist[buf == 2 ? 0 : buf + 1][tid] = 0u;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          if (j < per) {
            const unsigned key = r[j];
            if (key != 0u && (key & mask) == prefix) atomicAdd(&h[(key >> s) & 255u], 1u);
          }
        }
        __syncthreads();
        // every warp: lane l owns bins 255-8l .. 248-8l (two 16-byte
        // loads); the bin where the count from the top reaches rem holds the
        // threshold's digit
        const uint4* hp = reinterpret_cast<const uint4*>(h + 248 - 8 * lane);
        const uint4 u0 = hp[0], u1 = hp[1];
        const unsigned hv[8] = {u1.w, u1.z, u1.y, u1.x, u0.w, u0.z, u0.y, u0.x};
        unsigned own = 0u;
#pragma unroll
        for (int t = 0; t < 8; ++t) own += hv[t];
        const unsigned incl = warp_incl_scan(own, lane);
        const unsigned before = incl - own;
        const bool mine = before < rem && rem <= incl;
        const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        int bin = 0;
        unsigned acc = before, cb = 0u;
        if (mine) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            cb = hv[t];
            bin = 255 - 8 * lane - t;
            if (acc + cb >= rem) break;
            acc += cb;
          }
        }
        bin = __shfl_sync(0xffffffffu, bin, src);
        acc = __shfl_sync(0xffffffffu, acc, src);
        cb = __shfl_sync(0xffffffffu, cb, src);
        rem -= acc;
        prefix |= (unsigned)bin << s;
        mask |= 255u << s;
        // keys >= prefix: the kk_done = kk - rem keys above this bin, plus
        // the bin's cb keys
        const unsigned cand = (kk - rem) + cb;
        if (cand <= kCandStop || (s == 0 && cand <= (unsigned)kMaxK)) {
          low = prefix;
          break;
        }
        if (s == 0) {  // the full key: cb keys equal T, more than fit
          T = prefix;
          need = rem;
          cut_ties = true;
          break;
        }
      }
    }
  }

  // gather the candidates: every key >= low, or (cut_ties) every key > T and
  // the first `need` keys == T in position order
  unsigned tie_rank = 0u;
  if (cut_ties) {  // uniform over the block
    unsigned ties = 0u;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (j < per && r[j] == T) ++ties;
    const unsigned incl = warp_incl_scan(ties, lane);
    if (lane == 31) w_tie[warp] = incl;
    __syncthreads();
    unsigned off = 0u;
    for (int w = 0; w < warp; ++w) off += w_tie[w];
    tie_rank = off + incl - ties;
  }
  // each thread's candidates in position order, placed by a block prefix
  // count (no atomics, so the candidate order is fixed)
  bool tk[kPer];
  unsigned mine = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const unsigned key = r[j];
    bool take = false;
    if (j < per && key != 0u) {
      if (cut_ties) take = key > T || (key == T && tie_rank++ < need);
      else take = key >= low;
    }
    tk[j] = take;
    mine += take ? 1u : 0u;
  }
  const unsigned cincl = warp_incl_scan(mine, lane);
  if (lane == 31) w_cand[warp] = cincl;
  __syncthreads();
  unsigned coff = 0u, ctot = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const unsigned v = w_cand[w];
    coff += w < warp ? v : 0u;
    ctot += v;
  }
  unsigned slot = coff + cincl - mine;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if (tk[j]) {
      if (slot < (unsigned)kMaxK) cand[slot] = ((unsigned long long)r[j] << 32) | (unsigned)~(unsigned)(lo + j);
      ++slot;
    }
  }
  __syncthreads();
  const int m = (int)min(ctot, (unsigned)kMaxK);
  if (tid == 0 && (ctot > (unsigned)kMaxK || ctot < kk)) fdl::raise_error(err, FDL_DEVERR_SHAPE);
  // rank every candidate by (key desc, position asc) among the candidates
  // (which hold every key that can rank above it) and scatter the first kk
  for (int c = tid; c < m; c += kThreads) {
    const unsigned long long v = cand[c];
    const int pos = (int)~(unsigned)v;
    // branch-free count of the candidates above v, two per 16-byte load (an
    // odd count's last pair holds one candidate)
    int rank = 0;
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(cand);
#pragma unroll 4
    for (int o = 0; o < (m + 1) / 2; ++o) {
      const ulonglong2 w = c2[o];
      rank += (int)(w.x > v) + (int)((2 * o + 1 < m) & (w.y > v));
    }
    if (rank < (int)kk) idx_out[(size_t)b * k + rank] = pos;
  }
  for (int t = (int)kk + tid; t < k; t += kThreads) idx_out[(size_t)b * k + t] = -1;
  if (tid == 0) cnt_out[b] = (int)kk;
}

}  // namespace

cudaError_t fdl_launch_topk(fdl_ctx* ctx, const float* scores, const unsigned char* eligible, int ld,
                            const int* seq_len, int B, int k, int* idx_out, int* cnt_out) {
  if (ld <= kStage)
    return fdl_launch_pdl(topk_kernel, dim3(B), dim3(kThreads), 0, ctx->stream, 1, scores, eligible, ld, seq_len, k,
                          idx_out, cnt_out, ctx->err_word);
  return fdl_launch_pdl(topk_large_kernel, dim3(B), dim3(kThreads), 0, ctx->stream, 1, scores, eligible, ld, seq_len,
                        k, idx_out, cnt_out, ctx->err_word);
}
