// Top-k of the attention-mass tracker scores (next step's tracked set).
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...",
// section "Method steps in detail", Algorithm 2 step 4: the k decoded
// tokens with the largest a_i (Eq. (2)) are refreshed next step.
//
// One CTA per sequence. The order-preserving 32-bit images of the eligible
// scores are staged in shared memory once (sequences up to kStage positions;
// longer ones re-read global memory); the k-th largest key is found exactly
// by a 4-pass radix select whose bin search is a warp-parallel scan; ties at
// that threshold are resolved by lowest position with a block prefix count
// in position order; the <= k survivors are ranked by (score desc, position
// asc).
#include "fdl_internal.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kMaxK = 1024;
constexpr int kStage = 8192;

__global__ void __launch_bounds__(kThreads)
topk_kernel(const float* __restrict__ scores, const unsigned char* __restrict__ eligible, int ld,
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

}  // namespace

cudaError_t fdl_launch_topk(fdl_ctx* ctx, const float* scores, const unsigned char* eligible, int ld,
                            const int* seq_len, int B, int k, int* idx_out, int* cnt_out) {
  topk_kernel<<<B, kThreads, 0, ctx->stream>>>(scores, eligible, ld, seq_len, k, idx_out, cnt_out,
                                              ctx->err_word);
  return cudaGetLastError();
}
