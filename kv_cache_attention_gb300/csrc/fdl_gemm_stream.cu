// Weight-streaming GEMM on the 5th-generation tensor cores for the small
// row counts of a cached denoising step (up to 64 rows), in two kernels:
//
//   gemm_stream_kernel  one CTA per SM streams an equal share of the weight
//                       through tcgen05 and writes each of its accumulators
//                       out as an fp32 share of a tile. It merges nothing, so
//                       no CTA waits for another and the launch ends as soon
//                       as the last weight bytes have been multiplied.
//   merge kernels       every output element is the sum of its tile's shares
//                       in CTA order (so results do not depend on timing),
//                       then either
//     merge_dense_kernel  stored as bf16, or added into an fp32 residual
//                         stream (W_o, the SwiGLU gate/up and down
//                         projections of the transformer block), or
//     merge_qkv_kernel    rotated (RoPE) and written as Q and as rows of the
//                         preallocated K/V cache: the fused projection of
//                         paper digest "Flash-dLLM: IO-Aware KV Caching and
//                         Parallel Decoding ...", section "Core method" (the
//                         projection, RoPE and the cache write without a
//                         round trip of K and V through a dense buffer),
//                         "Method steps in detail", step 2 (the rows are the
//                         step's refresh set).
//
// Why. With 64 rows the product is bound by reading the weight once (64
// FLOP per byte, far below the tensor cores' ridge). The weight has only
// N/128 tiles of 128 output features, too few (32 for W_o and the down
// projection, 96 for QKV, 192 for gate/up) to give 152 SMs equal work, so K
// must be split. A split-K kernel that merges in the last CTA of each tile,
// or a stream-K kernel that merges in the last share, puts those merges at
// the end of the launch, after every SM's stream has finished; measured,
// they cost as much as a third of the launch. Here the shares go to an
// L2-resident workspace and the merge is a separate launch with a thread
// for every 8 or 16 output elements.
//
// Schedule (stream-K): the work is T tiles x nkb k-blocks of 64 ("units"),
// in tile-major order; CTA c of G takes the contiguous units [c*U/G,
// (c+1)*U/G), i.e. the tail of one tile, whole tiles, and the head of
// another. Each CTA writes the share of its j-th tile to slot (c, j) of the
// workspace; a tile's shares are those of the CTAs that own its first to
// its last unit.
//
// Orientation ("swap AB"): a tile is 128 output features on the TMEM lanes
// against the 64 rows (zero-filled past R by TMA) on the TMEM columns, which
// fills the M = 128 datapath. Warp roles (192 threads): warp 0 issues TMA
// loads into an 8-stage ring (W box 128 x 64, X box 64 x 64, 128-byte
// swizzle) that runs across tile boundaries, warp 1 owns TMEM and issues
// tcgen05.mma from one lane, warps 2-5 move finished accumulators (four of
// 64 columns) to the workspace while the next ones fill.
#include <cudaTypedefs.h>

#include "fdl_model.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kBM = 128;  // output features per tile
constexpr int kBK = 64;   // k-block: one 128-byte swizzled row of bf16
constexpr int kBN = 64;   // rows per tile (the largest row count served)
constexpr int kThreads = 192;
constexpr int kStages = 8;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kPipeBytes = kStages * kStageBytes;
constexpr int kNacc = 4;                     // TMEM accumulators of kBN columns
constexpr int kTmemCols = kNacc * kBN;
constexpr int kBarBytes = 256;
constexpr int kSmemBytes = 1024 + kPipeBytes + kBarBytes;
constexpr int kMaxSeg = 4;                   // tiles one CTA may touch (workspace slots per CTA)
constexpr size_t kShareFloats = (size_t)kBN * kBM;
constexpr int kMergeThreads = 256;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(8 * (2 * kStages + 2 * kNacc + 1) + 16 <= kBarBytes, "barriers and flags fit");

// (The launcher takes a schedule only while U * G < 2^32, so the unit
// arithmetic below is 32-bit.)
struct Sched {
  unsigned nkb;  // k-blocks per tile
  unsigned T;    // tiles (N / 128)
  unsigned G;    // CTAs
  unsigned U;    // units, T * nkb
};

__host__ __device__ __forceinline__ unsigned unit_begin(const Sched& s, unsigned c) { return s.U * c / s.G; }

// CTA whose range holds unit u (the largest c with unit_begin(c) <= u)
__device__ __forceinline__ unsigned unit_owner(const Sched& s, unsigned u) {
  unsigned c = ((u + 1) * s.G - 1) / s.U;
  c = min(c, s.G - 1);
  while (c + 1 < s.G && unit_begin(s, c + 1) <= u) ++c;
  while (c > 0 && unit_begin(s, c) > u) --c;
  return c;
}

// Segment j of CTA c: tile t and its k-blocks [kb_a, kb_b); false past the
// CTA's last segment.
__device__ __forceinline__ bool segment(const Sched& s, int c, int j, int& t, int& kb_a, int& kb_b) {
  const unsigned a = unit_begin(s, c), b = unit_begin(s, c + 1);
  const unsigned ts = a / s.nkb + j;
  if (j >= kMaxSeg || ts * s.nkb >= b) return false;
  kb_a = (int)(max(a, ts * s.nkb) - ts * s.nkb);
  kb_b = (int)(min(b, (ts + 1) * s.nkb) - ts * s.nkb);
  t = (int)ts;
  return true;
}

struct StreamParams {
  Sched s;
  int R;
  float* partials;        // [G][kMaxSeg][kBN][128] fp32 shares
  unsigned* err;
  long long wait_budget;  // cycles of the main loop's mbarrier waits
};

__global__ void __launch_bounds__(kThreads, 1)
    gemm_stream_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                       const StreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pipe = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPipeBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;  // [kNacc]
  uint64_t* acc_empty = acc_full + kNacc;   // [kNacc]
  uint64_t* mma_done = acc_empty + kNacc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  // Barriers, TMEM and the tensor-map prefetch touch no global memory, so
  // they overlap the end of the previous kernel in the stream.
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kNacc; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);  // one arrival per epilogue warp
    }
    tc::mbar_init(mma_done, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w);
    tc::prefetch_tensormap(&tmap_x);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }

  // The producer walks (segment, k-block) in order. The weight is never
  // written by a kernel of the stream, so the weight halves of the first
  // ring of stages are loaded before the programmatic-launch wait: the
  // stream starts while the previous kernel (typically the merge of the
  // previous product) is still running. The row halves (X, the previous
  // kernel's output) follow after the wait. (With a shortened wait budget,
  // for failure-path tests, the ring is filled only after the CTA barrier,
  // so that no load lands before the first wait.)
  int pj = 0, pt = 0, pkb = 0, pkb_b = 0, pit = 0;
  bool pvalid = false;
  int n_pre = 0;
  // the weight is read once: evict it from L2 first, so that it does not push
  // out the shares the merge reads back, nor the rows every CTA re-reads
  uint64_t pol_w = 0, pol_x = 0;
  if (threadIdx.x == 0) {
    pol_w = tc::l2_policy_evict_first();
    pol_x = tc::l2_policy_evict_last();
  }
  auto advance = [&]() {
    ++pit;
    if (++pkb >= pkb_b) pvalid = segment(p.s, cta, ++pj, pt, pkb, pkb_b);
  };
  auto issue = [&]() {
    const int s = pit % kStages;
    uint8_t* a = pipe + s * kStageBytes;
    tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
    tc::tma_load_2d_hint(a, &tmap_w, pkb * kBK, pt * kBM, &full[s], pol_w);
    tc::tma_load_2d_hint(a + kABytes, &tmap_x, pkb * kBK, 0, &full[s], pol_x);
    advance();
  };
  if (threadIdx.x == 0) {
    pvalid = segment(p.s, cta, 0, pt, pkb, pkb_b);
    if (p.wait_budget == tc::kWaitBudgetCycles) {
      while (pvalid && n_pre < kStages) {
        uint8_t* a = pipe + pit * kStageBytes;
        tc::mbar_arrive_expect_tx(&full[pit], kStageBytes);
        tc::tma_load_2d_hint(a, &tmap_w, pkb * kBK, pt * kBM, &full[pit], pol_w);
        ++n_pre;
        advance();
      }
    }
  }
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  if (threadIdx.x == 0 && n_pre > 0) {
    // the same walk again for the k-blocks of the pre-issued stages
    int wj = 0, wt = 0, wkb = 0, wkb_b = 0;
    segment(p.s, cta, 0, wt, wkb, wkb_b);
    for (int s = 0; s < n_pre; ++s) {
      tc::tma_load_2d_hint(pipe + s * kStageBytes + kABytes, &tmap_x, wkb * kBK, 0, &full[s], pol_x);
      if (++wkb >= wkb_b) segment(p.s, cta, ++wj, wt, wkb, wkb_b);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      while (pvalid) {
        const int s = pit % kStages;
        if (pit >= kStages &&
            !tc::mbar_wait(&empty[s], ((uint32_t)(pit / kStages) & 1u) ^ 1u, abort_flag, p.wait_budget))
          break;
        issue();
      }
      if (*abort_flag) {
        // let loads already in flight land before this CTA's memory is reused
        for (int j = max(0, pit - kStages); j < pit; ++j) {
          long long t0 = clock64();
          while (!tc::mbar_try_wait(&full[j % kStages], (uint32_t)(j / kStages) & 1u) &&
                 clock64() - t0 < tc::kWaitBudgetCycles / 8) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
      int it = 0, t = 0, kb_a = 0, kb_b = 0;
      bool ok = true;
      for (int j = 0; ok && segment(p.s, cta, j, t, kb_a, kb_b); ++j) {
        const int a = j % kNacc;
        // the epilogue has moved segment j - kNacc out of this accumulator
        if (j >= kNacc && !tc::mbar_wait(&acc_empty[a], (uint32_t)((j - kNacc) / kNacc) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(a * kBN);
        for (int kb = kb_a; kb < kb_b; ++kb, ++it) {
          const int s = it % kStages;
          if (!tc::mbar_wait(&full[s], (uint32_t)(it / kStages) & 1u, abort_flag, p.wait_budget)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_addr(pipe + s * kStageBytes);
          const uint64_t ad = tc::desc_kmajor_sw128(sa);
          const uint64_t bd = tc::desc_kmajor_sw128(sa + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16_ss(d, ad + 2 * k, bd + 2 * k, idesc, (kb > kb_a || k > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        if (ok) tc::mma_commit(&acc_full[a]);
      }
      // every product issued has finished before the CTA barrier below, also
      // when a wait gave up (the TMEM is freed after that barrier)
      tc::mma_commit(mma_done);
      long long t0 = clock64();
      while (!tc::mbar_try_wait(mma_done, 0) && clock64() - t0 < tc::kWaitBudgetCycles) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;        // TMEM lane quadrant of this warp
    const int ft = q * 32 + lane;  // tile row = output feature
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    const int rows = min(p.R, kBN);
    int t = 0, kb_a = 0, kb_b = 0;
    for (int j = 0; segment(p.s, cta, j, t, kb_a, kb_b); ++j) {
      const int a = j % kNacc;
      if (!tc::mbar_wait(&acc_full[a], (uint32_t)(j / kNacc) & 1u, abort_flag)) break;
      tc::fence_after_sync();
      // rows of 128 features, so a warp's stores of one row are 128
      // contiguous bytes
      float* dst = p.partials + ((size_t)cta * kMaxSeg + j) * kShareFloats + ft;
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 16) {
        float v[16];
        tc::tmem_ld_32x32b_x16(t_lane + (uint32_t)(a * kBN + c0), v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c0 + i < rows) dst[(size_t)(c0 + i) * kBM] = v[i];
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) fdl::raise_error(p.err, FDL_DEVERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// The merge kernels: one CTA per (tile, block of rows). The CTA first lists
// its tile's shares (their workspace offsets, in CTA order) in shared
// memory; then every thread sums the shares of its 8 or 16 features of one
// row with all of its loads in flight together.
constexpr int kMaxShares = 256;  // a tile's shares: at most one per CTA of the GEMM

struct ShareList {
  unsigned off[kMaxShares];  // float offset of each share's tile in the workspace
  int n;
};

// Fills `sl` for tile t (threads of warp 0; the caller synchronises).
__device__ __forceinline__ void list_shares(const Sched& s, unsigned t, ShareList& sl) {
  const unsigned ca = unit_owner(s, t * s.nkb), cb = unit_owner(s, (t + 1) * s.nkb - 1);
  for (unsigned c = ca + threadIdx.x; c <= cb; c += 32) {
    const unsigned j = t - unit_begin(s, c) / s.nkb;
    sl.off[c - ca] = (c * kMaxSeg + j) * (unsigned)kShareFloats;
  }
  if (threadIdx.x == 0) sl.n = (int)(cb - ca + 1);
}

// Sum over the listed shares of the 8 floats at `off` of each share, in
// list order.
__device__ __forceinline__ void sum8(const float* partials, const ShareList& sl, unsigned off, float (&acc)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const int n = sl.n;
  int k = 0;
  for (; k + 4 <= n; k += 4) {
    float4 x[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4* src = reinterpret_cast<const float4*>(partials + sl.off[k + u] + off);
      x[2 * u] = __ldcg(src);
      x[2 * u + 1] = __ldcg(src + 1);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc[0] += x[2 * u].x, acc[1] += x[2 * u].y, acc[2] += x[2 * u].z, acc[3] += x[2 * u].w;
      acc[4] += x[2 * u + 1].x, acc[5] += x[2 * u + 1].y, acc[6] += x[2 * u + 1].z, acc[7] += x[2 * u + 1].w;
    }
  }
  for (; k < n; ++k) {
    const float4* src = reinterpret_cast<const float4*>(partials + sl.off[k] + off);
    const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
    acc[0] += x0.x, acc[1] += x0.y, acc[2] += x0.z, acc[3] += x0.w;
    acc[4] += x1.x, acc[5] += x1.y, acc[6] += x1.z, acc[7] += x1.w;
  }
}

__device__ __forceinline__ int4 pack_bf16x8(const float (&v)[8]) {
  int4 o;
  __nv_bfloat162 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  o.x = *reinterpret_cast<int*>(&h[0]);
  o.y = *reinterpret_cast<int*>(&h[1]);
  o.z = *reinterpret_cast<int*>(&h[2]);
  o.w = *reinterpret_cast<int*>(&h[3]);
  return o;
}

struct MergeDenseParams {
  Sched s;
  int R, N;
  const float* partials;
  void* out;     // [R, N]: fp32 (add) or bf16 (store)
  bool add_f32;
};

constexpr int kDenseRows = kMergeThreads / (kBM / 8);  // rows per dense-merge CTA (16)

// Grid (row blocks, tiles): thread = (row, 8 consecutive features of the tile).
__global__ void __launch_bounds__(kMergeThreads) merge_dense_kernel(const MergeDenseParams p) {
  __shared__ ShareList sl;
  const unsigned t = blockIdx.y;
  if (threadIdx.x < 32) list_shares(p.s, t, sl);
  __syncthreads();
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int r = blockIdx.x * kDenseRows + (int)(threadIdx.x >> 4);
  const int fl = (int)(threadIdx.x & 15) * 8;
  if (r >= p.R) return;
  float acc[8];
  sum8(p.partials, sl, (unsigned)r * kBM + fl, acc);
  const size_t o = (size_t)r * p.N + t * kBM + fl;
  if (p.add_f32) {
    float4* h = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o);
    float4 h0 = h[0], h1 = h[1];
    h0.x += acc[0], h0.y += acc[1], h0.z += acc[2], h0.w += acc[3];
    h1.x += acc[4], h1.y += acc[5], h1.z += acc[6], h1.w += acc[7];
    h[0] = h0;
    h[1] = h1;
  } else {
    *reinterpret_cast<int4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o) = pack_bf16x8(acc);
  }
}

struct MergeQkvParams {
  Sched s;
  int R, d, hd;
  const float* partials;
  const int* row_seq;
  const int* row_rope_pos;
  const int* row_cache_pos;
  const int* block_table;
  int bt_stride, page_size, n_pages;
  __nv_bfloat16* q_out;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  const float* rope_cos;  // [rope_positions][hd / 2]
  const float* rope_sin;
  int rope_positions;
  unsigned* err;
};

constexpr int kQkvRows = kMergeThreads / (kBM / 16);  // rows per projection-merge CTA (32)

// Grid (row blocks, tiles); a tile holds whole heads (hd 64 or 128) of one
// section (Q, K or V). Thread = (row, 16 features of the tile): for Q and K
// the features i..i+7 and i+hd/2..i+hd/2+7 of one head (a RoPE pair each),
// for V 16 consecutive features. A row with an invalid RoPE position raises
// the index error and writes nothing; a row with a negative cache position
// writes Q only. The loads that do not depend on one another (the shares,
// the row's position, cache position and sequence) are issued together;
// the RoPE table and block table follow them.
__global__ void __launch_bounds__(kMergeThreads) merge_qkv_kernel(const MergeQkvParams p) {
  __shared__ ShareList sl;
  const unsigned t = blockIdx.y;
  const int f0 = (int)t * kBM, sec = f0 / p.d;
  if (threadIdx.x < 32) list_shares(p.s, t, sl);
  __syncthreads();
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int i = (int)(threadIdx.x >> 3), g = (int)(threadIdx.x & 7);
  const int r = blockIdx.x * kQkvRows + i;
  if (r >= p.R) return;
  const int half = p.hd / 2, gph = half / 8;  // 8-feature groups per half head
  int fl_lo, fl_hi, i0 = 0;
  if (sec < 2) {
    const int h = g / gph;
    i0 = (g - h * gph) * 8;
    fl_lo = h * p.hd + i0;
    fl_hi = fl_lo + half;
  } else {
    fl_lo = g * 16;
    fl_hi = fl_lo + 8;
  }
  const int pos = p.row_rope_pos[r];
  const int cp = sec > 0 ? p.row_cache_pos[r] : 0;
  const int b = sec > 0 ? p.row_seq[r] : 0;
  float lo[8], hi[8];
  sum8(p.partials, sl, (unsigned)r * kBM + fl_lo, lo);
  sum8(p.partials, sl, (unsigned)r * kBM + fl_hi, hi);
  if (pos < 0 || pos >= p.rope_positions) {
    if (g == 0) fdl::raise_error(p.err, FDL_DEVERR_INDEX);
    return;
  }
  long long dst = (long long)r * p.d;
  if (sec > 0) {
    if (cp < 0) return;
    const long long slot = fdl::cache_slot(p.block_table, p.bt_stride, p.page_size, p.n_pages, b, cp, p.err);
    if (slot < 0) return;
    dst = slot * p.d;
  }
  if (sec < 2) {
    const float4* cs4 = reinterpret_cast<const float4*>(p.rope_cos + (size_t)pos * half + i0);
    const float4* sn4 = reinterpret_cast<const float4*>(p.rope_sin + (size_t)pos * half + i0);
    const float4 c0 = __ldg(cs4), c1 = __ldg(cs4 + 1), s0 = __ldg(sn4), s1 = __ldg(sn4 + 1);
    const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float x = lo[k], y = hi[k];
      lo[k] = x * cs[k] - y * sn[k];
      hi[k] = x * sn[k] + y * cs[k];
    }
  }
  __nv_bfloat16* out = sec == 0 ? p.q_out : (sec == 1 ? p.k_cache : p.v_cache);
  const int fo = f0 - sec * p.d;  // the tile's first feature within its section
  *reinterpret_cast<int4*>(out + dst + fo + fl_lo) = pack_bf16x8(lo);
  *reinterpret_cast<int4*>(out + dst + fo + fl_hi) = pack_bf16x8(hi);
}

// ------------------------------------------------------------ consumers
// A kernel that merges the shares while consuming the product (the SwiGLU
// product of the gate/up projection), so that the product needs no launch
// of its own for the merge. (Folding the W_o and down merges into the
// residual add + RMSNorm, one CTA per row, was measured slower than the
// separate merge with a CTA per tile and row block.) CTA c's share of
// tile t gets index c + t in a flat table (CTA ranges are ordered like the
// tiles, so no two (c, t) pairs collide), filled from the schedule alone
// before the programmatic-launch wait.
constexpr int kMaxTable = 1024;  // G + T - 1 entries at most
constexpr int kRowThreads = 256;

__device__ __forceinline__ void fill_table(const Sched& s, unsigned* tab) {
  for (unsigned c = threadIdx.x; c < s.G; c += blockDim.x) {
    int t = 0, kb_a = 0, kb_b = 0;
    for (int j = 0; segment(s, (int)c, j, t, kb_a, kb_b); ++j) tab[c + t] = (c * kMaxSeg + j) * (unsigned)kShareFloats;
  }
}

// Merged product at (row r, features f..f+7), f a multiple of 8.
__device__ __forceinline__ void merged8(const Sched& s, const float* partials, const unsigned* tab, int r, int f,
                                        float (&acc)[8]) {
  const unsigned t = (unsigned)f / kBM;
  const unsigned ca = unit_owner(s, t * s.nkb), cb = unit_owner(s, (t + 1) * s.nkb - 1);
  const unsigned off = (unsigned)r * kBM + ((unsigned)f & (kBM - 1));
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (unsigned c = ca; c <= cb; ++c) {
    const float4* src = reinterpret_cast<const float4*>(partials + tab[c + t] + off);
    const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
    acc[0] += x0.x, acc[1] += x0.y, acc[2] += x0.z, acc[3] += x0.w;
    acc[4] += x1.x, acc[5] += x1.y, acc[6] += x1.z, acc[7] += x1.w;
  }
}

// Grid (rows, chunks of kRowThreads 8-feature groups): gate and up each
// rounded to bf16 as the stored product would be, then the SwiGLU product.
__global__ void __launch_bounds__(kRowThreads) swiglu_shares_kernel(const Sched s, const float* partials, int F,
                                                                    __nv_bfloat16* __restrict__ u) {
  __shared__ unsigned tab[kMaxTable];
  fill_table(s, tab);
  __syncthreads();
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int r = blockIdx.x;
  const int f = (blockIdx.y * kRowThreads + (int)threadIdx.x) * 8;
  if (f >= F) return;
  float a[8], b[8];
  merged8(s, partials, tab, r, f, a);
  merged8(s, partials, tab, r, F + f, b);
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float ga = __bfloat162float(__float2bfloat16_rn(a[i]));
    const float ub = __bfloat162float(__float2bfloat16_rn(b[i]));
    y[i] = ga / (1.f + expf(-ga)) * ub;
  }
  *reinterpret_cast<int4*>(u + (size_t)r * F + f) = pack_bf16x8(y);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 2-D bf16 row-major [rows, cols] map, box = 64 columns x box_rows rows,
// 128-byte swizzle (the layout desc_kmajor_sw128 describes).
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The schedule, or false when it does not fit: 32-bit unit arithmetic
// (U * G < 2^32), at most kMaxSeg tiles per CTA (a range of L units
// starting anywhere in a tile covers at most floor((L + nkb - 2) / nkb) + 1
// tiles), at most kMaxShares CTAs, and kMaxSeg workspace shares per CTA.
bool make_sched(const fdl_ctx* ctx, int K, int N, Sched& s) {
  if (K <= 0 || N <= 0 || K % kBK != 0 || N % kBM != 0) return false;
  const unsigned long long U = (unsigned long long)(K / kBK) * (unsigned long long)(N / kBM);
  const unsigned long long G = U < (unsigned long long)ctx->num_sms ? U : (unsigned long long)ctx->num_sms;
  if (G == 0 || G > (unsigned long long)kMaxShares || U * G >= (1ull << 32)) return false;
  s.nkb = (unsigned)(K / kBK);
  s.T = (unsigned)(N / kBM);
  s.U = (unsigned)U;
  s.G = (unsigned)G;
  const unsigned long long L = (U + G - 1) / G;
  const unsigned long long tiles = (L + s.nkb - 2) / s.nkb + 1;
  return tiles <= (unsigned long long)kMaxSeg && (size_t)G * kMaxSeg * kShareFloats <= ctx->qkv_partial_floats;
}

cudaError_t launch_stream(fdl_ctx* ctx, const Sched& s, int R, const void* X, const void* W, int K, int N) {
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)gemm_stream_kernel, ctx->device, kSmemBytes)) return e;
  CUtensorMap mw, mx;
  if (!make_map(&mw, W, (uint64_t)N, (uint64_t)K, kBM) || !make_map(&mx, X, (uint64_t)R, (uint64_t)K, kBN))
    return cudaErrorInvalidValue;
  StreamParams p;
  p.s = s;
  p.R = R;
  p.partials = ctx->qkv_partials;
  p.err = ctx->err_word;
  p.wait_budget = ctx->wait_budget > 0 ? ctx->wait_budget : tc::kWaitBudgetCycles;
  return fdl_launch_pdl(gemm_stream_kernel, dim3((unsigned)s.G), dim3(kThreads, 1, 1), kSmemBytes, ctx->stream, 1,
                        mw, mx, p);
}

}  // namespace

bool fdl_stream_gemm_applies(const fdl_ctx* ctx, int R, int K, int N) {
  Sched s;
  return R > 0 && R <= kBN && ctx->qkv_partials && make_sched(ctx, K, N, s);
}

cudaError_t fdl_launch_dense_stream(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N, void* out,
                                    bool add_f32) {
  Sched s;
  if (!fdl_stream_gemm_applies(ctx, R, K, N) || !make_sched(ctx, K, N, s)) return cudaErrorNotSupported;
  if (cudaError_t e = launch_stream(ctx, s, R, X, W, K, N)) return e;
  MergeDenseParams m;
  m.s = s;
  m.R = R;
  m.N = N;
  m.partials = ctx->qkv_partials;
  m.out = out;
  m.add_f32 = add_f32;
  return fdl_launch_pdl(merge_dense_kernel, dim3((unsigned)((R + kDenseRows - 1) / kDenseRows), s.T),
                        dim3(kMergeThreads, 1, 1), 0, ctx->stream, 1, m);
}

cudaError_t fdl_launch_qkv_stream(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                                  const int* row_rope_pos, const int* row_cache_pos, const int* block_table,
                                  int bt_stride, void* k_cache, void* v_cache, void* q_out) {
  const fdl_config& c = ctx->cfg;
  const int d = c.d_model;
  Sched s;
  if ((c.head_dim != 64 && c.head_dim != 128) || d % kBM != 0 || !fdl_stream_gemm_applies(ctx, R, d, 3 * d) ||
      !make_sched(ctx, d, 3 * d, s))
    return cudaErrorNotSupported;
  if (cudaError_t e = launch_stream(ctx, s, R, X, W, d, 3 * d)) return e;
  MergeQkvParams m;
  m.s = s;
  m.R = R;
  m.d = d;
  m.hd = c.head_dim;
  m.partials = ctx->qkv_partials;
  m.row_seq = row_seq;
  m.row_rope_pos = row_rope_pos;
  m.row_cache_pos = row_cache_pos;
  m.block_table = block_table;
  m.bt_stride = bt_stride;
  m.page_size = c.page_size;
  m.n_pages = c.n_pages;
  m.q_out = reinterpret_cast<__nv_bfloat16*>(q_out);
  m.k_cache = reinterpret_cast<__nv_bfloat16*>(k_cache);
  m.v_cache = reinterpret_cast<__nv_bfloat16*>(v_cache);
  m.rope_cos = ctx->rope_cos;
  m.rope_sin = ctx->rope_sin;
  m.rope_positions = ctx->rope_positions;
  m.err = ctx->err_word;
  return fdl_launch_pdl(merge_qkv_kernel, dim3((unsigned)((R + kQkvRows - 1) / kQkvRows), s.T),
                        dim3(kMergeThreads, 1, 1), 0, ctx->stream, 1, m);
}

bool fdl_stream_swiglu_applies(const fdl_ctx* ctx, int R, int d, int F) {
  Sched s;
  return F % 8 == 0 && fdl_stream_gemm_applies(ctx, R, d, 2 * F) && make_sched(ctx, d, 2 * F, s) &&
         s.G + s.T - 1 <= (unsigned)kMaxTable;
}

cudaError_t fdl_launch_dense_stream_shares(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N,
                                           fdl_stream_shares* out) {
  Sched s;
  if (!fdl_stream_gemm_applies(ctx, R, K, N) || !make_sched(ctx, K, N, s) || s.G + s.T - 1 > (unsigned)kMaxTable)
    return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W)) & 15) return cudaErrorMisalignedAddress;
  out->nkb = s.nkb;
  out->T = s.T;
  out->G = s.G;
  out->U = s.U;
  out->partials = ctx->qkv_partials;
  return launch_stream(ctx, s, R, X, W, K, N);
}

cudaError_t fdl_launch_swiglu_shares(fdl_ctx* ctx, const fdl_stream_shares& sh, int R, int F, void* u) {
  if (R <= 0) return cudaSuccess;
  if (sh.T * kBM != 2u * (unsigned)F || (reinterpret_cast<uintptr_t>(u) & 15)) return cudaErrorInvalidValue;
  const Sched s{sh.nkb, sh.T, sh.G, sh.U};
  const int chunks = (F / 8 + kRowThreads - 1) / kRowThreads;
  return fdl_launch_pdl(swiglu_shares_kernel, dim3(R, chunks), dim3(kRowThreads), 0, ctx->stream, 1, s, sh.partials,
                        F, reinterpret_cast<__nv_bfloat16*>(u));
}
