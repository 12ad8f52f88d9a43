// Block-table scheduled attention on the 5th-generation tensor cores, with the
// Flash-Verify two-view mask and the Eq. (2) attention-mass tracker fused in.
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...":
//   "Background"  exact softmax(QK^T/sqrt(d))V computed tile by tile, the
//                 score matrix never written to HBM;
//   "Core method" block-table scheduling of ragged per-sequence query blocks
//                 against their cached K/V; verify rows see the shared tracked
//                 context but not each other's view of the same token;
//   "Method steps in detail", step 4, Eq. (2): masked-window rows' attention
//                 probabilities, averaged over heads and rows, summed over
//                 layers.
//
// One CTA = (work item of <= 128 query rows of one sequence, head, KV split).
// The KV splits of an item form a thread-block cluster of C CTAs (C = 1 when
// items x heads already fill the GPU).
//
// Scores S = Q K^T and the products O += P V run on tcgen05 with fp32
// accumulators in TMEM. Eight softmax warps form two groups; group g takes
// the key tiles i with i % 2 == g and owns a P tile in shared memory and an O
// accumulator O_g in TMEM, so one group's softmax overlaps the other's
// products. An item takes one of two modes:
//   online    (C = 1, no masked-window row feeds the tracker) one pass: P =
//             exp(S - m) against a running row max m that moves only when a
//             tile's max exceeds it by more than 2^kRescale; O_g and the row
//             sum are then scaled to the new m in TMEM. At the end O =
//             (O_0 w_0 + O_1 w_1) / l with the two groups' weights w_g.
//   two-pass  (split items, and items whose WINDOW rows feed Eq. (2))
//             pass A gives each row's exact log-sum-exp (the C splits' (max,
//             sum) pairs meet through distributed shared memory); pass B
//             forms the final probabilities P = exp(S - lse), whose column
//             sums over WINDOW rows are the tracker's contribution, and O =
//             O_0 + O_1. K is read twice, the second time mostly from L2.
// The C partial O tiles are summed through distributed shared memory in rank
// order, so results do not depend on timing.
//
// Warp roles (352 threads): warp 0 TMA producer of Q and of a 4-stage K
// ring (a stage is released as soon as its S product finishes), warp 10 TMA
// producer of a 4-stage V ring, warp 1 TMEM owner and MMA issuer (one lane,
// issuing whichever of the next P V or the next S is ready, from four S
// buffers), warps 2-9 softmax and epilogue: one query row per thread (TMEM
// lane quadrant = warp % 4). The cache slot of every key tile of the CTA is
// looked up once, before the main loops, into shared memory.
#include <cudaTypedefs.h>
#include <math.h>

#include "fdl_internal.cuh"
#include "fdl_attn_tc.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kBM = 128;    // query rows per item
constexpr int kBN = 64;     // keys per tile
constexpr int kHD = 128;    // head dim handled here
constexpr int kThreads = 352;
constexpr int kVWarp = 10;  // V producer
constexpr int kKS = 4;      // K ring stages
constexpr int kVS = 4;      // V ring stages
constexpr int kSB = 4;      // S buffers in TMEM (64 columns each)
constexpr int kTmemCols = 512;  // O_0, O_1 (128 columns each) + kSB S buffers
constexpr float kRescale = 8.f;  // online mode: log2 headroom of P before the row max moves
constexpr int kMaxC = 8;
constexpr int kMaxTiles = 384;  // key tiles of one item: (max_seq + max_views) / 64

constexpr int Q_BYTES = kBM * kHD * 2;          // two 64-column halves of 16 KB
constexpr int KT_BYTES = kBN * kHD * 2;         // K tile: two halves of 8 KB
constexpr int VT_BYTES = kBN * kHD * 2;         // V tile: two halves of 8 KB
constexpr int P_BYTES = kBM * kBN * 2;          // bf16 P tile, 128 B rows (two alternate)
constexpr int ML_BYTES = kMaxC * kBM * 2 * 4;   // (max, sum) from every split

constexpr int OFF_Q = 0;
constexpr int OFF_KRING = OFF_Q + Q_BYTES;
constexpr int OFF_VRING = OFF_KRING + kKS * KT_BYTES;  // directly after the K ring
constexpr int OFF_P = OFF_VRING + kVS * VT_BYTES;
constexpr int OFF_ML = OFF_P + 2 * P_BYTES;
constexpr int OFF_MISC = OFF_ML + ML_BYTES;
// misc: barriers [0, 256), row kinds, the two groups' tracker column sums,
// the search bitmap (<= 768 words), the two groups' (max, sum) per row,
// flags, key-tile slots
constexpr int OFF_KINDS = 256;                      // int [128]
constexpr int OFF_COLACC = OFF_KINDS + 4 * kBM;     // float [2 groups][4 warps][64]
constexpr int OFF_BITMAP = OFF_COLACC + 2 * 4 * 64 * 4;  // uint32 [768]
constexpr int OFF_HALFML = OFF_BITMAP + 768 * 4;    // float [2][128][2]
constexpr int OFF_FLAGS = OFF_HALFML + 2 * kBM * 2 * 4;
constexpr int OFF_SLOTS = OFF_FLAGS + 256;          // int [kMaxTiles]
constexpr int OFF_ITEM = OFF_SLOTS + 4 * kMaxTiles;  // int [8]: item count, b, q0, qlen, n_keys, WINDOW rows of b
constexpr int kMaxDecodeB = 1024;                   // batch whose cu_seqlens_q the kernel stages
constexpr int OFF_CU = OFF_ITEM + 32;               // int [kMaxDecodeB + 1]
constexpr int OFF_WBITS = OFF_CU + 4 * (kMaxDecodeB + 1);  // uint32 [kTrkWords]: the sequence's WINDOW tiles, then 2 flags
constexpr int MISC_BYTES = OFF_WBITS + 4 * (kTrkWords + 2);
static_assert(8 * (1 + 2 * kKS + 2 * kVS + 2 * kSB + 5) + 8 <= OFF_KINDS, "barriers fit");
static_assert(256 + 64 * kSB <= kTmemCols, "TMEM columns");
constexpr int SMEM_BYTES = 1024 + OFF_MISC + MISC_BYTES;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(kKS * KT_BYTES + kVS * VT_BYTES >= kBM * (kHD + 4) * 4,
              "the two rings must hold an fp32 O tile for the cluster sum");

constexpr float kLn2 = 0.6931471805599453f;

struct TcAttnParams {
  const int* wl;            // count, then (b, q_start, q_len, n_keys); null: decode from cu
  const int* cu;            // cu_seqlens_q [B + 1] (decode mode)
  const int* n_search;      // [B] or null (decode mode)
  int B, max_seq, max_search_tokens;
  int* wl_out;              // decode mode: optional copy of the work list the kernel used
  const int* kv_len;
  const int* row_kind;
  const int* search_pos;
  int search_ld;
  const int* block_table;
  int bt_stride, page_size, n_pages, n_slots;
  const int* n_masked;
  __nv_bfloat16* o;
  float* lse;
  float* track;
  int track_ld;
  float* trk_part;          // deterministic tracker partials (null: atomics into track)
  int* trk_nslots;          // [B] slots of each sequence's partials (0: none, atomics)
  int trk_ld;
  int H, d, R;
  int C;                    // splits per item (cluster size)
  float scale_log2;         // log2(e) / sqrt(head_dim)
  int bitmap_words;         // search-position bitmap size
  unsigned* err;
};

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(tc::smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > tc::kWaitBudgetCycles) {
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
  const uint32_t a = tc::map_cluster(tc::smem_addr(bar), rank);
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a) : "memory");
}

__device__ __forceinline__ void st_cluster_v2(uint32_t caddr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(caddr), "f"(a), "f"(b) : "memory");
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Split `rank` of a C-CTA cluster sums its share of the item's qlen valid
// rows, [rank * qlen / C, (rank + 1) * qlen / C), over the C staged fp32 O
// tiles in rank order and stores them as bf16; each thread keeps the remote
// loads of two float4 columns (from every split) in flight together.
template <int CC>
__device__ __forceinline__ void merge_o(const TcAttnParams& p, uint32_t base, uint32_t rank, int t_local, int q0,
                                        int qlen, int h, bool aborted) {
  constexpr int kOStride = kHD + 4;
  constexpr int kVec = kHD / 4;  // float4 columns per row
  const int r0 = (int)rank * qlen / CC, r1 = ((int)rank + 1) * qlen / CC;
  const int n = (r1 - r0) * kVec;
  for (int e0 = t_local; e0 < n; e0 += 2 * 256) {
    float4 v[2][CC];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + 256 * u;
      if (e < n) {
        const int r = r0 + e / kVec, col = (e % kVec) * 4;
#pragma unroll
        for (int src = 0; src < CC; ++src)
          v[u][src] = ld_cluster_v4(tc::map_cluster(base + (uint32_t)(r * kOStride + col) * 4u, (uint32_t)src));
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + 256 * u;
      if (e >= n || aborted) continue;
      const int r = r0 + e / kVec, col = (e % kVec) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int src = 0; src < CC; ++src) {
        acc.x += v[u][src].x;
        acc.y += v[u][src].y;
        acc.z += v[u][src].z;
        acc.w += v[u][src].w;
      }
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 w = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      *reinterpret_cast<uint2*>(p.o + (size_t)(q0 + r) * p.d + h * kHD + col) = w;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const TcAttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem + OFF_Q;
  uint8_t* kring = smem + OFF_KRING;
  uint8_t* vring = smem + OFF_VRING;
  uint8_t* sp = smem + OFF_P;
  float* ml = reinterpret_cast<float*>(smem + OFF_ML);  // [C][128][2]
  uint8_t* misc = smem + OFF_MISC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;                   // [kKS]
  uint64_t* k_empty = k_full + kKS;              // [kKS]
  uint64_t* v_full = k_empty + kKS;              // [kVS]
  uint64_t* v_empty = v_full + kVS;              // [kVS]
  uint64_t* s_full = v_empty + kVS;              // [kSB]
  uint64_t* s_free = s_full + kSB;               // [kSB]
  uint64_t* p_full = s_free + kSB;               // [2], one per softmax group (P tile)
  uint64_t* pv_done = p_full + 2;                // [2], one per softmax group (P tile, O accumulator)
  uint64_t* ml_ready = pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ml_ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* kinds = reinterpret_cast<int*>(misc + OFF_KINDS);            // [128]
  float* colacc = reinterpret_cast<float*>(misc + OFF_COLACC);      // [2][4][64]
  uint32_t* wbits = reinterpret_cast<uint32_t*>(misc + OFF_WBITS);   // [kTrkWords], [kTrkWords]: overflow, +1: last
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(misc + OFF_BITMAP);  // [bitmap_words] (<= 768)
  float* halfml = reinterpret_cast<float*>(misc + OFF_HALFML);      // [2][128][2]
  // per row-staging warp: its 32 rows hold a WINDOW row (written by that
  // warp alone, so nothing has to clear it first)
  int* win_flags = reinterpret_cast<int*>(misc + OFF_FLAGS);  // [4]
  int* slots = reinterpret_cast<int*>(misc + OFF_SLOTS);            // [n_my] cache slot of each key tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = p.C;
  const uint32_t rank = C > 1 ? tc::cluster_ctarank() : 0u;
  const int item = blockIdx.z;
  const int h = blockIdx.y;
  const bool softmax_warp = warp >= 2 && warp < 10;
  const int t_local = threadIdx.x - 64;  // 0..255 over the softmax warps

  // ---------------------------------------------------------------- setup
  // Barriers, TMEM and the tensor-map prefetch touch no global memory, so
  // they overlap the end of the previous kernel in the stream; the work list,
  // Q and the cache are read only after the dependency wait.
  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < kKS; ++s) {
      tc::mbar_init(&k_full[s], 1);
      tc::mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVS; ++s) {
      tc::mbar_init(&v_full[s], 1);
      tc::mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < kSB; ++s) {
      tc::mbar_init(&s_full[s], 1);
      tc::mbar_init(&s_free[s], 4);  // the four warps of the group that reads it
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&p_full[s], 4);
      tc::mbar_init(&pv_done[s], 1);
    }
    tc::mbar_init(ml_ready, 4 * C);  // the four group-0 warps of every split
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tm_q);
    tc::prefetch_tensormap(&tm_k);
    tc::prefetch_tensormap(&tm_v);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  int* s_item = reinterpret_cast<int*>(misc + OFF_ITEM);
  if (!p.wl) {
    // The work item from cu_seqlens_q: sequence b contributes ceil(rows_b /
    // 128) items in order, item z of the grid is found by a prefix sum over
    // the staged offsets. Inconsistent offsets (cu[0] != 0, cu[B] != R, a
    // negative row count) leave no items and set the shape error.
    int* s_cu = reinterpret_cast<int*>(misc + OFF_CU);
    for (int i = threadIdx.x; i <= p.B; i += kThreads) s_cu[i] = p.cu[i];
    if (threadIdx.x == 0) s_item[5] = 0;
    if (threadIdx.x < kTrkWords + 1) wbits[threadIdx.x] = 0u;
    __syncthreads();
    if (warp == 0) {
      bool bad = s_cu[0] != 0 || s_cu[p.B] != p.R;
      int acc = 0, fb = -1, fbase = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int bb = base + lane;
        int rows = bb < p.B ? s_cu[bb + 1] - s_cu[bb] : 0;
        if (rows < 0) {
          bad = true;
          rows = 0;
        }
        const int tiles = (rows + kBM - 1) / kBM;
        const int incl = warp_incl_scan(tiles, lane);
        const bool mine = item >= acc + incl - tiles && item < acc + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, mine);
        if (hit) {
          const int src = __ffs(hit) - 1;
          fb = base + src;
          fbase = acc + __shfl_sync(0xffffffffu, incl - tiles, src);
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
      }
      bad = __any_sync(0xffffffffu, bad);
      const int count = bad ? 0 : acc;
      if (lane == 0) {
        s_item[0] = count;
        if (bad && item == 0 && h == 0 && rank == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
        if (item < count) {
          const int bq0 = s_cu[fb] + (item - fbase) * kBM;
          int kv = p.kv_len[fb];
          if (kv < 0 || kv > p.max_seq) {
            if (h == 0 && rank == 0) fdl::raise_error(p.err, FDL_DEVERR_INDEX);
            kv = max(0, min(kv, p.max_seq));
          }
          int m = 0;
          if (p.n_search) {
            m = p.n_search[fb];
            if (m < 0 || m > p.max_search_tokens) {
              if (h == 0 && rank == 0) fdl::raise_error(p.err, FDL_DEVERR_INDEX);
              m = max(0, min(m, p.max_search_tokens));
            }
          }
          s_item[1] = fb;
          s_item[2] = bq0;
          s_item[3] = min(kBM, s_cu[fb + 1] - bq0);
          s_item[4] = kv + 2 * m;
          if (p.wl_out && h == 0 && rank == 0) {
            int* w = p.wl_out + 1 + 4 * item;
            w[0] = fb;
            w[1] = bq0;
            w[2] = s_item[3];
            w[3] = s_item[4];
          }
        }
        if (p.wl_out && item == 0 && h == 0 && rank == 0) p.wl_out[0] = count;
      }
    }
    __syncthreads();
  } else if (threadIdx.x == 0) {
    s_item[0] = p.wl[0];
    if (item < s_item[0]) {
      const int* it = p.wl + 1 + 4 * item;
      s_item[1] = it[0];
      s_item[2] = it[1];
      s_item[3] = it[2];
      s_item[4] = it[3];
    }
  }
  if (p.wl) __syncthreads();
  if (item >= s_item[0]) {  // uniform over the cluster (a cluster spans x only)
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(*tmem_slot, kTmemCols);
    return;
  }
  const int b = s_item[1], q0 = s_item[2], qlen = s_item[3], nkeys = s_item[4];
  const int kvl = min(p.kv_len[b], nkeys);
  const int m_search = p.search_pos ? (nkeys - kvl) / 2 : 0;
  int n_tiles = (nkeys + kBN - 1) / kBN;
  if (n_tiles > kMaxTiles) {  // the launcher's limits rule this out; never index past the slot table
    if (threadIdx.x == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
    n_tiles = kMaxTiles;
  }
  const int t0 = (int)(rank * n_tiles / C), t1 = (int)((rank + 1) * n_tiles / C);
  const int n_my = t1 - t0;

  // slot of key tile j's first key; an unmapped page points past the cache
  // so the TMA zero-fills the tile (and the error word says so)
  auto tile_slot = [&](int j) -> int {
    const int c0 = j * kBN;
    const int pi = c0 / p.page_size;
    const int page = pi < p.bt_stride ? p.block_table[(size_t)b * p.bt_stride + pi] : -1;
    if (page >= 0 && page < p.n_pages) return page * p.page_size + c0 % p.page_size;
    fdl::raise_error(p.err, FDL_DEVERR_INDEX);
    return p.n_slots;
  };

  const int pre = min(n_my, kKS);  // key tiles issued before the CTA barrier
  if (warp == 0) {
    // every key tile's slot, looked up once by the whole warp
    for (int i = lane; i < n_my; i += 32) slots[i] = tile_slot(t0 + i);
    __syncwarp();
    if (lane == 0 && n_my > 0) {
      // Q and the first ring of key tiles need no free slot: the producer
      // (this thread) issues them now, so the loads overlap the rest of the setup
      tc::mbar_arrive_expect_tx(q_full, Q_BYTES);
      tc::tma_load_2d(sq, &tm_q, h * kHD, q0, q_full);
      tc::tma_load_2d(sq + Q_BYTES / 2, &tm_q, h * kHD + 64, q0, q_full);
      for (int lc = 0; lc < pre; ++lc) {
        uint8_t* st = kring + lc * KT_BYTES;
        tc::mbar_arrive_expect_tx(&k_full[lc], KT_BYTES);
        tc::tma_load_2d(st, &tm_k, h * kHD, slots[lc], &k_full[lc]);
        tc::tma_load_2d(st + KT_BYTES / 2, &tm_k, h * kHD + 64, slots[lc], &k_full[lc]);
      }
    }
  } else if (softmax_warp) {
    // row kinds (they decide the item's mode, so every warp needs them after
    // the barrier), a cleared search bitmap and cleared tracker column sums
    if (t_local < kBM) {  // warps 2-5, one row per thread
      const int r = t_local;
      int k = -1;
      if (r < qlen) {
        k = p.row_kind[q0 + r];
        if (k >= 2 && ((k - 2) >> 1) >= m_search) {
          fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
          k = -1;
        }
      }
      kinds[r] = k;
      const bool w = __any_sync(0xffffffffu, k == FDL_KIND_WINDOW);
      if (lane == 0) win_flags[r >> 5] = w ? 1 : 0;
    }
    for (int w = t_local; w < p.bitmap_words; w += 256) bitmap[w] = 0u;
    if (!p.wl && p.track) {
      // WINDOW rows of the whole sequence (the tracker's |M_b|), and the
      // sequence's 128-row tiles that hold them (the tracker's slots)
      const int* s_cu = reinterpret_cast<const int*>(misc + OFF_CU);
      int cnt = 0;
      for (int r = s_cu[b] + t_local; r < s_cu[b + 1]; r += 256) {
        if (p.row_kind[r] != FDL_KIND_WINDOW) continue;
        ++cnt;
        const int tt = (r - s_cu[b]) / kBM;
        if (tt < 32 * kTrkWords) atomicOr(&wbits[tt >> 5], 1u << (tt & 31));
        else wbits[kTrkWords] = 1u;
      }
      for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
      if (lane == 0 && cnt) atomicAdd(&s_item[5], cnt);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // peers' barriers and buffers must exist before any remote access: every
  // thread arrives now and waits just before its first remote access
  if (C > 1) tc::cluster_arrive();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s = tmem + 256;  // kSB 64-column S buffers; O accumulators at 0 and 128
  const int n_masked_b = p.wl ? p.n_masked[b] : s_item[5];
  const bool do_track = p.track != nullptr && n_masked_b > 0;
  const bool any_window = (win_flags[0] | win_flags[1] | win_flags[2] | win_flags[3]) != 0;
  const bool track_item = do_track && any_window;
  // deterministic tracker: this tile's slot among the sequence's WINDOW
  // tiles (decode mode with the context's partial buffer; the same decision
  // in every CTA of the sequence)
  // (found once, by one softmax thread, from the shared bitmap, and kept in
  // shared memory, s_item[6], so that it holds no register across the main
  // loops): the slot, or -1 for atomic adds
  auto trk_slot = [&]() -> int {
    if (p.wl || !p.trk_part || wbits[kTrkWords] != 0u) return -1;
    int n = 0;
    const int slot = trk_rank(wbits, (q0 - reinterpret_cast<const int*>(misc + OFF_CU)[b]) / kBM, n);
    return n <= FDL_TRK_SLOTS ? slot : -1;
  };
  // Split items and items that feed the tracker take two exact passes; the
  // others one online pass.
  const bool two_pass = C > 1 || track_item;
  // A two-pass item whose tiles all fit in the S buffers keeps pass A's
  // scores in TMEM for pass B instead of reloading K and recomputing them.
  const bool keep_s = two_pass && n_my <= kSB;
  const int n_s = two_pass && !keep_s ? 2 * n_my : n_my;  // S products = K tile loads

  if (warp == 0) {
    // ------------------------------------------------------------ K producer
    // K load lc = 0 .. n_s - 1: key tile lc % n_my (pass A, then pass B)
    if (lane == 0 && n_my > 0) {
      for (int lc = pre; lc < n_s; ++lc) {
        const int s = lc % kKS;
        if (!tc::mbar_wait(&k_empty[s], ((uint32_t)(lc / kKS) & 1u) ^ 1u, abort_flag)) break;
        const int slot = slots[lc % n_my];
        uint8_t* st = kring + s * KT_BYTES;
        tc::mbar_arrive_expect_tx(&k_full[s], KT_BYTES);
        tc::tma_load_2d(st, &tm_k, h * kHD, slot, &k_full[s]);
        tc::tma_load_2d(st + KT_BYTES / 2, &tm_k, h * kHD + 64, slot, &k_full[s]);
      }
    }
    __syncwarp();
    if (C > 1) tc::cluster_wait();  // matches the setup arrive
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ V producer
    if (lane == 0 && n_my > 0) {
      for (int i = 0; i < n_my; ++i) {
        const int s = i % kVS;
        if (!tc::mbar_wait(&v_empty[s], ((uint32_t)(i / kVS) & 1u) ^ 1u, abort_flag)) break;
        const int slot = slots[i];
        uint8_t* st = vring + s * VT_BYTES;
        tc::mbar_arrive_expect_tx(&v_full[s], VT_BYTES);
        tc::tma_load_2d(st, &tm_v, h * kHD, slot, &v_full[s]);
        tc::tma_load_2d(st + VT_BYTES / 2, &tm_v, h * kHD + 64, slot, &v_full[s]);
      }
    }
    __syncwarp();
    if (C > 1) tc::cluster_wait();  // matches the setup arrive
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The readiness checks are non-blocking (mbarrier.test_wait): a blocking
    // try_wait suspends the thread on the one barrier it tests, however soon
    // another product's operands land.
    // Issues whichever product is ready: O_g += P V for the next tile whose P
    // and V have landed (first, since it frees a P tile), else the next S =
    // Q K^T whose K tile and S buffer are free. Neither kind waits for the
    // other, so a late K load never holds back a P V product.
    if (lane == 0 && n_my > 0) {
      constexpr uint32_t id_s = tc::idesc_bf16_f32(kBM, kBN);
      constexpr uint32_t id_pv = idesc_pv(kBM, kHD);
      const uint32_t aq = tc::smem_addr(sq);
      const uint32_t ap = tc::smem_addr(sp);
      bool ok = tc::mbar_wait(q_full, 0, abort_flag);
      int si = 0, pi = 0;
      long long t_last = clock64();
      while (ok && pi < n_my) {
        bool progressed = false;
        if (tc::mbar_test_wait(&p_full[pi & 1], (uint32_t)(pi >> 1) & 1u) &&
            tc::mbar_test_wait(&v_full[pi % kVS], (uint32_t)(pi / kVS) & 1u)) {
          tc::fence_after_sync();
          const int g = pi & 1;
          const uint32_t av = tc::smem_addr(vring + (pi % kVS) * VT_BYTES);
          const uint32_t apg = ap + (uint32_t)(g * P_BYTES);
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k)
            tc::mma_bf16_ss(tmem + 128 * g, tc::desc_kmajor_sw128(apg + k * 32),
                            desc_mnmajor_sw128(av + k * 2048, VT_BYTES / 2), id_pv, (pi >= 2 || k > 0) ? 1u : 0u);
          tc::mma_commit(&pv_done[g]);
          tc::mma_commit(&v_empty[pi % kVS]);
          ++pi;
          progressed = true;
        }
        if (si < n_s && tc::mbar_test_wait(&k_full[si % kKS], (uint32_t)(si / kKS) & 1u) &&
            (si < kSB || tc::mbar_test_wait(&s_free[si % kSB], (uint32_t)((si - kSB) / kSB) & 1u))) {
          tc::fence_after_sync();
          const int sb = si % kSB;
          const uint32_t ak = tc::smem_addr(kring + (si % kKS) * KT_BYTES);
#pragma unroll
          for (int k = 0; k < kHD / 16; ++k) {
            const uint32_t half = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3) * 32u;
            tc::mma_bf16_ss(tm_s + 64 * sb, tc::desc_kmajor_sw128(aq + half * (Q_BYTES / 2) + kk),
                            tc::desc_kmajor_sw128(ak + half * (KT_BYTES / 2) + kk), id_s, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(&s_full[sb]);
          tc::mma_commit(&k_empty[si % kKS]);
          ++si;
          progressed = true;
        }
        if (progressed) {
          t_last = clock64();
        } else if (*abort_flag) {
          ok = false;
        } else if (clock64() - t_last > tc::kWaitBudgetCycles) {
          *abort_flag = 1;
          ok = false;
        }
      }
    }
    __syncwarp();
    if (C > 1) tc::cluster_wait();  // matches the setup arrive
  }

  // ------------------------------------------------------------ softmax warps
  // Two groups of four warps; group g takes the key tiles i with i % 2 == g
  // (all 64 columns of each), accumulates into its own O_g in TMEM and writes
  // its own P tile, so the two groups' tiles overlap. Warp w owns TMEM lane
  // quadrant w % 4 (32 query rows).
  const int qd = warp & 3;
  const int g = (warp - 2) >> 2;
  const int row = qd * 32 + lane;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  const uint32_t tm_og = tmem + 128 * (uint32_t)g;  // this group's O accumulator
  const int n_g = (n_my + 1 - g) / 2;               // tiles of this group
  const int n_g0 = (n_my + 1) / 2, n_g1 = n_my / 2;
  float lse2 = -INFINITY;  // log2-domain log-sum-exp of this row over all splits
  float beta0 = 1.f, beta1 = 1.f, inv_l = 1.f;  // epilogue weights of O_0, O_1 and the final scale
  if (softmax_warp) {
    for (int j = t_local; j < m_search; j += 256) {
      const int s = p.search_pos[(size_t)b * p.search_ld + j];
      if (s >= 0 && s < kvl && (s >> 5) < p.bitmap_words) atomicOr(&bitmap[s >> 5], 1u << (s & 31));
    }
    if (t_local == 0) s_item[6] = trk_slot();  // the tracker's slot, ordered by the barrier below
    tc::named_bar(3, 256);
    const int kind = kinds[row];

    // S of tile sc (global S index) into x[64]. Waits for the product and
    // releases the S buffer afterwards, except where keep_s holds the scores
    // for pass B: pass A then only waits, pass B (second) neither.
    auto load_s = [&](int sc, float (&x)[64], bool second) -> bool {
      const int sb = sc % kSB;
      // tcgen05.ld is warp-collective: the whole warp proceeds or none of it
      if (!second &&
          !__all_sync(0xffffffffu, tc::mbar_wait(&s_full[sb], (uint32_t)(sc / kSB) & 1u, abort_flag)))
        return false;
      tc::fence_after_sync();
      tc::tmem_ld_32x32b_x64(tm_s + 64 * sb + lane_off, x);
      tc::fence_before_sync();
      __syncwarp();
      if (!keep_s && lane == 0) tc::mbar_arrive(&s_free[sb]);
      return true;
    };
    // scaled scores of the visible keys, -inf elsewhere; returns the tile max
    auto mask_scale = [&](int c0, float (&x)[64]) -> float {
      const uint32_t vm0 = vis_mask(kind, c0, kvl, m_search, bitmap, p.bitmap_words);
      const uint32_t vm1 = vis_mask(kind, c0 + 32, kvl, m_search, bitmap, p.bitmap_words);
      if ((vm0 & vm1) == 0xffffffffu) {
#pragma unroll
        for (int k = 0; k < 64; ++k) x[k] *= p.scale_log2;
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          x[k] = ((vm0 >> k) & 1u) ? x[k] * p.scale_log2 : -INFINITY;
          x[k + 32] = ((vm1 >> k) & 1u) ? x[k + 32] * p.scale_log2 : -INFINITY;
        }
      }
      float t16[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) t16[k] = fmaxf(fmaxf(x[k], x[k + 16]), fmaxf(x[k + 32], x[k + 48]));
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) t16[k] = fmaxf(t16[k], t16[k + w]);
      return t16[0];
    };

    float m_run = -INFINITY, l_run = 0.f;
    if (two_pass) {
      // ---- pass A: exact running max and sum over this group's tiles
      for (int k = 0; k < n_g; ++k) {
        const int i = 2 * k + g;
        float x[64];
        if (!load_s(i, x, false)) break;
        const float tmax = mask_scale((t0 + i) * kBN, x);
        if (tmax == -INFINITY) continue;
        const float mnew = fmaxf(m_run, tmax);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          a0 += ex2(x[e] - mnew);
          a1 += ex2(x[e + 1] - mnew);
          a2 += ex2(x[e + 2] - mnew);
          a3 += ex2(x[e + 3] - mnew);
        }
        l_run = (m_run == -INFINITY ? 0.f : l_run * ex2(m_run - mnew)) + ((a0 + a1) + (a2 + a3));
        m_run = mnew;
      }
      // ---- the two groups of each row combine their (max, sum)
      halfml[(g * kBM + row) * 2] = m_run;
      halfml[(g * kBM + row) * 2 + 1] = l_run;
      tc::named_bar(2, 256);
      float mrow, lrow;
      {
        const float mo = halfml[((1 - g) * kBM + row) * 2], lo = halfml[((1 - g) * kBM + row) * 2 + 1];
        mrow = fmaxf(m_run, mo);
        lrow = 0.f;
        if (mrow != -INFINITY) {
          if (m_run != -INFINITY) lrow += l_run * ex2(m_run - mrow);
          if (mo != -INFINITY) lrow += lo * ex2(mo - mrow);
        }
      }
      // ---- combine (max, sum) over the cluster
      if (C > 1) {
        tc::cluster_wait();  // peers have initialised their barriers (setup arrive)
        if (g == 0) {
          // push this row's (max, sum) into every split, then release-arrive there
          const uint32_t mine = tc::smem_addr(ml + ((size_t)rank * kBM + row) * 2);
          for (int r = 0; r < C; ++r) st_cluster_v2(tc::map_cluster(mine, (uint32_t)r), mrow, lrow);
          // one release-arrive per warp and destination: every lane's remote
          // stores are ordered before lane 0's arrive by its cluster-scope
          // fence and the warp barrier
          fence_acq_rel_cluster();
          __syncwarp();
          if (lane == 0)
            for (int r = 0; r < C; ++r) mbar_arrive_remote(ml_ready, (uint32_t)r);
        }
        mbar_wait_cluster(ml_ready, 0, abort_flag);
        float mm = -INFINITY;
        for (int r = 0; r < C; ++r) mm = fmaxf(mm, ml[((size_t)r * kBM + row) * 2]);
        float ll = 0.f;
        if (mm != -INFINITY)
          for (int r = 0; r < C; ++r) {
            const float mr = ml[((size_t)r * kBM + row) * 2], lr = ml[((size_t)r * kBM + row) * 2 + 1];
            if (mr != -INFINITY) ll += lr * ex2(mr - mm);
          }
        lse2 = ll > 0.f ? mm + log2f(ll) : -INFINITY;
      } else {
        lse2 = lrow > 0.f ? mrow + log2f(lrow) : -INFINITY;
      }
      if (p.lse && rank == 0 && g == 0 && row < qlen) p.lse[(size_t)(q0 + row) * p.H + h] = lse2 * kLn2;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    // ---- pass B (two_pass: final probabilities P = exp(S - lse)) or the one
    // online pass (P = exp(S - m) against a running row max m that moves only
    // when a tile's max exceeds it by more than kRescale; O_g and the row sum
    // are then scaled down to the new m)
    const int sc0 = two_pass && !keep_s ? n_my : 0;
    const float wscale = do_track ? 1.f / ((float)p.H * (float)n_masked_b) : 0.f;
    const bool track_row = do_track && kind == FDL_KIND_WINDOW;
    const bool track_warp = __any_sync(0xffffffffu, track_row);
    const int t_g = t_local - 128 * g;  // 0..127 within the group
    for (int k = 0; k < n_g; ++k) {
      // a wait that gives up (abort) skips the work but never the barriers
      const int i = 2 * k + g;
      const int c0 = (t0 + i) * kBN;
      float pr[64];
      bool ok = load_s(sc0 + i, pr, keep_s);
      bool waited_pv = false;
      if (ok) {
        if (two_pass) {
          if (lse2 == -INFINITY) {
#pragma unroll
            for (int e = 0; e < 64; ++e) pr[e] = 0.f;
          } else {
            mask_scale(c0, pr);
#pragma unroll
            for (int e = 0; e < 64; ++e) pr[e] = ex2(pr[e] - lse2);
          }
        } else {
          const float tmax = mask_scale(c0, pr);
          float alpha = 1.f;
          bool resc = false;
          if (tmax != -INFINITY) {
            if (m_run == -INFINITY) {
              m_run = tmax;  // this row's O_g holds only zeros so far
            } else if (tmax > m_run + kRescale) {
              alpha = ex2(m_run - tmax);
              m_run = tmax;
              resc = true;
            }
          }
          if (m_run == -INFINITY) {
#pragma unroll
            for (int e = 0; e < 64; ++e) pr[e] = 0.f;
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) pr[e] = ex2(pr[e] - m_run);
          }
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            s0 += pr[e];
            s1 += pr[e + 1];
            s2 += pr[e + 2];
            s3 += pr[e + 3];
          }
          l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));
          if (__any_sync(0xffffffffu, resc)) {
            // O_g rows move to the new max once the group's previous P V
            // product (tile i - 2) has finished and before this tile's starts
            ok = i < 2 || __all_sync(0xffffffffu, tc::mbar_wait(&pv_done[g], (uint32_t)((i - 2) >> 1) & 1u, abort_flag));
            waited_pv = true;
            if (ok && i >= 2) {
              tc::fence_after_sync();
#pragma unroll 1
              for (int cc = 0; cc < kHD; cc += 32) {
                float o[32];
                tc::tmem_ld_32x32b_x32(tm_og + cc + lane_off, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] *= alpha;
                tc::tmem_st_32x32b_x32(tm_og + cc + lane_off, o);
              }
              tc::tmem_wait_st();
            }
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) pr[e] = 0.f;
      }
      // P tile g was last read by the P V product of tile i - 2
      if (!waited_pv) ok = ok && (i < 2 || tc::mbar_wait(&pv_done[g], (uint32_t)((i - 2) >> 1) & 1u, abort_flag));
      if (ok) {
        // P in the 128-byte swizzled K-major layout: row r, 16-byte chunk q at q ^ (r & 7)
        uint8_t* prow = sp + g * P_BYTES + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(pr[q * 8 + 2 * e], pr[q * 8 + 2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(prow + ((q ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // keys past the sequence end may hold anything: zero their V rows so
        // that 0 * V stays 0 in the P V product
        if (c0 + kBN > nkeys && tc::mbar_wait(&v_full[i % kVS], (uint32_t)(i / kVS) & 1u, abort_flag)) {
          uint8_t* vt = vring + (i % kVS) * VT_BYTES;
          const int first = max(0, nkeys - c0);
          for (int e = lane; e < (kBN - first) * 16; e += 32) {
            const int r = first + e / 16, part = e % 16;
            if ((r & 3) != qd) continue;  // the group's four warps split the rows
            *reinterpret_cast<uint4*>(vt + (part >> 3) * (VT_BYTES / 2) + r * 128 + (part & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
      }
      __syncwarp();
      if (ok && lane == 0) tc::mbar_arrive(&p_full[g]);
      if (two_pass && track_item) {
        if (track_warp) {  // a warp without WINDOW rows adds nothing
          if (!track_row) {
#pragma unroll
            for (int e = 0; e < 64; ++e) pr[e] = 0.f;
          }
          float* lo = pr;
          float* hi = pr + 32;
          warp_colsum32(*reinterpret_cast<float(*)[32]>(lo), lane);
          warp_colsum32(*reinterpret_cast<float(*)[32]>(hi), lane);
          colacc[(g * 4 + qd) * 64 + lane] = pr[0];
          colacc[(g * 4 + qd) * 64 + 32 + lane] = pr[32];
        } else {
          colacc[(g * 4 + qd) * 64 + lane] = 0.f;
          colacc[(g * 4 + qd) * 64 + 32 + lane] = 0.f;
        }
        // the group's four warps' column sums, added in a fixed order
        tc::named_bar(4 + g, 128);
        if (t_g < 64) {
          const int c = c0 + t_g;
          const float v = ((colacc[(g * 4 + 0) * 64 + t_g] + colacc[(g * 4 + 1) * 64 + t_g]) +
                           colacc[(g * 4 + 2) * 64 + t_g]) + colacc[(g * 4 + 3) * 64 + t_g];
          if (c < kvl) {
            const int slot = s_item[6];
            if (slot >= 0) {
              trk_row(p.trk_part, b, slot, h, p.H, p.trk_ld)[c] = v * wscale;
            } else if (v != 0.f) {
              atomicAdd(p.track + (size_t)b * p.track_ld + c, v * wscale);
            }
          }
        }
        tc::named_bar(4 + g, 128);
      }
    }
    // Every P V product of both groups has finished before O is read: each
    // group waits for its own last product (a parity wait is exact only one
    // phase ahead, which holds for the group that waited on the earlier
    // phases), then the two groups meet at barrier 2.
    if (n_g > 0) tc::mbar_wait(&pv_done[g], (uint32_t)(n_g - 1) & 1u, abort_flag);
    if (!two_pass) {
      halfml[(g * kBM + row) * 2] = m_run;
      halfml[(g * kBM + row) * 2 + 1] = l_run;
    }
    tc::fence_before_sync();
    tc::named_bar(2, 256);
    tc::fence_after_sync();
    if (!two_pass) {
      // the two groups' (max, sum) give the row's normaliser and the weights of O_0, O_1
      const float m0 = halfml[row * 2], l0 = halfml[row * 2 + 1];
      const float m1 = halfml[(kBM + row) * 2], l1 = halfml[(kBM + row) * 2 + 1];
      const float m = fmaxf(m0, m1);
      if (m != -INFINITY) {
        beta0 = m0 != -INFINITY ? ex2(m0 - m) : 0.f;
        beta1 = m1 != -INFINITY ? ex2(m1 - m) : 0.f;
        const float l = l0 * beta0 + l1 * beta1;
        lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
        inv_l = l > 0.f ? 1.f / l : 0.f;
      }
      if (p.lse && g == 0 && row < qlen) p.lse[(size_t)(q0 + row) * p.H + h] = lse2 * kLn2;
    }
    if (n_g0 == 0) beta0 = 0.f;  // an accumulator no product wrote holds garbage
    if (n_g1 == 0) beta1 = 0.f;
  }

  // ------------------------------------------------------------ output
  // Each softmax warp owns O columns [64 g, 64 g + 64) of its 32 rows and
  // combines O_0 and O_1 there. TMEM loads are warp-collective: issued by
  // whole warps, with per-row conditions only selecting values and guarding
  // stores.
  constexpr int kOStride = kHD + 4;  // padded fp32 staging rows: conflict-free float4 access
  auto o_cols = [&](int c0, float (&a)[32]) {
    float o1[32];
    tc::tmem_ld_32x32b_x32(tmem + c0 + lane_off, a);
    tc::tmem_ld_32x32b_x32(tmem + 128 + c0 + lane_off, o1);
    const bool live = n_my > 0 && lse2 != -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float v0 = beta0 != 0.f ? a[e] * beta0 : 0.f;
      const float v1 = beta1 != 0.f ? o1[e] * beta1 : 0.f;
      a[e] = live ? (v0 + v1) * inv_l : 0.f;
    }
  };
  if (C == 1) {
    if (softmax_warp) {
      const bool store = row < qlen && !*abort_flag;
      __nv_bfloat16* orow = p.o + (size_t)(q0 + row) * p.d + h * kHD;
#pragma unroll 1
      for (int cc = 0; cc < 64; cc += 32) {
        const int c0 = 64 * g + cc;
        float a[32];
        o_cols(c0, a);
        if (!store) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(a[q * 8 + 2 * e], a[q * 8 + 2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(orow + c0 + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  } else {
    // every split stages its fp32 partial O (already normalised) in its two
    // drained rings; split r then sums its share of the valid rows over all
    // splits in rank order
    float* ostage = reinterpret_cast<float*>(kring);  // [128][kOStride], over both rings
    if (softmax_warp) {
#pragma unroll 1
      for (int cc = 0; cc < 64; cc += 32) {
        const int c0 = 64 * g + cc;
        float a[32];
        o_cols(c0, a);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(ostage + row * kOStride + c0 + 4 * q) =
              make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
      }
    }
    tc::cluster_sync();
    if (softmax_warp) {
      const uint32_t base = tc::smem_addr(ostage);
      const bool ab = *abort_flag != 0;
      if (C == 2) merge_o<2>(p, base, rank, t_local, q0, qlen, h, ab);
      else if (C == 4) merge_o<4>(p, base, rank, t_local, q0, qlen, h, ab);
      else merge_o<8>(p, base, rank, t_local, q0, qlen, h, ab);
    }
    tc::cluster_sync();  // peers finished reading this CTA's staged O
  }

  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) fdl::raise_error(p.err, FDL_DEVERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
  // the sequence's first CTA records its partial slots for the sums below
  // (recomputed from the shared bitmap, which is still intact)
  // (everything re-read from shared memory and the grid indices, so that no
  // register stays live across the main loops for it)
  if (!p.wl && p.trk_part && threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.x == 0) {
    const int sb = s_item[1];
    if (s_item[2] == reinterpret_cast<const int*>(misc + OFF_CU)[sb]) {
      int n = 0;
      trk_rank(wbits, 0, n);
      p.trk_nslots[sb] = p.track && s_item[5] > 0 && wbits[kTrkWords] == 0u && n <= FDL_TRK_SLOTS ? n : 0;
    }
  }
}

// The tracker's fixed-order sums: grid (sequence, 64-column chunk), 256
// threads = 4 groups of a quarter of the heads x 64 columns. Each thread adds
// its group's heads for every slot (slots outer, heads in order), then each
// column adds the four group sums in group order into the scores.
constexpr int kFinThreads = 256;
__global__ void __launch_bounds__(kFinThreads)
    trk_finalize_kernel(const float* part, const int* nslots, const int* cu, const int* kv_len, int max_seq, int H,
                        int ld, float* track, int track_ld) {
  __shared__ float gsum[4][64];
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int b = blockIdx.x, c = blockIdx.y * 64 + (threadIdx.x & 63), grp = threadIdx.x >> 6;
  if (cu[b + 1] - cu[b] <= 0) return;  // no rows: no CTA recorded this sequence
  const int n = nslots[b];
  const int kvl = max(0, min(kv_len[b], max_seq));
  if (n <= 0 || blockIdx.y * 64 >= kvl) return;
  const int hpg = (H + 3) / 4, h0 = grp * hpg, h1 = min(H, h0 + hpg);
  float acc = 0.f;
  if (c < kvl) {
    for (int sl = 0; sl < n; ++sl) {
      const float* src = part + ((size_t)(b * FDL_TRK_SLOTS + sl) * H) * ld + c;
#pragma unroll 8
      for (int hh = h0; hh < h1; ++hh) acc += __ldcg(src + (size_t)hh * ld);
    }
  }
  gsum[grp][threadIdx.x & 63] = acc;
  __syncthreads();
  if (threadIdx.x < 64 && c < kvl)
    track[(size_t)b * track_ld + c] += ((gsum[0][threadIdx.x] + gsum[1][threadIdx.x]) + gsum[2][threadIdx.x]) +
                                       gsum[3][threadIdx.x];
}

}  // namespace

bool fdl_attn_pair_applies(int R, int B, int C);
cudaError_t fdl_launch_attn_pair(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                                 const int* block_table, int bt_stride, const int* cu_seqlens_q, const int* kv_len,
                                 int B, int R, const int* row_kind, const int* search_pos, int search_ld,
                                 const int* n_search, int max_search_tokens, void* o_out, float* lse_out, float* track,
                                 int track_ld, int* worklist_out);

bool fdl_attn_tc_supported(const fdl_config& c) {
  // head_dim 128, bf16, and every 64-key tile inside one page: pages are a
  // multiple of 64 slots, or one page holds a whole sequence plus its views
  return c.dtype == FDL_BF16 && c.head_dim == kHD &&
         (c.page_size % kBN == 0 || c.page_size >= c.max_seq + c.max_views) &&
         (c.max_seq + c.max_views + 31) / 32 <= 768;
}

int fdl_attn_tc_decode_max_batch() { return kMaxDecodeB; }

// decode: the kernel finds its work items from cu_seqlens_q itself (and
// writes them to worklist_out when given); otherwise it reads the work list
// built into the context's workspace.
cudaError_t fdl_launch_attn_tc(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                               const int* block_table, int bt_stride, const int* cu_seqlens_q, const int* kv_len,
                               int B, int R, const int* row_kind, const int* search_pos, int search_ld,
                               const int* n_search, int max_search_tokens, void* o_out, float* lse_out, float* track,
                               int track_ld, int cap, bool decode, int* worklist_out) {
  const fdl_config& c = ctx->cfg;
  if (decode && B > kMaxDecodeB) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(o_out)) & 15)
    return cudaErrorMisalignedAddress;
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)attn_tc_kernel, ctx->device, SMEM_BYTES)) return e;
  const int n_slots = c.n_pages * c.page_size;
  CUtensorMap mq, mk, mv;
  if (!map2d(&mq, q, R, c.d_model, kBM) || !map2d(&mk, k_cache, n_slots, c.d_model, kBN) ||
      !map2d(&mv, v_cache, n_slots, c.d_model, kBN))
    return cudaErrorInvalidValue;
  TcAttnParams p;
  p.wl = decode ? nullptr : ctx->worklist;
  p.cu = cu_seqlens_q;
  p.n_search = search_pos ? n_search : nullptr;
  p.B = B;
  p.max_seq = c.max_seq;
  p.max_search_tokens = max_search_tokens;
  p.wl_out = worklist_out;
  p.kv_len = kv_len;
  p.row_kind = row_kind;
  p.search_pos = search_pos;
  p.search_ld = search_ld;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.page_size = c.page_size;
  p.n_pages = c.n_pages;
  p.n_slots = n_slots;
  p.n_masked = ctx->n_masked;
  p.o = reinterpret_cast<__nv_bfloat16*>(o_out);
  p.lse = lse_out;
  p.track = track;
  p.track_ld = track_ld;
  p.trk_part = track ? ctx->trk_part : nullptr;
  p.trk_nslots = ctx->trk_nslots;
  p.trk_ld = ctx->trk_ld;
  p.H = c.n_heads;
  p.d = c.d_model;
  p.R = R;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
  p.bitmap_words = (c.max_seq + c.max_views + 31) / 32;
  p.err = ctx->err_word;
  // splits per item: fill the SMs when items x heads alone cannot
  const int est_items = (R + kBM - 1) / kBM + B - 1;
  int C = 1;
  while (C < kMaxC && est_items * c.n_heads * (2 * C) <= ctx->num_sms) C *= 2;
  p.C = C;
  // sequences of two or more query tiles without a KV split: two tiles per CTA
  // the tracker's fixed-order sums follow the attention launch (decode mode
  // with the context's partial buffer)
  auto finalize = [&](cudaError_t e) -> cudaError_t {
    if (e != cudaSuccess || !p.trk_part || !decode || B <= 0) return e;
    return fdl_launch_pdl(trk_finalize_kernel, dim3((unsigned)B, (unsigned)((c.max_seq + 63) / 64)),
                          dim3(kFinThreads, 1, 1), 0, ctx->stream, 1, (const float*)ctx->trk_part,
                          (const int*)ctx->trk_nslots, cu_seqlens_q, kv_len, c.max_seq, c.n_heads, ctx->trk_ld, track,
                          track_ld);
  };
  if (decode && fdl_attn_pair_applies(R, B, C))
    return finalize(fdl_launch_attn_pair(ctx, q, k_cache, v_cache, block_table, bt_stride, cu_seqlens_q, kv_len, B,
                                         R, row_kind, search_pos, search_ld, n_search, max_search_tokens, o_out,
                                         lse_out, track, track_ld, worklist_out));
  // grid (split, head, item): items vary slowest, so the CTAs of real items
  // are scheduled before any idle tail. Sequence b contributes
  // ceil(rows_b / 128) items, and summed over the sequences with rows that
  // is at most ceil(R / 128) + B - 1, so no more CTAs are launched.
  const int items = min(cap, est_items);
  if (items > 65535) return cudaErrorInvalidConfiguration;
  return finalize(fdl_launch_pdl(attn_tc_kernel, dim3((unsigned)C, (unsigned)c.n_heads, (unsigned)items),
                                 dim3(kThreads, 1, 1), SMEM_BYTES, ctx->stream, C, mq, mk, mv, p));
}
