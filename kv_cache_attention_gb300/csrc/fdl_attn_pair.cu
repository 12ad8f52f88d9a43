// Block-table scheduled attention for two query tiles of one sequence per
// CTA, on the 5th-generation tensor cores, with the Flash-Verify two-view
// mask and the Eq. (2) attention-mass tracker fused in.
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
// This kernel serves calls whose sequences mostly hold two or more 128-row
// query tiles (a full refresh: every position of a sequence is a query row).
// One CTA = (pair of consecutive 128-row query tiles of a sequence, head):
// every K/V tile it loads feeds both query tiles, so the K/V bytes per
// product are half those of one tile per CTA. A sequence with an odd tile
// count ends in a pair with one tile. Key tiles are 128 keys wide: a score
// product is 128 x 128 x 128, whose operands the tensor core reads from
// shared memory at its full rate (64-key tiles re-read the query tile twice
// as often per key and leave the products shared-memory bound).
//
// Per query tile g (0, 1) there is one softmax group of four warps (one per
// TMEM lane quadrant, one query row per thread), an O accumulator O_g and a
// 128-column S buffer in TMEM. The group writes the probabilities P as bf16
// back into the S buffer it read, and O_g += P V takes P straight from TMEM
// as its A operand: P never touches shared memory. The next scores of a
// group go into the same buffer, so its S product waits for its P V
// product; the MMA issuer fills that gap with the other group's products,
// and a group's O_g is never being written while the group works on a tile.
//
// Two modes per CTA:
//   online    (no WINDOW row of the pair feeds the tracker) one pass: P =
//             exp(S - m) against a running row max m that moves only when a
//             tile's max exceeds it by more than 2^kRescale; O_g and the row
//             sum are then scaled to the new m. O = O_g / l at the end. The
//             tile max comes from a first read of the scores' two halves.
//   two-pass  (a WINDOW row of the pair feeds Eq. (2)) pass A gives each
//             row's exact log-sum-exp; pass B forms the final probabilities
//             P = exp(S - lse), whose column sums over WINDOW rows are the
//             tracker's contribution (summed over the group's four warps in
//             a fixed order), and O = O_g. K is read twice.
//
// Warp roles (352 threads): warp 0 TMA producer of the two Q tiles and a
// 2-stage K ring (a stage is released once both groups' S products have
// read it), warp 10 TMA producer of a 2-stage V ring, warp 1 TMEM owner and
// MMA issuer (one lane; it issues whichever of the next P V or the next S is
// ready, polling without blocking), warps 2-5 group 0, warps 6-9 group 1.
#include <cudaTypedefs.h>
#include <math.h>

#include "fdl_internal.cuh"
#include "fdl_attn_tc.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kBM = 128;    // query rows per tile
constexpr int kBN = 128;    // keys per tile
constexpr int kSub = 64;    // keys per TMA box (and per entry of the slot table)
constexpr int kHD = 128;    // head dim handled here
constexpr int kThreads = 352;
constexpr int kVWarp = 10;  // V producer
constexpr int kKS = 2;      // K ring stages
constexpr int kVS = 2;      // V ring stages
constexpr int kTmemCols = 512;   // O_0, O_1, S_0, S_1 (128 columns each)
constexpr float kRescale = 8.f;  // online mode: log2 headroom of P before the row max moves
constexpr int kMaxSub = 384;     // 64-key sub-tiles of one sequence: (max_seq + max_views) / 64
constexpr int kMaxDecodeB = 1024;

constexpr int Q_BYTES = kBM * kHD * 2;   // one query tile: two 64-column halves of 16 KB
constexpr int KT_BYTES = kBN * kHD * 2;  // K tile: two halves of 16 KB (128 key rows of 128 B)
constexpr int VT_BYTES = kBN * kHD * 2;  // V tile: the same
constexpr int SUB_BYTES = kSub * 128;    // one 64-row TMA box of 128-byte rows

constexpr int OFF_Q = 0;  // query tiles 0 and 1
constexpr int OFF_KRING = OFF_Q + 2 * Q_BYTES;
constexpr int OFF_VRING = OFF_KRING + kKS * KT_BYTES;
constexpr int OFF_MISC = OFF_VRING + kVS * VT_BYTES;
// misc: barriers and flags [0, 512), row kinds of both tiles, the tracker's
// per-warp column sums, the search bitmap (<= 768 words), WINDOW flags,
// sub-tile slots, the work item, staged cu_seqlens_q
constexpr int OFF_KINDS = 512;                        // int [256]
constexpr int OFF_COLW = OFF_KINDS + 4 * 2 * kBM;     // float [8 warps][128]
constexpr int OFF_BITMAP = OFF_COLW + 8 * kBN * 4;    // uint32 [768]
constexpr int OFF_FLAGS = OFF_BITMAP + 768 * 4;       // int [8]: WINDOW rows in each 32-row group
constexpr int OFF_SLOTS = OFF_FLAGS + 64;             // int [kMaxSub]
constexpr int OFF_ITEM = OFF_SLOTS + 4 * kMaxSub;     // int [16]
constexpr int OFF_CU = OFF_ITEM + 64;                 // int [kMaxDecodeB + 1]
constexpr int OFF_WBITS = OFF_CU + 4 * (kMaxDecodeB + 1);  // uint32 [kTrkWords]: the sequence's WINDOW tiles, then 2 flags
constexpr int MISC_BYTES = OFF_WBITS + 4 * (kTrkWords + 2);
constexpr int SMEM_BYTES = 1024 + OFF_MISC + MISC_BYTES;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(8 * (1 + 2 * kKS + 2 * kVS + 10) + 16 <= OFF_KINDS, "barriers fit");

constexpr float kLn2 = 0.6931471805599453f;

struct PairParams {
  const int* cu;          // cu_seqlens_q [B + 1]
  const int* n_search;    // [B] or null
  int B, max_seq, max_search_tokens;
  int* wl_out;            // optional copy of the 128-row work items used
  const int* kv_len;
  const int* row_kind;
  const int* search_pos;
  int search_ld;
  const int* block_table;
  int bt_stride, page_size, n_pages, n_slots;
  __nv_bfloat16* o;
  float* lse;
  float* track;
  int track_ld;
  float* trk_part;        // deterministic tracker partials (null: atomics into track)
  int* trk_nslots;        // [B] slots of each sequence's partials (0: none, atomics)
  int trk_ld;
  int H, d, R;
  float scale_log2;       // log2(e) / sqrt(head_dim)
  int bitmap_words;
  unsigned* err;
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem + OFF_Q;
  uint8_t* kring = smem + OFF_KRING;
  uint8_t* vring = smem + OFF_VRING;
  uint8_t* misc = smem + OFF_MISC;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;           // [kKS]
  uint64_t* k_empty = k_full + kKS;      // [kKS]
  uint64_t* v_full = k_empty + kKS;      // [kVS]
  uint64_t* v_empty = v_full + kVS;      // [kVS]
  uint64_t* s_full = v_empty + kVS;      // [2 groups]: scores of the group's next product written
  uint64_t* s_free_a = s_full + 2;       // [2]: pass A, the group has read its scores
  uint64_t* s_free_b = s_free_a + 2;     // [2]: pass B / online, the P V product has read P
  uint64_t* p_full = s_free_b + 2;       // [2]: P of the group's tile written
  uint64_t* pv_done = p_full + 2;        // [2]: the group's P V product done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pv_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* kinds = reinterpret_cast<int*>(misc + OFF_KINDS);              // [256]
  float* colw = reinterpret_cast<float*>(misc + OFF_COLW);            // [8][128]
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(misc + OFF_BITMAP);  // [bitmap_words]
  int* win_flags = reinterpret_cast<int*>(misc + OFF_FLAGS);          // [8]
  int* slots = reinterpret_cast<int*>(misc + OFF_SLOTS);              // [n_sub]
  int* s_item = reinterpret_cast<int*>(misc + OFF_ITEM);
  int* s_cu = reinterpret_cast<int*>(misc + OFF_CU);
  uint32_t* wbits = reinterpret_cast<uint32_t*>(misc + OFF_WBITS);  // [kTrkWords], [kTrkWords]: overflow, +1: last

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int item = blockIdx.y;
  const bool softmax_warp = warp >= 2 && warp < 10;
  const int t_local = threadIdx.x - 64;  // 0..255 over the softmax warps

  // ---------------------------------------------------------------- setup
  // Barriers, TMEM and the tensor-map prefetch touch no global memory, so
  // they overlap the end of the previous kernel in the stream.
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
    for (int g = 0; g < 2; ++g) {
      tc::mbar_init(&s_full[g], 1);
      tc::mbar_init(&s_free_a[g], 4);  // the four warps of the group
      tc::mbar_init(&s_free_b[g], 1);
      tc::mbar_init(&p_full[g], 4);
      tc::mbar_init(&pv_done[g], 1);
    }
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

  // The work item from cu_seqlens_q: sequence b holds ceil(rows_b / 128)
  // query tiles and ceil(tiles_b / 2) pairs, in order; item z of the grid is
  // found by prefix sums over the staged offsets. Inconsistent offsets
  // (cu[0] != 0, cu[B] != R, a negative row count) leave no items and set
  // the shape error.
  for (int i = threadIdx.x; i <= p.B; i += kThreads) s_cu[i] = p.cu[i];
  if (threadIdx.x == 0) s_item[7] = 0;
  if (threadIdx.x < kTrkWords + 1) wbits[threadIdx.x] = 0u;
  __syncthreads();
  if (warp == 0) {
    bool bad = s_cu[0] != 0 || s_cu[p.B] != p.R;
    int accp = 0, acct = 0, fb = -1, fbase_p = 0, fbase_t = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int bb = base + lane;
      int rows = bb < p.B ? s_cu[bb + 1] - s_cu[bb] : 0;
      if (rows < 0) {
        bad = true;
        rows = 0;
      }
      const int tiles = (rows + kBM - 1) / kBM;
      const int pairs = (tiles + 1) / 2;
      const int incl_p = warp_incl_scan(pairs, lane);
      const int incl_t = warp_incl_scan(tiles, lane);
      const bool mine = item >= accp + incl_p - pairs && item < accp + incl_p;
      const unsigned hit = __ballot_sync(0xffffffffu, mine);
      if (hit) {
        const int src = __ffs(hit) - 1;
        fb = base + src;
        fbase_p = accp + __shfl_sync(0xffffffffu, incl_p - pairs, src);
        fbase_t = acct + __shfl_sync(0xffffffffu, incl_t - tiles, src);
      }
      accp += __shfl_sync(0xffffffffu, incl_p, 31);
      acct += __shfl_sync(0xffffffffu, incl_t, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    const int count = bad ? 0 : accp;
    if (lane == 0) {
      s_item[0] = count;
      if (bad && item == 0 && h == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
      if (item < count) {
        const int tile0 = 2 * (item - fbase_p);
        const int rows_b = s_cu[fb + 1] - s_cu[fb];
        const int bq0 = s_cu[fb] + tile0 * kBM;
        const int qlen0 = min(kBM, rows_b - tile0 * kBM);
        const int qlen1 = max(0, min(kBM, rows_b - (tile0 + 1) * kBM));
        int kv = p.kv_len[fb];
        if (kv < 0 || kv > p.max_seq) {
          if (h == 0) fdl::raise_error(p.err, FDL_DEVERR_INDEX);
          kv = max(0, min(kv, p.max_seq));
        }
        int m = 0;
        if (p.n_search) {
          m = p.n_search[fb];
          if (m < 0 || m > p.max_search_tokens) {
            if (h == 0) fdl::raise_error(p.err, FDL_DEVERR_INDEX);
            m = max(0, min(m, p.max_search_tokens));
          }
        }
        s_item[1] = fb;
        s_item[2] = bq0;
        s_item[3] = qlen0;
        s_item[4] = qlen1;
        s_item[5] = kv + 2 * m;
        s_item[6] = kv;
        if (p.wl_out && h == 0) {
          int* w = p.wl_out + 1 + 4 * (fbase_t + tile0);
          w[0] = fb;
          w[1] = bq0;
          w[2] = qlen0;
          w[3] = kv + 2 * m;
          if (qlen1 > 0) {
            w[4] = fb;
            w[5] = bq0 + kBM;
            w[6] = qlen1;
            w[7] = kv + 2 * m;
          }
        }
      }
      if (p.wl_out && item == 0 && h == 0) p.wl_out[0] = bad ? 0 : acct;
    }
  }
  __syncthreads();
  if (item >= s_item[0]) {
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(*tmem_slot, kTmemCols);
    return;
  }
  const int b = s_item[1], q0 = s_item[2], qlen0 = s_item[3], qlen1 = s_item[4], nkeys = s_item[5];
  const int kvl = s_item[6];
  const int m_search = p.search_pos ? (nkeys - kvl) / 2 : 0;
  const bool has1 = qlen1 > 0;
  const int n_g = has1 ? 2 : 1;  // query tiles of this CTA
  int n_sub = (nkeys + kSub - 1) / kSub;  // 64-key sub-tiles
  if (n_sub > kMaxSub) {  // the launcher's limits rule this out; never index past the slot table
    if (threadIdx.x == 0) fdl::raise_error(p.err, FDL_DEVERR_SHAPE);
    n_sub = kMaxSub;
  }
  const int n_tiles = (n_sub + 1) / 2;     // 128-key tiles

  // slot of 64-key sub-tile j's first key; an unmapped page, or the second
  // half of a sequence's last tile past its keys, points past the cache so
  // that the TMA zero-fills the box (an unmapped page sets the error word)
  auto sub_slot = [&](int j) -> int {
    if (j >= n_sub) return p.n_slots;
    const int c0 = j * kSub;
    const int pi = c0 / p.page_size;
    const int page = pi < p.bt_stride ? p.block_table[(size_t)b * p.bt_stride + pi] : -1;
    if (page >= 0 && page < p.n_pages) return page * p.page_size + c0 % p.page_size;
    fdl::raise_error(p.err, FDL_DEVERR_INDEX);
    return p.n_slots;
  };
  // key tile t (two sub-tiles, each two 64-dim halves) into ring stage st:
  // the boxes of a half stack into 128 rows of the 128-byte swizzle layout
  auto load_kv = [&](const CUtensorMap* map, uint8_t* st, int t, uint64_t* bar) {
    tc::mbar_arrive_expect_tx(bar, KT_BYTES);
    for (int hf = 0; hf < 2; ++hf)
      for (int sb = 0; sb < 2; ++sb)
        tc::tma_load_2d(st + hf * (KT_BYTES / 2) + sb * SUB_BYTES, map, h * kHD + hf * 64, slots[2 * t + sb], bar);
  };

  const int pre = min(n_tiles, kKS);  // key tiles issued before the CTA barrier
  if (warp == 0) {
    for (int i = lane; i < 2 * n_tiles; i += 32) slots[i] = sub_slot(i);
    __syncwarp();
    if (lane == 0 && n_tiles > 0) {
      // the query tiles and the first ring of key tiles need no free slot
      tc::mbar_arrive_expect_tx(q_full, (uint32_t)(Q_BYTES * n_g));
      for (int g = 0; g < n_g; ++g) {
        uint8_t* dq = sq + g * Q_BYTES;
        tc::tma_load_2d(dq, &tm_q, h * kHD, q0 + g * kBM, q_full);
        tc::tma_load_2d(dq + Q_BYTES / 2, &tm_q, h * kHD + 64, q0 + g * kBM, q_full);
      }
      for (int lc = 0; lc < pre; ++lc) load_kv(&tm_k, kring + lc * KT_BYTES, lc, &k_full[lc]);
    }
  } else if (softmax_warp) {
    // row kinds of both tiles (they decide the mode), a cleared search
    // bitmap, and the WINDOW rows of the whole sequence (the tracker's |M_b|)
    {
      const int r = t_local;  // 0..255: tile r / 128, row r % 128
      const int qlen = r < kBM ? qlen0 : qlen1;
      const int rr = r % kBM;
      int k = -1;
      if (rr < qlen) {
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
    if (p.track) {
      // and the sequence's 128-row tiles that hold them (the tracker's slots)
      int cnt = 0;
      for (int r = s_cu[b] + t_local; r < s_cu[b + 1]; r += 256) {
        if (p.row_kind[r] != FDL_KIND_WINDOW) continue;
        ++cnt;
        const int tt = (r - s_cu[b]) / kBM;
        if (tt < 32 * kTrkWords) atomicOr(&wbits[tt >> 5], 1u << (tt & 31));
        else wbits[kTrkWords] = 1u;
      }
      for (int off = 16; off; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
      if (lane == 0 && cnt) atomicAdd(&s_item[7], cnt);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int n_masked_b = s_item[7];
  const bool do_track = p.track != nullptr && n_masked_b > 0;
  bool any_window = false;
  for (int i = 0; i < 8; ++i) any_window |= win_flags[i] != 0;
  const bool two_pass = do_track && any_window;
  // deterministic tracker: each tile's slot among the sequence's WINDOW tiles
  const int tile0 = (q0 - s_cu[b]) / kBM;
  int trk_n = 0;
  const int trk_slot0 = trk_rank(wbits, tile0, trk_n);
  const int trk_slot1 = trk_slot0 + (int)((wbits[tile0 >> 5] >> (tile0 & 31)) & 1u);
  const bool trk_det = p.trk_part != nullptr && wbits[kTrkWords] == 0u && trk_n <= FDL_TRK_SLOTS;
  if (p.trk_part && threadIdx.x == 0 && h == 0 && tile0 == 0) p.trk_nslots[b] = trk_det && do_track ? trk_n : 0;
  const int sA = two_pass ? n_tiles : 0;  // S products of pass A per group
  const int n_s = sA + n_tiles;          // S products per group = K tile loads

  if (warp == 0) {
    // ------------------------------------------------------------ K producer
    // K load lc = 0 .. n_s - 1: key tile lc (pass A), then again (pass B)
    if (lane == 0 && n_tiles > 0) {
      for (int lc = pre; lc < n_s; ++lc) {
        const int s = lc % kKS;
        if (!tc::mbar_wait(&k_empty[s], ((uint32_t)(lc / kKS) & 1u) ^ 1u, abort_flag)) break;
        load_kv(&tm_k, kring + s * KT_BYTES, lc >= sA ? lc - sA : lc, &k_full[s]);
      }
    }
    __syncwarp();
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ V producer
    if (lane == 0 && n_tiles > 0) {
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kVS;
        if (!tc::mbar_wait(&v_empty[s], ((uint32_t)(i / kVS) & 1u) ^ 1u, abort_flag)) break;
        load_kv(&tm_v, vring + s * VT_BYTES, i, &v_full[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // S products in order (key tile j, then group g), P V products in order
    // (tile jj, group g). A P V product goes first when ready; an S product
    // needs its K tile and the group's S buffer, whose previous scores were
    // consumed (pass A: read by the group; pass B / online: read as P by the
    // group's P V product). Neither kind waits for the other. The readiness
    // checks do not block (mbarrier.test_wait): a blocking try_wait would
    // suspend the thread on the one barrier it tests, however soon another
    // product's operands landed.
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t id_s = tc::idesc_bf16_f32(kBM, kBN);
      constexpr uint32_t id_pv = idesc_pv(kBM, kHD);
      // descriptors of the first query tile and ring stages: the address
      // field counts 16-byte units, so a stage's or step's descriptor is the
      // base plus its byte offset / 16
      const uint64_t dq0 = tc::desc_kmajor_sw128(tc::smem_addr(sq));
      const uint64_t dk0 = tc::desc_kmajor_sw128(tc::smem_addr(kring));
      const uint64_t dv0 = desc_mnmajor_sw128(tc::smem_addr(vring), VT_BYTES / 2);
      bool ok = tc::mbar_wait(q_full, 0, abort_flag);
      const int total_s = n_s * n_g, total_pv = n_tiles * n_g;
      int si = 0, pi = 0;
      long long t_last = clock64();
      while (ok && pi < total_pv) {
        bool progressed = false;
        {
          const int jj = pi / n_g, g = pi - jj * n_g;
          const int vs = jj % kVS;
          if (tc::mbar_test_wait(&p_full[g], (uint32_t)jj & 1u) &&
              tc::mbar_test_wait(&v_full[vs], (uint32_t)(jj / kVS) & 1u)) {
            tc::fence_after_sync();
            const uint32_t a_p = tmem + 256u + 128u * (uint32_t)g;  // P: 64 columns of bf16 pairs
            const uint32_t d_o = tmem + 128u * (uint32_t)g;
            const uint64_t bv = dv0 + (uint64_t)(vs * (VT_BYTES >> 4));
            // 16 keys per step: 8 TMEM columns of P, 16 rows (2048 bytes) of V
#pragma unroll
            for (int k = 0; k < kBN / 16; ++k)
              tc::mma_bf16_ts(d_o, a_p + 8u * (uint32_t)k, bv + (uint64_t)(k * 128), id_pv, (jj > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(&pv_done[g]);
            tc::mma_commit(&s_free_b[g]);
            if (g == n_g - 1) tc::mma_commit(&v_empty[vs]);
            ++pi;
            progressed = true;
          }
        }
        if (si < total_s) {
          const int j = si / n_g, g = si - j * n_g;
          const int ks = j % kKS;
          bool ready = tc::mbar_test_wait(&k_full[ks], (uint32_t)(j / kKS) & 1u);
          if (ready && j >= 1) {
            const int jp = j - 1;  // the group's previous product, in the same buffer
            ready = jp < sA ? tc::mbar_test_wait(&s_free_a[g], (uint32_t)jp & 1u)
                            : tc::mbar_test_wait(&s_free_b[g], (uint32_t)(jp - sA) & 1u);
          }
          if (ready) {
            tc::fence_after_sync();
            const uint32_t d_s = tmem + 256u + 128u * (uint32_t)g;
            const uint64_t bq = dq0 + (uint64_t)(g * (Q_BYTES >> 4)), bk = dk0 + (uint64_t)(ks * (KT_BYTES >> 4));
            // 16 head dims (32 bytes) per step; the second 64 dims are the
            // second half of each tile (Q_BYTES / 2 and KT_BYTES / 2 on)
#pragma unroll
            for (int k = 0; k < kHD / 16; ++k) {
              const uint64_t oq = (uint64_t)((k >> 2) * (Q_BYTES / 2) + (k & 3) * 32) >> 4;
              const uint64_t okk = (uint64_t)((k >> 2) * (KT_BYTES / 2) + (k & 3) * 32) >> 4;
              tc::mma_bf16_ss(d_s, bq + oq, bk + okk, id_s, k > 0 ? 1u : 0u);
            }
            tc::mma_commit(&s_full[g]);
            if (g == n_g - 1) tc::mma_commit(&k_empty[ks]);
            ++si;
            progressed = true;
          }
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
  }

  // ------------------------------------------------------------ softmax warps
  // Group g (warps 2-5, 6-9) owns query tile g; warp w owns TMEM lane
  // quadrant w % 4 (32 query rows).
  const int qd = warp & 3;
  const int g = (warp - 2) >> 2;
  const int row = qd * 32 + lane;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  float lse2 = -INFINITY, inv_l = 0.f;
  bool live = false;
  if (softmax_warp) {
    for (int j = t_local; j < m_search; j += 256) {
      const int s = p.search_pos[(size_t)b * p.search_ld + j];
      if (s >= 0 && s < kvl && (s >> 5) < p.bitmap_words) atomicOr(&bitmap[s >> 5], 1u << (s & 31));
    }
    tc::named_bar(3, 256);
  }
  if (softmax_warp && g < n_g) {
    const int kind = kinds[g * kBM + row];
    const uint32_t tm_og = tmem + 128u * (uint32_t)g;
    const uint32_t s_buf = tmem + 256u + 128u * (uint32_t)g + lane_off;  // this warp's lanes
    const float sc = p.scale_log2;

    // waits for the group's product j (warp-collective: the whole warp
    // proceeds or none of it)
    auto wait_s = [&](int j) -> bool {
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&s_full[g], (uint32_t)j & 1u, abort_flag));
      if (ok) tc::fence_after_sync();
      return ok;
    };
    // raw scores of half hf (keys c0 + 64 hf ..) into x, the keys this row
    // does not see set to -inf (the scale is applied inside each exponent's
    // FFMA); with_max also returns the raw max of the half. A plain row sees
    // every key below the sequence length, so most halves need no mask.
    auto load_half = [&](int c0, int hf, float (&x)[64], bool with_max) -> float {
      tc::tmem_ld_32x32b_x64(s_buf + 64u * (uint32_t)hf, x);
      const int cb = c0 + 64 * hf;
      if (!(kind >= 0 && kind < 2 && cb + 64 <= kvl)) {
        const uint32_t vm0 = vis_mask(kind, cb, kvl, m_search, bitmap, p.bitmap_words);
        const uint32_t vm1 = vis_mask(kind, cb + 32, kvl, m_search, bitmap, p.bitmap_words);
        if ((vm0 & vm1) != 0xffffffffu) {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            x[k] = ((vm0 >> k) & 1u) ? x[k] : -INFINITY;
            x[k + 32] = ((vm1 >> k) & 1u) ? x[k + 32] : -INFINITY;
          }
        }
      }
      if (!with_max) return -INFINITY;
      float t16[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) t16[k] = fmaxf(fmaxf(x[k], x[k + 16]), fmaxf(x[k + 32], x[k + 48]));
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) t16[k] = fmaxf(t16[k], t16[k + w]);
      return t16[0];
    };
    // x <- exp2(x * sc - m) in place (zeros when m is -inf); returns the sum
    auto exp_sum = [&](float (&x)[64], float m) -> float {
      if (m == -INFINITY) {
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = 0.f;
        return 0.f;
      }
      const float nm = -m;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int e = 0; e < 64; e += 4) {
        ffma2(x[e], x[e + 1], x[e], x[e + 1], sc, sc, nm, nm);
        ffma2(x[e + 2], x[e + 3], x[e + 2], x[e + 3], sc, sc, nm, nm);
        x[e] = ex2(x[e]);
        x[e + 1] = ex2(x[e + 1]);
        x[e + 2] = ex2(x[e + 2]);
        x[e + 3] = ex2(x[e + 3]);
        fadd2(s0, s1, s0, s1, x[e], x[e + 1]);
        fadd2(s2, s3, s2, s3, x[e + 2], x[e + 3]);
      }
      return (s0 + s1) + (s2 + s3);
    };
    // P of half hf as bf16 pairs (the lower key in the low half) into
    // columns 32 hf .. 32 hf + 31 of the group's S buffer: the A operand of
    // P V.
    auto store_p = [&](int hf, const float (&x)[64]) {
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        pk[e] = *reinterpret_cast<uint32_t*>(&h2);
      }
      tc::tmem_st_32x32b_x32_u(s_buf + 32u * (uint32_t)hf, pk);
    };
    // Eq. (2): this warp's column sums of P over its WINDOW rows (half hf)
    // into its slot of colw
    auto colsum = [&](int hf, float (&x)[64], bool rows_count) {
      if (!rows_count) {
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = 0.f;
      }
      warp_colsum32(*reinterpret_cast<float(*)[32]>(x), lane);
      warp_colsum32(*reinterpret_cast<float(*)[32]>(x + 32), lane);
      colw[(g * 4 + qd) * kBN + 64 * hf + lane] = x[0];
      colw[(g * 4 + qd) * kBN + 64 * hf + 32 + lane] = x[32];
    };

    float m_run = -INFINITY, l_run = 0.f;  // log2 domain: m in units of scaled scores
    // the running reference max of a row: set by its first visible key, and
    // moved only when a tile's max exceeds it by more than 2^kRescale, when
    // alpha rescales what has accumulated
    auto update_max = [&](float tmax_raw, float& alpha) -> bool {
      alpha = 1.f;
      if (tmax_raw == -INFINITY) return false;
      const float t = tmax_raw * sc;
      if (m_run == -INFINITY) {
        m_run = t;
        return false;
      }
      if (t > m_run + kRescale) {
        alpha = ex2(m_run - t);
        m_run = t;
        return true;
      }
      return false;
    };

    if (two_pass) {
      // ---- pass A: each row's log-sum-exp
      for (int j = 0; j < n_tiles; ++j) {
        const bool ok = wait_s(j);
        if (ok) {
          const int c0 = j * kBN;
          float x[64];
          // each half's max moves the reference on its own (each score read
          // once); a move at half 1 rescales half 0's sum
          float a0, a1;
          update_max(load_half(c0, 0, x, true), a0);
          float sum = exp_sum(x, m_run);
          const float mx1 = load_half(c0, 1, x, true);
          tc::fence_before_sync();  // the scores are read: the buffer may be refilled
          if (update_max(mx1, a1)) sum *= a1;
          sum += exp_sum(x, m_run);
          l_run = l_run * (a0 * a1) + sum;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s_free_a[g]);
      }
      lse2 = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    // ---- pass B (two_pass: P = exp(S - lse)) or the one online pass
    const float wscale = do_track ? 1.f / ((float)p.H * (float)n_masked_b) : 0.f;
    const bool track_row = two_pass && kind == FDL_KIND_WINDOW;
    const int t_g = t_local - 128 * g;  // 0..127 within the group
    for (int jj = 0; jj < n_tiles; ++jj) {
      // a wait that gives up (abort) skips the work but never the barriers
      const int c0 = jj * kBN;
      const bool ok = wait_s(sA + jj);
      if (ok) {
        float x[64];
        // Online: each half's max moves the running reference on its own (a
        // move beyond 2^kRescale is rare), so each score is read once; a
        // move at half 1 rescales half 0's P (already in TMEM) and sum.
        // Two-pass: P = exp(S - lse).
        float a0 = 1.f, a1 = 1.f;
        bool r0 = false, r1 = false;
        if (!two_pass) r0 = update_max(load_half(c0, 0, x, true), a0);
        else load_half(c0, 0, x, false);
        // half 0's P goes into columns 0..31, whose scores (half 0) are
        // already read; half 1's scores (columns 64..127) are read next and
        // its P goes into columns 32..63
        float sum = exp_sum(x, two_pass ? lse2 : m_run);
        store_p(0, x);
        if (two_pass) colsum(0, x, track_row);
        if (!two_pass) {
          r1 = update_max(load_half(c0, 1, x, true), a1);
          if (__any_sync(0xffffffffu, r1)) {
            tc::tmem_wait_st();  // half 0's P has landed
            float pw[32];
            tc::tmem_ld_32x32b_x32(s_buf, pw);
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              uint32_t w = __float_as_uint(pw[e]);
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
              __nv_bfloat162 h2 = __floats2bfloat162_rn(f.x * a1, f.y * a1);
              pk[e] = *reinterpret_cast<uint32_t*>(&h2);
            }
            tc::tmem_st_32x32b_x32_u(s_buf, pk);
            sum *= a1;
          }
        } else {
          load_half(c0, 1, x, false);
        }
        sum += exp_sum(x, two_pass ? lse2 : m_run);
        store_p(1, x);
        if (two_pass) colsum(1, x, track_row);
        if (__any_sync(0xffffffffu, r0 || r1)) {
          // O_g rows move to the new max (the group's previous P V product
          // finished before this tile's scores were computed, and this
          // tile's is issued only after P is complete)
          const float alpha = a0 * a1;
#pragma unroll 1
          for (int cc = 0; cc < kHD; cc += 32) {
            float o[32];
            tc::tmem_ld_32x32b_x32(tm_og + cc + lane_off, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tc::tmem_st_32x32b_x32(tm_og + cc + lane_off, o);
          }
        }
        tc::tmem_wait_st();
        l_run = l_run * (a0 * a1) + sum;
        // keys past the sequence end may hold anything: zero their V rows so
        // that 0 * V stays 0 (group 0's product of the tile runs first)
        if (g == 0 && c0 + kBN > nkeys &&
            tc::mbar_wait(&v_full[jj % kVS], (uint32_t)(jj / kVS) & 1u, abort_flag)) {
          uint8_t* vt = vring + (jj % kVS) * VT_BYTES;
          const int first = max(0, nkeys - c0);
          for (int e = lane; e < (kBN - first) * 16; e += 32) {
            const int r = first + e / 16, part = e % 16;
            if ((r & 3) != qd) continue;  // the group's four warps split the rows
            *reinterpret_cast<uint4*>(vt + (part >> 3) * (VT_BYTES / 2) + r * 128 + (part & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        tc::fence_before_sync();
      }
      __syncwarp();
      if (ok && lane == 0) tc::mbar_arrive(&p_full[g]);
      if (two_pass) {
        if (!ok) {
          colw[(g * 4 + qd) * kBN + lane] = 0.f;
          colw[(g * 4 + qd) * kBN + 32 + lane] = 0.f;
          colw[(g * 4 + qd) * kBN + 64 + lane] = 0.f;
          colw[(g * 4 + qd) * kBN + 96 + lane] = 0.f;
        }
        // the four warps' column sums added in a fixed order
        tc::named_bar(4 + g, 128);
        {
          const int c = c0 + t_g;
          const float v = ((colw[(g * 4 + 0) * kBN + t_g] + colw[(g * 4 + 1) * kBN + t_g]) +
                           colw[(g * 4 + 2) * kBN + t_g]) + colw[(g * 4 + 3) * kBN + t_g];
          if (c < kvl) {
            const int tg = tile0 + g;
            if (!trk_det) {
              if (v != 0.f) atomicAdd(p.track + (size_t)b * p.track_ld + c, v * wscale);
            } else if ((wbits[tg >> 5] >> (tg & 31)) & 1u) {
              trk_row(p.trk_part, b, g ? trk_slot1 : trk_slot0, h, p.H, p.trk_ld)[c] = v * wscale;
            }
          }
        }
        tc::named_bar(4 + g, 128);
      }
    }
    // the group's last P V product has finished before O is read
    if (n_tiles > 0) tc::mbar_wait(&pv_done[g], (uint32_t)(n_tiles - 1) & 1u, abort_flag);
    tc::fence_after_sync();
    if (!two_pass) {
      lse2 = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
      inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    } else {
      inv_l = 1.f;
    }
    live = n_tiles > 0 && lse2 != -INFINITY;
  }

  // ------------------------------------------------------------ output
  if (softmax_warp && g < n_g) {
    const int qlen = g ? qlen1 : qlen0;
    const bool store = row < qlen && !*abort_flag;
    if (p.lse && row < qlen) p.lse[(size_t)(q0 + g * kBM + row) * p.H + h] = lse2 * kLn2;
    __nv_bfloat16* orow = p.o + (size_t)(q0 + g * kBM + row) * p.d + h * kHD;
#pragma unroll 1
    for (int cc = 0; cc < kHD; cc += 32) {
      float a[32];
      tc::tmem_ld_32x32b_x32(tmem + 128u * (uint32_t)g + cc + lane_off, a);
      if (!store) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = live ? a[q * 8 + 2 * e] * inv_l : 0.f;
          const float x1 = live ? a[q * 8 + 2 * e + 1] * inv_l : 0.f;
          __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
          w[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(orow + cc + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) fdl::raise_error(p.err, FDL_DEVERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// Whether the pair kernel takes a call: one CTA per key range (no KV split)
// and sequences of two or more query tiles on average.
bool fdl_attn_pair_applies(int R, int B, int C) { return C == 1 && R >= 2 * kBM * B; }

cudaError_t fdl_launch_attn_pair(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                                 const int* block_table, int bt_stride, const int* cu_seqlens_q, const int* kv_len,
                                 int B, int R, const int* row_kind, const int* search_pos, int search_ld,
                                 const int* n_search, int max_search_tokens, void* o_out, float* lse_out, float* track,
                                 int track_ld, int* worklist_out) {
  const fdl_config& c = ctx->cfg;
  if (B > kMaxDecodeB) return cudaErrorInvalidValue;
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)attn_pair_kernel, ctx->device, SMEM_BYTES)) return e;
  const int n_slots = c.n_pages * c.page_size;
  CUtensorMap mq, mk, mv;
  if (!map2d(&mq, q, R, c.d_model, kBM) || !map2d(&mk, k_cache, n_slots, c.d_model, kSub) ||
      !map2d(&mv, v_cache, n_slots, c.d_model, kSub))
    return cudaErrorInvalidValue;
  PairParams p;
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
  // grid (head, pair): sequence b contributes ceil(ceil(rows_b / 128) / 2)
  // pairs, at most ceil(R / 256) + B over the batch
  const int items = (R + 2 * kBM - 1) / (2 * kBM) + B;
  if (items > 65535) return cudaErrorInvalidConfiguration;
  return fdl_launch_pdl(attn_pair_kernel, dim3((unsigned)c.n_heads, (unsigned)items), dim3(kThreads, 1, 1),
                        SMEM_BYTES, ctx->stream, 1, mq, mk, mv, p);
}
