// Persistent GEMM on the 5th-generation tensor cores (tcgen05, accumulators
// in TMEM, operands staged by TMA) for row counts whose 128 x 256 tiles fill
// four or more waves of the GPU, with two epilogues:
//
//   fused projection  Paper digest "Flash-dLLM: IO-Aware KV Caching and
//                     Parallel Decoding ...", section "Core method": the QKV
//                     projection, RoPE and the cache write are one kernel; K
//                     and V leave the chip only as rows of the preallocated
//                     cache, Q only as the attention input. "Method steps in
//                     detail", step 2: the rows are the per-step refresh set
//                     (a full refresh: every position of every sequence).
//   dense             out (+)= X W^T for the rest of the transformer block
//                     (W_o, the SwiGLU gate/up and down projections): a bf16
//                     store, or an fp32 add into the residual stream.
// Up to 64 rows take the weight-streaming kernels (fdl_gemm_stream.cu), the
// row counts between those and four waves of tiles the split-K kernels
// (fdl_qkv_tc.cu, fdl_dense_tc.cu); fdl_launch_qkv_tc and
// fdl_launch_dense_tc below choose.
//
// Orientation ("swap AB"): a tile is 128 output features on the TMEM lanes
// against 256 rows on the TMEM columns. A projection tile covers whole
// heads, so every RoPE pair (i, i + hd/2) is in one tile (exchanged through
// shared memory).
//
// Scheduling. The work is T tiles x nkb k-blocks of 64 ("units"). One CTA
// per SM (G CTAs; a kernel that allocates tensor memory is resident once per
// SM). The first floor(T/G) - 1 waves of tiles are taken whole, round-robin
// (tile c + i*G), consecutive tiles sharing a weight tile so it is read once
// from DRAM; the remaining tiles (between one and two waves' worth) are
// split stream-K: CTA c takes the contiguous unit range [c*U/G, (c+1)*U/G)
// of them, so no wave runs part-empty.
//
// Warp roles (192 threads): warp 0 issues TMA loads into one 4-stage ring
// that runs across tile boundaries, warp 1 owns TMEM and issues tcgen05.mma
// (one lane), warps 2-5 run the epilogue. Two TMEM accumulators: the
// epilogue of one segment (a tile, or a CTA's share of a tile) overlaps the
// products of the next.
//
// A tile split over CTAs c_a..c_b: every share publishes its fp32 partial
// (rotated: RoPE is linear) to the slot of its CTA and takes an atomic
// ticket; the last to arrive sums the shares in CTA order, so results do not
// depend on timing, and stores the tile. Distinct split tiles have distinct
// first CTAs, so the ticket is indexed by c_a and G tickets and 2G partial
// slots (a CTA's first and last share) suffice. Tickets are plain counters,
// never waited on, and the last arrival resets them. A CTA's last share
// that finds every other share already published skips publishing its own;
// on the last segment the other shares are gathered with bulk copies into
// the drained ring; a merge won on an earlier segment waits until then.
#include <cudaTypedefs.h>

#include "fdl_model.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kBM = 128;          // output features per tile
constexpr int kBK = 64;           // k-block: one 128-byte swizzled row of bf16
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kCH = 16;           // accumulator columns per epilogue chunk
constexpr int kXStride = kCH + 1; // fp32 exchange rows (conflict-free)
constexpr unsigned kBadShare = 0x10000u;  // ticket increment of a share that published nothing

template <int BN>
struct Cfg {
  static constexpr int NACC = 2;  // TMEM accumulators
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int XBUF_BYTES = kBM * kXStride * 4;  // RoPE exchange; bf16 staging aliases it
  static constexpr int META_BYTES = BN * 16;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 + PIPE_BYTES + XBUF_BYTES + META_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = NACC * BN;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "TMEM budget");
  static_assert(8 * (2 * STAGES + 6) + 32 <= BAR_BYTES, "barriers and flags fit");
};

struct SkParams {
  int R, nkb, tiles_r, T, T_dp, G;
  long long U_sk;           // units of the stream-K tiles: (T - T_dp) * nkb
  int N;                    // output features (dense: row stride of out)
  bool add_f32;             // dense: add into fp32 out, else store bf16
  void* out;
  // fused projection
  int d, hd;
  const int* row_seq;
  const int* row_rope_pos;
  const int* row_cache_pos;
  const int* block_table;
  int bt_stride, page_size, n_pages;
  __nv_bfloat16* q_out;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  const float* rope_cos;
  const float* rope_sin;
  int rope_positions;
  float* partials;          // [G][2][BN][128] fp32 shares of split tiles
  unsigned* tickets;        // [G] arrival counters, zero between launches
  unsigned* err;
  long long wait_budget;    // cycles of the main loop's mbarrier waits
};

// kCH accumulator columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, float (&v)[kCH]) {
  static_assert(kCH == 16, "one TMEM load of 16 columns");
  tc::tmem_ld_32x32b_x16(taddr, v);
}

__device__ __forceinline__ long long sk_begin(const SkParams& p, int c) { return p.U_sk * c / p.G; }

// CTA whose stream-K range holds unit u (the largest c with sk_begin(c) <= u)
__device__ __forceinline__ int sk_owner(const SkParams& p, long long u) {
  int c = (int)(((u + 1) * p.G - 1) / p.U_sk);
  c = max(0, min(c, p.G - 1));
  while (c + 1 < p.G && sk_begin(p, c + 1) <= u) ++c;
  while (c > 0 && sk_begin(p, c) > u) --c;
  return c;
}

// Segment j of CTA c: tile t and its k-blocks [kb_a, kb_b); false past the
// CTA's last segment.
__device__ __forceinline__ bool segment(const SkParams& p, int c, int j, int& t, int& kb_a, int& kb_b) {
  const int n_dp = p.T_dp / p.G;
  if (j < n_dp) {
    t = c + j * p.G;
    kb_a = 0;
    kb_b = p.nkb;
    return true;
  }
  const long long a = sk_begin(p, c), b = sk_begin(p, c + 1);
  const long long ts = a / p.nkb + (j - n_dp);
  if (ts * p.nkb >= b) return false;
  kb_a = (int)(max(a, ts * p.nkb) - ts * p.nkb);
  kb_b = (int)(min(b, (ts + 1) * p.nkb) - ts * p.nkb);
  t = p.T_dp + (int)ts;
  return true;
}

template <int BN, bool QKV>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_sk_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                   const SkParams p) {
  using C = Cfg<BN>;
  constexpr int NACC = C::NACC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pipe = smem;
  float* xbuf = reinterpret_cast<float*>(smem + C::PIPE_BYTES);
  int* col_pos = reinterpret_cast<int*>(smem + C::PIPE_BYTES + C::XBUF_BYTES);
  long long* col_dst = reinterpret_cast<long long*>(col_pos + BN);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::PIPE_BYTES + C::XBUF_BYTES + C::META_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* acc_full = bars + 2 * C::STAGES;  // [NACC]
  uint64_t* acc_empty = acc_full + 2;         // [NACC]
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* mrg_bar = mma_done + 1;           // bulk copies into the drained ring
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mrg_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_flag = abort_flag + 1;  // epilogue: segment ok / last share / merge here
  volatile int* s_zero = abort_flag + 2;  // a flag nothing raises (waits that ignore the abort)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  // Barriers, TMEM and the tensor-map prefetch touch no global memory, so
  // they overlap the end of the previous kernel in the stream.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      tc::mbar_init(&acc_full[a], 1);
      tc::mbar_init(&acc_empty[a], 4);  // one arrival per epilogue warp
    }
    tc::mbar_init(mma_done, 1);
    tc::mbar_init(mrg_bar, 1);
    *abort_flag = 0;
    *s_zero = 0;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w);
    tc::prefetch_tensormap(&tmap_x);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();

  // The producer walks (segment, k-block) in order; the first ring of loads
  // needs no free slot and is issued before the CTA barrier, so the weight
  // stream starts while the other warps are still setting up.
  int pj = 0, pt = 0, pkb = 0, pkb_b = 0, pit = 0;
  bool pvalid = false;
  auto issue = [&]() {
    const int s = pit % C::STAGES;
    const int f = pt / p.tiles_r, r = pt - f * p.tiles_r;
    uint8_t* a = pipe + s * C::STAGE_BYTES;
    tc::mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
    tc::tma_load_2d(a, &tmap_w, pkb * kBK, f * kBM, &full[s]);
    tc::tma_load_2d(a + C::A_BYTES, &tmap_x, pkb * kBK, r * BN, &full[s]);
    ++pit;
    if (++pkb >= pkb_b) pvalid = segment(p, cta, ++pj, pt, pkb, pkb_b);
  };
  // (With a shortened wait budget, for failure-path tests, the ring is filled
  // only after the barrier, so that no load lands before the first wait.)
  if (threadIdx.x == 0) {
    pvalid = segment(p, cta, 0, pt, pkb, pkb_b);
    if (p.wait_budget == tc::kWaitBudgetCycles)
      while (pvalid && pit < C::STAGES) issue();
  }
  // the MMA issuer's first segment, also found before the barrier
  int mt = 0, mkb_a = 0, mkb_b = 0;
  bool mvalid = false;
  if (warp == 1 && lane == 0) mvalid = segment(p, cta, 0, mt, mkb_a, mkb_b);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      while (pvalid) {
        const int s = pit % C::STAGES;
        if (pit >= C::STAGES &&
            !tc::mbar_wait(&empty[s], ((uint32_t)(pit / C::STAGES) & 1u) ^ 1u, abort_flag, p.wait_budget))
          break;
        issue();
      }
      if (*abort_flag) {
        // let loads already in flight land before this CTA's memory is reused
        for (int j = max(0, pit - C::STAGES); j < pit; ++j) {
          long long t0 = clock64();
          while (!tc::mbar_try_wait(&full[j % C::STAGES], (uint32_t)(j / C::STAGES) & 1u) &&
                 clock64() - t0 < tc::kWaitBudgetCycles / 8) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, BN);
      int it = 0, t = mt, kb_a = mkb_a, kb_b = mkb_b;
      bool ok = true;
      for (int j = 0; ok && (j == 0 ? mvalid : segment(p, cta, j, t, kb_a, kb_b)); ++j) {
        const int a = j % NACC;
        // the epilogue has read segment j - NACC out of this accumulator
        if (j >= NACC && !tc::mbar_wait(&acc_empty[a], (uint32_t)((j - NACC) / NACC) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(a * BN);
        for (int kb = kb_a; kb < kb_b; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (!tc::mbar_wait(&full[s], (uint32_t)(it / C::STAGES) & 1u, abort_flag, p.wait_budget)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_addr(pipe + s * C::STAGE_BYTES);
          const uint64_t ad = tc::desc_kmajor_sw128(sa);
          const uint64_t bd = tc::desc_kmajor_sw128(sa + C::A_BYTES);
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
    const int ft = q * 32 + lane;  // tile row = output feature f0 + ft
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    __nv_bfloat16* obuf = reinterpret_cast<__nv_bfloat16*>(xbuf);  // [kCH][128] bf16, aliases xbuf
    constexpr size_t kTileF = (size_t)BN * kBM;                    // floats of one fp32 tile
    float* stage = reinterpret_cast<float*>(pipe);                  // the drained ring
    const int half = p.hd / 2;
    // the tile in hand: first feature and row, section (projection: 0 = Q,
    // 1 = K, 2 = V; tiles never straddle) and this thread's RoPE pair
    int f0 = 0, row0 = 0, section = 0, jj = 0, partner = ft;
    bool low = false, rope_on = false;
    uint32_t mrg_phase = 0;

    // tile t's per-row destinations and RoPE positions (projection)
    auto setup_tile = [&](int t) {
      const int f = t / p.tiles_r, r = t - f * p.tiles_r;
      f0 = f * kBM;
      row0 = r * BN;
      tc::named_bar(1, kEpiThreads);  // earlier readers of col_pos / col_dst / xbuf are done
      if constexpr (QKV) {
        section = f0 / p.d;
        const int fi = (f0 + ft) % p.hd;
        jj = fi % half;
        low = fi < half;
        partner = ft ^ half;
        rope_on = section < 2;
        for (int c = ft; c < BN; c += kEpiThreads) {
          const int rr = row0 + c;
          int pos = -1;
          long long dst = -1;
          if (rr < p.R) {
            pos = p.row_rope_pos[rr];
            if (pos < 0 || pos >= p.rope_positions) {
              fdl::raise_error(p.err, FDL_DEVERR_INDEX);
              pos = -1;
            } else if (section == 0) {
              dst = (long long)rr * p.d + f0;
            } else {
              const int cp = p.row_cache_pos[rr];
              if (cp >= 0) {
                const long long slot = fdl::cache_slot(p.block_table, p.bt_stride, p.page_size, p.n_pages,
                                                       p.row_seq[rr], cp, p.err);
                if (slot >= 0) dst = slot * p.d + (f0 - section * p.d);
              }
            }
          }
          col_pos[c] = pos;
          col_dst[c] = pos >= 0 ? dst : -1;
        }
      }
      tc::named_bar(1, kEpiThreads);
    };
    // RoPE on columns c0 .. c0 + kCH - 1 of this thread's feature (Q and K
    // only): rope_load fetches the table entries (issued before the TMEM
    // load, so their latency overlaps it), rope_apply exchanges the pair
    // partner's values through xbuf. The exchange barriers run in every
    // warp alike, whatever the segment's outcome.
    auto rope_load = [&](int c0, float (&cs)[kCH], float (&sn)[kCH]) {
      if (rope_on) {
#pragma unroll
        for (int e = 0; e < kCH; ++e) {
          const int pos = max(col_pos[c0 + e], 0);
          cs[e] = __ldg(p.rope_cos + (size_t)pos * half + jj);
          sn[e] = __ldg(p.rope_sin + (size_t)pos * half + jj);
        }
      }
    };
    auto rope_apply = [&](float (&v)[kCH], const float (&cs)[kCH], const float (&sn)[kCH]) {
      if constexpr (QKV) {
        tc::named_bar(1, kEpiThreads);  // earlier readers of xbuf / obuf are done
        if (rope_on) {
#pragma unroll
          for (int e = 0; e < kCH; ++e) xbuf[ft * kXStride + e] = v[e];
          tc::named_bar(1, kEpiThreads);
#pragma unroll
          for (int e = 0; e < kCH; ++e) {
            const float other = xbuf[partner * kXStride + e];
            v[e] = low ? (v[e] * cs[e] - other * sn[e]) : (other * sn[e] + v[e] * cs[e]);
          }
          tc::named_bar(1, kEpiThreads);  // exchange reads done before xbuf is reused
        }
      }
    };
    // final values of columns c0 .. c0 + kCH - 1: the projection stages
    // them as bf16 and writes whole 256-byte row pieces; the dense GEMM
    // writes (or adds) one element per thread and column
    auto emit = [&](int c0, const float (&v)[kCH], bool store) {
      if constexpr (QKV) {
        __nv_bfloat16* out = section == 0 ? p.q_out : (section == 1 ? p.k_cache : p.v_cache);
#pragma unroll
        for (int e = 0; e < kCH; ++e) obuf[e * kBM + ft] = __float2bfloat16_rn(v[e]);
        tc::named_bar(1, kEpiThreads);
        if (store) {
          for (int id = ft; id < kCH * 16; id += kEpiThreads) {
            const int e = id >> 4, part = id & 15;
            const long long dst = col_dst[c0 + e];
            if (dst >= 0)
              *reinterpret_cast<int4*>(out + dst + part * 8) = *reinterpret_cast<const int4*>(obuf + e * kBM + part * 8);
          }
        }
      } else {
        if (!store) return;
#pragma unroll
        for (int e = 0; e < kCH; ++e) {
          const int rr = row0 + c0 + e;
          if (rr < p.R) {
            const size_t at = (size_t)rr * p.N + f0 + ft;
            if (p.add_f32) {
              float* o = reinterpret_cast<float*>(p.out) + at;
              *o = *o + v[e];
            } else {
              reinterpret_cast<__nv_bfloat16*>(p.out)[at] = __float2bfloat16_rn(v[e]);
            }
          }
        }
      }
    };
    // Gathers into the drained ring, with a few large bulk copies on
    // mrg_bar, the published partial tiles of shares ca..cb (this CTA's
    // skipped when own_acc), share k at stage + k * kTileF. The wait ignores
    // the abort flag: bulk copies from global memory always complete, and
    // none may land after the CTA has exited.
    auto stage_issue = [&](long long ts, int ca, int cb, bool own_acc, int n_in) {
      if (ft == 0) tc::mbar_arrive_expect_tx(mrg_bar, (uint32_t)((size_t)n_in * kTileF * 4));
      tc::named_bar(1, kEpiThreads);  // armed before any copy can complete
      constexpr uint32_t kPiece = 8192;
      constexpr int kPieces = (int)(kTileF * 4 / kPiece);
      for (int cc = ca, k = 0; k < n_in; ++cc) {
        if (own_acc && cc == cta) continue;
        const int slot = sk_begin(p, cc) >= ts * p.nkb ? 0 : 1;
        const float* src = p.partials + ((size_t)cc * 2 + slot) * kTileF;
        float* dst = stage + (size_t)k * kTileF;
        for (int i = ft; i < kPieces; i += kEpiThreads)
          tc::bulk_load(dst + (size_t)i * (kPiece / 4), src + (size_t)i * (kPiece / 4), kPiece, mrg_bar);
        ++k;
      }
    };
    auto stage_wait = [&]() {
      tc::mbar_wait(mrg_bar, mrg_phase, s_zero);
      mrg_phase ^= 1u;
    };
    // Sums the shares ca..cb of stream-K tile ts in CTA order and stores the
    // tile, so results do not depend on timing. The published shares are
    // already rotated. own_acc: this CTA's share is still raw in its TMEM
    // accumulator at acc and is rotated here (else it is read back from its
    // published partial like the others). staged: the ring has drained and
    // the partials fit, so they are gathered into it first, the copies
    // landing while this share is rotated.
    auto merge_tile = [&](long long ts, int ca, int cb, bool own_acc, uint32_t acc, bool staged) {
      const int n_in = cb - ca + 1 - (own_acc ? 1 : 0);
      if (staged) stage_issue(ts, ca, cb, own_acc, n_in);
      for (int c0 = 0; c0 < BN; c0 += kCH) {
        float v[kCH], own[kCH];
        if (own_acc) {
          float cs[kCH], sn[kCH];
          rope_load(c0, cs, sn);
          tmem_ld_chunk(acc + c0, own);  // uniform over the CTA
          rope_apply(own, cs, sn);
        }
        if (staged && c0 == 0) stage_wait();
        for (int cc = ca, k = 0; cc <= cb; ++cc) {
          float x[kCH];
          if (own_acc && cc == cta) {
#pragma unroll
            for (int e = 0; e < kCH; ++e) x[e] = own[e];
          } else if (staged) {
            const float* src = stage + (size_t)k * kTileF + (size_t)c0 * kBM + ft;
#pragma unroll
            for (int e = 0; e < kCH; ++e) x[e] = src[e * kBM];
            ++k;
          } else {
            const int slot = sk_begin(p, cc) >= ts * p.nkb ? 0 : 1;
            const float* src = p.partials + ((size_t)cc * 2 + slot) * kTileF + (size_t)c0 * kBM + ft;
#pragma unroll
            for (int e = 0; e < kCH; ++e) x[e] = __ldcg(src + e * kBM);
          }
#pragma unroll
          for (int e = 0; e < kCH; ++e) v[e] = cc == ca ? x[e] : v[e] + x[e];
        }
        if constexpr (QKV) tc::named_bar(1, kEpiThreads);  // earlier readers of obuf are done
        emit(c0, v, true);
      }
    };

    // a merge won by a share that is not the CTA's last waits until the
    // ring has drained (at most two; more are merged at once)
    long long def_ts[2] = {0, 0};
    int def_ca[2] = {0, 0}, def_cb[2] = {0, 0}, n_def = 0;
    int t = 0, kb_a = 0, kb_b = 0;
    for (int j = 0; segment(p, cta, j, t, kb_a, kb_b); ++j) {
      const int a = j % NACC;
      const bool whole = kb_a == 0 && kb_b == p.nkb;
      int tn, kn_a, kn_b;
      const bool last_seg = !segment(p, cta, j + 1, tn, kn_a, kn_b);
      setup_tile(t);
      tc::mbar_wait(&acc_full[a], (uint32_t)(j / NACC) & 1u, abort_flag);
      tc::named_bar(1, kEpiThreads);
      // one snapshot of the abort flag decides, for all four warps alike,
      // whether this segment's products are complete
      if (ft == 0) *s_flag = *abort_flag ? 0 : 1;
      tc::named_bar(1, kEpiThreads);
      const bool seg_ok = *s_flag != 0;
      tc::fence_after_sync();
      const uint32_t acc = t_lane + (uint32_t)(a * BN);

      if (whole) {
        for (int c0 = 0; c0 < BN; c0 += kCH) {
          float v[kCH], cs[kCH], sn[kCH];
          rope_load(c0, cs, sn);
          tmem_ld_chunk(acc + c0, v);  // warp-collective: every warp, whatever seg_ok says
          rope_apply(v, cs, sn);
          emit(c0, v, seg_ok);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acc_empty[a]);
        continue;
      }

      // ---- a share of a split tile
      const long long ts = t - p.T_dp;  // tile index among the stream-K tiles
      const int ca = sk_owner(p, ts * p.nkb), cb = sk_owner(p, (ts + 1) * p.nkb - 1);
      const unsigned expect = (unsigned)(cb - ca + 1);
      // The CTA's last share finds, more often than not, every other share
      // of its tile already published: it is then the last to arrive, so it
      // skips publishing its own partial and merges straight from TMEM.
      bool sure_last = false;
      if (last_seg && seg_ok) {
        if (ft == 0) *s_flag = tc::ld_acquire_gpu(p.tickets + ca) == expect - 1u ? 1 : 0;
        tc::named_bar(1, kEpiThreads);
        sure_last = *s_flag != 0;
        tc::named_bar(1, kEpiThreads);
      }
      bool merge_here = sure_last;
      if (sure_last) {
        if (ft == 0) p.tickets[ca] = 0u;  // every other share has arrived: reset for the next launch
      } else {
        // publish the partial, rotated (RoPE is linear, so the sum of the
        // rotated shares is the rotated sum), and take the ticket
        const int my_slot = sk_begin(p, cta) >= ts * p.nkb ? 0 : 1;
        float* mine = p.partials + ((size_t)cta * 2 + my_slot) * kTileF;
        for (int c0 = 0; c0 < BN; c0 += kCH) {
          float v[kCH], cs[kCH], sn[kCH];
          rope_load(c0, cs, sn);
          tmem_ld_chunk(acc + c0, v);
          rope_apply(v, cs, sn);
          if (seg_ok) {
#pragma unroll
            for (int e = 0; e < kCH; ++e) __stcg(mine + (c0 + e) * kBM + ft, v[e]);
          }
        }
        __threadfence();  // release: this share's partial, before the ticket
        tc::named_bar(1, kEpiThreads);
        if (ft == 0) {
          const unsigned add = seg_ok ? 1u : 1u + kBadShare;
          const unsigned now = atomicAdd(p.tickets + ca, add) + add;
          const bool last = (now & (kBadShare - 1u)) == expect;
          if (last) {
            p.tickets[ca] = 0u;  // every share has arrived: reset for the next launch
            __threadfence();     // acquire: the other shares' partials
          }
          *s_flag = last && (now >> 16) == 0u ? 1 : 0;  // no share gave up
        }
        tc::named_bar(1, kEpiThreads);
        merge_here = *s_flag != 0;
        if (merge_here && !last_seg && n_def < 2) {
          def_ts[n_def] = ts;
          def_ca[n_def] = ca;
          def_cb[n_def] = cb;
          ++n_def;
          merge_here = false;
        }
      }
      if (merge_here) merge_tile(ts, ca, cb, true, acc, last_seg && (size_t)(cb - ca) * kTileF * 4 <= (size_t)C::PIPE_BYTES);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[a]);  // this share's accumulator is read
    }
    // merges deferred until the ring drained (every share already published)
    for (int d = 0; d < n_def; ++d) {
      setup_tile((int)(p.T_dp + def_ts[d]));
      merge_tile(def_ts[d], def_ca[d], def_cb[d], false, 0,
                 (size_t)(def_cb[d] - def_ca[d] + 1) * kTileF * 4 <= (size_t)C::PIPE_BYTES);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) fdl::raise_error(p.err, FDL_DEVERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
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

// The schedule: G = min(SMs, units); whole round-robin waves while more
// than two waves of tiles remain, the rest stream-K.
void schedule(const fdl_ctx* ctx, SkParams& p, int BN, int n_out, int K) {
  p.nkb = K / kBK;
  p.tiles_r = (p.R + BN - 1) / BN;
  p.T = p.tiles_r * (n_out / kBM);
  const long long units = (long long)p.T * p.nkb;
  p.G = (int)(units < ctx->num_sms ? units : ctx->num_sms);
  p.T_dp = p.T >= 2 * p.G ? (p.T / p.G - 1) * p.G : 0;
  p.U_sk = (long long)(p.T - p.T_dp) * p.nkb;
}

constexpr int kPersistBN = 256;

template <bool QKV>
cudaError_t launch(fdl_ctx* ctx, SkParams p, const void* X, const void* W, int K, int n_out) {
  constexpr int BN = kPersistBN;
  using Cf = Cfg<BN>;
  auto kernel = gemm_sk_kernel<BN, QKV>;
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)kernel, ctx->device, Cf::SMEM_BYTES)) return e;
  CUtensorMap mw, mx;
  if (!make_map(&mw, W, (uint64_t)n_out, (uint64_t)K, kBM) || !make_map(&mx, X, (uint64_t)p.R, (uint64_t)K, BN))
    return cudaErrorInvalidValue;
  schedule(ctx, p, BN, n_out, K);
  if ((size_t)p.G * 2 * BN * kBM > ctx->qkv_partial_floats || p.G > ctx->qkv_tickets) return cudaErrorNotSupported;
  p.partials = ctx->qkv_partials;
  p.tickets = ctx->qkv_ticket_buf;
  p.err = ctx->err_word;
  p.wait_budget = ctx->wait_budget > 0 ? ctx->wait_budget : tc::kWaitBudgetCycles;
  return fdl_launch_pdl(kernel, dim3((unsigned)p.G), dim3(kThreads, 1, 1), Cf::SMEM_BYTES, ctx->stream, 1, mw, mx,
                        p);
}

// The persistent form pays once its 256-row tiles fill four waves: below
// that the split-K kernels' two short waves overlap one wave's split-K
// merges with the other's weight stream, and finish first (measured: 64
// rows 26.8 against 32.6 us, 768 rows 70.5 against 88.1 us; 2048 rows 178
// against 145 us).
// (It also needs two partial tiles per CTA of context workspace.)
bool persistent_pays(const fdl_ctx* ctx, int R, int n_out) {
  const long long tiles = (long long)((R + kPersistBN - 1) / kPersistBN) * (n_out / kBM);
  return tiles >= 4LL * ctx->num_sms && (size_t)ctx->num_sms * 2 * kPersistBN * kBM <= ctx->qkv_partial_floats &&
         ctx->num_sms <= ctx->qkv_tickets;
}

}  // namespace

cudaError_t fdl_launch_qkv_splitk(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                                  const int* row_rope_pos, const int* row_cache_pos, const int* block_table,
                                  int bt_stride, void* k_cache, void* v_cache, void* q_out);
cudaError_t fdl_launch_dense_splitk(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N, void* out,
                                    bool add_f32);
size_t fdl_qkv_splitk_partial_floats(int num_sms);

size_t fdl_qkv_partial_floats(int num_sms, int max_rows) {
  // the split-K kernels' partial tiles, or two shares per CTA of the
  // persistent form's 256-row tiles when the context's rows can reach it
  const size_t splitk = fdl_qkv_splitk_partial_floats(num_sms);
  const size_t persistent = max_rows > kPersistBN ? (size_t)2 * num_sms * kPersistBN * kBM : 0;
  return splitk > persistent ? splitk : persistent;
}

cudaError_t fdl_launch_qkv_tc(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                              const int* row_rope_pos, const int* row_cache_pos, const int* block_table,
                              int bt_stride, void* k_cache, void* v_cache, void* q_out) {
  const fdl_config& c = ctx->cfg;
  if (c.d_model % kBM != 0 || (c.head_dim != 64 && c.head_dim != 128) || !ctx->qkv_partials)
    return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(X) & 15) || (reinterpret_cast<uintptr_t>(W) & 15) ||
      (reinterpret_cast<uintptr_t>(q_out) & 15) || (reinterpret_cast<uintptr_t>(k_cache) & 15) ||
      (reinterpret_cast<uintptr_t>(v_cache) & 15))
    return cudaErrorNotSupported;
  if (R <= 0) return cudaSuccess;
  if (fdl_stream_gemm_applies(ctx, R, c.d_model, 3 * c.d_model))
    return fdl_launch_qkv_stream(ctx, X, W, R, row_seq, row_rope_pos, row_cache_pos, block_table, bt_stride,
                                 k_cache, v_cache, q_out);
  if (!persistent_pays(ctx, R, 3 * c.d_model))
    return fdl_launch_qkv_splitk(ctx, X, W, R, row_seq, row_rope_pos, row_cache_pos, block_table, bt_stride,
                                 k_cache, v_cache, q_out);
  SkParams p = {};
  p.R = R;
  p.N = 3 * c.d_model;
  p.d = c.d_model;
  p.hd = c.head_dim;
  p.row_seq = row_seq;
  p.row_rope_pos = row_rope_pos;
  p.row_cache_pos = row_cache_pos;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.page_size = c.page_size;
  p.n_pages = c.n_pages;
  p.q_out = reinterpret_cast<__nv_bfloat16*>(q_out);
  p.k_cache = reinterpret_cast<__nv_bfloat16*>(k_cache);
  p.v_cache = reinterpret_cast<__nv_bfloat16*>(v_cache);
  p.rope_cos = ctx->rope_cos;
  p.rope_sin = ctx->rope_sin;
  p.rope_positions = ctx->rope_positions;
  return launch<true>(ctx, p, X, W, c.d_model, 3 * c.d_model);
}

cudaError_t fdl_launch_dense_tc(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N, void* out,
                                bool add_f32) {
  if (R <= 0) return cudaSuccess;
  if (ctx->cfg.dtype != FDL_BF16 || N % kBM != 0 || K % kBK != 0 || K <= 0 || !ctx->qkv_partials)
    return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(out)) & 15)
    return cudaErrorMisalignedAddress;
  if (fdl_stream_gemm_applies(ctx, R, K, N)) return fdl_launch_dense_stream(ctx, X, W, R, K, N, out, add_f32);
  if (!persistent_pays(ctx, R, N)) return fdl_launch_dense_splitk(ctx, X, W, R, K, N, out, add_f32);
  SkParams p = {};
  p.R = R;
  p.N = N;
  p.add_f32 = add_f32;
  p.out = out;
  p.hd = 1;
  return launch<false>(ctx, p, X, W, K, N);
}
