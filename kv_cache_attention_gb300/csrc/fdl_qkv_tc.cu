// Fused QKV projection + RoPE + KV-cache scatter on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM, operands staged by TMA): the
// split-K form for row counts whose tiles do not fill several waves of the
// GPU (the persistent form in fdl_gemm_tc.cu takes the larger ones).
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...",
// section "Core method": the projection, RoPE and cache write are one kernel;
// K and V leave the chip only as rows of the preallocated cache, Q only as
// the attention input. "Method steps in detail", step 2: the rows are the
// per-step refresh set (masked window + tracked tokens).
//
// Orientation ("swap AB"): the MMA computes D = W_tile . X_tile^T with the
// 128 output features of a tile on the TMEM lanes and up to BN query rows
// on the TMEM columns, so a refresh set of 64 rows still fills the M = 128
// datapath. A tile is aligned to whole heads, so every RoPE pair (i, i +
// head_dim/2) lives in the same CTA (exchanged through shared memory).
//
// Warp roles (192 threads): warp 0 issues TMA loads into a STAGES-deep
// ring, warp 1 owns TMEM and issues tcgen05.mma (one elected lane), warps
// 2-5 run the epilogue (TMEM -> registers -> RoPE -> bf16 -> 16-byte stores).
// When the tiles cannot fill the GPU (the small refresh sets of the cache
// phase), K is split across ks CTAs that stay resident together (two per
// SM for 64-row tiles). Each writes its fp32 partial tile to a workspace
// slot; the last CTA of a tile to arrive (an atomic ticket it resets) sums
// the ks partials in split order, so results do not depend on timing, and
// runs the epilogue. The ticket is a plain counter, never waited on.
#include <cudaTypedefs.h>

#include "fdl_internal.cuh"
#include "tc_ptx.cuh"

int qkv_ctas_per_sm(int bn);

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kXStride = 33;  // fp32 exchange buffer row stride (conflict-free)

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 64 ? 4 : (BN == 128 ? 6 : 4);
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int XBUF_BYTES = kBM * kXStride * 4;  // aliases the drained ring
  static constexpr int META_BYTES = BN * 16;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 + PIPE_BYTES + META_BYTES + BAR_BYTES;
  static_assert(XBUF_BYTES <= PIPE_BYTES, "exchange buffer must fit in the ring");
};

struct TcParams {
  int R, d, hd, nkb, ksplit;
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
  float* partials;     // [tiles * ksplit][BN][128] fp32 split-K partial tiles
  unsigned* tickets;   // [tiles] arrival counters, zero between launches
  unsigned* err;
  long long wait_budget;  // cycles of the main loop's mbarrier waits
};

template <int BN>
__global__ void __launch_bounds__(kThreads, BN == 64 ? 2 : 1)
    qkv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                  const TcParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pipe = smem;
  float* xbuf = reinterpret_cast<float*>(pipe);  // used only after the ring has drained
  int* col_pos = reinterpret_cast<int*>(smem + C::PIPE_BYTES);
  long long* col_dst = reinterpret_cast<long long*>(col_pos + BN);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::PIPE_BYTES + C::META_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tmem_full = bars + 2 * C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* is_last = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = p.ksplit;
  const uint32_t rank = blockIdx.x;  // split index along K
  const int tile_r = blockIdx.y, tile_f = blockIdx.z;
  const int tile_lin = tile_f * gridDim.y + tile_r;
  const int f0 = tile_f * kBM;
  const int section = f0 / p.d;  // 0 = Q, 1 = K, 2 = V (tiles never straddle)
  const int kb0 = (int)(rank * p.nkb / ks), kb1 = (int)((rank + 1) * p.nkb / ks);

  const int pre = min(kb1 - kb0, C::STAGES);  // loads issued before the CTA barrier
  // Barriers, TMEM and the tensor-map prefetch touch no global memory, so
  // they overlap the end of the previous kernel in the stream.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(tmem_full, 1);
    *abort_flag = 0;
    *is_last = ks == 1;
    tc::fence_mbar_init();
    tc::prefetch_tensormap(&tmap_w);
    tc::prefetch_tensormap(&tmap_x);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, BN);
    tc::tmem_relinquish();
  }
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  if (threadIdx.x == 0) {
    // The first ring of loads needs no free slot: the producer (this thread)
    // issues it before the CTA barrier, so the weight stream starts while
    // the other warps are still setting up.
    for (int it = 0; it < pre; ++it) {
      uint8_t* a = pipe + it * C::STAGE_BYTES;
      tc::mbar_arrive_expect_tx(&full[it], C::STAGE_BYTES);
      tc::tma_load_2d(a, &tmap_w, (kb0 + it) * kBK, f0, &full[it]);
      tc::tma_load_2d(a + C::A_BYTES, &tmap_x, (kb0 + it) * kBK, tile_r * BN, &full[it]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int it = pre;
      for (int kb = kb0 + pre; kb < kb1; ++kb, ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.wait_budget)) break;
        uint8_t* a = pipe + s * C::STAGE_BYTES;
        tc::mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        tc::tma_load_2d(a, &tmap_w, kb * kBK, f0, &full[s]);
        tc::tma_load_2d(a + C::A_BYTES, &tmap_x, kb * kBK, tile_r * BN, &full[s]);
      }
      if (*abort_flag) {
        // let loads already in flight land before this CTA's memory is reused
        for (int j = max(0, it - C::STAGES); j < it; ++j) {
          long long t0 = clock64();
          while (!tc::mbar_try_wait(&full[j % C::STAGES], (uint32_t)(j / C::STAGES) & 1u) &&
                 clock64() - t0 < tc::kWaitBudgetCycles / 8) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, BN);
      int it = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        if (!tc::mbar_wait(&full[s], ph, abort_flag, p.wait_budget)) break;
        tc::fence_after_sync();
        const uint32_t a = tc::smem_addr(pipe + s * C::STAGE_BYTES);
        const uint64_t ad = tc::desc_kmajor_sw128(a);
        const uint64_t bd = tc::desc_kmajor_sw128(a + C::A_BYTES);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc::mma_bf16_ss(tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(tmem_full);
      // every product issued has finished before the CTA barrier below, also
      // when the loop above gave up (the TMEM is freed after that barrier)
      long long t0 = clock64();
      while (!tc::mbar_try_wait(tmem_full, 0) && clock64() - t0 < tc::kWaitBudgetCycles) {
      }
    }
    __syncwarp();
  } else {
    // per-column (query row) destination and RoPE position, computed while
    // the main loop streams (only the epilogue warps read them)
    for (int c = threadIdx.x - 64; c < BN; c += kEpiThreads) {
      const int r = tile_r * BN + c;
      int pos = -1;
      long long dst = -1;
      if (r < p.R) {
        pos = p.row_rope_pos[r];
        if (pos < 0 || pos >= p.rope_positions) {
          fdl::raise_error(p.err, FDL_DEVERR_INDEX);
          pos = -1;
        } else if (section == 0) {
          dst = (long long)r * p.d + f0;
        } else {
          const int cp = p.row_cache_pos[r];
          if (cp >= 0) {
            long long slot = fdl::cache_slot(p.block_table, p.bt_stride, p.page_size, p.n_pages, p.row_seq[r], cp,
                                             p.err);
            if (slot >= 0) dst = slot * p.d + (f0 - section * p.d);
          }
        }
      }
      col_pos[c] = pos;
      col_dst[c] = pos >= 0 ? dst : -1;
    }
  }
  // After this barrier every load has landed (or been drained), every
  // product has finished and no thread waits on a barrier again, so the
  // abort flag is final and every thread reads the same value.
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool ok = !*abort_flag;

  const int q = warp & 3;          // TMEM lane quadrant of this warp
  const int t = q * 32 + lane;     // tile row = output feature f0 + t
  const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);

  if (warp >= 2) {
    const int half = p.hd / 2;
    const int i = (f0 + t) % p.hd;
    const int jj = i % half;
    const bool low = i < half;
    const int partner = t ^ half;
    __nv_bfloat16* out = section == 0 ? p.q_out : (section == 1 ? p.k_cache : p.v_cache);
    __nv_bfloat16* obuf = reinterpret_cast<__nv_bfloat16*>(xbuf);  // [32][128] bf16, aliases xbuf
    constexpr int CH = 16;  // columns per TMEM chunk

    // Columns c0..c0+CH-1 of this thread's output feature from TMEM, with
    // RoPE applied (each pair's partner is exchanged through shared memory).
    // RoPE is linear, so a K split may rotate its own partial sum.
    auto load_rotated = [&](int c0, float (&v)[CH]) {
      float cs[CH], sn[CH];
      if (section < 2) {
        // table loads first, so their latency overlaps the TMEM load
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int pos = max(col_pos[c0 + j], 0);
          cs[j] = __ldg(p.rope_cos + (size_t)pos * half + jj);
          sn[j] = __ldg(p.rope_sin + (size_t)pos * half + jj);
        }
      }
      tc::tmem_ld_32x32b_x16(t_lane + c0, v);
      tc::named_bar(1, kEpiThreads);  // earlier readers of xbuf / obuf are done
      if (section < 2) {
#pragma unroll
        for (int j = 0; j < CH; ++j) xbuf[t * kXStride + j] = v[j];
        tc::named_bar(1, kEpiThreads);
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const float other = xbuf[partner * kXStride + j];
          v[j] = low ? (v[j] * cs[j] - other * sn[j]) : (other * sn[j] + v[j] * cs[j]);
        }
        tc::named_bar(1, kEpiThreads);  // exchange reads done before xbuf is reused
      }
    };
    // nrows query rows x 256 bytes from obuf: 16-byte chunks, consecutive
    // threads on consecutive chunks
    auto store_rows = [&](int c0, int nrows) {
      for (int id = t; id < nrows * 16; id += kEpiThreads) {
        const int j = id >> 4, part = id & 15;
        const long long dst = col_dst[c0 + j];
        if (dst >= 0)
          *reinterpret_cast<int4*>(out + dst + part * 8) = *reinterpret_cast<const int4*>(obuf + j * kBM + part * 8);
      }
    };

    if (ks == 1) {
      for (int c0 = 0; ok && c0 < BN; c0 += CH) {
        float v[CH];
        load_rotated(c0, v);
#pragma unroll
        for (int j = 0; j < CH; ++j) obuf[j * kBM + t] = __float2bfloat16_rn(v[j]);
        tc::named_bar(1, kEpiThreads);
        store_rows(c0, CH);
      }
    } else {
      // publish this split's rotated partial tile, then take a ticket (a
      // split that gave up publishes nothing but still takes its ticket, so
      // the counter is back at zero for the next launch)
      float* mine = p.partials + ((size_t)tile_lin * ks + rank) * BN * kBM;
      for (int c0 = 0; ok && c0 < BN; c0 += CH) {
        float v[CH];
        load_rotated(c0, v);
#pragma unroll
        for (int j = 0; j < CH; ++j) __stcg(mine + (c0 + j) * kBM + t, v[j]);
      }
      __threadfence();
      tc::named_bar(1, kEpiThreads);
      if (t == 0) {
        const unsigned prev = atomicAdd(p.tickets + tile_lin, 1u);
        *is_last = prev == (unsigned)(ks - 1);
        if (*is_last) {
          p.tickets[tile_lin] = 0u;  // every split has arrived: reset for the next launch
          __threadfence();           // acquire: the other splits' partials, for every thread after the barrier
        }
      }
      tc::named_bar(1, kEpiThreads);
      if (*is_last && ok) {
        // sum the ks rotated partials in split order (all loads of a chunk
        // in flight together), round to bf16 and store
        const float* parts = p.partials + (size_t)tile_lin * ks * BN * kBM;
        constexpr int CHM = 32;
        const size_t split_stride = (size_t)BN * kBM;
        for (int c0 = 0; c0 < BN; c0 += CHM) {
          float a0[CHM], a1[CHM], a2[CHM];
#pragma unroll
          for (int j = 0; j < CHM; ++j) a0[j] = __ldcg(parts + (c0 + j) * kBM + t);
#pragma unroll
          for (int j = 0; j < CHM; ++j) a1[j] = __ldcg(parts + split_stride + (c0 + j) * kBM + t);
#pragma unroll
          for (int j = 0; j < CHM; ++j) a2[j] = ks > 2 ? __ldcg(parts + 2 * split_stride + (c0 + j) * kBM + t) : 0.f;
#pragma unroll
          for (int j = 0; j < CHM; ++j) a0[j] = (a0[j] + a1[j]) + a2[j];
          for (int sp = 3; sp < ks; ++sp) {
#pragma unroll
            for (int j = 0; j < CHM; ++j) a0[j] += __ldcg(parts + sp * split_stride + (c0 + j) * kBM + t);
          }
          tc::named_bar(1, kEpiThreads);  // earlier readers of xbuf / obuf are done
#pragma unroll
          for (int j = 0; j < CHM; ++j) obuf[j * kBM + t] = __float2bfloat16_rn(a0[j]);
          tc::named_bar(1, kEpiThreads);
          store_rows(c0, CHM);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) fdl::raise_error(p.err, FDL_DEVERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, BN);
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

template <int BN>
cudaError_t launch(fdl_ctx* ctx, const TcParams& p0, const void* X, const void* W) {
  static_assert(Cfg<BN>::SMEM_BYTES <= 227 * 1024, "shared memory budget");
  using Cf = Cfg<BN>;
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)qkv_tc_kernel<BN>, ctx->device, Cf::SMEM_BYTES)) return e;
  const fdl_config& c = ctx->cfg;
  CUtensorMap mw, mx;
  if (!make_map(&mw, W, (uint64_t)3 * c.d_model, c.d_model, kBM) || !make_map(&mx, X, p0.R, c.d_model, BN))
    return cudaErrorInvalidValue;
  TcParams p = p0;
  const int tiles_r = (p.R + BN - 1) / BN, tiles_f = 3 * c.d_model / kBM;
  const int tiles = tiles_r * tiles_f;
  const int per_sm = qkv_ctas_per_sm(BN);
  int ks = 1;
  if (tiles < ctx->num_sms * per_sm) ks = (ctx->num_sms * per_sm) / tiles;
  ks = max(1, min(ks, min(p.nkb, 8)));
  if ((size_t)tiles * ks * BN * kBM > ctx->qkv_partial_floats || tiles > ctx->qkv_tickets) ks = 1;
  p.ksplit = ks;
  p.partials = ctx->qkv_partials;
  p.tickets = ctx->qkv_ticket_buf;
  return fdl_launch_pdl(qkv_tc_kernel<BN>, dim3(ks, tiles_r, tiles_f), dim3(kThreads, 1, 1), Cf::SMEM_BYTES,
                        ctx->stream, 1, mw, mx, p);
}

}  // namespace

int qkv_ctas_per_sm(int bn) { return bn == 64 ? 2 : 1; }

size_t fdl_qkv_splitk_partial_floats(int num_sms) {
  // split-K is used only while tiles * ks <= resident CTAs
  size_t a = (size_t)2 * num_sms * 64 * kBM, b = (size_t)num_sms * 256 * kBM;
  return a > b ? a : b;
}

cudaError_t fdl_launch_qkv_splitk(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                              const int* row_rope_pos, const int* row_cache_pos, const int* block_table,
                              int bt_stride, void* k_cache, void* v_cache, void* q_out) {
  const fdl_config& c = ctx->cfg;
  if (c.d_model % kBM != 0 || (c.head_dim != 64 && c.head_dim != 128)) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(X) & 15) || (reinterpret_cast<uintptr_t>(W) & 15) ||
      (reinterpret_cast<uintptr_t>(q_out) & 15) || (reinterpret_cast<uintptr_t>(k_cache) & 15) ||
      (reinterpret_cast<uintptr_t>(v_cache) & 15))
    return cudaErrorNotSupported;
  TcParams p;
  p.R = R;
  p.d = c.d_model;
  p.hd = c.head_dim;
  p.nkb = c.d_model / kBK;
  p.ksplit = 1;
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
  p.err = ctx->err_word;
  p.wait_budget = ctx->wait_budget > 0 ? ctx->wait_budget : tc::kWaitBudgetCycles;
  if (R <= 64) return launch<64>(ctx, p, X, W);
  if (R <= 128) return launch<128>(ctx, p, X, W);
  return launch<256>(ctx, p, X, W);
}
