// Dense GEMM on the 5th-generation tensor cores for the rest of the
// transformer block (W_o, the SwiGLU gate/up and down projections), with the
// plain epilogues those need: a bf16 store, or an fp32 add into the residual
// stream. This is the split-K form for row counts whose tiles do not fill
// several waves of the GPU (the persistent form in fdl_gemm_tc.cu takes the
// larger ones).
//
// The design is the fused projection's ("swap AB", tcgen05 with the
// accumulator in TMEM, a TMA ring of 64-wide k-blocks, warp 0 loading,
// warp 1 issuing the MMAs, warps 2-5 in the epilogue, split-K across CTAs
// with a fixed-order merge by the last CTA of each tile): a tile is 128
// output features on the TMEM lanes against up to BN rows on the columns,
// which fills the M = 128 datapath for the small row counts of a cached
// denoising step.
#include <cudaTypedefs.h>

#include "fdl_model.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 64 ? 4 : (BN == 128 ? 6 : 4);
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 + PIPE_BYTES + BAR_BYTES;
};

struct DenseParams {
  int R, N, nkb, ksplit;
  bool add_f32;
  void* out;          // [R, N]: fp32 (add) or bf16 (store)
  float* partials;    // [tiles * ksplit][BN][128] fp32 split-K partial tiles
  unsigned* tickets;  // [tiles] arrival counters, zero between launches
  unsigned* err;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, BN == 64 ? 2 : 1)
    dense_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                    const DenseParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* pipe = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::PIPE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tmem_full = bars + 2 * C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* is_last = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = p.ksplit;
  const int rank = blockIdx.x;  // split index along K
  const int tile_r = blockIdx.y, tile_f = blockIdx.z;
  const int tile_lin = tile_f * gridDim.y + tile_r;
  const int f0 = tile_f * kBM;
  const int kb0 = rank * p.nkb / ks, kb1 = (rank + 1) * p.nkb / ks;
  const int pre = min(kb1 - kb0, C::STAGES);

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
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort_flag)) break;
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
        if (!tc::mbar_wait(&full[s], ph, abort_flag)) break;
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
    }
    __syncwarp();
  } else {
    tc::mbar_wait(tmem_full, 0, abort_flag);
    tc::fence_after_sync();
  }

  const int q = warp & 3;       // TMEM lane quadrant of this warp
  const int t = q * 32 + lane;  // tile row = output feature f0 + t
  const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
  const bool epi = warp >= 2 && !*abort_flag;
  constexpr int CH = 16;  // columns per TMEM chunk

  // row r's feature f0 + t: consecutive threads write consecutive features
  auto emit = [&](int c0, const float (&v)[CH]) {
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int r = tile_r * BN + c0 + j;
      if (r < p.R) {
        const size_t at = (size_t)r * p.N + f0 + t;
        if (p.add_f32) {
          float* o = reinterpret_cast<float*>(p.out) + at;
          *o = *o + v[j];
        } else {
          reinterpret_cast<__nv_bfloat16*>(p.out)[at] = __float2bfloat16_rn(v[j]);
        }
      }
    }
  };

  if (epi) {
    if (ks == 1) {
      for (int c0 = 0; c0 < BN; c0 += CH) {
        float v[CH];
        tc::tmem_ld_32x32b_x16(t_lane + c0, v);
        emit(c0, v);
      }
    } else {
      // publish this split's partial tile, then take a ticket
      float* mine = p.partials + ((size_t)tile_lin * ks + rank) * BN * kBM;
      for (int c0 = 0; c0 < BN; c0 += CH) {
        float v[CH];
        tc::tmem_ld_32x32b_x16(t_lane + c0, v);
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
          __threadfence();           // acquire: the other splits' partials
        }
      }
      tc::named_bar(1, kEpiThreads);
      if (*is_last) {
        // the ks partials summed in split order, so results do not depend on timing
        const float* parts = p.partials + (size_t)tile_lin * ks * BN * kBM;
        const size_t split_stride = (size_t)BN * kBM;
        for (int c0 = 0; c0 < BN; c0 += CH) {
          float v[CH];
#pragma unroll
          for (int j = 0; j < CH; ++j) v[j] = __ldcg(parts + (c0 + j) * kBM + t);
          for (int sp = 1; sp < ks; ++sp) {
#pragma unroll
            for (int j = 0; j < CH; ++j) v[j] += __ldcg(parts + sp * split_stride + (c0 + j) * kBM + t);
          }
          emit(c0, v);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) fdl::raise_error(p.err, FDL_DEVERR_TIMEOUT);
  if (warp == 1) tc::tmem_dealloc(tmem, BN);
}

PFN_cuTensorMapEncodeTiled_v12000 dense_map_encoder() {
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

// bf16 row-major [rows, cols], box 64 columns x box_rows rows, 128-byte swizzle
bool dense_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = dense_map_encoder();
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
cudaError_t launch(fdl_ctx* ctx, DenseParams p, const void* X, const void* W, int K) {
  using Cf = Cfg<BN>;
  static_assert(Cf::SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static fdl_smem_limit smem_limit;
  if (cudaError_t e = smem_limit.ensure((const void*)dense_tc_kernel<BN>, ctx->device, Cf::SMEM_BYTES)) return e;
  CUtensorMap mw, mx;
  if (!dense_map(&mw, W, (uint64_t)p.N, (uint64_t)K, kBM) || !dense_map(&mx, X, (uint64_t)p.R, (uint64_t)K, BN))
    return cudaErrorInvalidValue;
  const int tiles_r = (p.R + BN - 1) / BN, tiles_f = p.N / kBM;
  const int tiles = tiles_r * tiles_f;
  const int per_sm = BN == 64 ? 2 : 1;
  int ks = 1;
  if (tiles < ctx->num_sms * per_sm) ks = (ctx->num_sms * per_sm) / tiles;
  ks = max(1, min(ks, min(p.nkb, 8)));
  if ((size_t)tiles * ks * BN * kBM > ctx->qkv_partial_floats || tiles > ctx->qkv_tickets) ks = 1;
  p.ksplit = ks;
  p.partials = ctx->qkv_partials;
  p.tickets = ctx->qkv_ticket_buf;
  return fdl_launch_pdl(dense_tc_kernel<BN>, dim3(ks, tiles_r, tiles_f), dim3(kThreads, 1, 1), Cf::SMEM_BYTES,
                        ctx->stream, 1, mw, mx, p);
}

}  // namespace

cudaError_t fdl_launch_dense_splitk(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N, void* out,
                                    bool add_f32) {
  if (R <= 0) return cudaSuccess;
  if (ctx->cfg.dtype != FDL_BF16 || N % kBM != 0 || K % kBK != 0 || K <= 0 || !ctx->qkv_partials)
    return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(out)) & 15)
    return cudaErrorMisalignedAddress;
  DenseParams p = {};
  p.R = R;
  p.N = N;
  p.nkb = K / kBK;
  p.add_f32 = add_f32;
  p.out = out;
  p.err = ctx->err_word;
  if (R <= 64) return launch<64>(ctx, p, X, W, K);
  if (R <= 128) return launch<128>(ctx, p, X, W, K);
  return launch<256>(ctx, p, X, W, K);
}
