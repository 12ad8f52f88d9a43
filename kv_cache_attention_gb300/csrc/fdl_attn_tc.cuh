// Helpers shared by the two tensor-core attention kernels (fdl_attn_tc.cu,
// fdl_attn_pair.cu): operand descriptors for the P V product, the view
// visibility rule of the Flash-Verify mask, warp scans and column sums, the
// hardware exponential, and the tensor maps of Q and the K/V cache.
#pragma once

#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace {

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Instruction descriptor for O += P V: bf16 operands, fp32 D, A (P) K-major,
// B (V, stored keys x head_dim) MN-major.
__host__ __device__ constexpr uint32_t idesc_pv(int M, int N) {
  return tc::idesc_bf16_f32(M, N) | (1u << 16);
}

// MN-major operand in the 128-byte swizzle layout: 64-element (128 B) rows
// along MN, one row per K index; 8-row groups 1024 B apart (stride byte
// offset); the next 64-wide MN block lbo bytes further (leading byte offset).
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Visibility of key position c to a row of `kind` in a sequence with kvl
// base keys and m search tokens (is_search: c is a search position).
__device__ __forceinline__ bool visible(int kind, int c, int kvl, int m, bool is_search) {
  if (kind < 0) return false;
  if (kind < 2) return c < kvl;
  if (c < kvl) return !is_search;
  const int v = c - kvl;
  if (v >= 2 * m) return false;
  const int k = (kind - 2) >> 1;
  const bool mask_view = (kind - 2) & 1;
  if (v < m) return mask_view ? (v < k) : (v <= k);
  const int j = v - m;
  return mask_view ? (j >= k) : (j > k);
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += y;
  }
  return v;
}

// Hardware base-2 exponential (ex2.approx, relative error ~2^-22); ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two-wide fp32 arithmetic (one instruction for a pair, each element
// rounded as the scalar instruction would): d = a * b + c and d = a + b.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Visibility of keys cb .. cb+31 (cb a multiple of 32) to a row of `kind`,
// one bit per key. Plain rows only compare against the sequence length; view
// rows consult the search-position bitmap and the view-key rule.
__device__ __forceinline__ uint32_t vis_mask(int kind, int cb, int kvl, int m, const uint32_t* bm, int words) {
  if (kind < 0) return 0u;
  if (kind < 2) {
    const int n = kvl - cb;
    return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
  }
  const uint32_t srch = (cb < kvl && (cb >> 5) < words) ? bm[cb >> 5] : 0u;
  uint32_t mask = 0u;
#pragma unroll 4
  for (int k = 0; k < 32; ++k) mask |= (visible(kind, cb + k, kvl, m, (srch >> k) & 1u) ? 1u : 0u) << k;
  return mask;
}

// Reduce-scatter of 32 per-lane values over the warp: afterwards v[0] of
// lane l holds the warp's sum of column l.
__device__ __forceinline__ void warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int off = 16 >> step;
    const int half = 16 >> step;
    const bool hi = lane & off;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = hi ? v[k] : v[k + half];
      const float keep = hi ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

// ---------------------------------------------------------------------------
// Deterministic Eq. (2) tracker. A CTA whose query tile holds WINDOW rows
// stores its per-head column sums (already in a fixed order over its warps)
// into the context's partial buffer, at the slot of its tile among the
// sequence's tiles with WINDOW rows, and the first CTA of every sequence
// records how many slots the sequence has (0 when its WINDOW rows span more
// tiles than there are slots: those CTAs add with atomics instead). A
// separate kernel then adds, column by column, the slots' and heads'
// partials in a fixed order to the scores. Each (sequence, slot, head,
// column) has exactly one writer per call and every sum has a fixed order,
// so the scores do not depend on timing.
constexpr int kTrkWords = 16;  // bitmap of a sequence's 128-row tiles with WINDOW rows (<= 512 tiles)

// Rank of tile t among the set tiles of `bits`, and their count.
__device__ __forceinline__ int trk_rank(const uint32_t* bits, int t, int& n) {
  int below = 0;
  n = 0;
#pragma unroll
  for (int w = 0; w < kTrkWords; ++w) {
    const uint32_t x = bits[w];
    n += __popc(x);
    if (w < (t >> 5)) below += __popc(x);
    else if (w == (t >> 5)) below += __popc(x & ((1u << (t & 31)) - 1u));
  }
  return below;
}

// Row of partial sums of (sequence b, slot s, head h).
__device__ __forceinline__ float* trk_row(float* part, int b, int s, int h, int H, int ld) {
  return part + ((size_t)(b * FDL_TRK_SLOTS + s) * H + h) * ld;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

bool map2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
