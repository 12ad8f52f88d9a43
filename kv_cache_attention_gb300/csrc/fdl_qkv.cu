// Fused QKV projection + RoPE + KV-cache scatter: fp32 CUDA-core path.
//
// Paper digest "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding ...",
// section "Core method" (Flash-Cache: projection, RoPE and cache write fused
// so K/V go straight from on-chip storage into the preallocated cache) and
// "Method steps in detail", Algorithm 2 step 2 (only the refresh rows are
// projected).
//
// This translation unit holds the exact-fp32 variant used for fp32 contexts
// (the tensor-core tf32 path cannot meet a 1e-4 tolerance) and the launcher
// that routes bf16 contexts to the tcgen05 kernel. One warp produces one
// rotate-half pair (features i and i + head_dim/2 of one head) for one row,
// so RoPE needs no data exchange; the row's hidden vector is staged in
// shared memory and the two weight rows are read with coalesced loads.
#include "fdl_internal.cuh"

namespace {

constexpr int kWarps = 8;

struct QkvParams {
  const void* x;
  const void* w;
  int R, d, hd, H;
  const int* row_seq;
  const int* row_rope_pos;
  const int* row_cache_pos;
  const int* block_table;
  int bt_stride, page_size, n_pages;
  void* k_cache;
  void* v_cache;
  void* q_out;
  const float* rope_cos;
  const float* rope_sin;
  int rope_positions;
  unsigned* err;
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) qkv_simt_kernel(QkvParams p) {
  extern __shared__ float xs[];  // [d]
  const int r = blockIdx.x;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const T* x = reinterpret_cast<const T*>(p.x) + (size_t)r * p.d;
  for (int k = threadIdx.x; k < p.d; k += blockDim.x) xs[k] = fdl::io<T>::load(x + k);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = p.hd / 2;
  const int pairs_per_section = p.d / 2;
  const int pair = blockIdx.y * kWarps + warp;
  if (pair >= 3 * pairs_per_section) return;
  const int section = pair / pairs_per_section;  // 0 = q, 1 = k, 2 = v
  const int qidx = pair % pairs_per_section;
  const int h = qidx / half, i = qidx % half;
  const int f1 = section * p.d + h * p.hd + i, f2 = f1 + half;
  const T* w1 = reinterpret_cast<const T*>(p.w) + (size_t)f1 * p.d;
  const T* w2 = reinterpret_cast<const T*>(p.w) + (size_t)f2 * p.d;
  float a = 0.f, b = 0.f;
  for (int k = lane; k < p.d; k += 32) {
    a = fmaf(xs[k], fdl::io<T>::load(w1 + k), a);
    b = fmaf(xs[k], fdl::io<T>::load(w2 + k), b);
  }
  for (int off = 16; off; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
  if (lane != 0) return;
  const int pos = p.row_rope_pos[r];
  if (pos < 0 || pos >= p.rope_positions) {
    fdl::raise_error(p.err, FDL_DEVERR_INDEX);
    return;
  }
  if (section < 2) {
    const float c = p.rope_cos[(size_t)pos * half + i], s = p.rope_sin[(size_t)pos * half + i];
    const float ra = a * c - b * s, rb = a * s + b * c;
    a = ra;
    b = rb;
  }
  const int col = h * p.hd + i;
  if (section == 0) {
    T* q = reinterpret_cast<T*>(p.q_out) + (size_t)r * p.d;
    fdl::io<T>::store(q + col, a);
    fdl::io<T>::store(q + col + half, b);
    return;
  }
  const int c = p.row_cache_pos[r];
  if (c < 0) return;
  const int seq = p.row_seq[r];
  long long slot = fdl::cache_slot(p.block_table, p.bt_stride, p.page_size, p.n_pages, seq, c, p.err);
  if (slot < 0) return;
  T* dst = reinterpret_cast<T*>(section == 1 ? p.k_cache : p.v_cache) + slot * p.d;
  fdl::io<T>::store(dst + col, a);
  fdl::io<T>::store(dst + col + half, b);
}

}  // namespace

// tcgen05 path (fdl_qkv_tc.cu); returns cudaErrorNotSupported when the
// shape is outside what it handles.
cudaError_t fdl_launch_qkv_tc(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                              const int* row_rope_pos, const int* row_cache_pos, const int* block_table,
                              int bt_stride, void* k_cache, void* v_cache, void* q_out);

cudaError_t fdl_launch_qkv(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                           const int* row_rope_pos, const int* row_cache_pos,
                           const int* block_table, int bt_stride, void* k_cache, void* v_cache,
                           void* q_out) {
  const fdl_config& c = ctx->cfg;
  if (c.dtype == FDL_BF16) {
    cudaError_t e = fdl_launch_qkv_tc(ctx, X, W, R, row_seq, row_rope_pos, row_cache_pos, block_table,
                                      bt_stride, k_cache, v_cache, q_out);
    if (e != cudaErrorNotSupported) return e;
  }
  QkvParams p;
  p.x = X;
  p.w = W;
  p.R = R;
  p.d = c.d_model;
  p.hd = c.head_dim;
  p.H = c.n_heads;
  p.row_seq = row_seq;
  p.row_rope_pos = row_rope_pos;
  p.row_cache_pos = row_cache_pos;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.page_size = c.page_size;
  p.n_pages = c.n_pages;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.q_out = q_out;
  p.rope_cos = ctx->rope_cos;
  p.rope_sin = ctx->rope_sin;
  p.rope_positions = ctx->rope_positions;
  p.err = ctx->err_word;
  const int pairs = 3 * c.d_model / 2;
  const dim3 grid(R, (pairs + kWarps - 1) / kWarps), block(kWarps * 32);
  size_t smem = (size_t)c.d_model * sizeof(float);
  if (c.dtype == FDL_BF16) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(qkv_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return fdl_launch_pdl(qkv_simt_kernel<__nv_bfloat16>, grid, block, smem, ctx->stream, 1, p);
  }
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(qkv_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return fdl_launch_pdl(qkv_simt_kernel<float>, grid, block, smem, ctx->stream, 1, p);
}
