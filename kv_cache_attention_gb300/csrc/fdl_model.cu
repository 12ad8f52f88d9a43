// The whole masked-diffusion transformer forward over one step's refresh
// rows: embedding, then per layer RMSNorm -> fused QKV + RoPE + cache write
// -> scheduled attention (with the Eq. (2) tracker) -> W_o into the
// residual stream -> RMSNorm -> SwiGLU FFN into the residual stream, then
// the final RMSNorm. Paper digest, "Background" (dLLMs are bidirectional
// transformers such as LLaDA) and "Method steps in detail", Algorithm 2
// step 2 (each step's query rows go through the layers against the full
// cache). The block is LLaMA-style (LLaDA's): pre-norm RMSNorm, no biases,
// a SwiGLU FFN; the pages are silent on these internals.
//
// The residual stream stays fp32 in the caller's workspace; every matrix
// operand is bf16. Attention and the projection run through the library's
// own entry points; W_o and the FFN through the dense tensor-core GEMM.
#include <stdarg.h>
#include <stdio.h>

#include "fdl_model.cuh"

namespace {

constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) embed_kernel(const int* __restrict__ tokens, int vocab,
                                                            const __nv_bfloat16* __restrict__ embed, int d,
                                                            float* __restrict__ h, unsigned* err) {
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int r = blockIdx.x;
  const int tok = tokens[r];
  const bool ok = tok >= 0 && tok < vocab;
  if (!ok && threadIdx.x == 0) fdl::raise_error(err, FDL_DEVERR_INDEX);
  const __nv_bfloat16* src = embed + (size_t)(ok ? tok : 0) * d;
  float* dst = h + (size_t)r * d;
  for (int i = threadIdx.x; i < d; i += kRowThreads) dst[i] = ok ? __bfloat162float(src[i]) : 0.f;
}

// One CTA per row, four consecutive elements per thread and load (d is a
// multiple of 128), the loads of a thread issued together. The sum of squares
// is reduced in a fixed order (each thread's elements in order, a fixed xor
// tree per warp, the warps' sums in warp order), so the result does not
// depend on timing.
__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const float* __restrict__ h, int d,
                                                              const __nv_bfloat16* __restrict__ g, float eps,
                                                              __nv_bfloat16* __restrict__ out) {
  __shared__ float warp_sum[kRowThreads / 32];
  __shared__ float scale;
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int r = blockIdx.x;
  const float4* x = reinterpret_cast<const float4*>(h + (size_t)r * d);
  const int n4 = d / 4;
  float ss = 0.f;
#pragma unroll 4
  for (int i = threadIdx.x; i < n4; i += kRowThreads) {
    const float4 v = x[i];
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kRowThreads / 32; ++w) t += warp_sum[w];
    scale = rsqrtf(t / (float)d + eps);
  }
  __syncthreads();
  const float s = scale;
  const uint2* g4 = reinterpret_cast<const uint2*>(g);
  uint2* y = reinterpret_cast<uint2*>(out + (size_t)r * d);
#pragma unroll 4
  for (int i = threadIdx.x; i < n4; i += kRowThreads) {
    const float4 v = x[i];
    const uint2 gw = g4[i];
    const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&gw.x);
    const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&gw.y);
    const __nv_bfloat162 y01 = __floats2bfloat162_rn(v.x * s * __low2float(g01), v.y * s * __high2float(g01));
    const __nv_bfloat162 y23 = __floats2bfloat162_rn(v.z * s * __low2float(g23), v.w * s * __high2float(g23));
    uint2 o;
    o.x = *reinterpret_cast<const unsigned*>(&y01);
    o.y = *reinterpret_cast<const unsigned*>(&y23);
    y[i] = o;
  }
}

// Grid (rows, chunks of kRowThreads * 8 elements): each thread takes eight
// consecutive gate and up elements with one 16-byte load each (F is a
// multiple of 64).
__global__ void __launch_bounds__(kRowThreads) swiglu_kernel(const __nv_bfloat16* __restrict__ gu, int F,
                                                             __nv_bfloat16* __restrict__ u) {
  fdl::grid_dep_wait();
  fdl::grid_dep_launch();
  const int r = blockIdx.x;
  const int i8 = blockIdx.y * kRowThreads + threadIdx.x;  // index of an 8-element group
  if (i8 * 8 >= F) return;
  const uint4 gw = reinterpret_cast<const uint4*>(gu + (size_t)r * 2 * F)[i8];
  const uint4 uw = reinterpret_cast<const uint4*>(gu + (size_t)r * 2 * F + F)[i8];
  const __nv_bfloat162* ga = reinterpret_cast<const __nv_bfloat162*>(&gw);
  const __nv_bfloat162* ua = reinterpret_cast<const __nv_bfloat162*>(&uw);
  uint4 ow;
  __nv_bfloat162* oa = reinterpret_cast<__nv_bfloat162*>(&ow);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float a0 = __low2float(ga[k]), a1 = __high2float(ga[k]);
    const float s0 = a0 / (1.f + expf(-a0)), s1 = a1 / (1.f + expf(-a1));
    oa[k] = __floats2bfloat162_rn(s0 * __low2float(ua[k]), s1 * __high2float(ua[k]));
  }
  reinterpret_cast<uint4*>(u + (size_t)r * F)[i8] = ow;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace regions, in order: h fp32 [R, d]; normed rows bf16 [R, d]; Q bf16
// [R, d]; attention output bf16 [R, d]; gate/up bf16 [R, 2F]; SwiGLU bf16 [R, F].
struct Workspace {
  float* h;
  __nv_bfloat16 *xn, *q, *o, *gu, *u;
  size_t bytes;
};

Workspace carve(void* base, int R, int d, int F) {
  Workspace w{};
  size_t off = 0;
  char* b = reinterpret_cast<char*>(base);
  auto take = [&](size_t n) {
    char* p = b ? b + off : nullptr;
    off += align256(n);
    return p;
  };
  w.h = reinterpret_cast<float*>(take((size_t)R * d * 4));
  w.xn = reinterpret_cast<__nv_bfloat16*>(take((size_t)R * d * 2));
  w.q = reinterpret_cast<__nv_bfloat16*>(take((size_t)R * d * 2));
  w.o = reinterpret_cast<__nv_bfloat16*>(take((size_t)R * d * 2));
  w.gu = reinterpret_cast<__nv_bfloat16*>(take((size_t)R * 2 * F * 2));
  w.u = reinterpret_cast<__nv_bfloat16*>(take((size_t)R * F * 2));
  w.bytes = off;
  return w;
}

fdl_status model_fail(fdl_ctx* ctx, fdl_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(ctx->last_error, sizeof(ctx->last_error), fmt, ap);
  va_end(ap);
  return st;
}

}  // namespace

cudaError_t fdl_launch_embed(fdl_ctx* ctx, const int* tokens, int R, const void* embed, float* h) {
  if (R <= 0) return cudaSuccess;
  return fdl_launch_pdl(embed_kernel, dim3(R), dim3(kRowThreads), 0, ctx->stream, 1, tokens, ctx->cfg.vocab,
                        reinterpret_cast<const __nv_bfloat16*>(embed), ctx->cfg.d_model, h, ctx->err_word);
}

cudaError_t fdl_launch_rmsnorm(fdl_ctx* ctx, const float* h, int R, const void* g, float eps, void* out) {
  if (R <= 0) return cudaSuccess;
  if (ctx->cfg.d_model % 4 != 0 ||
      ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(out)) & 15) || (reinterpret_cast<uintptr_t>(g) & 7))
    return cudaErrorMisalignedAddress;
  return fdl_launch_pdl(rmsnorm_kernel, dim3(R), dim3(kRowThreads), 0, ctx->stream, 1, h, ctx->cfg.d_model,
                        reinterpret_cast<const __nv_bfloat16*>(g), eps, reinterpret_cast<__nv_bfloat16*>(out));
}

cudaError_t fdl_launch_swiglu(fdl_ctx* ctx, const void* gu, int R, int F, void* u) {
  if (R <= 0) return cudaSuccess;
  if (F % 8 != 0 || ((reinterpret_cast<uintptr_t>(gu) | reinterpret_cast<uintptr_t>(u)) & 15))
    return cudaErrorMisalignedAddress;
  const int chunks = (F / 8 + kRowThreads - 1) / kRowThreads;
  return fdl_launch_pdl(swiglu_kernel, dim3(R, chunks), dim3(kRowThreads), 0, ctx->stream, 1,
                        reinterpret_cast<const __nv_bfloat16*>(gu), F, reinterpret_cast<__nv_bfloat16*>(u));
}

extern "C" size_t fdl_model_workspace_bytes(const fdl_ctx* ctx, int ffn, int R) {
  if (!ctx || ffn <= 0 || R < 0) return 0;
  return carve(nullptr, R, ctx->cfg.d_model, ffn).bytes;
}

extern "C" fdl_status fdl_model_forward(fdl_ctx* ctx, const fdl_model* m, const int* tokens, int R,
                                        const int* row_seq, const int* row_rope_pos, const int* row_cache_pos,
                                        const int* row_kind, const int* cu_seqlens_q, const int* kv_len, int B,
                                        const int* block_table, int bt_stride, void* const* k_caches,
                                        void* const* v_caches, const int* search_pos, int search_ld,
                                        const int* n_search, float* track_scores, int track_ld, void* workspace,
                                        size_t workspace_bytes, void* final_out) {
  if (!ctx) return FDL_ERR_INVALID_ARG;
  if (!m || !tokens || !workspace || !final_out || !k_caches || !v_caches || !m->embed || !m->g_final ||
      !m->g_attn || !m->w_qkv || !m->w_o || !m->g_mlp || !m->w_gu || !m->w_down)
    return model_fail(ctx, FDL_ERR_INVALID_ARG, "fdl_model_forward: NULL argument");
  const fdl_config& c = ctx->cfg;
  if (c.dtype != FDL_BF16) return model_fail(ctx, FDL_ERR_UNSUPPORTED, "fdl_model_forward: bf16 contexts only");
  if (m->n_layers < 1) return model_fail(ctx, FDL_ERR_INVALID_ARG, "n_layers=%d < 1", m->n_layers);
  if (m->ffn < 64 || m->ffn % 64 != 0 || c.d_model % 128 != 0)
    return model_fail(ctx, FDL_ERR_UNSUPPORTED, "ffn=%d must be a multiple of 64 and d_model=%d of 128", m->ffn,
                      c.d_model);
  if (!(m->rms_eps >= 0.f)) return model_fail(ctx, FDL_ERR_INVALID_ARG, "rms_eps < 0");
  if (R < 0 || R > c.max_rows) return model_fail(ctx, FDL_ERR_INVALID_ARG, "R=%d outside [0, max_rows]", R);
  Workspace w = carve(workspace, R, c.d_model, m->ffn);
  if (workspace_bytes < w.bytes)
    return model_fail(ctx, FDL_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, w.bytes);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(final_out) & 15))
    return model_fail(ctx, FDL_ERR_INVALID_ARG, "workspace must be 256-byte and final_out 16-byte aligned");
  for (int l = 0; l < m->n_layers; ++l)
    if (!m->g_attn[l] || !m->w_qkv[l] || !m->w_o[l] || !m->g_mlp[l] || !m->w_gu[l] || !m->w_down[l] ||
        !k_caches[l] || !v_caches[l])
      return model_fail(ctx, FDL_ERR_INVALID_ARG, "fdl_model_forward: NULL pointer for layer %d", l);
  if (R == 0) return FDL_OK;

  const int d = c.d_model, F = m->ffn;
  // Up to 64 rows the gate/up product's fp32 shares (weight-streaming GEMM)
  // are merged by the SwiGLU kernel that consumes them.
  const bool fused_swiglu = fdl_stream_swiglu_applies(ctx, R, d, F);
  fdl_stream_shares sh{};
  fdl_status st = FDL_OK;
  cudaError_t e = fdl_launch_embed(ctx, tokens, R, m->embed, w.h);
  for (int l = 0; e == cudaSuccess && st == FDL_OK && l < m->n_layers; ++l) {
    e = fdl_launch_rmsnorm(ctx, w.h, R, m->g_attn[l], m->rms_eps, w.xn);
    if (e != cudaSuccess) break;
    st = fdl_qkv_rope_cache_write(ctx, w.xn, m->w_qkv[l], R, row_seq, row_rope_pos, row_cache_pos, block_table,
                                  bt_stride, k_caches[l], v_caches[l], w.q);
    if (st != FDL_OK) break;
    st = fdl_sched_attn(ctx, w.q, k_caches[l], v_caches[l], block_table, bt_stride, cu_seqlens_q, kv_len, B, R,
                        row_kind, search_pos, search_ld, n_search, w.o, nullptr, track_scores, track_ld, nullptr);
    if (st != FDL_OK) break;
    e = fdl_launch_dense_tc(ctx, w.o, m->w_o[l], R, d, d, w.h, true);
    if (e == cudaSuccess) e = fdl_launch_rmsnorm(ctx, w.h, R, m->g_mlp[l], m->rms_eps, w.xn);
    if (fused_swiglu) {
      if (e == cudaSuccess) e = fdl_launch_dense_stream_shares(ctx, w.xn, m->w_gu[l], R, d, 2 * F, &sh);
      if (e == cudaSuccess) e = fdl_launch_swiglu_shares(ctx, sh, R, F, w.u);
    } else {
      if (e == cudaSuccess) e = fdl_launch_dense_tc(ctx, w.xn, m->w_gu[l], R, d, 2 * F, w.gu, false);
      if (e == cudaSuccess) e = fdl_launch_swiglu(ctx, w.gu, R, F, w.u);
    }
    if (e == cudaSuccess) e = fdl_launch_dense_tc(ctx, w.u, m->w_down[l], R, F, d, w.h, true);
  }
  if (st != FDL_OK) return st;
  if (e == cudaSuccess) e = fdl_launch_rmsnorm(ctx, w.h, R, m->g_final, m->rms_eps, final_out);
  if (e != cudaSuccess)
    return model_fail(ctx, FDL_ERR_CUDA, "fdl_model_forward launch: %s", cudaGetErrorString(e));
  ctx->last_error[0] = 0;
  return FDL_OK;
}
