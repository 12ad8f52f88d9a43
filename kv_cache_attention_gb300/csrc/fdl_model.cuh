// Internal declarations of the whole-model forward: the dense tensor-core
// GEMM (W_o, the SwiGLU gate/up and down projections) and the row-wise
// kernels around it (embedding, RMSNorm, SwiGLU product).
#pragma once

#include "fdl_internal.cuh"

// out[r, n] (+)= sum_k X[r, k] W[n, k] for r < R, n < N: X [R, K] and W
// [N, K] bf16 row-major, 16-byte aligned, N % 128 == 0, K % 64 == 0. With
// add_f32 the product is added to the fp32 array out (a residual stream);
// otherwise it is stored as bf16.
cudaError_t fdl_launch_dense_tc(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N, void* out,
                                bool add_f32);

// h[r, :] = embed[tokens[r], :] widened to fp32 (a token outside [0, vocab)
// sets the device error word and gives a zero row).
cudaError_t fdl_launch_embed(fdl_ctx* ctx, const int* tokens, int R, const void* embed, float* h);

// out[r, :] = bf16(h[r, :] / sqrt(mean(h[r, :]^2) + eps) * g), fixed-order sums.
cudaError_t fdl_launch_rmsnorm(fdl_ctx* ctx, const float* h, int R, const void* g, float eps, void* out);

// u[r, i] = bf16(silu(gu[r, i]) * gu[r, F + i]) for i < F.
cudaError_t fdl_launch_swiglu(fdl_ctx* ctx, const void* gu, int R, int F, void* u);

// The weight-streaming GEMM's unmerged output (fdl_gemm_stream.cu): the
// schedule of the launch that wrote the fp32 shares, for kernels that merge
// them while consuming the product. Valid until the next launch on the
// context that uses its split-K workspace.
struct fdl_stream_shares {
  unsigned nkb, T, G, U;  // k-blocks per tile, tiles, CTAs, units
  const float* partials;
};

// Whether the model forward's gate/up product over R rows takes the
// weight-streaming GEMM with its merge in the SwiGLU kernel below (d =
// d_model, F = ffn).
bool fdl_stream_swiglu_applies(const fdl_ctx* ctx, int R, int d, int F);

// The GEMM alone: X [R, K] x W [N, K]^T into the context's share workspace.
cudaError_t fdl_launch_dense_stream_shares(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N,
                                           fdl_stream_shares* out);

// u[r, i] = bf16(silu(gate) * up) with gate = bf16(merged product[r, i]) and
// up = bf16(merged product[r, F + i]), as fdl_launch_swiglu over a bf16 store.
cudaError_t fdl_launch_swiglu_shares(fdl_ctx* ctx, const fdl_stream_shares& sh, int R, int F, void* u);

