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
