// tcgen05 path of the fused QKV projection (placeholder until written).
#include "fdl_internal.cuh"

cudaError_t fdl_launch_qkv_tc(fdl_ctx*, const void*, const void*, int, const int*, const int*, const int*,
                              const int*, int, void*, void*, void*) {
  return cudaErrorNotSupported;
}
