// Internal declarations shared by the translation units of libfdl.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/fdl.h"

// Device error-word bits (fdl_sync_status maps them to fdl_status).
#define FDL_DEVERR_INDEX 1u    // out-of-range page / position / row index
#define FDL_DEVERR_TIMEOUT 2u  // a bounded wait gave up
#define FDL_DEVERR_SHAPE 4u    // inconsistent device-side shape data (cu_seqlens, kinds)

// Rows per scheduled-attention work item.
#define FDL_TILE_M_SIMT 16
#define FDL_TILE_M_TC 128

// Eq. (2) tracker partial slots per sequence (the tensor-core attention's
// 128-row query tiles that hold WINDOW rows; a sequence whose WINDOW rows
// span more tiles adds its column sums with atomics instead).
#define FDL_TRK_SLOTS 2

struct fdl_ctx {
  fdl_config cfg;
  cudaStream_t stream;
  int device;
  int num_sms;
  int rope_positions;   // rows of the RoPE tables
  float* rope_cos;      // [rope_positions][head_dim/2]
  float* rope_sin;
  unsigned* err_word;   // device error word
  int attn_tile_m;      // query rows per attention work item
  int* worklist;        // [1 + 4 * worklist_items]: count then items
  int worklist_items;
  int* n_masked;        // [max_batch] WINDOW rows per sequence
  unsigned* tickets;    // [8] last-block tickets (left at zero between calls)
  float* qkv_partials;  // split-K partial tiles of the tensor-core projection
  size_t qkv_partial_floats;
  unsigned* qkv_ticket_buf;  // per-tile arrival counters (zero between calls)
  int qkv_tickets;
  float* lm_part;       // per-CTA row statistics of the fused LM head (bf16 contexts)
  size_t lm_part_floats;
  unsigned* lm_rt_tickets;  // per-row-tile arrival counters of the many-row LM head (zero between calls)
  int lm_rt_ticket_count;
  float* trk_part;       // tracker column sums [max_batch][FDL_TRK_SLOTS][n_heads][trk_ld] (tensor-core attention)
  int* trk_nslots;       // [max_batch] partial slots of each sequence in the last tracked attention call
  int trk_ld;
  long long wait_budget;  // projection main-loop wait budget in cycles (0 = the default ~2 s)
  char last_error[512];
};

namespace fdl {

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

template <typename T>
struct io;

template <>
struct io<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
};

template <>
struct io<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// Slot of (sequence b, cache position c); -1 (and the error bit) when the
// block table maps it outside the pool.
__device__ __forceinline__ long long cache_slot(const int* block_table, int bt_stride, int page_size,
                                                int n_pages, int b, int c, unsigned* err) {
  if (c < 0) return -1;
  int pi = c / page_size;
  if (pi >= bt_stride) {
    raise_error(err, FDL_DEVERR_INDEX);
    return -1;
  }
  int page = block_table[(long long)b * bt_stride + pi];
  if (page < 0 || page >= n_pages) {
    raise_error(err, FDL_DEVERR_INDEX);
    return -1;
  }
  return (long long)page * page_size + (c % page_size);
}

// Programmatic dependent launch. Every kernel of the library is launched
// with programmatic stream serialisation, so it may become resident while
// the previous kernel in the stream is still running. Work that touches no
// global memory (barrier initialisation, TMEM allocation, tensor-map
// prefetch) may run before grid_dep_wait(); every global-memory read or
// write comes after it, because the wait is what guarantees that the
// previous kernel has finished and its writes are visible. Without the
// launch attribute the wait returns at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream launch (it still waits for this one to
// finish before touching memory). Called once this kernel no longer needs
// SM room for CTAs of its own that have not started.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Order-preserving map of a float onto uint32 (-0.0 folded onto +0.0).
__device__ __forceinline__ unsigned float_order_key(float f) {
  unsigned u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace fdl

// Launches `kernel` on `stream` with programmatic stream serialisation (see
// grid_dep_wait). Setting FDL_DISABLE_PDL=1 in the environment launches
// plainly instead, so that each kernel starts only after the previous one
// has finished.
bool fdl_pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t fdl_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (fdl_pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Raises one kernel's dynamic shared-memory limit on the current device.
// The attribute belongs to a device, so it is set once per device (one bit
// per device ordinal below 64; higher ordinals set it on every launch).
// cudaFuncSetAttribute is thread-safe and idempotent, so two host threads
// that race here at most set it twice.
// The kernel also prefers the largest shared-memory carveout, so that
// kernels sized for two CTAs per SM get them.
struct fdl_smem_limit {
  std::atomic<unsigned long long> done{0};
  cudaError_t ensure(const void* kernel, int device, int bytes) {
    const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// Resident CTAs per SM of a kernel on a device, queried once per device
// ordinal below 64 (and on every call above).
struct fdl_occupancy {
  std::atomic<int> per_sm[64] = {};
  int get(const void* kernel, int device, int threads, int smem) {
    if (device >= 0 && device < 64) {
      const int v = per_sm[device].load(std::memory_order_acquire);
      if (v > 0) return v;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, (size_t)smem) != cudaSuccess || n < 1)
      n = 1;
    if (device >= 0 && device < 64) per_sm[device].store(n, std::memory_order_release);
    return n;
  }
};

// Checks a configuration as fdl_create does; false with the reason in `why`.
bool fdl_config_ok(const fdl_config* c, char* why, size_t n);

// Launchers implemented by the kernel translation units. Each returns a
// cudaError_t from the launch.
cudaError_t fdl_launch_qkv(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                           const int* row_rope_pos, const int* row_cache_pos,
                           const int* block_table, int bt_stride, void* k_cache, void* v_cache,
                           void* q_out);

cudaError_t fdl_launch_attn(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                            const int* block_table, int bt_stride, const int* cu_seqlens_q,
                            const int* kv_len, int B, int R, const int* row_kind,
                            const int* search_pos, int search_ld, const int* n_search, void* o_out,
                            float* lse_out, float* track, int track_ld, int* worklist_out);

cudaError_t fdl_launch_topk(fdl_ctx* ctx, const float* scores, const unsigned char* eligible, int ld,
                            const int* seq_len, int B, int k, int* idx_out, int* cnt_out);

cudaError_t fdl_launch_unmask_verify(fdl_ctx* ctx, const fdl_unmask_args* a);

// The fused LM head: unmask decisions from the window rows' hidden states
// (verify == false) or verify acceptance from the mask views' (verify == true).
cudaError_t fdl_launch_lm_head(fdl_ctx* ctx, const void* hidden, const void* w_lm, const fdl_unmask_args* a,
                               bool verify);
// Rows the fused LM head takes in one call, and its workspace floats
// (one set of per-row statistics per CTA of its persistent grid).
int fdl_lm_head_max_rows();
size_t fdl_lm_partial_floats(int num_sms, int max_rows);
int fdl_lm_row_tiles(int max_rows);

// Workspace floats the tensor-core projection needs for split-K partials.
size_t fdl_qkv_partial_floats(int num_sms, int max_rows);

// The weight-streaming GEMM for up to 64 rows (fdl_gemm_stream.cu): whether
// it takes an [R, K] x [N, K]^T product on this context, and its projection
// and dense forms (same contracts as fdl_launch_qkv_tc / fdl_launch_dense_tc).
bool fdl_stream_gemm_applies(const fdl_ctx* ctx, int R, int K, int N);
cudaError_t fdl_launch_qkv_stream(fdl_ctx* ctx, const void* X, const void* W, int R, const int* row_seq,
                                  const int* row_rope_pos, const int* row_cache_pos, const int* block_table,
                                  int bt_stride, void* k_cache, void* v_cache, void* q_out);
cudaError_t fdl_launch_dense_stream(fdl_ctx* ctx, const void* X, const void* W, int R, int K, int N, void* out,
                                    bool add_f32);
