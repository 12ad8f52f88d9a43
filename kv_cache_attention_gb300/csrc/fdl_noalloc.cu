// Scheduled attention for callers that cannot allocate device memory.
//
// fdl_sched_attn needs a context, and fdl_create allocates that context's
// workspace with cudaMalloc. Some callers cannot do that: code that runs
// under an external memory manager which owns the whole device heap and
// forbids further cudaMalloc, or code on a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not acceptable. This file
// gives them fdl_sched_attn_noalloc: the same attention kernels, with the
// only scratch they need (the device-built work list and the per-sequence
// masked-row counts) held in one file-scope __device__ array that is part of
// the loaded library image. Nothing is allocated on any call.
//
// The array is shared by every call on a device and keeps the last call's
// contents; each call rewrites every word it reads (the item count, the
// items and the counts of its B sequences), so nothing has to start at zero.
// Calls that overlap on the GPU (different streams, or concurrent host
// threads) race on the array and must be serialised by the caller.
#include <mutex>
#include <stdio.h>

#include "fdl_internal.cuh"

namespace {

// Largest call the scratch array holds: work items (query tiles of the
// attention kernel, ceil(rows_b / tile) summed over sequences) and sequences.
constexpr int kMaxItems = 4096;
constexpr int kMaxSeqs = 1024;
constexpr int kScratchInts = 1 + 4 * kMaxItems + kMaxSeqs;

// ~70 KB, held by every GPU that loads the library until the process exits.
static __device__ __align__(256) int g_attn_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
int* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device. The name
// g_attn_scratch in host code is only a host-side stand-in, so the address
// is looked up once per device (on that device's first call) and cached for
// the life of the process. A cudaDeviceReset unloads the module that holds
// the array, so the library must not be used on a device after resetting it
// (the same holds for every context created before the reset).
cudaError_t scratch_address(int device, int** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = static_cast<int*>(p);
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

fdl_status reject(const char* msg) {
  fprintf(stderr, "fdl_sched_attn_noalloc: %s\n", msg);
  return FDL_ERR_INVALID_ARG;
}

}  // namespace

bool fdl_attn_tc_supported(const fdl_config& c);

extern "C" fdl_status fdl_sched_attn_noalloc(const fdl_config* cfg, void* cuda_stream, const void* q,
                                             const void* k_cache, const void* v_cache, const int* block_table,
                                             int bt_stride, const int* cu_seqlens_q, const int* kv_len, int B,
                                             int R, const int* row_kind, const int* search_pos, int search_ld,
                                             const int* n_search, void* o_out, float* lse_out,
                                             float* track_scores, int track_ld, unsigned* device_error) {
  if (!cfg) return reject("NULL config");
  const fdl_config& c = *cfg;
  if (B < 0 || R < 0) return reject("negative B or R");
  {
    // the checks fdl_create makes, except the limits that size a context's
    // workspace (max_batch, max_rows, vocab): this call has none
    fdl_config cc = c;
    cc.max_batch = 1;
    cc.max_rows = 1;
    cc.vocab = 1;
    char why[256];
    if (!fdl_config_ok(&cc, why, sizeof(why))) return reject(why);
  }
  if (B == 0 || R == 0) return FDL_OK;
  if (B > kMaxSeqs) return reject("B exceeds the 1024 sequences the static scratch holds");
  const int tile = fdl_attn_tc_supported(c) ? FDL_TILE_M_TC : FDL_TILE_M_SIMT;
  if ((long long)(R + tile - 1) / tile + B > kMaxItems)
    return reject("rows need more than the 4096 work items the static scratch holds");
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !kv_len || !row_kind || !o_out)
    return reject("NULL pointer argument");
  if (bt_stride <= 0) return reject("bt_stride must be positive");
  if (search_pos && (!n_search || search_ld <= 0 || c.max_views == 0))
    return reject("search_pos needs n_search, search_ld > 0 and max_views > 0");
  if (track_scores && track_ld < c.max_seq) return reject("track_ld below max_seq");

  // A context on the stack: it points the kernels at the static scratch and
  // the caller's error word instead of an allocated workspace.
  fdl_ctx ctx = {};
  ctx.cfg = c;
  ctx.cfg.max_batch = B;
  ctx.cfg.max_rows = R;
  ctx.stream = static_cast<cudaStream_t>(cuda_stream);
  if (cudaGetDevice(&ctx.device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx.num_sms, cudaDevAttrMultiProcessorCount, ctx.device) != cudaSuccess)
    return FDL_ERR_CUDA;
  int* scratch = nullptr;
  cudaError_t e = scratch_address(ctx.device, &scratch);
  if (e != cudaSuccess) {
    fprintf(stderr, "fdl_sched_attn_noalloc: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
    return FDL_ERR_CUDA;
  }
  ctx.err_word = device_error;
  ctx.attn_tile_m = tile;
  ctx.worklist = scratch;
  ctx.worklist_items = kMaxItems;
  ctx.n_masked = scratch + 1 + 4 * kMaxItems;
  e = fdl_launch_attn(&ctx, q, k_cache, v_cache, block_table, bt_stride, cu_seqlens_q, kv_len, B, R, row_kind,
                      search_pos, search_ld, n_search, o_out, lse_out, track_scores, track_ld, nullptr);
  if (e != cudaSuccess) {
    fprintf(stderr, "fdl_sched_attn_noalloc: launch failed: %s\n", cudaGetErrorString(e));
    return FDL_ERR_CUDA;
  }
  return FDL_OK;
}
