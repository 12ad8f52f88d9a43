/*
 * fdl.h -- C ABI of the GB300 (sm_103a) Flash-dLLM layer-step hot path.
 *
 * The library computes, for one diffusion-LLM denoising step, the per-layer
 * Flash-Cache path and the per-step decoding decisions described by
 * "Flash-dLLM: IO-Aware KV Caching and Parallel Decoding for Fast,
 * Memory-Efficient Diffusion LLMs" (paper digest; sections "Core method" and
 * "Method steps in detail", Algorithm 2 steps 1-4 and Eq. (2)):
 *
 *   fdl_qkv_rope_cache_write  fused QKV projection + RoPE + K/V cache scatter
 *   fdl_sched_attn            block-table scheduled attention over the cache,
 *                             with the Flash-Verify two-view mask and the
 *                             Eq. (2) attention-mass tracker
 *   fdl_track_topk            top-k of the tracker scores (next tracked set)
 *   fdl_unmask_verify         confidence-threshold unmasking (search list) and
 *                             Flash-Verify prefix acceptance
 *   fdl_lm_head_unmask        the unmasking decisions straight from the window
 *                             rows' hidden states (LM head fused, logits never
 *                             stored)
 *   fdl_lm_head_verify        the verify acceptance straight from the mask
 *                             views' hidden states (LM head fused)
 *   fdl_model_forward         the whole transformer forward over a step's
 *                             refresh rows (embedding, every layer's norm,
 *                             projection, attention, W_o and SwiGLU FFN, the
 *                             final norm)
 *   fdl_flash_step            one Flash-dLLM denoising step of a whole model
 *                             (draft forward, unmasking, verify forward,
 *                             acceptance, next tracked set)
 *   fdl_refresh_rows          (host) the query rows of a step under a KV-cache
 *                             refresh policy: Fast-dLLM PrefixCache and
 *                             DualCache, FlashDLM FreeCache, the Flash-dLLM
 *                             draft forward
 *   fdl_verify_rows           (host) the query rows of a Flash-Verify forward
 *
 * Conventions shared by every entry point (exceptions: the two host row
 * builders take and return host arrays and touch no device; fdl_flash_step
 * keeps its sequences' state in host arrays and synchronises the stream;
 * the per-layer pointer arrays of fdl_model_forward and fdl_flash_step are
 * host arrays of device pointers)
 *   - All tensor arguments are DEVICE pointers owned by the caller (for
 *     example PyTorch allocations); the library never frees them.
 *   - Every call is asynchronous on the context's CUDA stream.
 *   - The return value reports host-side validation only: a NULL required
 *     pointer, a size beyond the limits fixed at fdl_create, an unsupported
 *     shape. On error nothing is launched and fdl_last_error() says why.
 *   - Data-dependent problems found on the device (a block-table entry
 *     outside the page pool, a position past the cache, inconsistent
 *     cu_seqlens, a bounded wait that gave up) never trap: the offending
 *     access is skipped and a device error word is set. fdl_sync_status()
 *     synchronises the stream and reports (and clears) that word as
 *     FDL_ERR_DEVICE_INDEX or FDL_ERR_TIMEOUT.
 *   - Floating-point tensors use the context dtype (FDL_F32 or FDL_BF16);
 *     accumulation is fp32. Index tensors are int32, masks are uint8.
 *   - A context is not thread-safe, and calls on one context must not overlap
 *     on the GPU (they share its workspace): use one context per host thread
 *     and one per stream when calls run concurrently.
 */
#ifndef FDL_H_
#define FDL_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FDL_OK = 0,
  FDL_ERR_INVALID_ARG = 1,   /* bad pointer / size / shape; nothing launched   */
  FDL_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 96)   */
  FDL_ERR_OOM = 3,           /* workspace allocation failed in fdl_create      */
  FDL_ERR_CUDA = 4,          /* a CUDA runtime call failed                     */
  FDL_ERR_DEVICE_INDEX = 5,  /* device saw an out-of-range index (skipped)     */
  FDL_ERR_TIMEOUT = 6        /* a bounded device wait gave up                  */
} fdl_status;

typedef enum { FDL_F32 = 0, FDL_BF16 = 1 } fdl_dtype;

/* Row kinds (row_kind arrays). j is the 0-based index of a search token in
 * the acceptance order of its sequence. */
#define FDL_KIND_NORMAL 0                 /* tracked / T_v / full-refresh row   */
#define FDL_KIND_WINDOW 1                 /* masked-window row: feeds Eq. (2)    */
#define FDL_KIND_DRAFT_VIEW(j) (2 + 2 * (j))
#define FDL_KIND_MASK_VIEW(j) (3 + 2 * (j))

/* Shape limits fixed for the life of a context. */
typedef struct {
  int d_model;        /* = n_heads * head_dim                                   */
  int n_heads;
  int head_dim;       /* 64 or 128                                              */
  double rope_theta;  /* RoPE base (LLaDA: 5e5)                                 */
  int max_batch;      /* most sequences in one call                             */
  int max_seq;        /* N_max: base cache positions per sequence               */
  int max_views;      /* view-key cache positions past a sequence's kv_len      */
  int page_size;      /* cache slots per block-table page                       */
  int n_pages;        /* pages in the pool: each cache holds n_pages*page_size  */
                      /* rows of d_model elements                               */
  int max_rows;       /* most query rows in one call                            */
  int vocab;          /* logits row length                                      */
  fdl_dtype dtype;    /* storage type of X, W, Q, caches, O and logits          */
} fdl_config;

typedef struct fdl_ctx fdl_ctx;

/* Creates a context on the current CUDA device and allocates its workspace
 * (RoPE cos/sin table for positions 0..max_seq+max_views-1 computed in
 * double on the host, the scheduled-attention work list, counters and the
 * device error word). cuda_stream is a cudaStream_t (NULL = legacy default
 * stream). Returns FDL_ERR_INVALID_ARG for inconsistent limits,
 * FDL_ERR_OOM / FDL_ERR_CUDA if allocation fails. */
fdl_status fdl_create(const fdl_config* cfg, void* cuda_stream, fdl_ctx** out);
void fdl_destroy(fdl_ctx* ctx);
fdl_status fdl_set_stream(fdl_ctx* ctx, void* cuda_stream);
/* Human-readable reason for the last non-OK status of this context. */
const char* fdl_last_error(const fdl_ctx* ctx);
/* Synchronises the context stream, then returns and clears the device error
 * word: FDL_OK, FDL_ERR_DEVICE_INDEX or FDL_ERR_TIMEOUT (FDL_ERR_CUDA if the
 * stream itself reported an error). */
fdl_status fdl_sync_status(fdl_ctx* ctx);
/* Query rows per scheduled-attention work item (the oracle rebuilds the
 * work list with this tile). */
int fdl_tile_m(const fdl_ctx* ctx);
/* Number of int32 a worklist_out buffer needs for R rows over B sequences:
 * 1 (item count) + 4 per possible item. */
int fdl_worklist_capacity(const fdl_ctx* ctx, int R, int B);
/* Failure-path testing: sets the budget, in SM clock cycles, of every wait
 * in the main loop of this context's tensor-core projection (the TMA ring's
 * full/empty mbarriers). 0 restores the default of about 2 s, far above any
 * legitimate wait. A budget shorter than a DRAM load makes the wait give up:
 * the kernel then lets its loads in flight land, waits for its issued
 * products, frees its TMEM, writes no output, keeps its split-K counters
 * consistent and sets the device error word, so fdl_sync_status returns
 * FDL_ERR_TIMEOUT and the context stays usable. The drain waits keep the
 * default budget. Returns FDL_ERR_INVALID_ARG for a negative budget. */
fdl_status fdl_set_wait_budget(fdl_ctx* ctx, long long cycles);

/* ------------------------------------------------------------------------
 * Flash-Cache fused projection (paper digest, "Core method": QKV projection,
 * RoPE and cache write fused so K/V go straight into the preallocated cache;
 * "Method steps" step 2: the refresh rows are the masked window plus the
 * tracked set).
 *
 * For every query row r (0 <= r < R):
 *   [q | k | v] = X[r] . Wqkv^T                    (fp32 accumulation)
 *   q, k <- RoPE(q, k) at position row_rope_pos[r]: rotate-half pairs
 *           (i, i + head_dim/2) by angle pos * rope_theta^(-2i/head_dim)
 *   q_out[r] = q                                   ([R, n_heads, head_dim])
 *   if row_cache_pos[r] >= 0:  with b = row_seq[r], c = row_cache_pos[r],
 *     slot = block_table[b*bt_stride + c/page_size]*page_size + c%page_size
 *     k_cache[slot] = k, v_cache[slot] = v         (rows of d_model)
 *
 * X: [R, d_model]; Wqkv: [3*d_model, d_model] row-major, Q rows then K rows
 * then V rows, head h in rows h*head_dim..(h+1)*head_dim-1 of each block.
 * R <= max_rows. Row r's writes are skipped (device error word set) when
 * its page lies outside [0, n_pages), c/page_size >= bt_stride, or its RoPE
 * position is outside the table. Two rows writing the same slot race.
 * ---------------------------------------------------------------------- */
fdl_status fdl_qkv_rope_cache_write(fdl_ctx* ctx, const void* X, const void* Wqkv, int R,
                                    const int* row_seq, const int* row_rope_pos,
                                    const int* row_cache_pos, const int* block_table,
                                    int bt_stride, void* k_cache, void* v_cache, void* q_out);

/* ------------------------------------------------------------------------
 * Scheduled attention (paper digest, "Background": exact IO-aware attention;
 * "Core method": block-table scheduled attention over ragged per-sequence
 * query blocks, and the two-view verify mask; "Method steps" step 4, Eq. (2)).
 *
 * Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q
 * ([R, n_heads, head_dim]); its base keys are cache positions
 * 0..kv_len[b]-1. When search_pos is not NULL, sequence b has
 * m = n_search[b] search tokens at base positions search_pos[b*search_ld + j]
 * (j < m <= min(search_ld, max_views/2), in acceptance order) whose draft-view keys sit at cache positions
 * kv_len[b]+j and mask-view keys at kv_len[b]+m+j.
 * Visibility by row_kind:
 *   NORMAL, WINDOW      all base keys;
 *   DRAFT_VIEW(k)       base keys except the search positions, draft keys
 *                       j <= k, mask keys j > k;
 *   MASK_VIEW(k)        base keys except the search positions, draft keys
 *                       j < k, mask keys j >= k.
 * For each row and head: o = softmax(q.K^T / sqrt(head_dim)) V over the
 * visible keys, lse = log sum exp of the scaled scores (natural log).
 * Tracker (track_scores != NULL): for every base key i of sequence b,
 *   track_scores[b*track_ld + i] += sum_h sum_{WINDOW rows j} p_{h,j,i} / (H*M_b)
 * with M_b the number of WINDOW rows of b; the caller zeroes the buffer
 * once per step and every layer's call accumulates into it. On the
 * tensor-core path (bf16, head_dim 128, B <= 1024) the sums are in a fixed
 * order, so a call reproduces its scores bit for bit, for every sequence
 * whose WINDOW rows lie within two 128-row query tiles; other sequences, and
 * the CUDA-core path, add with atomics (exact up to fp32 reassociation).
 * Several calls on one context must not overlap on the GPU (each call's
 * partial sums use the context's workspace).
 * o_out: [R, n_heads, head_dim] (context dtype); lse_out: [R, n_heads] fp32
 * (nullable); worklist_out (nullable, fdl_worklist_capacity ints): count,
 * then (b, q_start, q_len, n_keys) per item, n_keys = kv_len[b] + 2m.
 * Requires B <= max_batch, R <= max_rows; R must equal cu_seqlens_q[B]
 * (checked on the device).
 * ---------------------------------------------------------------------- */
fdl_status fdl_sched_attn(fdl_ctx* ctx, const void* q, const void* k_cache, const void* v_cache,
                          const int* block_table, int bt_stride, const int* cu_seqlens_q,
                          const int* kv_len, int B, int R, const int* row_kind,
                          const int* search_pos, int search_ld, const int* n_search, void* o_out,
                          float* lse_out, float* track_scores, int track_ld,
                          int* worklist_out);

/* ------------------------------------------------------------------------
 * Tracker top-k (paper digest, "Method steps" step 4: the top-k decoded
 * tokens by attention mass become the next tracked set).
 *
 * For each sequence b: among positions i < seq_len[b] with
 * eligible[b*ld + i] != 0, the k with the largest scores[b*ld + i], ordered
 * by score descending then position ascending. idx_out[b*k + t] holds the
 * t-th position (-1 past cnt_out[b] = min(k, #eligible)). 1 <= k <= 1024.
 * Scores must not be NaN; -0.0 and +0.0 compare equal.
 * ---------------------------------------------------------------------- */
fdl_status fdl_track_topk(fdl_ctx* ctx, const float* scores, const unsigned char* eligible,
                          int ld, const int* seq_len, int B, int k, int* idx_out, int* cnt_out);

/* ------------------------------------------------------------------------
 * Confidence unmasking and Flash-Verify acceptance (paper digest, "Method
 * steps" steps 2 and 3; Fast-dLLM "confidence-aware parallel decoding" for
 * the forced-progress fallback).
 *
 * Unmask phase (logits != NULL): for each window row r < R_w (rows grouped
 * by sequence: row_seq non-decreasing):
 *   conf[r] = max_v softmax(logits[r])_v = 1 / sum_v exp(l_v - max l)
 *   argmax[r] = lowest v attaining max l
 *   commit[r] = conf[r] >= eps
 *   if force_progress and sequence b committed nothing: commit its row of
 *   highest conf (lowest row_pos on ties).
 *   search_rows[b*max_search + j] = the uncommitted rows of b ordered by conf
 *   descending then row_pos ascending, j < n_search[b] <= max_search; -1 pad.
 * Verify phase (mask_logits != NULL): row b*max_search + j (j < n_search[b])
 *   of mask_logits is the mask view of b's j-th search token and
 *   draft_tok[b*max_search + j] its draft token. With c~ and x~ the mask
 *   view's confidence and argmax, accept[b*max_search + j] = 1 for the
 *   longest prefix j = 0, 1, ... with draft_tok == x~ and c~ >= gamma;
 *   n_accept[b] is its length. mask_conf / mask_argmax receive c~ and x~. If both phases run in one call, the verify phase reads the
 *   n_search the unmask phase wrote.
 * Logits rows have config.vocab entries of the context dtype.
 * ---------------------------------------------------------------------- */
typedef struct {
  int B;
  int max_search;
  /* unmask phase */
  const void* logits;          /* [R_w, vocab] or NULL to skip the phase */
  int R_w;
  const int* row_seq;          /* [R_w] */
  const int* row_pos;          /* [R_w] */
  float eps;
  int force_progress;
  float* conf;                 /* [R_w] */
  int* argmax;                 /* [R_w] */
  unsigned char* commit;       /* [R_w] */
  int* search_rows;            /* [B*max_search] */
  int* n_search;               /* [B]; output of unmask, input of verify */
  /* verify phase */
  const void* mask_logits;     /* [B*max_search, vocab] or NULL to skip */
  const int* draft_tok;        /* [B*max_search] */
  float gamma;
  unsigned char* accept;       /* [B*max_search] */
  int* n_accept;               /* [B] */
  float* mask_conf;            /* [B*max_search] */
  int* mask_argmax;            /* [B*max_search] */
} fdl_unmask_args;

fdl_status fdl_unmask_verify(fdl_ctx* ctx, const fdl_unmask_args* args);

/* ------------------------------------------------------------------------
 * Fused LM head + unmasking (paper digest, "Method steps in detail", step 2:
 * c_i = max_x p(x_i | x^t) is taken over the model's output distribution,
 * the softmax of the language-model head on each masked position's final
 * hidden state). The logits are never stored:
 *   logits[r] = hidden[r] . w_lm^T     (config.vocab entries, fp32 accumulation)
 * and the unmask phase of fdl_unmask_verify is applied to them: conf,
 * argmax, commit, search_rows and n_search exactly as documented above,
 * from args' R_w, row_seq, row_pos, eps, force_progress, max_search and B.
 * args->logits and args->mask_logits must be NULL (the verify phase runs
 * through fdl_unmask_verify on explicit mask-view logits).
 *
 * hidden: [R_w, d_model] bf16, the window rows' final hidden states (16-byte
 * aligned); w_lm: [vocab, d_model] bf16 row-major (16-byte aligned). bf16
 * contexts only, d_model a multiple of 64, 1 <= R_w <= max_rows: otherwise
 * FDL_ERR_UNSUPPORTED / FDL_ERR_INVALID_ARG. Up to 64 rows form one column
 * tile against 128-entry vocabulary tiles; more rows take 128-row tiles
 * against 256-entry vocabulary tiles (the batched Flash-Verify scale, e.g.
 * 32 sequences x 32 window rows). The reductions over the vocabulary run in
 * a fixed order, so results do not depend on timing.
 * ---------------------------------------------------------------------- */
fdl_status fdl_lm_head_unmask(fdl_ctx* ctx, const void* hidden, const void* w_lm, const fdl_unmask_args* args);

/* ------------------------------------------------------------------------
 * Fused LM head + Flash-Verify acceptance (paper digest, "Method steps in
 * detail", step 3: the mask view's prediction x~ and confidence c~ are the
 * argmax and the maximum of the model's output distribution at that view).
 * The logits are never stored:
 *   logits[r] = mask_hidden[r] . w_lm^T   for r = b*max_search + j, j < n_search[b]
 * and the verify phase of fdl_unmask_verify is applied to them: mask_conf,
 * mask_argmax (written for those rows only), accept and n_accept exactly as
 * documented above, from args' B, max_search, n_search (input), draft_tok
 * and gamma. args->logits and args->mask_logits must be NULL.
 *
 * mask_hidden: [B*max_search, d_model] bf16, the mask-view rows' final hidden
 * states in the verify forward's layout (rows j >= n_search[b] are read but
 * ignored); w_lm as for fdl_lm_head_unmask. bf16 contexts only,
 * 1 <= B*max_search <= max_rows: otherwise FDL_ERR_UNSUPPORTED /
 * FDL_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
fdl_status fdl_lm_head_verify(fdl_ctx* ctx, const void* mask_hidden, const void* w_lm,
                              const fdl_unmask_args* args);

/* ------------------------------------------------------------------------
 * Scheduled attention without any device allocation. The paper has no
 * counterpart: this is a deployment variant of fdl_sched_attn.
 *
 * For callers that cannot call cudaMalloc: code running under an external
 * memory manager that owns the whole device heap, or on a latency-critical
 * path where an allocation (which may synchronise the device) is not
 * acceptable. It needs no context (fdl_create allocates one) and allocates
 * nothing on any call. Its scratch (the device-built work list and the
 * per-sequence masked-row counts) lives in a static device array of about
 * 70 KB that every GPU loading the library holds until the process exits.
 *
 * Arguments and results are those of fdl_sched_attn (same kernels), with the
 * limits taken from *cfg and the work list not exported. *cfg is checked as
 * fdl_create checks it, except max_batch, max_rows and vocab, which are
 * ignored (the call's B and R apply). Limits of the static scratch:
 * B <= 1024 and ceil(R / fdl_tile_m) + B <= 4096 work items, where the tile
 * is 128 rows for bf16 contexts with head_dim 128 and 16 rows otherwise;
 * larger calls return FDL_ERR_INVALID_ARG (reason on stderr). Device-side
 * index errors are OR-ed into *device_error (a caller-owned device word, may
 * be NULL; the caller zeroes and reads it) with the bits of the device error
 * word: 1 index, 2 timeout, 4 shape.
 *
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress) and caches it for the life of the process; make
 * that first call before any stream capture, and do not use the library on
 * a device after a cudaDeviceReset of it (the reset unloads the array). Every call on a device shares the array and rewrites all
 * of it that it reads; calls that overlap on the GPU (several streams or host
 * threads) race on it and must be serialised by the caller.
 * ---------------------------------------------------------------------- */
fdl_status fdl_sched_attn_noalloc(const fdl_config* cfg, void* cuda_stream, const void* q,
                                  const void* k_cache, const void* v_cache, const int* block_table,
                                  int bt_stride, const int* cu_seqlens_q, const int* kv_len, int B, int R,
                                  const int* row_kind, const int* search_pos, int search_ld,
                                  const int* n_search, void* o_out, float* lse_out, float* track_scores,
                                  int track_ld, unsigned* device_error);

/* ------------------------------------------------------------------------
 * Whole-model forward over one step's refresh rows (the dLLM the path sits
 * in: paper digest, "Background", a bidirectional transformer such as LLaDA;
 * "Method steps in detail", Algorithm 2 step 2, each step's query rows go
 * through every layer against the full cache). The pages are silent on the
 * block's internals; it is LLaMA-style (LLaDA's), with no biases:
 *   h = embed[tokens[r]]                                  (fp32)
 *   per layer l:
 *     a  = RMSNorm(h) * g_attn[l]                         (bf16)
 *     fdl_qkv_rope_cache_write(a, w_qkv[l], ...) into k_caches[l], v_caches[l]
 *     o  = fdl_sched_attn(...)  (with track_scores: Eq. (2) summed over layers)
 *     h += o . w_o[l]^T
 *     m  = RMSNorm(h) * g_mlp[l]                          (bf16)
 *     h += (SiLU(m . W_gate^T) * (m . W_up^T)) . w_down[l]^T
 *   final_out = RMSNorm(h) * g_final                      (bf16 [R, d_model])
 * with RMSNorm(x) = x / sqrt(mean(x^2) + rms_eps). The rows, cu_seqlens,
 * kv_len, block table, views and tracker arguments are those of
 * fdl_qkv_rope_cache_write and fdl_sched_attn (same meaning, same checks);
 * tokens [R] are the rows' input token ids (the [MASK] id for a masked
 * position). k_caches / v_caches are HOST arrays of n_layers DEVICE pointers,
 * one cache pair per layer. workspace is caller-owned device memory of at
 * least fdl_model_workspace_bytes(ctx, ffn, R) bytes, 256-byte aligned
 * (the fp32 residual stream and the bf16 intermediates).
 *
 * bf16 contexts only, d_model a multiple of 128, ffn a multiple of 64:
 * otherwise FDL_ERR_UNSUPPORTED. A token id outside [0, vocab) gives a zero
 * input row and sets the device error word (FDL_ERR_DEVICE_INDEX).
 * ---------------------------------------------------------------------- */
typedef struct {
  int n_layers;
  int ffn;                    /* SwiGLU hidden size F                              */
  float rms_eps;
  const void* embed;          /* [vocab, d_model] bf16                             */
  const void* const* g_attn;  /* host array [n_layers] of [d_model] bf16 gains     */
  const void* const* w_qkv;   /* host array [n_layers] of [3 d_model, d_model] bf16 */
  const void* const* w_o;     /* host array [n_layers] of [d_model, d_model] bf16   */
  const void* const* g_mlp;   /* host array [n_layers] of [d_model] bf16 gains     */
  const void* const* w_gu;    /* host array [n_layers] of [2 ffn, d_model] bf16:
                                 the gate rows, then the up rows                   */
  const void* const* w_down;  /* host array [n_layers] of [d_model, ffn] bf16      */
  const void* g_final;        /* [d_model] bf16                                    */
} fdl_model;

size_t fdl_model_workspace_bytes(const fdl_ctx* ctx, int ffn, int R);

fdl_status fdl_model_forward(fdl_ctx* ctx, const fdl_model* model, const int* tokens, int R,
                             const int* row_seq, const int* row_rope_pos, const int* row_cache_pos,
                             const int* row_kind, const int* cu_seqlens_q, const int* kv_len, int B,
                             const int* block_table, int bt_stride, void* const* k_caches,
                             void* const* v_caches, const int* search_pos, int search_ld,
                             const int* n_search, float* track_scores, int track_ld, void* workspace,
                             size_t workspace_bytes, void* final_out);

/* ------------------------------------------------------------------------
 * Row descriptors of one step under a KV-cache refresh policy (HOST code:
 * every pointer below is a host pointer; no context, no GPU work).
 *
 * A refresh policy only chooses which positions a step recomputes. Each
 * chosen row gets rope position = cache position = its position (its K/V
 * overwrite the cache there) and attends over the whole cache (kv_len of its
 * sequence = seq_len). Positions not chosen keep the K/V last written.
 * Blocks start at the end of the prompt: block i of sequence b covers
 * [prompt_len[b] + i*block, min(prompt_len[b] + (i+1)*block, seq_len[b])).
 * The current block is the first one still holding a masked position.
 *
 *   FDL_REFRESH_FULL       every position, every step (no cache reuse).
 *   FDL_REFRESH_PREFIX     Fast-dLLM PrefixCache (Fast-dLLM news piece, the
 *                          key-value cache for block-wise decoding): the
 *                          current block and everything after it; at the
 *                          first step of every block (state != current
 *                          block) every position, which is how the cache of
 *                          all tokens is recomputed once a block is decoded.
 *   FDL_REFRESH_DUAL       Fast-dLLM DualCache: the current block only (the
 *                          masked suffix stays cached); every position at the
 *                          first step of every block.
 *   FDL_REFRESH_FREECACHE  FlashDLM FreeCache (FlashDLM note, key design 1):
 *                          every position at the first step (state == -1),
 *                          then the current block and every later block;
 *                          finished blocks and the prompt stay frozen.
 *   FDL_REFRESH_FLASH_DRAFT  Flash-dLLM (paper digest, Algorithm 2 steps 1
 *                          and 2): every position at the first step (state
 *                          == -1, the initial full forward), then the draft
 *                          forward's query: the window (the first `block` still-
 *                          masked positions at or after the prompt, in
 *                          position order) followed by the tracked positions
 *                          in the order given.
 *
 * Row kinds: FDL_KIND_WINDOW for the rows whose predictions are decoded (the
 * still-masked positions of the current block; for FLASH_DRAFT the window),
 * FDL_KIND_NORMAL for every other row. Rows of a sequence are contiguous
 * (cu_seqlens) and, except for FLASH_DRAFT, in ascending position order. A
 * sequence with no masked position left takes no rows and keeps its state.
 *
 * state[b] carries the policy's memory between steps: set it to -1 before a
 * sequence's first step; the call updates it (the block refreshed in full
 * last; 0 for FLASH_DRAFT after its first step).
 *
 * Errors (FDL_ERR_INVALID_ARG; nothing written, state untouched): a NULL
 * pointer the policy needs, B < 1, block < 1, an unknown policy, prompt_len
 * or seq_len outside 0 <= prompt_len <= seq_len <= max_seq, state < -1,
 * n_tracked outside [0, tracked_ld], a tracked position outside the sequence,
 * masked or repeated, or more rows than max_rows.
 * ---------------------------------------------------------------------- */
typedef enum {
  FDL_REFRESH_FULL = 0,
  FDL_REFRESH_PREFIX = 1,
  FDL_REFRESH_DUAL = 2,
  FDL_REFRESH_FREECACHE = 3,
  FDL_REFRESH_FLASH_DRAFT = 4
} fdl_refresh_policy;

typedef struct {
  int policy;                  /* fdl_refresh_policy                                */
  int B;                       /* sequences                                         */
  int max_seq;                 /* row stride of masked                              */
  int block;                   /* block size; the window size for FLASH_DRAFT       */
  const int* prompt_len;       /* [B]                                               */
  const int* seq_len;          /* [B] N_b                                           */
  const unsigned char* masked; /* [B*max_seq] 1 = position still masked             */
  int* state;                  /* [B] in/out, -1 before the first step              */
  const int* tracked;          /* FLASH_DRAFT only: [B*tracked_ld] positions        */
  int tracked_ld;
  const int* n_tracked;        /* FLASH_DRAFT only: [B]                             */
  int max_rows;                /* capacity of the four row arrays                   */
  int* row_seq;                /* [max_rows] out                                    */
  int* row_rope_pos;           /* [max_rows] out                                    */
  int* row_cache_pos;          /* [max_rows] out                                    */
  int* row_kind;               /* [max_rows] out                                    */
  int* cu_seqlens;             /* [B+1] out                                         */
  int* n_rows;                 /* [1] out: total rows                               */
} fdl_refresh_args;

fdl_status fdl_refresh_rows(const fdl_refresh_args* args);

/* ------------------------------------------------------------------------
 * Row descriptors of a Flash-dLLM verify forward (HOST code, host pointers;
 * paper digest, Algorithm 2 step 3, and the aiposthub article's Flash-Verify
 * section). For sequence b with m = n_search[b] search tokens s_0..s_{m-1}
 * (search_pos[b*search_ld + j], in acceptance order):
 *   - the first max(0, query_budget - 2m) tracked positions (tracked[b*
 *     tracked_ld ...], ordered by score, n_tracked[b] of them) as
 *     FDL_KIND_NORMAL rows at their own positions;
 *   - then s_j's draft view: rope position s_j, cache position seq_len[b] + j,
 *     kind FDL_KIND_DRAFT_VIEW(j);
 *   - then s_j's mask view: rope position s_j, cache position seq_len[b] + m
 *     + j, kind FDL_KIND_MASK_VIEW(j).
 * The attention of this forward takes kv_len = seq_len and search_pos /
 * n_search as given here. Errors (FDL_ERR_INVALID_ARG, nothing written): a
 * NULL pointer, B < 1, query_budget < 0, n_tracked or n_search outside
 * [0, ld], a tracked or search position outside [0, seq_len[b]), a repeated
 * search position, or more rows than max_rows.
 * ---------------------------------------------------------------------- */
fdl_status fdl_verify_rows(int B, const int* seq_len, const int* tracked, int tracked_ld,
                           const int* n_tracked, const int* search_pos, int search_ld,
                           const int* n_search, int query_budget, int max_rows, int* row_seq,
                           int* row_rope_pos, int* row_cache_pos, int* row_kind, int* cu_seqlens,
                           int* n_rows);

/* ------------------------------------------------------------------------
 * One Flash-dLLM denoising step of a whole model on a batch of sequences
 * (paper digest, "Method steps in detail", Algorithm 2 steps 2-4):
 *   1. draft forward (fdl_model_forward with the tracker) over the rows
 *      fdl_refresh_rows gives for FDL_REFRESH_FLASH_DRAFT: the tracked set
 *      and the window of the first `window` masked positions; at a
 *      sequence's first step (state -1) every position, which fills the
 *      caches (Algorithm 2 step 1);
 *   2. fdl_lm_head_unmask on the window rows: c >= eps is decoded, the
 *      uncommitted rows, most confident first, form the search list;
 *   3. if any sequence has search tokens, the verify forward over the rows
 *      of fdl_verify_rows (query budget track_budget + window; draft views
 *      hold their draft tokens, mask views mask_token), then
 *      fdl_lm_head_verify on the mask views: the accepted prefix is decoded;
 *   4. the committed, then the accepted tokens (each in position order) are
 *      written into tokens / masked; the next tracked set is those newly
 *      decoded positions, then the top (track_budget - their number) of the
 *      other decoded positions (prompt included) by the draft forward's
 *      tracker scores (fdl_track_topk), at most track_budget in all.
 * The sequences' state is HOST memory and is updated in place; the caches
 * (host array of per-layer device pointers, as in fdl_model_forward) and the
 * device block table must hold seq_len + 2*max_search slots per sequence
 * (the view keys). The call synchronises the context's stream (it reads the
 * decisions back three times). workspace: device memory of at least
 * fdl_flash_workspace_bytes bytes, 256-byte aligned. Limits: B*window and
 * B*max_search <= config.max_rows, 2*max_search <= config.max_views,
 * the first step's rows (every position of every sequence) <= max_rows.
 * A step on sequences with nothing left masked returns FDL_OK and does
 * nothing. An error before the decisions are applied (a bad argument, a
 * rejected row set, a device error reported at a read-back) leaves the
 * sequences as they were; an error while choosing the next tracked set leaves
 * the decoded tokens in place and the tracked set unchanged.
 * ---------------------------------------------------------------------- */
typedef struct {
  int window;         /* beta_m: masked-window rows per sequence          */
  int track_budget;   /* beta_t: tracked rows per sequence                 */
  int max_search;     /* search tokens per sequence (0: no verify forward) */
  float eps;          /* unmask threshold                                  */
  float gamma;        /* acceptance threshold                              */
  int force_progress; /* commit the most confident row when none reaches eps */
  int mask_token;     /* the [MASK] id                                     */
} fdl_flash_params;

typedef struct {
  int B;
  int max_seq;                 /* row stride of tokens / masked (and of the tracker) */
  const int* prompt_len;       /* host [B]                                           */
  const int* seq_len;          /* host [B] N_b <= max_seq                            */
  int* tokens;                 /* host [B*max_seq] in/out: current token ids         */
  unsigned char* masked;       /* host [B*max_seq] in/out: 1 = still masked          */
  int* tracked;                /* host [B*track_budget] in/out: tracked positions     */
  int* n_tracked;              /* host [B] in/out                                     */
  int* state;                  /* host [B] in/out: -1 before the first step           */
} fdl_flash_seqs;

typedef struct {               /* optional record of one step; any pointer may be NULL */
  int* n_rows;                 /* [2]: draft-forward rows, verify-forward rows (0 when none) */
  int* n_window;               /* [1]: window rows R_w                               */
  int* window_seq;             /* [B*window]: each window row's sequence             */
  int* window_pos;             /* [B*window]: and position                           */
  float* conf;                 /* [B*window]: confidence of each window row          */
  int* argmax;                 /* [B*window]: its prediction (the draft token)       */
  unsigned char* commit;       /* [B*window]                                         */
  int* search_rows;            /* [B*max_search]: window-row indices, -1 pad          */
  int* n_search;               /* [B]                                                */
  float* mask_conf;            /* [B*max_search]: the mask views' confidence          */
  int* mask_argmax;            /* [B*max_search]: and prediction                      */
  int* n_accept;               /* [B]                                                */
  float* track;                /* [B*max_seq]: the draft forward's tracker scores     */
  void* draft_final;           /* DEVICE [max_rows, d_model] bf16: the draft forward's
                                  final normed rows, in row order                    */
  void* verify_final;          /* DEVICE [max_rows, d_model] bf16: the verify forward's */
} fdl_flash_trace;

size_t fdl_flash_workspace_bytes(const fdl_ctx* ctx, int ffn, const fdl_flash_params* params, int B,
                                 int max_seq);

fdl_status fdl_flash_step(fdl_ctx* ctx, const fdl_model* model, const void* w_lm, void* const* k_caches,
                          void* const* v_caches, const int* block_table, int bt_stride,
                          const fdl_flash_params* params, fdl_flash_seqs* seqs, fdl_flash_trace* trace,
                          void* workspace, size_t workspace_bytes);

#ifdef __cplusplus
}
#endif
#endif /* FDL_H_ */
