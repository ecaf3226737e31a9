/*
 * lsr.h -- resident-prefix replay attention on one GB300 (sm_103a).
 *
 * What the library computes.  A long prompt is captured once, without
 * autograd, and only its K/V pages are kept resident ("LongStraw 2M RL"
 * explainer, section "The move: change the graph boundary": the resident
 * state is stopgrad(z_p(theta)), kept as model-native KV pages).  Each
 * policy response is then replayed: its query block attends to every prompt
 * key and causally to the response keys, the forward composes per-shard
 * softmax statistics (m, l, O) into the exact output, and the backward
 * returns dQ over prompt+response keys but dK/dV only for response-owned
 * pages, replaying response blocks in reverse and accumulating gradients
 * (explainer, section "Two incompatible architectures, same transaction",
 * the Qwen bullet; "Long-context RL is a state-lifetime problem", sections
 * "Make the prompt resident and the learning graph selective" and
 * "Preserve gradient semantics, not just forward outputs").
 *
 * Conventions shared by every entry point.
 *  - All device memory is owned by the caller.  The library calls no
 *    device allocator and never frees what it is given.  The one exception
 *    is a fixed 64 MiB scratch array in the library's own device memory,
 *    used only by lsr_replay_attn_bwd_noalloc and held by every GPU that
 *    loads the library until the process exits.
 *  - bf16 means IEEE bfloat16 stored as 2 bytes; fp32 is IEEE float.
 *  - Every device pointer must be 16-byte aligned.  Tensors are dense and
 *    row-major in the index order written next to them.
 *  - `stream` is a cudaStream_t cast to void* (NULL = the legacy default
 *    stream).  Every call validates its arguments on the host first and
 *    returns a status without launching anything when they are wrong; the
 *    work itself is asynchronous on `stream`.  A failed launch returns
 *    LSR_ERR_CUDA; an error raised later by a kernel shows up in the pool's
 *    device status word (lsr_pool_device_status) or as LSR_ERR_CUDA on a
 *    later call.
 *  - Logical pages: the prompt occupies logical pages [0, P/page_size) and
 *    the response starts at logical page P/page_size (P must be a multiple
 *    of page_size).  `page_table[i]` is the physical page holding logical
 *    page i; `table_len` is the number of entries the caller provides.
 *  - Query heads map to kv heads in contiguous groups:
 *    kv_head(h) = h / (Hq / Hkv).
 *  - Response query row i of a block starting at response position
 *    `resp_pos0` sees every prompt key and response key j iff
 *    j <= resp_pos0 + i.
 *  - Gradients are accumulated (+=) into caller-zeroed fp32 buffers; they
 *    are never overwritten, so one buffer spans an accumulation window of
 *    several replays.
 *  - No C++ exception crosses this interface.  Error text for the calling
 *    thread's most recent failure is returned by lsr_last_error().
 *  - A latent page pool (lsr_latent.h) is refused by every replay, write
 *    and group entry point here with LSR_ERR_INVALID_ARG.  The scoring
 *    calls (lsr_score_*) take either kind of pool.
 */
#ifndef LSR_H_
#define LSR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LSR_OK = 0,
  LSR_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or combination */
  LSR_ERR_UNSUPPORTED = 2, /* valid but not built (e.g. head_dim 96) */
  LSR_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  LSR_ERR_DEVICE = 4,      /* the device status word reports an error */
  LSR_ERR_STALE = 5,       /* resident state of another model version */
  LSR_ERR_DUPLICATE = 6,   /* replay already counted or in flight */
  LSR_ERR_STATE = 7        /* call not allowed in the window's state */
} lsr_status;

/* Bits of the device status word. */
#define LSR_DEV_WAIT_TIMEOUT 1 /* a bounded in-kernel wait gave up */
#define LSR_DEV_BAD_PAGE 2     /* a page-table entry was out of range */
#define LSR_DEV_BOUNDS 4       /* debug build: an output index failed its
                                  bounds check (the access was skipped) */

typedef struct lsr_pool* lsr_pool_t;
typedef struct lsr_window* lsr_window_t;

/*
 * lsr_page_pool_create -- describe a paged K/V pool (resident state).
 * Explainer, section "The move": the prompt's K/V are kept as pages.
 *  num_pages, page_size, num_kv_heads, head_dim: pool geometry.
 *    head_dim must be 64 or 128; page_size a multiple of 64;
 *    num_pages * num_kv_heads * page_size < 2^31.
 *  k_pages, v_pages: device bf16 [num_pages][num_kv_heads][page_size]
 *    [head_dim], caller-owned, alive while the pool is used.
 *  dev_status: device int32, caller-owned and zeroed; kernels OR
 *    LSR_DEV_* bits into it.
 *  out: receives an opaque host handle (host memory owned by the library,
 *    released by lsr_page_pool_destroy).
 */
lsr_status lsr_page_pool_create(int num_pages, int page_size, int num_kv_heads,
                                int head_dim, void* k_pages, void* v_pages,
                                int* dev_status, lsr_pool_t* out);

/* Release the handle.  Device memory is the caller's and is not touched. */
lsr_status lsr_page_pool_destroy(lsr_pool_t pool);

/*
 * lsr_write_prefix_pages -- scatter T tokens of K/V into the pool.
 * Used for the prompt capture (pos0 = 0, T = P) and for a response's own
 * pages (pos0 = P).  Token t goes to logical position pos0 + t, i.e. row
 * (pos0 + t) % page_size of physical page page_table[(pos0+t)/page_size].
 * The rows after the last written row of the last touched page are set to
 * zero, so a partial last page holds finite values.
 *  k, v: device bf16 [T][num_kv_heads][head_dim].
 *  page_table: device int32 [table_len]; table_len * page_size >= pos0 + T.
 *  Out-of-range entries are skipped and set LSR_DEV_BAD_PAGE.
 */
lsr_status lsr_write_prefix_pages(lsr_pool_t pool, const void* k,
                                  const void* v, int T, int pos0,
                                  const int32_t* page_table, int table_len,
                                  void* stream);

/*
 * lsr_replay_attn_fwd -- per-shard softmax statistics of one response block.
 * Explainer, Qwen bullet: rank-local softmax statistics are composed into
 * the exact global output; here the prompt's logical pages are split into
 * `num_shards` contiguous ranges (shard s holds pages
 * [s*np/num_shards, (s+1)*np/num_shards), np = P/page_size) and partial
 * number num_shards holds the visible response keys.
 *  q: device bf16 [R_b][Hq][head_dim], block rows at response positions
 *     resp_pos0 .. resp_pos0 + R_b - 1.  Hq must be a multiple of Hkv and
 *     Hq/Hkv must divide 128.
 *  P: prompt length (multiple of page_size).  The response keys
 *     0 .. resp_pos0 + R_b - 1 must already be in the pool.
 *  scale: softmax scale applied to q.k (e.g. 1/sqrt(head_dim)).
 *  m, l: device fp32 [num_shards+1][Hq][R_b]: a reference for the row's
 *     scaled logits (natural-log units) and the sum of exp(logit - m)
 *     against it; together they give the partial's log-sum-exp m + ln l.
 *     m is ln 2 times an integer that lies at most 8 below and less than 1
 *     above the row max in log2 units, so l stays within [2^-1, 2^8 n] for
 *     n visible keys.  An empty partial has m = -inf and l = 0.
 *  o_part: device fp32 [num_shards+1][R_b][Hq][head_dim]: the partial
 *     output normalised by its own l (0 when empty).
 */
lsr_status lsr_replay_attn_fwd(lsr_pool_t pool, const void* q, int Hq, int R_b,
                               int P, int resp_pos0, const int32_t* page_table,
                               int table_len, int num_shards, float scale,
                               float* m, float* l, float* o_part,
                               void* stream);

/*
 * lsr_lse_merge -- exact composition of partial statistics.
 * lse = log sum_s exp(m_s + ln l_s);  O = sum_s exp(m_s + ln l_s - lse) O_s.
 *  m, l: device fp32 [num_parts][Hq][R_b]; o_part: [num_parts][R_b][Hq][d].
 *  o: device fp32 [R_b][Hq][d].
 *  lse: device fp32 [Hq][R_b], natural log.
 *  head_dim must be 64 or 128.
 */
lsr_status lsr_lse_merge(const float* m, const float* l, const float* o_part,
                         int num_parts, int Hq, int R_b, int head_dim, float* o,
                         float* lse, void* stream);

/* Bytes of device workspace lsr_replay_attn_bwd needs: the dQ pass splits
 * each prompt shard in two contiguous halves (so that a half's K/V stream
 * fits in L2) and keeps one fp32 dQ slice [R_b][Hq][d] per half plus one
 * for the response keys, 2*num_shards + 1 slices in all, and the row dots
 * D [Hq][R_b]. */
lsr_status lsr_bwd_workspace_size(int num_shards, int Hq, int R_b,
                                  int head_dim, size_t* bytes);

/*
 * lsr_replay_attn_bwd -- response-only backward of one block.
 * The prompt K/V are stop-gradient (explainer, "The move": the direct
 * response gradient is kept and the prompt-side term is dropped), so only
 * dQ (over prompt and response keys) and the response pages' dK/dV are
 * produced; nothing is written for prompt pages (explainer, Qwen bullet:
 * K/V gradient pages exist only where a response backward touches them).
 *  q, dO: device bf16 [R_b][Hq][d]; o: the block's forward output (fp32,
 *     same layout); lse: device fp32 [Hq][R_b] from lsr_lse_merge.
 *  dq: device fp32 [R_b][Hq][d], accumulated (+=).
 *  dk_resp, dv_resp: device fp32 [n_resp_pages][Hkv][page_size][d], one
 *     gradient page per logical response page in logical order
 *     (n_resp_pages >= ceil((resp_pos0 + R_b) / page_size)); accumulated.
 *  workspace: device memory of lsr_bwd_workspace_size bytes (scratch for
 *     per-shard dQ partials and D = rowsum(dO * O)).
 */
lsr_status lsr_replay_attn_bwd(lsr_pool_t pool, const void* q, const float* o,
                               const void* dO, const float* lse, int Hq,
                               int R_b, int P, int resp_pos0,
                               const int32_t* page_table, int table_len,
                               int num_shards, float scale, float* dq,
                               float* dk_resp, float* dv_resp,
                               void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * lsr_replay_attn_bwd_noalloc -- lsr_replay_attn_bwd without a workspace.
 * The pages describe no such call; it exists for callers that cannot
 * allocate device memory where they run the backward (code that must not
 * call cudaMalloc/cudaFree, e.g. under an allocator-enforced memory budget
 * or where an allocation could block or fail, and plain C callers with no
 * device allocator).  Arguments, layouts and results are those of
 * lsr_replay_attn_bwd; the caller still passes every input and output.
 *  Scratch: a fixed 64 MiB array inside the library's device memory, which
 *    every GPU that loads the library holds until the process exits.  A
 *    block is accepted only if lsr_bwd_workspace_size(num_shards, Hq, R_b,
 *    head_dim) <= 64 MiB; larger ones return LSR_ERR_INVALID_ARG with the
 *    sizes in lsr_last_error() and launch nothing.
 *  Set-up: the first call on a device (made with that device current) looks
 *    up the array's device address; make that first call before any stream
 *    capture.
 *  Sharing: all calls share the one array and it keeps the last call's
 *    contents (nothing in it needs to start at zero).  Calls whose work
 *    overlaps on the GPU -- on different streams, or from several threads --
 *    race on the array; serialise them.
 *  No cudaMalloc, cudaFree or allocating library routine is called.
 */
lsr_status lsr_replay_attn_bwd_noalloc(lsr_pool_t pool, const void* q,
                                       const float* o, const void* dO,
                                       const float* lse, int Hq, int R_b,
                                       int P, int resp_pos0,
                                       const int32_t* page_table,
                                       int table_len, int num_shards,
                                       float scale, float* dq, float* dk_resp,
                                       float* dv_resp, void* stream);

/* Bytes of device workspace lsr_replay_response needs. */
lsr_status lsr_replay_workspace_size(int num_shards, int Hq, int R,
                                     int num_blocks, int head_dim,
                                     size_t* bytes);

/*
 * lsr_replay_response -- replay one response as num_blocks blocks, last
 * block first (explainer, Qwen bullet: response blocks are replayed in
 * reverse).  For each block: forward partials, merge, backward; the
 * response dK/dV of every block accumulate.  The response's K/V must
 * already be in the pool (lsr_write_prefix_pages with pos0 = P).
 *  q, dO: device bf16 [R][Hq][d]; o: device fp32 [R][Hq][d] (written);
 *  lse: device fp32 [Hq][R] (written); dq: fp32 [R][Hq][d] (+=);
 *  dk_resp, dv_resp: as in lsr_replay_attn_bwd (+=).
 *  Block b covers rows [b*(R/num_blocks), ...), the last block taking the
 *  remainder.
 */
lsr_status lsr_replay_response(lsr_pool_t pool, const void* q, const void* dO,
                               int Hq, int R, int num_blocks, int P,
                               const int32_t* page_table, int table_len,
                               int num_shards, float scale, float* o,
                               float* lse, float* dq, float* dk_resp,
                               float* dv_resp, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * K concurrent replays ("Long-context RL is a state-lifetime problem",
 * section "Make the prompt resident and the learning graph selective": K
 * responses replayed at once share the resident prompt).  The query rows of
 * num_resp (<= 32) responses are stacked in one tensor and go through one
 * forward (partials + merge) and one backward, so each prompt K/V tile
 * loaded serves all of them.  Each response is replayed whole (one block,
 * positions 0 .. R[k]-1) against its own response pages and causal mask.
 *  lsr_group_rows(Hq, Hkv, num_resp, R, row0): row0[0..num_resp] (host
 *    int) -- response k occupies rows [row0[k], row0[k+1]) of the stacked
 *    tensors, its R[k] real rows first; the rest pad to a pair of query
 *    tiles and must hold zeros in q and dO (their o, lse and dq rows are
 *    unspecified).
 *  R, resp_page0, grad_page0: host int [num_resp].  Response k's key j is
 *    at logical page resp_page0[k] + j/page_size (>= P/page_size; inside the
 *    table) and its dK/dV at gradient page grad_page0[k] + j/page_size of
 *    dk, dv [n_grad_pages][Hkv][page_size][d] (fp32, +=).  The gradient page
 *    ranges of different responses must not overlap.
 *  q, dO: device bf16 [row0[num_resp]][Hq][d]; o fp32 and lse fp32
 *    [Hq][rows] written; dq fp32 [rows][Hq][d] accumulated.
 *  workspace: lsr_group_workspace_size(num_shards, Hq, rows, d) bytes.
 */
lsr_status lsr_group_rows(int Hq, int num_kv_heads, int num_resp,
                          const int* R, int* row0);
lsr_status lsr_group_workspace_size(int num_shards, int Hq, int total_rows,
                                    int head_dim, size_t* bytes);
lsr_status lsr_replay_group(lsr_pool_t pool, int num_resp, const int* R,
                            const int* resp_page0, const int* grad_page0,
                            const void* q, const void* dO, int Hq, int P,
                            const int32_t* page_table, int table_len,
                            int num_shards, float scale, float* o, float* lse,
                            float* dq, float* dk, float* dv, int n_grad_pages,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Versioned identity and the accumulation window ("Long-context RL is a
 * state-lifetime problem", sections "Account for memory by lifetime" and
 * "Preserve gradient semantics, not just forward outputs": resident state
 * has a versioned identity and an invalidation point; compatible replays
 * accumulate until one optimizer step closes the window; retries must not
 * count a gradient twice and failures must not drop one silently; no
 * replay may run against an older model version).  Host-only bookkeeping.
 *  lsr_pool_set_version / lsr_pool_version: tag a pool with the model
 *    version its resident state was captured under (0 at creation).
 *  lsr_window_create(version): an empty window for that model version.
 *  lsr_window_begin_replay(w, resident_version, replay_id): before a
 *    replay's backward.  LSR_ERR_STALE if resident_version differs from
 *    the window's, LSR_ERR_DUPLICATE if replay_id is in flight or already
 *    committed, LSR_ERR_STATE if the window is poisoned.
 *  lsr_window_commit_replay(w, replay_id, n_tokens): after the backward of
 *    that replay finished; counts it (and its tokens) once.
 *  lsr_window_abort_replay(w, replay_id): a replay failed after it began.
 *    Its partial contribution may already be in the gradient buffers (the
 *    backward accumulates in place), so the window becomes poisoned: every
 *    later begin or close returns LSR_ERR_STATE, and the caller discards
 *    the window's gradients and opens a new window.
 *  lsr_window_close(w, next_version, &n_replays, &n_tokens): the optimizer
 *    step.  Fails with LSR_ERR_STATE while replays are in flight or the
 *    window is poisoned; otherwise returns the counted replays and tokens
 *    (the normalisation set), clears the window and moves it to
 *    next_version, after which state of the old version is stale.
 */
lsr_status lsr_pool_set_version(lsr_pool_t pool, uint64_t version);
lsr_status lsr_pool_version(lsr_pool_t pool, uint64_t* version);
lsr_status lsr_window_create(uint64_t model_version, lsr_window_t* out);
lsr_status lsr_window_destroy(lsr_window_t window);
lsr_status lsr_window_begin_replay(lsr_window_t window,
                                   uint64_t resident_version,
                                   uint64_t replay_id);
lsr_status lsr_window_commit_replay(lsr_window_t window, uint64_t replay_id,
                                    long long n_tokens);
lsr_status lsr_window_abort_replay(lsr_window_t window, uint64_t replay_id);
lsr_status lsr_window_close(lsr_window_t window, uint64_t next_version,
                            long long* n_replays, long long* n_tokens);

/*
 * Graph-free scoring (explainer, "The move": old-policy and reference
 * branches are scored without a training graph).  lsr_score_fwd runs the
 * forward partials and the LSE merge and keeps nothing for a backward; the
 * partials live in `workspace` (lsr_score_workspace_size bytes) only for
 * the duration of the call.  Arguments as in lsr_replay_attn_fwd and
 * lsr_lse_merge: q bf16 [R_b][Hq][d]; o fp32 [R_b][Hq][d] and lse fp32
 * [Hq][R_b] are written.  On a latent pool (lsr_latent.h) q is the absorbed
 * query [R_b][Hq][latent_dim + rope_dim], o is [R_b][Hq][latent_dim], and
 * lsr_score_workspace_size takes head_dim = latent_dim.
 * lsr_score_shards picks a prompt shard count that gives every SM at least
 * two CTAs for R_b query rows; with few rows (decoding against the resident
 * prompt) the call is then bound by one read of the prompt's K/V.
 */
lsr_status lsr_score_shards(lsr_pool_t pool, int Hq, int R_b, int P,
                            int* num_shards);
lsr_status lsr_score_workspace_size(int num_shards, int Hq, int R_b,
                                    int head_dim, size_t* bytes);
lsr_status lsr_score_fwd(lsr_pool_t pool, const void* q, int Hq, int R_b,
                         int P, int resp_pos0, const int32_t* page_table,
                         int table_len, int num_shards, float scale, float* o,
                         float* lse, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * lsr_selftest_bounded_wait -- check the bounded in-kernel wait.  The pages
 * describe no such call.  Every pipeline role of the attention kernels waits
 * on mbarriers with a time limit and, when it expires, sets
 * LSR_DEV_WAIT_TIMEOUT instead of spinning forever.  This launches one
 * thread that waits, with limit `limit_us` (1 .. 1e6 microseconds), on a
 * barrier nothing arrives on; afterwards `*dev_status` (device int32) has
 * LSR_DEV_WAIT_TIMEOUT set and the context remains usable.
 */
lsr_status lsr_selftest_bounded_wait(int* dev_status, int limit_us,
                                     void* stream);

/*
 * lsr_pool_set_wait_limit -- limit of the attention kernels' pipeline waits
 * for every later call on this pool (either kind).  The pages describe no
 * such call.  Each pipeline role (copy producer, MMA issuer, softmax and dS
 * warps) waits for the others on mbarriers; a wait that runs past the limit
 * makes the whole CTA give up: it sets LSR_DEV_WAIT_TIMEOUT in the pool's
 * status word, lets its issued copies and products finish, frees its tensor
 * memory and exits, leaving the outputs of that call undefined and the
 * context usable.  limit_us: 1 .. 4000000 microseconds, or 0 for the
 * default of 4 s.  A limit of a few microseconds makes waits run out on
 * purpose, which is how the abort path is tested.  Host-side only; takes
 * effect from the next launch.
 */
lsr_status lsr_pool_set_wait_limit(lsr_pool_t pool, int limit_us);

/*
 * lsr_pool_device_status -- synchronise `stream`, then copy the pool's
 * device status word to *out (0 = no device-side error).  Returns
 * LSR_ERR_DEVICE when the word is non-zero.
 */
lsr_status lsr_pool_device_status(lsr_pool_t pool, int* out, void* stream);

/*
 * Kernel profiling.  Every kernel the library launches is counted; while
 * timing is enabled each launch is also bracketed by two CUDA events
 * recorded on the launch's own stream.  Ids: */
enum {
  LSR_K_WRITE_PAGES = 0,
  LSR_K_ATTN_FWD = 1,
  LSR_K_LSE_MERGE = 2,
  LSR_K_BWD_PREPROCESS = 3,
  LSR_K_ATTN_BWD_DQ = 4,
  LSR_K_DQ_REDUCE = 5,
  LSR_K_ATTN_BWD_DKDV = 6,
  LSR_K_LATENT_BWD_DQ = 7,   /* latent pages (lsr_latent.h) */
  LSR_K_LATENT_BWD_DLAT = 8,
  LSR_K_COUNT = 9
};
/* Turn event timing on (1) or off (0).  Either way the launch counts and
 * the recorded events of every kernel are cleared. */
lsr_status lsr_profile_set(int enable);
/* Launch count and summed event time (ms) of kernel `kernel` since the
 * last lsr_profile_set; waits for the recorded events to complete. */
lsr_status lsr_profile_read(int kernel, long long* launches, double* total_ms);
/* Name of a kernel id ("" if out of range). */
const char* lsr_kernel_name(int kernel);

/* Text of the calling thread's most recent error ("" if none). */
const char* lsr_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* LSR_H_ */
