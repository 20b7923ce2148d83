/*
 * qasc — query-aware sparse KV selection and attention for NVIDIA GB300
 * (sm_103a).  Plain C ABI: device pointers, sizes and a CUDA stream handle;
 * no framework types cross this boundary.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *    library never allocates, frees or retains memory, and keeps no state
 *    between calls other than a per-device cache of attributes.
 *  - Calls are asynchronous: they validate their arguments on the host,
 *    enqueue kernels on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return.  Results are visible after the stream is synchronised.
 *  - On any validation failure the call returns a non-zero qasc_status and
 *    enqueues nothing.  A CUDA launch failure returns QASC_ERR_CUDA.
 *    qasc_last_error() gives a message for the calling thread.
 *  - The size queries (*_workspace_bytes, ts_expand_capacity) apply the
 *    shape and parameter checks of the call they size and return 0, with the
 *    reason in qasc_last_error(), for arguments that call would reject.
 *  - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 *  - All tensor base pointers must be 16-byte aligned; workspaces 256-byte.
 *  - Layouts are dense and row-major in the order written.
 *  - Query head h reads KV head g(h) = h / (Hq / Hkv): consecutive query heads
 *    share a KV head.
 *  - The compiled-in geometry is d = 128 (head dimension) and d_idx = 32
 *    (compressed index width, d/4).  Other values give QASC_ERR_UNSUPPORTED.
 *  - Device-side waits are bounded; a wait that runs out records an error
 *    that qasc_device_error() reports (QASC_ERR_TIMEOUT) instead of hanging.
 *
 * Source definitions are cited by page and section:
 *  [TokenSelect] "論文解説: TokenSelect — 動的トークンレベルKVキャッシュ選択による
 *                長文推論の高速化" (explainer of arXiv 2411.05159).
 *  [SnapKV]      "NeurIPS 2024論文解説: SnapKV — 生成前にKVキャッシュの重要トークンを
 *                選択する手法" (explainer of arXiv 2402.02938).
 *  [TokenButler] "Technische Zusammenfassung: TokenButler" (arXiv 2503.07518).
 */
#ifndef QASC_H_
#define QASC_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define QASC_API __attribute__((visibility("default")))
#else
#define QASC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QASC_OK = 0,
  QASC_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad shape or parameter */
  QASC_ERR_UNSUPPORTED = 2,  /* valid but not compiled in (d, d_idx, group size, GPU other than sm_103a) */
  QASC_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  QASC_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  QASC_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
  QASC_ERR_BAD_TABLE = 6,    /* a kernel met a block-table entry outside the page pool */
  QASC_ERR_INTERNAL = 7      /* a kernel met an index of its own outside its buffer (the access was skipped) */
} qasc_status;

/* Cache geometry.  n = tokens currently valid (rows 0..n-1); n_cap = row
 * capacity, i.e. the token stride of K, V and the index.  1 <= n <= n_cap,
 * n_cap < 2^24, 1 <= B, 1 <= Hkv <= Hq <= 64, Hq % Hkv == 0, B * Hkv <= 65535
 * and B * Hkv * n_cap < 2^31. */
typedef struct {
  int32_t B, Hq, Hkv, d, d_idx;
  int32_t reserved;
  int64_t n, n_cap;
} qasc_shape;

/* TokenSelect decode parameters.
 *   sink  = always-attended leading tokens (page default 4)
 *   local = always-attended trailing tokens (page default 256)
 *   K     = selected tokens from the candidates C = [sink, n - local);
 *           0 <= K <= |C|.  Sink and local are outside this budget.
 *   vmin  = minimum vote V_min >= 1 (page default 1).
 * [TokenSelect] section "Token-Level Selection と Sparse Attention", table of
 * always-included tokens; section "実装のポイント", TokenSelectConfig. */
typedef struct {
  int32_t K, sink, local, vmin;
} qasc_ts_params;

/* SnapKV parameters: c = kept entries per KV head (max_capacity_prompt),
 * window = observation rows w per query head, pool_k = odd pooling width.
 * c >= 1, window >= 1 and pool_k odd >= 1 (else QASC_ERR_INVALID_ARG).
 * [SnapKV] section "実装のポイント", hyper-parameter table (4096 / 32 / 3). */
typedef struct {
  int32_t c, window, pool_k, reserved;
} qasc_snap_params;

/* ---------------------------------------------------------------------------
 * ts_index_append — extend the compressed key index.
 * [TokenSelect] section "Query-Key Dot Product Index": a d' = d/4 key index
 * built incrementally during inference; [TokenButler] section
 * "Kernarchitektur": keys projected by a per-layer matrix into the
 * low-dimensional space.
 *
 *   index[b,g,i,:] = RNE_bf16( sum_e K[b,g,i,e] * W[g,e,:] )  for i in [start, start+count)
 *
 *   K      [B, Hkv, n_cap, d]      bf16, read
 *   W      [Hkv, d, d_idx]         bf16, read
 *   index  [B, Hkv, n_cap, d_idx]  bf16, rows [start, start+count) written
 * 0 <= start, start + count <= n_cap, count >= 0 (0 = no-op).  The rounded
 * value is the bf16 nearest to the exact dot product (ties to even).
 * ------------------------------------------------------------------------- */
QASC_API qasc_status ts_index_append(const qasc_shape* shape, const uint16_t* K, const uint16_t* W,
                            uint16_t* index, int64_t start, int64_t count, void* stream);

/* ---------------------------------------------------------------------------
 * ts_score_vote_select — pick the token set S for one decode step.
 * [TokenSelect] section "Query-Key Dot Product Index", eq. Score_h;
 * section "Voting Mechanism", eq. Vote; section "Token-Level Selection と
 * Sparse Attention", eq. S.
 *
 *   q'_h        = W[g(h)]^T q[b,h,:]                        (fp32)
 *   Score_h(i)  = q'_h . index[b,g(h),i,:] / sqrt(d_idx)    for i in C
 *   theta_h     = K-th largest Score_h(i) over C
 *   Vote(i)     = #{h : Score_h(i) > theta_h}
 *   S           = the K candidates first in the order (Vote desc,
 *                 sum_h Score_h(i) desc, i asc); sel[b,:] = S ascending.
 *
 *   q      [B, Hq, d]              bf16
 *   W      [Hkv, d, d_idx]         bf16
 *   index  [B, Hkv, n_cap, d_idx]  bf16 (rows of C must be valid)
 *   sel    [B, K]                  int32, written (token ids, ascending)
 *   workspace, ws_bytes >= ts_select_workspace_bytes(shape, params)
 * One S per sequence, shared by all heads.  Deterministic: same inputs give
 * the same S.  K == 0 enqueues nothing.
 * ------------------------------------------------------------------------- */
QASC_API size_t ts_select_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params);
QASC_API qasc_status ts_score_vote_select(const qasc_shape* shape, const qasc_ts_params* params,
                                 const uint16_t* q, const uint16_t* W, const uint16_t* index,
                                 int32_t* sel, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ts_sparse_attn — attention over T = sink + S + local.
 * [TokenSelect] section "Token-Level Selection と Sparse Attention",
 * eq. Attention and the always-included token table; section "統合の5
 * ステップ" step 5 (merging the sparse and local outputs: done as an exact
 * log-sum-exp merge of split-K partials, equal to one softmax over T).
 *
 *   out[b,h,:] = sum_{j in T} softmax_j(q[b,h].K[b,g(h),j] / sqrt(d)) V[b,g(h),j,:]
 *   lse[b,h]   = natural-log sum_j exp(q.K_j / sqrt(d))   (optional)
 *
 *   q      [B, Hq, d]           bf16
 *   K, V   [B, Hkv, n_cap, d]   bf16 (rows 0..n-1 valid)
 *   sel    [B, K]               int32, ascending, each in C (as written by
 *                               ts_score_vote_select; not re-validated)
 *   out    [B, Hq, d]           fp32, written
 *   lse    [B, Hq]              fp32, written if non-NULL
 *   workspace, ws_bytes >= ts_attn_workspace_bytes(shape, params)
 * ------------------------------------------------------------------------- */
QASC_API size_t ts_attn_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params);
QASC_API qasc_status ts_sparse_attn(const qasc_shape* shape, const qasc_ts_params* params,
                           const uint16_t* q, const uint16_t* K, const uint16_t* V,
                           const int32_t* sel, float* out, float* lse,
                           void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ts_score_select_per_head — one token set per KV head, without voting.
 * [TokenSelect] section "Ablation" (table アブレーション, "w/o Voting": an
 * independent selection per head); scores as in section "Query-Key Dot
 * Product Index", eq. Score_h.  Reading for GQA: KV head g ranks the
 * candidates C by the sum of its Gq query heads' scores (its own score when
 * Gq = 1), ties to the lower token index, and keeps the K best.
 *
 *   G_g(i)   = sum over h in group g of Score_h(i),  i in C
 *   S[b,g]   = the K candidates with the largest G_g, ascending
 *
 *   q, W, index as for ts_score_vote_select; params->vmin is ignored
 *   sel    [B, Hkv, K]          int32, written (ascending per (b, g))
 *   workspace, ws_bytes >= ts_head_select_workspace_bytes(shape, params)
 * Errors as for ts_score_vote_select; K = 0 returns QASC_OK without work.
 * ------------------------------------------------------------------------- */
QASC_API size_t ts_head_select_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params);
QASC_API qasc_status ts_score_select_per_head(const qasc_shape* shape, const qasc_ts_params* params,
                                              const uint16_t* q, const uint16_t* W, const uint16_t* index,
                                              int32_t* sel, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ts_sparse_attn_per_head — ts_sparse_attn with one selected set per KV
 * head: every query head of group g attends to sink + S[b,g] + local.
 *
 *   sel    [B, Hkv, K]          int32, ascending per (b, g), each in C (as
 *                               written by ts_score_select_per_head)
 *   other arguments, the workspace size (ts_attn_workspace_bytes) and the
 *   errors as for ts_sparse_attn.
 * ------------------------------------------------------------------------- */
QASC_API qasc_status ts_sparse_attn_per_head(const qasc_shape* shape, const qasc_ts_params* params,
                                             const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                             const int32_t* sel, float* out, float* lse, void* workspace,
                                             size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ts_expand_neighbors — grow selected sets by their neighbours.
 * [TokenButler] section "Optimierungen" (selected tokens expanded to their
 * spatial neighbours; a prediction interval reuses one selection for several
 * steps); [SnapKV] section "Top-k Selection と Cluster-based Retention", eq.
 * S_final (union of {j - k, ..., j + k} over the selected j).  Reading for
 * the decode step: the union is clipped to the candidates C.
 *
 *   S'[r] = ascending union over j in sel[r] of [j - radius, j + radius], within C
 *
 *   rows     number of sets: B for per-sequence sets, B * Hkv for per-KV-head sets
 *   sel      [rows, K]           int32, ascending tokens in [0, n) (normally
 *                                candidates; a token outside C adds its
 *                                neighbours that lie in C)
 *   sel_out  [rows, cap]         int32, written: S'[r] in its first len[r]
 *                                entries, the rest repeat its last entry (c0
 *                                when S'[r] is empty)
 *   len      [rows]              int32, written: |S'[r]|
 *   cap >= ts_expand_capacity(shape, params, radius) = min(|C|, (2 radius + 1) K)
 *   workspace  device, 256-byte aligned, ts_expand_workspace_bytes(shape,
 *            params, rows) bytes (a bitmap of C and a count per 4096
 *            candidates per row), owned by the caller, reusable once the call
 *            has finished on the stream
 * QASC_ERR_INVALID_ARG for rows outside [1, 65535], radius outside
 * [0, 2^20], a smaller cap or bad pointers, QASC_ERR_WORKSPACE for a missing
 * or short workspace, before any launch.  Rows that are not ascending give
 * some set within C (no out-of-range access), not the union.
 * ------------------------------------------------------------------------- */
QASC_API int32_t ts_expand_capacity(const qasc_shape* shape, const qasc_ts_params* params, int32_t radius);
QASC_API size_t ts_expand_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params, int32_t rows);
QASC_API qasc_status ts_expand_neighbors(const qasc_shape* shape, const qasc_ts_params* params, int32_t rows,
                                         const int32_t* sel, int32_t radius, int32_t* sel_out, int32_t cap,
                                         int32_t* len, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ts_sparse_attn_ex — ts_sparse_attn over lists that may be per KV head and
 * may carry lengths (as written by ts_expand_neighbors).
 *
 *   params->K        capacity of each list
 *   sel              [B, K] (sel_per_kv_head == 0) or [B, Hkv, K] (otherwise),
 *                    int32, ascending within the entries in use, each in C
 *   sel_len          NULL (every entry in use), or [B] / [B, Hkv] int32:
 *                    entries in use of each list, clamped to [0, K]; the
 *                    others are masked (they need not be valid tokens)
 *   other arguments, the workspace size (ts_attn_workspace_bytes) and the
 *   errors as for ts_sparse_attn.  Every query head must attend to at least
 *   one token (sink, local or an entry in use).
 * ------------------------------------------------------------------------- */
QASC_API qasc_status ts_sparse_attn_ex(const qasc_shape* shape, const qasc_ts_params* params, const uint16_t* q,
                                       const uint16_t* K, const uint16_t* V, const int32_t* sel,
                                       const int32_t* sel_len, int32_t sel_per_kv_head, float* out, float* lse,
                                       void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Paged cache and circular local buffer.
 * [TokenSelect] section "まとめ" (integration with vLLM's PagedAttention);
 * [TokenButler] section "Inferenzstrategie" (the cache as a sink, a circular
 * buffer of the newest tokens and the important tokens) and "Optimierungen"
 * (keys projected in batches of tokens).  The pages fix no layout; this one:
 *
 *   K_pool, V_pool  [num_pages, Hkv, P, d] bf16; index_pool [num_pages, Hkv, P, d_idx]
 *   block_table     [B, pages_per_seq] int32, device: token t of sequence b is
 *                   row t mod P of pool page block_table[b][t / P]; the index
 *                   uses the same pages.
 *   P               a power of two in [64, 65536]; shape->n_cap must equal
 *                   pages_per_seq * P; num_pages * Hkv * P < 2^31.
 *   ring            optional circular local buffer: K, V [B, Hkv, R, d] bf16,
 *                   token t at slot t mod R, local <= R <= 2^24 (a flush of
 *                   count tokens needs count <= R <= 2^24).
 *
 * Block-table entries are read on the device.  Those of the pages a call
 * touches must lie in [0, num_pages): the voting select reads tokens [0, c1),
 * attention the sink, the listed tokens and (without a ring) the local
 * tokens, the append and the flush the tokens they write.  An entry outside
 * the pool makes the kernel read row 0 of the pool (or skip the write) and
 * record QASC_ERR_BAD_TABLE for qasc_device_error().  Other arguments, the
 * workspaces (ts_select_workspace_bytes, ts_attn_workspace_bytes) and the
 * errors are those of the contiguous calls.  The results equal the
 * contiguous calls' on the same logical cache, bit for bit.
 * ------------------------------------------------------------------------- */
typedef struct {
  const int32_t* block_table;   /* device [B, pages_per_seq] */
  int32_t page_tokens;          /* P */
  int32_t pages_per_seq;
  int64_t num_pages;
} qasc_paged_cache;

typedef struct {
  const uint16_t* K;            /* device [B, Hkv, R, d] bf16 */
  const uint16_t* V;
  int32_t ring_tokens;          /* R */
} qasc_local_ring;

/* ts_index_append over the pool: index rows of tokens [start, start + count)
 * of every sequence from their K rows. */
QASC_API qasc_status ts_index_append_paged(const qasc_shape* shape, const qasc_paged_cache* cache,
                                           const uint16_t* K_pool, const uint16_t* W, uint16_t* index_pool,
                                           int64_t start, int64_t count, void* stream);

/* ts_score_vote_select over the pool's index rows (tokens [0, c1) must be
 * paged in). */
QASC_API qasc_status ts_score_vote_select_paged(const qasc_shape* shape, const qasc_ts_params* params,
                                                const qasc_paged_cache* cache, const uint16_t* q, const uint16_t* W,
                                                const uint16_t* index_pool, int32_t* sel, void* workspace,
                                                size_t ws_bytes, void* stream);

/* ts_score_select_per_head over the pool's index rows (workspace:
 * ts_head_select_workspace_bytes). */
QASC_API qasc_status ts_score_select_per_head_paged(const qasc_shape* shape, const qasc_ts_params* params,
                                                    const qasc_paged_cache* cache, const uint16_t* q,
                                                    const uint16_t* W, const uint16_t* index_pool, int32_t* sel,
                                                    void* workspace, size_t ws_bytes, void* stream);

/* ts_sparse_attn_ex over the pool; with a ring (non-NULL) the local tokens
 * [local_start, n) are read from it and need not be paged in. */
QASC_API qasc_status ts_sparse_attn_paged(const qasc_shape* shape, const qasc_ts_params* params,
                                          const qasc_paged_cache* cache, const qasc_local_ring* ring,
                                          const uint16_t* q, const uint16_t* K_pool, const uint16_t* V_pool,
                                          const int32_t* sel, const int32_t* sel_len, int32_t sel_per_kv_head,
                                          float* out, float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Moves tokens [start, start + count) of every sequence from the ring into
 * their pages: K and V rows copied from slot t mod R, index rows written
 * (the batched key projection).  count <= R; call it before the tokens leave
 * the local window and before their slots are reused. */
QASC_API qasc_status ts_ring_flush(const qasc_shape* shape, const qasc_paged_cache* cache,
                                   const qasc_local_ring* ring, const uint16_t* W, uint16_t* K_pool,
                                   uint16_t* V_pool, uint16_t* index_pool, int64_t start, int64_t count,
                                   void* stream);

/* ---------------------------------------------------------------------------
 * ts_dense_attn — full attention over all n cached tokens: the baseline the
 * TokenSelect page's speed table measures against ([TokenSelect] section
 * "速度性能": attention speed-up relative to full attention at 32K/64K/128K).
 *
 *   out[b,h,:] = sum_{j < n} softmax_j(q[b,h].K[b,g(h),j] / sqrt(d)) V[b,g(h),j,:]
 *   lse[b,h]   = natural-log sum_j exp(q.K_j / sqrt(d))   (optional)
 *
 * Same layouts, kernels and error behaviour as ts_sparse_attn with every
 * token attended (T = [0, n)); requires n >= 1.
 *   workspace, ws_bytes >= ts_dense_attn_workspace_bytes(shape)
 * ------------------------------------------------------------------------- */
QASC_API size_t ts_dense_attn_workspace_bytes(const qasc_shape* shape);
QASC_API qasc_status ts_dense_attn(const qasc_shape* shape, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                   float* out, float* lse, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ts_sparse_attn_noalloc — ts_sparse_attn for callers that cannot allocate.
 * No counterpart on the source pages: a library convenience.  Engines and
 * plugins that only receive input/output buffers, serving runtimes whose
 * memory planner forbids device allocations while requests run, and loops
 * that cannot pay for cudaMalloc's implicit synchronisation cannot supply a
 * workspace.  This call takes the same inputs and writes the same outputs as
 * ts_sparse_attn, but keeps its split-K scratch in a 16 MiB area built into
 * the library (reserved on every GPU that loads it, until the process exits).
 *  - It allocates and frees nothing.
 *  - A shape whose scratch exceeds 16 MiB returns QASC_ERR_WORKSPACE and
 *    enqueues nothing (ts_sparse_attn with a workspace has no such limit).
 *  - The first call on each device looks up the area's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before capturing any stream.  The address is kept for the life of the
 *    process: after cudaDeviceReset (or anything else that destroys and
 *    re-creates the device's primary context) it is stale, so do not call
 *    this entry point again in that process.
 *  - All calls share the area, which keeps the previous call's contents (none
 *    of it needs clearing); calls that can overlap on the GPU race, so
 *    serialise them.
 * ------------------------------------------------------------------------- */
QASC_API qasc_status ts_sparse_attn_noalloc(const qasc_shape* shape, const qasc_ts_params* params,
                                            const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                            const int32_t* sel, float* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * snapkv_compress — prefill-time compaction of one layer's cache.
 * [SnapKV] section "Attention Score計算とPooling", eqs. A and a-bar;
 * section "Top-k SelectionとCluster-based Retention", eq. S; section
 * "アルゴリズム" steps 1-5 (softmax, mean, average pool with padding
 * kernel//2 and stride 1, top-k of min(c, n), sort, gather).
 *
 *   A_h   = softmax_j(q_obs[b,h,r,:] . K[b,g(h),j,:] / sqrt(d)),  j in [0, n)
 *   a_j   = mean of A_h[r, j] over the window rows r and the Gq heads of g
 *   p_j   = (a_{j-k/2} + ... + a_{j+k/2}) / k   (zero padded)
 *   S     = the c' = min(c, n) largest p (ties: lower index), ascending
 *
 *   q_obs  [B, Hq, window, d]       bf16
 *   K, V   [B, Hkv, n_cap, d]       bf16
 *   idx    [B, Hkv, c']             int32, written
 *   K_out, V_out [B, Hkv, c', d]    bf16, written (bit copies of K[S], V[S])
 *   workspace, ws_bytes >= snapkv_workspace_bytes(shape, params)
 * Requires Hq / Hkv * window <= 128 (the window rows of a GQA group form one
 * 128-row tensor-core tile, padded when fewer; a group of 4 heads with
 * w = 32 fills it) and pool_k <= 65; larger values return
 * QASC_ERR_UNSUPPORTED before any launch.
 * ------------------------------------------------------------------------- */
QASC_API size_t snapkv_workspace_bytes(const qasc_shape* shape, const qasc_snap_params* params);
QASC_API qasc_status snapkv_compress(const qasc_shape* shape, const qasc_snap_params* params,
                            const uint16_t* q_obs, const uint16_t* K, const uint16_t* V,
                            int32_t* idx, uint16_t* K_out, uint16_t* V_out,
                            void* workspace, size_t ws_bytes, void* stream);

/* Human-readable name of a status code (static storage). */
QASC_API const char* qasc_status_string(qasc_status status);

/* Message describing the calling thread's most recent failure ("" if none). */
QASC_API const char* qasc_last_error(void);

/* The same message under the name the library's specification first gave it
 * (kept as an alias: both return the same string). */
QASC_API const char* qasc_last_cuda_error(void);

/* Synchronises `stream`, then reports and clears any error a kernel recorded
 * on the current device: QASC_ERR_TIMEOUT for a wait that ran out, else
 * QASC_ERR_BAD_TABLE for a block-table entry outside the pool (the kernel
 * skipped that row's write, or read row 0 of the pool instead), else
 * QASC_ERR_INTERNAL for an index one kernel handed another outside its
 * buffer (the access was skipped; no input can cause it). */
QASC_API qasc_status qasc_device_error(void* stream);

/* Self-test of the failure path shared by every kernel: launches one kernel
 * whose bounded wait (an mbarrier that nothing arrives on) gives up after
 * limit_us microseconds, records the timeout and returns, so that the next
 * qasc_device_error() reports QASC_ERR_TIMEOUT and the context stays usable.
 * QASC_ERR_INVALID_ARG for limit_us outside [1, 2000000]. */
QASC_API qasc_status qasc_selftest_bounded_wait(int32_t limit_us, void* stream);

/* Library version as 10000 * major + 100 * minor + patch. */
QASC_API int32_t qasc_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* QASC_H_ */
