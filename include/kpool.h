/*
 * kpool.h -- C ABI of the GB300 (sm_103a) KPool DSA indexer selection library.
 *
 * The operation (per packed batch of causal sequences):
 *   1. Mean-pool every kpool consecutive index keys of a sequence into one pooled
 *      key ("spark_model/layers/glm5next_dsa/tp.rs", module docs, "Why the
 *      indexer is REPLICATED": n_pools = seq / kpool). The pages do not name the
 *      pooling operator; this library reads it as the mean: an fp32 sum in key
 *      order, an IEEE fp32 division by kpool, round-to-nearest-even to the input
 *      dtype.
 *   2. Score every causally eligible (query row t, pool p) pair,
 *         s[t,p] = sum_h w[t,h] * relu(scale * q[t,h,:] . kpool[p,:]),
 *      a plain sum over heads taken before any top-k (same page and section).
 *      A row t (sequence-local) may use the pools p < floor((t+1)/kpool), i.e.
 *      the complete pools whose last key is at or before t.
 *   3. Keep the top budget = index_topk / kpool pools of each row, ordered by
 *      higher score first and then smaller pool index (tp.rs module docs: the
 *      deterministic tiebreak pinned because torch.topk's tie order is
 *      undefined). Rows with fewer eligible pools are padded with -1.
 *   4. Expand the chosen pools to token ids, append the row's own incomplete
 *      trailing pool and apply the causal / varlen mask ("NVIDIA/Megatron-LM
 *      pull request #8299", section "Change": pool expansion, tail append and
 *      mask filtering run on the [batch, sq, budget] pool ids).
 *
 * Sequences arrive packed (THD) with cumulative lengths cu_seqlens, as in the
 * pages' packed-THD tests (Megatron-LM #8299, section "Test plan"); a dense
 * batch [B, sq] is cu_seqlens = {0, sq, 2sq, ...}. Every index the library
 * returns is sequence-local.
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory. Scratch state lives in a caller-provided
 *     workspace of kpool_workspace_bytes() bytes (256-byte aligned).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). The returned status covers host-side validation and launch
 *     errors; errors found on the device (malformed cu_seqlens, a bounded wait
 *     that ran out) are recorded in the workspace and read back with
 *     kpool_last_device_error().
 *   - Validation happens before anything touches the GPU: a call that returns
 *     KPOOL_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE launched nothing.
 *   - Calls that share a workspace must not overlap on the GPU.
 *
 * Layouts (row-major, contiguous):
 *   q          [T, H, d]            dtype   (16-byte aligned)
 *   k          [T, d]               dtype   (16-byte aligned)
 *   w          [T, H]               fp32
 *   cu_seqlens [S + 1]              int32   cu[0] = 0, nondecreasing, cu[S] = T
 *   pool ids   [T, budget]          int32   rank order, -1 padded
 *   token ids  [T, index_topk+kpool] int32  slot j*kpool + r = pool_ids[j]*kpool + r;
 *                                           slots index_topk + r = the row's tail;
 *                                           -1 where empty or masked
 *   pool scores[T, budget]          fp32    score of each chosen pool, -INFINITY on -1 slots
 */
#ifndef KPOOL_H_
#define KPOOL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KPOOL_OK = 0,
  KPOOL_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, kpool < 1,
                                   index_topk % kpool != 0, malformed cu_seqlens */
  KPOOL_ERR_UNSUPPORTED = 2,    /* shape outside what the kernels implement */
  KPOOL_ERR_WORKSPACE = 3,      /* workspace null, misaligned or too small */
  KPOOL_ERR_CUDA = 4,           /* a CUDA runtime/driver call or launch failed */
  KPOOL_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait ran out */
  KPOOL_ERR_INTERNAL = 6        /* a device-side bounds guard fired (a library bug; the
                                   offending write was skipped) */
} kpool_status;

typedef enum { KPOOL_BF16 = 0, KPOOL_F32 = 1 } kpool_dtype;

/* Which score+select kernel kpool_select_ex runs. */
typedef enum {
  KPOOL_SCORE_AUTO = 0,   /* tensor-core kernel when the shape allows, else SIMT */
  KPOOL_SCORE_TC = 1,     /* tcgen05/TMEM kernel: bf16, H = 32, d = 128, budget <= 512 */
  KPOOL_SCORE_SIMT = 2    /* CUDA-core kernel: any H <= 64, d <= 256, budget <= 4096 */
} kpool_score_kernel;

typedef struct {
  int32_t score_kernel;       /* a kpool_score_kernel value */
  int32_t max_ctas;           /* 0: one persistent CTA per SM; > 0: cap (tests vary it) */
  void* const* stage_events;  /* NULL, or 5 cudaEvent_t (created by the caller) that are
                                 recorded on `stream` before the planning kernel and after
                                 the plan, pool, score+select and expand kernels, so a
                                 caller can time each kernel without a profiler; inside a
                                 stream capture they become event-record nodes of the
                                 graph, recorded again on every replay */
  int32_t row_begin;          /* with KPOOL_OPT_ROW_RANGE in flags: the call selects for the */
  int32_t row_end;            /* global rows [row_begin, row_end) only (else both zero)    */
  int32_t flags;              /* 0 or KPOOL_OPT_ROW_RANGE                                   */
  int32_t reserved;           /* must be zero */
} kpool_options;

/*
 * Query-row sharding ("NVIDIA/Megatron-LM pull request #8299", section "Change";
 * "NovaSky-AI/SkyRL pull request #2422", Summary): rows are independent, so a
 * group of G processes can each select a contiguous range of query rows and
 * all-gather the int32 pool ids; expansion then runs on the gathered
 * [T, budget] tensor (kpool_expand). With KPOOL_OPT_ROW_RANGE, kpool_select_ex
 * and kpool_select_pooled take the whole batch's q, k (or pooled keys), w and
 * cu_seqlens but score, select and expand only the global rows
 * [row_begin, row_end), 0 <= row_begin <= row_end <= T. Their outputs then hold
 * R = row_end - row_begin rows: out_pool_ids [R, budget], out_token_ids
 * [R, index_topk + kpool], row i being global row row_begin + i, each exactly
 * as the whole-batch call would write that row. An empty range is a no-op.
 * As on the pages, the sharded path returns no index scores: out_pool_scores
 * must be NULL (else KPOOL_ERR_INVALID_ARG). The workspace size is the
 * whole batch's. kpool_balanced_row_split() gives ranges of equal work.
 */
#define KPOOL_OPT_ROW_RANGE 1

/*
 * Workspace size, in bytes, for a call with these sizes. Pure host arithmetic;
 * never touches the GPU. Returns 0 for arguments kpool_select would reject.
 */
size_t kpool_workspace_bytes(int64_t total_tokens, int32_t num_seqs, int32_t heads, int32_t head_dim,
                             kpool_dtype dtype, int32_t kpool, int32_t index_topk);

/*
 * The whole selection (steps 1-4 above) for one packed batch.
 *   q, k, w, cu_seqlens  inputs as laid out above (device).
 *   scale                the fp32 factor inside the relu (any finite value).
 *   out_pool_ids         [T, budget] int32 (device), written for every row.
 *   out_token_ids        [T, index_topk + kpool] int32 (device), written for every row.
 *   out_pool_scores      [T, budget] fp32 (device) or NULL.
 *   workspace            device scratch of >= kpool_workspace_bytes(...) bytes.
 * T = 0 is a valid no-op. Requires d % 8 == 0 (16-byte rows) and heads >= 1.
 */
kpool_status kpool_select(const void* q, const void* k, const float* w, const int32_t* cu_seqlens,
                          int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                          kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                          int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                          void* workspace, size_t workspace_bytes, void* stream);

/* kpool_select with explicit options (NULL = defaults). */
kpool_status kpool_select_ex(const void* q, const void* k, const float* w, const int32_t* cu_seqlens,
                             int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                             kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                             int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                             void* workspace, size_t workspace_bytes, void* stream,
                             const kpool_options* options);

/*
 * Splits the rows of a packed batch into `parts` contiguous ranges of near-equal
 * work for query-row sharding. cu_seqlens is a HOST array [num_seqs + 1] (as the
 * device one); out_bounds, a HOST array of parts + 1 int32, receives
 * 0 = b[0] <= b[1] <= ... <= b[parts] = T, range g being rows [b[g], b[g+1]).
 * A row's work is its causal pair count floor((t+1)/kpool) (t sequence-local)
 * plus row_weight (the per-row cost of ranking, in pair units; 0 balances pairs
 * alone). The split minimises nothing globally: boundary g is the first row at
 * which the running work reaches g/parts of the total, so every range's work is
 * within one row's work of an equal share. The pages split rows evenly
 * (rank r takes rows [r*ceil(sq/G), ...)); under the causal mask that gives the
 * last rank about 2G-1 times the first rank's pairs, which this split avoids.
 * Pure host code; returns KPOOL_ERR_INVALID_ARG for malformed cu_seqlens,
 * kpool < 1, parts < 1 or row_weight < 0.
 */
kpool_status kpool_balanced_row_split(const int32_t* cu_seqlens, int32_t num_seqs, int32_t kpool,
                                      int64_t row_weight, int32_t parts, int32_t* out_bounds);

/*
 * Step 1 alone: writes the pooled keys [P, d] (dtype, P = sum_b floor(L_b/kpool),
 * sequences back to back) to out_pooled_keys, which must hold
 * floor(T/kpool) * d elements. Uses the workspace for the per-sequence offsets.
 */
kpool_status kpool_pool_keys(const void* k, const int32_t* cu_seqlens, int32_t num_seqs,
                             int64_t total_tokens, int32_t head_dim, kpool_dtype dtype, int32_t kpool,
                             void* out_pooled_keys, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Step 1 with gated pooling instead of the mean. The pages name a per-token,
 * per-channel compress gate (index_kpool_compress_gate, [head_dim, hidden]) and a
 * per-position embedding (index_kpool_compress_ape, [kpool, head_dim]) in the
 * GLM-5.3 DSA shard plan ("spark_model/layers/glm5next_dsa/tp.rs") and pass
 * "gate scores" to the fused top-k ("NVIDIA/Megatron-LM pull request #8299",
 * section "Mechanism"), but give no formula; this library reads them as gated
 * compression:
 *     kp[p,c] = sum_j softmax_j(gate[t_j,c]) * (k[t_j,c] + ape[j,c]),
 * t_j the pool's j-th token, computed in fp32 and rounded to the key dtype. A
 * zero gate and embedding reproduce the mean pooling bit for bit.
 *   gate  [T, d] fp32, 16-byte aligned (the gate scores, already projected from
 *         the hidden state)
 *   ape   [kpool, d] fp32, 16-byte aligned
 * Output and workspace as for kpool_pool_keys. Feed the result to
 * kpool_select_pooled.
 */
kpool_status kpool_pool_keys_gated(const void* k, const float* gate, const float* ape, const int32_t* cu_seqlens,
                                   int32_t num_seqs, int64_t total_tokens, int32_t head_dim, kpool_dtype dtype,
                                   int32_t kpool, void* out_pooled_keys, void* workspace, size_t workspace_bytes,
                                   void* stream);
/*
 * kpool_select_ex for pooled keys the caller already has (from kpool_pool_keys,
 * kpool_pool_keys_gated or a cache): steps 2-4 only. pooled_keys holds
 * floor(T/kpool) * d elements of dtype (the size kpool_pool_keys writes into),
 * the first P rows being the pools of cu_seqlens back to back; it is 16-byte
 * aligned and non-NULL even when no sequence holds a complete pool. Same workspace and
 * options as kpool_select_ex; the stage event after the pooling step is recorded
 * right after the planning one.
 */
kpool_status kpool_select_pooled(const void* q, const void* pooled_keys, const float* w, const int32_t* cu_seqlens,
                                 int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                                 kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                                 int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                                 void* workspace, size_t workspace_bytes, void* stream,
                                 const kpool_options* options);
/*
 * Full index scores, the pages' return_index_scores output ("NVIDIA/Megatron-LM
 * pull request #8299", section "Change": the op can return the index scores,
 * which it computes in row chunks of at most 2 GiB). Writes step 2's score of
 * every (row, pool) pair of a range of query rows instead of selecting:
 *   out_scores  [R, ld] fp32 (device, 4-byte aligned), R = row_end - row_begin:
 *               element (i, p), row i being global row row_begin + i (position t
 *               of its sequence), is s[t,p] for the sequence's pool p when
 *               p < floor((t+1)/kpool), and -INFINITY for every other p < ld.
 *   ld          row stride in elements, >= 1. Every row of the range needs
 *               ld >= floor((t+1)/kpool) (ld = floor(T/kpool) always suffices);
 *               a row that is wider keeps its first ld scores and the call records
 *               KPOOL_ERR_INVALID_ARG on the device (kpool_last_device_error).
 *   options     as for kpool_select_ex: KPOOL_OPT_ROW_RANGE picks the rows (the
 *               whole batch without it), so a caller bounds memory by calling once
 *               per chunk of rows; score_kernel picks the family, and the scores
 *               are bit-identical to the out_pool_scores a kpool_select_ex call with
 *               the same score kernel returns for the pools it selects.
 * q, k, w, cu_seqlens, the shape arguments, scale and the workspace are those of
 * kpool_select (workspace: kpool_workspace_bytes(T, S, H, d, dtype, kpool, 0)).
 * Supported shapes: the tensor-core kernel for bf16, H = 32, d = 128; the SIMT
 * kernel for H <= 64, d <= 256. The 4th and 5th stage events are both recorded
 * after the score kernel. An empty range or T = 0 is a no-op.
 */
kpool_status kpool_index_scores(const void* q, const void* k, const float* w, const int32_t* cu_seqlens,
                                int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                                kpool_dtype dtype, int32_t kpool, float scale, float* out_scores, int64_t ld,
                                void* workspace, size_t workspace_bytes, void* stream,
                                const kpool_options* options);

/* kpool_index_scores for pooled keys the caller already has (as kpool_select_pooled). */
kpool_status kpool_index_scores_pooled(const void* q, const void* pooled_keys, const float* w,
                                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                       int32_t heads, int32_t head_dim, kpool_dtype dtype, int32_t kpool, float scale,
                                       float* out_scores, int64_t ld, void* workspace, size_t workspace_bytes,
                                       void* stream, const kpool_options* options);

/*
 * Step 4 alone: expands pool ids [T, budget] (as kpool_select writes them) into
 * token ids [T, index_topk + kpool], appending each row's tail and applying the
 * causal/varlen mask. Ids outside [0, floor((t+1)/kpool)) are treated as -1.
 */
kpool_status kpool_expand(const int32_t* pool_ids, const int32_t* cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, int32_t kpool, int32_t index_topk,
                          int32_t* out_token_ids, void* stream);

/*
 * Selection for an explicit set of query rows against pooled keys that already
 * exist: the decode / short-query case, where a few new query tokens score a
 * long pooled-key cache ("spark_model/layers/glm5next_dsa/tp.rs", module docs,
 * "Why the indexer is REPLICATED": at a 262,144-token context one decode token
 * scores n_pools = 65,536 pools). Row r sits at sequence-local position
 * row_pos[r] of sequence row_seq[r] of the key batch described by cu_seqlens,
 * and gets exactly what row row_pos[r] of kpool_select would get for a query
 * q[r] with weights w[r]: the top budget of the pools p < floor((t+1)/kpool) of
 * its sequence (higher score, then smaller pool index), -1 padded, rank order,
 * expanded to token ids with its incomplete trailing pool appended.
 *   q               [R, H, d] dtype (16-byte aligned); row r is that row's query.
 *   w               [R, H] fp32.
 *   row_seq, row_pos [R] int32 (device): 0 <= row_seq < S, 0 <= row_pos < L_b.
 *   pooled_keys     [P, d] dtype, as kpool_pool_keys writes them for cu_seqlens
 *                   (16-byte aligned; may be NULL only when T / kpool == 0).
 *   cu_seqlens      [S + 1] int32 of the key sequences, as for kpool_pool_keys.
 *   out_pool_ids    [R, budget] int32; out_token_ids [R, index_topk + kpool] int32;
 *   out_pool_scores [R, budget] fp32 or NULL.
 *   workspace       >= kpool_rows_workspace_bytes(R, T, S, kpool, index_topk) bytes.
 * Supported: bf16, H = 32, d = 128, budget <= 512 (else KPOOL_ERR_UNSUPPORTED).
 * R = 0 is a valid no-op. A row whose row_seq or row_pos is out of range gets
 * all -1 outputs and the call records KPOOL_ERR_INVALID_ARG on the device
 * (kpool_last_device_error); malformed cu_seqlens records the same and every
 * row gets -1 outputs. The call allocates and synchronises nothing, so a decode
 * loop can capture it into a CUDA graph; its second to fourth kernels are
 * launched with programmatic stream serialization (each waits on the device for
 * the one before it).
 */
size_t kpool_rows_workspace_bytes(int32_t num_rows, int64_t total_tokens, int32_t num_seqs, int32_t kpool,
                                  int32_t index_topk);
kpool_status kpool_select_rows(const void* q, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                               int32_t num_rows, const void* pooled_keys, const int32_t* cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                               kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                               int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                               void* workspace, size_t workspace_bytes, void* stream);
/*
 * kpool_select_rows with options (NULL = defaults). score_kernel must be
 * KPOOL_SCORE_AUTO; max_ctas > 0 caps the score kernel's grid (CTAs); stage_events, when
 * not NULL, holds 4 cudaEvent_t recorded on `stream` before the planning kernel
 * and after the planning, score and select kernels (event-record nodes when the
 * stream is being captured into a graph).
 */
kpool_status kpool_select_rows_ex(const void* q, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                                  int32_t num_rows, const void* pooled_keys, const int32_t* cu_seqlens,
                                  int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                                  kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                                  int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                                  void* workspace, size_t workspace_bytes, void* stream,
                                  const kpool_options* options);

/*
 * Synchronises `stream`, then reads the device error word the last call on this
 * workspace recorded: KPOOL_OK, KPOOL_ERR_INVALID_ARG (malformed cu_seqlens),
 * KPOOL_ERR_DEVICE_TIMEOUT (a bounded wait ran out), KPOOL_ERR_INTERNAL (a
 * bounds guard fired), or KPOOL_ERR_CUDA if the synchronisation or copy failed.
 */
kpool_status kpool_last_device_error(const void* workspace, void* stream);

/*
 * Exercises the bounded device-side wait used by the pipelined kernel: one CTA
 * waits on a barrier that nothing ever completes, gives up after
 * `spin_limit` polls, records KPOOL_ERR_DEVICE_TIMEOUT in the workspace error
 * word and returns. No fault, trap or hang is involved. Asynchronous; read the
 * result with kpool_last_device_error().
 */
kpool_status kpool_wait_timeout_selftest(void* workspace, size_t workspace_bytes, int64_t spin_limit,
                                         void* stream);

/*
 * Capacity of the library's built-in scratch array used by
 * kpool_select_static_scratch: 48 MiB, enough for one batch of about 750,000
 * tokens at kpool 4, d 128, bf16 (kpool_workspace_bytes() <= this value).
 */
#define KPOOL_STATIC_SCRATCH_BYTES ((size_t)48 << 20)

/*
 * kpool_select for callers that cannot allocate device memory. The pages have
 * no counterpart to this entry point; it exists for callers such as a plugin or
 * custom operator inside a framework that owns all device memory, or a
 * real-time path that must never pay cudaMalloc's implicit synchronisation,
 * which have no workspace to pass. It runs the same kernels as kpool_select with
 * the scratch taken from a file-scope __device__ array of
 * KPOOL_STATIC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits. Inputs and outputs are still the caller's device buffers.
 *   - The arguments are checked as kpool_select checks them, so a shape the
 *     kernels do not implement returns KPOOL_ERR_UNSUPPORTED at any size. Only a
 *     call that passes those checks and whose kpool_workspace_bytes(...) exceeds
 *     KPOOL_STATIC_SCRATCH_BYTES returns KPOOL_ERR_WORKSPACE (split the batch),
 *     before any GPU work.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and caches it: make that first call before any
 *     stream capture.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents: calls that overlap on the GPU race and must be serialised.
 *   - It allocates nothing (no cudaMalloc/cudaFree or allocating library call).
 *   - Errors found on the device (malformed cu_seqlens, which leaves the outputs
 *     unwritten as with kpool_select; a bounded wait that ran out) land in the
 *     shared array's header: read them with
 *     kpool_static_scratch_last_device_error().
 */
kpool_status kpool_select_static_scratch(const void* q, const void* k, const float* w,
                                         const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                         int32_t heads, int32_t head_dim, kpool_dtype dtype, int32_t kpool,
                                         int32_t index_topk, float scale, int32_t* out_pool_ids,
                                         int32_t* out_token_ids, float* out_pool_scores, void* stream);

/*
 * kpool_last_device_error for kpool_select_static_scratch: synchronises `stream`,
 * then returns the device error word the last call on this device's built-in
 * scratch array recorded (KPOOL_OK, KPOOL_ERR_INVALID_ARG for malformed
 * cu_seqlens, KPOOL_ERR_DEVICE_TIMEOUT, KPOOL_ERR_INTERNAL), or KPOOL_ERR_CUDA if
 * the look-up, synchronisation or copy failed. Allocates nothing.
 */
kpool_status kpool_static_scratch_last_device_error(void* stream);

/* Static, human-readable name of a status code. */
const char* kpool_status_string(kpool_status status);

/*
 * Name of the CUDA error behind the most recent KPOOL_ERR_CUDA returned to the
 * calling host thread ("cudaSuccess" if none). Static string; never touches the GPU.
 */
const char* kpool_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KPOOL_H_ */
