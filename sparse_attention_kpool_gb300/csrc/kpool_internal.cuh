// kpool_internal.cuh -- shared pieces of the CUDA library: workspace layout,
// the ordered selection key, and the launch wrappers each .cu file provides.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kpool.h"

namespace kpool {

// Query rows handled together by one work item of the tensor-core kernel
// (8 rows x 32 heads = 256 MMA columns).
constexpr int kItemRows = 8;

// ---------------------------------------------------------------- workspace
//
// [header 256 B][pool_off S+1][qblk_off S+1][level_cnt L][level_start L]
// [level_fill L][items N x int2][pooled keys P x d]; every region 256-B aligned.
struct WorkspaceHeader {
  int32_t error;        // kpool_status recorded on the device (0 = OK)
  int32_t n_items;      // work items written by the planning kernel
  int32_t n_levels;     // distinct item depths
  int32_t total_pools;  // P
  int32_t reserved[59];
  int32_t next_item;    // work counter of the tensor-core kernel (reset by the planning kernel)
};
static_assert(sizeof(WorkspaceHeader) == 256, "header is one 256-byte block");

struct WorkspaceLayout {
  size_t header, pool_off, qblk_off, level_cnt, level_start, level_fill, items, pooled, total;
  int64_t max_items, max_levels, max_pools;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WorkspaceLayout workspace_layout(int64_t T, int32_t S, int32_t d, size_t elem_bytes, int32_t kpool) {
  WorkspaceLayout L{};
  L.max_items = (T + kItemRows - 1) / kItemRows + S + 1;
  L.max_levels = (T + kItemRows - 1) / kItemRows + 2;
  L.max_pools = T / kpool;
  size_t off = 0;
  L.header = off;      off = align256(off + sizeof(WorkspaceHeader));
  L.pool_off = off;    off = align256(off + sizeof(int32_t) * size_t(S + 1));
  L.qblk_off = off;    off = align256(off + sizeof(int32_t) * size_t(S + 1));
  L.level_cnt = off;   off = align256(off + sizeof(int32_t) * size_t(L.max_levels));
  L.level_start = off; off = align256(off + sizeof(int32_t) * size_t(L.max_levels));
  L.level_fill = off;  off = align256(off + sizeof(int32_t) * size_t(L.max_levels));
  L.items = off;       off = align256(off + sizeof(int2) * size_t(L.max_items));
  L.pooled = off;      off = align256(off + elem_bytes * size_t(d) * size_t(L.max_pools > 0 ? L.max_pools : 1));
  L.total = off;
  return L;
}

// ------------------------------------------------------------ selection key
//
// A 64-bit key whose unsigned order is the selection order: the high word is
// the score mapped to an order-preserving unsigned integer (sign bit set for
// non-negative scores, all bits flipped for negative ones), the low word is
// the bitwise complement of the pool index (so a smaller index ranks higher on
// equal scores). -0 is folded into +0 first, so the two zeros tie. Finite
// scores never produce the key 0, which therefore marks an empty slot.
__device__ __forceinline__ uint32_t score_order_bits(float s) {
  // x + 0.0f turns -0 into +0 (round to nearest) and leaves every other value as is
  const uint32_t u = __float_as_uint(__fadd_rn(s, 0.0f));
  return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(float s, uint32_t pool) {
  return (uint64_t(score_order_bits(s)) << 32) | uint64_t(~pool);
}

__device__ __forceinline__ uint32_t key_pool(uint64_t key) { return ~uint32_t(key); }

__device__ __forceinline__ float key_score(uint64_t key) {
  uint32_t u = uint32_t(key >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

// Sequence holding global row `row` (cu is nondecreasing, row < cu[S]).
__device__ __forceinline__ int seq_of_row(const int32_t* cu, int S, int64_t row) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (int64_t(__ldg(cu + mid)) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void record_error(WorkspaceHeader* hdr, int code) {
  atomicCAS(&hdr->error, 0, code);
}

// Records a caller's stage event on `stream`. Inside a stream capture it is added
// as an event-record node (cudaEventRecordExternal), so a replayed graph records it
// on every replay and the stage times can be read from graph launches too.
inline cudaError_t record_stage_event(void* ev, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), stream, cudaEventRecordExternal)
             : cudaEventRecord(static_cast<cudaEvent_t>(ev), stream);
}

// ------------------------------------------------------ launch wrappers
// Each returns cudaGetLastError() after enqueueing its kernel on `stream`.

// K0: validates cu_seqlens, writes pool/item offsets and the heavy-first item
// list of the rows [row_begin, row_end); clears the header. One CTA.
cudaError_t launch_plan(const int32_t* cu, int32_t S, int64_t T, int32_t kpool, int64_t row_begin,
                        int64_t row_end, char* ws, const WorkspaceLayout& L, cudaStream_t stream);

// K1: pooled keys [P, d] into `out` (dtype elements).
cudaError_t launch_pool(const void* k, kpool_dtype dtype, const int32_t* cu, int32_t S, int64_t T,
                        int32_t d, int32_t kpool, void* out, const char* ws, const WorkspaceLayout& L,
                        int num_sms, cudaStream_t stream);

// K1, gated: kp[p,c] = sum_j softmax_j(gate[t_j,c]) * (k[t_j,c] + ape[j,c]).
cudaError_t launch_pool_gated(const void* k, const float* gate, const float* ape, kpool_dtype dtype,
                              const int32_t* cu, int32_t S, int64_t T, int32_t d, int32_t kpool, void* out,
                              const char* ws, const WorkspaceLayout& L, int num_sms, cudaStream_t stream);

// K2 (CUDA cores): any supported shape. Selects the global rows [row_begin, row_end);
// output row i is global row row_begin + i.
cudaError_t launch_select_simt(const void* q, const void* kp, const float* w, kpool_dtype dtype,
                               const int32_t* cu, int32_t S, int64_t T, int32_t H, int32_t d, int32_t kpool,
                               int32_t budget, float scale, int64_t row_begin, int64_t row_end, int32_t* out_ids,
                               float* out_scores, char* ws, const WorkspaceLayout& L, int num_sms,
                               cudaStream_t stream);

// K2 (tensor cores): bf16, H = 32, d = 128, budget <= 512. Works through the items the
// planning kernel listed and writes the rows of [row_begin, row_end) only (row i of
// the outputs is global row row_begin + i).
bool select_tc_supported(kpool_dtype dtype, int32_t H, int32_t d, int32_t budget);
cudaError_t launch_select_tc(const void* q, const void* kp, const float* w, const int32_t* cu, int32_t S,
                             int64_t T, int32_t kpool, int32_t budget, float scale, int64_t row_begin,
                             int64_t row_end, int32_t* out_ids, float* out_scores, char* ws,
                             const WorkspaceLayout& L, int grid, cudaStream_t stream);

// Index scores (kpool_index_scores): the score of every (row, pool) pair of the global
// rows [row_begin, row_end) into out_scores [R, ld] (-inf where the pool is not
// eligible), with the same arithmetic as the selection kernel of the same family.
cudaError_t launch_scores_tc(const void* q, const void* kp, const float* w, const int32_t* cu, int64_t T,
                             int32_t kpool, float scale, int64_t row_begin, int64_t row_end, float* out_scores,
                             int64_t ld, char* ws, const WorkspaceLayout& L, int grid, cudaStream_t stream);
cudaError_t launch_scores_simt(const void* q, const void* kp, const float* w, kpool_dtype dtype, const int32_t* cu,
                               int32_t S, int64_t T, int32_t H, int32_t d, int32_t kpool, float scale,
                               int64_t row_begin, int64_t row_end, float* out_scores, int64_t ld, char* ws,
                               const WorkspaceLayout& L, int num_sms, cudaStream_t stream);

// K3: pool ids -> token ids for the global rows [row_begin, row_end) (pool_ids and
// out_tokens hold those rows only). `hdr` may be null; when given, the kernel does
// nothing if the planning kernel recorded an error.
cudaError_t launch_expand(const int32_t* pool_ids, const int32_t* cu, int32_t S, int64_t row_begin,
                          int64_t row_end, int32_t kpool, int32_t budget, int32_t* out_tokens,
                          const WorkspaceHeader* hdr, int num_sms, cudaStream_t stream);

// Selection for explicit query rows against an existing pooled-key cache
// (kpool_rows.cu): workspace layout, shape support and the R0-R2 launches.
struct RowsLayout {
  size_t header, pool_off, info, unit_off, hist, cand_cnt, tie_cnt, cleared_bytes, cand, ties, scores, total;
  int64_t stride;  // floats per row of the score buffer (>= T / kpool, multiple of 4)
};
RowsLayout rows_layout(int32_t R, int64_t T, int32_t S, int32_t kpool);
bool select_rows_supported(kpool_dtype dtype, int32_t H, int32_t d, int32_t budget);
cudaError_t launch_select_rows(const void* q, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                               int32_t R, const void* kp, const int32_t* cu, int32_t S, int64_t T, int32_t kpool,
                               int32_t budget, float scale, int32_t* out_ids, float* out_scores,
                               int32_t* out_tokens, char* ws, const RowsLayout& L, int num_sms, int max_ctas,
                               cudaStream_t stream, void* const* stage_events);

// Every check kpool_select_ex / kpool_select_pooled make before the workspace's:
// options, shape, the row range, pointers and alignment, kernel support (kin is k,
// or the pooled keys). On KPOOL_OK, *use_tc says which score kernel runs and
// [*row_begin, *row_end) which global rows are selected ([0, T) without a row
// range); T = 0 or an empty range passes and needs no further work.
kpool_status select_check_args(const void* q, const void* kin, const float* w, const int32_t* cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                               kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                               const int32_t* out_pool_ids, const int32_t* out_token_ids,
                               const float* out_pool_scores, const kpool_options* options, bool* use_tc,
                               int64_t* row_begin, int64_t* row_end);

// TMA descriptor of a [rows, 128] row-major bf16 matrix read in boxes of 64 columns x
// box_rows rows with 128-byte swizzle (kpool_tmap.cu). False if the driver's encoder is
// unavailable or rejects the arguments (base not 16-byte aligned, too many rows).
bool make_tmap_bf16_k128(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);

// Bounded-wait self test.
cudaError_t launch_wait_selftest(char* ws, int64_t spin_limit, cudaStream_t stream);

}  // namespace kpool
