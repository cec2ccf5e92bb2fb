// kpool_api.cu -- the C ABI declared in include/kpool.h: argument validation,
// workspace carve-up and the launch sequence K0 plan -> K1 pool -> K2 score +
// select -> K3 expand on the caller's stream. Nothing here allocates device
// memory or synchronises, except kpool_last_device_error (documented to sync).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kpool_internal.cuh"
#include "kpool_ptx.cuh"

namespace kpool {
namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// Remembers a failing CUDA call for kpool_last_cuda_error and maps it to a status.
bool cuda_ok(cudaError_t e) {
  if (e == cudaSuccess) return true;
  g_last_cuda_error = e;
  return false;
}

cudaError_t sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) {
    *out = g_sm_count[dev];
    return cudaSuccess;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev] = n;
  *out = n;
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_bytes(kpool_dtype dt) { return dt == KPOOL_BF16 ? 2 : 4; }

// Shape checks shared by every entry point; pointer checks are per entry point.
kpool_status check_shape(int64_t T, int32_t S, int32_t d, kpool_dtype dtype, int32_t kpool) {
  if (T < 0 || T > int64_t(INT32_MAX)) return KPOOL_ERR_INVALID_ARG;
  if (S < 0 || (T > 0 && S < 1)) return KPOOL_ERR_INVALID_ARG;
  if (dtype != KPOOL_BF16 && dtype != KPOOL_F32) return KPOOL_ERR_INVALID_ARG;
  if (kpool < 1 || d < 1) return KPOOL_ERR_INVALID_ARG;
  if ((size_t(d) * elem_bytes(dtype)) % 16 != 0) return KPOOL_ERR_INVALID_ARG;  // 16-byte rows
  return KPOOL_OK;
}

kpool_status check_workspace(const void* ws, size_t bytes, const WorkspaceLayout& L) {
  if (ws == nullptr || !aligned(ws, 256) || bytes < L.total) return KPOOL_ERR_WORKSPACE;
  return KPOOL_OK;
}

__global__ void wait_selftest_kernel(WorkspaceHeader* hdr, int64_t spin_limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  hdr->error = 0;
  ptx::mbar_init(&bar, 1);
  ptx::fence_mbar_init();
  // Nothing ever arrives on `bar`: the bounded wait must give up by itself.
  if (!ptx::mbar_wait_bounded(&bar, 0, spin_limit, 1000000000ull)) record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(char* ws, int64_t spin_limit, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<WorkspaceHeader*>(ws), spin_limit);
  return cudaGetLastError();
}

}  // namespace kpool

using namespace kpool;

extern "C" {

size_t kpool_workspace_bytes(int64_t total_tokens, int32_t num_seqs, int32_t heads, int32_t head_dim,
                             kpool_dtype dtype, int32_t kpool, int32_t index_topk) {
  if (check_shape(total_tokens, num_seqs, head_dim, dtype, kpool) != KPOOL_OK) return 0;
  if (heads < 1 || index_topk < 0 || index_topk % kpool != 0) return 0;
  return workspace_layout(total_tokens, num_seqs, head_dim, elem_bytes(dtype), kpool).total;
}

}  // extern "C"

namespace kpool {

kpool_status select_check_args(const void* q, const void* kin, const float* w, const int32_t* cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                               kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                               const int32_t* out_pool_ids, const int32_t* out_token_ids,
                               const float* out_pool_scores, const kpool_options* options, bool* use_tc,
                               int64_t* row_begin, int64_t* row_end) {
  kpool_options opt{};
  if (options) opt = *options;
  if (opt.reserved != 0 || (opt.flags & ~KPOOL_OPT_ROW_RANGE) != 0) return KPOOL_ERR_INVALID_ARG;
  if (opt.score_kernel < KPOOL_SCORE_AUTO || opt.score_kernel > KPOOL_SCORE_SIMT || opt.max_ctas < 0)
    return KPOOL_ERR_INVALID_ARG;

  kpool_status st = check_shape(total_tokens, num_seqs, head_dim, dtype, kpool);
  if (st != KPOOL_OK) return st;
  if (heads < 1 || index_topk < 0 || index_topk % kpool != 0 || !isfinite(scale)) return KPOOL_ERR_INVALID_ARG;
  *row_begin = 0;
  *row_end = total_tokens;
  if (opt.flags & KPOOL_OPT_ROW_RANGE) {
    // a shard of query rows; as on the pages, the sharded path returns no index scores
    if (opt.row_begin < 0 || opt.row_begin > opt.row_end || int64_t(opt.row_end) > total_tokens ||
        out_pool_scores != nullptr)
      return KPOOL_ERR_INVALID_ARG;
    *row_begin = opt.row_begin;
    *row_end = opt.row_end;
  } else if (opt.row_begin != 0 || opt.row_end != 0) {
    return KPOOL_ERR_INVALID_ARG;
  }
  const int32_t budget = index_topk / kpool;
  *use_tc = false;
  if (total_tokens == 0 || *row_end == *row_begin) return KPOOL_OK;
  if (!q || !kin || !w || !cu_seqlens || !out_token_ids || (budget > 0 && !out_pool_ids))
    return KPOOL_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kin, 16) || !aligned(w, 4) || !aligned(cu_seqlens, 4) ||
      !aligned(out_pool_ids, 4) || !aligned(out_token_ids, 4) || !aligned(out_pool_scores, 4))
    return KPOOL_ERR_INVALID_ARG;

  const bool tc_ok = select_tc_supported(dtype, heads, head_dim, budget);
  const bool simt_ok = heads <= 64 && head_dim <= 256 && budget <= 4096;
  switch (opt.score_kernel) {
    case KPOOL_SCORE_TC:
      if (!tc_ok) return KPOOL_ERR_UNSUPPORTED;
      *use_tc = true;
      break;
    case KPOOL_SCORE_SIMT:
      if (!simt_ok) return KPOOL_ERR_UNSUPPORTED;
      *use_tc = false;
      break;
    default:
      if (!tc_ok && !simt_ok) return KPOOL_ERR_UNSUPPORTED;
      *use_tc = tc_ok;
  }
  return KPOOL_OK;
}

}  // namespace kpool

namespace {

// The checks of kpool_index_scores(_pooled), in the order of select_check_args.
kpool_status scores_check_args(const void* q, const void* kin, const float* w, const int32_t* cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                               kpool_dtype dtype, int32_t kpool, float scale, const float* out_scores, int64_t ld,
                               const kpool_options* options, bool* use_tc, int64_t* row_begin, int64_t* row_end) {
  kpool_options opt{};
  if (options) opt = *options;
  if (opt.reserved != 0 || (opt.flags & ~KPOOL_OPT_ROW_RANGE) != 0) return KPOOL_ERR_INVALID_ARG;
  if (opt.score_kernel < KPOOL_SCORE_AUTO || opt.score_kernel > KPOOL_SCORE_SIMT || opt.max_ctas < 0)
    return KPOOL_ERR_INVALID_ARG;
  kpool_status st = check_shape(total_tokens, num_seqs, head_dim, dtype, kpool);
  if (st != KPOOL_OK) return st;
  if (heads < 1 || ld < 1 || !isfinite(scale)) return KPOOL_ERR_INVALID_ARG;
  *row_begin = 0;
  *row_end = total_tokens;
  if (opt.flags & KPOOL_OPT_ROW_RANGE) {
    if (opt.row_begin < 0 || opt.row_begin > opt.row_end || int64_t(opt.row_end) > total_tokens)
      return KPOOL_ERR_INVALID_ARG;
    *row_begin = opt.row_begin;
    *row_end = opt.row_end;
  } else if (opt.row_begin != 0 || opt.row_end != 0) {
    return KPOOL_ERR_INVALID_ARG;
  }
  *use_tc = false;
  if (total_tokens == 0 || *row_end == *row_begin) return KPOOL_OK;
  if ((*row_end - *row_begin) > INT64_MAX / ld) return KPOOL_ERR_INVALID_ARG;  // R * ld elements
  if (!q || !kin || !w || !cu_seqlens || !out_scores) return KPOOL_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kin, 16) || !aligned(w, 4) || !aligned(cu_seqlens, 4) || !aligned(out_scores, 4))
    return KPOOL_ERR_INVALID_ARG;
  const bool tc_ok = select_tc_supported(dtype, heads, head_dim, 1);
  const bool simt_ok = heads <= 64 && head_dim <= 256;
  switch (opt.score_kernel) {
    case KPOOL_SCORE_TC:
      if (!tc_ok) return KPOOL_ERR_UNSUPPORTED;
      *use_tc = true;
      break;
    case KPOOL_SCORE_SIMT:
      if (!simt_ok) return KPOOL_ERR_UNSUPPORTED;
      break;
    default:
      if (!tc_ok && !simt_ok) return KPOOL_ERR_UNSUPPORTED;
      *use_tc = tc_ok;
  }
  return KPOOL_OK;
}

// Index scores; pools k itself when `pooled_in` is null, else uses the caller's pooled keys.
kpool_status scores_impl(const void* q, const void* k, const void* pooled_in, const float* w,
                         const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t heads,
                         int32_t head_dim, kpool_dtype dtype, int32_t kpool, float scale, float* out_scores,
                         int64_t ld, void* workspace, size_t workspace_bytes, void* stream_ptr,
                         const kpool_options* options) {
  bool use_tc = false;
  int64_t rb = 0, re = 0;
  kpool_status st = scores_check_args(q, pooled_in ? pooled_in : k, w, cu_seqlens, num_seqs, total_tokens, heads,
                                      head_dim, dtype, kpool, scale, out_scores, ld, options, &use_tc, &rb, &re);
  if (st != KPOOL_OK) return st;
  const int64_t T = total_tokens;
  if (T == 0 || re == rb) return KPOOL_OK;
  kpool_options opt{};
  if (options) opt = *options;
  const WorkspaceLayout L = workspace_layout(T, num_seqs, head_dim, elem_bytes(dtype), kpool);
  st = check_workspace(workspace, workspace_bytes, L);
  if (st != KPOOL_OK) return st;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int sms = 0;
  if (!cuda_ok(sm_count(&sms))) return KPOOL_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  const void* pooled = pooled_in ? pooled_in : static_cast<const void*>(ws + L.pooled);
  void* const* ev = opt.stage_events;
  auto mark = [&](int i) {
    return ev == nullptr || cuda_ok(record_stage_event(ev[i], stream));
  };
  if (!mark(0)) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_plan(cu_seqlens, num_seqs, T, kpool, rb, re, ws, L, stream)) || !mark(1)) return KPOOL_ERR_CUDA;
  if (!pooled_in &&
      !cuda_ok(launch_pool(k, dtype, cu_seqlens, num_seqs, T, head_dim, kpool, ws + L.pooled, ws, L, sms, stream)))
    return KPOOL_ERR_CUDA;
  if (!mark(2)) return KPOOL_ERR_CUDA;
  cudaError_t e;
  if (use_tc) {
    int grid = sms;
    if (opt.max_ctas > 0 && opt.max_ctas < grid) grid = opt.max_ctas;
    e = launch_scores_tc(q, pooled, w, cu_seqlens, T, kpool, scale, rb, re, out_scores, ld, ws, L, grid, stream);
  } else {
    e = launch_scores_simt(q, pooled, w, dtype, cu_seqlens, num_seqs, T, heads, head_dim, kpool, scale, rb, re,
                           out_scores, ld, ws, L, opt.max_ctas > 0 ? opt.max_ctas : sms, stream);
  }
  if (!cuda_ok(e) || !mark(3) || !mark(4)) return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

// The whole selection; pools k itself when `pooled_in` is null, else scores the
// caller's pooled keys (k unused).
kpool_status select_impl(const void* q, const void* k, const void* pooled_in, const float* w,
                         const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t heads,
                         int32_t head_dim, kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                         int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores, void* workspace,
                         size_t workspace_bytes, void* stream_ptr, const kpool_options* options) {
  const void* kin = pooled_in ? pooled_in : k;
  bool use_tc = false;
  int64_t rb = 0, re = 0;
  kpool_status st = select_check_args(q, kin, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool,
                                      index_topk, scale, out_pool_ids, out_token_ids, out_pool_scores, options,
                                      &use_tc, &rb, &re);
  if (st != KPOOL_OK) return st;
  const int64_t T = total_tokens;
  if (T == 0 || re == rb) return KPOOL_OK;
  kpool_options opt{};
  if (options) opt = *options;
  const int32_t budget = index_topk / kpool;

  const WorkspaceLayout L = workspace_layout(T, num_seqs, head_dim, elem_bytes(dtype), kpool);
  st = check_workspace(workspace, workspace_bytes, L);
  if (st != KPOOL_OK) return st;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int sms = 0;
  if (!cuda_ok(sm_count(&sms))) return KPOOL_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  const void* pooled = pooled_in ? pooled_in : static_cast<const void*>(ws + L.pooled);

  void* const* ev = opt.stage_events;
  auto mark = [&](int i) {
    return ev == nullptr || cuda_ok(record_stage_event(ev[i], stream));
  };
  if (!mark(0)) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_plan(cu_seqlens, num_seqs, T, kpool, rb, re, ws, L, stream)) || !mark(1)) return KPOOL_ERR_CUDA;
  if (!pooled_in &&
      !cuda_ok(launch_pool(k, dtype, cu_seqlens, num_seqs, T, head_dim, kpool, ws + L.pooled, ws, L, sms, stream)))
    return KPOOL_ERR_CUDA;
  if (!mark(2)) return KPOOL_ERR_CUDA;
  if (budget > 0) {
    cudaError_t e;
    if (use_tc) {
      int grid = sms;
      if (opt.max_ctas > 0 && opt.max_ctas < grid) grid = opt.max_ctas;
      e = launch_select_tc(q, pooled, w, cu_seqlens, num_seqs, T, kpool, budget, scale, rb, re, out_pool_ids,
                           out_pool_scores, ws, L, grid, stream);
    } else {
      e = launch_select_simt(q, pooled, w, dtype, cu_seqlens, num_seqs, T, heads, head_dim, kpool, budget, scale, rb,
                             re, out_pool_ids, out_pool_scores, ws, L, opt.max_ctas > 0 ? opt.max_ctas : sms,
                             stream);
    }
    if (!cuda_ok(e)) return KPOOL_ERR_CUDA;
  }
  if (!mark(3)) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_expand(out_pool_ids, cu_seqlens, num_seqs, rb, re, kpool, budget, out_token_ids,
                             reinterpret_cast<const WorkspaceHeader*>(ws + L.header), sms, stream)) ||
      !mark(4))
    return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

}  // namespace

extern "C" {

kpool_status kpool_select_ex(const void* q, const void* k, const float* w, const int32_t* cu_seqlens,
                             int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                             kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                             int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                             void* workspace, size_t workspace_bytes, void* stream_ptr,
                             const kpool_options* options) {
  return select_impl(q, k, nullptr, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool,
                     index_topk, scale, out_pool_ids, out_token_ids, out_pool_scores, workspace, workspace_bytes,
                     stream_ptr, options);
}

kpool_status kpool_select_pooled(const void* q, const void* pooled_keys, const float* w, const int32_t* cu_seqlens,
                                 int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                                 kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                                 int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                                 void* workspace, size_t workspace_bytes, void* stream_ptr,
                                 const kpool_options* options) {
  return select_impl(q, nullptr, pooled_keys, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool,
                     index_topk, scale, out_pool_ids, out_token_ids, out_pool_scores, workspace, workspace_bytes,
                     stream_ptr, options);
}

kpool_status kpool_index_scores(const void* q, const void* k, const float* w, const int32_t* cu_seqlens,
                                int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                                kpool_dtype dtype, int32_t kpool, float scale, float* out_scores, int64_t ld,
                                void* workspace, size_t workspace_bytes, void* stream,
                                const kpool_options* options) {
  return scores_impl(q, k, nullptr, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool, scale,
                     out_scores, ld, workspace, workspace_bytes, stream, options);
}

kpool_status kpool_index_scores_pooled(const void* q, const void* pooled_keys, const float* w,
                                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                       int32_t heads, int32_t head_dim, kpool_dtype dtype, int32_t kpool, float scale,
                                       float* out_scores, int64_t ld, void* workspace, size_t workspace_bytes,
                                       void* stream, const kpool_options* options) {
  return scores_impl(q, nullptr, pooled_keys, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool,
                     scale, out_scores, ld, workspace, workspace_bytes, stream, options);
}

kpool_status kpool_select(const void* q, const void* k, const float* w, const int32_t* cu_seqlens,
                          int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                          kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                          int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return kpool_select_ex(q, k, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool, index_topk,
                         scale, out_pool_ids, out_token_ids, out_pool_scores, workspace, workspace_bytes, stream,
                         nullptr);
}

kpool_status kpool_pool_keys(const void* k, const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                             int32_t head_dim, kpool_dtype dtype, int32_t kpool, void* out_pooled_keys,
                             void* workspace, size_t workspace_bytes, void* stream_ptr) {
  kpool_status st = check_shape(total_tokens, num_seqs, head_dim, dtype, kpool);
  if (st != KPOOL_OK) return st;
  if (total_tokens == 0) return KPOOL_OK;
  if (!k || !cu_seqlens || (total_tokens / kpool > 0 && !out_pooled_keys)) return KPOOL_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(out_pooled_keys, 16) || !aligned(cu_seqlens, 4)) return KPOOL_ERR_INVALID_ARG;
  const WorkspaceLayout L = workspace_layout(total_tokens, num_seqs, head_dim, elem_bytes(dtype), kpool);
  st = check_workspace(workspace, workspace_bytes, L);
  if (st != KPOOL_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int sms = 0;
  if (!cuda_ok(sm_count(&sms))) return KPOOL_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  // pooling needs the checked bounds and the pool offsets only: an empty row range
  // leaves the work list empty
  if (!cuda_ok(launch_plan(cu_seqlens, num_seqs, total_tokens, kpool, 0, 0, ws, L, stream))) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_pool(k, dtype, cu_seqlens, num_seqs, total_tokens, head_dim, kpool, out_pooled_keys, ws, L,
                           sms, stream)))
    return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

kpool_status kpool_pool_keys_gated(const void* k, const float* gate, const float* ape, const int32_t* cu_seqlens,
                                   int32_t num_seqs, int64_t total_tokens, int32_t head_dim, kpool_dtype dtype,
                                   int32_t kpool, void* out_pooled_keys, void* workspace, size_t workspace_bytes,
                                   void* stream_ptr) {
  kpool_status st = check_shape(total_tokens, num_seqs, head_dim, dtype, kpool);
  if (st != KPOOL_OK) return st;
  if (total_tokens == 0) return KPOOL_OK;
  if (!k || !gate || !ape || !cu_seqlens || (total_tokens / kpool > 0 && !out_pooled_keys))
    return KPOOL_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(out_pooled_keys, 16) || !aligned(gate, 16) || !aligned(ape, 16) ||
      !aligned(cu_seqlens, 4))
    return KPOOL_ERR_INVALID_ARG;
  const WorkspaceLayout L = workspace_layout(total_tokens, num_seqs, head_dim, elem_bytes(dtype), kpool);
  st = check_workspace(workspace, workspace_bytes, L);
  if (st != KPOOL_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int sms = 0;
  if (!cuda_ok(sm_count(&sms))) return KPOOL_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  if (!cuda_ok(launch_plan(cu_seqlens, num_seqs, total_tokens, kpool, 0, 0, ws, L, stream))) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_pool_gated(k, gate, ape, dtype, cu_seqlens, num_seqs, total_tokens, head_dim, kpool,
                                 out_pooled_keys, ws, L, sms, stream)))
    return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

kpool_status kpool_expand(const int32_t* pool_ids, const int32_t* cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, int32_t kpool, int32_t index_topk, int32_t* out_token_ids,
                          void* stream_ptr) {
  if (total_tokens < 0 || total_tokens > int64_t(INT32_MAX) || num_seqs < 0 || (total_tokens > 0 && num_seqs < 1))
    return KPOOL_ERR_INVALID_ARG;
  if (kpool < 1 || index_topk < 0 || index_topk % kpool != 0) return KPOOL_ERR_INVALID_ARG;
  if (total_tokens == 0) return KPOOL_OK;
  const int32_t budget = index_topk / kpool;
  if (!cu_seqlens || !out_token_ids || (budget > 0 && !pool_ids)) return KPOOL_ERR_INVALID_ARG;
  if (!aligned(pool_ids, 4) || !aligned(out_token_ids, 4) || !aligned(cu_seqlens, 4)) return KPOOL_ERR_INVALID_ARG;
  int sms = 0;
  if (!cuda_ok(sm_count(&sms))) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_expand(pool_ids, cu_seqlens, num_seqs, 0, total_tokens, kpool, budget, out_token_ids, nullptr,
                             sms, static_cast<cudaStream_t>(stream_ptr))))
    return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

size_t kpool_rows_workspace_bytes(int32_t num_rows, int64_t total_tokens, int32_t num_seqs, int32_t kpool,
                                  int32_t index_topk) {
  if (num_rows < 0 || total_tokens < 0 || total_tokens > int64_t(INT32_MAX) || num_seqs < 0 ||
      (total_tokens > 0 && num_seqs < 1))
    return 0;
  if (kpool < 1 || index_topk < 0 || index_topk % kpool != 0) return 0;
  return rows_layout(num_rows, total_tokens, num_seqs, kpool).total;
}

kpool_status kpool_select_rows(const void* q, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                               int32_t num_rows, const void* pooled_keys, const int32_t* cu_seqlens,
                               int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                               kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                               int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                               void* workspace, size_t workspace_bytes, void* stream_ptr) {
  return kpool_select_rows_ex(q, w, row_seq, row_pos, num_rows, pooled_keys, cu_seqlens, num_seqs, total_tokens,
                              heads, head_dim, dtype, kpool, index_topk, scale, out_pool_ids, out_token_ids,
                              out_pool_scores, workspace, workspace_bytes, stream_ptr, nullptr);
}

kpool_status kpool_select_rows_ex(const void* q, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                                  int32_t num_rows, const void* pooled_keys, const int32_t* cu_seqlens,
                                  int32_t num_seqs, int64_t total_tokens, int32_t heads, int32_t head_dim,
                                  kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                                  int32_t* out_pool_ids, int32_t* out_token_ids, float* out_pool_scores,
                                  void* workspace, size_t workspace_bytes, void* stream_ptr,
                                  const kpool_options* options) {
  kpool_options opt{};
  if (options) opt = *options;
  if (opt.reserved != 0 || opt.flags != 0 || opt.row_begin != 0 || opt.row_end != 0) return KPOOL_ERR_INVALID_ARG;
  if (opt.score_kernel != KPOOL_SCORE_AUTO || opt.max_ctas < 0) return KPOOL_ERR_INVALID_ARG;
  kpool_status st = check_shape(total_tokens, num_seqs, head_dim, dtype, kpool);
  if (st != KPOOL_OK) return st;
  if (num_rows < 0 || heads < 1 || index_topk < 0 || index_topk % kpool != 0 || !isfinite(scale))
    return KPOOL_ERR_INVALID_ARG;
  if (num_rows == 0) return KPOOL_OK;
  if (total_tokens == 0) return KPOOL_ERR_INVALID_ARG;  // a row needs a sequence to sit in
  const int32_t budget = index_topk / kpool;
  if (!q || !w || !row_seq || !row_pos || !cu_seqlens || !out_token_ids || (budget > 0 && !out_pool_ids) ||
      (total_tokens / kpool > 0 && !pooled_keys))
    return KPOOL_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(pooled_keys, 16) || !aligned(w, 4) || !aligned(row_seq, 4) ||
      !aligned(row_pos, 4) || !aligned(cu_seqlens, 4) || !aligned(out_pool_ids, 4) ||
      !aligned(out_token_ids, 4) || !aligned(out_pool_scores, 4))
    return KPOOL_ERR_INVALID_ARG;
  if (!select_rows_supported(dtype, heads, head_dim, budget)) return KPOOL_ERR_UNSUPPORTED;
  const RowsLayout L = rows_layout(num_rows, total_tokens, num_seqs, kpool);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < L.total) return KPOOL_ERR_WORKSPACE;
  int sms = 0;
  if (!cuda_ok(sm_count(&sms))) return KPOOL_ERR_CUDA;
  if (!cuda_ok(launch_select_rows(q, w, row_seq, row_pos, num_rows, pooled_keys, cu_seqlens, num_seqs,
                                  total_tokens, kpool, budget, scale, out_pool_ids, out_pool_scores, out_token_ids,
                                  static_cast<char*>(workspace), L, sms, opt.max_ctas,
                                  static_cast<cudaStream_t>(stream_ptr), opt.stage_events)))
    return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

kpool_status kpool_last_device_error(const void* workspace, void* stream_ptr) {
  if (workspace == nullptr || !aligned(workspace, 256)) return KPOOL_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (!cuda_ok(cudaStreamSynchronize(stream))) return KPOOL_ERR_CUDA;
  int32_t code = 0;
  if (!cuda_ok(cudaMemcpy(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost))) return KPOOL_ERR_CUDA;
  if (code < 0 || code > KPOOL_ERR_INTERNAL) return KPOOL_ERR_CUDA;
  return static_cast<kpool_status>(code);
}

kpool_status kpool_wait_timeout_selftest(void* workspace, size_t workspace_bytes, int64_t spin_limit,
                                         void* stream_ptr) {
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < sizeof(WorkspaceHeader))
    return KPOOL_ERR_WORKSPACE;
  if (spin_limit < 1) return KPOOL_ERR_INVALID_ARG;
  if (!cuda_ok(launch_wait_selftest(static_cast<char*>(workspace), spin_limit,
                                    static_cast<cudaStream_t>(stream_ptr))))
    return KPOOL_ERR_CUDA;
  return KPOOL_OK;
}

kpool_status kpool_balanced_row_split(const int32_t* cu_seqlens, int32_t num_seqs, int32_t kpool, int64_t row_weight,
                                      int32_t parts, int32_t* out_bounds) {
  if (cu_seqlens == nullptr || out_bounds == nullptr || num_seqs < 0 || kpool < 1 || parts < 1 || row_weight < 0)
    return KPOOL_ERR_INVALID_ARG;
  if (cu_seqlens[0] != 0) return KPOOL_ERR_INVALID_ARG;
  for (int32_t b = 0; b < num_seqs; ++b)
    if (cu_seqlens[b + 1] < cu_seqlens[b]) return KPOOL_ERR_INVALID_ARG;
  const int64_t T = cu_seqlens[num_seqs];
  // pairs of the first m rows of a sequence: sum_{i=1..m} floor(i / kpool)
  auto pairs_prefix = [kpool](int64_t m) {
    const int64_t n = m / kpool, r = m % kpool;
    return int64_t(kpool) * n * (n - 1) / 2 + n * (r + 1);
  };
  auto work = [&](int64_t m) { return pairs_prefix(m) + m * row_weight; };  // first m rows of a sequence
  int64_t total = 0;
  for (int32_t b = 0; b < num_seqs; ++b) total += work(cu_seqlens[b + 1] - cu_seqlens[b]);
  // boundary g is the first row r whose preceding rows' work reaches g * total / parts
  const int64_t quot = total / parts, rem = total % parts;
  auto target = [&](int64_t g) { return quot * g + (rem * g) / parts; };
  out_bounds[0] = 0;
  int32_t g = 1;
  int64_t before = 0;  // work of the sequences before b
  for (int32_t b = 0; b < num_seqs && g < parts; ++b) {
    const int64_t len = cu_seqlens[b + 1] - cu_seqlens[b];
    const int64_t wb = work(len);
    while (g < parts && target(g) <= before + wb) {
      int64_t lo = 0, hi = len;  // smallest m in [0, len] with before + work(m) >= target(g)
      while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (before + work(mid) >= target(g)) hi = mid; else lo = mid + 1;
      }
      out_bounds[g++] = int32_t(cu_seqlens[b] + lo);
    }
    before += wb;
  }
  for (; g <= parts; ++g) out_bounds[g] = int32_t(T);
  return KPOOL_OK;
}

const char* kpool_status_string(kpool_status status) {
  switch (status) {
    case KPOOL_OK: return "ok";
    case KPOOL_ERR_INVALID_ARG: return "invalid argument";
    case KPOOL_ERR_UNSUPPORTED: return "unsupported shape";
    case KPOOL_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KPOOL_ERR_CUDA: return "CUDA error";
    case KPOOL_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case KPOOL_ERR_INTERNAL: return "device-side bounds guard fired";
  }
  return "unknown status";
}

const char* kpool_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

}  // extern "C"
