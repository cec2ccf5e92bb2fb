// kpool_static_scratch.cu -- kpool_select for callers that cannot allocate.
//
// Every other entry point takes its scratch space (the workspace) from the
// caller. Some callers have no way to provide it: code that runs where device
// allocation is forbidden or unsafe -- a plugin or custom operator inside a host
// framework that owns all device memory through its own allocator, a real-time
// path that must never hit cudaMalloc's implicit device synchronisation, or an
// embedding that simply has no allocator handle to offer. This entry point
// serves them: its scratch is a fixed, file-scope __device__ array that every
// GPU loading this library holds until the process exits.
//
// Rules (also stated in include/kpool.h):
//   * the arguments are checked exactly as kpool_select checks them (a shape the
//     kernels do not implement is KPOOL_ERR_UNSUPPORTED, whatever its size); only
//     then is the capacity checked: a call whose workspace requirement
//     (kpool_workspace_bytes) exceeds KPOOL_STATIC_SCRATCH_BYTES is rejected with
//     KPOOL_ERR_WORKSPACE, before any GPU work;
//   * the first call on a device looks up the array's device address with that
//     device current (cudaGetSymbolAddress) and caches it; make that first call
//     before any stream capture;
//   * every call on a device shares the one array, so calls that overlap on the
//     GPU (different streams, different host threads) race -- serialise them;
//   * nothing here allocates: no cudaMalloc, cudaFree or allocating library call;
//   * the array keeps the previous call's contents; the planning kernel rewrites
//     every field the later kernels read, so nothing needs clearing up front;
//   * errors found on the device land in the array's header, read back with
//     kpool_static_scratch_last_device_error.
#include <atomic>

#include <cuda_runtime.h>

#include "kpool_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KPOOL_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_kpool_scratch[kScratchBytes];

std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of g_kpool_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_kpool_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" kpool_status kpool_select_static_scratch(const void* q, const void* k, const float* w,
                                                    const int32_t* cu_seqlens, int32_t num_seqs,
                                                    int64_t total_tokens, int32_t heads, int32_t head_dim,
                                                    kpool_dtype dtype, int32_t kpool, int32_t index_topk, float scale,
                                                    int32_t* out_pool_ids, int32_t* out_token_ids,
                                                    float* out_pool_scores, void* stream) {
  bool use_tc = false;
  int64_t rb = 0, re = 0;
  const kpool_status st = kpool::select_check_args(q, k, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim,
                                                   dtype, kpool, index_topk, scale, out_pool_ids, out_token_ids,
                                                   out_pool_scores, nullptr, &use_tc, &rb, &re);
  if (st != KPOOL_OK || total_tokens == 0) return st;
  const size_t need = kpool_workspace_bytes(total_tokens, num_seqs, heads, head_dim, dtype, kpool, index_topk);
  if (need == 0) return KPOOL_ERR_INVALID_ARG;
  if (need > kScratchBytes) return KPOOL_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KPOOL_ERR_CUDA;
  return kpool_select(q, k, w, cu_seqlens, num_seqs, total_tokens, heads, head_dim, dtype, kpool, index_topk,
                      scale, out_pool_ids, out_token_ids, out_pool_scores, scratch, kScratchBytes, stream);
}

extern "C" kpool_status kpool_static_scratch_last_device_error(void* stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KPOOL_ERR_CUDA;
  return kpool_last_device_error(scratch, stream);
}
