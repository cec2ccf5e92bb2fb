// kpool_plan.cu -- K0: per-call planning on the device.
//
// From cu_seqlens alone (it lives on the device, so the host never has to wait
// for it) this kernel
//   * checks the packed-batch bounds (cu[0] = 0, nondecreasing, cu[S] = T) --
//     the varlen bounds of the pages' packed THD layout ("NVIDIA/Megatron-LM
//     pull request #8299", section "Test plan");
//   * writes the first pooled-key row of every sequence, pool_off[b] =
//     sum_{j<b} floor(L_j / kpool) (tp.rs module docs: n_pools = seq / kpool);
//   * lists the work items of the tensor-core kernel: one item per block of
//     kItemRows query rows of one sequence, ordered deepest-first. An item at
//     depth j (local rows j*kItemRows ...) scores about j*kItemRows/kpool pools
//     under the causal window, so deepest-first is heaviest-first and the
//     persistent kernel's static round-robin stays balanced;
//   * resets the header (error word, counts).
// One CTA of 1024 threads; the work is O(S + items).
#include "kpool_internal.cuh"

namespace kpool {
namespace {

constexpr int kThreads = 1024;

// Block-wide inclusive scan of one int per thread; returns the inclusive
// prefix, *total receives the block sum. All threads must call it.
__device__ int block_inclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  int res = v + (warp > 0 ? s_warp[warp - 1] : 0);
  *total = s_warp[31];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kThreads) plan_kernel(const int32_t* __restrict__ cu, int S, int64_t T,
                                                        int kpool, WorkspaceHeader* hdr, int32_t* pool_off,
                                                        int32_t* qblk_off, int32_t* level_cnt,
                                                        int32_t* level_start, int32_t* level_fill,
                                                        int2* items, int64_t max_levels) {
  __shared__ int s_bad;
  __shared__ int s_max_depth;
  __shared__ int s_warp[32];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (cu[0] != 0 || int64_t(cu[S]) != T) ? 1 : 0;
    s_max_depth = 0;
  }
  __syncthreads();
  for (int b = tid; b < S; b += kThreads)
    if (cu[b + 1] < cu[b]) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      hdr->error = KPOOL_ERR_INVALID_ARG;
      hdr->n_items = 0;
      hdr->n_levels = 0;
      hdr->total_pools = 0;
      hdr->next_item = 0;
    }
    return;
  }

  // pool and item offsets (exclusive scans over sequences)
  int carry_p = 0, carry_q = 0;
  for (int base = 0; base < S; base += kThreads) {
    const int b = base + tid;
    int np = 0, nq = 0;
    if (b < S) {
      const int len = cu[b + 1] - cu[b];
      np = len / kpool;
      nq = (len + kItemRows - 1) / kItemRows;
      atomicMax(&s_max_depth, nq);
    }
    int tp, tq;
    const int ip = block_inclusive_scan(np, &tp, s_warp);
    const int iq = block_inclusive_scan(nq, &tq, s_warp);
    if (b < S) {
      pool_off[b] = carry_p + ip - np;
      qblk_off[b] = carry_q + iq - nq;
    }
    carry_p += tp;
    carry_q += tq;
  }
  __syncthreads();
  const int n_items = carry_q;
  const int n_levels = s_max_depth;
  if (tid == 0) {
    pool_off[S] = carry_p;
    qblk_off[S] = carry_q;
  }
  if (n_levels > max_levels) {  // cannot happen with a workspace sized for T
    if (tid == 0) {
      hdr->error = KPOOL_ERR_WORKSPACE;
      hdr->n_items = 0;
      hdr->n_levels = 0;
      hdr->total_pools = 0;
      hdr->next_item = 0;
    }
    return;
  }

  // level_cnt[j] = number of sequences with exactly j+1 items
  for (int j = tid; j < n_levels; j += kThreads) {
    level_cnt[j] = 0;
    level_fill[j] = 0;
  }
  __syncthreads();
  for (int b = tid; b < S; b += kThreads) {
    const int nq = (cu[b + 1] - cu[b] + kItemRows - 1) / kItemRows;
    if (nq > 0) atomicAdd(&level_cnt[nq - 1], 1);
  }
  __syncthreads();

  // deep[j] = #sequences with more than j items (suffix sum of level_cnt);
  // level_start[j] = sum_{j' > j} deep[j'] (deeper levels come first).
  int carry_deep = 0, carry_start = 0;
  for (int base = 0; base < n_levels; base += kThreads) {
    const int r = base + tid;           // r-th level from the deepest
    const int j = n_levels - 1 - r;
    const int c = (r < n_levels) ? level_cnt[j] : 0;
    int tot;
    const int deep = carry_deep + block_inclusive_scan(c, &tot, s_warp);
    carry_deep += tot;
    const int d = (r < n_levels) ? deep : 0;
    int tot2;
    const int incl = block_inclusive_scan(d, &tot2, s_warp);
    if (r < n_levels) level_start[j] = carry_start + incl - d;
    carry_start += tot2;
  }
  __syncthreads();

  for (int i = tid; i < n_items; i += kThreads) {
    // the sequence whose item range holds i: last b with qblk_off[b] <= i
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (qblk_off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int j = i - qblk_off[lo];
    const int pos = level_start[j] + atomicAdd(&level_fill[j], 1);
    items[pos] = make_int2(lo, j);
  }
  if (tid == 0) {
    hdr->error = 0;
    hdr->n_items = n_items;
    hdr->n_levels = n_levels;
    hdr->total_pools = carry_p;
    hdr->next_item = 0;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* cu, int32_t S, int64_t T, int32_t kpool, char* ws,
                        const WorkspaceLayout& L, cudaStream_t stream) {
  plan_kernel<<<1, kThreads, 0, stream>>>(
      cu, S, T, kpool, reinterpret_cast<WorkspaceHeader*>(ws + L.header),
      reinterpret_cast<int32_t*>(ws + L.pool_off), reinterpret_cast<int32_t*>(ws + L.qblk_off),
      reinterpret_cast<int32_t*>(ws + L.level_cnt), reinterpret_cast<int32_t*>(ws + L.level_start),
      reinterpret_cast<int32_t*>(ws + L.level_fill), reinterpret_cast<int2*>(ws + L.items), L.max_levels);
  return cudaGetLastError();
}

}  // namespace kpool
