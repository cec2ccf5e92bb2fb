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
//     kItemRows query rows of one sequence that holds rows of the call's row
//     range (every row unless the caller selects a shard of rows), ordered
//     deepest-first. An item at
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

// Item blocks [j_lo, j_hi) of a sequence starting at global row c0 with `len` rows that
// hold rows of the range [row_begin, row_end) (empty when none does).
__device__ __forceinline__ int2 item_range(int64_t c0, int len, int64_t row_begin, int64_t row_end) {
  const int64_t lo = min(max(row_begin - c0, int64_t(0)), int64_t(len));
  const int64_t hi = min(max(row_end - c0, int64_t(0)), int64_t(len));
  if (lo >= hi) return make_int2(0, 0);
  return make_int2(int(lo / kItemRows), int((hi + kItemRows - 1) / kItemRows));
}

__global__ void __launch_bounds__(kThreads) plan_kernel(const int32_t* __restrict__ cu, int S, int64_t T,
                                                        int kpool, int64_t row_begin, int64_t row_end,
                                                        WorkspaceHeader* hdr, int32_t* pool_off,
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

  // pool and item offsets (exclusive scans over sequences); a sequence's items are the
  // blocks of kItemRows rows that hold rows of [row_begin, row_end)
  int carry_p = 0, carry_q = 0;
  for (int base = 0; base < S; base += kThreads) {
    const int b = base + tid;
    int np = 0, nq = 0;
    if (b < S) {
      const int len = cu[b + 1] - cu[b];
      np = len / kpool;
      const int2 jr = item_range(cu[b], len, row_begin, row_end);
      nq = jr.y - jr.x;
      atomicMax(&s_max_depth, jr.y);
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
  const int n_levels = s_max_depth;  // item depths 0 .. n_levels - 1
  if (tid == 0) {
    pool_off[S] = carry_p;
    qblk_off[S] = carry_q;
  }
  if (int64_t(n_levels) + 1 > max_levels) {  // cannot happen with a workspace sized for T
    if (tid == 0) {
      hdr->error = KPOOL_ERR_WORKSPACE;
      hdr->n_items = 0;
      hdr->n_levels = 0;
      hdr->total_pools = 0;
      hdr->next_item = 0;
    }
    return;
  }

  // level_cnt: +1 at each sequence's first item depth, -1 past its last, so its
  // prefix sum is the number of items at each depth
  for (int j = tid; j <= n_levels; j += kThreads) {
    level_cnt[j] = 0;
    level_fill[j] = 0;
  }
  __syncthreads();
  for (int b = tid; b < S; b += kThreads) {
    const int2 jr = item_range(cu[b], cu[b + 1] - cu[b], row_begin, row_end);
    if (jr.y > jr.x) {
      atomicAdd(&level_cnt[jr.x], 1);
      atomicAdd(&level_cnt[jr.y], -1);
    }
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < n_levels; base += kThreads) {
    const int j = base + tid;
    const int dv = j < n_levels ? level_cnt[j] : 0;
    int tot;
    const int incl = block_inclusive_scan(dv, &tot, s_warp);
    if (j < n_levels) level_cnt[j] = carry + incl;  // items at depth j
    carry += tot;
  }
  __syncthreads();
  // level_start[j] = items at depths deeper than j (deeper levels come first)
  carry = 0;
  for (int base = 0; base < n_levels; base += kThreads) {
    const int r = base + tid;  // r-th level from the deepest
    const int j = n_levels - 1 - r;
    const int c = r < n_levels ? level_cnt[j] : 0;
    int tot;
    const int incl = block_inclusive_scan(c, &tot, s_warp);
    if (r < n_levels) level_start[j] = carry + incl - c;
    carry += tot;
  }
  __syncthreads();

  for (int i = tid; i < n_items; i += kThreads) {
    // the sequence whose item range holds i: last b with qblk_off[b] <= i
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (qblk_off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int2 jr = item_range(cu[lo], cu[lo + 1] - cu[lo], row_begin, row_end);
    const int j = jr.x + (i - qblk_off[lo]);
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

cudaError_t launch_plan(const int32_t* cu, int32_t S, int64_t T, int32_t kpool, int64_t row_begin,
                        int64_t row_end, char* ws, const WorkspaceLayout& L, cudaStream_t stream) {
  plan_kernel<<<1, kThreads, 0, stream>>>(
      cu, S, T, kpool, row_begin, row_end, reinterpret_cast<WorkspaceHeader*>(ws + L.header),
      reinterpret_cast<int32_t*>(ws + L.pool_off), reinterpret_cast<int32_t*>(ws + L.qblk_off),
      reinterpret_cast<int32_t*>(ws + L.level_cnt), reinterpret_cast<int32_t*>(ws + L.level_start),
      reinterpret_cast<int32_t*>(ws + L.level_fill), reinterpret_cast<int2*>(ws + L.items), L.max_levels);
  return cudaGetLastError();
}

}  // namespace kpool
