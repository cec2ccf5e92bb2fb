// kpool_rows.cu -- selection for an explicit set of query rows against a pooled-key
// cache that already exists: the decode / short-query case. At a 262,144-token
// context one decode token scores 65,536 pools ("spark_model/layers/glm5next_dsa/
// tp.rs", module docs, "Why the indexer is REPLICATED": scores are [q_rows,
// n_pools] with n_pools = seq / kpool). Row r (sequence b, local position t)
// selects exactly what row t of the whole-batch selection would: the top budget
// of the pools p < floor((t+1)/kpool) of its sequence, by higher score and then
// smaller pool index, expanded to token ids with its own trailing pool appended.
//
// With a handful of rows the work is too small for the persistent tensor-core
// kernel's one-CTA-per-item layout, so this path splits every row's pool range
// over many CTAs and keeps the [rows, pools] scores (a few MiB, L2-resident):
//   R0 rows_plan_kernel   (1 CTA)   checks cu_seqlens and the rows, pool offsets,
//                                   per-row eligible counts and the work units
//   R1 rows_score_kernel  (grid)    one unit = up to 1024 pools of one row; bf16
//                                   mma.sync tensor-core products, relu / weight /
//                                   head sum in registers, fp32 scores out
//   R2 rows_select_kernel (1 CTA / row) exact top-budget by an MSD radix search
//                                   on the scores, ties to the smaller pool, a
//                                   register bitonic sort, ids / scores / tokens
// R1 streams the pooled keys once per row (HBM-bound: 256 B per pool); the
// contraction per pool is 32 heads x 128 channels, small enough that the
// warp-level mma.sync form keeps up with memory, so the tcgen05 pipeline of the
// batch kernel is not needed here.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kpool_internal.cuh"
#include "kpool_select_common.cuh"

namespace kpool {
namespace {

constexpr int kRowsHeads = 32;
constexpr int kRowsDim = 128;
constexpr int kUnitPools = 1024;       // pools per work unit of R1
constexpr int kScoreWarps = 8;         // R1: 8 warps x 128 pools = one unit
constexpr int kSelectThreads = 512;    // R2
constexpr int kRowsMaxBudget = 512;    // R2 sorts at most 512 keys in one warp

struct RowInfo {
  int32_t pool_base;  // global pooled-key row of the sequence's pool 0
  int32_t e;          // eligible pools floor((t+1)/kpool); -1 marks an invalid row
  int32_t t;          // sequence-local position
  int32_t pad;
};

__device__ int block_exclusive_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int res = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
  *total = s_warp[31];
  __syncthreads();
  return res;
}

// ------------------------------------------------------------------ R0 plan
__global__ void __launch_bounds__(1024) rows_plan_kernel(const int32_t* __restrict__ cu, int S, int64_t T,
                                                         const int32_t* __restrict__ row_seq,
                                                         const int32_t* __restrict__ row_pos, int R, int kpool,
                                                         WorkspaceHeader* hdr, int32_t* pool_off, RowInfo* info,
                                                         int32_t* unit_off) {
  __shared__ int s_bad, s_bad_row;
  __shared__ int s_warp[32];
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (cu[0] != 0 || int64_t(cu[S]) != T) ? 1 : 0;
    s_bad_row = 0;
  }
  __syncthreads();
  for (int b = tid; b < S; b += blockDim.x)
    if (cu[b + 1] < cu[b]) s_bad = 1;
  __syncthreads();
  if (s_bad) {  // nothing below runs; R2 sees n_levels == 0 and writes empty rows
    if (tid == 0) {
      hdr->error = KPOOL_ERR_INVALID_ARG;
      hdr->n_items = 0;
      hdr->n_levels = 0;
    }
    return;
  }
  int carry = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int b = base + tid;
    const int n = b < S ? (cu[b + 1] - cu[b]) / kpool : 0;
    int tot;
    const int ex = block_exclusive_scan(n, &tot, s_warp);
    if (b < S) pool_off[b] = carry + ex;
    carry += tot;
  }
  if (tid == 0) pool_off[S] = carry;
  __syncthreads();
  int ucarry = 0;
  for (int base = 0; base < R; base += blockDim.x) {
    const int r = base + tid;
    int units = 0;
    if (r < R) {
      const int b = row_seq[r], t = row_pos[r];
      RowInfo ri{0, -1, 0, 0};
      if (b >= 0 && b < S && t >= 0 && t < cu[b + 1] - cu[b]) {
        ri.pool_base = pool_off[b];
        ri.e = (t + 1) / kpool;
        ri.t = t;
        units = (ri.e + kUnitPools - 1) / kUnitPools;
      } else {
        s_bad_row = 1;
      }
      info[r] = ri;
    }
    int tot;
    const int ex = block_exclusive_scan(units, &tot, s_warp);
    if (r < R) unit_off[r] = ucarry + ex;
    ucarry += tot;
  }
  __syncthreads();
  if (tid == 0) {
    unit_off[R] = ucarry;
    hdr->n_items = ucarry;
    hdr->n_levels = 1;  // cu_seqlens valid: the row records are written
    hdr->total_pools = carry;
    hdr->error = s_bad_row ? KPOOL_ERR_INVALID_ARG : 0;
  }
}

// ----------------------------------------------------------------- R1 score
//
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate): a warp takes 16 pools (M) x 8
// heads (N) per instruction, 4 instructions cover the 32 heads and 8 k-steps the
// 128 channels. The channel order inside a 32-channel block is permuted the same
// way for both operands (a dot product does not depend on it), so every thread
// fills its fragments from 16-byte loads: thread (g = lane / 4, c = lane % 4)
// reads channels 32m + 8c .. 32m + 8c + 7 of pools g and g + 8 and of heads
// g + 8n. The first four of those eight channels feed k-step 2m, the last four
// k-step 2m + 1.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kScoreWarps * 32) rows_score_kernel(
    const uint4* __restrict__ q, const float* __restrict__ w, const uint4* __restrict__ kp,
    const RowInfo* __restrict__ info, const int32_t* __restrict__ unit_off, const WorkspaceHeader* hdr, int R,
    float scale, float* __restrict__ scores, int64_t stride) {
  const int n_units = hdr->n_items;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const float abs_scale = fabsf(scale);
  const bool neg = scale < 0.0f;
  constexpr int kVecPerRow = kRowsDim / 8;  // 16-byte vectors per pooled key / query head
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    // row of unit u: the last r with unit_off[r] <= u
    int lo = 0, hi = R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(unit_off + mid) <= u) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const RowInfo ri = info[r];
    const int p_begin = (u - unit_off[r]) * kUnitPools;
    const int e = ri.e;
    // query fragments of all 32 heads: qf[n][m] holds channels 32m + 8c .. + 7 of head g + 8n
    uint4 qf[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int m = 0; m < 4; ++m) qf[n][m] = __ldg(q + (int64_t(r) * kRowsHeads + g + 8 * n) * kVecPerRow + 4 * m + c);
    // this thread's accumulator columns are heads 8n + 2c and 8n + 2c + 1
    float wt[4][2];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      wt[n][0] = __ldg(w + int64_t(r) * kRowsHeads + 8 * n + 2 * c) * abs_scale;
      wt[n][1] = __ldg(w + int64_t(r) * kRowsHeads + 8 * n + 2 * c + 1) * abs_scale;
    }
    float* out = scores + int64_t(r) * stride;
    for (int p0 = p_begin + warp * 16; p0 < min(e, p_begin + kUnitPools); p0 += kScoreWarps * 16) {
      // pooled keys of pools p0 + g and p0 + g + 8 (clamped to an eligible pool; the
      // scores of clamped rows are not stored)
      const int pa = min(p0 + g, e - 1), pb = min(p0 + g + 8, e - 1);
      uint4 ka[4], kb[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        ka[m] = __ldg(kp + int64_t(ri.pool_base + pa) * kVecPerRow + 4 * m + c);
        kb[m] = __ldg(kp + int64_t(ri.pool_base + pb) * kVecPerRow + 4 * m + c);
      }
      float acc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[n][i] = 0.0f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t a_lo[4] = {ka[m].x, kb[m].x, ka[m].y, kb[m].y};  // k-step 2m
        const uint32_t a_hi[4] = {ka[m].z, kb[m].z, ka[m].w, kb[m].w};  // k-step 2m + 1
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          mma_bf16_16816(acc[n], a_lo, qf[n][m].x, qf[n][m].y);
          mma_bf16_16816(acc[n], a_hi, qf[n][m].z, qf[n][m].w);
        }
      }
      // acc[n][0..1]: pool g, heads 8n + 2c, +1; acc[n][2..3]: pool g + 8
      float sa = 0.0f, sb = 0.0f;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        sa = fmaf(wt[n][0], fmaxf(neg ? -acc[n][0] : acc[n][0], 0.0f), sa);
        sa = fmaf(wt[n][1], fmaxf(neg ? -acc[n][1] : acc[n][1], 0.0f), sa);
        sb = fmaf(wt[n][0], fmaxf(neg ? -acc[n][2] : acc[n][2], 0.0f), sb);
        sb = fmaf(wt[n][1], fmaxf(neg ? -acc[n][3] : acc[n][3], 0.0f), sb);
      }
      // head sum across the four threads of a pool
      sa += __shfl_xor_sync(0xffffffffu, sa, 1);
      sa += __shfl_xor_sync(0xffffffffu, sa, 2);
      sb += __shfl_xor_sync(0xffffffffu, sb, 1);
      sb += __shfl_xor_sync(0xffffffffu, sb, 2);
      if (c == 0 && p0 + g < e) out[p0 + g] = sa;
      if (c == 1 && p0 + g + 8 < e) out[p0 + g + 8] = sb;
    }
  }
}

// ---------------------------------------------------------------- R2 select
//
// Exact top-budget of one row's scores. The order is that of the 64-bit
// selection key (order-preserving score bits, then the complemented pool
// index), so the search runs on the 32 score bits with 8-bit digits (most
// significant first) to find the budget-th largest score value v, then takes
// every pool scoring above v and, of the pools scoring exactly v, the ones with
// the smallest indices until the budget is full.
__global__ void __launch_bounds__(kSelectThreads) rows_select_kernel(
    const float* __restrict__ scores, int64_t stride, const RowInfo* __restrict__ info,
    const WorkspaceHeader* hdr, int kpool, int budget, int32_t* __restrict__ out_ids,
    float* __restrict__ out_scores, int32_t* __restrict__ out_tokens) {
  __shared__ uint32_t s_hist[256];
  __shared__ int s_warp[32];
  __shared__ uint32_t s_digit, s_above;
  __shared__ int s_count;
  __shared__ uint64_t s_keys[kRowsMaxBudget];
  __shared__ int32_t s_ids[kRowsMaxBudget];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int width = budget * kpool + kpool;
  int32_t* tok = out_tokens + int64_t(r) * width;
  const RowInfo ri = hdr->n_levels != 0 ? info[r] : RowInfo{0, -1, 0, 0};
  if (ri.e < 0) {  // malformed cu_seqlens or an invalid row: every slot empty
    for (int s = tid; s < width; s += kSelectThreads) tok[s] = -1;
    for (int j = tid; j < budget; j += kSelectThreads) {
      out_ids[int64_t(r) * budget + j] = -1;
      if (out_scores) out_scores[int64_t(r) * budget + j] = -INFINITY;
    }
    return;
  }
  const int e = ri.e;
  const float* row = scores + int64_t(r) * stride;
  const int m = min(budget, e);
  if (tid == 0) s_count = 0;
  for (int j = tid; j < kRowsMaxBudget; j += kSelectThreads) s_keys[j] = 0ull;
  __syncthreads();

  if (e <= budget) {
    for (int p = tid; p < e; p += kSelectThreads) s_keys[p] = make_key(row[p], uint32_t(p));
  } else if (budget > 0) {
    // MSD radix search for v = the budget-th largest score_order_bits value
    uint32_t prefix = 0;
    int above = 0;  // pools whose bits exceed every value still in the bin
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
      for (int i = tid; i < 256; i += kSelectThreads) s_hist[i] = 0;
      __syncthreads();
      // whole warps iterate together (the bound is a multiple of 32) for the warp votes
      const int e_pad = (e + 31) & ~31;
      for (int p = tid; p < e_pad; p += kSelectThreads) {
        bool in = false;
        uint32_t dig = 0;
        if (p < e) {
          const uint32_t u = score_order_bits(row[p]);
          in = (u & hi_mask) == (prefix & hi_mask);
          dig = (u >> shift) & 255u;
        }
        // one shared atomic per distinct digit in the warp
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const unsigned peers = __match_any_sync(act, dig);
          if ((__ffs(peers) - 1) == lane) atomicAdd(s_hist + dig, uint32_t(__popc(peers)));
        }
      }
      __syncthreads();
      if (tid < 32) {
        // digit d (descending) where the count from the top first reaches budget - above
        uint32_t cnt[8];
        uint32_t tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          cnt[i] = s_hist[255 - (8 * lane + i)];
          tot += cnt[i];
        }
        uint32_t incl = tot;  // inclusive prefix over lanes (digits from 255 down)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        const uint32_t need = uint32_t(budget - above);
        const uint32_t before = incl - tot;
        const bool mine = before < need && incl >= need;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        if (mine) {
          uint32_t run = before;
          int i = 0;
          while (i < 8 && run + cnt[i] < need) run += cnt[i++];
          s_digit = 255u - uint32_t(8 * lane + i);
          s_above = run;
        }
        (void)who;
      }
      __syncthreads();
      prefix |= s_digit << shift;
      above += int(s_above);
      __syncthreads();
    }
    // every pool above v, then the pools equal to v in index order until the budget is full
    const int need_ties = budget - above;
    const int per = (e + kSelectThreads - 1) / kSelectThreads;
    const int p_lo = tid * per, p_hi = min(e, p_lo + per);
    int my_ties = 0;
    for (int p = p_lo; p < p_hi; ++p) my_ties += score_order_bits(row[p]) == prefix;
    int tot_ties;
    int tie_rank = block_exclusive_scan(my_ties, &tot_ties, s_warp);
    for (int p = p_lo; p < p_hi; ++p) {
      const float s = row[p];
      const uint32_t u = score_order_bits(s);
      bool take = u > prefix;
      if (u == prefix) take = tie_rank++ < need_ties;
      if (take) {
        const int slot = atomicAdd(&s_count, 1);
        if (slot < kRowsMaxBudget) s_keys[slot] = make_key(s, uint32_t(p));
      }
    }
  }
  __syncthreads();
  if (tid < 32) {
    uint64_t k[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) k[j] = s_keys[32 * j + lane];
    warp_sort512_blocked_desc(k);  // lane l holds ranks 16 l .. 16 l + 15
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int rank = 16 * lane + j;
      if (rank < budget) {
        const bool has = rank < m && k[j] != 0ull;
        const int32_t id = has ? int32_t(key_pool(k[j])) : -1;
        s_ids[rank] = id;
        out_ids[int64_t(r) * budget + rank] = id;
        if (out_scores) out_scores[int64_t(r) * budget + rank] = has ? key_score(k[j]) : -INFINITY;
      }
    }
  }
  __syncthreads();
  // expansion: slot j*kpool + i = id_j*kpool + i; tail slots budget*kpool + i hold the
  // row's incomplete pool e*kpool + i for i < (t+1) mod kpool
  const int tail = (ri.t + 1) % kpool;
  for (int s = tid; s < width; s += kSelectThreads) {
    int32_t v = -1;
    if (s < budget * kpool) {
      const int j = s / kpool, i = s - j * kpool;
      const int32_t id = s_ids[j];
      if (id >= 0) v = id * kpool + i;
    } else {
      const int i = s - budget * kpool;
      if (i < tail) v = e * kpool + i;
    }
    tok[s] = v;
  }
}

}  // namespace

// ------------------------------------------------------------------ host side

RowsLayout rows_layout(int32_t R, int64_t T, int32_t S, int32_t kpool) {
  RowsLayout L{};
  int64_t stride = T / kpool;
  stride = ((stride > 0 ? stride : 1) + 3) & ~int64_t(3);
  L.stride = stride;
  size_t off = 0;
  L.header = off;   off = align256(off + sizeof(WorkspaceHeader));
  L.pool_off = off; off = align256(off + sizeof(int32_t) * size_t(S + 1));
  L.info = off;     off = align256(off + sizeof(RowInfo) * size_t(R > 0 ? R : 1));
  L.unit_off = off; off = align256(off + sizeof(int32_t) * size_t(R + 1));
  L.scores = off;   off = align256(off + sizeof(float) * size_t(R) * size_t(stride));
  L.total = off;
  return L;
}

bool select_rows_supported(kpool_dtype dtype, int32_t H, int32_t d, int32_t budget) {
  return dtype == KPOOL_BF16 && H == kRowsHeads && d == kRowsDim && budget >= 0 && budget <= kRowsMaxBudget;
}

cudaError_t launch_select_rows(const void* q, const float* w, const int32_t* row_seq, const int32_t* row_pos,
                               int32_t R, const void* kp, const int32_t* cu, int32_t S, int64_t T, int32_t kpool,
                               int32_t budget, float scale, int32_t* out_ids, float* out_scores,
                               int32_t* out_tokens, char* ws, const RowsLayout& L, int num_sms,
                               cudaStream_t stream) {
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  int32_t* pool_off = reinterpret_cast<int32_t*>(ws + L.pool_off);
  RowInfo* info = reinterpret_cast<RowInfo*>(ws + L.info);
  int32_t* unit_off = reinterpret_cast<int32_t*>(ws + L.unit_off);
  float* scores = reinterpret_cast<float*>(ws + L.scores);
  rows_plan_kernel<<<1, 1024, 0, stream>>>(cu, S, T, row_seq, row_pos, R, kpool, hdr, pool_off, info, unit_off);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // units: at most R * ceil(max pools / kUnitPools); a few waves of 2 CTAs per SM
  const int64_t max_units = int64_t(R) * ((L.stride + kUnitPools - 1) / kUnitPools);
  const int grid = int(max_units < int64_t(4) * num_sms ? (max_units > 0 ? max_units : 1) : int64_t(4) * num_sms);
  rows_score_kernel<<<grid, kScoreWarps * 32, 0, stream>>>(static_cast<const uint4*>(q), w,
                                                             static_cast<const uint4*>(kp), info, unit_off, hdr,
                                                             R, scale, scores, L.stride);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  rows_select_kernel<<<R, kSelectThreads, 0, stream>>>(scores, L.stride, info, hdr, kpool, budget, out_ids,
                                                       out_scores, out_tokens);
  return cudaGetLastError();
}

}  // namespace kpool
