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
//   R1 rows_score_kernel  (grid)    each CTA a contiguous run of 128-pool units; bf16
//                                   mma.sync tensor-core products, relu / weight /
//                                   head sum in registers, fp32 scores out
//   R2 rows_collect_kernel (grid)   from a per-row histogram of the scores' top 12
//                                   bits (built by R1) finds the bin holding the
//                                   budget-th score, then gathers every pool above
//                                   that bin and the pools inside it
//   R3 rows_select_kernel (1 CTA / row) exact top-budget among the gathered pools
//                                   (ties to the smaller pool; a full MSD radix
//                                   search over the row when the bin overflows), a
//                                   256-thread bitonic sort, ids / scores / tokens
// R1-R3 use programmatic dependent launch (see wait_prior_kernel below).
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
constexpr int kUnitPools = 128;        // pools per work unit of R1 (the split granularity)
constexpr int kScoreWarps = 8;         // R1: 8 warps x 16 pools per round
constexpr int kSelectThreads = 256;    // R3 (block_sort512_desc takes exactly 256 threads)
constexpr int kRowsMaxBudget = 512;    // R3 sorts at most 512 keys
constexpr int kHistBits = 12;          // histogram of score_order_bits >> (32 - kHistBits)
constexpr int kHistBins = 1 << kHistBits;
constexpr int kTieCap = 4096;          // pools of the threshold bin R3 can finish in shared memory
static_assert(kTieCap >= 1024, "R3 sorts in the tie buffer (1024 keys)");
constexpr int kCollectPools = 2048;    // R2: pools per CTA and round
constexpr int kCollectTies = 2048;     // R2: threshold-bin pools one round can hold
constexpr int kCollectCtasPerRow = 64; // R2: grid width; CTAs loop over a row's slices
constexpr int kCollectThreads = 256;
constexpr int kCollectPer = kCollectPools / kCollectThreads;  // R2: scores per thread and round
static_assert(kCollectPer % 4 == 0, "R2 loads its scores 4 at a time");

// Programmatic dependent launch: R1-R3 are launched so they may start while the
// kernel before them is still running; each waits here, before its first read of
// anything an earlier kernel of the call wrote, until that kernel has completed
// and its writes are visible. (Launched without the attribute, the wait returns at
// once.) The trigger lets the next kernel's CTAs be scheduled as early as the
// resources they need free up.
__device__ __forceinline__ void wait_prior_kernel() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_kernel() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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
__global__ void __launch_bounds__(256) rows_plan_kernel(const int32_t* __restrict__ cu, int S, int64_t T,
                                                         const int32_t* __restrict__ row_seq,
                                                         const int32_t* __restrict__ row_pos, int R, int kpool,
                                                         WorkspaceHeader* hdr, int32_t* pool_off, RowInfo* info,
                                                         int32_t* unit_off) {
  __shared__ int s_bad, s_bad_row;
  __shared__ int s_warp[32];
  const int tid = threadIdx.x;
  allow_next_kernel();
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
    float scale, float* __restrict__ scores, int64_t stride, uint32_t* __restrict__ hist) {
  __shared__ uint32_t s_hist[kHistBins];  // this unit's histogram, flushed to the row's at the end
  __shared__ uint4 s_q[16][32];           // the row's query fragments (see below)
  wait_prior_kernel();  // the plan: n_items, row records, unit offsets (and the cleared histograms)
  allow_next_kernel();
  const int n_units = hdr->n_items;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const float abs_scale = fabsf(scale);
  const bool neg = scale < 0.0f;
  constexpr int kVecPerRow = kRowsDim / 8;  // 16-byte vectors per pooled key / query head
  // this CTA's share: a contiguous run of units, i.e. one or a few contiguous pool
  // ranges ("segments") of consecutive rows
  const int u_first = int(int64_t(n_units) * blockIdx.x / gridDim.x);
  const int u_last = int(int64_t(n_units) * (blockIdx.x + 1) / gridDim.x);
  for (int u = u_first; u < u_last;) {
    // row of unit u: the last r with unit_off[r] <= u
    int lo = 0, hi = R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(unit_off + mid) <= u) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const RowInfo ri = info[r];
    const int seg_end = min(u_last, __ldg(unit_off + r + 1));
    const int p_begin = (u - unit_off[r]) * kUnitPools;
    const int e = ri.e;
    const int p_end = min(e, (seg_end - unit_off[r]) * kUnitPools);
    u = seg_end;
    // query fragments of all 32 heads, one copy per lane slot in shared memory so the
    // registers stay free for a second set of pooled-key loads in flight:
    // s_q[n * 4 + m][lane] holds channels 32m + 8c .. + 7 of head g + 8n
    __syncthreads();  // the previous unit's fragments are no longer read
    for (int i = threadIdx.x; i < 16 * 32; i += blockDim.x) {
      const int f = i >> 5, l = i & 31, n = f >> 2, m = f & 3;
      s_q[f][l] = __ldg(q + (int64_t(r) * kRowsHeads + (l >> 2) + 8 * n) * kVecPerRow + 4 * m + (l & 3));
    }
    // this thread's accumulator columns are heads 8n + 2c and 8n + 2c + 1
    float wt[4][2];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      wt[n][0] = __ldg(w + int64_t(r) * kRowsHeads + 8 * n + 2 * c) * abs_scale;
      wt[n][1] = __ldg(w + int64_t(r) * kRowsHeads + 8 * n + 2 * c + 1) * abs_scale;
    }
    float* out = scores + int64_t(r) * stride;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) s_hist[i] = 0;
    __syncthreads();
    // pooled keys of pools p + g and p + g + 8, clamped to an eligible pool (the scores
    // of clamped rows are not stored); the next 16 pools load while these are scored
    auto load_keys = [&](int p, uint4 (&ka)[4], uint4 (&kb)[4]) {
      const int pa = min(p + g, e - 1), pb = min(p + g + 8, e - 1);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        ka[m] = __ldg(kp + int64_t(ri.pool_base + pa) * kVecPerRow + 4 * m + c);
        kb[m] = __ldg(kp + int64_t(ri.pool_base + pb) * kVecPerRow + 4 * m + c);
      }
    };
    uint4 ka[4], kb[4], na[4], nb[4];
    int p0 = p_begin + warp * 16;
    if (p0 < p_end) load_keys(p0, ka, kb);
    for (; p0 < p_end; p0 += kScoreWarps * 16) {
      const int pn = p0 + kScoreWarps * 16;
      if (pn < p_end) load_keys(pn, na, nb);
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
          const uint4 qf = s_q[n * 4 + m][lane];
          mma_bf16_16816(acc[n], a_lo, qf.x, qf.y);
          mma_bf16_16816(acc[n], a_hi, qf.z, qf.w);
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        ka[m] = na[m];
        kb[m] = nb[m];
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
      const int pm = c == 0 ? p0 + g : p0 + g + 8;
      const float sm = c == 0 ? sa : sb;
      const bool has = c < 2 && pm < e;
      if (has) out[pm] = sm;
      // histogram of the top bits, one shared atomic per distinct bin in the warp
      const uint32_t bin = score_order_bits(sm) >> (32 - kHistBits);
      const unsigned act = __ballot_sync(0xffffffffu, has);
      if (has) {
        const unsigned peers = __match_any_sync(act, bin);
        if ((__ffs(peers) - 1) == lane) atomicAdd(s_hist + bin, uint32_t(__popc(peers)));
      }
    }
    __syncthreads();
    uint32_t* h = hist + int64_t(r) * kHistBins;
    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) {
      const uint32_t v = s_hist[i];
      if (v) atomicAdd(h + i, v);
    }
    __syncthreads();
  }
}

// --------------------------------------------------------------- R2 collect
//
// Bin b of a row's histogram counts the pools whose score_order_bits has top
// bits b. Scanning the bins from the top, the threshold bin is the one where
// the running count first reaches the budget: every pool in a higher bin is
// chosen (fewer than budget of them), the rest of the budget comes from the
// threshold bin.
__device__ __forceinline__ void threshold_bin(const uint32_t* __restrict__ h, int budget, int* s_warp,
                                              int* out_bin, int* out_above) {
  constexpr int kPer = kHistBins / kCollectThreads;  // bins per thread, descending
  static_assert(kPer == 16, "four 16-byte loads per thread");
  const int tid = threadIdx.x;
  // thread t holds bins 4095 - 16 t down to 4080 - 16 t: cnt[i] is bin 4095 - 16 t - i
  const uint4* h4 = reinterpret_cast<const uint4*>(h + kHistBins - kPer * (tid + 1));
  uint4 v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = h4[j];
  uint32_t cnt[kPer];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    cnt[15 - 4 * j] = v[j].x;
    cnt[14 - 4 * j] = v[j].y;
    cnt[13 - 4 * j] = v[j].z;
    cnt[12 - 4 * j] = v[j].w;
  }
  int tot = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) tot += int(cnt[i]);
  int all;
  const int before = block_exclusive_scan(tot, &all, s_warp);
  if (before < budget && before + tot >= budget) {
    int run = before, i = 0;
    while (i < kPer - 1 && run + int(cnt[i]) < budget) run += int(cnt[i++]);
    *out_bin = kHistBins - 1 - (kPer * tid + i);
    *out_above = run;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kCollectThreads) rows_collect_kernel(
    const float* __restrict__ scores, int64_t stride, const RowInfo* __restrict__ info, const WorkspaceHeader* hdr,
    int budget, const uint32_t* __restrict__ hist, int32_t* cand_cnt, uint64_t* __restrict__ cand,
    int32_t* tie_cnt, uint64_t* __restrict__ ties) {
  __shared__ int s_warp[32];
  __shared__ int s_bin, s_above, s_na, s_nt, s_base_a, s_base_t;
  __shared__ uint64_t s_a[kRowsMaxBudget];
  __shared__ uint64_t s_t[kCollectTies];
  const int r = blockIdx.y;
  wait_prior_kernel();  // R1's scores and histograms
  allow_next_kernel();
  if (hdr->n_levels == 0) return;
  const RowInfo ri = info[r];
  const int e = ri.e;
  if (budget <= 0 || e <= budget || int(blockIdx.x) * kCollectPools >= e) return;  // includes invalid rows
  threshold_bin(hist + int64_t(r) * kHistBins, budget, s_warp, &s_bin, &s_above);
  const uint32_t thr = uint32_t(s_bin);
  const float* row = scores + int64_t(r) * stride;
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int p_lo = blockIdx.x * kCollectPools; p_lo < e; p_lo += gridDim.x * kCollectPools) {
    if (threadIdx.x == 0) {
      s_na = 0;
      s_nt = 0;
    }
    __syncthreads();
    const int p_hi = min(e, p_lo + kCollectPools);
    // gather this slice's pools above / inside the threshold bin in shared memory: the
    // thread's 8 consecutive scores come in two 16-byte loads (a row's stride is a
    // multiple of 4 floats, so a load that starts below e stays inside the row)
    const int p0 = p_lo + kCollectPer * threadIdx.x;
    float sv[kCollectPer];
#pragma unroll
    for (int j = 0; j < kCollectPer / 4; ++j) {
      float4 f = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (p0 + 4 * j < p_hi) f = *reinterpret_cast<const float4*>(row + p0 + 4 * j);
      sv[4 * j] = f.x;
      sv[4 * j + 1] = f.y;
      sv[4 * j + 2] = f.z;
      sv[4 * j + 3] = f.w;
    }
    // whole warps vote together on each of the eight
#pragma unroll
    for (int i = 0; i < kCollectPer; ++i) {
      const int p = p0 + i;
      const float s = sv[i];
      const bool in = p < p_hi;
      const uint32_t bin = score_order_bits(s) >> (32 - kHistBits);
      const bool above = in && bin > thr, tie = in && bin == thr;
      const unsigned ma = __ballot_sync(0xffffffffu, above), mt = __ballot_sync(0xffffffffu, tie);
      int base_a = 0, base_t = 0;
      if (lane == 0) {
        if (ma) base_a = atomicAdd(&s_na, __popc(ma));
        if (mt) base_t = atomicAdd(&s_nt, __popc(mt));
      }
      base_a = __shfl_sync(0xffffffffu, base_a, 0) + __popc(ma & lt);
      base_t = __shfl_sync(0xffffffffu, base_t, 0) + __popc(mt & lt);
      if (above && base_a < kRowsMaxBudget) s_a[base_a] = make_key(s, uint32_t(p));
      if (tie && base_t < kCollectTies) s_t[base_t] = make_key(s, uint32_t(p));
    }
    __syncthreads();
    // one reservation per slice in the row's gather lists; a slice with more ties than
    // it can hold reserves past the list's end, which sends the row to the full search
    if (threadIdx.x == 0) {
      s_base_a = s_na ? atomicAdd(cand_cnt + r, s_na) : 0;
      s_base_t = s_nt ? atomicAdd(tie_cnt + r, s_nt <= kCollectTies ? s_nt : kTieCap + 1) : 0;
    }
    __syncthreads();
    const int na = min(s_na, kRowsMaxBudget), nt = min(s_nt, kCollectTies);
    for (int i = threadIdx.x; i < na; i += kCollectThreads)
      if (s_base_a + i < kRowsMaxBudget) cand[int64_t(r) * kRowsMaxBudget + s_base_a + i] = s_a[i];
    for (int i = threadIdx.x; i < nt; i += kCollectThreads)
      if (s_base_t + i < kTieCap) ties[int64_t(r) * kTieCap + s_base_t + i] = s_t[i];
    __syncthreads();
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
    const WorkspaceHeader* hdr, int kpool, int budget, const int32_t* __restrict__ cand_cnt,
    const uint64_t* __restrict__ cand, const int32_t* __restrict__ tie_cnt, const uint64_t* __restrict__ ties,
    int32_t* __restrict__ out_ids, float* __restrict__ out_scores, int32_t* __restrict__ out_tokens) {
  __shared__ uint64_t s_ties[kTieCap];
  __shared__ SelectScratch s_sel;
  __shared__ uint32_t s_hist[256];
  __shared__ int s_warp[32];
  __shared__ uint32_t s_digit, s_above;
  __shared__ int s_count;
  __shared__ uint64_t s_keys[kRowsMaxBudget];
  __shared__ int32_t s_ids[kRowsMaxBudget];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int width = budget * kpool + kpool;
  int32_t* tok = out_tokens + int64_t(r) * width;
  wait_prior_kernel();  // R2's gather lists and counts
  // the row record and both gather counts in one round of loads (without valid
  // cu_seqlens the record is never read)
  const int n_levels = hdr->n_levels;
  const RowInfo ri_raw = info[r];
  const int cnt_above = cand_cnt[r], cnt_tie = tie_cnt[r];
  const RowInfo ri = n_levels != 0 ? ri_raw : RowInfo{0, -1, 0, 0};
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

  const int n_above = e > budget ? cnt_above : 0, n_tie = e > budget ? cnt_tie : 0;
  if (e <= budget) {
    for (int p = tid; p < e; p += kSelectThreads) s_keys[p] = make_key(row[p], uint32_t(p));
  } else if (budget > 0 && n_tie <= kTieCap) {
    // R2 gathered the n_above pools above the threshold bin and the n_tie pools in it:
    // keep the first, and the top budget - n_above of the second by full key
#pragma unroll
    for (int i = 0; i < kRowsMaxBudget / kSelectThreads; ++i) {
      const int j = tid + i * kSelectThreads;
      if (j < n_above) s_keys[j] = cand[int64_t(r) * kRowsMaxBudget + j];
    }
#pragma unroll
    for (int i = 0; i < kTieCap / kSelectThreads; ++i) {
      const int j = tid + i * kSelectThreads;
      if (j < n_tie) s_ties[j] = ties[int64_t(r) * kTieCap + j];
    }
    __syncthreads();
    const int need = budget - n_above;
    if (n_tie > need) {
      uint64_t edge;
      block_select_compact<kTieCap / kSelectThreads, kSelectThreads / 32>(s_ties, n_tie, need, 0, tid, 1, &s_sel,
                                                                         &edge);
    }
    for (int j = tid; j < need; j += kSelectThreads) s_keys[n_above + j] = s_ties[j];
  } else if (budget > 0) {
    // the threshold bin holds more pools than fit in shared memory (long runs of
    // equal scores): search the row itself
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
  {
    // the whole block ranks the (at most 512) kept keys; s_ties is free by now
    const int warp = tid >> 5;
    uint64_t k[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) k[h] = s_keys[64 * warp + 32 * h + lane];
    block_sort512_desc(k, s_ties, 1);  // k[h] is now rank 64 warp + 32 h + lane
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rank = 64 * warp + 32 * h + lane;
      if (rank < budget) {
        const bool has = rank < m && k[h] != 0ull;
        const int32_t id = has ? int32_t(key_pool(k[h])) : -1;
        s_ids[rank] = id;
        out_ids[int64_t(r) * budget + rank] = id;
        if (out_scores) out_scores[int64_t(r) * budget + rank] = has ? key_score(k[h]) : -INFINITY;
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

namespace {
// Launches `kern` with programmatic stream serialization: it may begin while the
// previous kernel on the stream runs and waits for it in wait_prior_kernel().
// Captured into a graph, the dependency becomes a programmatic edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_after_prior(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
}  // namespace

RowsLayout rows_layout(int32_t R, int64_t T, int32_t S, int32_t kpool) {
  RowsLayout L{};
  int64_t stride = T / kpool;
  stride = ((stride > 0 ? stride : 1) + 3) & ~int64_t(3);
  L.stride = stride;
  const size_t nr = size_t(R > 0 ? R : 1);
  size_t off = 0;
  L.header = off;   off = align256(off + sizeof(WorkspaceHeader));
  L.pool_off = off; off = align256(off + sizeof(int32_t) * size_t(S + 1));
  L.info = off;     off = align256(off + sizeof(RowInfo) * nr);
  L.unit_off = off; off = align256(off + sizeof(int32_t) * size_t(R + 1));
  // cleared before every call: histograms, then the two gather counters per row
  L.hist = off;     off += sizeof(uint32_t) * size_t(kHistBins) * nr;
  L.cand_cnt = off; off += sizeof(int32_t) * nr;
  L.tie_cnt = off;  off += sizeof(int32_t) * nr;
  L.cleared_bytes = off - L.hist;
  off = align256(off);
  L.cand = off;     off = align256(off + sizeof(uint64_t) * size_t(kRowsMaxBudget) * nr);
  L.ties = off;     off = align256(off + sizeof(uint64_t) * size_t(kTieCap) * nr);
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
                               int32_t* out_tokens, char* ws, const RowsLayout& L, int num_sms, int max_ctas,
                               cudaStream_t stream, void* const* stage_events) {
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  int32_t* pool_off = reinterpret_cast<int32_t*>(ws + L.pool_off);
  RowInfo* info = reinterpret_cast<RowInfo*>(ws + L.info);
  int32_t* unit_off = reinterpret_cast<int32_t*>(ws + L.unit_off);
  float* scores = reinterpret_cast<float*>(ws + L.scores);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  int32_t* cand_cnt = reinterpret_cast<int32_t*>(ws + L.cand_cnt);
  int32_t* tie_cnt = reinterpret_cast<int32_t*>(ws + L.tie_cnt);
  uint64_t* cand = reinterpret_cast<uint64_t*>(ws + L.cand);
  uint64_t* ties = reinterpret_cast<uint64_t*>(ws + L.ties);
  auto mark = [&](int i) {
    return stage_events == nullptr ? cudaSuccess
                                   : record_stage_event(stage_events[i], stream);
  };
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.hist, 0, L.cleared_bytes, stream);
  if (e != cudaSuccess) return e;
  rows_plan_kernel<<<1, 256, 0, stream>>>(cu, S, T, row_seq, row_pos, R, kpool, hdr, pool_off, info, unit_off);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return e;
  // units: at most R * ceil(max pools / kUnitPools); one wave of 2 CTAs per SM splits them
  const int64_t max_units = int64_t(R) * ((L.stride + kUnitPools - 1) / kUnitPools);
  int grid = int(max_units < int64_t(2) * num_sms ? (max_units > 0 ? max_units : 1) : int64_t(2) * num_sms);
  if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
  e = launch_after_prior(rows_score_kernel, dim3(grid), dim3(kScoreWarps * 32), stream, static_cast<const uint4*>(q),
                         w, static_cast<const uint4*>(kp), static_cast<const RowInfo*>(info),
                         static_cast<const int32_t*>(unit_off), static_cast<const WorkspaceHeader*>(hdr), R, scale,
                         scores, L.stride, hist);
  if (e == cudaSuccess) e = mark(2);
  if (e != cudaSuccess) return e;
  const int64_t slices = (L.stride + kCollectPools - 1) / kCollectPools;
  const dim3 cgrid(unsigned(slices < kCollectCtasPerRow ? slices : kCollectCtasPerRow), unsigned(R));
  e = launch_after_prior(rows_collect_kernel, cgrid, dim3(kCollectThreads), stream, static_cast<const float*>(scores),
                         L.stride, static_cast<const RowInfo*>(info), static_cast<const WorkspaceHeader*>(hdr), budget,
                         static_cast<const uint32_t*>(hist), cand_cnt, cand, tie_cnt, ties);
  if (e != cudaSuccess) return e;
  e = launch_after_prior(rows_select_kernel, dim3(R), dim3(kSelectThreads), stream, static_cast<const float*>(scores),
                         L.stride, static_cast<const RowInfo*>(info), static_cast<const WorkspaceHeader*>(hdr), kpool,
                         budget, static_cast<const int32_t*>(cand_cnt), static_cast<const uint64_t*>(cand),
                         static_cast<const int32_t*>(tie_cnt), static_cast<const uint64_t*>(ties), out_ids, out_scores,
                         out_tokens);
  if (e == cudaSuccess) e = mark(3);
  return e;
}

}  // namespace kpool
