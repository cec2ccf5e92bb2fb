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
//   R1 rows_score_kernel  (1 CTA/SM) each CTA a contiguous run of 128-pool units:
//                                   TMA pool tiles -> tcgen05.mma into TMEM ->
//                                   relu / weight / head sum per pool, fp32 scores out
//   R2 rows_collect_kernel (grid)   from a per-row histogram of the scores' top 12
//                                   bits (built by R1) finds the bin holding the
//                                   budget-th score, then gathers every pool above
//                                   that bin and the pools inside it
//   R3 rows_select_kernel (1 CTA / row) exact top-budget among the gathered pools
//                                   (ties to the smaller pool; a full MSD radix
//                                   search over the row when the bin overflows), a
//                                   256-thread bitonic sort, ids / scores / tokens
// R1-R3 use programmatic dependent launch (see wait_prior_kernel below).
// R1 streams the pooled keys once per row (HBM-bound: 256 B per pool, 8192 flop);
// its job is to keep enough of them in flight, which a deep TMA ring does.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kpool_internal.cuh"
#include "kpool_ptx.cuh"
#include "kpool_select_common.cuh"

namespace kpool {
namespace {

constexpr int kRowsHeads = 32;
constexpr int kRowsDim = 128;
constexpr int kUnitPools = 128;        // pools per work unit of R1 (the split granularity)
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
// CTA 0 plans; CTAs 1.. clear the histograms and gather counters (`clear`, n_clear
// 32-bit words, 16-byte aligned) that R1 and R2 accumulate into.
__global__ void __launch_bounds__(256) rows_plan_kernel(const int32_t* __restrict__ cu, int S, int64_t T,
                                                         const int32_t* __restrict__ row_seq,
                                                         const int32_t* __restrict__ row_pos, int R, int kpool,
                                                         WorkspaceHeader* hdr, int32_t* pool_off, RowInfo* info,
                                                         int32_t* unit_off, uint32_t* __restrict__ clear,
                                                         int64_t n_clear) {
  __shared__ int s_bad, s_bad_row;
  __shared__ int s_warp[32];
  const int tid = threadIdx.x;
  allow_next_kernel();
  if (blockIdx.x > 0) {
    const int64_t n4 = n_clear / 4;
    const int64_t stride = int64_t(gridDim.x - 1) * blockDim.x;
    uint4* c4 = reinterpret_cast<uint4*>(clear);
    for (int64_t i = int64_t(blockIdx.x - 1) * blockDim.x + tid; i < n4; i += stride) c4[i] = make_uint4(0, 0, 0, 0);
    for (int64_t i = 4 * n4 + int64_t(blockIdx.x - 1) * blockDim.x + tid; i < n_clear; i += stride) clear[i] = 0;
    return;
  }
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
// Per work unit (128 pools of one row) the TMA producer (warp 0) loads the
// [128 pools x 128] bf16 pooled-key tile (32 KB, 128-byte swizzle) into a 6-stage
// ring and, when the row changes, the row's [32 heads x 128] query tile. The MMA
// issuer (warp 1, owner of 128 TMEM columns) multiplies them as 8 tcgen05.mma
// (M = 128 pools, N = 32 heads, K = 16 each) into one of four 32-column fp32
// accumulators. Four epilogue warps (warp w reads TMEM lanes 32 (w % 4) ..) take one
// pool per thread: its 32 head products come in with one tcgen05.ld, then relu,
// |scale| and the head weights and the head sum, in the score kernel's arithmetic
// (x + |x| against halved weights, packed fp32 FMAs, pairs summed last), the score is
// stored and its top bits counted in the CTA's histogram of the row, which is added
// to the row's global histogram when the row ends. Every mbarrier wait is bounded;
// a wait that runs out records KPOOL_ERR_DEVICE_TIMEOUT and every role winds down.
namespace r1 {
constexpr int kThreads = 192;                                // producer, MMA issuer, 4 epilogue warps
constexpr int kStages = 6;                                   // pool tiles in flight
constexpr int kAccs = 4;                                     // TMEM accumulators
constexpr int kAccCols = kRowsHeads;                         // 32 fp32 columns each
constexpr int kTmemCols = kAccs * kAccCols;                  // 128 (a power of two >= 32)
constexpr uint32_t kPoolHalf = kUnitPools * 128;             // 128 pools x 64 bf16
constexpr uint32_t kStageBytes = 2 * kPoolHalf;              // 32 KB
constexpr uint32_t kQHalf = kRowsHeads * 128;                // 32 heads x 64 bf16
constexpr uint32_t kQBytes = 2 * kQHalf;                     // 8 KB
constexpr uint32_t kOffPool = 0;
constexpr uint32_t kOffQ = kOffPool + kStages * kStageBytes;  // 1024-byte aligned
constexpr uint32_t kOffHist = kOffQ + kQBytes;
constexpr uint32_t kOffBar = kOffHist + kHistBins * 4;
constexpr int kNumBars = 2 * kStages + 2 * kAccs + 3;        // full, empty, acc_full, acc_empty, q_full, q_empty, mma_done
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;        // TMEM base, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16;
static_assert(kOffQ % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
constexpr int64_t kMaxPolls = int64_t(1) << 40;
constexpr uint64_t kMaxWaitNs = 1000000000ull;  // 1 s; legitimate waits are microseconds
constexpr int kEpiBar = 1;                       // named barrier of the 4 epilogue warps
constexpr int kEndBar = 2;                       // named barrier of the whole CTA at teardown

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Row of unit u: the last r with unit_off[r] <= u (rows without units are skipped).
__device__ __forceinline__ int row_of_unit(const int32_t* unit_off, int R, int u) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(unit_off + mid) <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}
}  // namespace r1

__global__ void __launch_bounds__(r1::kThreads, 1) rows_score_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kp,
    const float* __restrict__ w, const RowInfo* __restrict__ info, const int32_t* __restrict__ unit_off,
    WorkspaceHeader* __restrict__ hdr, int R, float scale, float* __restrict__ scores, int64_t stride,
    uint32_t* __restrict__ hist) {
  using namespace r1;
  extern __shared__ __align__(1024) uint8_t smem[];
  allow_next_kernel();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a uniform exit, before any barrier or TMEM allocation (the error word is written
  // only after the planning kernel, which resets it, has finished)
  if ((ptx::smem_addr(smem) & 1023u) != 0) {
    wait_prior_kernel();
    if (threadIdx.x == 0) record_error(hdr, KPOOL_ERR_INTERNAL);
    return;
  }
  // the set-up below reads nothing the planning kernel writes, so it runs while that
  // kernel finishes (programmatic dependent launch)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + kAccs;
  uint64_t* q_full = acc_empty + kAccs;
  uint64_t* q_empty = q_full + 1;
  uint64_t* mma_done = q_empty + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + kOffMisc + 4);
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(full + i, 1);
      ptx::mbar_init(empty + i, 1);
    }
    for (int i = 0; i < kAccs; ++i) {
      ptx::mbar_init(acc_full + i, 1);
      ptx::mbar_init(acc_empty + i, 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    ptx::mbar_init(mma_done, 1);
    ptx::fence_mbar_init();
    *abort_flag = 0;
    ptx::prefetch_tmap(&tmap_q);
    ptx::prefetch_tmap(&tmap_kp);
  }
  if (warp == 1) {
    ptx::tmem_alloc(s_tmem, kTmemCols);
    ptx::tmem_relinquish();
  }
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) s_hist[i] = 0;
  wait_prior_kernel();  // the plan: n_items, row records, unit offsets (and the cleared histograms)
  const int n_units = hdr->n_items;  // 0 when the plan found cu_seqlens malformed
  const int u_first = int(int64_t(n_units) * blockIdx.x / gridDim.x);
  const int u_last = int(int64_t(n_units) * (blockIdx.x + 1) / gridDim.x);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (u_first >= u_last) {
    // no units for this CTA: straight to the teardown (TMEM is still freed there)
  } else if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- producer
      const uint64_t pol = ptx::policy_evict_first();  // every key tile is read once
      int stage = 0, r = row_of_unit(unit_off, R, u_first), cur = -1;
      uint32_t phase = 0, fills = 0, q_loads = 0;
      bool ok = true;
      for (int u = u_first; u < u_last; ++u) {
        while (__ldg(unit_off + r + 1) <= u) ++r;
        if (r != cur) {  // the row's query tile, once the previous row's MMAs are done with it
          if (q_loads > 0 && !ptx::mbar_wait_bounded(q_empty, (q_loads - 1) & 1, kMaxPolls, kMaxWaitNs)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(q_full, kQBytes);
          ptx::tma_load_2d_hint(smem + kOffQ, &tmap_q, q_full, 0, r * kRowsHeads, pol);
          ptx::tma_load_2d_hint(smem + kOffQ + kQHalf, &tmap_q, q_full, 64, r * kRowsHeads, pol);
          ++q_loads;
          cur = r;
        }
        if (!ptx::mbar_wait_bounded(empty + stage, phase ^ 1, kMaxPolls, kMaxWaitNs) || *abort_flag) {
          ok = false;
          break;
        }
        const int32_t prow = info[r].pool_base + (u - __ldg(unit_off + r)) * kUnitPools;
        uint8_t* dst = smem + kOffPool + stage * kStageBytes;
        ptx::mbar_arrive_expect_tx(full + stage, kStageBytes);
        ptx::tma_load_2d_hint(dst, &tmap_kp, full + stage, 0, prow, pol);
        ptx::tma_load_2d_hint(dst + kPoolHalf, &tmap_kp, full + stage, 64, prow, pol);
        ++fills;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      // every copy armed above lands before the CTA exits
      for (int s2 = 0; s2 < kStages; ++s2) {
        const uint32_t armed = (fills + kStages - 1 - s2) / kStages;
        if (armed) ptx::mbar_wait_bounded(full + s2, (armed - 1) & 1, kMaxPolls, kMaxWaitNs);
      }
      if (q_loads) ptx::mbar_wait_bounded(q_full, (q_loads - 1) & 1, kMaxPolls, kMaxWaitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------------ MMA
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kUnitPools, kRowsHeads);
      const uint32_t pool_addr = ptx::smem_addr(smem + kOffPool), q_addr = ptx::smem_addr(smem + kOffQ);
      int stage = 0, acc = 0, r = row_of_unit(unit_off, R, u_first), cur = -1;
      uint32_t phase = 0, acc_phase = 0, q_uses = 0;
      bool ok = true;
      for (int u = u_first; u < u_last; ++u) {
        while (__ldg(unit_off + r + 1) <= u) ++r;
        if (r != cur) {
          if (!ptx::mbar_wait_bounded(q_full, q_uses & 1, kMaxPolls, kMaxWaitNs)) {
            ok = false;
            break;
          }
          ++q_uses;
          cur = r;
        }
        if (!ptx::mbar_wait_bounded(acc_empty + acc, acc_phase ^ 1, kMaxPolls, kMaxWaitNs) ||
            !ptx::mbar_wait_bounded(full + stage, phase, kMaxPolls, kMaxWaitNs) || *abort_flag) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_base = pool_addr + stage * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a_addr = a_base + (kk >> 2) * kPoolHalf + (kk & 3) * 32;
          const uint32_t b_addr = q_addr + (kk >> 2) * kQHalf + (kk & 3) * 32;
          ptx::tc_mma_f16(tmem_base + uint32_t(acc * kAccCols), ptx::smem_desc_kmajor_sw128(a_addr),
                          ptx::smem_desc_kmajor_sw128(b_addr), idesc, kk > 0 ? 1u : 0u);
        }
        ptx::tc_commit(empty + stage);
        ptx::tc_commit(acc_full + acc);
        if (u + 1 == u_last || __ldg(unit_off + r + 1) <= u + 1) ptx::tc_commit(q_empty);  // row's last unit
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == kAccs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      ptx::tc_commit(mma_done);  // every MMA issued above completes before TMEM is freed
      ptx::mbar_wait_bounded(mma_done, 0, kMaxPolls, kMaxWaitNs);
    }
  } else {  // ---------------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64;  // 0..127
    const int lq = warp & 3;          // TMEM lane quarter this warp may read
    const uint32_t lane_addr = tmem_base + (uint32_t(lq * 32) << 16);
    const float abs_scale = fabsf(scale);
    const bool neg = scale < 0.0f;
    int acc = 0, r = row_of_unit(unit_off, R, u_first), cur = -1;
    uint32_t acc_phase = 0;
    uint64_t wp[kRowsHeads / 2];  // halved |scale| w of head pairs
    RowInfo ri{};
    auto flush_hist = [&](int row) {  // the CTA's counts of `row` into the row's histogram
      named_bar(kEpiBar, 128);
      uint32_t* h = hist + int64_t(row) * kHistBins;
      for (int i = et; i < kHistBins; i += 128) {
        const uint32_t v = s_hist[i];
        if (v) {
          atomicAdd(h + i, v);
          s_hist[i] = 0;
        }
      }
      named_bar(kEpiBar, 128);
    };
    for (int u = u_first; u < u_last; ++u) {
      while (__ldg(unit_off + r + 1) <= u) ++r;
      if (r != cur) {
        if (cur >= 0) flush_hist(cur);
        ri = info[r];
#pragma unroll
        for (int h2 = 0; h2 < kRowsHeads / 2; ++h2)
          wp[h2] = ptx::pack_f32x2((__ldg(w + int64_t(r) * kRowsHeads + 2 * h2) * abs_scale) * 0.5f,
                                   (__ldg(w + int64_t(r) * kRowsHeads + 2 * h2 + 1) * abs_scale) * 0.5f);
        cur = r;
      }
      // every lane tests the barrier; after an abort the units are only counted off
      const bool ready = *abort_flag == 0 &&
                         __all_sync(0xffffffffu, ptx::mbar_wait_bounded(acc_full + acc, acc_phase, kMaxPolls,
                                                                        kMaxWaitNs));
      if (ready) {
        ptx::tc_fence_after();
        uint32_t v[32];
        ptx::tc_ld_32x32b_x32(lane_addr + uint32_t(acc * kAccCols), v);
        ptx::tc_wait_ld();
        ptx::tc_reg_fence(v);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(acc_empty + acc);
        uint64_t a0 = 0, a1 = 0;
#pragma unroll
        for (int h4 = 0; h4 < kRowsHeads / 4; ++h4) {
          const float x0 = __uint_as_float(v[4 * h4 + 0]), x1 = __uint_as_float(v[4 * h4 + 1]);
          const float x2 = __uint_as_float(v[4 * h4 + 2]), x3 = __uint_as_float(v[4 * h4 + 3]);
          // x + |x| = 2 relu(x) exactly (|x| - x for a negative scale) against halved weights
          a0 = ptx::fma_f32x2(wp[2 * h4], ptx::pack_f32x2(neg ? fabsf(x0) - x0 : x0 + fabsf(x0),
                                                          neg ? fabsf(x1) - x1 : x1 + fabsf(x1)), a0);
          a1 = ptx::fma_f32x2(wp[2 * h4 + 1], ptx::pack_f32x2(neg ? fabsf(x2) - x2 : x2 + fabsf(x2),
                                                              neg ? fabsf(x3) - x3 : x3 + fabsf(x3)), a1);
        }
        float s0, s1, s2, s3;
        ptx::unpack_f32x2(a0, s0, s1);
        ptx::unpack_f32x2(a1, s2, s3);
        const float sc = (s0 + s1) + (s2 + s3);
        const int p = (u - __ldg(unit_off + r)) * kUnitPools + lq * 32 + lane;
        const bool has = p < ri.e;
        if (has) scores[int64_t(r) * stride + p] = sc;
        // histogram of the top bits, one shared atomic per distinct bin in the warp
        const uint32_t bin = score_order_bits(sc) >> (32 - kHistBits);
        const unsigned act = __ballot_sync(0xffffffffu, has);
        if (has) {
          const unsigned peers = __match_any_sync(act, bin);
          if ((__ffs(peers) - 1) == lane) atomicAdd(s_hist + bin, uint32_t(__popc(peers)));
        }
      } else if (lane == 0 && *abort_flag == 0) {
        record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
      }
      if (++acc == kAccs) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (cur >= 0) flush_hist(cur);
    ptx::tc_fence_before();
  }
  // ---------------------------------------------------------------------- teardown
  __syncwarp();
  named_bar(kEndBar, kThreads);
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
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

// ---------------------------------------------------------------- R3 select
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
cudaError_t launch_after_prior(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
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
  if (e != cudaSuccess) return e;
  // one planning CTA, and enough clearing CTAs that each clears about 32 KB
  const int64_t clear_ctas = (int64_t(L.cleared_bytes) + 32767) / 32768;
  const unsigned plan_grid = unsigned(1 + (clear_ctas < 2 * num_sms ? clear_ctas : 2 * num_sms));
  rows_plan_kernel<<<plan_grid, 256, 0, stream>>>(cu, S, T, row_seq, row_pos, R, kpool, hdr, pool_off, info,
                                                   unit_off, reinterpret_cast<uint32_t*>(ws + L.hist),
                                                   int64_t(L.cleared_bytes / 4));
  e = cudaGetLastError();
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return e;
  // units: at most R * ceil(max pools / kUnitPools); one persistent CTA per SM splits them
  const int64_t max_units = int64_t(R) * ((L.stride + kUnitPools - 1) / kUnitPools);
  int grid = int(max_units < num_sms ? (max_units > 0 ? max_units : 1) : num_sms);
  if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
  // no pooled keys (T / kpool == 0): every row has no eligible pool and no unit to score
  if (kp != nullptr && T / kpool > 0) {
    CUtensorMap map_q, map_kp;
    if (!make_tmap_bf16_k128(&map_q, q, uint64_t(R) * kRowsHeads, kRowsHeads) ||
        !make_tmap_bf16_k128(&map_kp, kp, uint64_t(T / kpool), kUnitPools))
      return cudaErrorInvalidValue;
    static bool attr_set[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= 64 || !attr_set[dev])) {
      e = cudaFuncSetAttribute(rows_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(r1::kSmemBytes));
      if (e == cudaSuccess && dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    if (e != cudaSuccess) return e;
    e = launch_after_prior(rows_score_kernel, dim3(grid), dim3(r1::kThreads), r1::kSmemBytes, stream, map_q, map_kp,
                           w, static_cast<const RowInfo*>(info), static_cast<const int32_t*>(unit_off), hdr, R, scale,
                           scores, L.stride, hist);
  }
  if (e == cudaSuccess) e = mark(2);
  if (e != cudaSuccess) return e;
  const int64_t slices = (L.stride + kCollectPools - 1) / kCollectPools;
  const dim3 cgrid(unsigned(slices < kCollectCtasPerRow ? slices : kCollectCtasPerRow), unsigned(R));
  e = launch_after_prior(rows_collect_kernel, cgrid, dim3(kCollectThreads), 0, stream, static_cast<const float*>(scores),
                         L.stride, static_cast<const RowInfo*>(info), static_cast<const WorkspaceHeader*>(hdr), budget,
                         static_cast<const uint32_t*>(hist), cand_cnt, cand, tie_cnt, ties);
  if (e != cudaSuccess) return e;
  e = launch_after_prior(rows_select_kernel, dim3(R), dim3(kSelectThreads), 0, stream, static_cast<const float*>(scores),
                         L.stride, static_cast<const RowInfo*>(info), static_cast<const WorkspaceHeader*>(hdr), kpool,
                         budget, static_cast<const int32_t*>(cand_cnt), static_cast<const uint64_t*>(cand),
                         static_cast<const int32_t*>(tie_cnt), static_cast<const uint64_t*>(ties), out_ids, out_scores,
                         out_tokens);
  if (e == cudaSuccess) e = mark(3);
  return e;
}

}  // namespace kpool
