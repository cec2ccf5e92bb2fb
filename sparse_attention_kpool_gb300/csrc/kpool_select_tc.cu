// kpool_select_tc.cu -- K2 on the 5th-generation tensor cores: fused score +
// streaming top-budget selection for bf16 inputs, 32 index heads, d = 128.
//
// What it computes, per query row t (sequence-local) and eligible pool
// p < floor((t+1)/kpool):
//   s[t,p] = sum_h w[t,h] * relu(scale * q[t,h,:] . kp[p,:])
// ("spark_model/layers/glm5next_dsa/tp.rs", module docs: index_scores
// accumulates weights[h] * relu(scale . dot) as a plain sum over heads, before
// any top-k), then the top budget = index_topk/kpool pools of the row under
// "higher score, then smaller pool index" (same page: the deterministic
// tiebreak). Every query scores every eligible pool, as on the pages ("NVIDIA/
// Megatron-LM pull request #8299", "What does this PR do": O(queries x pools)),
// but only the causally eligible tiles are visited and the [rows, pools] score
// matrix never leaves the SM.
//
// Work item = 8 consecutive query rows of one sequence (the planning kernel
// lists them deepest-first; CTAs take the next one from a global counter). Per
// item the dot products form one dense
// contraction per tile of 128 pools:
//   D[p, (t,h)] = kp[p,:] . q[t,h,:]     M = 128 pools, N = 8 rows x 32 heads = 256, K = 128
// issued as 8 tcgen05.mma (K = 16 each) with bf16 operands staged by TMA in
// 128-byte-swizzled shared memory and an fp32 accumulator in TMEM. Pools sit on
// the M axis (TMEM lanes) so each epilogue thread owns one pool and sums the 32
// heads of a query inside its own registers -- no shuffles.
//
// Warp roles (10 warps, one CTA per SM, persistent):
//   warp 0      TMA producer: fetches the next work item and hands its index to
//               the other roles through a 4-slot ring, then loads the item's q
//               tile (64 KB) and its pool tiles into a 2-stage ring (32 KB each);
//               a third stage measured no faster and its 32 KB buys 50% larger
//               candidate buffers instead.
//   warp 1      TMEM owner and MMA issuer: two 256-column accumulators, so the
//               epilogue drains one while the tensor core fills the other.
//   warps 2..9  epilogue, two groups of four warps; group g owns rows 4g..4g+3
//               of every item and reads their 128 columns of every accumulator;
//               warp w reads TMEM lanes 32*(w%4).. (the hardware rule). The
//               groups synchronise only within themselves. Per row: tcgen05.ld
//               (the next row's columns and head weights load meanwhile) -> relu,
//               |scale|*w, head sum in fp32 -> selection key -> threshold filter
//               -> candidate buffer in shared memory. The relu runs on the FMA
//               pipe as x + |x| (twice relu(x), exactly) against halved weights,
//               so packed f32x2 FMAs round the same products as w * relu(x) while
//               the ALU pipe carries only the selection's integer work.
// Selection: 1536 candidate slots per query row, in four 384-slot regions, one
// per warp of the owning group, so a warp appends with a register count and no
// atomics. A key enters only if it beats the row's threshold. When a region
// passes 352 entries the group's four warps run a radix threshold search over the
// row together and keep between budget and budget+64 keys, spread evenly over the
// regions; the threshold rises to the search's edge. After the last tile each row
// is cut to exactly `budget` keys the same way, then one warp per row sorts them
// in registers (bitonic) and writes the ranked ids.
//
// Index-score mode (kScores): the same producer, MMA issuer and scoring loop,
// but every epilogue thread stores its fp32 score to a [rows, ld] matrix (-inf
// where the pool is not eligible) instead of filtering it, and after an item's
// tiles the group writes -inf to the rest of its rows. This is the pages' full
// score output ("NVIDIA/Megatron-LM pull request #8299", section "Change":
// return_index_scores), bounded by the caller's row range as the pages bound
// their score chunks. The scores are bit-identical to the ones the selection
// ranks.
//
// The producer and MMA roles, the cooperative compaction and the final ranking
// are noinline functions: kept out of the kernel body, their code does not shape
// the register allocation of the epilogue's scoring loop (measured: 4-5 % faster at
// 512k tokens, 8 % at 128k).
//
// Every mbarrier wait is bounded (poll count and ~1 s of wall time). A wait that
// runs out records KPOOL_ERR_DEVICE_TIMEOUT in the workspace header; all roles
// then leave their loops through the same barriers, drain their in-flight copies
// and MMAs, and the TMEM owner frees TMEM before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include "kpool_internal.cuh"
#include "kpool_ptx.cuh"
#include "kpool_select_common.cuh"

namespace kpool {
namespace {

constexpr int kHeads = 32;
constexpr int kDim = 128;
constexpr int kRows = kItemRows;          // query rows per item
constexpr int kN = kRows * kHeads;        // 256 MMA columns
constexpr int kTilePools = 128;           // MMA M
#ifndef KPOOL_TC_STAGES
#define KPOOL_TC_STAGES 2
#endif
#ifndef KPOOL_TC_CAP
#define KPOOL_TC_CAP 1536
#endif
#ifndef KPOOL_TC_SLACK
#define KPOOL_TC_SLACK 64
#endif
constexpr int kStages = KPOOL_TC_STAGES;  // pool-tile ring depth
constexpr int kCap = KPOOL_TC_CAP;        // candidate slots per query row
constexpr int kMaxBudget = 512;
// A tile adds at most one candidate per pool to a row (128), so a row is
// compacted once it holds more than kCap - 128 after a tile.
constexpr int kCompactAt = kCap - kTilePools;
static_assert(kCap % 128 == 0, "a group's cooperative compaction gives each of 128 threads kCap/128 keys");
// Each row's buffer is split into four regions, one per warp of the owning group,
// so a warp inserts with a register count and no atomics. A warp adds at most 32
// candidates to a region per tile, so a row is compacted once a region passes
// kReg - 32.
constexpr int kReg = kCap / 4;
constexpr int kRegMark = kReg - 32;
// A compaction spreads the keys it keeps evenly over the four regions: a round's
// keeps at most budget + slack keys, the final one at most budget.
constexpr int kFinalChunk = kMaxBudget / 4;  // most keys a region holds after the final compaction
static_assert(kMaxBudget % 128 == 0 && kFinalChunk % 32 == 0, "the final sort reads whole warps per region");
static_assert((kMaxBudget + KPOOL_TC_SLACK + 3) / 4 < kRegMark, "a compaction must free room in every region");
constexpr int kSlack = KPOOL_TC_SLACK;    // a compaction keeps between budget and budget + kSlack keys
static_assert(kMaxBudget + kSlack < kCompactAt, "a compaction must free room for the next round");
constexpr int kThreads = 320;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kQHalfBytes = kN * 128;                  // 256 rows x 64 bf16
constexpr uint32_t kQBytes = 2 * kQHalfBytes;               // 64 KB
constexpr uint32_t kPoolHalfBytes = kTilePools * 128;       // 128 rows x 64 bf16
constexpr uint32_t kStageBytes = 2 * kPoolHalfBytes;        // 32 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffPool = kOffQ + kQBytes;
constexpr uint32_t kOffCand = kOffPool + kStages * kStageBytes;
constexpr uint32_t kOffW = kOffCand + kRows * kCap * 8;
constexpr uint32_t kOffBar = kOffW + kRows * kHeads * 4;
constexpr int kRing = 4;  // work items handed from the producer to the MMA issuer and the epilogue
constexpr int kNumBars = 2 + 2 * kStages + 4 + 1 + 2 * kRing;
constexpr uint32_t kOffCount = kOffBar + kNumBars * 8;         // [kRows][4] region counts
constexpr uint32_t kOffTau = (kOffCount + kRows * 4 * 4 + 7) & ~7u;
constexpr uint32_t kOffElig = kOffTau + kRows * 8;
constexpr uint32_t kOffMisc = kOffElig + kRows * 4;
constexpr uint32_t kOffRing = kOffMisc + 16;                // [kRing] item indices
constexpr uint32_t kOffSelect = kOffRing + 4 * kRing;       // SelectScratch
constexpr uint32_t kSelectBytes = (sizeof(SelectScratch) + 15) & ~size_t(15);
constexpr uint32_t kSmemUsed = kOffSelect + 2 * kSelectBytes;  // one SelectScratch per epilogue group
constexpr uint32_t kSmemBytes = kSmemUsed;
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

#ifndef KPOOL_TC_BACKOFF_NS
#define KPOOL_TC_BACKOFF_NS 0
#endif
constexpr int64_t kMaxPolls = int64_t(1) << 40;
constexpr uint32_t kBackoffNs = KPOOL_TC_BACKOFF_NS;  // producer / MMA poll back-off
constexpr uint64_t kMaxWaitNs = 1000000000ull;  // 1 s; legitimate waits are microseconds

struct Bars {
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* full;       // [kStages]
  uint64_t* empty;      // [kStages]
  uint64_t* acc_full;   // [2]
  uint64_t* acc_empty;  // [2]
  uint64_t* mma_done;
  uint64_t* ring_full;   // [kRing]: the producer wrote the slot's item index
  uint64_t* ring_empty;  // [kRing]: the MMA issuer and the 8 epilogue warps read it
};

__device__ __forceinline__ Bars bars_at(uint8_t* base) {
  uint64_t* b = reinterpret_cast<uint64_t*>(base + kOffBar);
  Bars r;
  r.q_full = b + 0;
  r.q_empty = b + 1;
  r.full = b + 2;
  r.empty = b + 2 + kStages;
  r.acc_full = b + 2 + 2 * kStages;
  r.acc_empty = b + 4 + 2 * kStages;
  r.mma_done = b + 6 + 2 * kStages;
  r.ring_full = b + 7 + 2 * kStages;
  r.ring_empty = b + 7 + 2 * kStages + kRing;
  return r;
}

// Non-.aligned barrier forms: a warp may arrive with its lanes diverged (the
// producer and MMA warps do their work on lane 0 only).
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a flag over the participating threads, so a
// decision taken after it is the same in every participating warp.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool flag) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "barrier.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(id), "r"(count), "r"(flag ? 1u : 0u)
      : "memory");
  return out != 0;
}

struct Item {
  int64_t seq_start;  // global row of the sequence's first token
  int32_t len;        // sequence length
  int32_t t0;         // first local row of the item
  int32_t rows;       // valid rows in the item (<= kRows)
  int32_t pool_base;  // global pooled-key row of the sequence's pool 0
  int32_t n_tiles;    // pool tiles covering the last row's eligible pools
};

__device__ __forceinline__ Item load_item(const int2* items, const int32_t* cu, const int32_t* pool_off, int idx,
                                          int kpool) {
  const int2 it = items[idx];
  Item m;
  m.seq_start = cu[it.x];
  m.len = cu[it.x + 1] - cu[it.x];
  m.t0 = it.y * kRows;
  m.rows = min(kRows, m.len - m.t0);
  m.pool_base = pool_off[it.x];
  const int e_max = (m.t0 + m.rows) / kpool;  // eligible pools of the item's last row
  m.n_tiles = (e_max + kTilePools - 1) / kTilePools;
  return m;
}

// Cooperative compaction of one row's candidates by the epilogue group's four warps
// (thread gt of 128, named barrier bar_id): keeps between budget and budget + slack
// keys (exactly budget for slack 0), dealt evenly back over the four regions, whose
// counts cnt4[0..3] it updates. With `tau`, thread 0 stores the new admission bound
// (edge - 1: from now on a key must reach the edge to matter). Kept out of line:
// inlined, its code costs the scoring loop around it 3-4 % (register allocation).
__device__ __noinline__ void compact_row(uint64_t* buf, int32_t* cnt4, int budget, int slack, int gt, int bar_id,
                                         SelectScratch* sel, uint64_t* tau) {
  using L = QuarteredLayout<kReg>;
  const int32_t* c = cnt4;
  uint64_t edge;
  const int kept = block_select_compact_in<kCap / 128, 4>(buf, c[0] + c[1] + c[2] + c[3], budget, slack, gt, bar_id,
                                                         sel, &edge, L{c});
  if (gt < 4) cnt4[gt] = L::region_count(kept, gt);  // block_select_compact_in ends with a group barrier
  if (tau != nullptr && gt == 0) *tau = edge - 1;
}

// Final ranking of one row by one warp: its candidates (at most kFinalChunk per
// region, at most budget in all) sorted, then the first `budget` ranks written as
// pool ids (-1 for empty slots) and, when sc_row is given, scores (-inf). Kept out of
// line: inlined, the unrolled sort network changes the register allocation of the
// scoring loop around it, which then runs slower than the sort gains.
__device__ __noinline__ void rank_and_write_row(const uint64_t* buf, const int32_t* c, int budget, int32_t* ids_row,
                                                float* sc_row) {
  const int lane = threadIdx.x & 31;
  uint64_t kk[kMaxBudget / 32];
#pragma unroll
  for (int j = 0; j < kMaxBudget / 32; ++j) {
    constexpr int kPerRegion = kFinalChunk / 32;
    const int r = j / kPerRegion, off = (j % kPerRegion) * 32 + lane;  // region, offset
    kk[j] = off < c[r] ? buf[r * kReg + off] : 0ull;
  }
  warp_sort512_blocked_desc(kk);  // lane l now holds ranks 16 l .. 16 l + 15
  const int o0 = 16 * lane;
  if (o0 + 16 <= budget && (reinterpret_cast<uintptr_t>(ids_row + o0) & 15u) == 0) {  // 16-byte vector stores
    int4* dst = reinterpret_cast<int4*>(ids_row + o0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int4 v;
      v.x = kk[4 * j + 0] ? int32_t(key_pool(kk[4 * j + 0])) : -1;
      v.y = kk[4 * j + 1] ? int32_t(key_pool(kk[4 * j + 1])) : -1;
      v.z = kk[4 * j + 2] ? int32_t(key_pool(kk[4 * j + 2])) : -1;
      v.w = kk[4 * j + 3] ? int32_t(key_pool(kk[4 * j + 3])) : -1;
      dst[j] = v;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (o0 + j < budget) ids_row[o0 + j] = kk[j] ? int32_t(key_pool(kk[j])) : -1;
  }
  if (sc_row) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (o0 + j < budget) sc_row[o0 + j] = kk[j] ? key_score(kk[j]) : -INFINITY;
  }
}

// Producer (one thread of warp 0): takes work items from the global counter and
// hands them to the MMA issuer and the epilogue through the ring, then streams each
// item's query block and pool tiles into shared memory with TMA. The two warp roles
// that run on a single thread are separate functions so the epilogue's code (the
// kernel body) is allocated on its own.
__device__ __noinline__ void producer_role(const CUtensorMap* tmap_q, const CUtensorMap* tmap_kp, const int32_t* cu,
                                           const int32_t* pool_off, const int2* items, WorkspaceHeader* hdr, int kpool,
                                           int n_items) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Bars bar = bars_at(smem);
  volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + kOffMisc + 4);
  volatile int32_t* s_ring = reinterpret_cast<volatile int32_t*>(smem + kOffRing);
  const uint64_t pol_q = ptx::policy_evict_first();
  const uint64_t pol_kp = ptx::policy_evict_last();
  int stage = 0;
  uint32_t phase = 0, q_phase = 0;
  uint32_t fills = 0;  // pool-tile fills armed so far (stage = fill index mod kStages)
  uint32_t q_armed = 0;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    // next work item from the global counter (heaviest first, as the plan sorted
    // them), handed to the MMA issuer and the epilogue through the ring
    const int slot = r % kRing;
    const uint32_t use = uint32_t(r / kRing);
    if (use > 0 && !ptx::mbar_wait_bounded(bar.ring_empty + slot, (use - 1) & 1, kMaxPolls, kMaxWaitNs,
                                           kBackoffNs)) {
      ok = false;
      break;
    }
    int idx = atomicAdd(&hdr->next_item, 1);
    if (idx >= n_items) idx = -1;
    s_ring[slot] = idx;
    ptx::mbar_arrive(bar.ring_full + slot);
    if (idx < 0) break;
    const Item it = load_item(items, cu, pool_off, idx, kpool);
    if (it.n_tiles == 0) continue;
    if (!ptx::mbar_wait_bounded(bar.q_empty, q_phase ^ 1, kMaxPolls, kMaxWaitNs, kBackoffNs) || *abort_flag) {
      ok = false;
      break;
    }
    q_phase ^= 1;
    uint8_t* qdst = smem + kOffQ;
    const int32_t qrow = int32_t((it.seq_start + it.t0) * kHeads);
    ptx::mbar_arrive_expect_tx(bar.q_full, kQBytes);
    ptx::tma_load_2d_hint(qdst, tmap_q, bar.q_full, 0, qrow, pol_q);
    ptx::tma_load_2d_hint(qdst + kQHalfBytes, tmap_q, bar.q_full, 64, qrow, pol_q);
    ++q_armed;
    for (int i = 0; i < it.n_tiles; ++i) {
      if (!ptx::mbar_wait_bounded(bar.empty + stage, phase ^ 1, kMaxPolls, kMaxWaitNs, kBackoffNs) ||
          *abort_flag) {
        ok = false;
        break;
      }
      uint8_t* dst = smem + kOffPool + stage * kStageBytes;
      const int32_t prow = it.pool_base + i * kTilePools;
      ptx::mbar_arrive_expect_tx(bar.full + stage, kStageBytes);
      ptx::tma_load_2d_hint(dst, tmap_kp, bar.full + stage, 0, prow, pol_kp);
      ptx::tma_load_2d_hint(dst + kPoolHalfBytes, tmap_kp, bar.full + stage, 64, prow, pol_kp);
      ++fills;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  if (!ok) {
    record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
    *abort_flag = 1;
  }
  // drain: the last fill armed on each barrier must land before the CTA exits
  for (uint32_t s = 0; s < kStages; ++s) {
    const uint32_t armed = (fills + kStages - 1 - s) / kStages;  // fills that went to stage s
    if (armed) ptx::mbar_wait_bounded(bar.full + s, (armed - 1) & 1, kMaxPolls, kMaxWaitNs);
  }
  if (q_armed) ptx::mbar_wait_bounded(bar.q_full, (q_armed - 1) & 1, kMaxPolls, kMaxWaitNs);
}

// MMA issuer (one thread of warp 1): for every pool tile of every item, 8 K16
// tcgen05 MMAs of [128 pools x 128] x [128 x 256 query-head columns] into one of the
// two TMEM accumulators, committed to the epilogue's acc_full barrier.
__device__ __noinline__ void mma_role(const int32_t* cu, const int32_t* pool_off, const int2* items,
                                      WorkspaceHeader* hdr, int kpool, uint32_t tmem_base) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Bars bar = bars_at(smem);
  volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + kOffMisc + 4);
  volatile int32_t* s_ring = reinterpret_cast<volatile int32_t*>(smem + kOffRing);
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTilePools, kN);
  const uint32_t q_addr = ptx::smem_addr(smem + kOffQ);
  const uint32_t pool_addr = ptx::smem_addr(smem + kOffPool);
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0, q_phase = 0;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int slot = r % kRing;
    if (!ptx::mbar_wait_bounded(bar.ring_full + slot, uint32_t(r / kRing) & 1, kMaxPolls, kMaxWaitNs,
                                kBackoffNs)) {
      ok = false;
      break;
    }
    const int idx = s_ring[slot];
    ptx::mbar_arrive(bar.ring_empty + slot);
    if (idx < 0) break;
    const Item it = load_item(items, cu, pool_off, idx, kpool);
    if (it.n_tiles == 0) continue;
    if (!ptx::mbar_wait_bounded(bar.q_full, q_phase, kMaxPolls, kMaxWaitNs, kBackoffNs) || *abort_flag) {
      ok = false;
      break;
    }
    q_phase ^= 1;
    ptx::tc_fence_after();
    for (int i = 0; i < it.n_tiles; ++i) {
      if (!ptx::mbar_wait_bounded(bar.acc_empty + acc, acc_phase ^ 1, kMaxPolls, kMaxWaitNs, kBackoffNs) ||
          !ptx::mbar_wait_bounded(bar.full + stage, phase, kMaxPolls, kMaxWaitNs, kBackoffNs) || *abort_flag) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccCols);
      const uint32_t a_base = pool_addr + stage * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < kDim / 16; ++kk) {
        const uint32_t a_addr = a_base + (kk >> 2) * kPoolHalfBytes + (kk & 3) * 32;
        const uint32_t b_addr = q_addr + (kk >> 2) * kQHalfBytes + (kk & 3) * 32;
        ptx::tc_mma_f16(d_tmem, ptx::smem_desc_kmajor_sw128(a_addr), ptx::smem_desc_kmajor_sw128(b_addr), idesc,
                        kk > 0 ? 1u : 0u);
      }
      ptx::tc_commit(bar.empty + stage);
      ptx::tc_commit(bar.acc_full + acc);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (!ok) break;
    ptx::tc_commit(bar.q_empty);
  }
  if (!ok) {
    record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
    *abort_flag = 1;
  }
  // every MMA issued above must complete before TMEM is released
  ptx::tc_commit(bar.mma_done);
  ptx::mbar_wait_bounded(bar.mma_done, 0, kMaxPolls, kMaxWaitNs);
}

// kScores = false: selection (out_ids [R, budget], out_scores [R, budget] or null).
// kScores = true: index scores (out_scores [R, ld]; out_ids and budget unused).
template <bool kNegScale, bool kScores>
__global__ void __launch_bounds__(kThreads, 1)
    select_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kp,
                     const float* __restrict__ w, const int32_t* __restrict__ cu,
                     const int32_t* __restrict__ pool_off, const int2* __restrict__ items,
                     WorkspaceHeader* __restrict__ hdr, int kpool, int budget, float abs_scale,
                     int64_t row_begin, int64_t row_end, int32_t* __restrict__ out_ids,
                     float* __restrict__ out_scores, int64_t ld) {
  // Pointers derived directly from the __shared__ array keep the shared address
  // space, so the compiler emits shared loads, stores and atomics (LDS/STS/ATOMS)
  // rather than generic ones.
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Bars bar = bars_at(smem);
  int32_t* s_count = reinterpret_cast<int32_t*>(smem + kOffCount);  // [row][region]
  uint64_t* s_tau = reinterpret_cast<uint64_t*>(smem + kOffTau);
  int32_t* s_elig = reinterpret_cast<int32_t*>(smem + kOffElig);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int32_t* s_abort = reinterpret_cast<int32_t*>(smem + kOffMisc + 4);
  float* s_w = reinterpret_cast<float*>(smem + kOffW);
  uint64_t* s_cand = reinterpret_cast<uint64_t*>(smem + kOffCand);

  // The 128-byte-swizzled TMA tiles need a 1024-byte aligned base. Every thread
  // sees the same address, so this early exit is uniform (before any barrier).
  if ((ptx::smem_addr(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(hdr, KPOOL_ERR_INTERNAL);
    return;
  }
  // n_items was written by the planning kernel before this launch and is 0 when
  // planning failed, so every thread reads the same value and the loops below
  // agree on how many items there are.
  const int n_items = hdr->n_items;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar.q_full, 1);
    ptx::mbar_init(bar.q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar.full + s, 1);
      ptx::mbar_init(bar.empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar.acc_full + a, 1);
      ptx::mbar_init(bar.acc_empty + a, 8);
    }
    ptx::mbar_init(bar.mma_done, 1);
    for (int i = 0; i < kRing; ++i) {
      ptx::mbar_init(bar.ring_full + i, 1);
      ptx::mbar_init(bar.ring_empty + i, 9);
    }
    ptx::fence_mbar_init();
    *s_abort = 0;
    ptx::prefetch_tmap(&tmap_q);
    ptx::prefetch_tmap(&tmap_kp);
  }
  if (warp == 1) {
    ptx::tmem_alloc(s_tmem, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  volatile int32_t* abort_flag = s_abort;
  volatile int32_t* s_ring = reinterpret_cast<volatile int32_t*>(smem + kOffRing);

  if (warp == 0) {
    if (lane == 0) producer_role(&tmap_q, &tmap_kp, cu, pool_off, items, hdr, kpool, n_items);
  } else if (warp == 1) {
    if (lane == 0) mma_role(cu, pool_off, items, hdr, kpool, tmem_base);
  } else {
    // ------------------------------------------------------------ epilogue
    // Row split: group grp (warps 2-5 -> 0, warps 6-9 -> 1) owns rows 4*grp .. 4*grp+3
    // of every item and reads those 128 columns of every accumulator. The groups share
    // only the accumulators (each released once all 8 warps have loaded it), so each
    // group synchronises just its own four warps and neither waits for the other's
    // compactions.
    const int ew = warp - 2;          // 0..7
    const int grp = ew >> 2;          // 0 or 1
    const int wq = ew & 3;            // row (within the group) this warp ranks at the end
    const int lg = warp & 3;          // TMEM lane group this warp may read
    const int gt = wq * 32 + lane;    // thread index within the group (0..127)
    const int rbase = 4 * grp;        // the group's first row
    const int bar_id = 1 + grp;
    SelectScratch* sel = reinterpret_cast<SelectScratch*>(smem + kOffSelect + grp * kSelectBytes);
    uint64_t* const my_region = s_cand + rbase * kCap + wq * kReg;  // this warp's region of the group's row 0
    const unsigned lt_mask = (1u << lane) - 1u;
    const uint32_t lane_addr = tmem_base + (uint32_t(lg * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int r = 0;; ++r) {
      // the next work item, as the producer fetched it
      const int slot = r % kRing;
      int idx = -1;
      bool got = true;
      if (lane == 0) {
        got = ptx::mbar_wait_bounded(bar.ring_full + slot, uint32_t(r / kRing) & 1, kMaxPolls, kMaxWaitNs);
        if (got) idx = s_ring[slot];
        ptx::mbar_arrive(bar.ring_empty + slot);
      }
      idx = __shfl_sync(0xffffffffu, idx, 0);
      // the group leaves together if any of its warps' waits ran out
      if (named_bar_or(bar_id, 128, __shfl_sync(0xffffffffu, got ? 0 : 1, 0) != 0)) {
        if (gt == 0) {
          record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      if (idx < 0) break;
      const Item it = load_item(items, cu, pool_off, idx, kpool);
      // per-item state of the group's 4 rows
      {
        const int q = rbase + (gt >> 5), h = gt & 31;
        const int row = it.t0 + q;
        // halved: the scoring loop multiplies by x + |x| = 2 relu(x) (exact)
        s_w[q * kHeads + h] = row < it.len ? (w[(it.seq_start + row) * kHeads + h] * abs_scale) * 0.5f : 0.0f;
      }
      if (gt < 4) {
        const int q = rbase + gt;
        const int row = it.t0 + q;
        s_elig[q] = row < it.len ? (row + 1) / kpool : 0;
        if constexpr (kScores) {
          // the output row, or -1 for rows past the sequence or outside the range
          const int64_t grow = it.seq_start + row;
          const bool written = row < it.len && grow >= row_begin && grow < row_end;
          s_tau[q] = written ? uint64_t(grow - row_begin) : ~0ull;
          if (written && s_elig[q] > ld) record_error(hdr, KPOOL_ERR_INVALID_ARG);  // row wider than ld
        } else {
          s_tau[q] = 0;
        }
      }
      int cnt[4] = {0, 0, 0, 0};  // this warp's region counts of the group's four rows
      named_bar(bar_id, 128);
      bool aborted = false;
      bool overflow = false;  // a region passed its capacity (a library bug; see the insertion)
      for (int i = 0; i < it.n_tiles; ++i) {
        if constexpr (kScores) {
          if (*abort_flag != 0) {  // another role gave up: leave the tiles, the item-end vote follows
            aborted = true;
            break;
          }
        }
        bool over = false;  // this warp's reservation pushed a row past the compaction mark
        // every lane tests the barrier (one warp-wide instruction, no divergent branch);
        // the vote keeps a wait that ran out uniform across the warp
        const bool ready = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar.acc_full + acc, acc_phase, kMaxPolls,
                                                                          kMaxWaitNs));
        if (!ready) {
          record_error(hdr, KPOOL_ERR_DEVICE_TIMEOUT);
          *abort_flag = 1;
        } else {
          ptx::tc_fence_after();
          const int p = i * kTilePools + lg * 32 + lane;  // sequence-local pool index of this thread
          const uint32_t col0 = lane_addr + uint32_t(acc * kAccCols + rbase * kHeads);
          // TMEM -> registers one row at a time; the next row's columns and head
          // weights are in flight while the current row is scored.
          uint32_t v[2][32];
          ulonglong2 wr[2][kHeads / 4];
          uint64_t key[4];
          unsigned m[4];
          bool pass[4];
          ptx::tc_ld_32x32b_x32(col0, v[0]);
          {
            const ulonglong2* wv = reinterpret_cast<const ulonglong2*>(s_w + rbase * kHeads);
#pragma unroll
            for (int h4 = 0; h4 < kHeads / 4; ++h4) wr[0][h4] = wv[h4];
          }
          ptx::tc_wait_ld();
          ptx::tc_reg_fence(v[0]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q = rbase + j;
            if (j < 3) {
              ptx::tc_ld_32x32b_x32(col0 + (j + 1) * kHeads, v[(j + 1) & 1]);
              const ulonglong2* wv = reinterpret_cast<const ulonglong2*>(s_w + (q + 1) * kHeads);
#pragma unroll
              for (int h4 = 0; h4 < kHeads / 4; ++h4) wr[(j + 1) & 1][h4] = wv[h4];
            } else {
              // every column this warp needs is in registers: release the accumulator
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(bar.acc_empty + acc);
            }
            const uint32_t (&cur)[32] = v[j & 1];
            const ulonglong2 (&wc)[kHeads / 4] = wr[j & 1];
            uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
            for (int h4 = 0; h4 < kHeads / 4; ++h4) {
              const ulonglong2 ww = wc[h4];
              const float x0 = __uint_as_float(cur[4 * h4 + 0]);
              const float x1 = __uint_as_float(cur[4 * h4 + 1]);
              const float x2 = __uint_as_float(cur[4 * h4 + 2]);
              const float x3 = __uint_as_float(cur[4 * h4 + 3]);
              // relu on the FMA pipe: x + |x| is exactly 2 relu(x) (|x| - x for a negative
              // scale; the absolute value is an operand modifier of the add), and the weights
              // are halved, so each fused multiply-add rounds the same exact product as
              // w * relu(x) would; the ALU pipe is left to the selection
              acc0 = ptx::fma_f32x2(ww.x, ptx::pack_f32x2(kNegScale ? fabsf(x0) - x0 : x0 + fabsf(x0),
                                                          kNegScale ? fabsf(x1) - x1 : x1 + fabsf(x1)), acc0);
              acc1 = ptx::fma_f32x2(ww.y, ptx::pack_f32x2(kNegScale ? fabsf(x2) - x2 : x2 + fabsf(x2),
                                                          kNegScale ? fabsf(x3) - x3 : x3 + fabsf(x3)), acc1);
            }
            float s0, s1, s2, s3;
            ptx::unpack_f32x2(acc0, s0, s1);
            ptx::unpack_f32x2(acc1, s2, s3);
            const float s = (s0 + s1) + (s2 + s3);
            if constexpr (kScores) {
              const int64_t orow = int64_t(s_tau[q]);
              if (orow >= 0 && p < ld) __stcs(out_scores + orow * ld + p, p < s_elig[q] ? s : -INFINITY);
            } else {
              key[j] = make_key(s, uint32_t(p));
              pass[j] = p < s_elig[q] && key[j] > s_tau[q];
              m[j] = __ballot_sync(0xffffffffu, pass[j]);
            }
            if (j < 3) {
              ptx::tc_wait_ld();
              ptx::tc_reg_fence(v[(j + 1) & 1]);
            }
          }
          // append to this warp's region of each row (warp-uniform counts, no atomics)
          // A region holds at most kRegMark keys when a tile starts (a compaction runs as
          // soon as one passes the mark) and a tile adds at most 32, so every slot below
          // is < kReg without a per-key check.
          if constexpr (!kScores) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (pass[j]) my_region[j * kCap + cnt[j] + __popc(m[j] & lt_mask)] = key[j];
              cnt[j] += __popc(m[j]);
            }
            const int cmax = max(max(cnt[0], cnt[1]), max(cnt[2], cnt[3]));
            over = cmax > kRegMark;
            overflow = overflow || cmax > kReg;  // cannot happen; reported at the end of the item
          }
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        if constexpr (kScores) {
          // no shared state changes between tiles: the warps run free, paced by the
          // accumulator barriers, and vote once at the end of the item
          if (!ready) {
            aborted = true;
            break;
          }
          continue;
        }
        // one group barrier per tile in the common case; its OR says whether any of the
        // group's rows needs compacting or a wait ran out
        if (named_bar_or(bar_id, 128, over || !ready || *abort_flag != 0)) {
          if (lane == 0)  // publish this warp's region counts for the cooperative compaction
            for (int j = 0; j < 4; ++j) s_count[(rbase + j) * 4 + wq] = cnt[j];
          if (named_bar_or(bar_id, 128, !ready || *abort_flag != 0)) {
            aborted = true;
            break;
          }
          // the group's four warps bring each row with a full region back down together
          for (int j = 0; j < 4; ++j) {
            const int q = rbase + j;
            const int32_t* c = s_count + q * 4;
            if (max(max(c[0], c[1]), max(c[2], c[3])) > kRegMark) {
              compact_row(s_cand + q * kCap, s_count + q * 4, budget, kSlack, gt, bar_id, sel, s_tau + q);
            }
          }
          named_bar(bar_id, 128);
#pragma unroll
          for (int j = 0; j < 4; ++j) cnt[j] = s_count[(rbase + j) * 4 + wq];
        }
      }
      if constexpr (kScores) {
        // every warp of the group reaches this vote, including one whose wait ran out
        if (named_bar_or(bar_id, 128, aborted)) break;
        // the pools no tile covered: -inf up to ld for each of the group's rows, in
        // 16-byte stores where the row allows (the next item's row state is written
        // only after the group barrier at the top of the item loop)
        const int64_t p_from = int64_t(it.n_tiles) * kTilePools;
        for (int j = 0; j < 4; ++j) {
          const int64_t orow = int64_t(s_tau[rbase + j]);
          if (orow < 0) continue;
          float* orow_p = out_scores + orow * ld;
          int64_t pp = p_from;
          if (pp < ld && (reinterpret_cast<uintptr_t>(orow_p + pp) & 15) == 0) {
            const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            for (int64_t v = pp + 4 * gt; v + 4 <= ld; v += 4 * 128) __stcs(reinterpret_cast<float4*>(orow_p + v), ninf);
            pp += (ld - pp) / 4 * 4;  // the scalar loop below writes the last (ld - p_from) % 4
          }
          for (int64_t v = pp + gt; v < ld; v += 128) __stcs(orow_p + v, -INFINITY);
        }
        continue;
      }
      if (aborted) break;
      if (overflow && lane == 0) record_error(hdr, KPOOL_ERR_INTERNAL);
      // final ranking: cut each of the group's rows to its top `budget` keys, dealt
      // evenly over the four regions (the group's four warps together), then warp wq
      // sorts row rbase + wq and writes it
      if (lane == 0)
        for (int j = 0; j < 4; ++j) s_count[(rbase + j) * 4 + wq] = cnt[j];
      named_bar(bar_id, 128);
      for (int j = 0; j < 4; ++j) {
        const int q = rbase + j;
        const int32_t* c = s_count + q * 4;
        const int n = c[0] + c[1] + c[2] + c[3];
        const int64_t grow = it.seq_start + it.t0 + q;
        const bool written = grow >= row_begin && grow < row_end;  // rows past the sequence have n = 0
        // the sort below reads the first kFinalChunk slots of each region
        if (written && (n > budget || max(max(c[0], c[1]), max(c[2], c[3])) > kFinalChunk)) {
          compact_row(s_cand + q * kCap, s_count + q * 4, budget, 0, gt, bar_id, sel, nullptr);
        }
      }
      named_bar(bar_id, 128);
      {
        const int q = rbase + wq;
        const int row = it.t0 + q;
        const int64_t grow = it.seq_start + row;
        if (row < it.len && grow >= row_begin && grow < row_end) {  // items may straddle the row range
          const int64_t orow = grow - row_begin;
          rank_and_write_row(s_cand + q * kCap, s_count + q * 4, budget, out_ids + orow * budget,
                             out_scores ? out_scores + orow * budget : nullptr);
          __syncwarp();
        }
      }
      named_bar(bar_id, 128);
    }
    ptx::tc_fence_before();
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  named_bar(3, kThreads);
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

bool g_attr_set[64][4] = {};

}  // namespace

bool select_tc_supported(kpool_dtype dtype, int32_t H, int32_t d, int32_t budget) {
  return dtype == KPOOL_BF16 && H == kHeads && d == kDim && budget >= 1 && budget <= kMaxBudget;
}

namespace {

cudaError_t launch_tc(bool scores, const void* q, const void* kp, const float* w, const int32_t* cu, int64_t T,
                      int32_t kpool, int32_t budget, float scale, int64_t row_begin, int64_t row_end, int32_t* out_ids,
                      float* out_scores, int64_t ld, char* ws, const WorkspaceLayout& L, int grid,
                      cudaStream_t stream) {
  if (T == 0 || row_end <= row_begin) return cudaSuccess;
  if (T * kHeads > int64_t(INT32_MAX)) return cudaErrorInvalidValue;
  CUtensorMap map_q, map_kp;
  if (!make_tmap_bf16_k128(&map_q, q, uint64_t(T) * kHeads, kN)) return cudaErrorInvalidValue;
  const uint64_t kp_rows = L.max_pools > 0 ? uint64_t(L.max_pools) : 1;
  if (!make_tmap_bf16_k128(&map_kp, kp, kp_rows, kTilePools)) return cudaErrorInvalidValue;
  const bool neg = scale < 0.0f;
  const float abs_scale = neg ? -scale : scale;
  auto kern = scores ? (neg ? select_tc_kernel<true, true> : select_tc_kernel<false, true>)
                     : (neg ? select_tc_kernel<true, false> : select_tc_kernel<false, false>);
  const int variant = (neg ? 1 : 0) + (scores ? 2 : 0);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !g_attr_set[dev][variant]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_set[dev][variant] = true;
  }
  kern<<<grid, kThreads, kSmemBytes, stream>>>(
      map_q, map_kp, w, cu, reinterpret_cast<const int32_t*>(ws + L.pool_off),
      reinterpret_cast<const int2*>(ws + L.items), reinterpret_cast<WorkspaceHeader*>(ws + L.header), kpool, budget,
      abs_scale, row_begin, row_end, out_ids, out_scores, ld);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select_tc(const void* q, const void* kp, const float* w, const int32_t* cu, int32_t S, int64_t T,
                             int32_t kpool, int32_t budget, float scale, int64_t row_begin, int64_t row_end,
                             int32_t* out_ids, float* out_scores, char* ws, const WorkspaceLayout& L, int grid,
                             cudaStream_t stream) {
  (void)S;
  return launch_tc(false, q, kp, w, cu, T, kpool, budget, scale, row_begin, row_end, out_ids, out_scores, 0, ws, L,
                   grid, stream);
}

cudaError_t launch_scores_tc(const void* q, const void* kp, const float* w, const int32_t* cu, int64_t T,
                             int32_t kpool, float scale, int64_t row_begin, int64_t row_end, float* out_scores,
                             int64_t ld, char* ws, const WorkspaceLayout& L, int grid, cudaStream_t stream) {
  return launch_tc(true, q, kp, w, cu, T, kpool, 0, scale, row_begin, row_end, nullptr, out_scores, ld, ws, L, grid,
                   stream);
}

}  // namespace kpool
