// kpool_select_common.cuh -- warp-level selection primitives on 64-bit
// selection keys held in shared memory (key order = selection order; key 0 is
// an empty slot). Used by the score+select kernels.
#pragma once

#include <stdint.h>

namespace kpool {

// Descending bitonic sort of n (a power of two) keys in shared memory, one warp.
__device__ inline void warp_sort_desc(uint64_t* buf, int n) {
  const int lane = threadIdx.x & 31;
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = lane; i < n; i += 32) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t a = buf[i], b = buf[l];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            buf[i] = b;
            buf[l] = a;
          }
        }
      }
      __syncwarp();
    }
  }
}

// Compare-exchange of a bitonic network on 64-bit keys: returns the key this
// position keeps, the larger of (mine, other) when keep_max, else the smaller.
__device__ __forceinline__ uint64_t bitonic_keep(uint64_t mine, uint64_t other, bool keep_max) {
  return (mine > other) == keep_max ? mine : other;
}

// Descending bitonic sort of 512 keys in one warp, blocked layout: key index
// i = 16 * lane + r (k[r] of lane `lane`). Strides below 16 pair registers of the
// same lane (30 of the 45 stages), larger strides exchange with lane ^ (stride / 16)
// through shuffles (15 stages). The starting placement of the keys does not matter
// to a sorting network, so callers load them striped (conflict-free) and read the
// result as blocked: lane l ends up holding ranks 16 l .. 16 l + 15. Every stage is
// unrolled (with rolled stage loops a lone warp spends a third more time on loop
// control and reconvergence); a caller whose own code is register-hungry keeps the
// network out of line so its allocation does not depend on this one.
__device__ __forceinline__ void warp_sort512_blocked_desc(uint64_t (&k)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 512; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < 16) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          if ((r & stride) == 0) {
            const int r2 = r | stride;
            const bool desc = ((16 * lane + r) & size) == 0;
            const uint64_t a = k[r], c = k[r2];
            const bool swap = (a > c) != desc;
            k[r] = swap ? c : a;
            k[r2] = swap ? a : c;
          }
        }
      } else {
        const int ls = stride >> 4;
        const bool keep_max = ((lane & ls) == 0) == (((16 * lane) & size) == 0);
#pragma unroll
        for (int r = 0; r < 16; ++r) k[r] = bitonic_keep(k[r], __shfl_xor_sync(0xffffffffu, k[r], ls), keep_max);
      }
    }
  }
}

__device__ __forceinline__ void group_bar(int id, int count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Descending bitonic sort of 512 keys by the 256 threads of warps 0-7 (named
// barrier bar_id): k[h] of thread (warp w, lane l) is key 64 w + 32 h + l. Strides
// up to 16 go through shuffles, stride 32 swaps the thread's two keys, strides
// 64..256 cross warps through s_buf (1024 keys of shared memory, two alternating
// halves, so each such stage needs one barrier). On return the thread holds ranks
// 64 w + 32 h + l.
__device__ __forceinline__ void block_sort512_desc(uint64_t (&k)[2], uint64_t* s_buf, int bar_id) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int half = 0;
#pragma unroll
  for (int size = 2; size <= 512; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 64) {
        uint64_t* b = s_buf + 512 * half;
        half ^= 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) b[64 * warp + 32 * h + lane] = k[h];
        group_bar(bar_id, 256);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = 64 * warp + 32 * h + lane;
          k[h] = bitonic_keep(k[h], b[i ^ stride], ((i & stride) == 0) == ((i & size) == 0));
        }
      } else if (stride == 32) {
        const bool desc = ((64 * warp + lane) & size) == 0;
        const uint64_t a = k[0], c = k[1];
        const bool swap = (a > c) != desc;
        k[0] = swap ? c : a;
        k[1] = swap ? a : c;
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = 64 * warp + 32 * h + lane;
          k[h] = bitonic_keep(k[h], __shfl_xor_sync(0xffffffffu, k[h], stride),
                              ((i & stride) == 0) == ((i & size) == 0));
        }
      }
    }
  }
}

// Scratch (shared memory) of block_select_compact: per-warp OR/AND words, three
// rotating 32-bin histograms and per-warp kept counts.
struct SelectScratch {
  unsigned long long red_or[8];
  unsigned long long red_and[8];
  uint32_t hist[3][32];
  int32_t kept[8];
};

// Threshold search + compaction of one candidate buffer by the kWarps warps
// (barrier `bar_id`) that call it together. Same search as
// warp_select_compact -- 5-bit most-significant-digit passes starting below the
// keys' common leading bits -- with each thread holding kPer of the (at most
// 32 * kWarps * kPer) keys and the histograms shared, so a compaction costs a handful of
// barriers instead of one warp's long dependent chain. Returns the kept count
// (between budget and budget + slack, or all keys when n <= budget); *edge_out
// gets the edge. Ends with a barrier: buf and the count are consistent for all.
// Where a candidate buffer's keys live. Contiguous: slots [0, n). Quartered: four
// regions of kReg slots, region r holding counts[r] keys (one region per warp of
// an epilogue group, so insertion needs no atomics); the kept keys are written
// back as four consecutive blocks, region r receiving region_count(kept, r) =
// kept / 4 (+1 for r < kept % 4) of them, so the regions restart level and a
// warp's 32 consecutive keys land in consecutive slots (no bank conflicts).
// load<kT, j>(buf, t): the j-th key of thread t of kT, i.e. slot t + kT * j.
struct ContiguousLayout {
  int n;
  template <int kT, int j>
  __device__ __forceinline__ uint64_t load(const uint64_t* buf, int t) const {
    return t + kT * j < n ? buf[t + kT * j] : 0ull;
  }
  __device__ __forceinline__ int pos(int e, int) const { return e; }
};

template <int kReg>
struct QuarteredLayout {
  const int32_t* counts;  // 4 region counts (shared memory)
  template <int kT, int j>
  __device__ __forceinline__ uint64_t load(const uint64_t* buf, int t) const {
    static_assert(kReg % kT == 0, "a thread's slot t + kT * j stays in one region for every t < kT");
    constexpr int r = kT * j / kReg, off = kT * j % kReg;  // region and offset of thread 0's slot
    return off + t < counts[r] ? buf[kT * j + t] : 0ull;
  }
  // slot of kept key e (0 <= e < kept); callers keep kept <= 4 * kReg
  __device__ __forceinline__ int pos(int e, int kept) const {
    const int q = kept >> 2, rem = kept & 3;
    const int s1 = q + (rem > 0), s2 = 2 * q + min(rem, 2), s3 = 3 * q + rem;  // block starts
    const int r = (e >= s1) + (e >= s2) + (e >= s3);
    const int start = r * q + min(r, rem);
    return r * kReg + (e - start);
  }
  __device__ __forceinline__ static int region_count(int kept, int r) { return (kept >> 2) + (r < (kept & 3)); }
};

template <class Layout, int kT, int kPer, int j = 0>
__device__ __forceinline__ void load_keys(const Layout& layout, const uint64_t* buf, int t, uint64_t (&k)[kPer]) {
  if constexpr (j < kPer) {
    k[j] = layout.template load<kT, j>(buf, t);
    load_keys<Layout, kT, kPer, j + 1>(layout, buf, t, k);
  }
}

template <int kPer, int kWarps, class Layout>
__device__ inline int block_select_compact_in(uint64_t* buf, int n, int budget, int slack, int et, int bar_id,
                                              SelectScratch* sc, uint64_t* edge_out, Layout layout) {
  static_assert(kWarps <= 8, "SelectScratch holds 8 warps");
  constexpr int kT = 32 * kWarps;
  const int lane = et & 31, wid = et >> 5;
  const unsigned full = 0xffffffffu;
  uint64_t k[kPer];
  load_keys<Layout, kT, kPer>(layout, buf, et, k);
  uint64_t o = 0, a = ~0ull;
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (k[j] != 0) {
      o |= k[j];
      a &= k[j];
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    o |= __shfl_xor_sync(full, o, off);
    a &= __shfl_xor_sync(full, a, off);
  }
  if (lane == 0) {
    sc->red_or[wid] = o;
    sc->red_and[wid] = a;
  }
  if (wid == 0) {
    sc->hist[0][lane] = 0;
    sc->hist[1][lane] = 0;
  }
  group_bar(bar_id, kT);
  o = 0;
  a = ~0ull;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    o |= sc->red_or[w];
    a &= sc->red_and[w];
  }
  const uint64_t diff = o ^ a;
  uint64_t edge = a;  // one distinct key (or none): keep it
  if (n > budget && diff != 0) {
    int pbits = __clzll(static_cast<long long>(diff));  // leading bits common to every key
    uint64_t prefix = pbits == 0 ? 0ull : (a & ~(~0ull >> pbits));
    int above = 0;
    for (int pass = 0;; ++pass) {
      uint32_t* hist = sc->hist[pass % 3];
      const int width = (64 - pbits) < 5 ? (64 - pbits) : 5;
      const int dshift = 64 - pbits - width;
      const uint64_t dmask = (1ull << width) - 1ull;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const bool in = k[j] != 0 && (pbits == 0 || (k[j] >> (64 - pbits)) == (prefix >> (64 - pbits)));
        if (in) atomicAdd(hist + int((k[j] >> dshift) & dmask), 1u);
      }
      group_bar(bar_id, kT);
      if (wid == 0) sc->hist[(pass + 2) % 3][lane] = 0;  // read by every warp before this barrier
      const int cnt = int(hist[lane]);
      int suffix = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_down_sync(full, suffix, off);
        if (lane + off < 32) suffix += v;
      }
      const int higher = suffix - cnt;
      const unsigned hit = __ballot_sync(full, above + higher < budget && above + suffix >= budget);
      const int d = hit ? __ffs(hit) - 1 : 0;  // a crossing bin always exists (above < budget <= bin total)
      const int d_higher = __shfl_sync(full, higher, d);
      const int d_cnt = __shfl_sync(full, cnt, d);
      prefix |= uint64_t(d) << dshift;
      pbits += width;
      if (above + d_higher + d_cnt <= budget + slack || pbits == 64) {
        edge = prefix;
        break;
      }
      above += d_higher;
    }
  } else if (n <= budget) {
    edge = 1;  // keep everything
  }
  // write the kept keys back (front of buf, or dealt over the regions), in thread order
  unsigned m[kPer];
  int mine = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    m[j] = __ballot_sync(full, k[j] != 0 && k[j] >= edge);
    mine += __popc(m[j]);
  }
  if (lane == 0) sc->kept[wid] = mine;
  group_bar(bar_id, kT);
  int off = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = sc->kept[w];
    off += w < wid ? c : 0;
    total += c;
  }
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if ((m[j] >> lane) & 1u) buf[layout.pos(off + __popc(m[j] & lt), total)] = k[j];
    off += __popc(m[j]);
  }
  *edge_out = edge;
  group_bar(bar_id, kT);
  return total;
}

// Contiguous buffer of n keys.
template <int kPer, int kWarps>
__device__ inline int block_select_compact(uint64_t* buf, int n, int budget, int slack, int et, int bar_id,
                                           SelectScratch* sc, uint64_t* edge_out) {
  return block_select_compact_in<kPer, kWarps>(buf, n, budget, slack, et, bar_id, sc, edge_out,
                                               ContiguousLayout{n});
}

}  // namespace kpool
