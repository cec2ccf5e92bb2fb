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

// Threshold search + compaction, one warp, n <= 32 * kSlots keys.
//
// Finds an edge such that budget <= #{keys >= edge} <= budget + slack by a
// most-significant-digit search with 5-bit digits: each pass histograms the
// keys of the current bin on the five bits just below their highest differing
// bit (so common leading bits cost nothing) and descends into the bin where the
// running count crosses `budget`, until the whole bin can be kept. Keys are
// distinct, so every pass splits the bin and the search ends. The kept keys are
// then written back to the front of buf (unordered). Requires budget <= n.
// `hist` is 16 words of shared memory private to the warp holding 32 16-bit
// bin counts (n < 65536). Returns the kept count; *edge_out receives the edge
// (keys below it cannot be in the top budget).
template <int kSlots>
__device__ inline int warp_select_compact(uint64_t* buf, int n, int budget, int slack, uint32_t* hist,
                                          uint64_t* edge_out) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  uint64_t key[kSlots];
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    const int idx = i * 32 + lane;
    key[i] = idx < n ? buf[idx] : 0ull;
  }
  __syncwarp();

  bool all = true;   // the current bin is every nonzero key
  int bin_shift = 0; // otherwise: keys with (key >> bin_shift) == bin_hi
  uint64_t bin_hi = 0;
  int above = 0;     // keys above the current bin (all kept)
  uint64_t edge = 1;
  for (int pass = 0; pass < 64; ++pass) {
    // common bits of the bin's keys
    uint64_t o = 0, a = ~0ull;
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const bool in = key[i] != 0 && (all || (key[i] >> bin_shift) == bin_hi);
      if (in) {
        o |= key[i];
        a &= key[i];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      o |= __shfl_xor_sync(full, o, off);
      a &= __shfl_xor_sync(full, a, off);
    }
    const uint64_t diff = o ^ a;
    if (diff == 0) {  // one key left in the bin: it completes the budget
      edge = a;
      break;
    }
    const int top = 63 - __clzll(static_cast<long long>(diff));
    const int dshift = top >= 4 ? top - 4 : 0;
    if (lane < 16) hist[lane] = 0;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const bool in = key[i] != 0 && (all || (key[i] >> bin_shift) == bin_hi);
      if (in) {
        const uint32_t digit = uint32_t(key[i] >> dshift) & 31u;
        atomicAdd(hist + (digit >> 1), 1u << (16 * (digit & 1u)));
      }
    }
    __syncwarp();
    const int cnt = int((hist[lane >> 1] >> (16 * (lane & 1))) & 0xFFFFu);
    int suffix = cnt;  // sum of counts of digits >= lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_down_sync(full, suffix, off);
      if (lane + off < 32) suffix += v;
    }
    const int higher = suffix - cnt;  // digits > lane
    const unsigned hit = __ballot_sync(full, above + higher < budget && above + suffix >= budget);
    const int d = __ffs(hit) - 1;
    const int d_higher = __shfl_sync(full, higher, d);
    const int d_cnt = __shfl_sync(full, cnt, d);
    __syncwarp();
    // bits above the digit are common to the whole bin (taken from the AND)
    const uint64_t upper = (dshift + 5 >= 64) ? 0ull : ((a >> (dshift + 5)) << 5);
    const uint64_t new_hi = upper | uint64_t(d);
    if (above + d_higher + d_cnt <= budget + slack || dshift == 0) {
      edge = new_hi << dshift;
      break;
    }
    above += d_higher;
    all = false;
    bin_shift = dshift;
    bin_hi = new_hi;
  }

  // write the kept keys back to the front of buf
  int base = 0;
#pragma unroll
  for (int i = 0; i < kSlots; ++i) {
    const bool keep = key[i] != 0 && key[i] >= edge;
    const unsigned m = __ballot_sync(full, keep);
    if (keep) buf[base + __popc(m & ((1u << lane) - 1u))] = key[i];
    base += __popc(m);
  }
  __syncwarp();
  *edge_out = edge;
  return base;
}

// Descending bitonic sort of 32 * kSlots keys held in registers, one warp.
// Key index i = 32 * r + lane (k[r] of lane `lane`), so loads and stores of a
// buffer are coalesced: strides below 32 exchange with another lane through
// shuffles, larger strides swap registers of the same lane.
template <int kSlots>
__device__ __forceinline__ void warp_sort_regs_desc(uint64_t (&k)[kSlots]) {
  constexpr int kN = 32 * kSlots;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= kN; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32) {
        const int rs = stride >> 5;
#pragma unroll
        for (int r = 0; r < kSlots; ++r) {
          if ((r & rs) == 0) {
            const int r2 = r | rs;
            const bool desc = ((32 * r) & size) == 0;
            const uint64_t a = k[r], b = k[r2];
            const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
            k[r] = desc ? hi : lo;
            k[r2] = desc ? lo : hi;
          }
        }
      } else {
        const bool lower = (lane & stride) == 0;
#pragma unroll
        for (int r = 0; r < kSlots; ++r) {
          const uint64_t other = __shfl_xor_sync(0xffffffffu, k[r], stride);
          const bool desc = ((32 * r + lane) & size) == 0;
          const bool take_max = lower == desc;
          const uint64_t hi = k[r] > other ? k[r] : other, lo = k[r] > other ? other : k[r];
          k[r] = take_max ? hi : lo;
        }
      }
    }
  }
}

}  // namespace kpool
