// kpool_expand.cu -- K3: pool expansion, tail append and mask filtering.
//
// "NVIDIA/Megatron-LM pull request #8299", section "Change": after the pool
// ids are chosen, pool expansion, tail append and mask filtering run on the
// full [batch, sq, budget] pool-id tensor. For sequence-local row t of a
// sequence of length L, with e = floor((t+1)/kpool) eligible pools:
//   slot j*kpool + r      = pool_ids[t, j]*kpool + r   (pool id in [0, e), else -1)
//   slot index_topk + r   = e*kpool + r  if r < (t+1) mod kpool, else -1
//                           (the row's own incomplete trailing pool)
//   any id > t or >= L    -> -1 (causal / varlen mask)
//
// HBM-bound (reads budget ints, writes index_topk + kpool ints per row). One
// CTA strides over rows; each thread writes 16-byte chunks when kpool is a
// multiple of 4 and the output is 16-byte aligned, single ints otherwise.
#include "kpool_internal.cuh"

namespace kpool {
namespace {

struct RowInfo {
  int64_t t, len, eligible, tail;
};

__device__ __forceinline__ RowInfo row_info(const int32_t* cu, int S, int64_t row, int kpool) {
  const int b = seq_of_row(cu, S, row);
  RowInfo r;
  const int64_t start = __ldg(cu + b);
  r.t = row - start;
  r.len = int64_t(__ldg(cu + b + 1)) - start;
  r.eligible = (r.t + 1) / kpool;
  r.tail = (r.t + 1) % kpool;
  return r;
}

__device__ __forceinline__ int32_t token_at(const RowInfo& ri, int32_t pool, int64_t slot, int kpool, int budget) {
  int64_t tok;
  if (slot < int64_t(budget) * kpool) {
    const int64_t r = slot % kpool;
    tok = (pool >= 0 && pool < ri.eligible) ? int64_t(pool) * kpool + r : -1;
  } else {
    const int64_t r = slot - int64_t(budget) * kpool;
    tok = r < ri.tail ? ri.eligible * kpool + r : -1;
  }
  if (tok > ri.t || tok >= ri.len) tok = -1;
  return int32_t(tok);
}

// kpool == 4 (16 bytes of tokens per pool): one warp per row, lane l writes the
// row's 16-byte chunks l, l + 32, ...; chunk j < budget expands pool rank j, chunk
// budget holds the tail. 32-bit arithmetic throughout.
__global__ void __launch_bounds__(256) expand_kernel_k4(const int32_t* __restrict__ pool_ids,
                                                        const int32_t* __restrict__ cu, int S, int64_t row_begin,
                                                        int64_t R, int budget, int32_t* __restrict__ out,
                                                        const WorkspaceHeader* __restrict__ hdr) {
  if (hdr != nullptr && hdr->error != 0) return;
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t W4 = int64_t(budget) + 1;  // 16-byte chunks per row
  for (int64_t i = int64_t(blockIdx.x) * warps + (threadIdx.x >> 5); i < R; i += int64_t(gridDim.x) * warps) {
    const int64_t row = row_begin + i;
    const int b = seq_of_row(cu, S, row);
    const int t = int(row - __ldg(cu + b));
    const int e = (t + 1) >> 2, tail = (t + 1) & 3;
    const int32_t* ids = pool_ids + i * budget;
    int4* dst = reinterpret_cast<int4*>(out + i * (W4 * 4));
    for (int j = lane; j < budget; j += 32) {
      const int32_t id = __ldg(ids + j);
      dst[j] = (id >= 0 && id < e) ? make_int4(4 * id, 4 * id + 1, 4 * id + 2, 4 * id + 3)
                                   : make_int4(-1, -1, -1, -1);
    }
    if (lane == 0)
      dst[budget] = make_int4(tail > 0 ? 4 * e : -1, tail > 1 ? 4 * e + 1 : -1, tail > 2 ? 4 * e + 2 : -1, -1);
  }
}

__global__ void __launch_bounds__(256) expand_kernel_vec4(const int32_t* __restrict__ pool_ids,
                                                          const int32_t* __restrict__ cu, int S, int64_t row_begin,
                                                          int64_t R, int kpool, int budget,
                                                          int32_t* __restrict__ out,
                                                          const WorkspaceHeader* __restrict__ hdr) {
  if (hdr != nullptr && hdr->error != 0) return;
  const int64_t W = int64_t(budget) * kpool + kpool;
  const int chunks = int(W / 4);
  for (int64_t i = blockIdx.x; i < R; i += gridDim.x) {
    const RowInfo ri = row_info(cu, S, row_begin + i, kpool);
    const int32_t* ids = pool_ids + i * budget;
    int4* dst = reinterpret_cast<int4*>(out + i * W);
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const int64_t s0 = int64_t(c) * 4;
      const int64_t j = s0 / kpool;  // the 4 slots share one pool (kpool % 4 == 0)
      const int32_t pool = j < budget ? __ldg(ids + j) : -1;
      int4 v;
      v.x = token_at(ri, pool, s0 + 0, kpool, budget);
      v.y = token_at(ri, pool, s0 + 1, kpool, budget);
      v.z = token_at(ri, pool, s0 + 2, kpool, budget);
      v.w = token_at(ri, pool, s0 + 3, kpool, budget);
      dst[c] = v;
    }
  }
}

__global__ void __launch_bounds__(256) expand_kernel_scalar(const int32_t* __restrict__ pool_ids,
                                                            const int32_t* __restrict__ cu, int S,
                                                            int64_t row_begin, int64_t R, int kpool, int budget,
                                                            int32_t* __restrict__ out,
                                                            const WorkspaceHeader* __restrict__ hdr) {
  if (hdr != nullptr && hdr->error != 0) return;
  const int64_t W = int64_t(budget) * kpool + kpool;
  for (int64_t i = blockIdx.x; i < R; i += gridDim.x) {
    const RowInfo ri = row_info(cu, S, row_begin + i, kpool);
    const int32_t* ids = pool_ids + i * budget;
    for (int64_t s = threadIdx.x; s < W; s += blockDim.x) {
      const int64_t j = s / kpool;
      const int32_t pool = j < budget ? __ldg(ids + j) : -1;
      out[i * W + s] = token_at(ri, pool, s, kpool, budget);
    }
  }
}

}  // namespace

cudaError_t launch_expand(const int32_t* pool_ids, const int32_t* cu, int32_t S, int64_t row_begin,
                          int64_t row_end, int32_t kpool, int32_t budget, int32_t* out_tokens,
                          const WorkspaceHeader* hdr, int num_sms, cudaStream_t stream) {
  const int64_t R = row_end - row_begin;
  if (R <= 0) return cudaSuccess;
  int64_t blocks = R;
  const int64_t cap = int64_t(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  const bool vec = (kpool % 4 == 0) && (reinterpret_cast<uintptr_t>(out_tokens) % 16 == 0);
  if (vec && kpool == 4) {
    int64_t b4 = (R + 7) / 8;  // 8 rows (warps) per CTA
    if (b4 > int64_t(num_sms) * 16) b4 = int64_t(num_sms) * 16;
    expand_kernel_k4<<<unsigned(b4), 256, 0, stream>>>(pool_ids, cu, S, row_begin, R, budget, out_tokens, hdr);
  } else if (vec)
    expand_kernel_vec4<<<unsigned(blocks), 256, 0, stream>>>(pool_ids, cu, S, row_begin, R, kpool, budget,
                                                              out_tokens, hdr);
  else
    expand_kernel_scalar<<<unsigned(blocks), 256, 0, stream>>>(pool_ids, cu, S, row_begin, R, kpool, budget,
                                                                out_tokens, hdr);
  return cudaGetLastError();
}

}  // namespace kpool
