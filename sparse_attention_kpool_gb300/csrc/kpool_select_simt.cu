// kpool_select_simt.cu -- K2 on CUDA cores: score + streaming top-budget.
//
// Serves the shapes the tensor-core kernel does not (fp32 inputs, H != 32,
// d != 128, budget > 512). One warp owns one query row t of sequence b:
//   s[t,p] = sum_h w[t,h] * relu(scale * q[t,h,:] . kp[p,:])
// ("spark_model/layers/glm5next_dsa/tp.rs", module docs: index_scores
// accumulates weights[h] * relu(scale . dot) as a plain sum over heads) for
// every eligible pool p < floor((t+1)/kpool), 32 pools per step, one per lane.
// relu(scale*x) = |scale| * relu(sign(scale)*x), so |scale| is folded into the
// weight and the sign picks which side of zero survives.
//
// Selection keeps a per-warp candidate buffer of selection keys in shared
// memory (unsigned key order = higher score, then smaller pool index: tp.rs
// module docs, the deterministic tiebreak). A lane's key enters only if it
// beats the running threshold -- the budget-th best key seen so far. When the
// buffer is nearly full it is sorted and cut back to `budget`, which
// raises the threshold. The [rows, pools] score matrix is never materialised.
#include <cuda_bf16.h>

#include "kpool_internal.cuh"
#include "kpool_select_common.cuh"

namespace kpool {
namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// s[t,p] of one (row, pool) pair: an fp32 FMA chain over the channels per head, then
// an FMA of |scale| * w[h] and the surviving side of zero per head. The selection
// and the index-score kernels both call this, so their scores agree bit for bit.
template <typename T, bool kNegScale>
__device__ __forceinline__ float simt_score(const T* __restrict__ qr, const T* __restrict__ kr,
                                            const float* __restrict__ wr, int H, int d, float abs_scale) {
  float s = 0.0f;
  for (int h = 0; h < H; ++h) {
    float dot = 0.0f;
    for (int c = 0; c < d; ++c) dot = fmaf(to_f32(qr[h * d + c]), to_f32(kr[c]), dot);
    const float v = kNegScale ? -dot : dot;
    s = fmaf(__ldg(wr + h) * abs_scale, fmaxf(v, 0.0f), s);
  }
  return s;
}

template <typename T, bool kNegScale>
__global__ void __launch_bounds__(128) select_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ kp, const float* __restrict__ w,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ pool_off, const WorkspaceHeader* __restrict__ hdr,
    int S, int64_t row_begin, int64_t row_end, int H, int d, int kpool, int budget, int cap, float abs_scale,
    int32_t* __restrict__ out_ids, float* __restrict__ out_scores) {
  extern __shared__ uint64_t smem_keys[];
  if (hdr->error != 0) return;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int warps = blockDim.x >> 5;
  uint64_t* buf = smem_keys + size_t(warp) * cap;
  const unsigned lt_mask = (1u << lane) - 1u;

  for (int64_t row = row_begin + int64_t(blockIdx.x) * warps + warp; row < row_end;
       row += int64_t(gridDim.x) * warps) {
    const int64_t orow = row - row_begin;  // output row
    const int b = seq_of_row(cu, S, row);
    const int64_t t = row - __ldg(cu + b);
    const int64_t eligible = (t + 1) / kpool;
    const T* qr = q + row * int64_t(H) * d;
    const float* wr = w + row * int64_t(H);
    const T* kseq = kp + int64_t(__ldg(pool_off + b)) * d;

    int count = 0;
    uint64_t tau = 0;
    for (int64_t p0 = 0; p0 < eligible; p0 += 32) {
      const int64_t p = p0 + lane;
      uint64_t key = 0;
      if (p < eligible) key = make_key(simt_score<T, kNegScale>(qr, kseq + p * d, wr, H, d, abs_scale), uint32_t(p));
      const bool pass = key > tau;
      const unsigned m = __ballot_sync(0xffffffffu, pass);
      if (pass) buf[count + __popc(m & lt_mask)] = key;
      count += __popc(m);
      if (count > cap - 32) {  // room for one more step is no longer guaranteed
        __syncwarp();
        for (int i = count + lane; i < cap; i += 32) buf[i] = 0;  // drop stale slots
        __syncwarp();
        warp_sort_desc(buf, cap);
        count = budget;  // count > cap - 32 >= budget here
        tau = buf[budget - 1];
        __syncwarp();
      }
    }
    // final: clear the unused tail, sort, emit in rank order
    __syncwarp();
    for (int i = count + lane; i < cap; i += 32) buf[i] = 0;
    __syncwarp();
    warp_sort_desc(buf, cap);
    for (int j = lane; j < budget; j += 32) {
      const uint64_t key = buf[j];
      out_ids[orow * budget + j] = key ? int32_t(key_pool(key)) : -1;
      if (out_scores) out_scores[orow * budget + j] = key ? key_score(key) : -INFINITY;
    }
    __syncwarp();
  }
}

// Index scores on CUDA cores: one warp per row of [row_begin, row_end), lanes over
// the pools 0 .. ld-1 of the row's sequence; eligible pools get simt_score, every
// other column -inf.
template <typename T, bool kNegScale>
__global__ void __launch_bounds__(128) scores_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ kp, const float* __restrict__ w,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ pool_off, WorkspaceHeader* __restrict__ hdr,
    int S, int64_t row_begin, int64_t row_end, int H, int d, int kpool, float abs_scale,
    float* __restrict__ out, int64_t ld) {
  // planning failed (malformed cu_seqlens); n_items, unlike the error word, is not
  // written again during this kernel, so every block takes the same decision
  if (hdr->n_items == 0) return;
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int64_t row = row_begin + int64_t(blockIdx.x) * warps + (threadIdx.x >> 5); row < row_end;
       row += int64_t(gridDim.x) * warps) {
    const int b = seq_of_row(cu, S, row);
    const int64_t t = row - __ldg(cu + b);
    const int64_t eligible = (t + 1) / kpool;
    if (eligible > ld && lane == 0) record_error(hdr, KPOOL_ERR_INVALID_ARG);  // row wider than ld
    const T* qr = q + row * int64_t(H) * d;
    const float* wr = w + row * int64_t(H);
    const T* kseq = kp + int64_t(__ldg(pool_off + b)) * d;
    float* o = out + (row - row_begin) * ld;
    for (int64_t p = lane; p < ld; p += 32)
      __stcs(o + p, p < eligible ? simt_score<T, kNegScale>(qr, kseq + p * d, wr, H, d, abs_scale) : -INFINITY);
  }
}

int simt_capacity(int budget) {
  int cap = 64;
  while (cap < 2 * budget + 32) cap <<= 1;
  return cap;
}

template <typename Elem, bool kNeg>
cudaError_t launch_typed(const void* q, const void* kp, const float* w, const int32_t* cu, int32_t S,
                         int64_t row_begin, int64_t row_end, int32_t H, int32_t d, int32_t kpool, int32_t budget,
                         float abs_scale, int32_t* out_ids, float* out_scores, const char* ws,
                         const WorkspaceLayout& L, int num_sms, cudaStream_t stream) {
  const int cap = simt_capacity(budget);
  const size_t per_warp = size_t(cap) * sizeof(uint64_t);
  int warps = int((96 * 1024) / per_warp);
  if (warps > 4) warps = 4;
  if (warps < 1) warps = 1;
  const size_t smem = per_warp * warps;
  auto kern = select_simt_kernel<Elem, kNeg>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  int64_t blocks = (row_end - row_begin + warps - 1) / warps;
  const int64_t cap_blocks = int64_t(num_sms) * 16;
  if (blocks > cap_blocks) blocks = cap_blocks;
  kern<<<unsigned(blocks), warps * 32, smem, stream>>>(
      static_cast<const Elem*>(q), static_cast<const Elem*>(kp), w, cu, reinterpret_cast<const int32_t*>(ws + L.pool_off),
      reinterpret_cast<const WorkspaceHeader*>(ws + L.header), S, row_begin, row_end, H, d, kpool, budget, cap,
      abs_scale, out_ids, out_scores);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select_simt(const void* q, const void* kp, const float* w, kpool_dtype dtype, const int32_t* cu,
                               int32_t S, int64_t T, int32_t H, int32_t d, int32_t kpool, int32_t budget, float scale,
                               int64_t row_begin, int64_t row_end, int32_t* out_ids, float* out_scores, char* ws,
                               const WorkspaceLayout& L, int num_sms, cudaStream_t stream) {
  if (T == 0 || budget == 0 || row_end <= row_begin) return cudaSuccess;
  const bool neg = scale < 0.0f;
  const float abs_scale = neg ? -scale : scale;
  const int64_t rb = row_begin, re = row_end;
  if (dtype == KPOOL_BF16)
    return neg ? launch_typed<__nv_bfloat16, true>(q, kp, w, cu, S, rb, re, H, d, kpool, budget, abs_scale, out_ids,
                                                    out_scores, ws, L, num_sms, stream)
               : launch_typed<__nv_bfloat16, false>(q, kp, w, cu, S, rb, re, H, d, kpool, budget, abs_scale, out_ids,
                                                     out_scores, ws, L, num_sms, stream);
  return neg ? launch_typed<float, true>(q, kp, w, cu, S, rb, re, H, d, kpool, budget, abs_scale, out_ids, out_scores,
                                         ws, L, num_sms, stream)
             : launch_typed<float, false>(q, kp, w, cu, S, rb, re, H, d, kpool, budget, abs_scale, out_ids,
                                          out_scores, ws, L, num_sms, stream);
}

cudaError_t launch_scores_simt(const void* q, const void* kp, const float* w, kpool_dtype dtype, const int32_t* cu,
                               int32_t S, int64_t T, int32_t H, int32_t d, int32_t kpool, float scale,
                               int64_t row_begin, int64_t row_end, float* out_scores, int64_t ld, char* ws,
                               const WorkspaceLayout& L, int num_sms, cudaStream_t stream) {
  if (T == 0 || row_end <= row_begin) return cudaSuccess;
  const bool neg = scale < 0.0f;
  const float abs_scale = neg ? -scale : scale;
  constexpr int kWarps = 4;
  int64_t blocks = (row_end - row_begin + kWarps - 1) / kWarps;
  if (blocks > int64_t(num_sms) * 16) blocks = int64_t(num_sms) * 16;
  const int32_t* po = reinterpret_cast<const int32_t*>(ws + L.pool_off);
  WorkspaceHeader* hdr = reinterpret_cast<WorkspaceHeader*>(ws + L.header);
  const unsigned g = unsigned(blocks);
  if (dtype == KPOOL_BF16) {
    const auto* qq = static_cast<const __nv_bfloat16*>(q);
    const auto* kk = static_cast<const __nv_bfloat16*>(kp);
    if (neg)
      scores_simt_kernel<__nv_bfloat16, true><<<g, 32 * kWarps, 0, stream>>>(qq, kk, w, cu, po, hdr, S, row_begin,
                                                                           row_end, H, d, kpool, abs_scale,
                                                                           out_scores, ld);
    else
      scores_simt_kernel<__nv_bfloat16, false><<<g, 32 * kWarps, 0, stream>>>(qq, kk, w, cu, po, hdr, S, row_begin,
                                                                            row_end, H, d, kpool, abs_scale,
                                                                            out_scores, ld);
  } else {
    const auto* qq = static_cast<const float*>(q);
    const auto* kk = static_cast<const float*>(kp);
    if (neg)
      scores_simt_kernel<float, true><<<g, 32 * kWarps, 0, stream>>>(qq, kk, w, cu, po, hdr, S, row_begin, row_end, H,
                                                                   d, kpool, abs_scale, out_scores, ld);
    else
      scores_simt_kernel<float, false><<<g, 32 * kWarps, 0, stream>>>(qq, kk, w, cu, po, hdr, S, row_begin, row_end,
                                                                    H, d, kpool, abs_scale, out_scores, ld);
  }
  return cudaGetLastError();
}

}  // namespace kpool
