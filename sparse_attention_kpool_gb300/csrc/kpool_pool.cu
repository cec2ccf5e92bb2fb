// kpool_pool.cu -- K1: mean-pooling of index keys.
//
// kp[pool_off[b] + p, c] = round_to_dtype( (sum_{j<kpool} k[cu[b] + p*kpool + j, c]) / kpool )
// The pages group kpool consecutive index keys into one pool ("spark_model/
// layers/glm5next_dsa/tp.rs", module docs: n_pools = seq / kpool) but never
// name the operator; the mean is this library's stated reading. The sum runs in
// fp32 in key order, the division is IEEE-rounded, the result is rounded to
// nearest even in the input dtype -- so a bf16 MMA consumes it exactly.
//
// HBM-bound: each thread owns one 16-byte chunk (8 bf16 / 4 fp32 channels) of
// one pooled row at a time, reads kpool 16-byte vectors (coalesced across the
// chunk threads of a row) and writes one. Grid-stride over P * d/vec chunks;
// kpool = 4 has its own kernels that keep more loads in flight.
#include <cuda_bf16.h>

#include "kpool_internal.cuh"

namespace kpool {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kLanes = 8;
};
template <>
struct Vec<float> {
  static constexpr int kLanes = 4;
};

__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], __nv_bfloat16*) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 x = __bfloat1622float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], __nv_bfloat16*) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}

template <typename T>
__global__ void __launch_bounds__(256) pool_kernel(const T* __restrict__ k, const int32_t* __restrict__ cu,
                                                   const int32_t* __restrict__ pool_off,
                                                   const WorkspaceHeader* __restrict__ hdr, int S, int d,
                                                   int kpool, T* __restrict__ out) {
  constexpr int V = Vec<T>::kLanes;
  if (hdr->error != 0) return;
  const int64_t P = hdr->total_pools;
  const int chunks = d / V;
  const int64_t total = P * chunks;
  const float divisor = float(kpool);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t g = i / chunks;  // global pool row
    const int c = int(i - g * chunks) * V;
    // sequence of pool g: last b with pool_off[b] <= g
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (int64_t(__ldg(pool_off + mid)) <= g) lo = mid; else hi = mid - 1;
    }
    const int64_t p = g - __ldg(pool_off + lo);
    const int64_t first = int64_t(__ldg(cu + lo)) + p * kpool;
    float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    for (int j = 0; j < kpool; ++j) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(k + (first + j) * d + c));
      float f[8];
      unpack(v, f, static_cast<T*>(nullptr));
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
    }
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = __fdiv_rn(acc[e], divisor);
    *reinterpret_cast<uint4*>(out + g * d + c) = pack(acc, static_cast<T*>(nullptr));
  }
}

// Sequence of global pool row g: last b with pool_off[b] <= g.
__device__ __forceinline__ int seq_of_pool(const int32_t* __restrict__ pool_off, int S, int64_t g) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (int64_t(__ldg(pool_off + mid)) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// pool_kernel for a compile-time kpool (the pages' kpool is 4): each thread takes
// kUnroll chunks per round and issues all kUnroll * KP 16-byte loads before any add,
// so a warp keeps kUnroll * KP independent loads in flight instead of one per
// dependent add. The keys are read once (evict-first loads); the pooled keys are
// written with the default policy so the score kernel that follows finds them in L2.
// Dividing by KP = 4 is an exact power-of-two scaling, so multiplying by 1/KP rounds
// to the same value as the IEEE division of the generic kernel.
template <typename T, int KP>
__global__ void __launch_bounds__(256) pool_kernel_fixed(const T* __restrict__ k, const int32_t* __restrict__ cu,
                                                         const int32_t* __restrict__ pool_off,
                                                         const WorkspaceHeader* __restrict__ hdr, int S, int d,
                                                         T* __restrict__ out) {
  constexpr int V = Vec<T>::kLanes;
  constexpr int kUnroll = 2;
  static_assert((KP & (KP - 1)) == 0, "1/KP must be exact");
  if (hdr->error != 0) return;
  const int64_t P = hdr->total_pools;
  const int chunks = d / V;
  const int64_t total = P * chunks;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i0 = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i0 < total; i0 += kUnroll * stride) {
    uint4 v[kUnroll][KP];
    int64_t dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      dst[u] = -1;
      if (i < total) {
        const int64_t g = i / chunks;  // global pool row
        const int c = int(i - g * chunks) * V;
        const int b = seq_of_pool(pool_off, S, g);
        const int64_t first = int64_t(__ldg(cu + b)) + (g - __ldg(pool_off + b)) * KP;
        const uint4* src = reinterpret_cast<const uint4*>(k + first * d + c);
#pragma unroll
        for (int j = 0; j < KP; ++j) v[u][j] = __ldcs(src + j * (d / V));
        dst[u] = g * d + c;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] < 0) continue;
      float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        float f[8];
        unpack(v[u][j], f, static_cast<T*>(nullptr));
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
      }
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = __fmul_rn(acc[e], 1.0f / KP);
      *reinterpret_cast<uint4*>(out + dst[u]) = pack(acc, static_cast<T*>(nullptr));
    }
  }
}

// Gated pooling, the library's reading of the pages' compress gate and position
// embedding (parameters index_kpool_compress_gate [head_dim, hidden] and
// index_kpool_compress_ape [kpool, head_dim] in the GLM-5.3 DSA shard plan,
// "spark_model/layers/glm5next_dsa/tp.rs"; "gate scores" passed to the fused
// top-k in "NVIDIA/Megatron-LM pull request #8299", section "Mechanism"):
//   kp[p,c] = sum_j softmax_j(gate[t_j,c]) * (k[t_j,c] + ape[j,c]),  t_j = first + j,
// in fp32 (max-subtracted exponentials, the normalisation applied once at the end),
// rounded to the key dtype. A zero gate and embedding give exactly the mean pooling.
template <typename T>
__global__ void __launch_bounds__(256) pool_gated_kernel(const T* __restrict__ k, const float* __restrict__ gate,
                                                         const float* __restrict__ ape,
                                                         const int32_t* __restrict__ cu,
                                                         const int32_t* __restrict__ pool_off,
                                                         const WorkspaceHeader* __restrict__ hdr, int S, int d,
                                                         int kpool, T* __restrict__ out) {
  constexpr int V = Vec<T>::kLanes;
  if (hdr->error != 0) return;
  const int64_t P = hdr->total_pools;
  const int chunks = d / V;
  const int64_t total = P * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t g = i / chunks;  // global pool row
    const int c = int(i - g * chunks) * V;
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (int64_t(__ldg(pool_off + mid)) <= g) lo = mid; else hi = mid - 1;
    }
    const int64_t first = int64_t(__ldg(cu + lo)) + (g - __ldg(pool_off + lo)) * kpool;
    float m[8], den[8], num[8];
#pragma unroll
    for (int e = 0; e < V; ++e) {
      m[e] = -INFINITY;
      den[e] = 0.0f;
      num[e] = 0.0f;
    }
    // gate scores of the chunk's V channels, 16-byte loads; kept for the second pass
    // when the pool is short enough to hold in registers
    constexpr int kHold = 4;
    float gh[kHold][8];
    for (int j = 0; j < kpool; ++j) {
      float gv[8];
      const float4* gp = reinterpret_cast<const float4*>(gate + (first + j) * d + c);
#pragma unroll
      for (int h = 0; h < V / 4; ++h) {
        const float4 x = __ldg(gp + h);
        gv[4 * h] = x.x;
        gv[4 * h + 1] = x.y;
        gv[4 * h + 2] = x.z;
        gv[4 * h + 3] = x.w;
      }
#pragma unroll
      for (int e = 0; e < V; ++e) m[e] = fmaxf(m[e], gv[e]);
#pragma unroll
      for (int hj = 0; hj < kHold; ++hj)
        if (hj == j)
#pragma unroll
          for (int e = 0; e < V; ++e) gh[hj][e] = gv[e];
    }
    for (int j = 0; j < kpool; ++j) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(k + (first + j) * d + c));
      float f[8];
      unpack(v, f, static_cast<T*>(nullptr));
      float gv[8];
      if (j < kHold) {
#pragma unroll
        for (int hj = 0; hj < kHold; ++hj)
          if (hj == j)
#pragma unroll
            for (int e = 0; e < V; ++e) gv[e] = gh[hj][e];
      } else {
        const float4* gp = reinterpret_cast<const float4*>(gate + (first + j) * d + c);
#pragma unroll
        for (int h = 0; h < V / 4; ++h) {
          const float4 x = __ldg(gp + h);
          gv[4 * h] = x.x;
          gv[4 * h + 1] = x.y;
          gv[4 * h + 2] = x.z;
          gv[4 * h + 3] = x.w;
        }
      }
      const float4* ap = reinterpret_cast<const float4*>(ape + int64_t(j) * d + c);
      float av[8];
#pragma unroll
      for (int h = 0; h < V / 4; ++h) {
        const float4 x = __ldg(ap + h);
        av[4 * h] = x.x;
        av[4 * h + 1] = x.y;
        av[4 * h + 2] = x.z;
        av[4 * h + 3] = x.w;
      }
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float ge = expf(gv[e] - m[e]);
        den[e] = __fadd_rn(den[e], ge);
        num[e] = __fadd_rn(num[e], __fmul_rn(ge, __fadd_rn(f[e], av[e])));
      }
    }
#pragma unroll
    for (int e = 0; e < V; ++e) num[e] = __fdiv_rn(num[e], den[e]);
    *reinterpret_cast<uint4*>(out + g * d + c) = pack(num, static_cast<T*>(nullptr));
  }
}

// pool_gated_kernel for a compile-time kpool: every load of a chunk (KP keys, KP
// rows of gate scores, the embedding) is issued before the arithmetic, which is the
// generic kernel's, term for term and in the same order.
template <typename T, int KP>
__global__ void __launch_bounds__(256) pool_gated_kernel_fixed(const T* __restrict__ k,
                                                               const float* __restrict__ gate,
                                                               const float* __restrict__ ape,
                                                               const int32_t* __restrict__ cu,
                                                               const int32_t* __restrict__ pool_off,
                                                               const WorkspaceHeader* __restrict__ hdr, int S, int d,
                                                               T* __restrict__ out) {
  constexpr int V = Vec<T>::kLanes;
  if (hdr->error != 0) return;
  const int64_t P = hdr->total_pools;
  const int chunks = d / V;
  const int64_t total = P * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t g = i / chunks;  // global pool row
    const int c = int(i - g * chunks) * V;
    const int b = seq_of_pool(pool_off, S, g);
    const int64_t first = int64_t(__ldg(cu + b)) + (g - __ldg(pool_off + b)) * KP;
    uint4 kv[KP];
    float4 gv4[KP][V / 4];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      kv[j] = __ldcs(reinterpret_cast<const uint4*>(k + (first + j) * d + c));
#pragma unroll
      for (int h = 0; h < V / 4; ++h) gv4[j][h] = __ldcs(reinterpret_cast<const float4*>(gate + (first + j) * d + c) + h);
    }
    float m[8], den[8], num[8];
#pragma unroll
    for (int e = 0; e < V; ++e) {
      m[e] = -INFINITY;
      den[e] = 0.0f;
      num[e] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      const float* gv = reinterpret_cast<const float*>(&gv4[j][0]);
#pragma unroll
      for (int e = 0; e < V; ++e) m[e] = fmaxf(m[e], gv[e]);
    }
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      float f[8];
      unpack(kv[j], f, static_cast<T*>(nullptr));
      const float* gv = reinterpret_cast<const float*>(&gv4[j][0]);
      const float4* ap = reinterpret_cast<const float4*>(ape + int64_t(j) * d + c);
      float av[8];
#pragma unroll
      for (int h = 0; h < V / 4; ++h) {
        const float4 x = __ldg(ap + h);
        av[4 * h] = x.x;
        av[4 * h + 1] = x.y;
        av[4 * h + 2] = x.z;
        av[4 * h + 3] = x.w;
      }
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const float ge = expf(gv[e] - m[e]);
        den[e] = __fadd_rn(den[e], ge);
        num[e] = __fadd_rn(num[e], __fmul_rn(ge, __fadd_rn(f[e], av[e])));
      }
    }
#pragma unroll
    for (int e = 0; e < V; ++e) num[e] = __fdiv_rn(num[e], den[e]);
    *reinterpret_cast<uint4*>(out + g * d + c) = pack(num, static_cast<T*>(nullptr));
  }
}

}  // namespace

cudaError_t launch_pool_gated(const void* k, const float* gate, const float* ape, kpool_dtype dtype,
                              const int32_t* cu, int32_t S, int64_t T, int32_t d, int32_t kpool, void* out,
                              const char* ws, const WorkspaceLayout& L, int num_sms, cudaStream_t stream) {
  const int64_t max_chunks = (T / kpool) * (d / (dtype == KPOOL_BF16 ? 8 : 4));
  if (max_chunks == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (max_chunks + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const auto* hdr = reinterpret_cast<const WorkspaceHeader*>(ws + L.header);
  const auto* pool_off = reinterpret_cast<const int32_t*>(ws + L.pool_off);
  if (kpool == 4) {
    if (dtype == KPOOL_BF16)
      pool_gated_kernel_fixed<__nv_bfloat16, 4><<<unsigned(blocks), threads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(k), gate, ape, cu, pool_off, hdr, S, d,
          static_cast<__nv_bfloat16*>(out));
    else
      pool_gated_kernel_fixed<float, 4><<<unsigned(blocks), threads, 0, stream>>>(
          static_cast<const float*>(k), gate, ape, cu, pool_off, hdr, S, d, static_cast<float*>(out));
  } else if (dtype == KPOOL_BF16)
    pool_gated_kernel<__nv_bfloat16><<<unsigned(blocks), threads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(k), gate, ape, cu, pool_off, hdr, S, d, kpool,
        static_cast<__nv_bfloat16*>(out));
  else
    pool_gated_kernel<float><<<unsigned(blocks), threads, 0, stream>>>(static_cast<const float*>(k), gate, ape, cu,
                                                                       pool_off, hdr, S, d, kpool,
                                                                       static_cast<float*>(out));
  return cudaGetLastError();
}

cudaError_t launch_pool(const void* k, kpool_dtype dtype, const int32_t* cu, int32_t S, int64_t T, int32_t d,
                        int32_t kpool, void* out, const char* ws, const WorkspaceLayout& L, int num_sms,
                        cudaStream_t stream) {
  const int64_t max_chunks = (T / kpool) * (d / (dtype == KPOOL_BF16 ? 8 : 4));
  if (max_chunks == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (max_chunks + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const auto* hdr = reinterpret_cast<const WorkspaceHeader*>(ws + L.header);
  const auto* pool_off = reinterpret_cast<const int32_t*>(ws + L.pool_off);
  if (kpool == 4) {
    // one wave: the fixed kernel's registers allow 4 CTAs of 256 threads per SM
    if (blocks > int64_t(num_sms) * 4) blocks = int64_t(num_sms) * 4;
    if (dtype == KPOOL_BF16)
      pool_kernel_fixed<__nv_bfloat16, 4><<<unsigned(blocks), threads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(k), cu, pool_off, hdr, S, d, static_cast<__nv_bfloat16*>(out));
    else
      pool_kernel_fixed<float, 4><<<unsigned(blocks), threads, 0, stream>>>(static_cast<const float*>(k), cu,
                                                                           pool_off, hdr, S, d,
                                                                           static_cast<float*>(out));
  } else if (dtype == KPOOL_BF16)
    pool_kernel<__nv_bfloat16><<<unsigned(blocks), threads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(k), cu, pool_off, hdr, S, d, kpool, static_cast<__nv_bfloat16*>(out));
  else
    pool_kernel<float><<<unsigned(blocks), threads, 0, stream>>>(static_cast<const float*>(k), cu, pool_off, hdr,
                                                                 S, d, kpool, static_cast<float*>(out));
  return cudaGetLastError();
}

}  // namespace kpool
