// combine.cu -- un-permute, gate-weighted sum over the k slots, plus the shared expert.
//
// "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps
//   y_routed = sum_i G_i E_i ;  D_ffn = y_routed + y_shared
// and the back half of the `moe_infer` code excerpt on "Kimi K3 · Latent up-projection" (put the
// expert outputs back in (token, slot) order, multiply by the gate weights, sum over the slots).
// One CTA per token (grid-stride); 16-byte vectors; the sum is kept in fp32 and rounded once.
//
// K3 latent: the same weighted sum in the latent width, then (optionally) RMSNorm with unit weight
// y / sqrt(mean(y^2) + eps) in fp32, stored bf16 as the input of the up-projection GEMM.
#include "common.cuh"
#include "internal.h"

namespace moe {

template <typename TY>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {  // 8 x bf16 per 16 bytes
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 raw;
    raw.x = pack_bf16x2(v[0], v[1]);
    raw.y = pack_bf16x2(v[2], v[3]);
    raw.z = pack_bf16x2(v[4], v[5]);
    raw.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = raw;
  }
};
template <>
struct Vec<float> {  // 4 x fp32 per 16 bytes
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

constexpr int kMaxK = 32;

template <typename TY>
__global__ void __launch_bounds__(256)
    combine_kernel(const TY* __restrict__ y_perm, const TY* __restrict__ y_shared,
                   const int32_t* __restrict__ perm_dst, const float* __restrict__ weight,
                   int64_t T, int k, int d, TY* __restrict__ out) {
  constexpr int N = Vec<TY>::N;
  __shared__ int64_t rows[kMaxK];
  __shared__ float gw[kMaxK];
  const int64_t P = T * k;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      const int r = perm_dst[t * k + threadIdx.x];
      rows[threadIdx.x] = (r >= 0 && r < P) ? (int64_t)r : -1;
      gw[threadIdx.x] = weight[t * k + threadIdx.x];
    }
    __syncthreads();
    for (int c = threadIdx.x * N; c < d; c += blockDim.x * N) {
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.0f;
      for (int j = 0; j < k; ++j) {
        if (rows[j] < 0) continue;
        float v[N];
        Vec<TY>::load(y_perm + rows[j] * d + c, v);
        const float w = gw[j];
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = fmaf(w, v[i], acc[i]);
      }
      if (y_shared) {
        float v[N];
        Vec<TY>::load(y_shared + t * d + c, v);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] += v[i];
      }
      Vec<TY>::store(out + t * d + c, acc);
    }
  }
}

cudaError_t launch_combine(int act_dtype, const void* y_perm, const void* y_shared,
                           const int32_t* perm_dst, const float* weight, int64_t T, int k, int d,
                           void* out, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (k > kMaxK) return cudaErrorInvalidValue;
  const int64_t blocks = T < (int64_t)num_sms * 8 ? T : (int64_t)num_sms * 8;
  if (act_dtype == MOE_BF16) {
    if (d % 8) return cudaErrorInvalidValue;
    combine_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        (const __nv_bfloat16*)y_perm, (const __nv_bfloat16*)y_shared, perm_dst, weight, T, k, d,
        (__nv_bfloat16*)out);
  } else {
    if (d % 4) return cudaErrorInvalidValue;
    combine_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(
        (const float*)y_perm, (const float*)y_shared, perm_dst, weight, T, k, d, (float*)out);
  }
  count_launch();
  return cudaGetLastError();
}

// K3: weighted latent sum -> optional RMSNorm -> bf16 u_hat.  One CTA per token, the fp32 sum kept
// in shared memory (L <= 8192).
constexpr int kMaxLatent = 8192;

__global__ void __launch_bounds__(256)
    latent_combine_kernel(const __nv_bfloat16* __restrict__ y_perm,
                          const int32_t* __restrict__ perm_dst, const float* __restrict__ weight,
                          int64_t T, int k, int L, int norm, float eps,
                          __nv_bfloat16* __restrict__ u_hat) {
  __shared__ float ysum[kMaxLatent];
  __shared__ int64_t rows[kMaxK];
  __shared__ float gw[kMaxK];
  __shared__ float red[32];
  const int64_t P = T * k;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      const int r = perm_dst[t * k + threadIdx.x];
      rows[threadIdx.x] = (r >= 0 && r < P) ? (int64_t)r : -1;
      gw[threadIdx.x] = weight[t * k + threadIdx.x];
    }
    __syncthreads();
    float ss = 0.0f;
    for (int c = threadIdx.x * 8; c < L; c += blockDim.x * 8) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int j = 0; j < k; ++j) {
        if (rows[j] < 0) continue;
        float v[8];
        Vec<__nv_bfloat16>::load(y_perm + rows[j] * L + c, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(gw[j], v[i], acc[i]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ysum[c + i] = acc[i];
        ss = fmaf(acc[i], acc[i], ss);
      }
    }
    float scale = 1.0f;
    if (norm) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
      __syncthreads();
      if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (threadIdx.x == 0) red[0] = v;
      }
      __syncthreads();
      scale = rsqrtf(red[0] / (float)L + eps);
    }
    for (int c = threadIdx.x * 8; c < L; c += blockDim.x * 8) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ysum[c + i] * scale;
      Vec<__nv_bfloat16>::store(u_hat + t * L + c, v);
    }
  }
}

cudaError_t launch_latent_combine(const void* y_perm, const int32_t* perm_dst,
                                  const float* weight, int64_t T, int k, int L, int norm,
                                  float eps, void* u_hat, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (k > kMaxK || L > kMaxLatent || L % 8) return cudaErrorInvalidValue;
  const int64_t blocks = T < (int64_t)num_sms * 8 ? T : (int64_t)num_sms * 8;
  latent_combine_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      (const __nv_bfloat16*)y_perm, perm_dst, weight, T, k, L, norm, eps,
      (__nv_bfloat16*)u_hat);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
