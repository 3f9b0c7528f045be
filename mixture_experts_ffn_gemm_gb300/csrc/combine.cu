// combine.cu -- un-permute, gate-weighted sum over the k slots, plus the shared expert.
//
// "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps
//   y_routed = sum_i G_i E_i ;  D_ffn = y_routed + y_shared
// and the back half of the `moe_infer` code excerpt on "Kimi K3 · Latent up-projection" (put the
// expert outputs back in (token, slot) order, multiply by the gate weights, sum over the slots).
// One CTA per token (grid-stride); the expert outputs arrive in fp32, the sum is kept in fp32 and
// rounded once to the output type.
//
// K3 latent: the same weighted sum in the latent width, then (optionally) RMSNorm with unit weight
// y / sqrt(mean(y^2) + eps) in fp32, stored bf16 as the input of the up-projection GEMM.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kMaxK = 32;

// y_perm and y_shared hold the expert outputs (fp32, or bf16 on request); resid (optional, the
// block's residual stream) is in the output type; out is bf16 or fp32, rounded once from the fp32
// sum.  T tokens (a chunk of
// the batch when the caller offsets perm_dst, weight, y_shared, resid and out); P is the number of
// rows of y_perm, so that perm_dst entries outside [0, P) read nothing.
// acc[0..N-1] += sum over the token's k slots of gw[j] * y[rows[j]][c .. c+N-1], in slot order.
// Four rows are loaded before any is used (a skipped slot, rows[j] < 0, reads nothing and adds
// zero), so each thread has four row loads in flight instead of one.  N is a multiple of 8.
template <int N, typename TY>
__device__ __forceinline__ void gather_rows(const TY* __restrict__ y, const int64_t* rows,
                                            const float* gw, int k, int64_t width, int c,
                                            float (&acc)[N]) {
  for (int j0 = 0; j0 < k; j0 += 4) {
    float v[4][N];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u;
      if (j < k && rows[j] >= 0) {
#pragma unroll
        for (int h = 0; h < N / 8; ++h)
          load8(y + rows[j] * width + c + 8 * h, *reinterpret_cast<float(*)[8]>(&v[u][8 * h]));
      } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[u][i] = 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float g = j0 + u < k ? gw[j0 + u] : 0.0f;
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(g, v[u][i], acc[i]);
    }
  }
}

// N consecutive values as fp32 (N a multiple of 8), and back.
template <int N, typename T>
__device__ __forceinline__ void loadn(const T* p, float (&v)[N]) {
#pragma unroll
  for (int h = 0; h < N / 8; ++h) load8(p + 8 * h, *reinterpret_cast<float(*)[8]>(&v[8 * h]));
}
template <int N, typename T>
__device__ __forceinline__ void storen(T* p, const float (&v)[N]) {
#pragma unroll
  for (int h = 0; h < N / 8; ++h)
    store8(p + 8 * h, *reinterpret_cast<const float(*)[8]>(&v[8 * h]));
}

// TY: the expert outputs' type (fp32, or bf16 on request); a thread takes 8 columns of every row
// per step (16 bf16 columns per step measured slower: 0.73 against 0.65 ms at prefill).
template <typename TO, typename TY>
__global__ void __launch_bounds__(256)
    combine_kernel(const TY* __restrict__ y_perm, const TY* __restrict__ y_shared,
                   const int32_t* __restrict__ perm_dst, const float* __restrict__ weight,
                   int64_t T, int k, int64_t P, int d, const TO* __restrict__ resid,
                   TO* __restrict__ out, int cols_per_block) {
  constexpr int N = 8;
  __shared__ int64_t rows[kMaxK];
  __shared__ float gw[kMaxK];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      const int r = perm_dst[t * k + threadIdx.x];
      rows[threadIdx.x] = (r >= 0 && r < P) ? (int64_t)r : -1;
      gw[threadIdx.x] = weight[t * k + threadIdx.x];
    }
    __syncthreads();
    // columns [c_begin, c_end) of the row: the whole row, or one slice of it when few tokens
    // spread over blockIdx.y
    const int c_begin = blockIdx.y * cols_per_block;
    const int c_end = min(d, c_begin + cols_per_block);
    for (int c = c_begin + threadIdx.x * N; c < c_end; c += blockDim.x * N) {
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.0f;
      gather_rows<N>(y_perm, rows, gw, k, d, c, acc);
      if (y_shared) {
        float v[N];
        loadn<N>(y_shared + t * d + c, v);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] += v[i];
      }
      if (resid) {
        float v[N];
        loadn<N>(resid + t * d + c, v);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] += v[i];
      }
      storen<N>(out + t * d + c, acc);
    }
  }
}

cudaError_t launch_combine(int act_dtype, bool y_bf16, const void* y_perm, const void* y_shared,
                           const int32_t* perm_dst, const float* weight, int64_t T, int k,
                           int64_t P, int d, const void* resid, void* out, int num_sms,
                           cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (k > kMaxK || d % 8) return cudaErrorInvalidValue;
  // few tokens: each row in slices of 2048 columns (one 8-column chunk per thread) over
  // blockIdx.y, so that every slice's loads are in flight at once
  const int slices = T < (int64_t)num_sms * 4 ? (d + 2047) / 2048 : 1;
  // many tokens with bf16 expert outputs: blocks of 128 threads, twice as many tokens in flight
  // per SM (0.30 against 0.33 ms at the fp8 layer; fp32 outputs measured no better that way)
  const int threads = (slices == 1 && y_bf16) ? 128 : 256;
  const int64_t per_sm = 2048 / threads;
  const int64_t blocks = T < (int64_t)num_sms * per_sm ? T : (int64_t)num_sms * per_sm;
  const int cols = slices > 1 ? 2048 : d;
  const dim3 grid((unsigned)blocks, (unsigned)slices);
  LaunchScope ls("combine", st);
  if (act_dtype == MOE_BF16 && y_bf16)
    combine_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, threads, 0, st>>>(
        (const __nv_bfloat16*)y_perm, (const __nv_bfloat16*)y_shared, perm_dst, weight, T, k, P,
        d, (const __nv_bfloat16*)resid, (__nv_bfloat16*)out, cols);
  else if (act_dtype == MOE_BF16)
    combine_kernel<__nv_bfloat16, float><<<grid, threads, 0, st>>>(
        (const float*)y_perm, (const float*)y_shared, perm_dst, weight, T, k, P, d,
        (const __nv_bfloat16*)resid, (__nv_bfloat16*)out, cols);
  else if (!y_bf16)
    combine_kernel<float, float><<<grid, threads, 0, st>>>(
        (const float*)y_perm, (const float*)y_shared, perm_dst, weight, T, k, P, d,
        (const float*)resid, (float*)out, cols);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// K3: weighted latent sum -> optional RMSNorm -> bf16 u_hat.  One CTA per token, the fp32 sum kept
// in shared memory (L <= 8192).
constexpr int kMaxLatent = 8192;

__global__ void __launch_bounds__(256)
    latent_combine_kernel(const float* __restrict__ y_perm,
                          const int32_t* __restrict__ perm_dst, const float* __restrict__ weight,
                          int64_t T, int k, int64_t P, int L, int norm, float eps,
                          __nv_bfloat16* __restrict__ u_hat) {
  __shared__ float ysum[kMaxLatent];
  __shared__ int64_t rows[kMaxK];
  __shared__ float gw[kMaxK];
  __shared__ float red[32];
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
      gather_rows<8>(y_perm, rows, gw, k, L, c, acc);
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
      store8(u_hat + t * L + c, v);
    }
  }
}

cudaError_t launch_latent_combine(const void* y_perm, const int32_t* perm_dst,
                                  const float* weight, int64_t T, int k, int64_t P, int L,
                                  int norm, float eps, void* u_hat, int num_sms,
                                  cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (k > kMaxK || L > kMaxLatent || L % 8) return cudaErrorInvalidValue;
  const int64_t blocks = T < (int64_t)num_sms * 8 ? T : (int64_t)num_sms * 8;
  LaunchScope ls("latent_combine", st);
  latent_combine_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      (const float*)y_perm, perm_dst, weight, T, k, P, L, norm, eps,
      (__nv_bfloat16*)u_hat);
  return cudaGetLastError();
}

// out[i] = RN(sum_s part[s * n + i]) over the k-split partials in slice order (fp32 sum, one
// rounding to bf16): the last step of a split-K dense projection.  8 values per thread; the S
// slices' loads are issued before any is added.
template <int S>
__global__ void splitk_sum_kernel(const float* __restrict__ part, int64_t n,
                                  __nv_bfloat16* __restrict__ out) {
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < n;
       i += (int64_t)gridDim.x * blockDim.x * 8) {
    float v[S][8];
#pragma unroll
    for (int sl = 0; sl < S; ++sl) load8(part + (int64_t)sl * n + i, v[sl]);
#pragma unroll
    for (int sl = 1; sl < S; ++sl)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[0][j] += v[sl][j];
    store8(out + i, v[0]);
  }
}

cudaError_t launch_splitk_sum(const float* part, int S, int64_t n, void* out, int num_sms,
                              cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (S < 1 || S > 8 || n % 8) return cudaErrorInvalidValue;
  const int64_t want = (n / 8 + 255) / 256;
  const unsigned blocks = (unsigned)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
  LaunchScope ls("splitk_sum", st);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  switch (S) {
#define MOE_SPLITK_CASE(NS) \
  case NS:                  \
    splitk_sum_kernel<NS><<<blocks, 256, 0, st>>>(part, n, o); \
    break;
    MOE_SPLITK_CASE(1)
    MOE_SPLITK_CASE(2)
    MOE_SPLITK_CASE(3)
    MOE_SPLITK_CASE(4)
    MOE_SPLITK_CASE(5)
    MOE_SPLITK_CASE(6)
    MOE_SPLITK_CASE(7)
    MOE_SPLITK_CASE(8)
#undef MOE_SPLITK_CASE
  }
  return cudaGetLastError();
}

}  // namespace moe
