// block.cu -- the steps on either side of the MoE layer inside a transformer block.
//
// "Kimi K2 · Transformer blocks > MoE transformer block":
//   x_ffn = RMSNorm(x'_n) ;  ... Mixture of experts ... ;  x_{n+1} = x'_n + D_ffn
// with the post-attention RMSNorm a DeepseekV3RMSNorm((7168,), eps=1e-06) of 7168 learned weights
// (nnterp "kimi_k2", "Printout"; the "Parameters" table's "MoE RMSNorm 7,168").
//
// rmsnorm_rows_kernel: y = w * x / sqrt(mean(x^2) + eps) per row, in fp32, rounded once to the
//   activation type (the input of the router and expert GEMMs).  One CTA per row (grid-stride).
// add_residual_kernel: y_f32 += r, for the K3 path, whose output is written by the up-projection
//   epilogue as u_hat W_up^T + (fp32 addend): the residual joins the shared-expert rows there, so
//   the block output is still rounded once.
#include "common.cuh"
#include "internal.h"

namespace moe {

template <typename TX>
__global__ void __launch_bounds__(256)
    rmsnorm_rows_kernel(const TX* __restrict__ x, const TX* __restrict__ w, float eps, int64_t T,
                        int d, TX* __restrict__ y) {
  __shared__ float red[32];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const TX* xr = x + t * d;
    float ss = 0.0f;
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float v[8];
      load8(xr + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __syncthreads();  // red[] of the previous row has been read
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
      float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float inv = 1.0f / sqrtf(red[0] / (float)d + eps);
    for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
      float v[8], g[8];
      load8(xr + c, v);
      load8(w + c, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = g[i] * (v[i] * inv);
      store8(y + t * d + c, v);
    }
  }
}

template <typename TR>
__global__ void __launch_bounds__(256)
    add_residual_kernel(float* __restrict__ y, const TR* __restrict__ r, int64_t n8) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float a[8], b[8];
    load8(y + i * 8, a);
    load8(r + i * 8, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] += b[j];
    store8(y + i * 8, a);
  }
}

cudaError_t launch_rmsnorm_rows(int act_dtype, const void* x, const void* w, float eps, int64_t T,
                                int d, void* y, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (d % 8) return cudaErrorInvalidValue;
  const int64_t blocks = T < (int64_t)num_sms * 8 ? T : (int64_t)num_sms * 8;
  LaunchScope ls("block_rmsnorm", st);
  if (act_dtype == MOE_BF16)
    rmsnorm_rows_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        (const __nv_bfloat16*)x, (const __nv_bfloat16*)w, eps, T, d, (__nv_bfloat16*)y);
  else
    rmsnorm_rows_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(
        (const float*)x, (const float*)w, eps, T, d, (float*)y);
  return cudaGetLastError();
}

cudaError_t launch_add_residual(float* y, int act_dtype, const void* r, int64_t n, int num_sms,
                                cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  const int64_t n8 = n / 8;
  const int64_t want = (n8 + 255) / 256;
  const int64_t blocks = want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8;
  LaunchScope ls("block_residual", st);
  if (act_dtype == MOE_BF16)
    add_residual_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        y, (const __nv_bfloat16*)r, n8);
  else
    add_residual_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(y, (const float*)r, n8);
  return cudaGetLastError();
}

}  // namespace moe
