// quant.cu -- e4m3 activation quantisation for the fp8 expert path, and the copy of the quantised
// rows with their scales into the expert-major order.
//
// Expert weights stored as e4m3 with block scales, the form the nnterp "kimi_k2" note gives for the
// K2 checkpoints ("FP8 blocks"); activations entering the expert GEMMs are quantised per token per
// 128 channels with scale = amax / 448 (1 for an all-zero group) and code = e4m3(x / scale), round
// to nearest even with saturation.  Both the scale and the quotient are IEEE fp32 divisions.
// Scales are stored transposed, [groups][rows], so that the GEMM epilogue (one thread per row)
// reads them coalesced.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  // cvt.rn.satfinite.e4m3x2.f32 packs (hi, lo): the first source goes to the upper byte
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// One warp per (row, 128-channel group): each lane converts 4 consecutive channels.
__global__ void __launch_bounds__(256)
    quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int d,
                         uint8_t* __restrict__ q, float* __restrict__ sT) {
  const int lane = threadIdx.x & 31;
  const int groups = d / 128;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= rows * groups) return;
  const int64_t r = w / groups;
  const int g = (int)(w - r * groups);
  const __nv_bfloat16* src = x + r * d + g * 128 + lane * 4;
  const uint2 raw = *reinterpret_cast<const uint2*>(src);
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
  const float2 a = __bfloat1622float2(h2[0]);
  const float2 b = __bfloat1622float2(h2[1]);
  float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const uint32_t packed = e4m3x4(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale),
                                 __fdiv_rn(b.x, scale), __fdiv_rn(b.y, scale));
  *reinterpret_cast<uint32_t*>(q + r * d + g * 128 + lane * 4) = packed;
  if (lane == 0) sT[(int64_t)g * rows + r] = scale;
}

cudaError_t launch_quantize_rows(const void* x, int64_t rows, int d, uint8_t* q, float* sT,
                                 cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (d % 128) return cudaErrorInvalidValue;
  const int64_t warps = rows * (d / 128);
  const int64_t blocks = (warps + 7) / 8;
  LaunchScope ls("quantize_x_e4m3", st);
  quantize_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>((const __nv_bfloat16*)x, rows, d, q, sT);
  return cudaGetLastError();
}

// dst[r] = src[perm_src[r] / k] (d bytes of e4m3 codes) and dst_sT[g][r] = src_sT[g][t].
// The e4m3 rows in the permuted order, token by token: each token's codes and scales are read
// once and written to its k permuted rows (perm_dst); pairs whose destination is outside [0, P)
// are skipped.
__global__ void __launch_bounds__(256)
    scatter_q_kernel(const uint8_t* __restrict__ src, const float* __restrict__ src_sT, int64_t T,
                     const int32_t* __restrict__ perm_dst, int k, int64_t P, int d,
                     uint8_t* __restrict__ dst, float* __restrict__ dst_sT) {
  __shared__ int64_t rows[32];
  const int vec = d / 16;
  const int groups = d / 128;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      const int r = perm_dst[t * k + threadIdx.x];
      rows[threadIdx.x] = (r >= 0 && r < P) ? (int64_t)r : -1;
    }
    __syncthreads();
    const uint4* in = reinterpret_cast<const uint4*>(src + t * d);
    for (int v = threadIdx.x; v < vec; v += blockDim.x) {
      const uint4 val = __ldg(in + v);
      for (int j = 0; j < k; ++j)
        if (rows[j] >= 0) reinterpret_cast<uint4*>(dst + rows[j] * d)[v] = val;
    }
    for (int g = threadIdx.x; g < groups; g += blockDim.x) {
      const float sc = src_sT[(int64_t)g * T + t];
      for (int j = 0; j < k; ++j)
        if (rows[j] >= 0) dst_sT[(int64_t)g * P + rows[j]] = sc;
    }
  }
}

cudaError_t launch_scatter_q(const uint8_t* src, const float* src_sT, int64_t T,
                             const int32_t* perm_dst, int k, int64_t P, int d, uint8_t* dst,
                             float* dst_sT, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (d % 128 || k > 32) return cudaErrorInvalidValue;
  const int64_t blocks = T < (int64_t)num_sms * 8 ? T : (int64_t)num_sms * 8;
  LaunchScope ls("scatter_rows_e4m3", st);
  scatter_q_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, src_sT, T, perm_dst, k, P, d, dst,
                                                     dst_sT);
  return cudaGetLastError();
}

}  // namespace moe
