// gemm_simt.cu -- CUDA-core grouped GEMM with fp32 accumulation.
//
// Serves the fp32 layer (the tensor cores have no fp32-exact mode: tf32 keeps 10 mantissa bits)
// and the split-K router GEMM for few tokens, where a tensor-core tile would be mostly empty.
// Computes, per group, out[row][f] = sum_k act[row][k] * w[wrow(f)][k] with the SwiGLU epilogue
// h = SiLU(x W1) * (x W3) ("Mixture of experts" steps g, u, a, h) or a plain store.
// 64 x 64 output tiles, 256 threads with 4 x 4 outputs each, K in steps of 16 through shared memory.
#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

struct SimtParams {
  const void* act;
  const void* w;
  const void* act_d;
  const void* w_d;
  const int32_t* offsets;
  int n_routed, w_group_rows, u_off, u_off_d;
  int dense_rows, dense_act_row0, dense_out_row0;
  int64_t act_rows, act_d_rows;
  int K, k_wrap, F, k_splits;
  int64_t split_stride;
  void* out;
  int64_t ldo;
  int out_f32;
  uint32_t* err;
};

constexpr int kSimtTile = 64;
constexpr int kSimtK = 16;
constexpr int kSimtThreads = 256;
constexpr int kSimtMaxGroups = 1025;

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p) {
  return to_f32<T>(p[0]);
}

// Four consecutive values as fp32 with one vector load (p 16-byte aligned for fp32, 8 for bf16).
__device__ __forceinline__ void ld4_f32(const float* p, float (&v)[4]) {
  const float4 q = *reinterpret_cast<const float4*>(p);
  v[0] = q.x;
  v[1] = q.y;
  v[2] = q.z;
  v[3] = q.w;
}
__device__ __forceinline__ void ld4_f32(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
  v[0] = a.x;
  v[1] = a.y;
  v[2] = b.x;
  v[3] = b.y;
}

template <typename TA, typename TW, bool kSwiGLU>
__global__ void __launch_bounds__(kSimtThreads) moe_gemm_simt_kernel(const SimtParams p) {
  __shared__ int tile_start[kSimtMaxGroups + 1];
  __shared__ int row_start[kSimtMaxGroups + 1];
  __shared__ int scratch[kSimtThreads];
  __shared__ float As[kSimtK][kSimtTile + 4];
  __shared__ float Bg[kSimtK][kSimtTile + 4];
  __shared__ float Bu[kSwiGLU ? kSimtK : 1][kSwiGLU ? kSimtTile + 4 : 1];

  const int feat_tiles = (p.F + kSimtTile - 1) / kSimtTile;
  build_tile_table(tile_start, row_start, scratch, p.offsets, p.n_routed, p.dense_rows,
                   kSimtTile, feat_tiles);
  const int G = p.n_routed + (p.dense_rows > 0 ? 1 : 0);
  const int total = tile_start[G];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int ksplit = blockIdx.y;
  const int klen = p.K / p.k_splits;
  const int k_begin = ksplit * klen;

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                    p.dense_rows, p.dense_act_row0, kSimtTile);
    const TA* A = (const TA*)(ti.dense ? p.act_d : p.act);
    const TW* W = (const TW*)(ti.dense ? p.w_d : p.w);
    const int64_t a_row0 = (int64_t)ti.grp_row0 + (int64_t)ti.rt * kSimtTile;
    const int64_t w_row0 = (ti.dense ? 0 : (int64_t)ti.g * p.w_group_rows) +
                           (int64_t)ti.ft * kSimtTile;
    const int f0 = ti.ft * kSimtTile;
    const int uoff = ti.dense ? p.u_off_d : p.u_off;

    float accg[4][4], accu[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) accg[i][j] = accu[i][j] = 0.0f;

    // each thread stages 4 consecutive k of one row of A and of W (and W3); the next K-step's
    // values are loaded into registers while the current one is multiplied out of shared memory
    const int lr = threadIdx.x / 4;
    const int lk = (threadIdx.x % 4) * 4;
    const bool a_ok = lr < ti.valid, w_ok = f0 + lr < p.F;
    const bool wrap = p.k_wrap != p.K;
    const TA* a_row = A + (a_row0 + lr) * p.k_wrap;
    const TW* wg_row = W + (w_row0 + lr) * p.K;
    const TW* wu_row = W + (w_row0 + uoff + lr) * p.K;
    float ra[4], rg[4], ru[4];
    // 4 consecutive k per row: one vector load each (k0 + lk is a multiple of 4, and a wrapped
    // activation row repeats with a period that is a multiple of 16)
    auto fetch = [&](int k0) {
      const int kk = k0 + lk;
#pragma unroll
      for (int j = 0; j < 4; ++j) ra[j] = rg[j] = ru[j] = 0.0f;
      if (a_ok) ld4_f32(a_row + (wrap ? kk % p.k_wrap : kk), ra);
      if (w_ok) {
        ld4_f32(wg_row + kk, rg);
        if (kSwiGLU) ld4_f32(wu_row + kk, ru);
      }
    };
    fetch(k_begin);
    for (int k0 = k_begin; k0 < k_begin + klen; k0 += kSimtK) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        As[lk + j][lr] = ra[j];
        Bg[lk + j][lr] = rg[j];
        if (kSwiGLU) Bu[lk + j][lr] = ru[j];
      }
      __syncthreads();
      if (k0 + kSimtK < k_begin + klen) fetch(k0 + kSimtK);
#pragma unroll
      for (int kk = 0; kk < kSimtK; ++kk) {
        float a[4], bg[4], bu[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bg[j] = Bg[kk][tx * 4 + j];
          if (kSwiGLU) bu[j] = Bu[kk][tx * 4 + j];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            accg[i][j] = fmaf(a[i], bg[j], accg[i][j]);
            if (kSwiGLU) accu[i][j] = fmaf(a[i], bu[j], accu[i][j]);
          }
      }
      __syncthreads();
    }

    const int64_t out_row0 =
        (ti.dense ? (int64_t)p.dense_out_row0 : (int64_t)ti.grp_row0) + (int64_t)ti.rt * kSimtTile;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty * 4 + i;
      if (r >= ti.valid) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int f = f0 + tx * 4 + j;
        if (f >= p.F) continue;
        const float v = kSwiGLU ? silu_accurate(accg[i][j]) * accu[i][j] : accg[i][j];
        const int64_t o = (out_row0 + r) * p.ldo + f + (int64_t)ksplit * p.split_stride;
        if (p.out_f32)
          ((float*)p.out)[o] = v;
        else
          ((__nv_bfloat16*)p.out)[o] = __float2bfloat16_rn(v);
      }
    }
  }
}

cudaError_t launch_gemm_simt(const GroupedGemm& g, int num_sms, cudaStream_t st) {
  if (g.n_routed > kSimtMaxGroups - 1) return cudaErrorInvalidValue;
  if (g.K % (kSimtK * g.k_splits) || (g.K / g.k_splits) % kSimtK) return cudaErrorInvalidValue;
  // operands are read 4 consecutive values at a time with vector loads
  auto aligned16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  if (!aligned16(g.act) || !aligned16(g.w) || !aligned16(g.act_d) || !aligned16(g.w_d))
    return cudaErrorInvalidValue;
  if (g.k_wrap > 0 && g.k_wrap % kSimtK) return cudaErrorInvalidValue;
  if (g.epi == EPI_STORE_ADD) return cudaErrorInvalidValue;
  SimtParams p;
  p.act = g.act;
  p.w = g.w;
  p.act_d = g.act_d;
  p.w_d = g.w_d;
  p.offsets = g.offsets;
  p.n_routed = g.n_routed;
  p.w_group_rows = g.w_group_rows;
  p.u_off = g.u_off;
  p.u_off_d = g.u_off_d;
  p.dense_rows = g.dense_rows;
  p.dense_act_row0 = g.dense_act_row0;
  p.dense_out_row0 = g.dense_out_row0;
  p.act_rows = g.act_rows;
  p.act_d_rows = g.act_d_rows;
  p.K = g.K;
  p.k_wrap = g.k_wrap > 0 ? g.k_wrap : g.K;
  p.F = g.F;
  p.k_splits = g.k_splits;
  p.split_stride = g.split_stride;
  p.out = g.out;
  p.ldo = g.ldo;
  p.out_f32 = g.out_dtype == MOE_F32;
  p.err = g.err;
  // at most as many CTAs as tiles can exist: routed groups have at most P/64 + n_routed row
  // tiles in total, the dense group ceil(rows/64)
  const int64_t ftiles = (g.F + kSimtTile - 1) / kSimtTile;
  const int64_t rtiles = (g.n_routed > 0 ? g.act_rows / kSimtTile + g.n_routed : 0) +
                         (g.dense_rows + kSimtTile - 1) / kSimtTile;
  const int64_t bound = rtiles * ftiles;
  dim3 grid((unsigned)(bound < num_sms * 4 ? (bound > 0 ? bound : 1) : num_sms * 4), g.k_splits);
  const bool swiglu = g.epi == EPI_SWIGLU;
  LaunchScope ls(g.label, st);
  if (g.act_dtype == MOE_F32 && g.w_dtype == MOE_F32) {
    if (swiglu)
      moe_gemm_simt_kernel<float, float, true><<<grid, kSimtThreads, 0, st>>>(p);
    else
      moe_gemm_simt_kernel<float, float, false><<<grid, kSimtThreads, 0, st>>>(p);
  } else if (g.act_dtype == MOE_BF16 && g.w_dtype == MOE_F32) {
    if (swiglu)
      moe_gemm_simt_kernel<__nv_bfloat16, float, true><<<grid, kSimtThreads, 0, st>>>(p);
    else
      moe_gemm_simt_kernel<__nv_bfloat16, float, false><<<grid, kSimtThreads, 0, st>>>(p);
  } else if (g.act_dtype == MOE_BF16 && g.w_dtype == MOE_BF16) {
    if (swiglu)
      moe_gemm_simt_kernel<__nv_bfloat16, __nv_bfloat16, true><<<grid, kSimtThreads, 0, st>>>(p);
    else
      moe_gemm_simt_kernel<__nv_bfloat16, __nv_bfloat16, false><<<grid, kSimtThreads, 0, st>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
