// router.cu -- selection and gates.
//
// "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps:
//   s = sigma(z) ; E_sel_i = [i in top_8(s + b)] ; G_i = 2.827 s_i E_sel_i / sum_j s_j E_sel_j
// and nnterp "kimi_k2", note "The mixture of experts": the bias b only selects, the gates are the
// unbiased sigmoids of the selected experts renormalised and scaled by routed_scaling_factor.
//
// One warp per token.  The logits come either from one buffer or from split-K partial slices
// (summed here in a fixed order, so the result does not depend on scheduling).  Each lane holds the
// keys of experts lane, lane+32, ...; k rounds of a warp arg-max (key descending, ties to the lower
// expert index) pick the experts in slot order.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kTopkWarps = 8;
constexpr int kMaxExpertsPerLane = 32;  // E <= 1024

// EPL = experts per lane (ceil(E / 32)), a compile-time bound so that only real slots are kept.
template <int EPL>
__global__ void __launch_bounds__(kTopkWarps * 32)
    router_topk_kernel(const float* __restrict__ partial, int S, int64_t split_stride, int64_t T,
                       int E, int k, const float* __restrict__ b, float gate_scale,
                       float* __restrict__ logits_out, int32_t* __restrict__ idx,
                       float* __restrict__ weight) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform

  float key[EPL];
  float sig[EPL];
  // the split-K slices summed in slice order; the loads of U slices are issued before any of
  // them is added, so that a lane has U * EPL loads in flight
  constexpr int U = EPL <= 12 ? 4 : 1;
  float zs[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) zs[j] = 0.0f;
  int s = 0;
  for (; s + U <= S; s += U) {
    float v[U][EPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float* ps = partial + (s + u) * split_stride + t * E;
#pragma unroll
      for (int j = 0; j < EPL; ++j) v[u][j] = lane + 32 * j < E ? ps[lane + 32 * j] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < EPL; ++j) zs[j] += v[u][j];
  }
  for (; s < S; ++s) {
    const float* ps = partial + s * split_stride + t * E;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (lane + 32 * j < E) zs[j] += ps[lane + 32 * j];
  }
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    key[j] = -INFINITY;
    sig[j] = 0.0f;
    if (e < E) {
      const float z = zs[j];
      if (logits_out) logits_out[t * E + e] = z;
      const float sg = 1.0f / (1.0f + expf(-z));
      const float kv = sg + b[e];
      sig[j] = sg;
      key[j] = isnan(kv) ? -INFINITY : kv;
    }
  }

  uint32_t taken = 0;
  int my_e = 0;
  float my_s = 0.0f;
  float den = 0.0f;
  for (int slot = 0; slot < k; ++slot) {
    float bk = -INFINITY;
    int be = 0x7fffffff;
    float bs = 0.0f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && (key[j] > bk || (key[j] == bk && e < be))) {
        bk = key[j];
        be = e;
        bs = sig[j];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      const float os = __shfl_xor_sync(0xffffffffu, bs, off);
      if (ok > bk || (ok == bk && oe < be)) {
        bk = ok;
        be = oe;
        bs = os;
      }
    }
    if (lane == slot) {
      my_e = be;
      my_s = bs;
    }
    den += bs;  // same order on every lane
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
  }
  if (lane < k) {
    idx[t * k + lane] = my_e;
    weight[t * k + lane] = gate_scale * my_s / den;
  }
}

cudaError_t launch_router_topk(const float* partial, int S, int64_t split_stride, int64_t T,
                               int E, int k, const float* b, float gate_scale, float* logits_out,
                               int32_t* idx, float* weight, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (E > 32 * kMaxExpertsPerLane || k > 32 || k > E) return cudaErrorInvalidValue;
  const int64_t blocks = (T + kTopkWarps - 1) / kTopkWarps;
  const int epl = (E + 31) / 32;
  LaunchScope ls("router_topk", st);
#define MOE_TOPK_CASE(N)                                                               \
  if (epl <= N) {                                                                      \
    router_topk_kernel<N><<<(unsigned)blocks, kTopkWarps * 32, 0, st>>>(               \
        partial, S, split_stride, T, E, k, b, gate_scale, logits_out, idx, weight);    \
    return cudaGetLastError();                                                         \
  }
  MOE_TOPK_CASE(1)
  MOE_TOPK_CASE(2)
  MOE_TOPK_CASE(4)
  MOE_TOPK_CASE(8)
  MOE_TOPK_CASE(12)
  MOE_TOPK_CASE(16)
  MOE_TOPK_CASE(24)
  MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
  return cudaErrorInvalidValue;
}

// W [E][d] fp32 -> [E][3d] bf16: hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid).  Each
// difference is exact in fp32, so hi + mid + lo carries the weight to within a few units of its
// last fp32 bit; a bf16 x times the split weights, accumulated in fp32 by the tensor cores, is an
// fp32-faithful router GEMM.
__global__ void split_router_weights_kernel(const float* __restrict__ W, int E, int d,
                                            __nv_bfloat16* __restrict__ out) {
  const int64_t n = (int64_t)E * d;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / d;
    const int64_t c = i - e * d;
    const float w = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    __nv_bfloat16* row = out + e * 3 * d;
    row[c] = hi;
    row[d + c] = mid;
    row[2 * d + c] = lo;
  }
}

cudaError_t launch_split_router_weights(const float* W_r, int E, int d, __nv_bfloat16* out,
                                        cudaStream_t st) {
  const int64_t n = (int64_t)E * d;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  LaunchScope ls("split_router_weights", st);
  split_router_weights_kernel<<<blocks, 256, 0, st>>>(W_r, E, d, out);
  return cudaGetLastError();
}

}  // namespace moe
