// router_tc.cu -- router logits for small batches on the tensor cores, split over K.
//
// "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts": z = W_r x with
// fp32 logits (nnterp "kimi_k2": the gate's weight is kept in fp32).  x is bf16, W_r fp32.  Each
// fp32 weight is split into three bf16 parts, hi = bf16(w), mid = bf16(w - hi), lo =
// bf16(w - hi - mid) (each difference exact in fp32), and the tensor cores accumulate x * hi +
// x * mid + x * lo in fp32: an fp32-faithful product of the bf16 activations and the fp32 weights.
//
// A batch of a few hundred tokens gives too few 128-token tiles to fill the GPU, so the K range
// is split into S slices and every CTA takes one (token tile, 64-expert block, K slice); the slices'
// partial logits go to S separate buffers, which the selection kernel sums in slice order (the
// result does not depend on scheduling).  The weights are split inside the kernel, so no split
// copy of W_r has to be written per call:
//   warp 0       TMA producer of the token tile's bf16 activations (one 128 x 64 box per K-block);
//   warps 1..4   converters: each thread loads 32 consecutive fp32 weights of one expert row,
//                splits them and writes the three parts into the stage's 128-byte-swizzled
//                K-major operands (the layout TMA would produce), then the epilogue: TMEM lane
//                quarter (warp % 4) holds tokens 32 (warp % 4) .. +31;
//   warp 5       MMA issuer: per K-block 4 K-steps x 3 parts of M = 128 tokens, N = 64 experts.
// Every wait is bounded as in the other kernels.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kRtThreads = 192;
constexpr int kRtStages = 3;
constexpr int kRtXBox = 128 * 128;           // 128 tokens x 64 bf16
constexpr int kRtPart = 64 * 128;            // 64 experts x 64 bf16
constexpr int kRtWStage = 3 * kRtPart;       // hi, mid, lo
constexpr int kRtSmem = 1024 + kRtStages * (kRtXBox + kRtWStage) + 256;

struct RtParams {
  CUtensorMap map_x;   // bf16 [T][d], box {64, 128}, 128-byte swizzle
  const float* W_r;    // fp32 [E][d]
  float* z;            // partial logits: slice s at z + s * split_stride, [T][E]
  int64_t split_stride;
  int T, E, d, S, eblocks, nkb;  // nkb: K-blocks per slice
  uint32_t* err;
};

// Splits four fp32 weights into their bf16 hi / mid / lo parts, two bf16 per 32-bit word.
__device__ __forceinline__ void split3(const float4 w, uint2& hi, uint2& mid, uint2& lo) {
  const float v[4] = {w.x, w.y, w.z, w.w};
  uint32_t h[4], m[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat16 bh = __float2bfloat16_rn(v[i]);
    const float r1 = v[i] - __bfloat162float(bh);
    const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(bm);
    const __nv_bfloat16 bl = __float2bfloat16_rn(r2);
    h[i] = __bfloat16_as_ushort(bh);
    m[i] = __bfloat16_as_ushort(bm);
    l[i] = __bfloat16_as_ushort(bl);
  }
  hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  mid = make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
  lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_splitk_tc_kernel(const __grid_constant__ RtParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* xs = smem;                                 // [stage] 16 KB
  uint8_t* wsm = smem + kRtStages * kRtXBox;          // [stage][part] 8 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(wsm + kRtStages * kRtWStage);
  uint64_t* xfull = bars;
  uint64_t* xempty = bars + kRtStages;
  uint64_t* wfull = bars + 2 * kRtStages;
  uint64_t* wempty = bars + 3 * kRtStages;
  uint64_t* accfull = bars + 4 * kRtStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 4 * kRtStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x % p.S;
  const int rest = blockIdx.x / p.S;
  const int eb = rest % p.eblocks;
  const int tt = rest / p.eblocks;
  const int kb0 = s * p.nkb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRtStages; ++i) {
      mbar_init(&xfull[i], 1);
      mbar_init(&xempty[i], 1);
      mbar_init(&wfull[i], 128);
      mbar_init(&wempty[i], 1);
    }
    mbar_init(accfull, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_map(&p.map_x);
  if (warp == 5) {
    tmem_alloc(tmem_holder, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ activations (TMA)
    if (lane == 0) {
      for (int i = 0; i < p.nkb; ++i) {
        const int st = i % kRtStages;
        if (!mbar_wait(&xempty[st], ((i / kRtStages) & 1) ^ 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&xfull[st], kRtXBox);
        tma_load_2d(xs + st * kRtXBox, &p.map_x, &xfull[st], (kb0 + i) * 64, tt * 128);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32<128, 64>();
      bool ok = true;
      for (int i = 0; i < p.nkb && ok; ++i) {
        const int st = i % kRtStages;
        const uint32_t ph = (i / kRtStages) & 1;
        if (!mbar_wait(&xfull[st], ph, abort_flag, p.err) ||
            !mbar_wait(&wfull[st], ph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xa = smem_u32(xs + st * kRtXBox);
        const uint32_t wa = smem_u32(wsm + st * kRtWStage);
#pragma unroll
        for (int k16 = 0; k16 < 4; ++k16)
#pragma unroll
          for (int part = 0; part < 3; ++part)
            mma_bf16(tmem, sw128_kmajor_desc(xa + k16 * 32),
                     sw128_kmajor_desc(wa + part * kRtPart + k16 * 32), kIdesc,
                     (i | k16 | part) != 0);
        mma_commit(&xempty[st]);
        mma_commit(&wempty[st]);
      }
      if (ok) mma_commit(accfull);
    }
  } else {
    // ------------------------------------------------------------ converters, then epilogue
    const int t = threadIdx.x - 32;          // 0..127
    const int e = t >> 1;                    // expert row of the block
    const int kh = (t & 1) * 32;             // first of this thread's 32 channels in the K-block
    const int64_t erow = (int64_t)eb * 64 + e;
    const float* wrow = p.W_r + erow * p.d + (int64_t)kb0 * 64 + kh;
    // the slice's later K-blocks of this row are pulled into L2 now (one 128-byte line per
    // K-block), so that the loads below wait on L2 rather than DRAM
    for (int i = 1; i < p.nkb; ++i)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(wrow + i * 64));
    float4 cur[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = __ldg(reinterpret_cast<const float4*>(wrow) + j);
    bool ok = true;
    for (int i = 0; i < p.nkb; ++i) {
      const int st = i % kRtStages;
      float4 nxt[8];
      if (i + 1 < p.nkb) {  // the next K-block's weights are in flight while this one is split
#pragma unroll
        for (int j = 0; j < 8; ++j)
          nxt[j] = __ldg(reinterpret_cast<const float4*>(wrow + (i + 1) * 64) + j);
      }
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&wempty[st], ((i / kRtStages) & 1) ^ 1, abort_flag, p.err);
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!w_ok) {
        ok = false;
        break;
      }
      uint8_t* base = wsm + st * kRtWStage + e * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16-byte chunk (kh / 8 + c) of the row: 8 channels
        uint2 h0, m0, l0, h1, m1, l1;
        split3(cur[2 * c], h0, m0, l0);
        split3(cur[2 * c + 1], h1, m1, l1);
        const int off = (((kh >> 3) + c) ^ (e & 7)) << 4;
        *reinterpret_cast<uint4*>(base + off) = make_uint4(h0.x, h0.y, h1.x, h1.y);
        *reinterpret_cast<uint4*>(base + kRtPart + off) = make_uint4(m0.x, m0.y, m1.x, m1.y);
        *reinterpret_cast<uint4*>(base + 2 * kRtPart + off) = make_uint4(l0.x, l0.y, l1.x, l1.y);
      }
      // the generic-proxy stores become visible to the tensor core's reads
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&wfull[st]);
      if (i + 1 < p.nkb) {
#pragma unroll
        for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
      }
    }
    // epilogue: tokens on TMEM lanes, the block's 64 experts on columns
    const int quarter = warp & 3;
    int a_ok = 0;
    if (ok) {
      if (lane == 0) a_ok = mbar_wait(accfull, 0, abort_flag, p.err) ? 1 : 0;
      a_ok = __shfl_sync(0xffffffffu, a_ok, 0);
    }
    if (a_ok) {
      tc_fence_after();
      const int row = tt * 128 + quarter * 32 + lane;
      float* dst = p.z + (int64_t)s * p.split_stride + (int64_t)row * p.E + (int64_t)eb * 64;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + c, v);
        tmem_ld_wait();
        if (row < p.T) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(dst + c + 4 * q) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

bool router_splitk_tc_supported(int64_t T, int E, int d) {
  return T > 0 && T <= (int64_t)1 << 20 && E % 64 == 0 && d % 64 == 0 && E <= 4096;
}

// Slices of K for T tokens: the largest divisor of d / 64 that keeps one wave of CTAs.
int router_splitk_tc_slices(int64_t T, int E, int d, int num_sms) {
  const int64_t tiles = ((T + 127) / 128) * (E / 64);
  const int nkb = d / 64;
  int best = 1;
  for (int s = 1; s <= nkb; ++s)
    if (nkb % s == 0 && tiles * s <= num_sms) best = s;
  return best;
}

cudaError_t launch_router_splitk_tc(const void* x, const float* W_r, int64_t T, int E, int d,
                                    int S, float* z, int64_t split_stride, uint32_t* err,
                                    cudaStream_t st) {
  if (!router_splitk_tc_supported(T, E, d) || S <= 0 || (d / 64) % S) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(W_r) & 15) || (reinterpret_cast<uintptr_t>(z) & 15))
    return cudaErrorInvalidValue;
  RtParams p;
  memset(&p, 0, sizeof(p));
  if (!make_map_bf16(&p.map_x, x, T, d, 128)) return cudaErrorInvalidValue;
  p.W_r = W_r;
  p.z = z;
  p.split_stride = split_stride;
  p.T = (int)T;
  p.E = E;
  p.d = d;
  p.S = S;
  p.eblocks = E / 64;
  p.nkb = d / 64 / S;
  p.err = err;
  static int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(router_splitk_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  const int64_t blocks = ((T + 127) / 128) * p.eblocks * S;
  LaunchScope ls("router_gemm_tc_splitk", st);
  router_splitk_tc_kernel<<<(unsigned)blocks, kRtThreads, kRtSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
