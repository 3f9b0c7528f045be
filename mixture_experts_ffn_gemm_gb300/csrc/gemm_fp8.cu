// gemm_fp8.cu -- grouped expert GEMMs with e4m3 operands and per-block scales, on tcgen05
// (kind::f8f6f4), fp32 accumulation.
//
// Expert weights are e4m3 with one fp32 scale per 128 x 128 block (the nnterp "kimi_k2" note:
// the K2 checkpoints store "FP8 blocks"); activations are e4m3 with one fp32 scale per row per 128
// channels.  The value of one output is
//     y[r][f] = sum_kb  sx[r][kb] * sw[f/128][kb] * sum_{k in block kb} qx[r][k] * qw[f][k],
// so every 128-wide K-block is a separate MMA product that is scaled and added in fp32.
//
// Kernel shape: persistent, one CTA per SM, 320 threads:
//   warp 0      TMA producer: one K-block (128 e4m3 = one 128-byte swizzle row) per stage;
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) per K-block into one of two
//               TMEM partial buffers (M = 128 rows x N = 256 columns), commit -> partial_full;
//   warps 2..9  epilogue/promotion: two warps per TMEM lane quarter, each owning 128 of the 256
//               columns; per K-block they read the partial, multiply by the row's activation
//               scale times the block's weight scale and add into 128 fp32 registers, then free
//               the buffer, so the MMA of block kb+1 overlaps the promotion of block kb.
// Tiles are token rows (M = 128) x 256 weight rows, as in the bf16 rows orientation:
//   SwiGLU: columns 0..127 are the W1 rows of 128 features, 128..255 the W3 rows of the same
//           features; warp half 0 owns features 0..63 (g and u), half 1 features 64..127.  The
//           epilogue forms h = SiLU(g) * u and quantises it per row per 128 features -- exactly one
//           tile -- to e4m3 with scale amax/448 (the two halves exchange their amax).
//   store:  half 0 owns output features 0..127 (weight block 0), half 1 128..255 (block 1);
//           fp32 output.
// Every wait is bounded as in the bf16 kernel.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

constexpr int kF8Threads = 320;
constexpr int kF8BK = 128;                // e4m3 per K-block = bytes per row of a stage
constexpr int kF8BN = 256;
constexpr int kF8Box = 128 * 128;         // one 128-row x 128-byte box
constexpr int kF8Stage = kF8Box + 2 * kF8Box;
constexpr int kF8MaxGroups = 1025;
constexpr int kF8Table = 2 * (kF8MaxGroups + 1) * 4 + kF8Threads * 4;
constexpr int kF8Bars = 256 + 64;
constexpr int kF8Xchg = 2 * 2 * 128 * 4;  // [tile parity][half][row] amax exchange
constexpr int kF8Stages = 4;
constexpr int kF8Smem = 1024 + kF8Stages * kF8Stage + kF8Bars + kF8Xchg + kF8Table;
static_assert(kF8Smem <= 232448, "fp8 GEMM shared memory");

struct F8Params {
  CUtensorMap map_act, map_w, map_act_d, map_w_d;  // uint8 [rows][K], box {128, 128}
  const int32_t* offsets;
  const float* act_sT;    // routed activation scales [K/128][act_s_ld]
  int64_t act_s_ld;
  const float* act_sT_d;  // dense-group activation scales [K/128][act_s_ld_d]
  int64_t act_s_ld_d;
  const float* w_s;       // routed weight scales [E][w_group_rows/128][K/128]
  const float* w_s_d;     // dense weight scales [rows/128][K/128]
  int32_t n_routed, w_group_rows, u_off, u_off_d;
  int32_t dense_rows, dense_act_row0, dense_out_row0;
  int32_t K, F;
  void* out;              // SwiGLU: e4m3 h [rows][ldo]; store: fp32 [rows][ldo]
  int64_t ldo;
  float* out_sT;          // SwiGLU: h scales [F/128][out_s_ld]
  int64_t out_s_ld;
  uint32_t* err;
};

__device__ __forceinline__ uint32_t e4m3x4_pack(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <bool kSwiGLU>
__global__ void __launch_bounds__(kF8Threads, 1) moe_gemm_fp8_kernel(const __grid_constant__ F8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF8Stages * kF8Stage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kF8Stages;
  uint64_t* pfull = bars + 2 * kF8Stages;
  uint64_t* pempty = pfull + 2;
  uint64_t* drain = pempty + 2;
  uint64_t* xbar = drain + 1;  // [2]: amax exchange between the two epilogue halves
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* xchg = reinterpret_cast<float*>(smem + kF8Stages * kF8Stage + kF8Bars);  // [2][128]
  int* tile_start = reinterpret_cast<int*>(smem + kF8Stages * kF8Stage + kF8Bars + kF8Xchg);
  int* row_start = tile_start + (kF8MaxGroups + 1);
  int* scratch = row_start + (kF8MaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int FPT = kSwiGLU ? 128 : kF8BN;  // output features per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], 256);
    }
    mbar_init(drain, 1);
    mbar_init(&xbar[0], 256);
    mbar_init(&xbar[1], 256);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_act);
    tma_prefetch_map(&p.map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  build_tile_table(tile_start, row_start, scratch, p.offsets, p.n_routed, p.dense_rows, 128,
                   p.F / FPT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int G = p.n_routed + (p.dense_rows > 0 ? 1 : 0);
  const int total = tile_start[G];
  const int nkb = p.K / kF8BK;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      int armed = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                        p.dense_rows, p.dense_act_row0, 128);
        const CUtensorMap* ma = ti.dense ? &p.map_act_d : &p.map_act;
        const CUtensorMap* mw = ti.dense ? &p.map_w_d : &p.map_w;
        const int act_y = ti.grp_row0 + ti.rt * 128;
        const int w_y = (ti.dense ? 0 : ti.g * p.w_group_rows) + ti.ft * FPT;
        const int u_off = ti.dense ? p.u_off_d : p.u_off;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kF8Stage;
          uint8_t* sb = sa + kF8Box;
          mbar_arrive_expect_tx(&full[stage], kF8Stage);
          const int kx = kb * kF8BK;
          tma_load_2d(sa, ma, &full[stage], kx, act_y);
          tma_load_2d(sb, mw, &full[stage], kx, w_y);
          tma_load_2d(sb + kF8Box, mw, &full[stage], kx, kSwiGLU ? w_y + u_off : w_y + 128);
          if (armed < kF8Stages) ++armed;
          if (++stage == kF8Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int i = 0; i < armed; ++i) {
          if (stage == 0) {
            stage = kF8Stages;
            phase ^= 1u;
          }
          --stage;
          mbar_wait(&full[stage], phase, nullptr, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      constexpr uint32_t kIdesc = idesc_e4m3_f32<128, kF8BN>();
      uint32_t stage = 0, phase = 0;
      uint32_t kbg = 0;  // K-blocks issued so far (all tiles): buffer = kbg & 1
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++kbg) {
          const uint32_t buf = kbg & 1u, bph = (kbg >> 1) & 1u;
          if (!mbar_wait(&pempty[buf], bph ^ 1u, abort_flag, p.err) ||
              !mbar_wait(&full[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kF8Stage);
          const uint32_t sb = sa + kF8Box;
          const uint32_t d = tmem_base + buf * kF8BN;
#pragma unroll
          for (int k32 = 0; k32 < kF8BK / 32; ++k32)
            mma_e4m3(d, sw128_kmajor_desc(sa + k32 * 32), sw128_kmajor_desc(sb + k32 * 32), kIdesc,
                     k32 != 0);
          mma_commit(&empty[stage]);
          mma_commit(&pfull[buf]);
          if (++stage == kF8Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, nullptr, kDrainLimitNs);
    }
  } else {
    // ---------------------------------------------------------------- promotion + epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    uint32_t kbg = 0;
    uint32_t it = 0;  // tiles finished by this thread: exchange slot it & 1
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                      p.dense_rows, p.dense_act_row0, 128);
      const bool valid = r < ti.valid;
      const int64_t act_row = (int64_t)ti.grp_row0 + ti.rt * 128 + r;
      const float* sx_col = ti.dense ? p.act_sT_d : p.act_sT;
      const int64_t sx_ld = ti.dense ? p.act_s_ld_d : p.act_s_ld;
      const int wblocks = p.w_group_rows / 128;
      // weight scale rows of the two 128-row halves this warp reads
      const float* ws0;
      const float* ws1;
      if (kSwiGLU) {
        const int u_off = ti.dense ? p.u_off_d : p.u_off;
        const int rb_g = ti.ft, rb_u = (u_off + ti.ft * 128) / 128;
        const float* base = ti.dense ? p.w_s_d : p.w_s + (int64_t)ti.g * wblocks * nkb;
        ws0 = base + (int64_t)rb_g * nkb;
        ws1 = base + (int64_t)rb_u * nkb;
      } else {
        const int rb = ti.ft * 2 + half;
        const float* base = ti.dense ? p.w_s_d : p.w_s + (int64_t)ti.g * wblocks * nkb;
        ws0 = base + (int64_t)rb * nkb;
        ws1 = ws0;
      }
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      // the scales of K-block kb + 1 are loaded while block kb is promoted (their global-memory
      // latency then hides behind the MMA instead of stalling every block)
      const float* sx_ptr = sx_col + act_row;
      float sx_n = valid ? __ldg(sx_ptr) : 0.0f;
      float w0_n = __ldg(ws0), w1_n = __ldg(ws1);
      for (int kb = 0; kb < nkb; ++kb, ++kbg) {
        const float sx = sx_n, w0 = w0_n, w1 = w1_n;
        if (kb + 1 < nkb) {
          sx_n = valid ? __ldg(sx_ptr + (int64_t)(kb + 1) * sx_ld) : 0.0f;
          w0_n = __ldg(ws0 + kb + 1);
          w1_n = __ldg(ws1 + kb + 1);
        }
        const uint32_t buf = kbg & 1u, bph = (kbg >> 1) & 1u;
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&pfull[buf], bph, abort_flag, p.err) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float s0 = sx * w0;
        const float s1 = sx * w1;
        const uint32_t tb = tmem_base + buf * kF8BN + ((uint32_t)(quarter * 32) << 16);
        if (kSwiGLU) {
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t g[16], u[16];
            tmem_ld16(tb + half * 64 + c, g);
            tmem_ld16(tb + 128 + half * 64 + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              fma2(acc[c + i], acc[c + i + 1], s0, g[i], g[i + 1]);
              fma2(acc[64 + c + i], acc[64 + c + i + 1], s1, u[i], u[i + 1]);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; c += 32) {
            uint32_t v0[16], v1[16];
            tmem_ld16(tb + half * 128 + c, v0);
            tmem_ld16(tb + half * 128 + c + 16, v1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              fma2(acc[c + i], acc[c + i + 1], s0, v0[i], v0[i + 1]);
              fma2(acc[c + 16 + i], acc[c + 16 + i + 1], s0, v1[i], v1[i + 1]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&pempty[buf]);
      }
      if (!ok) break;
      const int64_t orow =
          (ti.dense ? (int64_t)p.dense_out_row0 : (int64_t)ti.grp_row0) + ti.rt * 128 + r;
      if (kSwiGLU) {
        // h = SiLU(g) * u for this thread's 64 features, then e4m3 per 128-feature group
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = silu_fast(acc[j]) * acc[64 + j];
          amax = fmaxf(amax, fabsf(acc[j]));
        }
        // exchange with the other half through a double-buffered slot and a bounded mbarrier wait:
        // slot it&1 is rewritten two tiles later, after the partner has passed the barrier of the
        // tile in between, i.e. after it read this one
        float* slot = xchg + (it & 1u) * 256;
        slot[half * 128 + r] = amax;
        mbar_arrive(&xbar[it & 1u]);
        int x_ok = 1;
        if (lane == 0) x_ok = mbar_wait(&xbar[it & 1u], (it >> 1) & 1u, abort_flag, p.err) ? 1 : 0;
        x_ok = __shfl_sync(0xffffffffu, x_ok, 0);
        if (!x_ok) break;
        amax = fmaxf(amax, slot[(half ^ 1) * 128 + r]);
        const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (valid) {
          uint8_t* dst = (uint8_t*)p.out + orow * p.ldo + (int64_t)ti.ft * 128 + half * 64;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int j = v * 16 + q * 4;
              w[q] = e4m3x4_pack(__fdiv_rn(acc[j], scale), __fdiv_rn(acc[j + 1], scale),
                                 __fdiv_rn(acc[j + 2], scale), __fdiv_rn(acc[j + 3], scale));
            }
            reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (half == 0) p.out_sT[(int64_t)ti.ft * p.out_s_ld + orow] = scale;
        }
      } else if (valid) {
        float* dst = (float*)p.out + orow * p.ldo + (int64_t)ti.ft * kF8BN + half * 128;
#pragma unroll
        for (int j = 0; j < 128; j += 4)
          reinterpret_cast<float4*>(dst)[j / 4] = make_float4(acc[j], acc[j + 1], acc[j + 2],
                                                              acc[j + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFnF8)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnF8 encode_fn_f8() {
  static EncodeTiledFnF8 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnF8>(ptr);
  });
  return fn;
}

// 2D uint8 map over [rows][cols], box {128 bytes, 128 rows}, 128-byte swizzle, zero fill.
static bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFnF8 enc = encode_fn_f8();
  if (!enc || !base || rows <= 0 || cols <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <bool kSwiGLU>
static cudaError_t launch_f8_variant(const F8Params& p, int grid, cudaStream_t st,
                                     const char* label) {
  auto kern = moe_gemm_fp8_kernel<kSwiGLU>;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  LaunchScope ls(label, st);
  kern<<<grid, kF8Threads, kF8Smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp8(const Fp8Gemm& g, int num_sms, cudaStream_t st) {
  if (g.K % kF8BK || g.n_routed > kF8MaxGroups - 1) return cudaErrorInvalidValue;
  if (g.swiglu ? g.F % 128 : g.F % kF8BN) return cudaErrorInvalidValue;
  if (g.w_group_rows % 128 || g.ldo % 16) return cudaErrorInvalidValue;
  F8Params p;
  memset(&p, 0, sizeof(p));
  if (g.n_routed > 0) {
    if (!make_map_u8(&p.map_act, g.act, g.act_rows, g.K)) return cudaErrorInvalidValue;
    if (!make_map_u8(&p.map_w, g.w, g.w_rows, g.K)) return cudaErrorInvalidValue;
  }
  if (g.dense_rows > 0) {
    if (!make_map_u8(&p.map_act_d, g.act_d, g.act_d_rows, g.K)) return cudaErrorInvalidValue;
    if (!make_map_u8(&p.map_w_d, g.w_d, g.w_d_rows, g.K)) return cudaErrorInvalidValue;
  }
  if (g.n_routed == 0) {
    p.map_act = p.map_act_d;
    p.map_w = p.map_w_d;
  }
  if (g.dense_rows == 0) {
    p.map_act_d = p.map_act;
    p.map_w_d = p.map_w;
  }
  p.offsets = g.offsets;
  p.act_sT = g.act_sT;
  p.act_s_ld = g.act_s_ld;
  p.act_sT_d = g.act_sT_d;
  p.act_s_ld_d = g.act_s_ld_d;
  p.w_s = g.w_s;
  p.w_s_d = g.w_s_d;
  p.n_routed = g.n_routed;
  p.w_group_rows = g.w_group_rows;
  p.u_off = g.u_off;
  p.u_off_d = g.u_off_d;
  p.dense_rows = g.dense_rows;
  p.dense_act_row0 = g.dense_act_row0;
  p.dense_out_row0 = g.dense_out_row0;
  p.K = g.K;
  p.F = g.F;
  p.out = g.out;
  p.ldo = g.ldo;
  p.out_sT = g.out_sT;
  p.out_s_ld = g.out_s_ld;
  p.err = g.err;
  if (g.swiglu) return launch_f8_variant<true>(p, num_sms, st, g.label);
  return launch_f8_variant<false>(p, num_sms, st, g.label);
}

}  // namespace moe
