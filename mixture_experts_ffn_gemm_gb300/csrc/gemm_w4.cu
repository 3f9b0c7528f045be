// gemm_w4.cu -- grouped expert GEMMs with 4-bit integer group-quantised weights and bf16
// activations, on tcgen05 (kind::f16), fp32 accumulation in TMEM.
//
// The nnterp "kimi_k2" page lists "4-bit integer groups (compressed-tensors)" as the weight storage
// of K2-Thinking and the K2.5 line.  Format (include/moe.h): per weight row, K/2 bytes of packed
// excess-8 nibbles and one bf16 scale per 32 input channels (stored [K/32][rows]); the weight is
// RN_bf16((u - 8) * scale), rounded once as the MMA operand.
//
// Orientation: swap-AB as in the bf16 kernel's decode tiles -- M = 128 weight rows (the features
// of one tile), N = the tile's tokens (at most 32, rounded up to 16).  Decode streams the weights,
// so the weight bytes (0.5 B + 1/16 B per weight instead of 2 B) bound the layer.
//
// Kernel shape: persistent, one CTA per SM, 320 threads:
//   warp 0      TMA producer: per K-block (64 input channels) the packed boxes (128 rows x 32 B)
//               and scale boxes (2 groups x 128 rows) of the tile's weight rows (W1 and W3 for
//               SwiGLU) and the token box (32 rows x 128 B), into one stage, on full[s];
//   warps 2..5  converters: thread = weight row; expand its 64 codes per box to bf16 with one
//               mask-and-OR per pair of codes ((0x4300 | u) is the bf16 of 128 + u), a bf16x2
//               subtract of 136 and a bf16x2 multiply by the scale, and store them in the
//               stage's 128-byte-swizzled A tile; fence the async proxy, arrive on conv[s];
//   warp 1      MMA issuer: tcgen05.mma (A = the converted tile, B = the tokens) into one of two
//               TMEM accumulators (W1 and W3 side by side for SwiGLU), frees the stage;
//   warps 6..9  epilogue (TMEM lane quarters): SwiGLU -> bf16 h, or a plain fp32 store.
// Every wait is bounded as in the other kernels.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

constexpr int kW4Conv = 8;                            // converter warps
constexpr int kW4Threads = 32 * (2 + kW4Conv + 4);    // producer, MMA, converters, epilogue
constexpr int kW4BK = 64;                  // input channels per stage
constexpr int kW4BN = 32;                  // tokens per tile
constexpr int kW4ABox = 128 * 128;         // converted bf16 A tile: 128 rows x 128 bytes
constexpr int kW4PackBox = 128 * 32;       // packed codes: 128 rows x 32 bytes
constexpr int kW4ScaleBox = 2 * 128 * 2;   // 2 groups x 128 rows of bf16 scales
constexpr int kW4TokBox = kW4BN * 128;     // 32 token rows x 128 bytes
constexpr int kW4MaxGroups = 1025;
constexpr int kW4SmemLimit = 232448;

// Two rings: copy stages (tokens, packed codes, scales: what the TMA brings, small, so that several
// are in flight while the weights stream from HBM) and converted stages (the bf16 A tiles and a
// copy of the tokens: what the MMA reads; enough of them to cover the converter -> MMA -> release
// round trip).
template <bool kSwiGLU>
struct W4Shape {
  static constexpr int NW = kSwiGLU ? 2 : 1;  // weight boxes per K-block
  static constexpr int P_TOK = 0;
  static constexpr int P_PACK = kW4TokBox;
  static constexpr int P_SCALE = P_PACK + NW * kW4PackBox;
  static constexpr int PSTAGE = (P_SCALE + NW * kW4ScaleBox + 1023) & ~1023;
  static constexpr int TX = kW4TokBox + NW * (kW4PackBox + kW4ScaleBox);  // TMA bytes per stage
  static constexpr int C_TOK = NW * kW4ABox;
  static constexpr int CSTAGE = C_TOK + kW4TokBox;
  static constexpr int CSTAGES = kSwiGLU ? 4 : 6;
  static constexpr int ACC_COLS = NW * kW4BN;
  static constexpr int TMEM_COLS = 2 * ACC_COLS <= 64 ? 64 : 128;
  static constexpr int TABLE_BYTES = 2 * (kW4MaxGroups + 1) * 4 + kW4Threads * 4;
  static constexpr int BAR_BYTES = 256 + 64;
  static constexpr int PSTAGES_FIT =
      (kW4SmemLimit - 1024 - BAR_BYTES - TABLE_BYTES - CSTAGES * CSTAGE) / PSTAGE;
  static constexpr int PSTAGES_MAX = kSwiGLU ? 5 : 7;
  static constexpr int PSTAGES = PSTAGES_FIT > PSTAGES_MAX ? PSTAGES_MAX : PSTAGES_FIT;
  static constexpr int RINGS = CSTAGES * CSTAGE + PSTAGES * PSTAGE;
  static constexpr int SMEM = 1024 + RINGS + BAR_BYTES + TABLE_BYTES;
  static_assert(PSTAGES >= 4, "not enough shared memory for the copy ring");
  static_assert(SMEM <= kW4SmemLimit, "shared memory");
  static_assert(2 * PSTAGES + 2 * CSTAGES + 5 <= 32, "barrier area too small");
  static_assert(CSTAGE % 1024 == 0 && PSTAGE % 1024 == 0 && P_SCALE % 128 == 0,
                "TMA and MMA operands misaligned");
};

struct W4Params {
  CUtensorMap map_act, map_act_d;  // tokens, bf16 [rows][K], box {64, 32}, 128-byte swizzle
  CUtensorMap map_wq, map_wq_d;    // packed codes, uint8 [w_rows][K/2], box {32, 128}
  CUtensorMap map_ws, map_ws_d;    // scales, bf16: routed [E * K/32][w_group_rows] (each expert's
                                   // [K/32][rows] in turn), dense [K/32][w_d_rows]; box {128, 2}
  const int32_t* offsets;
  int32_t n_routed, w_group_rows, u_off, u_off_d;
  int32_t dense_rows, dense_act_row0, dense_out_row0;
  int32_t K, F;
  void* out;  // SwiGLU: bf16 h [rows][ldo]; store: fp32 [rows][ldo]
  int64_t ldo;
  uint32_t* err;
};

// Four bf16 pairs (one 16-byte chunk: input channels 8i .. 8i+7) from one packed word.
__device__ __forceinline__ uint4 w4_expand_word(uint32_t w, __nv_bfloat162 s2) {
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
  uint32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t bits = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;  // bf16(128 + u) pair
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&bits);
    v = __hmul2(__hsub2(v, off), s2);  // (u - 8) exact, then one rounding of the product
    r[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

template <bool kSwiGLU>
__global__ void __launch_bounds__(kW4Threads, 1) moe_gemm_w4_kernel(const __grid_constant__ W4Params p) {
  using S = W4Shape<kSwiGLU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* cring = smem;                             // [CSTAGES][CSTAGE]
  uint8_t* pring = smem + S::CSTAGES * S::CSTAGE;    // [PSTAGES][PSTAGE]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::RINGS);
  uint64_t* pfull = bars;
  uint64_t* pempty = pfull + S::PSTAGES;
  uint64_t* cfull = pempty + S::PSTAGES;
  uint64_t* cempty = cfull + S::CSTAGES;
  uint64_t* tfull = cempty + S::CSTAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* tile_start = reinterpret_cast<int*>(smem + S::RINGS + S::BAR_BYTES);
  int* row_start = tile_start + (kW4MaxGroups + 1);
  int* scratch = row_start + (kW4MaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::PSTAGES; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], kW4Conv);  // one arrival per converter warp
    }
    for (int s = 0; s < S::CSTAGES; ++s) {
      mbar_init(&cfull[s], kW4Conv);
      mbar_init(&cempty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_act);
    tma_prefetch_map(&p.map_wq);
    tma_prefetch_map(&p.map_ws);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, S::TMEM_COLS);
    tmem_relinquish();
  }
  build_tile_table(tile_start, row_start, scratch, p.offsets, p.n_routed, p.dense_rows, kW4BN,
                   p.F / 128);  // ends with __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int G = p.n_routed + (p.dense_rows > 0 ? 1 : 0);
  const int total = tile_start[G];
  const int nkb = p.K / kW4BK;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      int armed = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                        p.dense_rows, p.dense_act_row0, kW4BN);
        const CUtensorMap* ma = ti.dense ? &p.map_act_d : &p.map_act;
        const CUtensorMap* mq = ti.dense ? &p.map_wq_d : &p.map_wq;
        const CUtensorMap* ms = ti.dense ? &p.map_ws_d : &p.map_ws;
        const int act_y = ti.grp_row0 + ti.rt * kW4BN;
        const int w_local = ti.ft * 128;  // the tile's first row within its group's weights
        const int w_y = (ti.dense ? 0 : ti.g * p.w_group_rows) + w_local;
        const int s_y = ti.dense ? 0 : ti.g * (p.K / 32);  // the group's first scale row
        const int u_off = ti.dense ? p.u_off_d : p.u_off;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&pempty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* st = pring + stage * S::PSTAGE;
          mbar_arrive_expect_tx(&pfull[stage], S::TX);
          tma_load_2d(st + S::P_TOK, ma, &pfull[stage], kb * kW4BK, act_y);
#pragma unroll
          for (int j = 0; j < S::NW; ++j) {
            tma_load_2d(st + S::P_PACK + j * kW4PackBox, mq, &pfull[stage], kb * (kW4BK / 2),
                        w_y + j * u_off);
            tma_load_2d(st + S::P_SCALE + j * kW4ScaleBox, ms, &pfull[stage], w_local + j * u_off,
                        s_y + kb * 2);
          }
          if (armed < S::PSTAGES) ++armed;
          if (++stage == S::PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // wait (briefly) for the copies still in flight before leaving
        for (int i = 0; i < armed; ++i) {
          if (stage == 0) {
            stage = S::PSTAGES;
            phase ^= 1u;
          }
          --stage;
          mbar_wait(&pfull[stage], phase, nullptr, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + kW4Conv) {
    // ---------------------------------------------------------------- converters
    const int ct = (warp - 2) * 32 + lane;  // 0 .. 255
    uint32_t ps = 0, pph = 0, cs = 0, cph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb) {
        int w_ok = 1;
        if (lane == 0)
          w_ok = (mbar_wait(&pfull[ps], pph, abort_flag, p.err) &&
                  mbar_wait(&cempty[cs], cph ^ 1u, abort_flag, p.err)) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        const uint8_t* src = pring + ps * S::PSTAGE;
        uint8_t* dst = cring + cs * S::CSTAGE;
        // units (box j, scale group g, row): lanes take consecutive rows
#pragma unroll
        for (int u = ct; u < S::NW * 256; u += 256) {
          const int j = u >> 8, g = (u >> 7) & 1, row = u & 127;
          const uint4 q = *reinterpret_cast<const uint4*>(src + S::P_PACK + j * kW4PackBox +
                                                          row * 32 + g * 16);
          const __nv_bfloat16 sc = *reinterpret_cast<const __nv_bfloat16*>(
              src + S::P_SCALE + j * kW4ScaleBox + (g * 128 + row) * 2);
          const __nv_bfloat162 s2 = __bfloat162bfloat162(sc);
          const uint32_t words[4] = {q.x, q.y, q.z, q.w};
          uint8_t* a_row = dst + j * kW4ABox + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int chunk = g * 4 + i;  // 16-byte chunk of the 128-byte row
            *reinterpret_cast<uint4*>(a_row + ((chunk ^ (row & 7)) << 4)) =
                w4_expand_word(words[i], s2);
          }
        }
        // the token box moves as is (both stages are 1024-byte aligned: the swizzle is kept)
        reinterpret_cast<uint4*>(dst + S::C_TOK)[ct] =
            reinterpret_cast<const uint4*>(src + S::P_TOK)[ct];
        // the tensor core reads the converted stage through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&cfull[cs]);
          mbar_arrive(&pempty[ps]);
        }
        if (++ps == S::PSTAGES) {
          ps = 0;
          pph ^= 1u;
        }
        if (++cs == S::CSTAGES) {
          cs = 0;
          cph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      uint32_t cs = 0, cph = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                        p.dense_rows, p.dense_act_row0, kW4BN);
        const int n = ti.valid >= kW4BN ? kW4BN : ((ti.valid + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32_n(n);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * S::ACC_COLS;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&cfull[cs], cph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(cring + cs * S::CSTAGE);
#pragma unroll
          for (int k16 = 0; k16 < kW4BK / 16; ++k16) {
            const uint32_t accum = (kb | k16) != 0;
            const uint64_t bdesc = sw128_kmajor_desc(st + S::C_TOK + k16 * 32);
#pragma unroll
            for (int j = 0; j < S::NW; ++j)
              mma_bf16(d0 + j * kW4BN, sw128_kmajor_desc(st + j * kW4ABox + k16 * 32), bdesc,
                       idesc, accum);
          }
          mma_commit(&cempty[cs]);
          if (++cs == S::CSTAGES) {
            cs = 0;
            cph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, nullptr, kDrainLimitNs);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (4 warps)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                      p.dense_rows, p.dense_act_row0, kW4BN);
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err) ? 1 : 0;
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!w_ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * S::ACC_COLS + ((uint32_t)(quarter * 32) << 16);
      const int64_t out_row0 = (ti.dense ? (int64_t)p.dense_out_row0 : (int64_t)ti.grp_row0) +
                               (int64_t)ti.rt * kW4BN;
      const int64_t feat = (int64_t)ti.ft * 128 + r;
#pragma unroll 1
      for (int c = 0; c < kW4BN && c < ti.valid; c += 16) {
        uint32_t gv[16], uv[16];
        tmem_ld16(tb + c, gv);
        if (kSwiGLU) tmem_ld16(tb + kW4BN + c, uv);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (c + i < ti.valid) {
            const int64_t orow = out_row0 + c + i;
            if (kSwiGLU) {
              const float h = silu_fast(__uint_as_float(gv[i])) * __uint_as_float(uv[i]);
              ((__nv_bfloat16*)p.out)[orow * p.ldo + feat] = __float2bfloat16_rn(h);
            } else {
              ((float*)p.out)[orow * p.ldo + feat] = __uint_as_float(gv[i]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFnW4)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnW4 encode_fn_w4() {
  static EncodeTiledFnW4 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnW4>(ptr);
  });
  return fn;
}

// 2D map over [outer][inner] elements with a dense row pitch, box {box_in, box_out}, zero fill.
static bool make_map_w4(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base,
                        int64_t outer, int64_t inner, int box_in, int box_out,
                        CUtensorMapSwizzle swz) {
  EncodeTiledFnW4 enc = encode_fn_w4();
  if (!enc || !base || outer <= 0 || inner <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(inner * esize)};
  cuuint32_t box[2] = {(cuuint32_t)box_in, (cuuint32_t)box_out};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// groups: the weight groups the scales come in (n experts each [K/32][rows_per_group]).
static bool w4_maps(CUtensorMap* act, CUtensorMap* wq, CUtensorMap* ws, const void* a,
                    int64_t a_rows, const void* q, const void* s, int64_t groups,
                    int64_t rows_per_group, int K) {
  return make_map_w4(act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a, a_rows, K, kW4BK, kW4BN,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_w4(wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q, groups * rows_per_group, K / 2,
                     kW4BK / 2, 128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         make_map_w4(ws, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s, groups * (K / 32), rows_per_group,
                     128, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <bool kSwiGLU>
static cudaError_t launch_w4_variant(const W4Params& p, int grid, cudaStream_t st,
                                     const char* label) {
  using S = W4Shape<kSwiGLU>;
  auto kern = moe_gemm_w4_kernel<kSwiGLU>;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  LaunchScope ls(label, st);
  kern<<<grid, kW4Threads, S::SMEM, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_w4(const W4Gemm& g, int num_sms, cudaStream_t st) {
  if (g.K % kW4BK || g.F % 128 || g.n_routed > kW4MaxGroups - 1) return cudaErrorInvalidValue;
  if (g.w_group_rows % 128 || g.ldo % 8) return cudaErrorInvalidValue;
  W4Params p;
  memset(&p, 0, sizeof(p));
  if (g.n_routed > 0 && (g.w_rows != (int64_t)g.n_routed * g.w_group_rows ||
                         !w4_maps(&p.map_act, &p.map_wq, &p.map_ws, g.act, g.act_rows, g.wq, g.ws,
                                  g.n_routed, g.w_group_rows, g.K)))
    return cudaErrorInvalidValue;
  if (g.dense_rows > 0 && !w4_maps(&p.map_act_d, &p.map_wq_d, &p.map_ws_d, g.act_d, g.act_d_rows,
                                   g.wq_d, g.ws_d, 1, g.w_d_rows, g.K))
    return cudaErrorInvalidValue;
  if (g.n_routed == 0) {  // keep the unused maps valid objects
    p.map_act = p.map_act_d;
    p.map_wq = p.map_wq_d;
    p.map_ws = p.map_ws_d;
  }
  if (g.dense_rows == 0) {
    p.map_act_d = p.map_act;
    p.map_wq_d = p.map_wq;
    p.map_ws_d = p.map_ws;
  }
  p.offsets = g.offsets;
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
  p.err = g.err;
  if (g.swiglu) return launch_w4_variant<true>(p, num_sms, st, g.label);
  return launch_w4_variant<false>(p, num_sms, st, g.label);
}

}  // namespace moe
