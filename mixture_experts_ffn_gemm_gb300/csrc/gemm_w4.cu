// gemm_w4.cu -- grouped expert GEMMs with 4-bit integer group-quantised weights and bf16
// activations, on tcgen05 (kind::f16), fp32 accumulation in TMEM.
//
// The nnterp "kimi_k2" page lists "4-bit integer groups (compressed-tensors)" as the weight storage
// of K2-Thinking and the K2.5 line.  Format (include/moe.h): per weight row, K/2 bytes of packed
// excess-8 nibbles and one bf16 scale per 32 input channels (stored [K/32][rows]); the weight is
// RN_bf16((u - 8) * scale), rounded once as the MMA operand.
//
// Orientation: swap-AB as in the bf16 kernel's decode tiles -- M = 128 weight rows per MMA, N = the
// tile's tokens (at most 32, rounded up to 16).  Decode streams the weights, so the weight bytes
// (0.5 B + 1/16 B per weight instead of 2 B) bound the layer, and everything per input channel
// has to run four times faster than in the bf16 kernel:
//   * copies: a TMA engine finishes only a few boxes at a time, so a small box costs about as much
//     as a large one.  One copy stage covers 256 input channels with three boxes: the packed codes
//     of two 128-row blocks (128 B a row, 32 KB), their scales (8 groups, 4 KB) and the tokens
//     (4 chunks of 32 rows x 64 channels, 16 KB, each chunk in the MMA's 128-byte swizzled layout);
//   * the expanded weights never touch shared memory: a converter thread owns one weight row,
//     expands 64 codes into 32 bf16 pairs in registers and writes them to TMEM with one tcgen05.st;
//     the MMA takes A from TMEM (row m on lane m, two bf16 per 32-bit column).
//   * the MMA floor: an M = 128, K = 16 MMA with N <= 32 costs a fixed ~45 cycles, so 32 MMAs per
//     copy stage stay just under the stage's HBM time -- but only with two issuing warps: one
//     thread that waits on an mbarrier (or touches shared memory at all) between groups of MMAs
//     lets the tensor pipe drain and runs at ~90 cycles per MMA.  The two issuers take alternate
//     64-channel sub-blocks into their own accumulators (split K); the epilogue adds the halves.
// Blocks: SwiGLU tiles pair 128 W1 rows with the matching 128 W3 rows (h = SiLU(W1 x) * W3 x for
// 128 features); store tiles take 256 consecutive rows as two blocks (two accumulators).
//
// Kernel shape: persistent, one CTA per SM, 736 threads (23 warps):
//   warp 0       TMA producer, copy ring (pfull / pempty);
//   warps 2..17  converters in two groups: group g = (w - 2) / 8 expands the sub-blocks of parity
//                g (those MMA issuer g takes), block ((w - 2) / 4) % 2, and writes TMEM lanes
//                32 (w % 4) .. +31 (thread = weight row).  Per copy stage a warp reads its row's
//                codes and scales of its two sub-blocks before any tcgen05 operation (a shared-
//                memory read behind outstanding tcgen05 work stalls), releases the stage, then
//                fills its group's TMEM sub-stage with both (cfull / cempty).  Per pair of codes: one
//                mask-and-OR ((0x4300 | u) is the bf16 of 128 + u), a bf16x2 subtract of 136 and a
//                bf16x2 multiply by the scale;
//   warps 1, 22  MMA issuers i = 0, 1: the tile's sub-blocks of parity i (4 K-steps x 2 blocks
//                each) into accumulator half i; their commits free the TMEM sub-stage and, with
//                the converters, the copy stage;
//   warps 18..21 epilogue (TMEM lane quarters): reads and adds the two halves, frees the
//                accumulator at once, then SwiGLU -> bf16 h, or plain fp32 stores.
// TMEM columns: [0, 128) the accumulator [issuer][block] x 32 columns (one buffer: the epilogue
// holds it only for its reads), then 3 sub-stages of [block][sub-block] x 32 columns.  Per copy
// stage each converter group fills one sub-stage with both of its 64-channel sub-blocks (one wait,
// two TMEM stores, one release), and the two groups take the three sub-stages in turn (the group's
// u-th use, u = 2 * copy stage + group, is sub-stage u % 3).
// Every wait is bounded as in the other kernels.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

constexpr int kW4Conv = 16;                         // converter warps: 2 groups x 2 blocks x 4
constexpr int kW4Threads = 32 * (3 + kW4Conv + 4);  // producer, 2 MMA, converters, epilogue
constexpr int kW4Mma1Warp = 2 + kW4Conv + 4;        // the second MMA issuer (the last warp)
constexpr int kW4BK = 256;                 // input channels per copy stage
constexpr int kW4Sub = 64;                 // input channels per TMEM sub-stage
constexpr int kW4BN = 32;                  // tokens per tile
constexpr int kW4ACols = kW4Sub / 2;       // TMEM columns of one block's sub-stage (bf16 pairs)
constexpr int kW4TokChunk = kW4BN * 128;   // 32 token rows x 128 bytes
constexpr int kW4PackBlock = 128 * 128;    // 128 rows x 128 code bytes
constexpr int kW4ScaleBlock = 8 * 128 * 2; // 8 groups x 128 rows of bf16 scales
constexpr int kW4MaxGroups = 1025;
constexpr int kW4SmemLimit = 232448;
constexpr int kW4TmemCols = 512;

struct W4Shape {
  static constexpr int P_TOK = 0;                           // [4 chunks][32 rows][128 B]
  static constexpr int P_PACK = 4 * kW4TokChunk;            // [2 blocks][128 rows][128 B]
  static constexpr int P_SCALE = P_PACK + 2 * kW4PackBlock; // [2 blocks][8 groups][128 rows]
  static constexpr int PSTAGE = P_SCALE + 2 * kW4ScaleBlock;
  static constexpr int TX = PSTAGE;                         // TMA bytes per copy stage
  static constexpr int ACC_COLS = 2 * 2 * kW4BN;  // [issuer][block] x 32 columns
  static constexpr int A_COL0 = ACC_COLS;
  // one sub-stage holds a converter group's two 64-channel sub-blocks of a copy stage for both
  // blocks: [block][sub-block] x 32 columns
  static constexpr int CSTAGE_COLS = 2 * 2 * kW4ACols;
  static constexpr int CSTAGES = (kW4TmemCols - A_COL0) / CSTAGE_COLS;
  static constexpr int TABLE_BYTES = 2 * (kW4MaxGroups + 1) * 4 + kW4Threads * 4;
  static constexpr int NBARS = 32;
  static constexpr int BAR_BYTES = NBARS * 8 + 64;
  static constexpr int PSTAGES = (kW4SmemLimit - 1024 - BAR_BYTES - TABLE_BYTES) / PSTAGE;
  static constexpr int RINGS = PSTAGES * PSTAGE;
  static constexpr int SMEM = 1024 + RINGS + BAR_BYTES + TABLE_BYTES;
  static_assert(PSTAGES >= 3, "not enough shared memory for the copy ring");
  static_assert(CSTAGES == 3, "TMEM ring: three sub-stages shared by the two groups in turn");
  static_assert(SMEM <= kW4SmemLimit, "shared memory");
  static_assert(2 * PSTAGES + 2 * CSTAGES + 6 <= NBARS, "barrier area too small");
  static_assert(PSTAGE % 1024 == 0 && P_PACK % 1024 == 0 && P_SCALE % 128 == 0,
                "TMA and MMA operands misaligned");
};

struct W4Params {
  CUtensorMap map_act, map_act_d;  // tokens, bf16, 3D {64, rows, K/64}, box {64, 32, 4}, swizzled
  CUtensorMap map_wq, map_wq_d;    // codes, uint8, 3D {K/2, rows - blk, 2}, box {128, 128, 2}
  CUtensorMap map_ws, map_ws_d;    // scales, bf16, 3D {rows_per_group - blk, groups K/32, 2},
                                   // box {128, 8, 2}: routed experts' [K/32][rows] in turn
  const int32_t* offsets;
  int32_t n_routed, w_group_rows;
  int32_t dense_rows, dense_act_row0, dense_out_row0;
  int32_t K, F;
  void* out;  // SwiGLU: bf16 h [rows][ldo]; store: fp32 [rows][ldo]
  int64_t ldo;
  uint32_t* err;
};

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Four bf16 pairs (input channels 8i .. 8i+7, the even channel in each low half) from one packed
// word, whose code c sits in nibble c/2 + 4 (c % 2).
__device__ __forceinline__ void w4_expand_word(uint32_t w, __nv_bfloat162 s2, uint32_t* r) {
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t bits = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;  // bf16(128 + u) pair
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&bits);
    v = __hmul2(__hsub2(v, off), s2);  // (u - 8) exact, then one rounding of the product
    r[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// Whole warp: each lane writes 4 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

// One sub-block (64 input channels) of one weight row: its 32 code bytes (q0: channels 0..31,
// q1: 32..63) and the scales of its two groups, expanded word by word; each word's four bf16
// pairs go to TMEM columns t + 4i as soon as they exist (a 32-column store of the whole
// sub-block measured 1-2% slower).
__device__ __forceinline__ void w4_expand_sub_st(uint4 q0, uint4 q1, __nv_bfloat16 sc0,
                                                 __nv_bfloat16 sc1, uint32_t t) {
  const __nv_bfloat162 s0 = __bfloat162bfloat162(sc0);
  const __nv_bfloat162 s1 = __bfloat162bfloat162(sc1);
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t r[4];
    w4_expand_word(w[i], i < 4 ? s0 : s1, r);
    tmem_st4(t + 4 * i, r);
  }
}

template <bool kSwiGLU>
__global__ void __launch_bounds__(kW4Threads, 1) moe_gemm_w4_kernel(const __grid_constant__ W4Params p) {
  using S = W4Shape;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* pring = smem;  // [PSTAGES][PSTAGE]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::RINGS);
  uint64_t* pfull = bars;
  uint64_t* pempty = pfull + S::PSTAGES;
  uint64_t* cfull = pempty + S::PSTAGES;
  uint64_t* cempty = cfull + S::CSTAGES;
  uint64_t* tfull = cempty + S::CSTAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;  // one per issuer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* tile_start = reinterpret_cast<int*>(smem + S::RINGS + S::BAR_BYTES);
  int* row_start = tile_start + (kW4MaxGroups + 1);
  int* scratch = row_start + (kW4MaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rows_per_tile = kSwiGLU ? 128 : 256;  // features a tile covers

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::PSTAGES; ++s) {
      mbar_init(&pfull[s], 1);
      mbar_init(&pempty[s], kW4Conv + 2);  // every converter warp and both issuers
    }
    for (int s = 0; s < S::CSTAGES; ++s) {
      mbar_init(&cfull[s], kW4Conv / 2);  // the converter group of the sub-stage's parity
      mbar_init(&cempty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 2);
      mbar_init(&tempty[a], 128);
      mbar_init(&drain[a], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_act);
    tma_prefetch_map(&p.map_wq);
    tma_prefetch_map(&p.map_ws);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kW4TmemCols);
    tmem_relinquish();
  }
  build_tile_table(tile_start, row_start, scratch, p.offsets, p.n_routed, p.dense_rows, kW4BN,
                   p.F / rows_per_tile);  // ends with __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int G = p.n_routed + (p.dense_rows > 0 ? 1 : 0);
  const int total = tile_start[G];
  const int nsub_all = p.K / kW4Sub;                // TMEM sub-stages per tile (even)
  const int nkb = (nsub_all + 3) / 4;               // copy stages per tile (the last may be short)

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
        const int w_local = ti.ft * rows_per_tile;  // block 0's first row within its group
        const int w_y = (ti.dense ? 0 : ti.g * p.w_group_rows) + w_local;
        const int s_y = ti.dense ? 0 : ti.g * (p.K / 32);  // the group's first scale row
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_sleep(&pempty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* st = pring + stage * S::PSTAGE;
          mbar_arrive_expect_tx(&pfull[stage], S::TX);
          tma_load_3d(st + S::P_TOK, ma, &pfull[stage], 0, act_y, kb * 4);
          tma_load_3d(st + S::P_PACK, mq, &pfull[stage], kb * (kW4BK / 2), w_y, 0);
          tma_load_3d(st + S::P_SCALE, ms, &pfull[stage], w_local, s_y + kb * 8, 0);
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
          mbar_wait_sleep(&pfull[stage], phase, nullptr, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + kW4Conv) {
    // ---------------------------------------------------------------- converters
    const int grp = (warp - 2) >> 3;      // the sub-blocks of this parity (MMA issuer grp's)
    const int j = ((warp - 2) >> 2) & 1;  // the block this warp expands
    const int quarter = warp & 3;         // the TMEM lanes this warp may write
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16) + j * 2 * kW4ACols;
    uint32_t ps = 0, pph = 0, c = 0;  // c: copy stages seen (this group's sub-stage use 2c + grp)
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int nsub = min(4, nsub_all - kb * 4);  // 2 or 4
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait_sleep(&pfull[ps], pph, abort_flag, p.err) ? 1 : 0;
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
          ok = false;
          break;
        }
        // this warp's sub-blocks b = grp, grp + 2 of the stage: codes (128-byte swizzled row, 16-byte
        // chunk c at c ^ (row % 8)) and scales, read before any tcgen05 operation of the stage
        const uint8_t* src = pring + ps * S::PSTAGE;
        const uint8_t* qrow = src + S::P_PACK + j * kW4PackBlock + row * 128;
        const __nv_bfloat16* srow =
            reinterpret_cast<const __nv_bfloat16*>(src + S::P_SCALE + j * kW4ScaleBlock) + row;
        uint4 q[4];
        __nv_bfloat16 sc[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int b = grp + 2 * h;
          if (b < nsub) {
            q[2 * h] = *reinterpret_cast<const uint4*>(qrow + (((2 * b) ^ (row & 7)) << 4));
            q[2 * h + 1] = *reinterpret_cast<const uint4*>(qrow + (((2 * b + 1) ^ (row & 7)) << 4));
            sc[2 * h] = srow[(2 * b) * 128];
            sc[2 * h + 1] = srow[(2 * b + 1) * 128];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[ps]);
        {
          // the two groups take the three sub-stages in turn: use u = 2c + grp of the ring
          const uint32_t u = 2 * c + grp, cs = u % S::CSTAGES, cph = (u / S::CSTAGES) & 1u;
          if (lane == 0) w_ok = mbar_wait_sleep(&cempty[cs], cph ^ 1u, abort_flag, p.err) ? 1 : 0;
          w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
          if (!w_ok) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (grp + 2 * h >= nsub) break;
            w4_expand_sub_st(q[2 * h], q[2 * h + 1], sc[2 * h], sc[2 * h + 1],
                             t_lane + S::A_COL0 + cs * S::CSTAGE_COLS + h * kW4ACols);
          }
          tmem_st_wait();  // both sub-blocks' stores, then one release
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&cfull[cs]);
        }
        ++c;
        if (++ps == S::PSTAGES) {
          ps = 0;
          pph ^= 1u;
        }
      }
    }
  } else if (warp == 1 || warp == kW4Mma1Warp) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuers
      const int me = warp == 1 ? 0 : 1;
      uint32_t ps = 0, pph = 0, c = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                        p.dense_rows, p.dense_act_row0, kW4BN);
        const int n = ti.valid >= kW4BN ? kW4BN : ((ti.valid + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32_n(n);
        if (!mbar_wait_sleep(tempty, acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + me * 2 * kW4BN;
        uint32_t accum = 0;
        for (int kb = 0; kb < nkb && ok; ++kb) {
          const int nsub = min(4, nsub_all - kb * 4);  // 2 or 4: every stage has work for both
          if (!mbar_wait_sleep(&pfull[ps], pph, abort_flag, p.err)) {  // the stage's tokens
            ok = false;
            break;
          }
          const uint32_t tok = smem_u32(pring + ps * S::PSTAGE + S::P_TOK);
          {
            const uint32_t u = 2 * c + me, cs = u % S::CSTAGES, cph = (u / S::CSTAGES) & 1u;
            if (!mbar_wait_sleep(&cfull[cs], cph, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = tmem_base + S::A_COL0 + cs * S::CSTAGE_COLS;
            for (int h = 0; h < 2 && me + 2 * h < nsub; ++h) {
              const int b = me + 2 * h;  // this issuer's sub-blocks of the stage
#pragma unroll
              for (int k16 = 0; k16 < kW4Sub / 16; ++k16) {
                const uint64_t bdesc = sw128_kmajor_desc(tok + b * kW4TokChunk + k16 * 32);
                mma_bf16_tmem_a(d0, a0 + h * kW4ACols + k16 * 8, bdesc, idesc, accum);
                mma_bf16_tmem_a(d0 + kW4BN, a0 + 2 * kW4ACols + h * kW4ACols + k16 * 8, bdesc,
                                idesc, accum);
                accum = 1;
              }
            }
            mma_commit(&cempty[cs]);
          }
          ++c;
          mma_commit(&pempty[ps]);
          if (++ps == S::PSTAGES) {
            ps = 0;
            pph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull);
        acc_phase ^= 1u;
      }
      mma_commit(&drain[me]);
      mbar_wait_sleep(&drain[me], 0, nullptr, nullptr, kDrainLimitNs);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (4 warps)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                      p.dense_rows, p.dense_act_row0, kW4BN);
      int w_ok = 1;
      if (lane == 0) w_ok = mbar_wait_sleep(tfull, acc_phase, abort_flag, p.err) ? 1 : 0;
      w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
      if (!w_ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16);
      // y_b = issuer 0's half + issuer 1's half of block b, tokens 0..31 of the tile.  SwiGLU keeps
      // h = SiLU(y_0) * y_1 as bf16 pairs and stores after freeing the accumulator; the plain store
      // writes each 8-token chunk as soon as it is read.
      const int64_t out_row0 = (ti.dense ? (int64_t)p.dense_out_row0 : (int64_t)ti.grp_row0) +
                               (int64_t)ti.rt * kW4BN;
      const int64_t feat = (int64_t)ti.ft * rows_per_tile + r;
      uint32_t hpair[kSwiGLU ? kW4BN / 2 : 1];
#pragma unroll
      for (int c = 0; c < kW4BN; c += 8) {
        if (c < ti.valid) {
          uint32_t g0[8], g1[8], u0[8], u1[8];
          tmem_ld8(tb + c, g0);
          tmem_ld8(tb + 2 * kW4BN + c, g1);
          tmem_ld8(tb + kW4BN + c, u0);
          tmem_ld8(tb + 3 * kW4BN + c, u1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float ga = __uint_as_float(g0[i]) + __uint_as_float(g1[i]);
            const float gb = __uint_as_float(g0[i + 1]) + __uint_as_float(g1[i + 1]);
            const float ua = __uint_as_float(u0[i]) + __uint_as_float(u1[i]);
            const float ub = __uint_as_float(u0[i + 1]) + __uint_as_float(u1[i + 1]);
            if (kSwiGLU) {
              hpair[kSwiGLU ? (c + i) / 2 : 0] = pack_bf16x2(silu_fast(ga) * ua, silu_fast(gb) * ub);
            } else {
              if (c + i < ti.valid) {
                float* o = (float*)p.out + (out_row0 + c + i) * p.ldo + feat;
                o[0] = ga;
                o[128] = ua;
              }
              if (c + i + 1 < ti.valid) {
                float* o = (float*)p.out + (out_row0 + c + i + 1) * p.ldo + feat;
                o[0] = gb;
                o[128] = ub;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);  // the accumulator is free for the next tile
      acc_phase ^= 1u;
      if (kSwiGLU) {
        __nv_bfloat16* o = (__nv_bfloat16*)p.out + out_row0 * p.ldo + feat;
#pragma unroll
        for (int i = 0; i < kW4BN; ++i)
          if (i < ti.valid) {
            const uint32_t v = hpair[kSwiGLU ? i / 2 : 0] >> (16 * (i & 1));
            o[(int64_t)i * p.ldo] = __ushort_as_bfloat16((unsigned short)(v & 0xFFFFu));
          }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kW4TmemCols);
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

// 3D map: dims {d0, d1, d2} elements, byte strides {s1, s2} of dims 1 and 2, box {b0, b1, b2}.
static bool make_map_w4(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int64_t d0,
                        int64_t d1, int64_t d2, int64_t s1, int64_t s2, int b0, int b1, int b2,
                        CUtensorMapSwizzle swz) {
  EncodeTiledFnW4 enc = encode_fn_w4();
  if (!enc || !base || d0 <= 0 || d1 <= 0 || d2 <= 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)s1, (cuuint64_t)s2};
  cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, (cuuint32_t)b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The three maps of one weight set.  groups: how many [rows_per_group] weight groups (each with
// its [K/32][rows_per_group] scales); blk: rows from block 0 to block 1.  The row extents stop
// `blk` rows short of the end, so that block 1 of the last tile is still inside the tensor.
static bool w4_maps(CUtensorMap* act, CUtensorMap* wq, CUtensorMap* ws, const void* a,
                    int64_t a_rows, const void* q, const void* s, int64_t groups,
                    int64_t rows_per_group, int64_t blk, int K) {
  const int64_t half_k = K / 2;
  return make_map_w4(act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, kW4Sub, a_rows, K / kW4Sub,
                     (int64_t)K * 2, kW4Sub * 2, kW4Sub, kW4BN, 4, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_w4(wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, half_k, groups * rows_per_group - blk, 2,
                     half_k, blk * half_k, kW4BK / 2, 128, 2, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_w4(ws, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, s, rows_per_group - blk,
                     groups * (K / 32), 2, rows_per_group * 2, blk * 2, 128, kW4BK / 32, 2,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <bool kSwiGLU>
static cudaError_t launch_w4_variant(const W4Params& p, int grid, cudaStream_t st,
                                     const char* label) {
  auto kern = moe_gemm_w4_kernel<kSwiGLU>;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W4Shape::SMEM);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  LaunchScope ls(label, st);
  kern<<<grid, kW4Threads, W4Shape::SMEM, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_w4(const W4Gemm& g, int num_sms, cudaStream_t st) {
  // SwiGLU tiles: 128 features from W1 rows and the W3 rows u_off further; store tiles: 256 rows
  const int tile_rows = g.swiglu ? 128 : 256;
  if (g.K % (2 * kW4Sub) || g.F % tile_rows || g.n_routed > kW4MaxGroups - 1)
    return cudaErrorInvalidValue;
  if (g.w_group_rows % 128 || g.ldo % 8) return cudaErrorInvalidValue;
  const int blk = g.swiglu ? g.u_off : 128;
  const int blk_d = g.swiglu ? g.u_off_d : 128;
  if (g.swiglu && (blk < g.F || (g.dense_rows > 0 && blk_d < g.F))) return cudaErrorInvalidValue;
  W4Params p;
  memset(&p, 0, sizeof(p));
  if (g.n_routed > 0 && (g.w_rows != (int64_t)g.n_routed * g.w_group_rows ||
                         g.w_group_rows < blk + g.F - (g.swiglu ? 0 : 128) ||
                         !w4_maps(&p.map_act, &p.map_wq, &p.map_ws, g.act, g.act_rows, g.wq, g.ws,
                                  g.n_routed, g.w_group_rows, blk, g.K)))
    return cudaErrorInvalidValue;
  if (g.dense_rows > 0 && (g.w_d_rows < blk_d + g.F - (g.swiglu ? 0 : 128) ||
                           !w4_maps(&p.map_act_d, &p.map_wq_d, &p.map_ws_d, g.act_d, g.act_d_rows,
                                    g.wq_d, g.ws_d, 1, g.w_d_rows, blk_d, g.K)))
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
