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
//   warp 1      MMA issuer: per K-block one product, 4 x tcgen05.mma kind::f8f6f4 (M = 128,
//               N = 256, K = 32), into the next slot of a ring of two 256-column TMEM partial
//               buffers, commit -> partial_full[slot] (kF8SPK = 2 splits it into one N = 128
//               product per weight box over four 128-column slots);
//   warps 2..9  epilogue/promotion: kF8Parts = 2 warps per TMEM lane quarter; warp part p owns
//               columns [64p, 64p + 64) of each 128-column weight box of every slot.  Per slot
//               they read the partial, multiply by the row's activation scale times the box's
//               weight scale and add into fp32 registers, then free the slot.  The TMEM reads are
//               the long pole of that hand-off: one warp reads at a fixed rate whatever the load
//               shape, so a slot's 128 KB is read faster by more warps (1000, 820 and 740 cycles
//               per K-block with 4, 8 and 16 warps in a microbenchmark, against 512 cycles of
//               MMA).  Four parts (16 warps) measured slower in the kernel itself: at 576
//               threads a thread gets 96 registers, and the loop no longer fits.
// Tiles are token rows (M = 128) x 256 weight rows, as in the bf16 rows orientation:
//   SwiGLU: the first box holds the W1 rows of 128 features, the second the W3 rows of the same
//           features; warp part p owns features 64p..64p + 63 (g and u).  The epilogue forms
//           h = SiLU(g) * u and quantises it per row per 128 features -- exactly one tile -- to
//           e4m3 with scale amax/448 (the parts exchange their amax).
//   store:  the boxes are weight blocks 2 ft and 2 ft + 1 (output features 0..127 and
//           128..255 of the tile); fp32 output, written through a per-warp staging buffer.
// Every wait is bounded as in the bf16 kernel.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

constexpr int kF8Parts = 2;                  // promotion warps per TMEM lane quarter (2 or 4)
constexpr int kF8PartCols = 128 / kF8Parts;  // columns of each weight box per promotion warp
constexpr int kF8PromoWarps = 4 * kF8Parts;
constexpr int kF8Threads = 64 + 32 * kF8PromoWarps;
constexpr int kF8BK = 128;                // e4m3 per K-block = bytes per row of a stage
constexpr int kF8BN = 256;
constexpr int kF8Box = 128 * 128;         // one 128-row x 128-byte box
constexpr int kF8Stage = kF8Box + 2 * kF8Box;
constexpr int kF8MaxGroups = 1025;
constexpr int kF8Table = 2 * (kF8MaxGroups + 1) * 4 + kF8Threads * 4;
constexpr int kF8Bars = 256 + 64;
constexpr int kF8Xchg = 2 * kF8Parts * 128 * 4;  // [tile parity][part][row] amax exchange
constexpr int kF8Stages = 3;  // measured as fast as four (2.71 vs 2.75 ms at 8192 tokens)
// Partial products per K-block: 1 = one N = 256 product into a ring of two 256-column TMEM
// buffers; 2 = one N = 128 product per 128-row weight box into a ring of four 128-column slots.
constexpr int kF8SPK = 1;
constexpr int kF8SlotCols = 256 / kF8SPK;
constexpr int kF8Slots = 512 / kF8SlotCols;
// per epilogue warp, for row stores: 32 rows x 256 bytes of fp32 with two parts (the W2
// epilogue stages a whole weight box per row), 32 rows x 64 bytes with four
constexpr int kF8WarpStaging = kF8PartCols == 64 ? 8192 : 2048;
constexpr int kF8Staging = kF8PromoWarps * kF8WarpStaging;
constexpr int kF8Acc = 2 * kF8PartCols;            // fp32 accumulators per promotion thread
constexpr int kF8Smem = 1024 + kF8Stages * kF8Stage + kF8Bars + kF8Xchg + kF8Table + kF8Staging;
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
  void* out;              // SwiGLU: e4m3 h [rows][ldo]; store: fp32 (or bf16) [rows][ldo]
  int64_t ldo;
  int32_t out_bf16;       // store: bf16 outputs instead of fp32
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

// Warp-cooperative store of 32 rows x 64 bytes (lane l holds row l) through a 2 KB XOR-swizzled
// shared buffer: each store instruction then writes 8 whole 64-byte row pieces instead of 32
// scattered 16-byte ones.  Rows >= valid_rows are not written.
__device__ __forceinline__ void store_rows_64B(uint8_t* buf, int lane, const uint4 (&v)[4],
                                               uint8_t* row0, int pitch, int valid_rows) {
  __syncwarp();  // the previous chunk's read-back has finished
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v[j];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2);
    const int j = lane & 3;
    const uint4 w = *reinterpret_cast<const uint4*>(buf + r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
    if (r < valid_rows) *reinterpret_cast<uint4*>(row0 + (r * pitch + j * 16)) = w;
  }
}

// The same for 32 rows x 32 bytes (1 KB of the buffer): each read-back instruction writes 16
// whole 32-byte row pieces.
__device__ __forceinline__ void store_rows_32B(uint8_t* buf, int lane, const uint4 (&v)[2],
                                               uint8_t* row0, int pitch, int valid_rows) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 2; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 32 + ((j ^ ((lane >> 2) & 1)) << 4)) = v[j];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = i * 16 + (lane >> 1);
    const int j = lane & 1;
    const uint4 w = *reinterpret_cast<const uint4*>(buf + r * 32 + ((j ^ ((r >> 2) & 1)) << 4));
    if (r < valid_rows) *reinterpret_cast<uint4*>(row0 + (r * pitch + j * 16)) = w;
  }
}

// A warp's piece of h rows: 64 or 32 bytes of e4m3 per row, by the width of its part.
__device__ __forceinline__ void store_h_rows(uint8_t* buf, int lane, const uint4 (&v)[4],
                                             uint8_t* row0, int pitch, int valid_rows) {
  store_rows_64B(buf, lane, v, row0, pitch, valid_rows);
}
__device__ __forceinline__ void store_h_rows(uint8_t* buf, int lane, const uint4 (&v)[2],
                                             uint8_t* row0, int pitch, int valid_rows) {
  store_rows_32B(buf, lane, v, row0, pitch, valid_rows);
}

// Warp-cooperative store of 32 rows x 256 bytes (lane l holds row l: 64 fp32 from acc[a0..])
// through an 8 KB XOR-swizzled buffer.  All 64 values go to shared memory before any is read
// back, so their registers are free for the read-back; each store instruction then writes two
// whole 256-byte row pieces.  Rows >= valid_rows are not written.
__device__ __forceinline__ void store_rows_256B(uint8_t* buf, int lane, const float (&acc)[kF8Acc],
                                                int a0, uint8_t* row0, int pitch, int valid_rows) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 16; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 256 + ((j ^ (lane & 15)) << 4)) =
        make_uint4(__float_as_uint(acc[a0 + 4 * j]), __float_as_uint(acc[a0 + 4 * j + 1]),
                   __float_as_uint(acc[a0 + 4 * j + 2]), __float_as_uint(acc[a0 + 4 * j + 3]));
  __syncwarp();
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int r = i * 2 + (lane >> 4);
    const int j = lane & 15;
    const uint4 w = *reinterpret_cast<const uint4*>(buf + r * 256 + ((j ^ (r & 15)) << 4));
    if (r < valid_rows) *reinterpret_cast<uint4*>(row0 + (r * pitch + j * 16)) = w;
  }
}

// The same for 32 rows x 128 bytes (lane l holds row l: 64 bf16 as 8 x 16 bytes) through 4 KB of
// the buffer: each read-back instruction writes four whole 128-byte row pieces.
__device__ __forceinline__ void store_rows_128B_f8(uint8_t* buf, int lane, const uint4 (&v)[8],
                                                   uint8_t* row0, int pitch, int valid_rows) {
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = v[j];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const int j = lane & 7;
    const uint4 w = *reinterpret_cast<const uint4*>(buf + r * 128 + ((j ^ (r & 7)) << 4));
    if (r < valid_rows) *reinterpret_cast<uint4*>(row0 + (r * pitch + j * 16)) = w;
  }
}

// SiLU for the fp8 epilogue: the quotient with the fast division (h is quantised to e4m3 next)
__device__ __forceinline__ float silu_fp8(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// One promotion step of a warp: wait for partial product ks (slot ks % kF8Slots), which holds
// weight boxes BOX0 .. BOX0 + kF8SlotCols / 128 - 1; add s_box * partial[box column c] into
// acc[box * kF8PartCols + c] for this thread's kF8PartCols columns of each box (tq addresses its
// lane and first column; box 0 is scaled by s0, box 1 by s1), then release the slot.  False when
// the wait gave up.
template <int BOX0>
__device__ __forceinline__ bool promote_slot(float (&acc)[kF8Acc], float s0, float s1, uint32_t tq,
                                             uint32_t ks,
                                             uint64_t* pfull, uint64_t* pempty, int lane,
                                             volatile int* abort_flag, uint32_t* err) {
  const uint32_t slot = ks % kF8Slots, sph = (ks / kF8Slots) & 1u;
  int w_ok = 1;
  if (lane == 0) w_ok = mbar_wait(&pfull[slot], sph, abort_flag, err) ? 1 : 0;
  w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
  if (!w_ok) return false;
  tc_fence_after();
  const uint32_t tb = tq + slot * kF8SlotCols;
#pragma unroll
  for (int j = 0; j < kF8SlotCols / 128; ++j) {  // the weight boxes this slot holds
    constexpr int kBase = BOX0 * kF8PartCols;
    const float sc = (BOX0 + j) ? s1 : s0;
#pragma unroll
    for (int c = 0; c < kF8PartCols; c += 16) {  // 16 columns per TMEM load and wait
      uint32_t v[16];
      tmem_ld16(tb + j * 128 + c, v);
      tmem_ld_wait();
      float* a = acc + kBase + j * kF8PartCols + c;
#pragma unroll
      for (int i = 0; i < 16; i += 2) fma2(a[i], a[i + 1], sc, v[i], v[i + 1]);
    }
  }
  // every lane's loads of this slot have completed (tcgen05.wait::ld); one arrival per warp
  // after a warp barrier releases the slot to the MMA issuer
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&pempty[slot]);
  return true;
}

template <bool kSwiGLU>
__global__ void __launch_bounds__(kF8Threads, 1) moe_gemm_fp8_kernel(const __grid_constant__ F8Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF8Stages * kF8Stage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kF8Stages;
  uint64_t* pfull = bars + 2 * kF8Stages;  // [kF8Slots]
  uint64_t* pempty = pfull + kF8Slots;     // [kF8Slots]
  uint64_t* drain = pempty + kF8Slots;
  uint64_t* xbar = drain + 1;  // [2]: amax exchange between the epilogue parts
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* xchg = reinterpret_cast<float*>(smem + kF8Stages * kF8Stage + kF8Bars);  // [2][parts][128]
  int* tile_start = reinterpret_cast<int*>(smem + kF8Stages * kF8Stage + kF8Bars + kF8Xchg);
  int* row_start = tile_start + (kF8MaxGroups + 1);
  int* scratch = row_start + (kF8MaxGroups + 1);
  uint8_t* staging = smem + kF8Stages * kF8Stage + kF8Bars + kF8Xchg + kF8Table;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int FPT = kSwiGLU ? 128 : kF8BN;  // output features per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kF8Slots; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], kF8PromoWarps);  // one arrival per promotion warp
    }
    mbar_init(drain, 1);
    mbar_init(&xbar[0], kF8PromoWarps);
    mbar_init(&xbar[1], kF8PromoWarps);
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
      // the boxes of (tile, kb): activation rows, then the two 128-row weight boxes
      auto boxes = [&](const TileInfo& ti, const CUtensorMap*& ma, const CUtensorMap*& mw,
                       int& act_y, int& w_y0, int& w_y1) {
        ma = ti.dense ? &p.map_act_d : &p.map_act;
        mw = ti.dense ? &p.map_w_d : &p.map_w;
        act_y = ti.grp_row0 + ti.rt * 128;
        w_y0 = (ti.dense ? 0 : ti.g * p.w_group_rows) + ti.ft * FPT;
        w_y1 = kSwiGLU ? w_y0 + (ti.dense ? p.u_off_d : p.u_off) : w_y0 + 128;
      };
      uint32_t stage = 0, phase = 0;
      int armed = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                        p.dense_rows, p.dense_act_row0, 128);
        const CUtensorMap* ma;
        const CUtensorMap* mw;
        int act_y, w_y0, w_y1;
        boxes(ti, ma, mw, act_y, w_y0, w_y1);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kF8Stage;
          uint8_t* sb = sa + kF8Box;
          mbar_arrive_expect_tx(&full[stage], kF8Stage);
          const int kx = kb * (kF8BK / 8);  // in the maps' 8-byte elements
          tma_load_2d(sa, ma, &full[stage], kx, act_y);
          tma_load_2d(sb, mw, &full[stage], kx, w_y0);
          tma_load_2d(sb + kF8Box, mw, &full[stage], kx, w_y1);
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
      constexpr uint32_t kIdesc = idesc_e4m3_f32<128, kF8SlotCols>();
      uint32_t stage = 0, phase = 0;
      uint32_t ks = 0;  // partial products issued so far (all tiles): slot = ks % kF8Slots
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nkb && ok; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * kF8Stage);
          // the K-block's two 128-row weight boxes go to two slots, so that the promotion can
          // free one slot while the MMA fills the next ones
#pragma unroll 1
          for (int hb = 0; hb < kF8SPK; ++hb, ++ks) {
            const uint32_t slot = ks % kF8Slots, sph = (ks / kF8Slots) & 1u;
            if (!mbar_wait(&pempty[slot], sph ^ 1u, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sb = sa + kF8Box + hb * (kF8SlotCols / 128) * kF8Box;
            const uint32_t d = tmem_base + slot * kF8SlotCols;
#pragma unroll
            for (int k32 = 0; k32 < kF8BK / 32; ++k32)
              mma_e4m3(d, sw128_kmajor_desc(sa + k32 * 32), sw128_kmajor_desc(sb + k32 * 32),
                       kIdesc, k32 != 0);
            mma_commit(&pfull[slot]);
          }
          if (!ok) break;
          mma_commit(&empty[stage]);
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
    const int part = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    uint8_t* wbuf = staging + (warp - 2) * kF8WarpStaging;
    uint32_t ks = 0;  // partial products consumed so far (all tiles), as counted by the MMA issuer
    uint32_t it = 0;  // tiles finished by this thread: exchange slot it & 1
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                      p.dense_rows, p.dense_act_row0, 128);
      const bool valid = r < ti.valid;
      const int vrows = ti.valid - quarter * 32;  // rows of this warp's 32 that are real
      const int64_t act_row = (int64_t)ti.grp_row0 + ti.rt * 128 + r;
      const float* sx_col = ti.dense ? p.act_sT_d : p.act_sT;
      const int64_t sx_ld = ti.dense ? p.act_s_ld_d : p.act_s_ld;
      const int wblocks = p.w_group_rows / 128;
      // weight-scale rows of the tile's two 128-row weight boxes (slot hb = 0 and hb = 1)
      const float* ws0;
      const float* ws1;
      if (kSwiGLU) {
        const int u_off = ti.dense ? p.u_off_d : p.u_off;
        const int rb_g = ti.ft, rb_u = (u_off + ti.ft * 128) / 128;
        const float* base = ti.dense ? p.w_s_d : p.w_s + (int64_t)ti.g * wblocks * nkb;
        ws0 = base + (int64_t)rb_g * nkb;
        ws1 = base + (int64_t)rb_u * nkb;
      } else {
        const float* base = ti.dense ? p.w_s_d : p.w_s + (int64_t)ti.g * wblocks * nkb;
        ws0 = base + (int64_t)(ti.ft * 2) * nkb;
        ws1 = ws0 + nkb;
      }
      float acc[kF8Acc];
#pragma unroll
      for (int i = 0; i < kF8Acc; ++i) acc[i] = 0.0f;
      // the scales of K-block kb + 1 are loaded while block kb is promoted (their global-memory
      // latency then hides behind the MMA instead of stalling every block)
      const float* sx_ptr = sx_col + act_row;
      float sx_n = valid ? __ldg(sx_ptr) : 0.0f;
      float w0_n = __ldg(ws0), w1_n = __ldg(ws1);
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const float sx = sx_n, w0 = w0_n, w1 = w1_n;
        if (kb + 1 < nkb) {
          sx_n = valid ? __ldg(sx_ptr + (int64_t)(kb + 1) * sx_ld) : 0.0f;
          w0_n = __ldg(ws0 + kb + 1);
          w1_n = __ldg(ws1 + kb + 1);
        }
        // this thread owns columns [part * P, part * P + P) of both weight boxes of the
        // K-block, P = kF8PartCols: acc[0..P-1] from the first box, acc[P..2P-1] from the second
        const uint32_t tq = tmem_base + part * kF8PartCols + ((uint32_t)(quarter * 32) << 16);
        const float s0 = sx * w0, s1 = sx * w1;
        if constexpr (kF8SPK == 1) {
          ok = promote_slot<0>(acc, s0, s1, tq, ks, pfull, pempty, lane, abort_flag, p.err);
        } else {
          ok = promote_slot<0>(acc, s0, s1, tq, ks, pfull, pempty, lane, abort_flag, p.err) &&
               promote_slot<1>(acc, s0, s1, tq, ks + 1, pfull, pempty, lane, abort_flag, p.err);
        }
        ks += kF8SPK;
      }
      if (!ok) break;
      const int64_t orow =
          (ti.dense ? (int64_t)p.dense_out_row0 : (int64_t)ti.grp_row0) + ti.rt * 128 + r;
      if (kSwiGLU) {
        // h = SiLU(g) * u for this thread's features, then e4m3 per 128-feature group
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < kF8PartCols; ++j) {
          acc[j] = silu_fp8(acc[j]) * acc[kF8PartCols + j];
          amax = fmaxf(amax, fabsf(acc[j]));
        }
        // exchange with the other parts through a double-buffered slot and a bounded mbarrier
        // wait: slot it&1 is rewritten two tiles later, after every part has passed the barrier of
        // the tile in between, i.e. after each has read this one
        float* slot = xchg + (it & 1u) * (kF8Parts * 128);
        slot[part * 128 + r] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[it & 1u]);
        int x_ok = 1;
        if (lane == 0) x_ok = mbar_wait(&xbar[it & 1u], (it >> 1) & 1u, abort_flag, p.err) ? 1 : 0;
        x_ok = __shfl_sync(0xffffffffu, x_ok, 0);
        __syncwarp();
        if (!x_ok) break;
#pragma unroll
        for (int q = 0; q < kF8Parts; ++q) amax = fmaxf(amax, slot[q * 128 + r]);
        const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        const float rscale = __frcp_rn(scale);
        uint4 v[kF8PartCols / 16];
#pragma unroll
        for (int c = 0; c < kF8PartCols / 16; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = c * 16 + q * 4;
            w[q] = e4m3x4_pack(div_rn_by_recip(acc[j], scale, rscale),
                               div_rn_by_recip(acc[j + 1], scale, rscale),
                               div_rn_by_recip(acc[j + 2], scale, rscale),
                               div_rn_by_recip(acc[j + 3], scale, rscale));
          }
          v[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        uint8_t* dst0 =
            (uint8_t*)p.out + (orow - lane) * p.ldo + (int64_t)ti.ft * 128 + part * kF8PartCols;
        store_h_rows(wbuf, lane, v, dst0, (int)p.ldo, vrows);
        if (valid && part == 0) p.out_sT[(int64_t)ti.ft * p.out_s_ld + orow] = scale;
      } else {
        // acc[j], j < P, is output column ft*256 + part*P + j; acc[P + j] the same + 128
        uint8_t* dst0 = (uint8_t*)p.out +
                        ((orow - lane) * p.ldo + (int64_t)ti.ft * kF8BN + part * kF8PartCols) * 4;
        if (kF8PartCols == 64 && p.out_bf16) {  // bf16: 128 bytes of each row per box
          uint8_t* b0 = (uint8_t*)p.out +
                        ((orow - lane) * p.ldo + (int64_t)ti.ft * kF8BN + part * kF8PartCols) * 2;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            uint4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float* a = acc + hb * 64 + 8 * q;
              v[q] = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
            }
            store_rows_128B_f8(wbuf, lane, v, b0 + hb * 128 * 2, (int)p.ldo * 2, vrows);
          }
        } else if constexpr (kF8PartCols == 64) {
          store_rows_256B(wbuf, lane, acc, 0, dst0, (int)p.ldo * 4, vrows);
          store_rows_256B(wbuf, lane, acc, 64, dst0 + 128 * 4, (int)p.ldo * 4, vrows);
        } else {
#pragma unroll
          for (int c = 0; c < kF8Acc; c += 16) {
            uint4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              v[q] = make_uint4(__float_as_uint(acc[c + 4 * q]), __float_as_uint(acc[c + 4 * q + 1]),
                                __float_as_uint(acc[c + 4 * q + 2]), __float_as_uint(acc[c + 4 * q + 3]));
            const int col = (c < kF8PartCols ? c : 128 + (c - kF8PartCols));
            store_rows_64B(wbuf, lane, v, dst0 + col * 4, (int)p.ldo * 4, vrows);
          }
        }
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

// 2D map over a byte matrix [rows][cols] (cols % 8 == 0), box {128 bytes, 128 rows}, 128-byte
// swizzle, zero fill.  The copy moves bytes unchanged, so the map describes each row as cols / 8
// 8-byte elements: a 16 KB box is then 2048 elements instead of 16384 single bytes, which the TMA
// unit moves faster.  x coordinates passed to the copies are in these 8-byte units.
static bool make_map_u8(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFnF8 enc = encode_fn_f8();
  if (!enc || !base || rows <= 0 || cols <= 0 || cols % 8) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(cols / 8), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {16, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides, box,
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
  if (g.w_group_rows % 128 || g.ldo % 16 || g.ldo > (1 << 24)) return cudaErrorInvalidValue;
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
  p.out_bf16 = !g.swiglu && g.out_bf16 ? 1 : 0;
  p.err = g.err;
  if (g.swiglu) return launch_f8_variant<true>(p, num_sms, st, g.label);
  return launch_f8_variant<false>(p, num_sms, st, g.label);
}

}  // namespace moe
