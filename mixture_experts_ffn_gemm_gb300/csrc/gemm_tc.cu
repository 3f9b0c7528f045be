// gemm_tc.cu -- grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM, TMA), bf16 in,
// fp32 accumulation.
//
// The expert MLPs of the "Mixture of experts" steps (g = x W1, u = x W3, a = g sigma(g), h = a * u,
// E_i = h W2; the shared expert the same) run as grouped GEMMs over the permuted rows: one group per
// routed expert (rows [offsets[g], offsets[g+1])) plus a trailing dense group (the shared expert,
// every token, or a plain dense projection).  This replaces the per-expert host loop of the
// `moe_infer` excerpt on "Kimi K3 · Latent up-projection"; group sizes stay on the device.
//
// Kernel shape: persistent, one CTA per SM, 192 threads, warp-specialised:
//   warp 0      TMA producer: K-blocks of 64 bf16 (one 128-byte swizzle row) into a ring of
//               shared-memory stages, completion counted on full[s] mbarriers;
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, M = 128, into one of two TMEM
//               accumulators, frees stages with tcgen05.commit -> empty[s], signals tmem_full[a];
//   warps 2..5  epilogue: tcgen05.ld from TMEM (each warp reads its 32-lane quarter), SwiGLU or a
//               plain store, then release the accumulator (tmem_empty[a]) so the next tile's
//               mainloop overlaps this tile's epilogue.
// Two tile orientations:
//   rows  (swap = 0): MMA M = 128 token rows, N = 256 weight rows.  SwiGLU tiles load 128 W1 rows and
//                     the matching 128 W3 rows, so each thread (= one token row) holds g and u of the
//                     same features in its own TMEM lane and the epilogue needs no exchange.
//                     With two M halves (kMH = 2) a tile is 256 token rows: two M = 128 MMAs share
//                     each staged weight K-block, so a CTA copies 64 KB per 1024 MMA cycles instead
//                     of 48 KB per 512, and three 64 KB stages hide about 3000 cycles of copy
//                     latency.  A tile whose rows end within its first half issues only that half
//                     (the padding stays at 128 rows).  The two halves fill all 512 TMEM columns,
//                     so the epilogue of a tile no longer overlaps the next tile's mainloop.
//   swap  (swap = 1): MMA M = 128 weight rows, N = 32 tokens, for groups with few rows (decode):
//                     the weights stream once per 32 tokens instead of once per 128-row tile padded
//                     with empty rows.  SwiGLU keeps a W1 accumulator and a W3 accumulator.
// Every wait is bounded (common.cuh): on expiry the kernel flags kErrTimeout, drains its in-flight
// copies and MMAs, frees TMEM and returns.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

constexpr int kTcThreads = 192;
constexpr int kBK = 64;                  // bf16 K-elements per stage (128 bytes per row)
constexpr int kBoxBytes = 128 * 128;     // one 128-row x 128-byte operand box
constexpr int kTcMaxGroups = 1025;
constexpr int kSmemLimit = 232448;       // 227 KB per CTA

struct TcParams {
  CUtensorMap map_act;    // routed activations [rows][K]
  CUtensorMap map_w;      // routed weights [E * w_group_rows][K]
  CUtensorMap map_act_d;  // dense-group activations
  CUtensorMap map_w_d;    // dense-group weights
  CUtensorMap map_out;    // fp32 output [rows][ldo], box {32, 32}, 128-byte swizzle (tma_out)
  // token-rows N = 256 tiles with one weight box per stage (big_boxes): SwiGLU, a 3D map
  // {K, rows of one half, halves} with box {64, 128, 2} (a feature tile's W1 and W3 rows in one
  // copy); store, a 2D map with box {64, 256}
  CUtensorMap map_wb;
  CUtensorMap map_wb_d;
  const int32_t* offsets;
  int32_t n_routed, w_group_rows, u_off, u_off_d;
  int32_t dense_rows, dense_act_row0, dense_out_row0;
  int32_t K, k_wrap, F;          // routed groups
  int32_t K_d, k_wrap_d, F_d;    // the dense group (its own reduction length and features)
  void* out;
  int64_t ldo;
  void* out_d;                   // the dense group's output and row pitch
  int64_t ldo_d;
  int32_t out_f32;
  int32_t tma_out;      // token-rows fp32 stores: whole 32-row chunks leave by TMA from staging
  const float* addend;  // EPI_STORE_ADD: fp32 [rows][ld_add]
  int64_t ld_add;
  uint32_t* err;
  uint64_t wait_ns;     // limit of every mbarrier wait
  int32_t test_stall;   // test hook: the producer issues no copy, so the MMA's wait expires
  int32_t dense_band;   // the dense group's tiles in bands of this many row tiles (0: one band)
  int32_t big_boxes;    // weights copied in one box per stage (map_wb / map_wb_d): one copy
                        // fewer per stage, measured 1-1.5% faster at prefill
  // split-K (a dense-only fp32 store launch with few row tiles): every output tile is computed
  // as ksplit partial sums over consecutive K ranges, partial s written split_rows rows further
  int32_t ksplit;
  int64_t split_rows;
};

__device__ __forceinline__ void tma_load_3d_tc(void* smem_dst, const CUtensorMap* map,
                                               uint64_t* bar, int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

template <bool kSwap, int kBN, int kEpi, int kMH = 1, bool kPair = false>
struct TcShape {
  static_assert(kMH == 1 || (kMH == 2 && !kSwap && kBN == 256), "two M halves: token rows, N = 256");
  static_assert(!kPair || (!kSwap && kBN == 256 && kMH == 1 && kEpi != EPI_STORE_ADD),
                "CTA pairs: token-rows SwiGLU / store tiles, N = 256");
  static constexpr bool kSwiGLU = kEpi == EPI_SWIGLU;
  // 256-token swap-AB SwiGLU tiles stack 64 W1 rows over the matching 64 W3 rows in one M = 128
  // operand, so that one 256-column accumulator holds both and two of them fit in TMEM
  static constexpr bool kStack = kSwap && kSwiGLU && kBN == 256;
  static constexpr int RPT = kSwap ? kBN : 128 * kMH * (kPair ? 2 : 1);  // token rows per tile
  static constexpr int FPT = kSwap ? (kStack ? 64 : 128) : (kSwiGLU ? kBN / 2 : kBN);  // features
  static constexpr int OPA =
      (kSwap && kSwiGLU && !kStack) ? 2 * kBoxBytes : kMH * kBoxBytes;  // A bytes / stage
  static constexpr int OPB = (kPair ? kBN / 2 : kBN) * 128;  // B bytes / stage (a pair: half)
  static constexpr int STAGE = OPA + OPB;
  static constexpr int ACC_COLS =
      (kSwap && kSwiGLU && !kStack) ? 2 * kBN : kMH * kBN;  // fp32 columns of one accumulator
  // two accumulators (the epilogue of tile i overlaps the mainloop of tile i+1) when they fit
  static constexpr int NACC = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr int TMEM_NEED = NACC * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                   : TMEM_NEED <= 64  ? 64
                                   : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256
                                                      : 512;
  static constexpr int TABLE_BYTES = 2 * (kTcMaxGroups + 1) * 4 + kTcThreads * 4;
  static constexpr int BAR_BYTES = 256 + 64;  // barriers, TMEM base, abort flag
  // token-rows epilogues stage each warp's 32 rows x 128 bytes through shared memory so that
  // the global stores are whole rows (4 KB per epilogue warp)
  static constexpr bool kStaged = !kSwap && kEpi != EPI_STORE_ADD;
  static constexpr int STAGING = kStaged ? 4 * 4096 : 0;
  // stacked tiles: g and u of 64 features x 16 tokens meet here (rows padded to 17 words)
  static constexpr int XCH = kStack ? 2 * 64 * 17 * 4 : 0;
  static constexpr int STAGES_FIT =
      (kSmemLimit - 1024 - TABLE_BYTES - BAR_BYTES - STAGING - XCH) / STAGE;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM = 1024 + STAGES * STAGE + BAR_BYTES + TABLE_BYTES + STAGING + XCH;
  static_assert(STAGES >= 2, "not enough shared memory for two stages");
  static_assert(TMEM_NEED <= 512, "accumulators exceed TMEM");
  static_assert(STAGE % 1024 == 0, "stages must keep 1024-byte alignment for SWIZZLE_128B");
  static_assert(2 * STAGES + 5 <= 32, "barrier area too small");
};

// One epilogue warp writes a chunk of 32 rows x 128 bytes: lane l holds row l's 128 bytes in v.
// The chunk goes through a 4 KB shared buffer (16-byte pieces XOR-swizzled by row % 8, free of
// bank conflicts both ways) and leaves as 4 whole 128-byte rows per store instruction.
__device__ __forceinline__ void store_rows_128B(uint8_t* buf, int lane, const uint4 (&v)[8],
                                                uint8_t* row0, int64_t pitch, int valid_rows) {
  __syncwarp();  // the previous chunk's read-back has finished
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = v[j];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const int j = lane & 7;
    const uint4 w = *reinterpret_cast<const uint4*>(buf + r * 128 + ((j ^ (r & 7)) << 4));
    if (r < valid_rows) *reinterpret_cast<uint4*>(row0 + r * pitch + j * 16) = w;
  }
}

template <bool kSwap, int kBN, int kEpi, int kMH = 1, bool kPair = false>
__global__ void __launch_bounds__(kTcThreads, 1) moe_gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using S = TcShape<kSwap, kBN, kEpi, kMH, kPair>;
  // CTA pairs: the two CTAs of a cluster share every tile (256 token rows, 128 each) and one
  // M = 256 MMA per K-step issued by the even CTA; each CTA copies its own 128 activation rows and
  // its half of the weight rows, so a stage is 32 KB per SM for the MMA work a 48 KB stage feeds
  // in a CTA alone, and six stages are in flight.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int tile0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int tstep = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // stages, then the staging / exchange buffers (1024-byte aligned: TMA reads them swizzled),
  // then barriers and the tile table
  uint8_t* staging = smem + S::STAGES * S::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + S::STAGING + S::XCH);
  uint64_t* full = bars;
  uint64_t* empty = bars + S::STAGES;
  uint64_t* tfull = bars + 2 * S::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* tile_start = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + S::BAR_BYTES);
  int* row_start = tile_start + (kTcMaxGroups + 1);
  int* scratch = row_start + (kTcMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kPair ? 256 : 128);  // a pair: both CTAs' epilogue threads
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_act);
    tma_prefetch_map(&p.map_w);
    if (p.dense_rows > 0) {
      tma_prefetch_map(&p.map_act_d);
      tma_prefetch_map(&p.map_w_d);
    }
  }
  if (warp == 1) {
    if constexpr (kPair) {  // one warp of each CTA of the pair, together
      tmem_alloc_pair(tmem_holder, S::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, S::TMEM_COLS);
      tmem_relinquish();
    }
  }
  build_tile_table(tile_start, row_start, scratch, p.offsets, p.n_routed, p.dense_rows, S::RPT,
                   p.F / S::FPT, p.F_d / S::FPT);  // ends with __syncthreads
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int G = p.n_routed + (p.dense_rows > 0 ? 1 : 0);
  const int total = tile_start[G] * p.ksplit;  // (tile, K range) pairs
  const int nkb_r = p.K / kBK, nkb_d = p.K_d / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && !p.test_stall) {
      uint32_t stage = 0, phase = 0;
      int armed = 0;
      bool ok = true;
      for (int tile = tile0; tile < total && ok; tile += tstep) {
        const int ks = tile % p.ksplit;
        const TileInfo ti = decode_tile(tile / p.ksplit, tile_start, row_start, p.offsets,
                                        p.n_routed, p.dense_rows, p.dense_act_row0, S::RPT,
                                        p.dense_band);
        const CUtensorMap* ma = ti.dense ? &p.map_act_d : &p.map_act;
        const CUtensorMap* mw = ti.dense ? &p.map_w_d : &p.map_w;
        const int act_y = ti.grp_row0 + ti.rt * S::RPT;
        const int w_y = (ti.dense ? 0 : ti.g * p.w_group_rows) + ti.ft * S::FPT;
        const int u_off = ti.dense ? p.u_off_d : p.u_off;
        const int nkb_all = ti.dense ? nkb_d : nkb_r;
        const int kb0 = ks * nkb_all / p.ksplit, nkb = (ks + 1) * nkb_all / p.ksplit;
        const int kwrap = ti.dense ? p.k_wrap_d : p.k_wrap;
        // the second M half's rows are copied only when the tile has rows there
        const bool half1 = kMH == 2 && ti.valid > 128;
        const uint32_t tx = (kMH == 2 && !half1) ? S::STAGE - kBoxBytes : S::STAGE;
        for (int kb = kb0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * S::STAGE;
          uint8_t* sb = sa + S::OPA;
          const int kx = kb * kBK;
          const int ax = kx % kwrap;
          if constexpr (kPair) {
            // this CTA's 128 activation rows and its half of the weight rows (SwiGLU: the W1 rows
            // on the even CTA, the matching W3 rows on the odd one); both CTAs' copies complete
            // on the even CTA's barrier, which expects the bytes of both
            const uint32_t bar = cluster_addr(&full[stage], 0);
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * S::STAGE);
            tma_load_2d_pair(sa, ma, bar, ax, act_y + (int)rank * 128);
            tma_load_2d_pair(sb, mw, bar, kx,
                             S::kSwiGLU ? (rank ? w_y + u_off : w_y) : w_y + (int)rank * 128);
          } else {
          mbar_arrive_expect_tx(&full[stage], tx);
          if (!kSwap) {
            tma_load_2d(sa, ma, &full[stage], ax, act_y);
            if (half1) tma_load_2d(sa + kBoxBytes, ma, &full[stage], ax, act_y + 128);
            if (kBN == 256 && kMH == 1 && p.big_boxes) {
              const CUtensorMap* mwb = ti.dense ? &p.map_wb_d : &p.map_wb;
              if (S::kSwiGLU)  // W1 rows (half 2g) and W3 rows (half 2g + 1) of the feature tile
                tma_load_3d_tc(sb, mwb, &full[stage], kx, ti.ft * S::FPT,
                               ti.dense ? 0 : 2 * ti.g);
              else
                tma_load_2d(sb, mwb, &full[stage], kx, w_y);
            } else if (S::kSwiGLU) {
              tma_load_2d(sb, mw, &full[stage], kx, w_y);
              tma_load_2d(sb + kBoxBytes, mw, &full[stage], kx, w_y + u_off);
            } else {
#pragma unroll
              for (int j = 0; j < kBN / 128; ++j)
                tma_load_2d(sb + j * kBoxBytes, mw, &full[stage], kx, w_y + j * 128);
            }
          } else {
            // stacked tiles: the weight map's box is 64 rows, W3 lands in operand rows 64..127
            tma_load_2d(sa, mw, &full[stage], kx, w_y);
            if (S::kSwiGLU)
              tma_load_2d(sa + (S::kStack ? kBoxBytes / 2 : kBoxBytes), mw, &full[stage], kx,
                          w_y + u_off);
            tma_load_2d(sb, ma, &full[stage], ax, act_y);
          }
          }
          if (armed < S::STAGES) ++armed;
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // drain: wait (briefly) for the copies of the most recent stage uses to land (a pair's
        // copies all complete on the even CTA's barriers)
        for (int i = 0; i < armed; ++i) {
          if (stage == 0) {
            stage = S::STAGES;
            phase ^= 1u;
          }
          --stage;
          mbar_wait(&full[stage], phase, nullptr, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {  // a pair's MMAs are issued by its even CTA
      constexpr uint32_t kIdesc = idesc_bf16_f32<128, (kBN > 256 ? 256 : kBN)>();
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = tile0; tile < total && ok; tile += tstep) {
        const int ks = tile % p.ksplit;
        const TileInfo ti = decode_tile(tile / p.ksplit, tile_start, row_start, p.offsets,
                                        p.n_routed, p.dense_rows, p.dense_act_row0, S::RPT,
                                        p.dense_band);
        const int nkb_all = ti.dense ? nkb_d : nkb_r;
        const int kb0 = ks * nkb_all / p.ksplit, nkb = (ks + 1) * nkb_all / p.ksplit;
        // swap-AB tiles: the MMA's N is the tile's token count rounded up to 16, so a group's
        // last, partial tile costs only the tokens it holds
        uint32_t idesc = kIdesc;
        if constexpr (kSwap) {
          const int n = ti.valid >= kBN ? kBN : ((ti.valid + 15) & ~15);
          idesc = idesc_bf16_f32_n(n);
        }
        const bool half1 = kMH == 2 && ti.valid > 128;
        // the accumulator is free once both CTAs' epilogues have read it (a pair: arrivals from
        // the odd CTA, released at cluster scope)
        if (!(kPair ? mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, p.wait_ns)
                    : mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, p.wait_ns)))
          break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * S::ACC_COLS;
        for (int kb = kb0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE);
          const uint32_t sb = sa + S::OPA;
#pragma unroll
          for (int k16 = 0; k16 < kBK / 16; ++k16) {
            const uint32_t accum = ((kb - kb0) | k16) != 0;
            const uint64_t bdesc = sw128_kmajor_desc(sb + k16 * 32);
            if constexpr (kBN > 256) {  // N = 384: an N = 256 and an N = 128 MMA side by side
              const uint64_t adesc = sw128_kmajor_desc(sa + k16 * 32);
              mma_bf16(d0, adesc, bdesc, idesc_bf16_f32<128, 256>(), accum);
              mma_bf16(d0 + 256, adesc, sw128_kmajor_desc(sb + 2 * kBoxBytes + k16 * 32),
                       idesc_bf16_f32<128, kBN - 256>(), accum);
              continue;
            }
            if constexpr (kPair) {  // M = 256 over both CTAs' rows, N = 256 over both halves
              mma_bf16_pair(d0, sw128_kmajor_desc(sa + k16 * 32), bdesc, idesc_bf16_f32_pair(256),
                            accum);
              continue;
            }
            mma_bf16(d0, sw128_kmajor_desc(sa + k16 * 32), bdesc, idesc, accum);
            if (half1)  // the second 128 token rows against the same weight K-block
              mma_bf16(d0 + kBN, sw128_kmajor_desc(sa + kBoxBytes + k16 * 32), bdesc, idesc, accum);
            if (kSwap && S::kSwiGLU && !S::kStack)
              mma_bf16(d0 + kBN, sw128_kmajor_desc(sa + kBoxBytes + k16 * 32), bdesc, idesc,
                       accum);
          }
          if constexpr (kPair)
            mma_commit_pair(&empty[stage]);  // frees the stage in both CTAs
          else
            mma_commit(&empty[stage]);
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kPair)
          mma_commit_pair(&tfull[acc]);  // both CTAs' epilogues may read their rows
        else
          mma_commit(&tfull[acc]);
        if (S::NACC == 2) acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued above has completed once this commit arrives
      if constexpr (kPair)
        mma_commit_pair(drain);
      else
        mma_commit(drain);
      mbar_wait(drain, 0, nullptr, nullptr, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;       // TMEM lanes this warp may read: 32 * quarter + [0, 32)
    const int r = quarter * 32 + lane;  // tile row (rows) or tile feature (swap)
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = tile0; tile < total; tile += tstep) {
      const int ks = tile % p.ksplit;
      const TileInfo ti = decode_tile(tile / p.ksplit, tile_start, row_start, p.offsets,
                                      p.n_routed, p.dense_rows, p.dense_act_row0, S::RPT,
                                      p.dense_band);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err, p.wait_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // stacked tiles meet at a named barrier below: all four warps leave together or none does
      if (S::kStack) ok = named_barrier_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * S::ACC_COLS + ((uint32_t)(quarter * 32) << 16);
      // a pair: this CTA's accumulator holds the tile's rows 128 * rank .. +127
      const int64_t out_row0 = (ti.dense ? (int64_t)p.dense_out_row0 : (int64_t)ti.grp_row0) +
                               (int64_t)ti.rt * S::RPT + (kPair ? (int64_t)rank * 128 : 0) +
                               (int64_t)ks * p.split_rows;
      const int vt = kPair ? ti.valid - (int)rank * 128 : ti.valid;  // rows of this CTA's part
      void* const out = ti.dense ? p.out_d : p.out;
      const int64_t ldo = ti.dense ? p.ldo_d : p.ldo;
      if (!kSwap && S::kStaged) {
        uint8_t* buf = staging + (warp - 2) * 4096;
#pragma unroll 1
        for (int mh = 0; mh < kMH && mh * 128 < vt; ++mh) {
          const uint32_t th = tmem_base + acc * S::ACC_COLS + mh * kBN +
                              ((uint32_t)(quarter * 32) << 16);  // this M half's columns
          const int vrows = min(32, max(0, vt - mh * 128 - quarter * 32));
          const int64_t row0 = out_row0 + mh * 128 + quarter * 32;
          if (S::kSwiGLU) {  // h in bf16: chunks of 64 features = 128 bytes per row
#pragma unroll 1
            for (int c = 0; c < S::FPT; c += 64) {
              uint4 v[8];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t g0[16], u0[16], g1[16], u1[16];
                tmem_ld16(th + c + 32 * h, g0);
                tmem_ld16(th + S::FPT + c + 32 * h, u0);
                tmem_ld16(th + c + 32 * h + 16, g1);
                tmem_ld16(th + S::FPT + c + 32 * h + 16, u1);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  pk[i] = pack_bf16x2(
                      silu_fast(__uint_as_float(g0[2 * i])) * __uint_as_float(u0[2 * i]),
                      silu_fast(__uint_as_float(g0[2 * i + 1])) * __uint_as_float(u0[2 * i + 1]));
                  pk[8 + i] = pack_bf16x2(
                      silu_fast(__uint_as_float(g1[2 * i])) * __uint_as_float(u1[2 * i]),
                      silu_fast(__uint_as_float(g1[2 * i + 1])) * __uint_as_float(u1[2 * i + 1]));
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  v[4 * h + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
              }
              uint8_t* dst = (uint8_t*)out + (row0 * ldo + (int64_t)ti.ft * S::FPT + c) * 2;
              store_rows_128B(buf, lane, v, dst, ldo * 2, vrows);
            }
          } else if (p.out_f32) {  // fp32: chunks of 32 columns
#pragma unroll 1
            for (int c = 0; c < S::FPT; c += 32) {
              uint32_t a[16], b[16];
              tmem_ld16(th + c, a);
              tmem_ld16(th + c + 16, b);
              tmem_ld_wait();
              uint4 v[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                v[q] = make_uint4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
                v[4 + q] = make_uint4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
              }
              if (p.tma_out && vrows == 32) {
                // the chunk in the 128-byte swizzled layout; the TMA unswizzles it on the way out
                if (lane == 0) tma_store_wait_read();  // the previous chunk has left the buffer
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) = v[j];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) tma_store_2d_stream(&p.map_out, buf, ti.ft * S::FPT + c, (int)row0);
              } else {
                if (p.tma_out && lane == 0) tma_store_wait_read();
                __syncwarp();
                uint8_t* dst = (uint8_t*)out + (row0 * ldo + (int64_t)ti.ft * S::FPT + c) * 4;
                store_rows_128B(buf, lane, v, dst, ldo * 4, vrows);
              }
            }
          } else {  // bf16: chunks of 64 columns
#pragma unroll 1
            for (int c = 0; c < S::FPT; c += 64) {
              uint4 v[8];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t a[16], b[16];
                tmem_ld16(th + c + 32 * h, a);
                tmem_ld16(th + c + 32 * h + 16, b);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  pk[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                  pk[8 + i] = pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  v[4 * h + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
              }
              uint8_t* dst = (uint8_t*)out + (row0 * ldo + (int64_t)ti.ft * S::FPT + c) * 2;
              store_rows_128B(buf, lane, v, dst, ldo * 2, vrows);
            }
          }
        }
      } else if (!kSwap) {
        // store + fp32 addend (bf16 out): one row per thread
        const bool valid = r < ti.valid;
        const int64_t orow = out_row0 + r;
        const int64_t col0 = (int64_t)ti.ft * S::FPT;
#pragma unroll 1
        for (int c = 0; c < S::FPT; c += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c, v);
          tmem_ld_wait();
          if (valid) {
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
            if (kEpi == EPI_STORE_ADD) {
              const float4* a4 = reinterpret_cast<const float4*>(p.addend + orow * p.ld_add + col0 + c);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float4 av = __ldg(a4 + h);
                f[4 * h] += av.x;
                f[4 * h + 1] += av.y;
                f[4 * h + 2] += av.z;
                f[4 * h + 3] += av.w;
              }
            }
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
            uint4* d4 = reinterpret_cast<uint4*>((__nv_bfloat16*)out + orow * ldo + col0 + c);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else if constexpr (S::kStack) {
        // stacked SwiGLU: lanes 0..63 hold g = x W1 and lanes 64..127 u = x W3 of features
        // ft * 64 + (lane % 64); the pair meets in shared memory, 16 tokens at a time
        float* xch = reinterpret_cast<float*>(staging);
        const int t = threadIdx.x - 64;          // epilogue thread 0..127
        const int cf = t & 63, th = t >> 6;      // the feature and token half it computes
        float* mine = xch + r * 17;               // row r: (r >> 6 ? u : g) of feature r % 64
        const int64_t feat = (int64_t)ti.ft * 64 + cf;
#pragma unroll 1
        for (int c = 0; c < kBN && c < ti.valid; c += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) mine[i] = __uint_as_float(v[i]);
          named_barrier(1, 128);
          const float* gr = xch + cf * 17 + th * 8;
          const float* ur = xch + (64 + cf) * 17 + th * 8;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int tok = c + th * 8 + i;
            if (tok < ti.valid)
              ((__nv_bfloat16*)out)[(out_row0 + tok) * ldo + feat] =
                  __float2bfloat16_rn(silu_fast(gr[i]) * ur[i]);
          }
          named_barrier(1, 128);  // the buffer is read before the next chunk overwrites it
        }
      } else {
        // swap: TMEM lane = output feature, columns = tokens of this tile
        const int64_t feat = (int64_t)ti.ft * 128 + r;
#pragma unroll 1
        for (int c = 0; c < kBN && c < ti.valid; c += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tb + c, g);
          if (S::kSwiGLU) tmem_ld16(tb + kBN + c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (c + i < ti.valid) {
              const int64_t orow = out_row0 + c + i;
              float v = __uint_as_float(g[i]);
              if (S::kSwiGLU) v = silu_fast(v) * __uint_as_float(u[i]);
              if (p.out_f32) {
                ((float*)out)[orow * ldo + feat] = v;
              } else {
                if (kEpi == EPI_STORE_ADD) v += p.addend[orow * p.ld_add + feat];
                ((__nv_bfloat16*)out)[orow * ldo + feat] = __float2bfloat16_rn(v);
              }
            }
          }
        }
      }
      tc_fence_before();
      if constexpr (kPair)
        mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));  // the even CTA's accumulator barrier
      else
        mbar_arrive(&tempty[acc]);
      if (S::NACC == 2) acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  if (S::kStaged && p.tma_out && warp >= 2 && lane == 0) tma_store_wait_all();
  tc_fence_before();
  __syncthreads();
  // a pair: no arrival on the peer's barriers and no MMA into the peer's TMEM after this point
  if constexpr (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2D bf16 map over [rows][cols] (cols contiguous), box {64 cols, box_rows rows}, 128-byte swizzle,
// out-of-range elements read as zero.
bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                          int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base || rows <= 0 || cols <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 3D bf16 map over [halves][rows][cols] (halves rows apart), box {64 cols, 128 rows, 2 halves},
// 128-byte swizzle: one copy of the W1 rows of a feature tile and the matching W3 rows.
static bool make_map_bf16_3d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows,
                             int64_t halves) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base || rows <= 0 || cols <= 0 || halves < 2) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)halves};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)kBK, 128, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// fp32 output [rows][cols] for bulk stores of 32 x 32 chunks (128-byte swizzle in shared memory).
static bool make_map_f32_out(CUtensorMap* m, void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !base || rows <= 0 || cols <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kSwap, int kBN, int kEpi, int kMH = 1, bool kPair = false>
static cudaError_t launch_variant(const TcParams& p, int grid, cudaStream_t st, const char* label) {
  using S = TcShape<kSwap, kBN, kEpi, kMH, kPair>;
  auto kern = moe_gemm_tc_kernel<kSwap, kBN, kEpi, kMH, kPair>;
  static int attr_set_device = -1;  // the attribute is per device; refreshed when it changes
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_device != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    attr_set_device = dev;
  }
  LaunchScope ls(label, st);
  if constexpr (kPair) {  // clusters of two CTAs (one pair each), one CTA per SM
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(grid & ~1));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
  }
  kern<<<grid, kTcThreads, S::SMEM, st>>>(p);
  return cudaGetLastError();
}

bool gemm_tc_supported(const GroupedGemm& g, int swap) {
  if (g.act_dtype != MOE_BF16 || g.w_dtype != MOE_BF16) return false;
  if (g.K <= 0 || g.K % kBK) return false;
  if (g.K_d % kBK || (g.F_d && g.F_d % (g.epi == EPI_SWIGLU || swap ? 128 : 256))) return false;
  if (g.out_d && g.ldo_d % 8) return false;
  const int kw = g.k_wrap > 0 ? g.k_wrap : g.K;
  if (kw % kBK || g.K % kw) return false;
  if (g.n_routed > kTcMaxGroups - 1) return false;
  if (g.epi == EPI_SWIGLU) {
    if (g.F % 128) return false;
    if (g.out_dtype != MOE_BF16) return false;
  } else {
    if (g.F % (swap ? 128 : 256) && !(g.F % 128 == 0 && !swap && g.out_dtype == MOE_F32))
      return false;
  }
  if (g.ldo % 8) return false;
  if (g.epi == EPI_STORE_ADD && (!g.addend || g.ld_add % 4 || g.out_dtype != MOE_BF16))
    return false;
  return true;
}

cudaError_t launch_gemm_tc(const GroupedGemm& g, int swap, int num_sms, cudaStream_t st) {
  if (!gemm_tc_supported(g, swap)) return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const bool f32_router = !swap && g.epi == EPI_STORE && g.out_dtype == MOE_F32 && g.F % 256;
  if (g.n128 && g.epi == EPI_STORE && (g.F % 128 || (g.F_d && g.F_d % 128)))
    return cudaErrorInvalidValue;
  const int act_box = swap == 2 ? 256 : swap ? 32 : 128;
  const int w_box = swap == 2 && g.epi == EPI_SWIGLU ? 64 : 128;  // stacked W1 / W3 halves
  const int kw = g.k_wrap > 0 ? g.k_wrap : g.K;
  if (g.n_routed > 0) {
    if (!make_map_bf16(&p.map_act, g.act, g.act_rows, kw, act_box)) return cudaErrorInvalidValue;
    if (!make_map_bf16(&p.map_w, g.w, g.w_rows, g.K, w_box)) return cudaErrorInvalidValue;
  }
  const int K_d = g.K_d > 0 ? g.K_d : g.K;
  const int kw_d = g.k_wrap_d > 0 ? g.k_wrap_d : (g.K_d > 0 ? g.K_d : kw);
  if (g.dense_rows > 0) {
    if (!make_map_bf16(&p.map_act_d, g.act_d, g.act_d_rows, kw_d, act_box))
      return cudaErrorInvalidValue;
    if (!make_map_bf16(&p.map_w_d, g.w_d, g.w_d_rows, K_d, w_box)) return cudaErrorInvalidValue;
  }
  if (g.n_routed == 0) {  // keep the unused maps valid objects
    p.map_act = p.map_act_d;
    p.map_w = p.map_w_d;
  }
  if (g.dense_rows == 0) {
    p.map_act_d = p.map_act;
    p.map_w_d = p.map_w;
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
  p.k_wrap = kw;
  p.F = g.F;
  p.K_d = K_d;
  p.k_wrap_d = kw_d;
  p.F_d = g.F_d > 0 ? g.F_d : g.F;
  p.out = g.out;
  p.ldo = g.ldo;
  p.out_d = g.out_d ? g.out_d : g.out;
  p.ldo_d = g.out_d ? g.ldo_d : g.ldo;
  p.out_f32 = g.out_dtype == MOE_F32;
  // token-rows fp32 stores by TMA when every group writes the same tensor: its rows end at the
  // routed rows or at the dense group's last row, whichever is later
  if (!swap && g.epi == EPI_STORE && p.out_f32 && p.out_d == p.out && p.ldo_d == p.ldo &&
      g.ldo % 4 == 0 &&
      (reinterpret_cast<uintptr_t>(g.out) & 15) == 0) {
    const int64_t routed_end = g.n_routed > 0 ? g.act_rows : 0;
    const int64_t dense_end = g.dense_rows > 0 ? (int64_t)g.dense_out_row0 + g.dense_rows : 0;
    int64_t out_rows = routed_end > dense_end ? routed_end : dense_end;
    if (g.k_splits > 1 && g.ldo > 0)  // every partial
      out_rows = (int64_t)g.k_splits * (g.split_stride / g.ldo);
    if (out_rows > 0 && make_map_f32_out(&p.map_out, g.out, out_rows, g.ldo)) p.tma_out = 1;
  }
  p.addend = (const float*)g.addend;
  p.ld_add = g.ld_add;
  p.err = g.err;
  p.ksplit = 1;
  if (g.k_splits > 1) {
    // dense-only token-rows fp32 stores into one tensor; every K range at least one K-block;
    // the partials a whole number of rows apart, none overlapping the next
    if (swap || g.n_routed > 0 || g.epi != EPI_STORE || !p.out_f32 || g.pair || g.n128 ||
        g.out_d || g.k_splits > K_d / kBK || g.ldo <= 0 || g.split_stride % g.ldo ||
        g.split_stride / g.ldo < (int64_t)g.dense_out_row0 + g.dense_rows)
      return cudaErrorInvalidValue;
    p.ksplit = g.k_splits;
    p.split_rows = g.split_stride / g.ldo;
  }
  // Tile order of the dense group.  Activations that fit in L2 are re-read from there by every
  // feature tile (one band: the weights stream once).  Larger activations with weights that fit in
  // L2 stream once, row tile by row tile (the K3 down-projection: 117 MB of x, 51 MB of W_down;
  // the prefill shared expert: 235 MB of x, 58 MB of W1|W3).  When neither fits, bands of 16 row
  // tiles: the CTAs running at once then share 16 activation row tiles and about 152 / 16 weight
  // tiles, near the fewest distinct bytes in flight for 128 x 256 tiles.
  if (g.dense_rows > 0) {
    const int64_t act_bytes = (int64_t)g.dense_rows * K_d * 2;
    const int64_t w_bytes = (int64_t)p.F_d * (g.epi == EPI_SWIGLU ? 2 : 1) * K_d * 2;
    const int64_t l2_share = 48ll << 20;
    if (swap || act_bytes <= l2_share)
      p.dense_band = 0;
    else if (w_bytes <= 64ll << 20)
      p.dense_band = 1;
    else
      p.dense_band = 16;
  }
  // one weight box per stage for token-rows N = 256 tiles (not the pair / two-M-half variants)
  if (!swap && g.big_boxes && !g.pair && g.m_halves != 2 &&
      (g.epi == EPI_SWIGLU || (g.epi == EPI_STORE && !f32_router && !g.n128))) {
    bool ok = true;
    if (g.epi == EPI_SWIGLU) {
      // W1 | W3 stacked per expert: [groups * 2 halves][half rows][K]
      if (g.n_routed > 0)
        ok = ok && g.u_off % 128 == 0 && g.w_group_rows == 2 * g.u_off &&
             make_map_bf16_3d(&p.map_wb, g.w, g.K, g.u_off, g.w_rows / g.u_off);
      if (g.dense_rows > 0)
        ok = ok && g.u_off_d % 128 == 0 && g.w_d_rows == 2 * g.u_off_d &&
             make_map_bf16_3d(&p.map_wb_d, g.w_d, K_d, g.u_off_d, 2);
    } else {
      if (g.n_routed > 0) ok = ok && make_map_bf16(&p.map_wb, g.w, g.w_rows, g.K, 256);
      if (g.dense_rows > 0) ok = ok && make_map_bf16(&p.map_wb_d, g.w_d, g.w_d_rows, K_d, 256);
    }
    if (ok) {
      if (g.n_routed == 0) p.map_wb = p.map_wb_d;
      if (g.dense_rows == 0) p.map_wb_d = p.map_wb;
      p.big_boxes = 1;
    }
  }
  p.test_stall = g.test_stall ? 1 : 0;
  p.wait_ns = g.test_stall ? 50000000ull : kWaitLimitNs;
  const int grid = num_sms;
  if (!swap) {
    if (g.epi == EPI_SWIGLU) {
      // two M halves per tile only on request: measured slower at prefill (gemm13 6.6 -> 8.1 ms)
      // and K3 (2.4 -> 3.1 ms), the SwiGLU epilogue no longer hidden behind the next mainloop
      if (g.m_halves == 2) return launch_variant<false, 256, EPI_SWIGLU, 2>(p, grid, st, g.label);
      if (g.pair) return launch_variant<false, 256, EPI_SWIGLU, 1, true>(p, grid, st, g.label);
      return launch_variant<false, 256, EPI_SWIGLU>(p, grid, st, g.label);
    }
    if (g.pair && g.epi == EPI_STORE && !f32_router && !g.n128)
      return launch_variant<false, 256, EPI_STORE, 1, true>(p, grid, st, g.label);
    if (f32_router && g.F % 384 == 0) return launch_variant<false, 384, EPI_STORE>(p, grid, st, g.label);
    if (f32_router || (g.n128 && g.epi == EPI_STORE))
      return launch_variant<false, 128, EPI_STORE>(p, grid, st, g.label);
    if (g.epi == EPI_STORE) return launch_variant<false, 256, EPI_STORE>(p, grid, st, g.label);
    return launch_variant<false, 256, EPI_STORE_ADD>(p, grid, st, g.label);
  }
  if (swap == 2) {  // 256-token tiles (the MMA's N follows each tile's token count)
    if (g.epi == EPI_SWIGLU) return launch_variant<true, 256, EPI_SWIGLU>(p, grid, st, g.label);
    if (g.epi == EPI_STORE) return launch_variant<true, 256, EPI_STORE>(p, grid, st, g.label);
    return cudaErrorInvalidValue;
  }
  if (g.epi == EPI_SWIGLU) return launch_variant<true, 32, EPI_SWIGLU>(p, grid, st, g.label);
  if (g.epi == EPI_STORE) return launch_variant<true, 32, EPI_STORE>(p, grid, st, g.label);
  return launch_variant<true, 32, EPI_STORE_ADD>(p, grid, st, g.label);
}

}  // namespace moe
