// decode_fused.cu -- the decode experts in one persistent launch.
//
// "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps g = x W1,
// u = x W3, a = g sigma(g), h = a * u, E_i = h W2, for every routed expert and the shared expert:
// phase 1 computes h in 128-feature x 32-token tiles (the W1 and W3 rows of the same features
// against the tile's tokens), phase 2 the expert outputs in 128-feature x 32-token tiles of W2
// against h.  Both phases stream their weights once; the kernel is HBM-bound like the two
// swap-AB launches it replaces, and what it removes is the boundary between them: the last wave
// of W1|W3 tiles no longer waits for the slowest CTA, and W2 needs no second launch or pipeline
// fill.
//
// Order and waits.  Every CTA takes tiles blockIdx.x, blockIdx.x + gridDim.x, ... of one list:
// all phase-1 tiles, then all phase-2 tiles.  A phase-2 tile needs the h rows of its row tile,
// i.e. the I/128 phase-1 tiles of that row tile, which come earlier in the list; each of those
// counts itself in `ready[row tile]` once its h values are written, and the copy producer of the
// phase-2 tile waits (bounded) for the count before it loads h.  A CTA reaches a phase-2 tile only
// after its own phase-1 tiles, so with every CTA resident at once (a cooperative launch of one CTA
// per SM) no wait can depend on a CTA that is itself waiting.
//
// Measured on the K2 decode batch (128 tokens, 384 experts): 3.21 ms against 1.99 + 1.01 ms for
// the two launches, with identical outputs.  Phase 1 alone runs as fast as the stand-alone W1|W3
// launch, and phase 2 alone, with no wait at all, takes 1.23 ms against 1.01 for the same W2 tiles
// in their own launch; neither the waits, the fences nor the stage ring account for it.  The
// library therefore runs it only on request (MOE_FLAG_DECODE_FUSED).
//
// Warp roles as in the grouped GEMM (gemm_tc.cu): warp 0 copies (TMA), warp 1 issues tcgen05.mma
// (M = 128 weight rows, N = the tile's tokens rounded up to 16, fp32 accumulators in TMEM), warps
// 2..5 run the epilogues.  Every wait is bounded; on expiry the kernel flags kErrTimeout, drains
// its copies and MMAs, frees TMEM and returns.
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "sched.cuh"

namespace moe {

constexpr int kFdThreads = 192;
constexpr int kFdBK = 64;                       // K elements per stage (one 128-byte row)
constexpr int kFdTok = 32;                      // tokens per tile (the MMA's N at most)
constexpr int kFdFeat = 128;                    // output features per tile (the MMA's M)
constexpr int kFdBox = 128 * 128;               // 128 weight rows x 128 bytes
constexpr int kFdTokBox = kFdTok * 128;         // 32 token rows x 128 bytes
// Two stage rings over the same shared memory, one per phase, so that each phase keeps as many
// bytes in flight as fit: phase 1 stages hold a W1 box, a W3 box and the tokens (36 KB), phase 2
// stages a W2 box and the h tokens (20 KB).  An HBM stream of about 45 GB/s per SM with a few
// microseconds of latency needs well over 120 KB in flight, which six 20 KB W2 stages in the
// phase-1 ring would not give.  A CTA switches rings once, after its last phase-1 copies have
// been consumed.
constexpr int kFdStage1 = 2 * kFdBox + kFdTokBox;
constexpr int kFdStage2 = kFdBox + kFdTokBox;
constexpr int kFdMaxGroups = 1025;
constexpr int kFdTable = 2 * (kFdMaxGroups + 1) * 4 + kFdThreads * 4;
constexpr int kFdBars = 512;
constexpr int kFdRing = 232448 - 1024 - kFdTable - kFdBars;  // bytes for either ring
constexpr int kFdStages1 = kFdRing / kFdStage1;
constexpr int kFdStages2 = kFdRing / kFdStage2 < 12 ? kFdRing / kFdStage2 : 12;
constexpr int kFdRingUsed =
    kFdStages1 * kFdStage1 > kFdStages2 * kFdStage2 ? kFdStages1 * kFdStage1 : kFdStages2 * kFdStage2;
constexpr int kFdSmem = 1024 + kFdRingUsed + kFdBars + kFdTable;
constexpr int kFdAcc = 2 * kFdTok;  // columns of one accumulator: g (W1) then u (W3) in phase 1
constexpr int kFdTmemCols = 128;    // two accumulators
static_assert(kFdStages1 >= 4 && kFdStages2 >= 8, "stage rings");
static_assert(2 * (kFdStages1 + kFdStages2) + 5 + 1 <= kFdBars / 8, "barrier area");
static_assert(kFdStage1 % 1024 == 0 && kFdStage2 % 1024 == 0,
              "stages keep 1024-byte alignment for the 128-byte swizzle");
static_assert(kFdSmem <= 232448, "shared memory");

struct FdParams {
  CUtensorMap map_x;      // x_perm [P][d]      box {64, 32}
  CUtensorMap map_x_d;    // x [T][d]           box {64, 32}
  CUtensorMap map_w13;    // W13 [E * 2I][d]    box {64, 128}
  CUtensorMap map_w13_d;  // Ws13 [2I][d]
  CUtensorMap map_h;      // h [P + T][I]       box {64, 32}
  CUtensorMap map_w2;     // W2 [E * d][I]      box {64, 128}
  CUtensorMap map_w2_d;   // Ws2 [d][I]
  const int32_t* offsets;
  int32_t n_routed, dense_rows, d, I, P;
  __nv_bfloat16* h;
  float* y;
  uint32_t* ready;
  uint32_t* err;
  uint64_t wait_ns;
};

// Phase-2 tile -> group, row tile, feature tile: the groups and row tiles of phase 1 with d/128
// feature tiles per row tile instead of I/128, so group g's tiles start at
// tile_start1[g] / nft1 * nft2 (a group's phase-1 tile count is a multiple of nft1).
__device__ __forceinline__ TileInfo decode_phase2(int t2, const int* tile_start1,
                                                  const int* row_start, int n_routed,
                                                  int dense_rows, int nft1, int nft2) {
  const int G = n_routed + (dense_rows > 0 ? 1 : 0);
  int lo = 0, hi = G - 1;  // the largest g whose tiles start at or before t2
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start1[mid] / nft1 * nft2 <= t2)
      lo = mid;
    else
      hi = mid - 1;
  }
  TileInfo ti;
  ti.g = lo;
  ti.dense = lo == n_routed ? 1 : 0;
  if (ti.dense) {
    ti.rows = dense_rows;
    ti.grp_row0 = 0;
  } else {
    ti.grp_row0 = row_start[lo];
    ti.rows = row_start[lo + 1] - ti.grp_row0;
  }
  const int nrt = (ti.rows + kFdTok - 1) / kFdTok;
  const int local = t2 - tile_start1[lo] / nft1 * nft2;
  ti.ft = local / nrt;
  ti.rt = local - ti.ft * nrt;
  ti.valid = min(kFdTok, ti.rows - ti.rt * kFdTok);
  return ti;
}

// Waits (bounded) until *cnt >= target, with acquire semantics at GPU scope, then orders the
// caller's later async-proxy (TMA) reads after it.  False on expiry (kErrTimeout raised, *abort
// set) or when another warp has set *abort.
__device__ __forceinline__ bool wait_ready(const uint32_t* cnt, uint32_t target,
                                           volatile int* abort, uint32_t* err, uint64_t limit_ns) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
  if (v < target) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      __nanosleep(128);
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= target) break;
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        raise_flag(err, kErrTimeout);
        return false;
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__global__ void __launch_bounds__(kFdThreads, 1) decode_fused_kernel(const __grid_constant__ FdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFdRingUsed);
  uint64_t* full1 = bars;  // phase-1 ring
  uint64_t* empty1 = full1 + kFdStages1;
  uint64_t* full2 = empty1 + kFdStages1;  // phase-2 ring
  uint64_t* empty2 = full2 + kFdStages2;
  uint64_t* tfull = empty2 + kFdStages2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* tile_start = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + kFdBars);
  int* row_start = tile_start + (kFdMaxGroups + 1);
  int* scratch = row_start + (kFdMaxGroups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFdStages1; ++s) {
      mbar_init(&full1[s], 1);
      mbar_init(&empty1[s], 1);
    }
    for (int s = 0; s < kFdStages2; ++s) {
      mbar_init(&full2[s], 1);
      mbar_init(&empty2[s], 1);
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
    tma_prefetch_map(&p.map_x);
    tma_prefetch_map(&p.map_w13);
    tma_prefetch_map(&p.map_h);
    tma_prefetch_map(&p.map_w2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kFdTmemCols);
    tmem_relinquish();
  }
  const int nft1 = p.I / kFdFeat, nft2 = p.d / kFdFeat;
  build_tile_table(tile_start, row_start, scratch, p.offsets, p.n_routed, p.dense_rows, kFdTok,
                   nft1);  // ends with __syncthreads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int G = p.n_routed + (p.dense_rows > 0 ? 1 : 0);
  const int total1 = tile_start[G];
  const int total = total1 + total1 / nft1 * nft2;
  const int nkb1 = p.d / kFdBK, nkb2 = p.I / kFdBK;

  auto tile_at = [&](int tile) -> TileInfo {
    return tile < total1 ? decode_tile(tile, tile_start, row_start, p.offsets, p.n_routed,
                                       p.dense_rows, 0, kFdTok)
                         : decode_phase2(tile - total1, tile_start, row_start, p.n_routed,
                                         p.dense_rows, nft1, nft2);
  };
  // first row of the tile in h / y (the shared expert's rows follow the P routed rows)
  auto row0_of = [&](const TileInfo& ti) -> int64_t {
    return (ti.dense ? (int64_t)p.P : (int64_t)ti.grp_row0) + (int64_t)ti.rt * kFdTok;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int armed = 0;  // fills of the current ring (for the drain after an abort)
      bool ring2 = false, ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const bool p2 = tile >= total1;
        const TileInfo ti = tile_at(tile);
        if (p2 && !ring2) {
          // the phase-2 ring overlays the phase-1 ring: wait until the MMA has released the last
          // phase-1 fill (it releases in order), then start the phase-2 ring at its first stage
          if (armed > 0) {
            const uint32_t ls = stage == 0 ? kFdStages1 - 1 : stage - 1;
            const uint32_t lp = stage == 0 ? phase ^ 1u : phase;
            if (!mbar_wait(&empty1[ls], lp, abort_flag, p.err, p.wait_ns)) break;
          }
          ring2 = true;
          stage = phase = 0;
          armed = 0;
        }
        if (p2) {
          // h of this row tile is complete once its nft1 phase-1 tiles have counted themselves
          const int unit = tile_start[ti.g] / nft1 + ti.rt;
          if (!wait_ready(p.ready + unit, (uint32_t)nft1, abort_flag, p.err, p.wait_ns)) break;
        }
        const int nkb = p2 ? nkb2 : nkb1;
        const int nst = p2 ? kFdStages2 : kFdStages1;
        uint64_t* const full = p2 ? full2 : full1;
        uint64_t* const empty = p2 ? empty2 : empty1;
        const int64_t row0 = row0_of(ti);
        const int act_y = p2 ? (int)row0
                             : (ti.dense ? 0 : ti.grp_row0) + ti.rt * kFdTok;  // x or x_perm
        const int w_y = p2 ? (ti.dense ? 0 : ti.g * p.d) + ti.ft * kFdFeat
                           : (ti.dense ? 0 : ti.g * 2 * p.I) + ti.ft * kFdFeat;
        const CUtensorMap* mw = p2 ? (ti.dense ? &p.map_w2_d : &p.map_w2)
                                   : (ti.dense ? &p.map_w13_d : &p.map_w13);
        const CUtensorMap* ma = p2 ? &p.map_h : (ti.dense ? &p.map_x_d : &p.map_x);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * (p2 ? kFdStage2 : kFdStage1);
          uint8_t* sb = sa + (p2 ? kFdBox : 2 * kFdBox);
          const int kx = kb * kFdBK;
          mbar_arrive_expect_tx(&full[stage], p2 ? kFdStage2 : kFdStage1);
          tma_load_2d(sa, mw, &full[stage], kx, w_y);
          if (!p2) tma_load_2d(sa + kFdBox, mw, &full[stage], kx, w_y + p.I);  // W3 rows
          tma_load_2d(sb, ma, &full[stage], kx, act_y);
          if (armed < nst) ++armed;
          if (++stage == (uint32_t)nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        // drain: wait (briefly) for the copies of the most recent stage uses to land
        const int nst = ring2 ? kFdStages2 : kFdStages1;
        uint64_t* const full = ring2 ? full2 : full1;
        for (int i = 0; i < armed; ++i) {
          if (stage == 0) {
            stage = nst;
            phase ^= 1u;
          }
          --stage;
          mbar_wait(&full[stage], phase, nullptr, nullptr, kDrainLimitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true, ring2 = false;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const bool p2 = tile >= total1;
        const TileInfo ti = tile_at(tile);
        if (p2 && !ring2) {  // every phase-1 stage has been consumed: the phase-2 ring starts
          ring2 = true;
          stage = phase = 0;
        }
        const int nkb = p2 ? nkb2 : nkb1;
        const int nst = p2 ? kFdStages2 : kFdStages1;
        uint64_t* const full = p2 ? full2 : full1;
        uint64_t* const empty = p2 ? empty2 : empty1;
        const uint32_t idesc = idesc_bf16_f32_n((ti.valid + 15) & ~15);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.err, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc * kFdAcc;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * (p2 ? kFdStage2 : kFdStage1));
          const uint32_t sb = sa + (p2 ? kFdBox : 2 * kFdBox);
#pragma unroll
          for (int k16 = 0; k16 < kFdBK / 16; ++k16) {
            const uint32_t accum = (kb | k16) != 0;
            const uint64_t bdesc = sw128_kmajor_desc(sb + k16 * 32);
            mma_bf16(d0, sw128_kmajor_desc(sa + k16 * 32), bdesc, idesc, accum);
            if (!p2)  // u = x W3 beside g = x W1
              mma_bf16(d0 + kFdTok, sw128_kmajor_desc(sa + kFdBox + k16 * 32), bdesc, idesc, accum);
          }
          mma_commit(&empty[stage]);
          if (++stage == (uint32_t)nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      mma_commit(drain);  // arrives once every MMA issued above has completed
      mbar_wait(drain, 0, nullptr, nullptr, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;       // TMEM lanes 32 * quarter + [0, 32)
    const int r = quarter * 32 + lane;  // the tile's feature this thread holds
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const bool p2 = tile >= total1;
      const TileInfo ti = tile_at(tile);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err, p.wait_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ok = named_barrier_and(1, 128, ok);  // the four warps leave together or not at all
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * kFdAcc + ((uint32_t)(quarter * 32) << 16);
      const int64_t row0 = row0_of(ti);
      const int64_t feat = (int64_t)ti.ft * kFdFeat + r;
      if (!p2) {
#pragma unroll 1
        for (int c = 0; c < ti.valid; c += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tb + c, g);
          tmem_ld16(tb + kFdTok + c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < ti.valid)
              p.h[(row0 + c + i) * p.I + feat] =
                  __float2bfloat16_rn(silu_fast(__uint_as_float(g[i])) * __uint_as_float(u[i]));
        }
        // publish: this thread's h values are visible to every CTA's copies (async proxy) before
        // the tile is counted; the count is released once all four warps have stored
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        named_barrier(2, 128);
        if (threadIdx.x == 64) {
          const int unit = tile_start[ti.g] / nft1 + ti.rt;
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.ready + unit) : "memory");
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < ti.valid; c += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < ti.valid) p.y[(row0 + c + i) * p.d + feat] = __uint_as_float(v[i]);
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
    tmem_dealloc(tmem_base, kFdTmemCols);
  }
}

int64_t fused_ready_count(int64_t T, int k, int E) {
  // row tiles: at most P / 32 + E over the routed groups (each adds at most one partial tile),
  // plus ceil(T / 32) for the shared expert
  return T * k / kFdTok + E + (T + kFdTok - 1) / kFdTok + 1;
}

cudaError_t launch_decode_fused(const FusedDecode& f, int num_sms, cudaStream_t st) {
  if (f.d % kFdFeat || f.I % kFdFeat || f.n_routed < 1 || f.n_routed > kFdMaxGroups - 1)
    return cudaErrorInvalidValue;
  if (f.P < 1 || f.P + f.T >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  FdParams p;
  memset(&p, 0, sizeof(p));
  const int64_t E = f.n_routed;
  const int64_t rows_h = f.P + f.T;
  if (!make_map_bf16(&p.map_x, f.x_perm, f.P, f.d, kFdTok) ||
      !make_map_bf16(&p.map_w13, f.W13, E * 2 * f.I, f.d, kFdFeat) ||
      !make_map_bf16(&p.map_h, f.h, rows_h, f.I, kFdTok) ||
      !make_map_bf16(&p.map_w2, f.W2, E * f.d, f.I, kFdFeat))
    return cudaErrorInvalidValue;
  if (f.T > 0) {
    if (!make_map_bf16(&p.map_x_d, f.x, f.T, f.d, kFdTok) ||
        !make_map_bf16(&p.map_w13_d, f.Ws13, 2 * (int64_t)f.I, f.d, kFdFeat) ||
        !make_map_bf16(&p.map_w2_d, f.Ws2, f.d, f.I, kFdFeat))
      return cudaErrorInvalidValue;
  } else {  // keep the unused maps valid objects
    p.map_x_d = p.map_x;
    p.map_w13_d = p.map_w13;
    p.map_w2_d = p.map_w2;
  }
  p.offsets = f.offsets;
  p.n_routed = f.n_routed;
  p.dense_rows = (int)f.T;
  p.d = f.d;
  p.I = f.I;
  p.P = (int)f.P;
  p.h = static_cast<__nv_bfloat16*>(f.h);
  p.y = f.y;
  p.ready = f.ready;
  p.err = f.err;
  p.wait_ns = kWaitLimitNs;

  static int attr_set_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFdSmem);
    if (e != cudaSuccess) return e;
    attr_set_device = dev;
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kFdThreads);
  cfg.dynamicSmemBytes = kFdSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once (the W2 tiles wait)
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchScope ls(f.label, st);
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel, p);
}

}  // namespace moe
