// sched.cuh -- tile schedule of a grouped GEMM whose group sizes live on the device.
//
// Groups 0..n_routed-1 are the routed experts; their rows are the permuted (token, slot) rows
// [offsets[g], offsets[g+1]).  An optional trailing "dense" group (the shared expert, or a plain
// dense GEMM) has dense_rows rows.  Every group is cut into row tiles of RPT rows and feature tiles
// of FPT output features; a group's tiles are numbered feature-tile-major, row-tile-minor, so that
// consecutive tile numbers (run at the same time by neighbouring CTAs) share one weight tile and
// the weights stream from HBM once.  The dense group may instead be numbered in bands of
// `dense_band` row tiles, feature-tile-major inside a band: a projection of every token of a large
// batch has more activation bytes than fit in L2, and with bands the running CTAs share both a few
// activation row tiles and a few weight tiles (a band of one row tile is row-tile-major order: the
// activations stream from HBM once and a weight matrix that fits in L2 is re-read from there).
#pragma once

#include <stdint.h>

namespace moe {

struct TileInfo {
  int g;          // group
  int dense;      // 1 for the trailing dense group
  int rows;       // rows of the group
  int rt;         // row tile within the group
  int ft;         // feature tile
  int valid;      // rows of this tile inside the group (1..RPT)
  int grp_row0;   // first row of the group in the routed (permuted) row space, or dense_act_row0
};

// Block-wide: fills tile_start[0..G] (exclusive prefix of tiles per group) and row_start[0..G]
// (row_start[g] = offsets[g] for the routed groups g <= n_routed, so that a routed group's row count
// is row_start[g+1] - row_start[g] without touching global memory again).  Ends with
// __syncthreads(); tile_start[G] is the total number of tiles.
__device__ __forceinline__ void build_tile_table(int* tile_start, int* row_start,
                                                 int* scratch /* blockDim.x ints */,
                                                 const int32_t* offsets, int n_routed,
                                                 int dense_rows, int rpt, int feat_tiles,
                                                 int feat_tiles_d = -1) {
  const int G = n_routed + (dense_rows > 0 ? 1 : 0);
  const int nt = blockDim.x;
  const int per = (G + nt - 1) / nt;
  const int lo = threadIdx.x * per;
  const int hi = min(G, lo + per);
  int local = 0;
  for (int g = lo; g < hi; ++g) {
    int rows, r0;
    if (g < n_routed) {
      r0 = offsets[g];
      rows = offsets[g + 1] - r0;
    } else {
      r0 = 0;
      rows = dense_rows;
    }
    rows = rows < 0 ? 0 : rows;
    if (g < n_routed) row_start[g] = r0;  // the dense group's entry is never read
    if (g == n_routed - 1) row_start[n_routed] = offsets[n_routed];
    const int ft = (g < n_routed || feat_tiles_d < 0) ? feat_tiles : feat_tiles_d;
    const int t = ((rows + rpt - 1) / rpt) * ft;
    tile_start[g] = t;  // count for now
    local += t;
  }
  scratch[threadIdx.x] = local;
  __syncthreads();
  // inclusive Hillis-Steele scan of the per-thread sums
  for (int off = 1; off < nt; off <<= 1) {
    const int v = threadIdx.x >= off ? scratch[threadIdx.x - off] : 0;
    __syncthreads();
    scratch[threadIdx.x] += v;
    __syncthreads();
  }
  int run = scratch[threadIdx.x] - local;  // exclusive prefix of this thread's range
  for (int g = lo; g < hi; ++g) {
    const int t = tile_start[g];
    tile_start[g] = run;
    run += t;
  }
  if (threadIdx.x == nt - 1) tile_start[G] = scratch[nt - 1];
  __syncthreads();
}

__device__ __forceinline__ TileInfo decode_tile(int tile, const int* tile_start,
                                                const int* row_start, const int32_t* offsets,
                                                int n_routed, int dense_rows, int dense_row0,
                                                int rpt, int dense_band = 0) {
  const int G = n_routed + (dense_rows > 0 ? 1 : 0);
  int lo = 0, hi = G - 1;  // largest g with tile_start[g] <= tile (empty groups share starts)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile)
      lo = mid;
    else
      hi = mid - 1;
  }
  TileInfo ti;
  ti.g = lo;
  ti.dense = (lo == n_routed) ? 1 : 0;
  if (ti.dense) {
    ti.rows = dense_rows;
    ti.grp_row0 = dense_row0;
  } else {
    ti.grp_row0 = row_start[lo];
    ti.rows = row_start[lo + 1] - ti.grp_row0;
  }
  const int nrt = (ti.rows + rpt - 1) / rpt;
  const int local = tile - tile_start[lo];
  if (ti.dense && dense_band > 0 && dense_band < nrt) {
    const int nft = (tile_start[G] - tile_start[lo]) / nrt;  // the dense group is the last
    const int band = local / (dense_band * nft);
    const int rem = local - band * dense_band * nft;
    const int in_band = min(dense_band, nrt - band * dense_band);  // the last band may be short
    ti.ft = rem / in_band;
    ti.rt = band * dense_band + (rem - ti.ft * in_band);
  } else {
    ti.ft = local / nrt;
    ti.rt = local - ti.ft * nrt;
  }
  ti.valid = min(rpt, ti.rows - ti.rt * rpt);
  return ti;
}

}  // namespace moe
