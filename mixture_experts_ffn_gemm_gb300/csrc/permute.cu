// permute.cu -- dispatch bookkeeping: group the (token, slot) pairs by expert.
//
// "Kimi K3 · Latent up-projection", `moe_infer` code excerpt: count tokens per expert, sort the
// flattened top-k expert ids, gather the token rows in that order (then, per expert, run its MLP).
// Here the sort is a stable counting sort done in three kernels, with no host synchronisation:
//   1. count:   per chunk of pairs, a shared-memory histogram over experts -> chunk_counts[c][e]
//   2. scan:    per expert, exclusive prefix over chunks; counts[e]; offsets = exclusive prefix of
//               counts over experts (the shared expert appended as group E with T*n_shared rows)
//   3. scatter: per chunk, one warp walks the pairs in order; lanes with the same expert get
//               consecutive slots (__match_any_sync ranks), so each expert's rows stay in
//               increasing pair order -- a deterministic layout.
// The scatter copies token rows into the permuted order (16-byte vectors), token by token.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kChunk = 1024;     // pairs per chunk
constexpr int kMaxExperts = 1024;

int permute_chunks(int64_t P) { return (int)((P + kChunk - 1) / kChunk); }

__global__ void __launch_bounds__(256)
    permute_count_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                         int32_t* __restrict__ chunk_counts, uint32_t* err) {
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t p0 = (int64_t)blockIdx.x * kChunk;
  const int64_t p1 = min(P, p0 + kChunk);
  bool bad = false;
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = idx[p];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      bad = true;
  }
  if (bad) raise_flag(err, kErrIndex);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

__global__ void __launch_bounds__(1024)
    permute_scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E, int64_t P,
                        int64_t shared_rows, int32_t* __restrict__ counts,
                        int32_t* __restrict__ offsets) {
  __shared__ int sc[1024];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = chunk_counts[(int64_t)c * E + e];
      chunk_counts[(int64_t)c * E + e] = run;  // rows of expert e in the chunks before c
      run += v;
    }
    counts[e] = run;
  }
  sc[e] = (e < E) ? run : 0;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan over experts
    const int v = e >= off ? sc[e - off] : 0;
    __syncthreads();
    sc[e] += v;
    __syncthreads();
  }
  if (e < E) offsets[e] = sc[e] - run;
  if (e == 0) {
    counts[E] = (int32_t)shared_rows;
    offsets[E] = (int32_t)P;
    offsets[E + 1] = (int32_t)(P + shared_rows);
  }
}

__global__ void __launch_bounds__(32)
    permute_scatter_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                           const int32_t* __restrict__ chunk_counts,
                           const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
                           int32_t* __restrict__ perm_dst) {
  __shared__ int base[kMaxExperts];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32)
    base[e] = offsets[e] + chunk_counts[(int64_t)blockIdx.x * E + e];
  __syncwarp();
  const int64_t p0 = (int64_t)blockIdx.x * kChunk;
  const int64_t p1 = min(P, p0 + kChunk);
  const uint32_t lt = (1u << lane) - 1u;
  // the chunk's expert ids, all loaded before the in-order walk (no load latency per step)
  int ids[kChunk / 32];
#pragma unroll
  for (int i = 0; i < kChunk / 32; ++i) {
    const int64_t p = p0 + i * 32 + lane;
    int e = -2;  // -2: lane past the chunk end
    if (p < p1) {
      e = idx[p];
      if (e < 0 || e >= E) e = -1;  // out of range: skipped (the count kernel raised the flag)
    }
    ids[i] = e;
  }
#pragma unroll
  for (int i = 0; i < kChunk / 32; ++i) {
    const int64_t q = p0 + i * 32;
    if (q >= p1) break;  // warp-uniform
    const int64_t p = q + lane;
    const int e = ids[i];
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    const int leader = __ffs(peers) - 1;
    int pos = 0;
    if (e >= 0) pos = base[e] + rank;
    __syncwarp();
    if (e >= 0 && lane == leader) base[e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      perm_src[pos] = (int32_t)p;
      perm_dst[p] = pos;
    } else if (e == -1) {
      perm_dst[p] = -1;
    }
  }
}

// All P <= kChunk pairs in one CTA of 1024 threads: the count, the scan and the ordered walk of
// the three kernels above, without their launch gaps (decode batches).  Same result.
__global__ void __launch_bounds__(1024)
    permute_small_kernel(const int32_t* __restrict__ idx, int P, int E, int64_t shared_rows,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ perm_src, int32_t* __restrict__ perm_dst,
                         uint32_t* err) {
  __shared__ int hist[kMaxExperts];
  __shared__ int sc[1024];
  const int tid = threadIdx.x;
  for (int e = tid; e < kMaxExperts; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  int my_e = -2;  // this thread's pair: -2 none, -1 out of range
  if (tid < P) {
    my_e = idx[tid];
    if (my_e >= 0 && my_e < E)
      atomicAdd(&hist[my_e], 1);
    else
      my_e = -1;
  }
  if (my_e == -1) raise_flag(err, kErrIndex);
  __syncthreads();
  const int run = tid < E ? hist[tid] : 0;
  sc[tid] = run;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan over experts
    const int v = tid >= off ? sc[tid - off] : 0;
    __syncthreads();
    sc[tid] += v;
    __syncthreads();
  }
  if (tid < E) {
    counts[tid] = run;
    offsets[tid] = sc[tid] - run;
    hist[tid] = sc[tid] - run;  // from here: the next free row of expert tid
  }
  if (tid == 0) {
    counts[E] = (int32_t)shared_rows;
    offsets[E] = P;
    offsets[E + 1] = (int32_t)(P + shared_rows);
  }
  __syncthreads();
  if (tid >= 32) return;
  // warp 0 walks the pairs in order; lanes with the same expert take consecutive rows
  const int lane = tid;
  const uint32_t lt = (1u << lane) - 1u;
  for (int q = 0; q < P; q += 32) {
    const int p = q + lane;
    int e = -2;
    if (p < P) {
      e = idx[p];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    const int leader = __ffs(peers) - 1;
    int pos = 0;
    if (e >= 0) pos = hist[e] + rank;
    __syncwarp();
    if (e >= 0 && lane == leader) hist[e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      perm_src[pos] = p;
      perm_dst[p] = pos;
    } else if (e == -1) {
      perm_dst[p] = -1;
    }
  }
}

cudaError_t launch_permute(const int32_t* idx, int64_t T, int k, int E, int n_shared,
                           int32_t* chunk_counts, int32_t* counts, int32_t* offsets,
                           int32_t* perm_src, int32_t* perm_dst, uint32_t* err, cudaStream_t st) {
  if (E > kMaxExperts - 1) return cudaErrorInvalidValue;
  const int64_t P = T * k;
  const int nchunks = permute_chunks(P);
  if (P > 0 && P <= kChunk) {
    LaunchScope ls("permute_small", st);
    permute_small_kernel<<<1, 1024, 0, st>>>(idx, (int)P, E, T * n_shared, counts, offsets,
                                             perm_src, perm_dst, err);
    return cudaGetLastError();
  }
  if (nchunks > 0) {
    LaunchScope ls("permute_count", st);
    permute_count_kernel<<<nchunks, 256, 0, st>>>(idx, P, E, chunk_counts, err);
  }
  {
    LaunchScope ls("permute_scan", st);
    permute_scan_kernel<<<1, 1024, 0, st>>>(chunk_counts, nchunks, E, P, T * n_shared, counts,
                                            offsets);
  }
  if (nchunks > 0) {
    LaunchScope ls("permute_scatter", st);
    permute_scatter_kernel<<<nchunks, 32, 0, st>>>(idx, P, E, chunk_counts, offsets, perm_src,
                                                   perm_dst);
  }
  return cudaGetLastError();
}

// dst[perm_dst[t*k + j]][:] = src[t][:] for every token t and slot j: each source row is read
// once and written k times, where a copy in permuted-row order reads every row k times (the K2
// prefill x, 235 MB, is larger than L2, so those reads reach DRAM).  A pair whose destination is
// outside [0, P) (a skipped, out-of-range expert index) is not written; neither are the rows it
// would have filled, which lie past every expert's group.
__global__ void __launch_bounds__(256)
    scatter_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ perm_dst,
                        int64_t T, int k, int64_t P, int vec_per_row, uint4* __restrict__ dst) {
  __shared__ int64_t rows[32];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      const int r = perm_dst[t * k + threadIdx.x];
      rows[threadIdx.x] = (r >= 0 && r < P) ? (int64_t)r : -1;
    }
    __syncthreads();
    const uint4* s = src + t * vec_per_row;
#pragma unroll 4
    for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
      const uint4 val = __ldg(s + v);
      for (int j = 0; j < k; ++j)
        if (rows[j] >= 0) dst[rows[j] * vec_per_row + v] = val;
    }
  }
}

cudaError_t launch_scatter_rows(const void* src, const int32_t* perm_dst, int64_t T, int k,
                                int64_t P, int width, int elem_bytes, void* dst, int num_sms,
                                cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int64_t row_bytes = (int64_t)width * elem_bytes;
  if (row_bytes % 16 || k > 32) return cudaErrorInvalidValue;
  const int64_t blocks = T < (int64_t)num_sms * 8 ? T : (int64_t)num_sms * 8;
  LaunchScope ls("scatter_rows", st);
  scatter_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>((const uint4*)src, perm_dst, T, k, P,
                                                        (int)(row_bytes / 16), (uint4*)dst);
  return cudaGetLastError();
}

// perm_dst[perm_src[r]] = r for r < P: the inverse of the expert-major order (the layer's own
// permute writes both; the stage entry point for the experts receives only perm_src).
__global__ void invert_perm_kernel(const int32_t* __restrict__ perm_src, int64_t P,
                                   int32_t* __restrict__ perm_dst) {
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < P;
       r += (int64_t)gridDim.x * blockDim.x) {
    const int p = perm_src[r];
    if (p >= 0 && p < P) perm_dst[p] = (int32_t)r;
  }
}

cudaError_t launch_invert_perm(const int32_t* perm_src, int64_t P, int32_t* perm_dst, int num_sms,
                               cudaStream_t st) {
  if (P <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(perm_dst, 0xff, (size_t)P * 4, st);  // -1: no pair
  if (e != cudaSuccess) return e;
  const int64_t blocks = (P + 255) / 256 < (int64_t)num_sms * 8 ? (P + 255) / 256 : num_sms * 8;
  LaunchScope ls("invert_perm", st);
  invert_perm_kernel<<<(unsigned)blocks, 256, 0, st>>>(perm_src, P, perm_dst);
  return cudaGetLastError();
}

}  // namespace moe
