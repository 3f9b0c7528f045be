// permute_noalloc.cu -- moe_permute without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc at the point where they route tokens.  One case is a serving
// process that reserved the GPU's free memory for its own pool at start-up, where any later
// allocation fails or evicts cached state.  Another is a latency-critical loop where cudaMalloc
// is not allowed because it can synchronise the device and stall the other streams.  For them
// this entry point keeps its only scratch, the per-chunk expert counts of the counting sort, in a
// fixed array in device global memory, part of the library image.  Every GPU that loads the
// library holds the array (1 MiB) until the process exits.
//
// The array is shared by every call on a device and keeps the last call's contents.  Nothing in it
// needs to start at zero: each call overwrites every count it reads before reading it.  Calls whose
// work overlaps on the GPU (two streams at once) race on it and give wrong results; serialise them.
#include <mutex>

#include "internal.h"

namespace moe {

constexpr int kNoAllocMaxExperts = 1024;                       // E + 1 <= 1024
constexpr int kNoAllocMaxPairs = 262144;                       // T * k
constexpr int kNoAllocChunk = 1024;                            // pairs per chunk (permute.cu)
constexpr int kNoAllocMaxChunks = kNoAllocMaxPairs / kNoAllocChunk;
constexpr int kMaxDevices = 64;

// The scratch: chunk counts [chunks][E], 1 MiB.
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocMaxChunks * kNoAllocMaxExperts];

// Device address of g_permute_scratch for the current device.  In host code the array's name is
// only a host-side stand-in, never a device address, so the address is asked of the runtime with
// that device current.  It is looked up again on every call made outside stream capture (a
// cudaDeviceReset reloads the module, and the array may then sit elsewhere); during capture the
// address found by the last call outside capture on that device is used, since a lookup may have
// to load the module, which capture does not allow.
static int32_t* scratch_for_current_device(cudaStream_t st, cudaError_t* err) {
  static std::mutex mu;
  static int32_t* ptr[kMaxDevices] = {nullptr};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  *err = cudaStreamIsCapturing(st, &cap);
  if (*err != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (*err != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<int32_t*>(p);
  } else if (!ptr[dev]) {
    *err = cudaErrorStreamCaptureUnsupported;  // no call outside capture on this device yet
    return nullptr;
  }
  return ptr[dev];
}

}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_idx,
                                            int32_t* counts, int32_t* offsets, int32_t* perm_src,
                                            int32_t* perm_dst, void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (cfg->T < 0 || cfg->E < 1 || cfg->k < 1 || cfg->k > cfg->E ||
      (cfg->n_shared != 0 && cfg->n_shared != 1))
    return MOE_ERR_INVALID_ARG;
  // sizes beyond the fixed scratch are refused before anything is enqueued
  if (cfg->E + 1 > kNoAllocMaxExperts || cfg->T * (int64_t)cfg->k > kNoAllocMaxPairs)
    return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!topk_idx || !counts || !offsets || !perm_src || !perm_dst) return MOE_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  int32_t* scratch = scratch_for_current_device(st, &e);
  if (!scratch) return status_from_cuda(e);
  (void)cudaGetLastError();
  // No status word: an expert index outside [0, E) is skipped (not counted) and its perm_dst
  // entry is set to -1.
  e = launch_permute(topk_idx, cfg->T, cfg->k, cfg->E, cfg->n_shared, scratch, counts, offsets,
                     perm_src, perm_dst, nullptr, st);
  return status_from_cuda(e);
}
