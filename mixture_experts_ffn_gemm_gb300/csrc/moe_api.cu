// moe_api.cu -- the C ABI of include/moe.h: host validation, workspace layout and the order of
// kernel launches for each entry point.  No allocation, no host synchronisation on the layer path.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace moe {

// ---------------------------------------------------------------------------------------------
// Launch counter and launch profiler
// ---------------------------------------------------------------------------------------------
static thread_local uint64_t g_launches = 0;

struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
struct ProfTotal {
  std::string name;
  double ms;
  uint64_t launches;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<ProfRecord> g_prof_pending;
static std::vector<cudaEvent_t> g_prof_pool;
static std::vector<ProfTotal> g_prof_totals;

static cudaEvent_t prof_event() {  // caller holds g_prof_mu
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

LaunchScope::LaunchScope(const char* name, cudaStream_t st) : name_(name), st_(st) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  start_ = prof_event();
  if (start_ && cudaEventRecord(start_, st_) != cudaSuccess) {
    g_prof_pool.push_back(start_);
    start_ = nullptr;
  }
}

LaunchScope::~LaunchScope() {
  ++g_launches;
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t stop = prof_event();
  if (stop && cudaEventRecord(stop, st_) == cudaSuccess) {
    g_prof_pending.push_back({name_, start_, stop});
  } else {
    g_prof_pool.push_back(start_);
    if (stop) g_prof_pool.push_back(stop);
  }
}

static int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

static size_t dtype_bytes(int dt) { return dt == MOE_F32 ? 4 : dt == MOE_BF16 ? 2 : 1; }
static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Choices that depend only on the configuration (so that the workspace size is deterministic).
struct Plan {
  bool latent;
  int de;             // expert width: d or d_latent
  bool router_tc;     // tensor-core router (3 x bf16 split weights)
  bool router_splitk; // tensor-core router for small batches, split over K (weights split inside)
  int router_splits;  // K slices of the router GEMM (partial logits the selection adds in order)
  int swap;           // expert GEMM tiles: 0 token rows as M; 1 weight rows as M with 32-token
                      // tiles; 2 the same with 256-token tiles
  bool tc;            // tensor-core expert GEMMs
  bool fp8;           // e4m3 experts with block scales
  bool w4;            // 4-bit integer group-quantised experts
  bool fused;         // decode experts in one persistent launch (32-token swap-AB tiles)
  bool y_bf16;        // expert outputs (y_perm and the shared rows) in bf16 instead of fp32
};

struct Layout {
  size_t status, zbuf, wsplit, idx, weight, chunk_counts, counts, offsets, perm_src, perm_dst,
      x_lat, x_perm, h, y_perm, u_hat, x_io, out_io;
  size_t ready;       // fused decode experts: W1|W3 tiles done per row tile
  size_t xq, xq_s, xpq, xpq_s, hq, hq_s;  // fp8 experts: e4m3 activations + [K/128][rows] scales
  size_t total;
};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static moe_status_t validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->T > (int64_t)1 << 26) return MOE_ERR_INVALID_ARG;
  if (c->d <= 0 || c->E < 1 || c->k < 1 || c->k > c->E || c->I <= 0) return MOE_ERR_INVALID_ARG;
  if (c->n_shared != 0 && c->n_shared != 1) return MOE_ERR_INVALID_ARG;
  if (c->d_latent < 0 || c->reserved_ != 0) return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->w_dtype != MOE_F32 && c->w_dtype != MOE_BF16 && c->w_dtype != MOE_FP8_E4M3 &&
      c->w_dtype != MOE_INT4)
    return MOE_ERR_INVALID_ARG;
  if (c->k > 32 || c->E > 1023) return MOE_ERR_UNSUPPORTED;
  // bf16 expert outputs: bf16 or e4m3 experts on the K2 path
  if ((c->flags & MOE_FLAG_EXPERT_OUT_BF16) &&
      (c->act_dtype != MOE_BF16 || (c->w_dtype != MOE_BF16 && c->w_dtype != MOE_FP8_E4M3) ||
       c->d_latent > 0))
    return MOE_ERR_UNSUPPORTED;
  if (c->n_shared && c->I_shared != c->I) return MOE_ERR_UNSUPPORTED;
  if (c->T * c->k + c->T >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (c->w_dtype == MOE_FP8_E4M3) {
    // e4m3 experts: bf16 activations, 128 x 128 weight blocks, K2 path only
    if (c->act_dtype != MOE_BF16 || c->quant_block != 128 || c->d_latent > 0)
      return MOE_ERR_UNSUPPORTED;
    if (c->d % 256 || c->I % 128) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
  }
  if (c->w_dtype == MOE_INT4) {
    // 4-bit groups of 32 input channels: bf16 activations, K2 path only
    if (c->act_dtype != MOE_BF16 || c->quant_block != 32 || c->d_latent > 0)
      return MOE_ERR_UNSUPPORTED;
    if (c->d % 256 || c->I % 128) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
  }
  if (c->w_dtype != c->act_dtype) return MOE_ERR_UNSUPPORTED;
  if (c->act_dtype == MOE_F32) {
    if (c->d % 16 || c->I % 16 || c->d % 4) return MOE_ERR_UNSUPPORTED;
    if (c->d_latent > 0) return MOE_ERR_UNSUPPORTED;
  } else {
    if (c->d % 256 || c->I % 128) return MOE_ERR_UNSUPPORTED;
    if (c->d_latent > 0 && (c->d_latent % 256 || c->d_latent > 8192)) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

static Plan make_plan(const moe_config_t* c) {
  Plan p;
  p.latent = c->d_latent > 0;
  p.de = p.latent ? c->d_latent : c->d;
  p.tc = c->act_dtype == MOE_BF16;
  p.fp8 = c->w_dtype == MOE_FP8_E4M3;
  p.w4 = c->w_dtype == MOE_INT4;
  // router
  const bool tc_ok = c->act_dtype == MOE_BF16 && c->E % 128 == 0 && c->d % 64 == 0;
  if (c->flags & MOE_FLAG_ROUTER_SIMT)
    p.router_tc = false;
  else if (c->flags & MOE_FLAG_ROUTER_TC)
    p.router_tc = tc_ok;
  else
    p.router_tc = tc_ok && c->T >= 1024;
  p.router_splits = 1;
  if (p.router_tc) {
    // few 128-token row tiles (one CTA each, all experts in one N = 384 tile) leave SMs idle: the
    // 3 * d reduction is split into as many K ranges as one wave of 152 CTAs holds (at most 8),
    // whose fp32 partial logits the selection kernel adds in range order
    const int64_t tiles = (c->T + 127) / 128;
    const int64_t s = tiles > 0 ? 152 / tiles : 1;
    p.router_splits = s < 1 ? 1 : s > 8 ? 8 : (int)s;
  }
  // small bf16 batches: the split-K tensor-core router, slices for one wave of CTAs on 152 SMs
  p.router_splitk = !p.router_tc && !(c->flags & MOE_FLAG_ROUTER_SIMT) &&
                    c->act_dtype == MOE_BF16 && router_splitk_tc_supported(c->T, c->E, c->d);
  if (p.router_splitk) {
    p.router_splits = router_splitk_tc_slices(c->T, c->E, c->d, 152);
  } else if (!p.router_tc) {
    const int64_t tiles = ((c->T + 63) / 64) * ((c->E + 63) / 64);
    int s = (int)((304 + (tiles > 0 ? tiles : 1) - 1) / (tiles > 0 ? tiles : 1));
    if (s > 32) s = 32;
    while (s > 1 && (c->d % (16 * s) != 0)) --s;
    p.router_splits = s < 1 ? 1 : s;
  }
  // expert GEMM tile orientation.  Few tokens: 32-token swap-AB tiles (each expert's weights
  // stream once).  Otherwise 128-token rows tiles.  The 256-token swap-AB tiles (MMA N shrinks to
  // a group's last tokens) waste far less padding in the K3 regime of ~171 rows per expert, but
  // measured slower there: the SwiGLU accumulators take all of TMEM, so the epilogue no longer
  // overlaps the next tile, and MMAs with N < 256 read more shared memory per FLOP.  They stay
  // available through MOE_FLAG_GEMM_SWAP_WIDE.
  if (c->flags & MOE_FLAG_GEMM_SWAP_AB)
    p.swap = 1;
  else if (c->flags & MOE_FLAG_GEMM_SWAP_WIDE)
    p.swap = 2;
  else if (c->flags & MOE_FLAG_GEMM_ROWS_MAJOR)
    p.swap = 0;
  else
    p.swap = c->T <= 512 ? 1 : 0;
  // the one-launch decode experts on request only: measured slower than the two launches
  // bf16 expert outputs on request, and by default for e4m3 experts: their quantisation error is
  // far above one more bf16 rounding of each expert output, and the outputs' bytes are a large
  // part of the W2 launch
  p.y_bf16 = (c->flags & MOE_FLAG_EXPERT_OUT_BF16) ||
             (p.fp8 && !(c->flags & MOE_FLAG_EXPERT_OUT_F32));
  p.fused = p.tc && !p.fp8 && !p.w4 && !p.latent && p.swap == 1 && !p.y_bf16 &&
            (c->flags & MOE_FLAG_DECODE_FUSED) && !(c->flags & MOE_FLAG_TEST_STALL_EXPERTS) &&
            c->I % 128 == 0;
  return p;
}

static Layout make_layout(const moe_config_t* c, const Plan& pl) {
  Layout L;
  const int64_t T = c->T, P = T * c->k, E = c->E, d = c->d, I = c->I;
  const size_t ab = dtype_bytes(c->act_dtype);
  const int64_t shared_rows = T * c->n_shared;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  L.status = take(256);
  L.zbuf = take((size_t)pl.router_splits * T * E * 4);
  L.wsplit = take(pl.router_tc ? (size_t)E * 3 * d * 2 : 0);
  L.idx = take((size_t)P * 4);
  L.weight = take((size_t)P * 4);
  L.chunk_counts = take((size_t)permute_chunks(P) * E * 4);
  L.counts = take((size_t)(E + 1) * 4);
  L.offsets = take((size_t)(E + 2) * 4);
  L.perm_src = take((size_t)P * 4);
  L.perm_dst = take((size_t)P * 4);
  L.x_lat = take(pl.latent ? (size_t)T * c->d_latent * ab : 0);
  L.x_perm = take(pl.fp8 ? 0 : (size_t)P * pl.de * ab);
  L.h = take(pl.fp8 ? 0 : (size_t)(P + shared_rows) * I * ab);
  L.xq = take(pl.fp8 ? (size_t)T * d : 0);
  L.xq_s = take(pl.fp8 ? (size_t)(d / 128) * T * 4 : 0);
  L.xpq = take(pl.fp8 ? (size_t)P * d : 0);
  L.xpq_s = take(pl.fp8 ? (size_t)(d / 128) * P * 4 : 0);
  L.hq = take(pl.fp8 ? (size_t)(P + shared_rows) * I : 0);
  L.hq_s = take(pl.fp8 ? (size_t)(I / 128) * (P + shared_rows) * 4 : 0);
  L.y_perm = take(((size_t)P * pl.de + (size_t)shared_rows * d) * 4);  // fp32 expert outputs
  L.ready = take(pl.fused ? (size_t)fused_ready_count(T, c->k, E) * 4 : 0);
  L.u_hat = take(pl.latent ? (size_t)T * c->d_latent * 2 : 0);
  L.x_io = take((size_t)T * d * ab);
  L.out_io = take((size_t)T * d * ab);
  L.total = off;
  return L;
}

static thread_local char g_last_error[256] = "";

static moe_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

moe_status_t status_from_cuda(cudaError_t e) { return from_cuda(e); }

template <typename T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

struct Ctx {
  const moe_config_t* c;
  Plan pl;
  Layout L;
  void* ws;
  cudaStream_t st;
  int sms;
  uint32_t* err;
  // the shared expert's rows are already computed (host-I/O path, chunk by chunk as the input
  // arrives) and the status word already reset: the routed launches carry no dense group
  bool shared_done = false;
};

static moe_status_t begin(Ctx& x, const moe_config_t* c, void* ws, size_t ws_bytes,
                          void* stream) {
  moe_status_t s = validate(c);
  if (s != MOE_OK) return s;
  x.c = c;
  x.pl = make_plan(c);
  x.L = make_layout(c, x.pl);
  if (!ws || ws_bytes < x.L.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  x.ws = ws;
  x.st = static_cast<cudaStream_t>(stream);
  x.sms = 0;
  x.err = at<uint32_t>(ws, x.L.status);
  return MOE_OK;
}

// T == 0: every entry point is a no-op once the configuration and workspace are valid (empty
// tensors may come with NULL data pointers).
#define MOE_RETURN_IF_EMPTY(cfg) \
  do {                           \
    if ((cfg)->T == 0) return MOE_OK; \
  } while (0)

// First CUDA runtime calls of an entry point, made only after every host-side check passed.
static void ready(Ctx& x) {
  x.sms = num_sms();
  (void)cudaGetLastError();  // start from a clean launch-error state
}

// Host-I/O overlap: inputs of at least kIoOverlapBytes arrive in kIoStreams pieces at once, or,
// for bf16 layers with a shared expert, in up to kIoChunks token chunks of at least
// kIoMinChunkTokens, each chunk's shared-expert rows computed while the next chunk is copied; the
// output leaves in kIoChunks chunks, each behind its part of the combine.
constexpr size_t kIoOverlapBytes = 32u << 20;
constexpr int kIoStreams = 2;
constexpr int kIoChunks = 8;
constexpr int64_t kIoMinChunkTokens = 2048;
constexpr int kIoMaxDevices = 64;

struct OutCopy {
  void* host;
  int n;
  cudaStream_t cs[kIoStreams];
  cudaEvent_t ev[kIoChunks];
};

struct IoStreams {
  bool ok = false;
  cudaStream_t cs[kIoStreams] = {};
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_in[kIoStreams] = {};
  cudaEvent_t ev_out[kIoStreams] = {};
  cudaEvent_t ev_chunk[kIoChunks] = {};
  cudaEvent_t ev_in_chunk[kIoChunks] = {};
};
static std::mutex g_io_mutex;
static IoStreams g_io[kIoMaxDevices];

// Creates the current device's copy streams and events (kept for the life of the process).
static moe_status_t io_streams_init(IoStreams& io) {
  const unsigned ef = cudaEventDisableTiming;
  for (int i = 0; i < kIoStreams; ++i) {
    if (cudaStreamCreateWithFlags(&io.cs[i], cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&io.ev_in[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&io.ev_out[i], ef) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (cudaEventCreateWithFlags(&io.ev_start, ef) != cudaSuccess) return MOE_ERR_CUDA;
  for (int i = 0; i < kIoChunks; ++i)
    if (cudaEventCreateWithFlags(&io.ev_chunk[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&io.ev_in_chunk[i], ef) != cudaSuccess)
      return MOE_ERR_CUDA;
  io.ok = true;
  return MOE_OK;
}

static moe_status_t forward_impl(Ctx& c, const void* x, const float* W_r, const float* b,
                                 const void* W13, const void* W2, const float* W13_scale,
                                 const float* W2_scale, const void* Ws13, const void* Ws2,
                                 const float* Ws13_scale, const float* Ws2_scale,
                                 const void* W_down, const void* W_up, void* out,
                                 const OutCopy* oc);

// ---------------------------------------------------------------------------------------------
// Stages
// ---------------------------------------------------------------------------------------------
static moe_status_t run_router(Ctx& x, const void* xin, const float* W_r, const float* b,
                               float* logits, int32_t* idx, float* weight) {
  const moe_config_t* c = x.c;
  if (c->T == 0) return MOE_OK;
  cudaError_t e;
  if (x.pl.router_tc) {
    __nv_bfloat16* ws_split = at<__nv_bfloat16>(x.ws, x.L.wsplit);
    e = launch_split_router_weights(W_r, c->E, c->d, ws_split, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    const int S = x.pl.router_splits;
    float* z = (S == 1 && logits) ? logits : at<float>(x.ws, x.L.zbuf);
    GroupedGemm g;
    g.act_d = xin;
    g.act_d_rows = c->T;
    g.w_d = ws_split;
    g.w_d_rows = c->E;
    g.dense_rows = (int)c->T;
    g.K = 3 * c->d;
    g.k_wrap = c->d;
    g.F = c->E;
    g.epi = EPI_STORE;
    g.out = z;
    g.ldo = c->E;
    g.out_dtype = MOE_F32;
    g.k_splits = S;
    g.split_stride = c->T * c->E;
    g.err = x.err;
    g.label = "router_gemm_tc";
    e = launch_gemm_tc(g, 0, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    e = launch_router_topk(z, S, c->T * c->E, c->T, c->E, c->k, b, c->gate_scale,
                           S == 1 ? nullptr : logits, idx, weight, x.st);
    return from_cuda(e);
  }
  float* zp = at<float>(x.ws, x.L.zbuf);
  if (x.pl.router_splitk) {
    e = launch_router_splitk_tc(xin, W_r, c->T, c->E, c->d, x.pl.router_splits, zp,
                                c->T * c->E, x.err, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    e = launch_router_topk(zp, x.pl.router_splits, c->T * c->E, c->T, c->E, c->k, b,
                           c->gate_scale, logits, idx, weight, x.st);
    return from_cuda(e);
  }
  GroupedGemm g;
  g.act_d = xin;
  g.act_d_rows = c->T;
  g.w_d = W_r;
  g.w_d_rows = c->E;
  g.dense_rows = (int)c->T;
  g.K = c->d;
  g.k_wrap = c->d;
  g.F = c->E;
  g.epi = EPI_STORE;
  g.act_dtype = c->act_dtype;
  g.w_dtype = MOE_F32;
  g.out = zp;
  g.ldo = c->E;
  g.out_dtype = MOE_F32;
  g.k_splits = x.pl.router_splits;
  g.split_stride = c->T * c->E;
  g.err = x.err;
  g.label = "router_gemm_simt";
  e = launch_gemm_simt(g, x.sms, x.st);
  if (e != cudaSuccess) return from_cuda(e);
  e = launch_router_topk(zp, x.pl.router_splits, c->T * c->E, c->T, c->E, c->k, b,
                         c->gate_scale, logits, idx, weight, x.st);
  return from_cuda(e);
}

static moe_status_t run_permute(Ctx& x, const int32_t* idx, int32_t* counts, int32_t* offsets,
                                int32_t* perm_src, int32_t* perm_dst) {
  const moe_config_t* c = x.c;
  return from_cuda(launch_permute(idx, c->T, c->k, c->E, c->n_shared,
                                  at<int32_t>(x.ws, x.L.chunk_counts), counts, offsets, perm_src,
                                  perm_dst, x.err, x.st));
}

// The routed expert GEMMs: tensor cores (token-rows or swap-AB tiles) for bf16, CUDA cores for
// fp32.  The profiler name carries the variant ("<label>_rows" / "_swap" / "_simt").
static cudaError_t gemm(Ctx& x, GroupedGemm g, const char* rows_label, const char* swap_label,
                        const char* wide_label, const char* simt_label) {
  if (x.pl.tc) {
    g.label = x.pl.swap == 2 ? wide_label : x.pl.swap ? swap_label : rows_label;
    return launch_gemm_tc(g, x.pl.swap, x.sms, x.st);
  }
  g.label = simt_label;
  return launch_gemm_simt(g, x.sms, x.st);
}

// perm_dst may be null (the experts' stage entry point receives only perm_src): its inverse is
// then rebuilt in the workspace, since the activation rows are copied token by token.
static moe_status_t run_experts(Ctx& x, const void* xin, const int32_t* offsets,
                                const int32_t* perm_src, const int32_t* perm_dst, const void* W13,
                                const void* W2, const float* W13_scale, const float* W2_scale,
                                const void* Ws13, const void* Ws2, const float* Ws13_scale,
                                const float* Ws2_scale, const void* W_down, void* y_perm) {
  const moe_config_t* c = x.c;
  if (c->T == 0) return MOE_OK;
  if (!perm_dst) {
    int32_t* inv = at<int32_t>(x.ws, x.L.perm_dst);
    cudaError_t ei = launch_invert_perm(perm_src, c->T * c->k, inv, x.sms, x.st);
    if (ei != cudaSuccess) return from_cuda(ei);
    perm_dst = inv;
  }
  const int64_t T = c->T, P = T * c->k;
  const int de = x.pl.de, I = c->I, d = c->d, E = c->E;
  const size_t ab = dtype_bytes(c->act_dtype);
  void* h = at<void>(x.ws, x.L.h);
  void* x_perm = at<void>(x.ws, x.L.x_perm);
  cudaError_t e;

  if (x.pl.fp8) {  // e4m3 experts: quantise x once, gather codes + scales, two fp8 GEMMs
    uint8_t* xq = at<uint8_t>(x.ws, x.L.xq);
    float* xq_s = at<float>(x.ws, x.L.xq_s);
    uint8_t* xpq = at<uint8_t>(x.ws, x.L.xpq);
    float* xpq_s = at<float>(x.ws, x.L.xpq_s);
    uint8_t* hq = at<uint8_t>(x.ws, x.L.hq);
    float* hq_s = at<float>(x.ws, x.L.hq_s);
    const int64_t rows_h = P + (c->n_shared ? T : 0);
    e = launch_quantize_rows(xin, T, d, xq, xq_s, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    e = launch_scatter_q(xq, xq_s, T, perm_dst, c->k, P, d, xpq, xpq_s, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    Fp8Gemm g;
    g.act = xpq;
    g.act_rows = P;
    g.act_sT = xpq_s;
    g.act_s_ld = P;
    g.w = W13;
    g.w_rows = (int64_t)E * 2 * I;
    g.w_s = W13_scale;
    g.offsets = offsets;
    g.n_routed = E;
    g.w_group_rows = 2 * I;
    g.u_off = I;
    if (c->n_shared) {
      g.act_d = xq;
      g.act_d_rows = T;
      g.act_sT_d = xq_s;
      g.act_s_ld_d = T;
      g.w_d = Ws13;
      g.w_d_rows = 2 * I;
      g.w_s_d = Ws13_scale;
      g.dense_rows = (int)T;
      g.dense_out_row0 = (int)P;
      g.u_off_d = I;
    }
    g.K = d;
    g.F = I;
    g.swiglu = true;
    g.out = hq;
    g.ldo = I;
    g.out_sT = hq_s;
    g.out_s_ld = rows_h;
    g.err = x.err;
    g.label = "gemm13_swiglu_fp8";
    e = launch_gemm_fp8(g, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    Fp8Gemm g2;
    g2.act = hq;
    g2.act_rows = rows_h;
    g2.act_sT = hq_s;
    g2.act_s_ld = rows_h;
    g2.w = W2;
    g2.w_rows = (int64_t)E * d;
    g2.w_s = W2_scale;
    g2.offsets = offsets;
    g2.n_routed = E;
    g2.w_group_rows = d;
    if (c->n_shared) {
      g2.act_d = hq;
      g2.act_d_rows = rows_h;
      g2.act_sT_d = hq_s;
      g2.act_s_ld_d = rows_h;
      g2.dense_act_row0 = (int)P;
      g2.w_d = Ws2;
      g2.w_d_rows = d;
      g2.w_s_d = Ws2_scale;
      g2.dense_rows = (int)T;
      g2.dense_out_row0 = (int)P;
    }
    g2.K = I;
    g2.F = d;
    g2.swiglu = false;
    g2.out = y_perm;
    g2.ldo = d;
    g2.out_bf16 = x.pl.y_bf16;
    g2.err = x.err;
    g2.label = "gemm2_fp8";
    return from_cuda(launch_gemm_fp8(g2, x.sms, x.st));
  }

  if (x.pl.w4) {  // 4-bit experts: gather bf16 x, two grouped GEMMs that expand the weights
    e = launch_scatter_rows(xin, perm_dst, T, c->k, P, d, (int)ab, x_perm, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    const bool sh = c->n_shared != 0;
    W4Gemm g;
    g.act = x_perm;
    g.act_rows = P;
    g.wq = W13;
    g.ws = W13_scale;
    g.w_rows = (int64_t)E * 2 * I;
    g.offsets = offsets;
    g.n_routed = E;
    g.w_group_rows = 2 * I;
    g.u_off = I;
    if (sh) {
      g.act_d = xin;
      g.act_d_rows = T;
      g.wq_d = Ws13;
      g.ws_d = Ws13_scale;
      g.w_d_rows = 2 * I;
      g.dense_rows = (int)T;
      g.dense_out_row0 = (int)P;
      g.u_off_d = I;
    }
    g.K = d;
    g.F = I;
    g.swiglu = true;
    g.out = h;
    g.ldo = I;
    g.err = x.err;
    g.label = "gemm13_swiglu_w4";
    e = launch_gemm_w4(g, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    W4Gemm g2;
    g2.act = h;
    g2.act_rows = P + (sh ? T : 0);
    g2.wq = W2;
    g2.ws = W2_scale;
    g2.w_rows = (int64_t)E * d;
    g2.offsets = offsets;
    g2.n_routed = E;
    g2.w_group_rows = d;
    if (sh) {
      g2.act_d = h;
      g2.act_d_rows = P + T;
      g2.dense_act_row0 = (int)P;
      g2.wq_d = Ws2;
      g2.ws_d = Ws2_scale;
      g2.w_d_rows = d;
      g2.dense_rows = (int)T;
      g2.dense_out_row0 = (int)P;
    }
    g2.K = I;
    g2.F = d;
    g2.swiglu = false;
    g2.out = y_perm;
    g2.ldo = d;
    g2.err = x.err;
    g2.label = "gemm2_w4";
    return from_cuda(launch_gemm_w4(g2, x.sms, x.st));
  }

  const void* route_src = xin;
  if (x.pl.latent) {  // x_lat = x W_down^T on every token (the router saw the full width)
    void* x_lat = at<void>(x.ws, x.L.x_lat);
    GroupedGemm g;
    g.act_d = xin;
    g.act_d_rows = T;
    g.w_d = W_down;
    g.w_d_rows = de;
    g.dense_rows = (int)T;
    g.K = d;
    g.k_wrap = d;
    g.F = de;
    g.epi = EPI_STORE;
    g.act_dtype = g.w_dtype = c->act_dtype;
    g.out = x_lat;
    g.ldo = de;
    g.out_dtype = c->act_dtype;
    g.err = x.err;
    g.label = "down_proj";
    e = launch_gemm_tc(g, 0, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    route_src = x_lat;
  }
  e = launch_scatter_rows(route_src, perm_dst, T, c->k, P, de, (int)ab, x_perm, x.sms, x.st);
  if (e != cudaSuccess) return from_cuda(e);

  if (x.pl.fused) {  // decode: both expert GEMMs in one persistent launch
    uint32_t* ready = at<uint32_t>(x.ws, x.L.ready);
    e = cudaMemsetAsync(ready, 0, (size_t)fused_ready_count(T, c->k, E) * 4, x.st);
    if (e != cudaSuccess) return from_cuda(e);
    FusedDecode f;
    f.x_perm = x_perm;
    f.x = xin;
    f.W13 = W13;
    f.Ws13 = Ws13;
    f.W2 = W2;
    f.Ws2 = Ws2;
    f.offsets = offsets;
    f.n_routed = E;
    f.T = c->n_shared ? T : 0;
    f.P = P;
    f.d = d;
    f.I = I;
    f.h = h;
    f.y = static_cast<float*>(y_perm);
    f.ready = ready;
    f.err = x.err;
    e = launch_decode_fused(f, x.sms, x.st);
    if (e != cudaErrorCooperativeLaunchTooLarge) return from_cuda(e);
    (void)cudaGetLastError();  // not every SM free for a cooperative launch: two launches instead
  }

  // W1 | W3 with the SwiGLU epilogue -> h [P + T][I]; the shared expert is the trailing dense
  // group of the same launch (on the K3 path with its own reduction length d, since it reads the
  // full-width x while the routed experts read the latent)
  const bool fuse_shared = c->n_shared && !x.shared_done && (x.pl.tc || !x.pl.latent);
  void* y_sh = static_cast<uint8_t*>(y_perm) + (size_t)P * de * (x.pl.y_bf16 ? 2 : 4);
  {
    GroupedGemm g;
    g.act = x_perm;
    g.act_rows = P;
    g.w = W13;
    g.w_rows = (int64_t)E * 2 * I;
    g.offsets = offsets;
    g.n_routed = E;
    g.w_group_rows = 2 * I;
    g.u_off = I;
    if (fuse_shared) {
      g.act_d = xin;
      g.act_d_rows = T;
      g.w_d = Ws13;
      g.w_d_rows = 2 * I;
      g.dense_rows = (int)T;
      g.dense_out_row0 = (int)P;
      g.u_off_d = I;
      if (x.pl.latent) g.K_d = d;
    }
    g.K = de;
    g.k_wrap = de;
    g.F = I;
    g.epi = EPI_SWIGLU;
    g.act_dtype = g.w_dtype = c->act_dtype;
    g.out = h;
    g.ldo = I;
    g.out_dtype = c->act_dtype;
    g.err = x.err;
    g.test_stall = (c->flags & MOE_FLAG_TEST_STALL_EXPERTS) != 0;
    g.m_halves = (c->flags & MOE_FLAG_GEMM_M1) ? 1 : (c->flags & MOE_FLAG_GEMM_M2) ? 2 : 0;
    g.pair = (c->flags & MOE_FLAG_GEMM_PAIR) && !g.test_stall && g.m_halves != 2;
    e = gemm(x, g, "gemm13_swiglu_rows", "gemm13_swiglu_swap", "gemm13_swiglu_swap256",
             "gemm13_swiglu_simt");
    if (e != cudaSuccess) return from_cuda(e);
  }
  // W2 -> y_perm [P][de] (+ shared rows [T][d])
  {
    GroupedGemm g;
    g.act = h;
    g.act_rows = P + (fuse_shared ? T : 0);
    g.w = W2;
    g.w_rows = (int64_t)E * de;
    g.offsets = offsets;
    g.n_routed = E;
    g.w_group_rows = de;
    if (fuse_shared) {
      g.act_d = h;
      g.act_d_rows = P + T;
      g.dense_act_row0 = (int)P;
      g.w_d = Ws2;
      g.w_d_rows = d;
      g.dense_rows = (int)T;
      g.dense_out_row0 = (int)P;
      if (x.pl.latent) {  // shared outputs are full width, in their own region after y_perm
        g.F_d = d;
        g.out_d = y_sh;
        g.ldo_d = d;
        g.dense_out_row0 = 0;
      }
    }
    g.K = I;
    g.k_wrap = I;
    g.F = de;
    g.epi = EPI_STORE;
    g.act_dtype = g.w_dtype = c->act_dtype;
    g.out = y_perm;
    g.ldo = de;
    g.out_dtype = x.pl.y_bf16 ? MOE_BF16 : MOE_F32;
    g.err = x.err;
    g.n128 = (c->flags & MOE_FLAG_GEMM_N128) != 0;
    g.pair = (c->flags & MOE_FLAG_GEMM_PAIR) && !g.n128;
    e = gemm(x, g, "gemm2_rows", "gemm2_swap", "gemm2_swap256", "gemm2_simt");
    if (e != cudaSuccess) return from_cuda(e);
  }
  return MOE_OK;
}

// The shared expert of tokens [t0, t0 + nt) in two launches of its own: dense groups of the
// token-rows expert GEMMs, with the tiles and K order it has as the trailing group of the routed
// launches, so its rows come out bit for bit the same.  h rows P + t0 .., then its expert-output
// rows (K2: rows P + t0 .. of y_perm; K3: rows t0 .. of the full-width region after y_perm).
static moe_status_t run_shared_rows(Ctx& x, const void* xin, const void* Ws13, const void* Ws2,
                                    int64_t t0, int64_t nt) {
  const moe_config_t* c = x.c;
  const int64_t T = c->T, P = T * c->k;
  const int de = x.pl.de, I = c->I, d = c->d;
  void* h = at<void>(x.ws, x.L.h);
  uint8_t* y_perm = at<uint8_t>(x.ws, x.L.y_perm);
  const size_t yb = x.pl.y_bf16 ? 2 : 4;
  cudaError_t e;
  {
    GroupedGemm g;
    g.act_d = xin;
    g.act_d_rows = T;
    g.dense_act_row0 = (int)t0;
    g.w_d = Ws13;
    g.w_d_rows = 2 * I;
    g.dense_rows = (int)nt;
    g.dense_out_row0 = (int)(P + t0);
    g.u_off_d = I;
    g.K = d;
    g.k_wrap = d;
    g.F = I;
    g.epi = EPI_SWIGLU;
    g.act_dtype = g.w_dtype = c->act_dtype;
    g.out = h;
    g.ldo = I;
    g.out_dtype = c->act_dtype;
    g.err = x.err;
    g.label = "shared_gemm13_swiglu_rows";
    e = launch_gemm_tc(g, 0, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  {
    GroupedGemm g;
    g.act_d = h;
    g.act_d_rows = P + T;
    g.dense_act_row0 = (int)(P + t0);
    g.w_d = Ws2;
    g.w_d_rows = d;
    g.dense_rows = (int)nt;
    g.K = I;
    g.k_wrap = I;
    g.F = d;
    g.epi = EPI_STORE;
    g.act_dtype = g.w_dtype = c->act_dtype;
    g.out = y_perm + (x.pl.latent ? (size_t)P * de * yb : 0);
    g.dense_out_row0 = (int)(x.pl.latent ? t0 : P + t0);
    g.ldo = x.pl.latent ? d : de;
    g.out_dtype = x.pl.y_bf16 ? MOE_BF16 : MOE_F32;
    g.err = x.err;
    g.label = "shared_gemm2_rows";
    e = launch_gemm_tc(g, 0, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return MOE_OK;
}

// The combine of tokens [t0, t0 + nt) (all tokens by default): every step of it is per token.
static moe_status_t run_combine(Ctx& x, const void* y_perm, const int32_t* perm_dst,
                                const float* weight, const void* W_up, void* out,
                                const void* resid = nullptr, int64_t t0 = 0, int64_t nt = -1) {
  const moe_config_t* c = x.c;
  if (nt < 0) nt = c->T - t0;
  if (nt <= 0) return MOE_OK;
  const int64_t T = nt, P = c->T * c->k;
  const int de = x.pl.de, d = c->d;
  const size_t ab = dtype_bytes(c->act_dtype);
  perm_dst += t0 * c->k;
  weight += t0 * c->k;
  out = static_cast<uint8_t*>(out) + (size_t)t0 * d * ab;
  if (resid) resid = static_cast<const uint8_t*>(resid) + (size_t)t0 * d * ab;
  // the shared expert's fp32 rows [T][d] follow the routed rows
  const size_t yb = x.pl.y_bf16 ? 2 : 4;  // bytes per expert output
  const void* y_sh = c->n_shared ? static_cast<const uint8_t*>(y_perm) + (size_t)P * de * yb +
                                       (size_t)t0 * d * yb
                                 : nullptr;
  if (!x.pl.latent)
    return from_cuda(launch_combine(c->act_dtype, x.pl.y_bf16, y_perm, y_sh, perm_dst, weight, T,
                                    c->k, P, d, resid, out, x.sms, x.st));
  if (resid) {  // the residual joins the fp32 shared-expert rows the up-projection adds
    if (!y_sh) return MOE_ERR_UNSUPPORTED;
    cudaError_t e = launch_add_residual(static_cast<float*>(const_cast<void*>(y_sh)),
                                        c->act_dtype, resid, T * d, x.sms, x.st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  void* u_hat = at<uint8_t>(x.ws, x.L.u_hat) + (size_t)t0 * de * 2;
  cudaError_t e = launch_latent_combine(y_perm, perm_dst, weight, T, c->k, P, de,
                                        c->latent_norm, c->rms_eps, u_hat, x.sms, x.st);
  if (e != cudaSuccess) return from_cuda(e);
  GroupedGemm g;  // y_routed = u_hat W_up^T (+ y_shared)
  g.act_d = u_hat;
  g.act_d_rows = T;
  g.w_d = W_up;
  g.w_d_rows = d;
  g.dense_rows = (int)T;
  g.K = de;
  g.k_wrap = de;
  g.F = d;
  g.epi = y_sh ? EPI_STORE_ADD : EPI_STORE;
  g.act_dtype = g.w_dtype = c->act_dtype;
  g.out = out;
  g.ldo = d;
  g.out_dtype = c->act_dtype;
  g.addend = y_sh;
  g.ld_add = d;
  g.err = x.err;
  g.label = "up_proj";
  return from_cuda(launch_gemm_tc(g, 0, x.sms, x.st));
}

}  // namespace moe

using namespace moe;

// ---------------------------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------------------------
extern "C" {

size_t moe_workspace_size(const moe_config_t* cfg) {
  if (validate(cfg) != MOE_OK) return 0;
  return make_layout(cfg, make_plan(cfg)).total;
}

moe_status_t moe_router(const moe_config_t* cfg, const void* x, const float* W_r, const float* b,
                        float* logits, int32_t* topk_idx, float* topk_weight, void* ws,
                        size_t ws_bytes, void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  MOE_RETURN_IF_EMPTY(cfg);
  if (!x || !W_r || !b || !topk_idx || !topk_weight) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_r) || (logits && !aligned16(logits)))
    return MOE_ERR_INVALID_ARG;
  ready(c);
  return run_router(c, x, W_r, b, logits, topk_idx, topk_weight);
}

moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_idx, int32_t* counts,
                         int32_t* offsets, int32_t* perm_src, int32_t* perm_dst, void* ws,
                         size_t ws_bytes, void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  MOE_RETURN_IF_EMPTY(cfg);
  if (!topk_idx || !counts || !offsets || !perm_src || !perm_dst) return MOE_ERR_INVALID_ARG;
  ready(c);
  return run_permute(c, topk_idx, counts, offsets, perm_src, perm_dst);
}

moe_status_t moe_experts(const moe_config_t* cfg, const void* x, const int32_t* offsets,
                         const int32_t* perm_src, const void* W13, const void* W2,
                         const float* W13_scale, const float* W2_scale, const void* Ws13,
                         const void* Ws2, const float* Ws13_scale, const float* Ws2_scale,
                         const void* W_down, void* y_perm, void* ws, size_t ws_bytes,
                         void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  MOE_RETURN_IF_EMPTY(cfg);
  if (!x || !offsets || !perm_src || !W13 || !W2 || !y_perm) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared && (!Ws13 || !Ws2)) return MOE_ERR_INVALID_ARG;
  if ((cfg->w_dtype == MOE_FP8_E4M3 || cfg->w_dtype == MOE_INT4) &&
      (!W13_scale || !W2_scale || (cfg->n_shared && (!Ws13_scale || !Ws2_scale))))
    return MOE_ERR_INVALID_ARG;
  if (cfg->d_latent > 0 && !W_down) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, W13, W2, Ws13, Ws2, W_down, y_perm};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  ready(c);
  return run_experts(c, x, offsets, perm_src, nullptr, W13, W2, W13_scale, W2_scale, Ws13, Ws2,
                     Ws13_scale, Ws2_scale, W_down, y_perm);
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* perm_dst,
                         const float* topk_weight, const void* W_up, void* out, void* ws,
                         size_t ws_bytes, void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  MOE_RETURN_IF_EMPTY(cfg);
  if (!y_perm || !perm_dst || !topk_weight || !out) return MOE_ERR_INVALID_ARG;
  if (cfg->d_latent > 0 && !W_up) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (W_up && !aligned16(W_up)))
    return MOE_ERR_INVALID_ARG;
  ready(c);
  return run_combine(c, y_perm, perm_dst, topk_weight, W_up, out);
}

moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const float* W_r, const float* b,
                         const void* W13, const void* W2, const float* W13_scale,
                         const float* W2_scale, const void* Ws13, const void* Ws2,
                         const float* Ws13_scale, const float* Ws2_scale, const void* W_down,
                         const void* W_up, void* out, void* ws, size_t ws_bytes, void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  MOE_RETURN_IF_EMPTY(cfg);
  return forward_impl(c, x, W_r, b, W13, W2, W13_scale, W2_scale, Ws13, Ws2, Ws13_scale,
                      Ws2_scale, W_down, W_up, out, nullptr);
}

}  // extern "C"

namespace moe {

static moe_status_t forward_impl(Ctx& c, const void* x, const float* W_r, const float* b,
                                 const void* W13, const void* W2, const float* W13_scale,
                                 const float* W2_scale, const void* Ws13, const void* Ws2,
                                 const float* Ws13_scale, const float* Ws2_scale,
                                 const void* W_down, const void* W_up, void* out,
                                 const OutCopy* oc) {
  const moe_config_t* cfg = c.c;
  moe_status_t s;
  void* ws = c.ws;
  if (!x || !W_r || !b || !W13 || !W2 || !out) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared && (!Ws13 || !Ws2)) return MOE_ERR_INVALID_ARG;
  if ((cfg->w_dtype == MOE_FP8_E4M3 || cfg->w_dtype == MOE_INT4) &&
      (!W13_scale || !W2_scale || (cfg->n_shared && (!Ws13_scale || !Ws2_scale))))
    return MOE_ERR_INVALID_ARG;
  if (cfg->d_latent > 0 && (!W_down || !W_up)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, W_r, W13, W2, Ws13, Ws2, W_down, W_up, out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  ready(c);
  if (!c.shared_done && cudaMemsetAsync(c.err, 0, 256, c.st) != cudaSuccess) return MOE_ERR_CUDA;
  const Layout& L = c.L;
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* wgt = at<float>(ws, L.weight);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm_src = at<int32_t>(ws, L.perm_src);
  int32_t* perm_dst = at<int32_t>(ws, L.perm_dst);
  void* y_perm = at<void>(ws, L.y_perm);
  if ((s = run_router(c, x, W_r, b, nullptr, idx, wgt)) != MOE_OK) return s;
  if ((s = run_permute(c, idx, at<int32_t>(ws, L.counts), offsets, perm_src, perm_dst)) != MOE_OK)
    return s;
  if ((s = run_experts(c, x, offsets, perm_src, perm_dst, W13, W2, W13_scale, W2_scale, Ws13, Ws2,
                       Ws13_scale, Ws2_scale, W_down, y_perm)) != MOE_OK)
    return s;
  if (!oc) return run_combine(c, y_perm, perm_dst, wgt, W_up, out);
  // the combine in token chunks; each chunk's output leaves for the host on a copy stream while
  // the next chunk is combined
  const int64_t T = cfg->T;
  const size_t row = (size_t)cfg->d * dtype_bytes(cfg->act_dtype);
  const int64_t chunk = (T + oc->n - 1) / oc->n;
  for (int i = 0; i * chunk < T; ++i) {
    const int64_t t0 = i * chunk, nt = T - t0 < chunk ? T - t0 : chunk;
    if ((s = run_combine(c, y_perm, perm_dst, wgt, W_up, out, nullptr, t0, nt)) != MOE_OK)
      return s;
    cudaStream_t cs = oc->cs[i % kIoStreams];
    if (cudaEventRecord(oc->ev[i], c.st) != cudaSuccess ||
        cudaStreamWaitEvent(cs, oc->ev[i], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(oc->host) + (size_t)t0 * row,
                        static_cast<const uint8_t*>(out) + (size_t)t0 * row, (size_t)nt * row,
                        cudaMemcpyDeviceToHost, cs) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe

extern "C" {

moe_status_t moe_forward_block(const moe_config_t* cfg, const void* x_resid, const void* norm_w,
                               const float* W_r, const float* b, const void* W13, const void* W2,
                               const float* W13_scale, const float* W2_scale, const void* Ws13,
                               const void* Ws2, const float* Ws13_scale, const float* Ws2_scale,
                               const void* W_down, const void* W_up, void* out, void* ws,
                               size_t ws_bytes, void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  if (cfg->d_latent > 0 && !cfg->n_shared) return MOE_ERR_UNSUPPORTED;
  MOE_RETURN_IF_EMPTY(cfg);
  if (!x_resid || !norm_w || !W_r || !b || !W13 || !W2 || !out) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared && (!Ws13 || !Ws2)) return MOE_ERR_INVALID_ARG;
  if ((cfg->w_dtype == MOE_FP8_E4M3 || cfg->w_dtype == MOE_INT4) &&
      (!W13_scale || !W2_scale || (cfg->n_shared && (!Ws13_scale || !Ws2_scale))))
    return MOE_ERR_INVALID_ARG;
  if (cfg->d_latent > 0 && (!W_down || !W_up)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_resid, norm_w, W_r, W13, W2, Ws13, Ws2, W_down, W_up, out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  ready(c);
  if (cudaMemsetAsync(c.err, 0, 256, c.st) != cudaSuccess) return MOE_ERR_CUDA;
  const Layout& L = c.L;
  // x_ffn = RMSNorm(x'_n) in the host-I/O staging region, which this entry point does not use
  void* x_ffn = at<void>(ws, L.x_io);
  cudaError_t e = launch_rmsnorm_rows(cfg->act_dtype, x_resid, norm_w, cfg->rms_eps, cfg->T, cfg->d,
                                      x_ffn, c.sms, c.st);
  if (e != cudaSuccess) return from_cuda(e);
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* wgt = at<float>(ws, L.weight);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm_src = at<int32_t>(ws, L.perm_src);
  int32_t* perm_dst = at<int32_t>(ws, L.perm_dst);
  void* y_perm = at<void>(ws, L.y_perm);
  if ((s = run_router(c, x_ffn, W_r, b, nullptr, idx, wgt)) != MOE_OK) return s;
  if ((s = run_permute(c, idx, at<int32_t>(ws, L.counts), offsets, perm_src, perm_dst)) != MOE_OK)
    return s;
  if ((s = run_experts(c, x_ffn, offsets, perm_src, perm_dst, W13, W2, W13_scale, W2_scale, Ws13, Ws2,
                       Ws13_scale, Ws2_scale, W_down, y_perm)) != MOE_OK)
    return s;
  return run_combine(c, y_perm, perm_dst, wgt, W_up, out, x_resid);
}

moe_status_t moe_forward_host_io(const moe_config_t* cfg, const void* x_host, const float* W_r,
                                 const float* b, const void* W13, const void* W2,
                                 const float* W13_scale, const float* W2_scale, const void* Ws13,
                                 const void* Ws2, const float* Ws13_scale, const float* Ws2_scale,
                                 const void* W_down, const void* W_up, void* out_host, void* ws,
                                 size_t ws_bytes, void* stream) {
  Ctx c;
  moe_status_t s = begin(c, cfg, ws, ws_bytes, stream);
  if (s != MOE_OK) return s;
  MOE_RETURN_IF_EMPTY(cfg);
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (!W_r || !b || !W13 || !W2) return MOE_ERR_INVALID_ARG;
  ready(c);
  const size_t bytes = (size_t)cfg->T * cfg->d * dtype_bytes(cfg->act_dtype);
  void* x_dev = at<void>(ws, c.L.x_io);
  void* out_dev = at<void>(ws, c.L.out_io);
  if (bytes < kIoOverlapBytes) {  // one copy each way on the caller's stream
    if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, c.st) != cudaSuccess)
      return MOE_ERR_CUDA;
    s = forward_impl(c, x_dev, W_r, b, W13, W2, W13_scale, W2_scale, Ws13, Ws2, Ws13_scale,
                     Ws2_scale, W_down, W_up, out_dev, nullptr);
    if (s != MOE_OK) return s;
    if (cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, c.st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return from_cuda(cudaStreamSynchronize(c.st));
  }
  // Large batches: the input arrives in kIoStreams pieces on as many copy streams at once, and
  // the output leaves in chunks behind the combine.  The copy streams and their events belong to
  // the device; one such call per device runs at a time (the call synchronises before returning).
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kIoMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_io_mutex);
  IoStreams& io = g_io[dev];
  if (!io.ok && (s = io_streams_init(io)) != MOE_OK) return s;
  // the copies start after the work already queued on the caller's stream (the workspace may
  // still be in use there), and the layer starts after the input copies
  if (cudaEventRecord(io.ev_start, c.st) != cudaSuccess) return MOE_ERR_CUDA;
  // the shared expert chunk by chunk: bf16 token-rows layers in the default tile shapes (the
  // shared rows then equal those of the fused launches bit for bit)
  const bool pipe = c.pl.tc && !c.pl.fp8 && !c.pl.w4 && c.pl.swap == 0 && cfg->n_shared &&
                    Ws13 && Ws2 && aligned16(Ws13) && aligned16(Ws2) &&
                    !(cfg->flags & (MOE_FLAG_GEMM_PAIR | MOE_FLAG_GEMM_M2 | MOE_FLAG_GEMM_N128 |
                                    MOE_FLAG_TEST_STALL_EXPERTS));
  if (pipe) {
    if (cudaMemsetAsync(c.err, 0, 256, c.st) != cudaSuccess) return MOE_ERR_CUDA;
    const int64_t T = cfg->T;
    int64_t chunk = ((T + kIoChunks - 1) / kIoChunks + 127) / 128 * 128;
    if (chunk < kIoMinChunkTokens) chunk = kIoMinChunkTokens;
    const size_t row = (size_t)cfg->d * dtype_bytes(cfg->act_dtype);
    for (int i = 0; i * chunk < T && s == MOE_OK; ++i) {
      const int64_t t0 = i * chunk, nt = T - t0 < chunk ? T - t0 : chunk;
      cudaStream_t cs = io.cs[i % kIoStreams];
      if (cudaStreamWaitEvent(cs, io.ev_start, 0) != cudaSuccess ||
          cudaMemcpyAsync(static_cast<uint8_t*>(x_dev) + (size_t)t0 * row,
                          static_cast<const uint8_t*>(x_host) + (size_t)t0 * row,
                          (size_t)nt * row, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
          cudaEventRecord(io.ev_in_chunk[i], cs) != cudaSuccess ||
          cudaStreamWaitEvent(c.st, io.ev_in_chunk[i], 0) != cudaSuccess)
        s = MOE_ERR_CUDA;
      else
        s = run_shared_rows(c, x_dev, Ws13, Ws2, t0, nt);
    }
    c.shared_done = true;
  } else {
    const size_t piece = (bytes / kIoStreams + 255) & ~size_t(255);
    for (int i = 0; i < kIoStreams; ++i) {
      const size_t o = (size_t)i * piece;
      if (o >= bytes) break;
      const size_t n = bytes - o < piece ? bytes - o : piece;
      if (cudaStreamWaitEvent(io.cs[i], io.ev_start, 0) != cudaSuccess ||
          cudaMemcpyAsync(static_cast<uint8_t*>(x_dev) + o,
                          static_cast<const uint8_t*>(x_host) + o, n, cudaMemcpyHostToDevice,
                          io.cs[i]) != cudaSuccess ||
          cudaEventRecord(io.ev_in[i], io.cs[i]) != cudaSuccess ||
          cudaStreamWaitEvent(c.st, io.ev_in[i], 0) != cudaSuccess) {
        s = MOE_ERR_CUDA;
        break;
      }
    }
  }
  OutCopy oc;
  oc.host = out_host;
  oc.n = kIoChunks;
  for (int i = 0; i < kIoStreams; ++i) oc.cs[i] = io.cs[i];
  for (int i = 0; i < kIoChunks; ++i) oc.ev[i] = io.ev_chunk[i];
  if (s == MOE_OK)
    s = forward_impl(c, x_dev, W_r, b, W13, W2, W13_scale, W2_scale, Ws13, Ws2, Ws13_scale,
                     Ws2_scale, W_down, W_up, out_dev, &oc);
  // whatever was queued on the copy streams (also after a failure above) finishes before the
  // caller's stream goes on
  for (int i = 0; i < kIoStreams; ++i) {
    if (cudaEventRecord(io.ev_out[i], io.cs[i]) != cudaSuccess ||
        cudaStreamWaitEvent(c.st, io.ev_out[i], 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (s != MOE_OK) return s;
  return from_cuda(cudaStreamSynchronize(c.st));
}

// K ranges of the W2 launch: with few tokens its d / 256 output tiles leave most SMs idle, so
// each tile is computed as partial sums over consecutive K ranges (fp32 partials, then one sum
// kernel), as many as one wave of CTAs on 152 SMs holds, at most 8.  1: no split.
static int dense_w2_splits(int64_t T, int32_t d, int32_t I, moe_dtype_t act_dtype) {
  if (act_dtype != MOE_BF16 || T <= 0 || d % 256 || I % 128) return 1;
  const int64_t tiles = ((T + 127) / 128) * (d / 256);
  int64_t s = 152 / tiles;
  if (s > I / 64) s = I / 64;
  if (s > 8) s = 8;
  return s >= 2 ? (int)s : 1;
}

// The dense SwiGLU MLP: one dense group through the expert GEMMs (W1|W3 + SwiGLU -> h in the
// workspace, then W2 straight into `out`, or through fp32 partials over K ranges): token-rows
// tensor-core tiles for bf16, CUDA cores for fp32.
size_t moe_dense_mlp_workspace_size(int64_t T, int32_t d, int32_t I, moe_dtype_t act_dtype) {
  if (T < 0 || d <= 0 || I <= 0 || (act_dtype != MOE_BF16 && act_dtype != MOE_F32)) return 0;
  const int splits = dense_w2_splits(T, d, I, act_dtype);
  return 256 + moe::align256((size_t)T * (size_t)I * moe::dtype_bytes(act_dtype)) +
         (splits > 1 ? moe::align256((size_t)splits * T * d * 4) : 0);
}

moe_status_t moe_dense_mlp(int64_t T, int32_t d, int32_t I, moe_dtype_t act_dtype, const void* x,
                           const void* W13, const void* W2, void* out, void* ws, size_t ws_bytes,
                           void* stream) {
  using namespace moe;
  if (T < 0 || d <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (act_dtype != MOE_BF16 && act_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  const bool tc = act_dtype == MOE_BF16;
  if (tc && (d % 256 || I % 128)) return MOE_ERR_UNSUPPORTED;
  if (!tc && (d % 16 || I % 16)) return MOE_ERR_UNSUPPORTED;
  if (T > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_dense_mlp_workspace_size(T, d, I, act_dtype)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {x, W13, W2, out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = num_sms();
  (void)cudaGetLastError();
  uint32_t* err = at<uint32_t>(ws, 0);
  void* h = at<void>(ws, 256);
  const int splits = dense_w2_splits(T, d, I, act_dtype);
  float* part = at<float>(ws, 256 + align256((size_t)T * (size_t)I * dtype_bytes(act_dtype)));
  if (cudaMemsetAsync(err, 0, 256, st) != cudaSuccess) return MOE_ERR_CUDA;
  // Token-rows tiles in every regime: with few tokens one CTA streams each weight tile once
  // (swap-AB tiles of 32 tokens would have several CTAs stream the same tile, so that only a
  // fraction of the bytes in flight are distinct and HBM runs latency-bound).  W2 then has only
  // d / 256 feature tiles; at small T it is split over K (dense_w2_splits), else its 128-column
  // variant doubles the CTAs streaming it.
  const bool n128_2 = T <= 256 && splits == 1;
  cudaError_t e;
  {
    GroupedGemm g;
    g.act_d = x;
    g.act_d_rows = T;
    g.w_d = W13;
    g.w_d_rows = 2 * (int64_t)I;
    g.dense_rows = (int)T;
    g.u_off_d = I;
    g.K = d;
    g.k_wrap = d;
    g.F = I;
    g.epi = EPI_SWIGLU;
    g.act_dtype = g.w_dtype = act_dtype;
    g.out = h;
    g.ldo = I;
    g.out_dtype = act_dtype;
    g.err = err;
    g.label = tc ? "dense_gemm13_swiglu_rows" : "dense_gemm13_swiglu_simt";
    e = tc ? launch_gemm_tc(g, 0, sms, st) : launch_gemm_simt(g, sms, st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  {
    GroupedGemm g;
    g.act_d = h;
    g.act_d_rows = T;
    g.w_d = W2;
    g.w_d_rows = d;
    g.dense_rows = (int)T;
    g.K = I;
    g.k_wrap = I;
    g.F = d;
    g.epi = EPI_STORE;
    g.act_dtype = g.w_dtype = act_dtype;
    g.out = splits > 1 ? static_cast<void*>(part) : out;
    g.ldo = d;
    g.out_dtype = splits > 1 ? MOE_F32 : act_dtype;
    g.k_splits = splits;
    g.split_stride = T * d;
    g.err = err;
    g.n128 = n128_2;
    g.label = !tc ? "dense_gemm2_simt" : splits > 1 ? "dense_gemm2_rows_splitk" : "dense_gemm2_rows";
    e = tc ? launch_gemm_tc(g, 0, sms, st) : launch_gemm_simt(g, sms, st);
    if (e != cudaSuccess) return from_cuda(e);
    if (splits > 1) {
      e = launch_splitk_sum(part, splits, T * d, out, sms, st);
      if (e != cudaSuccess) return from_cuda(e);
    }
  }
  return MOE_OK;
}

moe_status_t moe_reset_device_status(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  return from_cuda(cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_device_status(const void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t flags = 0;
  if (cudaMemcpy(&flags, ws, sizeof flags, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (flags & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (flags & kErrIndex) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error_string(void) { return g_last_error; }

uint64_t moe_launch_count(void) { return g_launches; }
void moe_reset_launch_count(void) { g_launches = 0; }

moe_status_t moe_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return MOE_OK;
}

int moe_profile_read(int max_entries, char* names, size_t name_len, double* total_ms,
                     uint64_t* launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const ProfRecord& r : g_prof_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      bool found = false;
      for (ProfTotal& t : g_prof_totals)
        if (t.name == r.name) {
          t.ms += ms;
          ++t.launches;
          found = true;
          break;
        }
      if (!found) g_prof_totals.push_back({r.name, (double)ms, 1});
    }
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_pending.clear();
  int n = 0;
  for (const ProfTotal& t : g_prof_totals) {
    if (n >= max_entries) break;
    if (names && name_len > 0) {
      std::strncpy(names + (size_t)n * name_len, t.name.c_str(), name_len - 1);
      names[(size_t)n * name_len + name_len - 1] = '\0';
    }
    if (total_ms) total_ms[n] = t.ms;
    if (launches) launches[n] = t.launches;
    ++n;
  }
  g_prof_totals.clear();
  return n;
}

}  // extern "C"
