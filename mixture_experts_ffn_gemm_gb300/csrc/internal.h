// internal.h -- host-side interfaces between the C ABI (moe_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Flags of the device status word (first word of the workspace).
enum : uint32_t {
  kErrTimeout = 1u,  // a bounded wait expired
  kErrIndex = 2u,    // an expert index / row outside its range was skipped
};

enum Epi { EPI_SWIGLU = 0, EPI_STORE = 1, EPI_STORE_ADD = 2 };

// A grouped GEMM  out[row][f] = sum_k act[row][k] * w[wrow(f)][k]  over groups of rows, with the
// SwiGLU epilogue h = SiLU(g) * u (g from the W1 row f, u from the W3 row f + u_off) or a plain
// store (optionally plus a bf16 addend).
struct GroupedGemm {
  // routed groups: rows [offsets[g], offsets[g+1]) of act, weights rows [g*w_group_rows, ...)
  const void* act = nullptr;  // [act_rows][K]
  int64_t act_rows = 0;
  const void* w = nullptr;    // [w_rows][K]
  int64_t w_rows = 0;
  const int32_t* offsets = nullptr;  // device [n_routed + 1]
  int n_routed = 0;
  int w_group_rows = 0;
  int u_off = 0;
  // trailing dense group (shared expert or a dense projection)
  const void* act_d = nullptr;  // [act_d_rows][K]
  int64_t act_d_rows = 0;
  int dense_act_row0 = 0;
  const void* w_d = nullptr;    // [w_d_rows][K]
  int64_t w_d_rows = 0;
  int dense_rows = 0;
  int dense_out_row0 = 0;
  int u_off_d = 0;
  // shapes
  int K = 0;
  int k_wrap = 0;  // activation column = k mod k_wrap (3-way split router); K when unused
  int F = 0;       // output features per group
  // the dense group's own reduction length, features and output (0 / null: as the routed ones)
  int K_d = 0;
  int k_wrap_d = 0;
  int F_d = 0;
  void* out_d = nullptr;
  int64_t ldo_d = 0;
  int epi = EPI_STORE;
  int act_dtype = MOE_BF16;
  int w_dtype = MOE_BF16;
  // output
  void* out = nullptr;
  int64_t ldo = 0;
  int out_dtype = MOE_BF16;
  const void* addend = nullptr;  // EPI_STORE_ADD: fp32 [rows][ld_add], indexed like out
  int64_t ld_add = 0;
  // split-K (the SIMT router; dense-only tensor-core fp32 stores): the partial sum over the s-th
  // of k_splits consecutive K ranges at out + s * split_stride elements
  int k_splits = 1;
  int64_t split_stride = 0;
  uint32_t* err = nullptr;
  const char* label = "gemm";  // kernel name for the launch profiler
  bool test_stall = false;     // test hook (MOE_FLAG_TEST_STALL_EXPERTS): see moe.h
  bool n128 = false;           // token-rows store tiles with N = 128 (MOE_FLAG_GEMM_N128)
  int m_halves = 0;            // token-rows SwiGLU tiles of 1 or 2 M halves (0: one)
  bool pair = false;           // token-rows tiles of 256 rows on a CTA pair (cta_group::2)
  bool big_boxes = true;       // token-rows N = 256 tiles: the weights in one copy per stage
};

// Tensor-core grouped GEMM (tcgen05 + TMA), bf16 operands, fp32 accumulation in TMEM.
// swap = 0: token rows are the MMA M side (128-row tiles), weights the N side.
// swap = 1: weight rows are the M side, tokens the N side (32-token tiles), for few rows per group.
// swap = 2: as 1 with 256-token tiles; the MMA's N is each tile's token count rounded up to 16
//           (SwiGLU and plain store only).
// Requires K % 64 == 0, F % 128 == 0 (F % 256 == 0 for swap = 0 stores).  Returns a CUDA error or
// cudaErrorInvalidValue when the shapes are not supported (nothing launched).
cudaError_t launch_gemm_tc(const GroupedGemm& g, int swap, int num_sms, cudaStream_t st);
bool gemm_tc_supported(const GroupedGemm& g, int swap);
// A TMA map over a bf16 [rows][cols] matrix (cols contiguous): box {64 cols, box_rows rows},
// 128-byte swizzle, out-of-range elements read as zero.  False when the driver refuses it.
bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows);

// The decode experts in one persistent launch (bf16, 32-token swap-AB tiles): W1|W3 + SwiGLU into
// h, then W2 into the fp32 expert outputs, each W2 tile starting once the h tiles of its rows are
// written.  Routed groups by offsets plus the shared expert as a trailing dense group of T rows.
//   x_perm [P][d], x [T][d], W13 [E][2I][d], Ws13 [2I][d], W2 [E][d][I], Ws2 [d][I],
//   h [P+T][I] (out, then in), y [P+T][d] fp32 (out), ready [fused_ready_count(T, k, E)] zeroed.
// Needs d % 128 == 0, I % 128 == 0 and a cooperative launch of one CTA per SM (the W2 tiles wait
// on W1|W3 tiles of other CTAs); returns cudaErrorCooperativeLaunchTooLarge when that is refused.
struct FusedDecode {
  const void* x_perm = nullptr;
  const void* x = nullptr;
  const void* W13 = nullptr;
  const void* Ws13 = nullptr;
  const void* W2 = nullptr;
  const void* Ws2 = nullptr;
  const int32_t* offsets = nullptr;
  int n_routed = 0;
  int64_t T = 0;   // tokens (the shared expert's rows; 0 without a shared expert)
  int64_t P = 0;   // routed rows (T * k)
  int d = 0;
  int I = 0;
  void* h = nullptr;
  float* y = nullptr;
  uint32_t* ready = nullptr;
  uint32_t* err = nullptr;
  const char* label = "experts_fused_swap";
};
int64_t fused_ready_count(int64_t T, int k, int E);
cudaError_t launch_decode_fused(const FusedDecode& f, int num_sms, cudaStream_t st);

// Grouped GEMM with e4m3 operands and fp32 block scales (tcgen05 kind::f8f6f4), token-rows tiles
// M = 128 x 256 weight rows.  Activation scales per row per 128 channels, stored [K/128][ld];
// weight scales per 128 x 128 block, [rows/128][K/128].  swiglu: out = e4m3 h [rows][ldo] with
// scales out_sT [F/128][out_s_ld]; else fp32 out [rows][ldo].
struct Fp8Gemm {
  const void* act = nullptr;
  int64_t act_rows = 0;
  const float* act_sT = nullptr;
  int64_t act_s_ld = 0;
  const void* w = nullptr;
  int64_t w_rows = 0;
  const float* w_s = nullptr;
  const int32_t* offsets = nullptr;
  int n_routed = 0;
  int w_group_rows = 0;
  int u_off = 0;
  const void* act_d = nullptr;
  int64_t act_d_rows = 0;
  const float* act_sT_d = nullptr;
  int64_t act_s_ld_d = 0;
  int dense_act_row0 = 0;
  const void* w_d = nullptr;
  int64_t w_d_rows = 0;
  const float* w_s_d = nullptr;
  int dense_rows = 0;
  int dense_out_row0 = 0;
  int u_off_d = 0;
  int K = 0;
  int F = 0;
  bool swiglu = false;
  void* out = nullptr;
  int64_t ldo = 0;
  float* out_sT = nullptr;
  int64_t out_s_ld = 0;
  bool out_bf16 = false;  // store mode: bf16 outputs instead of fp32
  uint32_t* err = nullptr;
  const char* label = "gemm_fp8";
};
cudaError_t launch_gemm_fp8(const Fp8Gemm& g, int num_sms, cudaStream_t st);

// Grouped GEMM with 4-bit integer group-quantised weights (packed [w_rows][K/2]; bf16 scales per
// weight group, [n_routed][K/32][w_group_rows] for the routed experts and [K/32][w_d_rows] for the
// dense group) and bf16 activations, swap-AB tiles: M = 128 weight rows, N = up to 32 tokens.
// swiglu: out = bf16 h [rows][ldo] (W3 rows at +u_off); else fp32 out [rows][ldo].
struct W4Gemm {
  const void* act = nullptr;
  int64_t act_rows = 0;
  const void* wq = nullptr;
  const void* ws = nullptr;
  int64_t w_rows = 0;
  const int32_t* offsets = nullptr;
  int n_routed = 0;
  int w_group_rows = 0;
  int u_off = 0;
  const void* act_d = nullptr;
  int64_t act_d_rows = 0;
  int dense_act_row0 = 0;
  const void* wq_d = nullptr;
  const void* ws_d = nullptr;
  int64_t w_d_rows = 0;
  int dense_rows = 0;
  int dense_out_row0 = 0;
  int u_off_d = 0;
  int K = 0;
  int F = 0;
  bool swiglu = false;
  void* out = nullptr;
  int64_t ldo = 0;
  uint32_t* err = nullptr;
  const char* label = "gemm_w4";
};
cudaError_t launch_gemm_w4(const W4Gemm& g, int num_sms, cudaStream_t st);

// x bf16 [rows][d] -> e4m3 codes [rows][d] and scales sT [d/128][rows] (amax / 448 per 128).
cudaError_t launch_quantize_rows(const void* x, int64_t rows, int d, uint8_t* q, float* sT,
                                 cudaStream_t st);

// CUDA-core grouped GEMM (fp32 or bf16 operands, fp32 accumulation), 64x64 tiles.
cudaError_t launch_gemm_simt(const GroupedGemm& g, int num_sms, cudaStream_t st);

// Router: selection and gates from logits (split-K partial slices summed in a fixed order).
cudaError_t launch_router_topk(const float* partial, int S, int64_t split_stride, int64_t T,
                               int E, int k, const float* b, float gate_scale, float* logits_out,
                               int32_t* idx, float* weight, cudaStream_t st);
// Router logits of a small batch on the tensor cores: bf16 x [T][d] times fp32 W_r [E][d] (split
// into three bf16 parts inside the kernel), K cut into S slices of partial logits at
// z + s * split_stride ([T][E] each), summed in order by launch_router_topk.
bool router_splitk_tc_supported(int64_t T, int E, int d);
int router_splitk_tc_slices(int64_t T, int E, int d, int num_sms);
cudaError_t launch_router_splitk_tc(const void* x, const float* W_r, int64_t T, int E, int d,
                                    int S, float* z, int64_t split_stride, uint32_t* err,
                                    cudaStream_t st);
// fp32 [E][d] -> bf16 [E][3d] (hi | mid | lo) so that hi + mid + lo reproduces each weight.
cudaError_t launch_split_router_weights(const float* W_r, int E, int d, __nv_bfloat16* out,
                                        cudaStream_t st);

// Permute: histogram, scan, stable scatter.
int permute_chunks(int64_t P);
cudaError_t launch_permute(const int32_t* idx, int64_t T, int k, int E, int n_shared,
                           int32_t* chunk_counts, int32_t* counts, int32_t* offsets,
                           int32_t* perm_src, int32_t* perm_dst, uint32_t* err, cudaStream_t st);
// dst[perm_dst[t*k + j]] = src[t] for every token and slot: the activation rows in the
// expert-major order, each source row read once (rows of `width` elements of elem_bytes each);
// destinations outside [0, P) are skipped.
cudaError_t launch_scatter_rows(const void* src, const int32_t* perm_dst, int64_t T, int k,
                                int64_t P, int width, int elem_bytes, void* dst, int num_sms,
                                cudaStream_t st);
// e4m3 rows of d bytes with their scales (transposed layouts), token-major likewise.
cudaError_t launch_scatter_q(const uint8_t* src, const float* src_sT, int64_t T,
                             const int32_t* perm_dst, int k, int64_t P, int d, uint8_t* dst,
                             float* dst_sT, int num_sms, cudaStream_t st);
// perm_dst = the inverse of perm_src (-1 where no pair lands).
cudaError_t launch_invert_perm(const int32_t* perm_src, int64_t P, int32_t* perm_dst, int num_sms,
                               cudaStream_t st);

// Combine: out[t] = sum_j w[t,j] * y[perm_dst[t*k+j]] + y_shared[t] (+ resid[t]); y fp32, fp32
// sum, one rounding to act_dtype.  resid (act_dtype) and y_shared may be null.
// y_perm and y_shared in fp32, or in bf16 when y_bf16 is set.
cudaError_t launch_combine(int act_dtype, bool y_bf16, const void* y_perm, const void* y_shared,
                           const int32_t* perm_dst, const float* weight, int64_t T, int k,
                           int64_t P, int d, const void* resid, void* out, int num_sms,
                           cudaStream_t st);
// Block steps: y = w * x / sqrt(mean(x^2) + eps) per row (fp32, one rounding to act_dtype); and
// y_f32 += r (r in act_dtype, n elements, n % 8 == 0).
cudaError_t launch_rmsnorm_rows(int act_dtype, const void* x, const void* w, float eps, int64_t T,
                                int d, void* y, int num_sms, cudaStream_t st);
cudaError_t launch_add_residual(float* y, int act_dtype, const void* r, int64_t n, int num_sms,
                                cudaStream_t st);
// out (bf16, n values) = the fp32 sum of S partials part[s * n .. s * n + n), in slice order,
// rounded once; 1 <= S <= 8, n % 8 == 0.
cudaError_t launch_splitk_sum(const float* part, int S, int64_t n, void* out, int num_sms,
                              cudaStream_t st);
// K3: u_hat[t] = RMSNorm?( sum_j w[t,j] * y[perm_dst[t*k+j]] ) in bf16, width L, y fp32 [P][L].
cudaError_t launch_latent_combine(const void* y_perm, const int32_t* perm_dst,
                                  const float* weight, int64_t T, int k, int64_t P, int L,
                                  int norm, float eps, void* u_hat, int num_sms,
                                  cudaStream_t st);

// A failed CUDA call as a status: MOE_OK for cudaSuccess, else MOE_ERR_CUDA with the error's name
// and text kept for moe_last_error_string() (per host thread).
moe_status_t status_from_cuda(cudaError_t e);

// Brackets one kernel launch: counts it (per host thread) and, while profiling is enabled
// (moe_profile_enable), records a CUDA event pair around it on the launch stream.
class LaunchScope {
 public:
  LaunchScope(const char* name, cudaStream_t st);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  const char* name_;
  cudaStream_t st_;
  cudaEvent_t start_ = nullptr;
};

}  // namespace moe
