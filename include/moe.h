/*
 * moe.h -- C ABI of the GB300 (sm_103a) mixture-of-experts FFN layer library (libmoe_gb300.so).
 *
 * The layer is the Kimi K2 / DeepSeek-V3 MoE feed-forward block and the Kimi K3 latent variant:
 *
 *   z = x W_r ; s = sigma(z) ; selected = top_k(s + b) ; G_i = gate_scale * s_i / sum_sel s_j
 *   E_i(x) = (SiLU(x W1_i) * (x W3_i)) W2_i ;  y = sum_sel G_i E_i(x) + E_shared(x)
 *
 * Sources (page title and section):
 *   [K2-MoE]   "Kimi K2 · Transformer blocks > MoE transformer block", "Mixture of experts" steps.
 *   [K2-PARAM] same page, "Parameters" table (exact per-instance accounting).
 *   [NN-MOE]   nnterp encyclopedia "kimi_k2", note "The mixture of experts" (bias selects only;
 *              gates are renormalised unbiased sigmoids times 2.827; routed + shared = output).
 *   [NN-API]   nnterp "kimi_k2", "02 · support()" (router_logits, expert_weights, expert_indices,
 *              routed_output, shared_expert_output and their layouts).
 *   [NN-CFG]   nnterp "kimi_k2", "Config" table (hidden 7168, 384 experts, top 8, moe intermediate
 *              2048, 1 shared expert, routed_scaling_factor 2.827, n_group 1, rms_norm_eps 1e-6).
 *   [K3-UP]    "Kimi K3 · Latent up-projection": equation y_routed = u_hat W_up, parameter table,
 *              and the `__init__`, `forward` and `moe_infer` code excerpts (dispatch by expert,
 *              per-expert MLP, un-permute, gate-weighted sum; latent down/up projections, RMSNorm).
 *   [NN-PRINT] nnterp "kimi_k2", "Printout": layer 0's `mlp` is a dense DeepseekV3MLP
 *              (gate_proj, up_proj 7168 -> 18432, down_proj 18432 -> 7168, SiLU).
 *   [K2-CODE]  "Kimi K2 · Transformer blocks", the modeling_deepseek excerpt that builds the dense
 *              MLP instead of the MoE for blocks below first_k_dense_replace.
 *
 * Conventions for every entry point
 *   - Pointers named x, W*, b, out, logits, topk_*, counts, offsets, perm_*, y_perm and ws are
 *     DEVICE pointers on the current CUDA device; the library never allocates, frees or copies to
 *     the host on these paths.  The caller owns every buffer, the workspace included.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).  Calls
 *     return once the work is enqueued: execution errors surface at the caller's next
 *     synchronisation, and device-side checks (index range, bounded waits) raise flags in the first
 *     word of the workspace, read with moe_device_status().
 *   - Layouts are row-major.  Weights are stored [out][in] as on the pages ("The reference module
 *     holds the weight output by input"), i.e. K-contiguous.
 *   - Every pointer must be 16-byte aligned; every row pitch is the row's width (no padding).
 *   - Errors are return codes; nothing is launched when host validation fails.
 *   - T == 0 is valid: once the configuration and workspace pass validation every entry point
 *     returns MOE_OK without touching any other pointer (empty tensors may be NULL).
 *   - The functions hold no state between calls other than cached kernel attributes and the
 *     driver entry point of cuTensorMapEncodeTiled; they are safe to call from several threads on
 *     distinct workspaces.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, inconsistent shape                     */
  MOE_ERR_UNSUPPORTED = 2,  /* a shape or dtype combination this build does not implement        */
  MOE_ERR_WORKSPACE = 3,    /* ws is null or smaller than moe_workspace_size()                   */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed at launch time                */
  MOE_ERR_DEVICE_CHECK = 5, /* a kernel found an out-of-range expert index or row                */
  MOE_ERR_TIMEOUT = 6       /* a kernel gave up a bounded wait (pipeline stalled) and returned   */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8_E4M3 = 2, MOE_INT4 = 3 } moe_dtype_t;

/* MOE_INT4 expert weights ("4-bit integer groups", the storage of K2-Thinking and K2.5 per the
 * nnterp "kimi_k2" page; bf16 activations):
 *   - a weight matrix [rows][K] is stored packed, [rows][K/2] bytes, eight codes per 32-bit
 *     little-endian word: code i of the word (input channel 8w + i) is the 4-bit nibble number
 *     (i / 2) + 4 * (i % 2), counted from bit 0;
 *   - a nibble u encodes the integer u - 8 (excess-8, -8..7);
 *   - one bf16 scale per 32 consecutive input channels of each row, stored transposed,
 *     [K/32][rows];
 *   - the weight is RN_bf16((u - 8) * scale): the product rounded once to bf16, the MMA operand.
 * W13 is then [E][2I][d/2] packed with W13_scale [E][d/32][2I]; W2 [E][d][I/2] with W2_scale
 * [E][I/32][d]; the shared expert likewise ([2 I_s][d/2], [d/32][2 I_s]; [d][I_s/2], [I_s/32][d]).
 * The *_scale arguments then point to bf16 data.  quant_block must be 32. */

/* moe_config_t.flags */
#define MOE_FLAG_GEMM_ROWS_MAJOR 0x1u /* force the token-rows-as-M tensor-core GEMM tiles       */
#define MOE_FLAG_GEMM_SWAP_AB 0x2u    /* force the weight-rows-as-M (swap-AB) GEMM tiles         */
#define MOE_FLAG_ROUTER_SIMT 0x4u     /* force the CUDA-core fp32 router GEMM                    */
#define MOE_FLAG_ROUTER_TC 0x8u       /* force the tensor-core (3 x bf16 split) router GEMM      */
#define MOE_FLAG_GEMM_N128 0x10u      /* token-rows tiles of the store GEMMs with N = 128 columns  */
#define MOE_FLAG_GEMM_SWAP_WIDE 0x20u /* force weight-rows-as-M tiles of 256 tokens (runtime N)  */
#define MOE_FLAG_GEMM_M1 0x40u        /* token-rows SwiGLU tiles of one 128-row M half            */
#define MOE_FLAG_GEMM_M2 0x80u        /* token-rows SwiGLU tiles of two 128-row M halves (256 rows)
                                       * sharing each weight K-block (slower: kept for comparison) */
#define MOE_FLAG_DECODE_FUSED 0x200u  /* decode batches (32-token swap-AB tiles): the expert
                                       * GEMMs in one persistent launch (W1|W3 + SwiGLU tiles,
                                       * then W2 tiles that wait for their h rows) instead of two
                                       * launches; same results bit for bit, measured slower      */
#define MOE_FLAG_GEMM_PAIR 0x400u     /* token-rows expert GEMM tiles of 256 rows on a pair of SMs
                                       * (one M = 256 tensor-core MMA over both SMs' operands)     */
#define MOE_FLAG_EXPERT_OUT_BF16 0x800u /* expert outputs (y_perm, the shared expert's rows) in
                                       * bf16 instead of fp32: half their bytes, one more rounding
                                       * of every expert output before the gated sum.  bf16 or
                                       * e4m3 experts on the K2 path only (else
                                       * MOE_ERR_UNSUPPORTED); moe_experts then writes, and
                                       * moe_combine reads, bf16 y_perm.  The default for e4m3
                                       * experts                                                  */
#define MOE_FLAG_EXPERT_OUT_F32 0x1000u /* fp32 expert outputs for e4m3 experts too            */
/* Test hook for the failure path: the tensor-core W1|W3 expert GEMM's copy producer issues no
 * copy, so its MMA issuer's bounded wait (shortened to 50 ms under this flag) expires; the kernel
 * flags MOE_ERR_TIMEOUT in the device status, drains, frees its tensor memory and returns, and
 * the layer's output is incomplete.  Never set in normal use. */
#define MOE_FLAG_TEST_STALL_EXPERTS 0x100u

/* Layer shapes and constants.  Names follow [NN-CFG]. */
typedef struct {
  int64_t T;           /* tokens (batch x positions), >= 0                                       */
  int32_t d;           /* hidden size (7168)                                                     */
  int32_t E;           /* routed experts (384)                                                   */
  int32_t k;           /* experts per token (8), 1 <= k <= E, k <= 32                            */
  int32_t I;           /* routed expert intermediate size (2048)                                 */
  int32_t I_shared;    /* shared expert intermediate size (2048 = I x n_shared_experts)          */
  int32_t n_shared;    /* 0 or 1 shared expert                                                   */
  int32_t d_latent;    /* 0: K2 path; L > 0: K3 latent width (3584) [K3-UP]                      */
  int32_t latent_norm; /* 1: RMSNorm with unit weight on the latent gate-weighted sum [K3-UP]    */
  int32_t act_dtype;   /* MOE_F32 or MOE_BF16: x, out, W_down, W_up, intermediates               */
  int32_t w_dtype;     /* expert weights: act_dtype, MOE_FP8_E4M3 (block scales) or MOE_INT4      */
  int32_t quant_block; /* fp8: block edge 128 (weights 128x128, activations 1x128); int4: group 32 */
  uint32_t flags;      /* MOE_FLAG_* tuning overrides; 0 = automatic choice                      */
  float gate_scale;    /* routed_scaling_factor (2.827) [NN-CFG]                                 */
  float rms_eps;       /* rms_norm_eps (1e-6) [NN-CFG]                                           */
  int32_t reserved_;   /* must be 0                                                              */
} moe_config_t;

/* Bytes of device workspace every entry point below needs for this configuration.  The first
 * 256 bytes hold the device status word (see moe_device_status).  Returns 0 for an invalid
 * configuration. */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Router, selection and gates [K2-MoE] steps z, s, E_sel, G; [NN-MOE]; [NN-API] router_logits,
 * expert_indices, expert_weights.
 *   x            [T][d]  act_dtype
 *   W_r          [E][d]  fp32 (one logit per expert)
 *   b            [E]     fp32 selection bias (used for the selection only)
 *   logits       [T][E]  fp32 out, z = x W_r^T, or NULL
 *   topk_idx     [T][k]  int32 out: the k experts with the largest s + b, slot order by s + b
 *                        descending, equal keys ordered by the lower expert index
 *   topk_weight  [T][k]  fp32 out: gate_scale * s_i / sum of the selected s (unbiased sigmoids);
 *                        sums to gate_scale per token
 * s = 1/(1+exp(-z)) and s + b are evaluated in fp32. */
moe_status_t moe_router(const moe_config_t* cfg, const void* x, const float* W_r, const float* b,
                        float* logits, int32_t* topk_idx, float* topk_weight, void* ws,
                        size_t ws_bytes, void* stream);

/* Dispatch bookkeeping: the `moe_infer` front half of [K3-UP] (per-expert token counts and the
 * expert-major order of the (token, slot) pairs), without the host synchronisation.
 *   topk_idx  [T][k]   int32 in; pair p = t*k + j
 *   counts    [E+1]    int32 out: rows of each routed expert; counts[E] = T*n_shared (the shared
 *                      expert's rows, every token)
 *   offsets   [E+2]    int32 out: exclusive prefix sum of counts (offsets[E] = T*k,
 *                      offsets[E+1] = T*k + T*n_shared)
 *   perm_src  [T*k]    int32 out: permuted row r holds pair perm_src[r]; rows of one expert are
 *                      contiguous and in increasing pair order (a stable sort by expert)
 *   perm_dst  [T*k]    int32 out: inverse permutation, perm_src[perm_dst[p]] == p
 * An index outside [0, E) raises MOE_ERR_DEVICE_CHECK in the device status and is not counted. */
moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_idx, int32_t* counts,
                         int32_t* offsets, int32_t* perm_src, int32_t* perm_dst, void* ws,
                         size_t ws_bytes, void* stream);

/* moe_permute for callers that cannot allocate device memory.  The pages have no counterpart:
 * this is a deployment variant of the dispatch bookkeeping above, with the same arguments and
 * results except the workspace.  Callers that cannot call cudaMalloc at routing time need it: a
 * serving process that gave the GPU's free memory to its own pool at start-up, or a
 * latency-critical loop where cudaMalloc may synchronise the device.  Its scratch (the per-chunk
 * expert counts) is a fixed 1 MiB array of device global memory inside the library, held by every
 * GPU that loads the library until the process exits; no memory is allocated.
 *   Limits: T*k <= 262144 and E <= 1023; larger sizes return MOE_ERR_UNSUPPORTED and enqueue
 *   nothing.  There is no status word: an expert index outside [0, E) is skipped (not counted)
 *   and its perm_dst entry is set to -1.
 *   Every call made outside stream capture looks up the array's device address
 *   (cudaGetSymbolAddress) with the current device, so the address stays right after a
 *   cudaDeviceReset.  A call made during capture uses the address found by the last call outside
 *   capture on that device: make at least one call on each device before any stream capture
 *   (otherwise the captured call returns MOE_ERR_CUDA and enqueues nothing).  CUDA errors leave
 *   their text for moe_last_error_string().
 *   Every call on a device shares the one array: calls whose GPU work overlaps (for example on
 *   two streams at once) race on it and produce wrong results, so serialise them. */
moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_idx,
                                 int32_t* counts, int32_t* offsets, int32_t* perm_src,
                                 int32_t* perm_dst, void* stream);

/* Expert MLPs [K2-MoE] steps g, u, a, h, E_i and y_shared; the per-expert loop of `moe_infer`
 * [K3-UP] as grouped GEMMs over the permuted rows; on the K3 path the down-projection
 * x_lat = x W_down^T first [K3-UP].
 *   x         [T][d]               act_dtype
 *   offsets   [E+2], perm_src [T*k] from moe_permute
 *   W13       [E][2I][d_e]         rows 0..I-1 = W1 (gate_proj), rows I..2I-1 = W3 (up_proj);
 *                                  d_e = d (K2) or d_latent (K3); w_dtype
 *   W2        [E][d_e][I]          down_proj; w_dtype
 *   W13_scale [E][2I/qb][d_e/qb], W2_scale [E][d_e/qb][I/qb]   fp32 block scales, fp8 only
 *   Ws13      [2 I_shared][d], Ws2 [d][I_shared] (+ Ws13_scale, Ws2_scale for fp8); NULL when
 *             n_shared == 0
 *   W_down    [d_latent][d] act_dtype, K3 only (else NULL)
 *   y_perm    out, fp32: [T*k][d_e] un-weighted expert outputs in permuted row order, followed
 *             by [T*n_shared][d] shared-expert outputs in token order (kept in fp32 so that the
 *             gate-weighted sum in moe_combine rounds only once).  bf16, same layout, for e4m3
 *             experts (unless MOE_FLAG_EXPERT_OUT_F32) and under MOE_FLAG_EXPERT_OUT_BF16.
 * fp8 (w_dtype MOE_FP8_E4M3): the activations entering both GEMMs are quantised per token per
 * quant_block channels to e4m3 with scale = amax/448 (1 for an all-zero group), accumulation in
 * fp32. */
moe_status_t moe_experts(const moe_config_t* cfg, const void* x, const int32_t* offsets,
                         const int32_t* perm_src, const void* W13, const void* W2,
                         const float* W13_scale, const float* W2_scale, const void* Ws13,
                         const void* Ws2, const float* Ws13_scale, const float* Ws2_scale,
                         const void* W_down, void* y_perm, void* ws, size_t ws_bytes,
                         void* stream);

/* Un-permute and gate-weighted sum, plus the shared expert: [K2-MoE] y_routed = sum_i G_i E_i,
 * D_ffn = y_routed + y_shared; the `moe_infer` back half of [K3-UP]; on the K3 path the RMSNorm of
 * the latent sum (when latent_norm) and the up-projection y_routed = u_hat W_up^T [K3-UP].
 *   y_perm       from moe_experts;  perm_dst [T*k] from moe_permute
 *   topk_weight  [T][k] fp32 from moe_router
 *   W_up         [d][d_latent] act_dtype, K3 only (else NULL)
 *   out          [T][d] act_dtype: D_ffn.  The sum is taken in fp32 and rounded once. */
moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* perm_dst,
                         const float* topk_weight, const void* W_up, void* out, void* ws,
                         size_t ws_bytes, void* stream);

/* The whole layer: moe_router -> moe_permute -> moe_experts -> moe_combine, with every
 * intermediate in the workspace, enqueued on one stream with no host synchronisation.
 * Arguments as above.  Clears the device status word on entry. */
moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const float* W_r, const float* b,
                         const void* W13, const void* W2, const float* W13_scale,
                         const float* W2_scale, const void* Ws13, const void* Ws2,
                         const float* Ws13_scale, const float* Ws2_scale, const void* W_down,
                         const void* W_up, void* out, void* ws, size_t ws_bytes, void* stream);

/* The FFN half of a transformer block with the layer inside it, [K2-MoE] "x_ffn = RMSNorm(x'_n)",
 * the "Mixture of experts" steps, and "x_{n+1} = x'_n + D_ffn" ([NN-PRINT]: the post-attention
 * norm is DeepseekV3RMSNorm((7168,), eps=1e-06); [K2-PARAM]: "MoE RMSNorm" has 7168 weights).
 *   x_resid   [T][d] act_dtype: x'_n, the residual stream entering the FFN half
 *   norm_w    [d] act_dtype: the RMSNorm weight
 *   out       [T][d] act_dtype: x'_n + D_ffn(norm_w * x'_n / sqrt(mean(x'_n^2) + rms_eps))
 *   other arguments as moe_forward
 * The normalised input is computed in fp32 and rounded once to act_dtype (the router and expert
 * GEMMs' operand); the residual is added inside the combine (on the K3 path, to the fp32
 * shared-expert rows that the up-projection adds), before the output's single rounding.  The K3
 * path needs its shared expert (n_shared = 1), else MOE_ERR_UNSUPPORTED. */
moe_status_t moe_forward_block(const moe_config_t* cfg, const void* x_resid, const void* norm_w,
                               const float* W_r, const float* b, const void* W13, const void* W2,
                               const float* W13_scale, const float* W2_scale, const void* Ws13,
                               const void* Ws2, const float* Ws13_scale, const float* Ws2_scale,
                               const void* W_down, const void* W_up, void* out, void* ws,
                               size_t ws_bytes, void* stream);

/* The whole layer from HOST buffers: copies x (pinned or pageable host memory, [T][d] act_dtype)
 * to the workspace, runs moe_forward on resident device weights, and copies the output back to
 * out_host ([T][d] act_dtype).  Synchronises `stream` before returning.  Weights stay device
 * pointers.  From 32 MB of input on, the copies overlap: x arrives in up to eight token chunks of
 * at least 2048 tokens on two copy streams, and for bf16 layers with a shared expert (default
 * tile shapes) each chunk's shared-expert rows are computed while the next chunk is copied, with
 * the same kernels and results bit for bit as in moe_forward, where the shared expert rides in
 * the routed launches; otherwise x arrives in two pieces at once.  The output leaves in eight
 * token chunks, each copied while the next is combined.  Those copy streams and their events are
 * created once per device and shared, so such calls on one device are serialised by a lock for
 * their duration. */
moe_status_t moe_forward_host_io(const moe_config_t* cfg, const void* x_host, const float* W_r,
                                 const float* b, const void* W13, const void* W2,
                                 const float* W13_scale, const float* W2_scale, const void* Ws13,
                                 const void* Ws2, const float* Ws13_scale, const float* Ws2_scale,
                                 const void* W_down, const void* W_up, void* out_host, void* ws,
                                 size_t ws_bytes, void* stream);

/* The dense SwiGLU MLP of the first block(s), [NN-PRINT] and [K2-CODE]:
 *   y = (SiLU(x W1^T) * (x W3^T)) W2^T, with no router, experts or gates.
 * It runs on the same grouped GEMM kernels as the experts, as one dense group (token-rows tiles).
 * With bf16 and few tokens the W2 GEMM has too few output tiles to keep the GPU's memory busy: its
 * tiles are then split over up to 8 consecutive ranges of I into fp32 partial sums, which one
 * more kernel adds in range order and rounds once to bf16 (T <= 256 with no split: 128-column
 * tiles instead).
 *   T, d, I     tokens, hidden width, intermediate width (d % 256 == 0 and I % 128 == 0 for
 *               bf16; d % 16 == 0 and I % 16 == 0 for fp32)
 *   act_dtype   MOE_BF16 (tensor cores, fp32 accumulation, h rounded to bf16) or MOE_F32
 *               (CUDA cores); x, W13, W2 and out all have this type
 *   x           [T][d]
 *   W13         [2I][d]: the I rows of W1 (gate_proj), then the I rows of W3 (up_proj)
 *   W2          [d][I]   (down_proj)
 *   out         [T][d]   y, each element rounded once from its fp32 accumulation
 *   ws          workspace of at least moe_dense_mlp_workspace_size() bytes (holds h [T][I], the
 *               status word and any fp32 partial sums of W2); ws_bytes its size
 * Errors: MOE_ERR_INVALID_ARG (null pointer, non-positive width, misalignment),
 * MOE_ERR_UNSUPPORTED (dtype or width the kernels do not take), MOE_ERR_WORKSPACE (ws too small),
 * MOE_ERR_CUDA.  T == 0 is a no-op. */
size_t moe_dense_mlp_workspace_size(int64_t T, int32_t d, int32_t I, moe_dtype_t act_dtype);
moe_status_t moe_dense_mlp(int64_t T, int32_t d, int32_t I, moe_dtype_t act_dtype, const void* x,
                           const void* W13, const void* W2, void* out, void* ws, size_t ws_bytes,
                           void* stream);

/* Reset the device status word (first 256 bytes of ws) to "no error", enqueued on stream. */
moe_status_t moe_reset_device_status(void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream`, read the device status word and translate it: MOE_OK,
 * MOE_ERR_DEVICE_CHECK (an index or row out of range was skipped) or MOE_ERR_TIMEOUT (a kernel's
 * bounded wait expired; its outputs are incomplete).  MOE_ERR_CUDA if the stream reports an
 * error. */
moe_status_t moe_device_status(const void* ws, size_t ws_bytes, void* stream);

/* A static, human-readable name of a status code. */
const char* moe_status_string(moe_status_t status);

/* Name and message of the CUDA error behind the calling thread's last MOE_ERR_CUDA ("" if none);
 * valid until the thread's next call into the library. */
const char* moe_last_error_string(void);

/* Number of this library's kernels enqueued by the calling thread since the last reset (a launch
 * counter for benchmarks), and its reset. */
uint64_t moe_launch_count(void);
void moe_reset_launch_count(void);

/* Launch profiler (the trace of the layer's kernels; off by default).  While enabled, every kernel
 * this library enqueues is bracketed by a CUDA event pair recorded on its own stream (events are
 * created once and reused; no device memory is allocated).  moe_profile_read() synchronises on
 * the recorded events, sums the elapsed time and the launch count per kernel name, writes at most
 * max_entries entries (names as NUL-terminated strings in slots of name_len bytes) and clears the
 * totals; it returns the number of entries written. */
moe_status_t moe_profile_enable(int on);
int moe_profile_read(int max_entries, char* names, size_t name_len, double* total_ms,
                     uint64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
