/*
 * moe_oracle.h -- plain, slow, fp64 CPU oracle of the mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the timed CPU baseline of the
 * benchmark may load this library.  The product path (the CUDA library) never calls it, links it
 * or shares a header, helper or table with it.
 *
 * What it computes (sources, cited by page title and section):
 *   - "Kimi K2 · Transformer blocks > MoE transformer block", the "Mixture of experts" steps:
 *       z = x W_r ;  s = sigma(z) ;  E_sel_i = [i in top_8(s + b)] ;
 *       G_i = 2.827 s_i E_sel_i / sum_j s_j E_sel_j ;
 *       g = x W1 ; u = x W3 ; a = g sigma(g) ; h = a (.) u ; E_i = h W2 ;
 *       y_routed = sum_i G_i E_i ; y_shared = (same SwiGLU, shared weights) ; D_ffn = y_routed + y_shared.
 *   - nnterp encyclopedia "kimi_k2", note "The mixture of experts": the bias is used only for the
 *     selection, the gates are the unbiased sigmoids renormalised and scaled by 2.827 and sum to 2.827.
 *   - "Kimi K3 · Latent up-projection", its equation y_routed = u_hat W_up and the `forward` /
 *     `moe_infer` code excerpts: router on the full-width input, down-projection to the latent,
 *     experts in the latent, gate-weighted sum, optional RMSNorm, up-projection, shared expert on the
 *     full-width input.
 *
 * Weight layout is the pages' [out, in] ("The reference module holds the weight output by input").
 * Every routed expert's W13 is [2I][d_e]: rows 0..I-1 are W1 (gate_proj), rows I..2I-1 are W3 (up_proj).
 * W2 is [d_e][I].  d_e = d on the K2 path, d_latent on the K3 path.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_F64 = 3, ORC_INT4 = 4 };

typedef struct {
  int64_t T;            /* tokens                                                     */
  int32_t d;            /* hidden size                                                */
  int32_t E;            /* routed experts                                             */
  int32_t k;            /* experts per token                                          */
  int32_t I;            /* routed expert intermediate size                            */
  int32_t I_shared;     /* shared expert intermediate size                            */
  int32_t n_shared;     /* 0 or 1 shared expert                                       */
  int32_t d_latent;     /* 0: K2 path; >0: K3 latent width                            */
  int32_t latent_norm;  /* 1: RMSNorm (unit weight) on the latent gate-weighted sum   */
  int32_t fp8;          /* 1: e4m3 expert weights with block scales, activations
                           quantised to e4m3 per token per quant_block channels       */
  int32_t quant_block;  /* 128                                                        */
  int32_t pad_;
  double gate_scale;    /* 2.827                                                      */
  double rms_eps;       /* 1e-6                                                       */
} orc_config;

/* A row-major matrix in one of the ORC_* types.  For ORC_E4M3, `scale` holds one fp32 scale per
 * quant_block x quant_block block, row-major over [ceil(rows/qb)][ceil(cols/qb)].  For ORC_INT4
 * ("4-bit integer groups"), `data` holds [rows][cols/2] packed bytes: code i of each 32-bit
 * little-endian word w (input channel 8w + i) is nibble (i / 2) + 4 (i % 2), and a nibble u
 * stands for u - 8; `scale` holds one scale per 32 input channels of each row, transposed,
 * [cols/32][rows] (bf16 values widened to fp32); `rows` is the row count; the element is the
 * product (u - 8) * scale rounded once to bf16 (the GEMM operand). */
typedef struct {
  const void* data;
  int32_t dtype;
  int32_t rows;         /* ORC_INT4 only: rows of the matrix (the scale layout's pitch) */
  const float* scale;
} orc_tensor;

/* Status codes. */
enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_EMISSING = 2 };

/* Full layer forward in fp64, with the oracle's own routing (fp64 logits and keys).
 *  x       [T][d]          ORC_F32 / ORC_BF16 / ORC_F64
 *  W_r     [E][d]          fp32 router weight ; b [E] fp32 selection bias
 *  W13     E entries, each [2I][d_e] ; W2 E entries, each [d_e][I]; an entry whose data is NULL
 *          marks an expert that is not supplied (an error if a token selects it)
 *  Ws13    [2 I_shared][d] ; Ws2 [d][I_shared]      (ignored when n_shared == 0)
 *  W_down  [d_latent][d]   ; W_up [d][d_latent]     (K3 only)
 *  outputs: out [T][d]; optional (may be NULL): idx [T][k] (slot order: key descending, ties to the
 *  lower index), gates [T][k], margin [T] (k-th minus (k+1)-th largest key), logits [T][E],
 *  routed [T][d] (y_routed alone), shared [T][d] (y_shared alone).
 *  nthreads >= 1 worker threads split the tokens. */
int orc_forward(const orc_config* cfg, int nthreads, orc_tensor x, const float* W_r, const float* b,
                const orc_tensor* W13, const orc_tensor* W2, orc_tensor Ws13, orc_tensor Ws2,
                orc_tensor W_down, orc_tensor W_up, double* out, int32_t* idx, double* gates,
                double* margin, double* logits, double* routed, double* shared);

/* The routing alone, in fp64 (the forward's first steps): no expert weight is read. */
int orc_route(const orc_config* cfg, orc_tensor x, const float* W_r, const float* b, int32_t* idx,
              double* gates, double* margin, double* logits);

/* Routing from given fp32 logits z [T][E] (the selection rule fed another implementation's logits).
 * Key = fp32( fp32(sigma(z)) + b ), sigma evaluated in fp64 and rounded to fp32.  Gates in fp64 from
 * the unbiased sigma(z).  idx [T][k], gates [T][k], margin [T] (in the fp32 key); sel_keys [T][k]
 * (may be NULL) receives the keys of the selected experts in slot order. */
int orc_route_from_logits(const orc_config* cfg, const float* z, const float* b, int32_t* idx,
                          double* gates, double* margin, float* sel_keys);

/* Number of learned parameters of one MoE layer, from the shapes the forward indexes. */
int64_t orc_param_count(const orc_config* cfg);
/* The same count by component: [0] router W_r, [1] selection bias b, [2] routed experts,
 * [3] shared expert, [4] latent down-projection, [5] latent up-projection. */
void orc_param_breakdown(const orc_config* cfg, int64_t out[6]);

/* e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, one NaN pattern per
 * sign) decoded from its definition. */
double orc_e4m3_decode(uint8_t code);
/* fp32 -> e4m3, round to nearest with ties to even, saturating to +-448; NaN -> 0x7F. */
uint8_t orc_e4m3_encode(float v);
/* Quantise n values (fp32) as groups of qb channels: scale = fp32(amax / 448) (1 for an all-zero
 * group), code = e4m3(fp32(v / scale)).  q [n] codes, scales [ceil(n/qb)]. */
void orc_quantize_group_e4m3(const float* v, int64_t n, int qb, uint8_t* q, float* scales);

/* One dense SwiGLU MLP on one row (the expert / shared-expert equations), fp64 in and out:
 *  x [din], W13 [2 I][din] (W1 rows then W3 rows), W2 [dout][I], y [dout]. */
int orc_swiglu_row(const double* x, int din, int I, int dout, orc_tensor W13, orc_tensor W2,
                   int qb, int quant_act, double* y);

/* The dense SwiGLU MLP of the first block(s) (nnterp "kimi_k2", "Printout": layer 0's mlp is a
 * DeepseekV3MLP with gate_proj / up_proj d -> I and down_proj I -> d): per token the expert
 * equations with no routing, y = (SiLU(x W1) (.) (x W3)) W2, in fp64.
 *  x [T][d] (ORC_F32 / ORC_BF16 / ORC_F64), W13 [2I][d] (W1 rows then W3 rows), W2 [d][I],
 *  out [T][d] fp64.  nthreads >= 1 worker threads split the tokens. */
int orc_dense_mlp(int64_t T, int d, int I, int nthreads, orc_tensor x, orc_tensor W13,
                  orc_tensor W2, double* out);

/* Row r of a matrix [rows][cols] of any ORC_* type widened to fp64, the values the oracle's GEMMs
 * use (e4m3: code value x block scale; int4: RN_bf16((u - 8) x group scale)). */
int orc_dequant_row(orc_tensor t, int64_t cols, int qb, int64_t r, double* out);

/* RMSNorm with unit weight: y = v / sqrt(mean(v^2) + eps). */
void orc_rmsnorm_unit(const double* v, int n, double eps, double* y);

#ifdef __cplusplus
}
#endif
#endif
