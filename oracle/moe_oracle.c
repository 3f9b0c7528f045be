/*
 * moe_oracle.c -- plain fp64 CPU oracle of the mixture-of-experts FFN layer (Kimi K2 /
 * DeepSeek-V3 shape, and the Kimi K3 latent variant).
 *
 * TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the benchmark's timed CPU baseline
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * Every step is the plain definition from the pages, evaluated per token in fp64 with no blocking,
 * fusion or reordering: there is no permutation, no grouping and no tiling here.  The function
 * comments name the passage each step follows.
 *
 * Where the pages are silent the readings are:
 *   - slot order of the selected experts: key descending, ties to the lower expert index;
 *   - the renormalisation has no epsilon (every sigmoid is > 0);
 *   - the K3 gate is the same sigmoid / bias / top-k / renormalise / x2.827 router, on the full-width
 *     input; the K3 RMSNorm has unit weight;
 *   - fp8: weights are e4m3 codes times one fp32 scale per 128x128 block; activations entering both
 *     expert GEMMs are quantised per token per 128 channels with scale = amax/448 (1 for an all-zero
 *     group); the quantisation decisions are taken in fp32 (the precision of the GPU kernel), the
 *     rest of the arithmetic in fp64.
 */
#include "moe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* Number formats                                                                              */
/* ------------------------------------------------------------------------------------------ */

static double bf16_bits_to_double(uint16_t v) {
  uint32_t u = (uint32_t)v << 16; /* bf16 is the top half of an IEEE binary32 */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* e4m3 ("E4M3FN"): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.  Exponent field 0
 * holds the subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity; the largest finite
 * magnitude is S.1111.110 = 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t code) {
  const int sign = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Nearest e4m3 value by a search over the 127 non-negative finite codes (their values increase with
 * the code), ties to the even code (the even mantissa), saturating at 448. */
uint8_t orc_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 126; /* largest code c with decode(c) <= a; decode(0) = 0 <= a */
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (orc_e4m3_decode((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int c = lo;
  if (c == 126) return (uint8_t)(sign | 126);
  const double below = a - orc_e4m3_decode((uint8_t)c);
  const double above = orc_e4m3_decode((uint8_t)(c + 1)) - a;
  int r;
  if (below < above)
    r = c;
  else if (above < below)
    r = c + 1;
  else
    r = (c % 2 == 0) ? c : c + 1;
  return (uint8_t)(sign | r);
}

void orc_quantize_group_e4m3(const float* v, int64_t n, int qb, uint8_t* q, float* scales) {
  for (int64_t g0 = 0; g0 < n; g0 += qb) {
    const int64_t g1 = (g0 + qb < n) ? g0 + qb : n;
    float amax = 0.0f;
    for (int64_t i = g0; i < g1; ++i) {
      const float m = fabsf(v[i]);
      if (m > amax) amax = m;
    }
    const float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    scales[g0 / qb] = scale;
    for (int64_t i = g0; i < g1; ++i) q[i] = orc_e4m3_encode(v[i] / scale);
  }
}

static double e4m3_table[256];
static pthread_once_t e4m3_table_once = PTHREAD_ONCE_INIT;
static void e4m3_table_init(void) {
  for (int c = 0; c < 256; ++c) e4m3_table[c] = orc_e4m3_decode((uint8_t)c);
}

/* Round to the nearest bf16 value (8 significant bits, ties to even) in fp64: v = m 2^e with
 * 0.5 <= |m| < 1, and m keeps 8 bits.  Normal-range values (every use here is O(1) or a small
 * integer times a weight scale). */
static double round_bf16(double v) {
  int e;
  const double m = frexp(v, &e);
  return ldexp(nearbyint(m * 256.0), e - 8); /* the default rounding mode is to nearest even */
}

/* int4 element (r, c): the nibble of input channel c in row r's packed words, value u - 8, times
 * the row's scale for its group of 32 channels, rounded once to bf16. */
static double int4_elem(const orc_tensor* t, int64_t cols, int64_t r, int64_t c) {
  const int64_t w = c / 8;
  const int i = (int)(c % 8);
  const int nib = i / 2 + 4 * (i % 2);
  const uint8_t byte = ((const uint8_t*)t->data)[r * (cols / 2) + w * 4 + nib / 2];
  const int u = (byte >> (4 * (nib % 2))) & 0xF;
  const double s = (double)t->scale[(c / 32) * (int64_t)t->rows + r];
  return round_bf16((double)(u - 8) * s);
}

/* Element (r, c) of a row-major [rows][cols] tensor, widened to fp64.  For e4m3 the value is the
 * code's value times the fp32 scale of its qb x qb block. */
static double elem(const orc_tensor* t, int64_t cols, int qb, int64_t r, int64_t c) {
  switch (t->dtype) {
    case ORC_F32: return (double)((const float*)t->data)[r * cols + c];
    case ORC_F64: return ((const double*)t->data)[r * cols + c];
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t*)t->data)[r * cols + c]);
    case ORC_E4M3: {
      const int64_t nbc = (cols + qb - 1) / qb;
      const double s = (double)t->scale[(r / qb) * nbc + c / qb];
      return e4m3_table[((const uint8_t*)t->data)[r * cols + c]] * s;
    }
    case ORC_INT4: return int4_elem(t, cols, r, c);
    default: return NAN;
  }
}

/* sum_c W[r][c] * v[c] over one row of W (a Linear's output r, weight stored [out][in]). */
static double row_dot(const orc_tensor* W, int64_t cols, int qb, int64_t r, const double* v) {
  double acc = 0.0;
  switch (W->dtype) {
    case ORC_F32: {
      const float* w = (const float*)W->data + r * cols;
      for (int64_t c = 0; c < cols; ++c) acc += (double)w[c] * v[c];
      return acc;
    }
    case ORC_F64: {
      const double* w = (const double*)W->data + r * cols;
      for (int64_t c = 0; c < cols; ++c) acc += w[c] * v[c];
      return acc;
    }
    case ORC_BF16: {
      const uint16_t* w = (const uint16_t*)W->data + r * cols;
      for (int64_t c = 0; c < cols; ++c) acc += bf16_bits_to_double(w[c]) * v[c];
      return acc;
    }
    case ORC_INT4: { /* int4_elem per channel, with the 16 values of each group's scale tabled */
      for (int64_t c0 = 0; c0 < cols; c0 += 32) {
        double val[16];
        const double s = (double)W->scale[(c0 / 32) * (int64_t)W->rows + r];
        for (int u = 0; u < 16; ++u) val[u] = round_bf16((double)(u - 8) * s);
        const uint8_t* bytes = (const uint8_t*)W->data + r * (cols / 2) + c0 / 2;
        for (int i = 0; i < 32 && c0 + i < cols; ++i) {
          const int nib = (i % 8) / 2 + 4 * (i % 2);
          const int u = (bytes[(i / 8) * 4 + nib / 2] >> (4 * (nib % 2))) & 0xF;
          acc += val[u] * v[c0 + i];
        }
      }
      return acc;
    }
    default:
      for (int64_t c = 0; c < cols; ++c) acc += elem(W, cols, qb, r, c) * v[c];
      return acc;
  }
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------------------------ */
/* Shapes (the only place the layer's tensor shapes are stated; the parameter count reuses them) */
/* ------------------------------------------------------------------------------------------ */

static int64_t expert_width(const orc_config* c) { return c->d_latent > 0 ? c->d_latent : c->d; }
static int64_t w13_rows(int64_t I) { return 2 * I; } /* W1 rows then W3 rows */
static int64_t swiglu_params(int64_t din, int64_t I, int64_t dout) {
  return w13_rows(I) * din + dout * I;
}

void orc_param_breakdown(const orc_config* c, int64_t out[6]) {
  const int64_t de = expert_width(c);
  out[0] = (int64_t)c->E * c->d; /* router W_r [E][d] */
  out[1] = c->E;                 /* selection bias b [E] */
  out[2] = (int64_t)c->E * swiglu_params(de, c->I, de);
  out[3] = (int64_t)c->n_shared * swiglu_params(c->d, c->I_shared, c->d);
  out[4] = c->d_latent > 0 ? (int64_t)c->d_latent * c->d : 0; /* down [L][d] */
  out[5] = c->d_latent > 0 ? (int64_t)c->d * c->d_latent : 0; /* up [d][L]   */
}

int64_t orc_param_count(const orc_config* c) {
  int64_t p[6];
  orc_param_breakdown(c, p);
  return p[0] + p[1] + p[2] + p[3] + p[4] + p[5];
}

/* ------------------------------------------------------------------------------------------ */
/* Routing: "Mixture of experts" steps z, s, E_sel, G                                          */
/* ------------------------------------------------------------------------------------------ */

/* top_k by rank: expert i's rank is the number of experts ordered before it (larger key, or equal
 * key and lower index).  The k experts of rank 0..k-1 are selected, in rank order.  margin is the
 * key of rank k-1 minus the key of rank k (infinite when k == E). */
static void topk_by_rank_f64(const double* key, int E, int k, int32_t* idx, double* margin) {
  double kth = 0.0, next = 0.0;
  for (int i = 0; i < E; ++i) {
    int rank = 0;
    for (int j = 0; j < E; ++j)
      if (key[j] > key[i] || (key[j] == key[i] && j < i)) ++rank;
    if (rank < k) idx[rank] = i;
    if (rank == k - 1) kth = key[i];
    if (rank == k) next = key[i];
  }
  if (margin) *margin = (k < E) ? kth - next : INFINITY;
}

static void topk_by_rank_f32(const float* key, int E, int k, int32_t* idx, double* margin) {
  float kth = 0.0f, next = 0.0f;
  for (int i = 0; i < E; ++i) {
    int rank = 0;
    for (int j = 0; j < E; ++j)
      if (key[j] > key[i] || (key[j] == key[i] && j < i)) ++rank;
    if (rank < k) idx[rank] = i;
    if (rank == k - 1) kth = key[i];
    if (rank == k) next = key[i];
  }
  if (margin) *margin = (k < E) ? (double)kth - (double)next : INFINITY;
}

/* G_j = gate_scale * s_{idx_j} / sum_{j'} s_{idx_j'}  (unbiased sigmoids; no epsilon). */
static void gates_from_scores(const double* s, const int32_t* idx, int k, double gate_scale,
                              double* g) {
  double den = 0.0;
  for (int j = 0; j < k; ++j) den += s[idx[j]];
  for (int j = 0; j < k; ++j) g[j] = gate_scale * s[idx[j]] / den;
}

int orc_route_from_logits(const orc_config* c, const float* z, const float* b, int32_t* idx,
                          double* gates, double* margin, float* sel_keys) {
  if (!c || !z || !b || !idx || c->k < 1 || c->k > c->E) return ORC_EINVAL;
  double* s = (double*)malloc(sizeof(double) * c->E);
  float* key = (float*)malloc(sizeof(float) * c->E);
  double g[1024];
  if (!s || !key || c->k > 1024) {
    free(s);
    free(key);
    return ORC_EINVAL;
  }
  for (int64_t t = 0; t < c->T; ++t) {
    const float* zt = z + t * c->E;
    for (int e = 0; e < c->E; ++e) {
      s[e] = sigmoid((double)zt[e]);
      const float s32 = (float)s[e];
      key[e] = s32 + b[e]; /* fp32 add, rounded to fp32 */
    }
    topk_by_rank_f32(key, c->E, c->k, idx + t * c->k, margin ? margin + t : NULL);
    gates_from_scores(s, idx + t * c->k, c->k, c->gate_scale, g);
    if (gates)
      for (int j = 0; j < c->k; ++j) gates[t * c->k + j] = g[j];
    if (sel_keys)
      for (int j = 0; j < c->k; ++j) sel_keys[t * c->k + j] = key[idx[t * c->k + j]];
  }
  free(s);
  free(key);
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Experts: g = x W1 ; u = x W3 ; a = g sigma(g) ; h = a (.) u ; E = h W2                       */
/* ------------------------------------------------------------------------------------------ */

/* fp8: quantise a vector per qb-channel group (decisions in fp32), return the dequantised fp64
 * values code_value * scale. */
static void fake_quant_e4m3(const double* v, int64_t n, int qb, double* out, float* tmp_f,
                            uint8_t* tmp_q, float* tmp_s) {
  for (int64_t i = 0; i < n; ++i) tmp_f[i] = (float)v[i];
  orc_quantize_group_e4m3(tmp_f, n, qb, tmp_q, tmp_s);
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_table[tmp_q[i]] * (double)tmp_s[i / qb];
}

int orc_swiglu_row(const double* x, int din, int I, int dout, orc_tensor W13, orc_tensor W2,
                   int qb, int quant_act, double* y) {
  if (!x || !y || !W13.data || !W2.data || din < 1 || I < 1 || dout < 1) return ORC_EINVAL;
  pthread_once(&e4m3_table_once, e4m3_table_init);
  const int64_t nmax = din > I ? din : I;
  double* xin = (double*)malloc(sizeof(double) * din);
  double* h = (double*)malloc(sizeof(double) * I);
  float* tf = (float*)malloc(sizeof(float) * nmax);
  uint8_t* tq = (uint8_t*)malloc(nmax);
  float* ts = (float*)malloc(sizeof(float) * (nmax / (qb > 0 ? qb : 1) + 1));
  if (!xin || !h || !tf || !tq || !ts) {
    free(xin); free(h); free(tf); free(tq); free(ts);
    return ORC_EINVAL;
  }
  if (quant_act)
    fake_quant_e4m3(x, din, qb, xin, tf, tq, ts);
  else
    memcpy(xin, x, sizeof(double) * din);
  for (int j = 0; j < I; ++j) {
    const double g = row_dot(&W13, din, qb, j, xin);     /* W1 = gate_proj */
    const double u = row_dot(&W13, din, qb, I + j, xin); /* W3 = up_proj   */
    const double a = g * sigmoid(g);                     /* SiLU           */
    h[j] = a * u;
  }
  if (quant_act) fake_quant_e4m3(h, I, qb, h, tf, tq, ts);
  for (int o = 0; o < dout; ++o) y[o] = row_dot(&W2, I, qb, o, h); /* W2 = down_proj */
  free(xin); free(h); free(tf); free(tq); free(ts);
  return ORC_OK;
}

void orc_rmsnorm_unit(const double* v, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += v[i] * v[i];
  const double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = v[i] * inv;
}

/* One token's routing, the "Mixture of experts" steps z = x W_r, s = sigma(z), selection by
 * top_k(s + b) (the bias only selects), and the gates G = 2.827 s_i / sum_selected s_j, in fp64. */
static void route_token(const orc_config* c, const double* xr, const float* W_r, const float* b,
                        double* z, double* s, double* key, int32_t* id, double* g, double* mg) {
  const int64_t d = c->d, E = c->E;
  for (int64_t e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int64_t ch = 0; ch < d; ++ch) acc += (double)W_r[e * d + ch] * xr[ch];
    z[e] = acc;
    s[e] = sigmoid(acc);
    key[e] = s[e] + (double)b[e];
  }
  topk_by_rank_f64(key, (int)E, c->k, id, mg);
  gates_from_scores(s, id, c->k, c->gate_scale, g);
}

int orc_route(const orc_config* c, orc_tensor x, const float* W_r, const float* b, int32_t* idx,
              double* gates, double* margin, double* logits) {
  if (!c || !x.data || !W_r || !b || c->k < 1 || c->k > c->E) return ORC_EINVAL;
  const int64_t d = c->d, E = c->E, k = c->k;
  const int qb = c->quant_block > 0 ? c->quant_block : 128;
  double* xr = (double*)malloc(sizeof(double) * d);
  double* z = (double*)malloc(sizeof(double) * E);
  double* s = (double*)malloc(sizeof(double) * E);
  double* key = (double*)malloc(sizeof(double) * E);
  int32_t* id = (int32_t*)malloc(sizeof(int32_t) * k);
  double* g = (double*)malloc(sizeof(double) * k);
  int status = (xr && z && s && key && id && g) ? ORC_OK : ORC_EINVAL;
  for (int64_t t = 0; status == ORC_OK && t < c->T; ++t) {
    for (int64_t ch = 0; ch < d; ++ch) xr[ch] = elem(&x, d, qb, t, ch);
    double mg;
    route_token(c, xr, W_r, b, z, s, key, id, g, &mg);
    for (int64_t j = 0; j < k; ++j) {
      if (idx) idx[t * k + j] = id[j];
      if (gates) gates[t * k + j] = g[j];
    }
    if (margin) margin[t] = mg;
    if (logits)
      for (int64_t e = 0; e < E; ++e) logits[t * E + e] = z[e];
  }
  free(xr); free(z); free(s); free(key); free(id); free(g);
  return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Layer forward                                                                               */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
  const orc_config* c;
  int tid, nthreads;
  orc_tensor x;
  const float* W_r;
  const float* b;
  const orc_tensor* W13;
  const orc_tensor* W2;
  orc_tensor Ws13, Ws2, W_down, W_up;
  double *out, *gates, *margin, *logits, *routed, *shared;
  int32_t* idx;
  int status;
} fwd_job;

static void* forward_worker(void* arg) {
  fwd_job* J = (fwd_job*)arg;
  const orc_config* c = J->c;
  const int64_t d = c->d, E = c->E, k = c->k, de = expert_width(c);
  const int qb = c->quant_block > 0 ? c->quant_block : 128;
  double* xr = (double*)malloc(sizeof(double) * d);
  double* xe = (double*)malloc(sizeof(double) * de);
  double* z = (double*)malloc(sizeof(double) * E);
  double* s = (double*)malloc(sizeof(double) * E);
  double* key = (double*)malloc(sizeof(double) * E);
  double* ex = (double*)malloc(sizeof(double) * de);
  double* yr = (double*)malloc(sizeof(double) * de);
  double* yn = (double*)malloc(sizeof(double) * de);
  double* ro = (double*)malloc(sizeof(double) * d);
  double* sh = (double*)malloc(sizeof(double) * d);
  int32_t* id = (int32_t*)malloc(sizeof(int32_t) * k);
  double* g = (double*)malloc(sizeof(double) * k);
  J->status = ORC_OK;
  if (!xr || !xe || !z || !s || !key || !ex || !yr || !yn || !ro || !sh || !id || !g) {
    J->status = ORC_EINVAL;
    goto done;
  }
  for (int64_t t = J->tid; t < c->T; t += J->nthreads) {
    for (int64_t ch = 0; ch < d; ++ch) xr[ch] = elem(&J->x, d, qb, t, ch);

    double mg;
    route_token(c, xr, J->W_r, J->b, z, s, key, id, g, &mg);

    /* K3: the routed path runs in the latent, x_lat = x W_down (the router saw the full width). */
    if (c->d_latent > 0) {
      for (int64_t l = 0; l < de; ++l) xe[l] = row_dot(&J->W_down, d, qb, l, xr);
    } else {
      memcpy(xe, xr, sizeof(double) * d);
    }

    /* y_routed = sum_j G_j E_{idx_j}(x) over the selected experts (G is 0 for the others). */
    for (int64_t o = 0; o < de; ++o) yr[o] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      const int e = id[j];
      if (!J->W13[e].data || !J->W2[e].data) {
        J->status = ORC_EMISSING;
        goto done;
      }
      int st = orc_swiglu_row(xe, (int)de, c->I, (int)de, J->W13[e], J->W2[e], qb, c->fp8, ex);
      if (st) {
        J->status = st;
        goto done;
      }
      for (int64_t o = 0; o < de; ++o) yr[o] += g[j] * ex[o];
    }

    /* K3: optional RMSNorm on the latent sum, then y_routed = u_hat W_up. */
    if (c->d_latent > 0) {
      if (c->latent_norm)
        orc_rmsnorm_unit(yr, (int)de, c->rms_eps, yn);
      else
        memcpy(yn, yr, sizeof(double) * de);
      for (int64_t o = 0; o < d; ++o) ro[o] = row_dot(&J->W_up, de, qb, o, yn);
    } else {
      memcpy(ro, yr, sizeof(double) * d);
    }

    /* y_shared: the same SwiGLU with the shared weights, on the full-width input. */
    for (int64_t o = 0; o < d; ++o) sh[o] = 0.0;
    if (c->n_shared > 0) {
      int st = orc_swiglu_row(xr, (int)d, c->I_shared, (int)d, J->Ws13, J->Ws2, qb, c->fp8, sh);
      if (st) {
        J->status = st;
        goto done;
      }
    }

    /* D_ffn = y_routed + y_shared */
    for (int64_t o = 0; o < d; ++o) J->out[t * d + o] = ro[o] + sh[o];
    if (J->routed)
      for (int64_t o = 0; o < d; ++o) J->routed[t * d + o] = ro[o];
    if (J->shared)
      for (int64_t o = 0; o < d; ++o) J->shared[t * d + o] = sh[o];
    if (J->idx)
      for (int64_t j = 0; j < k; ++j) J->idx[t * k + j] = id[j];
    if (J->gates)
      for (int64_t j = 0; j < k; ++j) J->gates[t * k + j] = g[j];
    if (J->margin) J->margin[t] = mg;
    if (J->logits)
      for (int64_t e = 0; e < E; ++e) J->logits[t * E + e] = z[e];
  }
done:
  free(xr); free(xe); free(z); free(s); free(key); free(ex); free(yr); free(yn);
  free(ro); free(sh); free(id); free(g);
  return NULL;
}

int orc_forward(const orc_config* c, int nthreads, orc_tensor x, const float* W_r, const float* b,
                const orc_tensor* W13, const orc_tensor* W2, orc_tensor Ws13, orc_tensor Ws2,
                orc_tensor W_down, orc_tensor W_up, double* out, int32_t* idx, double* gates,
                double* margin, double* logits, double* routed, double* shared) {
  if (!c || !x.data || !W_r || !b || !W13 || !W2 || !out) return ORC_EINVAL;
  if (c->T < 0 || c->d < 1 || c->E < 1 || c->k < 1 || c->k > c->E || c->I < 1) return ORC_EINVAL;
  if (c->n_shared && (!Ws13.data || !Ws2.data || c->I_shared < 1)) return ORC_EINVAL;
  if (c->d_latent > 0 && (!W_down.data || !W_up.data)) return ORC_EINVAL;
  if (c->fp8 && c->d_latent > 0) return ORC_EINVAL; /* no fp8 latent variant is defined */
  pthread_once(&e4m3_table_once, e4m3_table_init);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  fwd_job* jobs = (fwd_job*)calloc((size_t)nthreads, sizeof(fwd_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return ORC_EINVAL;
  }
  for (int i = 0; i < nthreads; ++i) {
    fwd_job j = {c, i, nthreads, x, W_r, b, W13, W2, Ws13, Ws2, W_down, W_up,
                 out, gates, margin, logits, routed, shared, idx, ORC_OK};
    jobs[i] = j;
  }
  char* started = (char*)calloc((size_t)nthreads, 1);
  for (int i = 1; i < nthreads; ++i)
    started[i] = started && pthread_create(&th[i], NULL, forward_worker, &jobs[i]) == 0;
  forward_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int i = 1; i < nthreads; ++i) {
    if (started && started[i])
      pthread_join(th[i], NULL);
    else
      forward_worker(&jobs[i]);
    if (!status) status = jobs[i].status;
  }
  free(started);
  free(jobs);
  free(th);
  return status;
}

/* ------------------------------------------------------------------------------------------ */
/* Dense block MLP (nnterp "kimi_k2", "Printout": layer 0's mlp is a DeepseekV3MLP; the Kimi K2  */
/* "Transformer blocks" modeling_deepseek excerpt builds it for blocks below                     */
/* first_k_dense_replace): y = (SiLU(x W1) (.) (x W3)) W2 per token, the expert equations with   */
/* no routing.                                                                                   */
/* ------------------------------------------------------------------------------------------ */
typedef struct {
  int64_t T;
  int d, I, tid, nthreads;
  orc_tensor x, W13, W2;
  double* out;
  int status;
} dense_job;

static void* dense_worker(void* arg) {
  dense_job* J = (dense_job*)arg;
  double* xr = (double*)malloc(sizeof(double) * J->d);
  if (!xr) {
    J->status = ORC_EINVAL;
    return NULL;
  }
  for (int64_t t = J->tid; t < J->T; t += J->nthreads) {
    for (int ch = 0; ch < J->d; ++ch) xr[ch] = elem(&J->x, J->d, 1, t, ch);
    const int st = orc_swiglu_row(xr, J->d, J->I, J->d, J->W13, J->W2, 128, 0,
                                  J->out + t * (int64_t)J->d);
    if (st != ORC_OK) {
      J->status = st;
      break;
    }
  }
  free(xr);
  return NULL;
}

int orc_dense_mlp(int64_t T, int d, int I, int nthreads, orc_tensor x, orc_tensor W13,
                  orc_tensor W2, double* out) {
  if (T < 0 || d < 1 || I < 1 || !x.data || !W13.data || !W2.data || !out) return ORC_EINVAL;
  if (x.dtype == ORC_E4M3 || W13.dtype == ORC_E4M3 || W2.dtype == ORC_E4M3) return ORC_EINVAL;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  dense_job* jobs = (dense_job*)calloc((size_t)nthreads, sizeof(dense_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* started = (char*)calloc((size_t)nthreads, 1);
  if (!jobs || !th || !started) {
    free(jobs); free(th); free(started);
    return ORC_EINVAL;
  }
  for (int i = 0; i < nthreads; ++i) {
    dense_job j = {T, d, I, i, nthreads, x, W13, W2, out, ORC_OK};
    jobs[i] = j;
  }
  for (int i = 1; i < nthreads; ++i)
    started[i] = pthread_create(&th[i], NULL, dense_worker, &jobs[i]) == 0;
  dense_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int i = 1; i < nthreads; ++i) {
    if (started[i])
      pthread_join(th[i], NULL);
    else
      dense_worker(&jobs[i]);
    if (!status) status = jobs[i].status;
  }
  free(started); free(jobs); free(th);
  return status;
}

/* Row r of a matrix [rows][cols] in any ORC_* type, widened to fp64 (the values every GEMM of the
 * oracle multiplies with). */
int orc_dequant_row(orc_tensor t, int64_t cols, int qb, int64_t r, double* out) {
  if (!t.data || !out || cols < 1 || r < 0) return ORC_EINVAL;
  if ((t.dtype == ORC_E4M3 || t.dtype == ORC_INT4) && !t.scale) return ORC_EINVAL;
  if (t.dtype == ORC_INT4 && (cols % 32 || r >= t.rows)) return ORC_EINVAL;
  pthread_once(&e4m3_table_once, e4m3_table_init);
  for (int64_t c = 0; c < cols; ++c) out[c] = elem(&t, cols, qb, r, c);
  return ORC_OK;
}
