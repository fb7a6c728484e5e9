/*
 * pace_oracle.c -- plain, slow, obviously correct CPU statement of the PACE decode path.
 *
 * TEST INFRASTRUCTURE. Only tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares nothing with the CUDA library. Build: -O2 -ffp-contract=off (no FMA contraction, so
 * every fp32 operation of the quantizers rounds exactly once, as written).
 *
 * Page shorthand (title, then the section cited):
 *   [P1] "PACE는 4비트 순환 상태를 주기적으로 반올림해 추론 메모리를 줄인다" (onedev.kr)
 *   [P2] "[논문리뷰] PACE: Periodic and Channel-Aligned Encoding of Four-Bit Recurrent States"
 *   [P3] "PACE сжимает состояние линейных LLM до 4 бит и экономит треть памяти"
 *
 * Arithmetic: recurrences in fp64; quantizers in fp32 on the fp32-rounded state.
 * Readings taken where the pages are silent (listed again in the design notes):
 *   - rounding is to nearest, ties to even (rintf under the default rounding mode);
 *   - symmetric codes use +-(2^(b-1)-1); scales are stored as bf16; codes use the reciprocal of the
 *     stored scale; a scale that is zero or subnormal makes the whole group zero;
 *   - the zero-point range always contains 0 and the zero point is an integer code;
 *   - the decode buffer also holds beta_t (the rule needs it);
 *   - the current token enters its own output through its buffered (quantized) values;
 *   - the state is rounded right after the output of the dP-th buffered token;
 *   - prefill inputs are not buffered; a partial final chunk is rounded at its end too.
 */
#include "pace_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------------------------- */
/* bf16 rounding: keep the upper 16 bits of the fp32 pattern, rounding the dropped 16 bits to      */
/* nearest with ties going to the even upper half.                                                 */
float orc_bf16_rn(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) {           /* inf or nan */
    if (u & 0x007fffffu) u |= 0x00400000u;           /* nan stays a (quiet) nan */
    u &= 0xffff0000u;
  } else {
    uint32_t keep_odd = (u >> 16) & 1u;
    u += 0x7fffu + keep_odd;
    u &= 0xffff0000u;
  }
  float y;
  memcpy(&y, &u, sizeof y);
  return y;
}

void orc_bf16_rn_array(const float *x, float *y, long n) {
  for (long i = 0; i < n; ++i) y[i] = orc_bf16_rn(x[i]);
}

static int32_t clamp_i(int32_t v, int32_t lo, int32_t hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* ---------------------------------------------------------------------------------------------- */
/* Symmetric quantizer of one key-axis group ([P1] 무엇과 다른가: g contiguous elements along the key */
/* axis of one column share one scale; PACE-4 is symmetric).                                       */
void orc_quant_group_sym(const float *x, int n, int stride, int bits, float *s_out, int32_t *c, int cstride) {
  const int qmax = (1 << (bits - 1)) - 1;
  float A = 0.0f;
  for (int i = 0; i < n; ++i) {
    float ax = fabsf(x[(long)i * stride]);
    if (ax > A) A = ax;
  }
  float q = A / (float)qmax;
  float s = orc_bf16_rn(q);
  if (!(s >= FLT_MIN)) {                              /* zero (or subnormal) scale: all-zero group */
    *s_out = 0.0f;
    for (int i = 0; i < n; ++i) c[(long)i * cstride] = 0;
    return;
  }
  float r = 1.0f / s;
  for (int i = 0; i < n; ++i) {
    float t = x[(long)i * stride] * r;
    float rt = rintf(t);
    c[(long)i * cstride] = clamp_i((int32_t)rt, -qmax, qmax);
  }
  *s_out = s;
}

/* Integer zero-point quantizer of one group ([P1] 무엇과 다른가: PACE-4/8 uses an integer zero point). */
void orc_quant_group_zp(const float *x, int n, int stride, int bits, float *s_out, int32_t *z_out, int32_t *c,
                        int cstride) {
  const int qm = (1 << bits) - 1;
  float lo = 0.0f, hi = 0.0f;                         /* the range always contains zero */
  for (int i = 0; i < n; ++i) {
    float v = x[(long)i * stride];
    if (v < lo) lo = v;
    if (v > hi) hi = v;
  }
  float span = hi - lo;
  float s = orc_bf16_rn(span / (float)qm);
  if (!(s >= FLT_MIN)) {
    *s_out = 0.0f;
    *z_out = 0;
    for (int i = 0; i < n; ++i) c[(long)i * cstride] = 0;
    return;
  }
  float r = 1.0f / s;
  float nl = -lo;
  float zt = nl * r;
  int32_t z = clamp_i((int32_t)rintf(zt), 0, qm);
  for (int i = 0; i < n; ++i) {
    float t = x[(long)i * stride] * r;
    int32_t ci = (int32_t)rintf(t) + z;
    c[(long)i * cstride] = clamp_i(ci, 0, qm);
  }
  *s_out = s;
  *z_out = z;
}

void orc_quantize_state(const orc_cfg *cfg, const float *S32, int32_t *code, float *scale, int32_t *zp) {
  const int dk = cfg->d_k, dv = cfg->d_v, g = cfg->g, ng = dk / g;
  for (int j = 0; j < dv; ++j) {
    for (int gi = 0; gi < ng; ++gi) {
      const float *x = S32 + (long)gi * g * dv + j;   /* rows gi*g .. gi*g+g-1 of column j */
      int32_t *c = code + (long)gi * g * dv + j;
      if (cfg->zero_point)
        orc_quant_group_zp(x, g, dv, cfg->bits, &scale[gi * dv + j], &zp[gi * dv + j], c, dv);
      else
        orc_quant_group_sym(x, g, dv, cfg->bits, &scale[gi * dv + j], c, dv);
    }
  }
}

void orc_dequantize_state(const orc_cfg *cfg, const int32_t *code, const float *scale, const int32_t *zp,
                          double *S) {
  const int dk = cfg->d_k, dv = cfg->d_v, g = cfg->g;
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) {
      int gi = i / g;
      int32_t c = code[(long)i * dv + j];
      int32_t z = cfg->zero_point ? zp[gi * dv + j] : 0;
      S[(long)i * dv + j] = (double)scale[gi * dv + j] * (double)(c - z);
    }
}

/* Decode-buffer quantizer ([P1] 어떻게 동작하나: the buffer is int8 by default; keys 4-bit in the    */
/* mixed configuration). One symmetric fp32 scale per token vector.                                */
void orc_buffer_quant(const float *x, int n, int qmax, int32_t *c, float *s_out) {
  float A = 0.0f;
  for (int i = 0; i < n; ++i) {
    float ax = fabsf(x[i]);
    if (ax > A) A = ax;
  }
  if (!(A >= FLT_MIN)) {
    *s_out = 0.0f;
    for (int i = 0; i < n; ++i) c[i] = 0;
    return;
  }
  float fq = (float)qmax;
  float s = A / fq;
  float r = fq / A;
  for (int i = 0; i < n; ++i) {
    float t = x[i] * r;
    c[i] = clamp_i((int32_t)rintf(t), -qmax, qmax);
  }
  *s_out = s;
}

/* ---------------------------------------------------------------------------------------------- */
/* Gated delta rule ([P2] 1. Key Terms & Definitions, "Delta Value"):                             */
/*   S_t = a_t S_{t-1} + k_t u_t^T,  u_t = beta_t (v_t - (a_t S_{t-1})^T k_t).                     */
void orc_token_update(int dk, int dv, double *S, const double *k, const double *v, double a, double beta,
                      double *u_out) {
  double *u = (double *)malloc(sizeof(double) * dv);
  for (int j = 0; j < dv; ++j) {
    double w = 0.0;
    for (int i = 0; i < dk; ++i) w += a * S[(long)i * dv + j] * k[i];
    u[j] = beta * (v[j] - w);
  }
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) S[(long)i * dv + j] = a * S[(long)i * dv + j] + k[i] * u[j];
  if (u_out) memcpy(u_out, u, sizeof(double) * dv);
  free(u);
}

/* Readout o = S^T q. */
void orc_readout(int dk, int dv, const double *S, const double *q, double *o) {
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < dk; ++i) acc += S[(long)i * dv + j] * q[i];
    o[j] = acc;
  }
}

/* ---------------------------------------------------------------------------------------------- */
/* Resident state <-> fp64 working state.                                                          */
static void load_state(const orc_cfg *cfg, const orc_unit *u, double *S) {
  const long n = (long)cfg->d_k * cfg->d_v;
  if (cfg->state_mode == ORC_STATE_QUANT)
    orc_dequantize_state(cfg, u->code, u->scale, u->zp, S);
  else
    memcpy(S, u->S, sizeof(double) * n);
}

/* Round the working state once and store it: quantized mode rounds the fp32 image with the       */
/* key-axis quantizer; fp32 (test) mode keeps it exact; both bf16 modes store bf16(fp32(S)).      */
static void store_state(const orc_cfg *cfg, orc_unit *u, const double *S) {
  const long n = (long)cfg->d_k * cfg->d_v;
  if (cfg->state_mode == ORC_STATE_QUANT) {
    float *S32 = (float *)malloc(sizeof(float) * n);
    for (long e = 0; e < n; ++e) S32[e] = (float)S[e];
    orc_quantize_state(cfg, S32, u->code, u->scale, u->zp);
    free(S32);
  } else if (cfg->state_mode == ORC_STATE_BF16 || cfg->state_mode == ORC_STATE_BF16_BUF) {
    for (long e = 0; e < n; ++e) u->S[e] = (double)orc_bf16_rn((float)S[e]);
  } else {
    memcpy(u->S, S, sizeof(double) * n);
  }
}

/* Buffer slot -> dequantized (k, v) in fp64. */
static void buffer_token(const orc_cfg *cfg, const orc_unit *u, int slot, double *k, double *v) {
  const int dk = cfg->d_k, dv = cfg->d_v;
  if (cfg->buf_mode == ORC_BUF_FP32) {
    for (int i = 0; i < dk; ++i) k[i] = (double)u->bkf[(long)slot * dk + i];
    for (int j = 0; j < dv; ++j) v[j] = (double)u->bvf[(long)slot * dv + j];
    return;
  }
  for (int i = 0; i < dk; ++i) k[i] = (double)u->bsk[slot] * (double)u->bk[(long)slot * dk + i];
  if (cfg->buf_mode == ORC_BUF_MIXED) {
    for (int j = 0; j < dv; ++j) v[j] = (double)u->bvf[(long)slot * dv + j];
  } else {
    for (int j = 0; j < dv; ++j) v[j] = (double)u->bsv[slot] * (double)u->bv[(long)slot * dv + j];
  }
}

/* Buffer append ([P1] 어떻게 동작하나: the tokens since the last rounding wait in the decode buffer). */
static void buffer_append(const orc_cfg *cfg, orc_unit *u, int slot, const float *k, const float *v, float a,
                          float beta) {
  const int dk = cfg->d_k, dv = cfg->d_v;
  if (cfg->buf_mode == ORC_BUF_FP32) {
    memcpy(u->bkf + (long)slot * dk, k, sizeof(float) * dk);
    memcpy(u->bvf + (long)slot * dv, v, sizeof(float) * dv);
  } else if (cfg->buf_mode == ORC_BUF_MIXED) {
    orc_buffer_quant(k, dk, 7, u->bk + (long)slot * dk, &u->bsk[slot]);
    for (int j = 0; j < dv; ++j) u->bvf[(long)slot * dv + j] = orc_bf16_rn(v[j]);
  } else {
    orc_buffer_quant(k, dk, 127, u->bk + (long)slot * dk, &u->bsk[slot]);
    orc_buffer_quant(v, dv, 127, u->bv + (long)slot * dv, &u->bsv[slot]);
  }
  u->ba[slot] = a;
  u->bb[slot] = beta;
}

static void replay(const orc_cfg *cfg, const orc_unit *u, double *S) {
  double *k = (double *)malloc(sizeof(double) * cfg->d_k);
  double *v = (double *)malloc(sizeof(double) * cfg->d_v);
  for (int t = 0; t < u->m; ++t) {
    buffer_token(cfg, u, t, k, v);
    orc_token_update(cfg->d_k, cfg->d_v, S, k, v, (double)u->ba[t], (double)u->bb[t], NULL);
  }
  free(k);
  free(v);
}

/* One decode step ([P1] 어떻게 동작하나: the state is rounded once per dP generated tokens; the     */
/* buffered tokens are applied to the state all at once at the flush). Per-token bf16 mode is the  */
/* pages' comparison point ([P1] 전제와 한계, throughput study): no buffer, bf16 state every token;  */
/* the output is read from the state before it is rounded, as in the PACE path. Buffered bf16 mode */
/* ([P1] 전제와 한계: most of the TPOT gain comes from the decode buffer with a bf16 state) takes    */
/* the PACE path below with bf16 rounding in place of the key-axis quantizer.                      */
void orc_decode_step(const orc_cfg *cfg, orc_unit *u, const float *q, const float *k, const float *v, float a,
                     float beta, double *o) {
  const int dk = cfg->d_k, dv = cfg->d_v;
  double *S = (double *)malloc(sizeof(double) * (long)dk * dv);
  double *qd = (double *)malloc(sizeof(double) * dk);
  for (int i = 0; i < dk; ++i) qd[i] = (double)q[i];
  load_state(cfg, u, S);
  if (cfg->state_mode == ORC_STATE_BF16) {
    double *kd = (double *)malloc(sizeof(double) * dk);
    double *vd = (double *)malloc(sizeof(double) * dv);
    for (int i = 0; i < dk; ++i) kd[i] = (double)k[i];
    for (int j = 0; j < dv; ++j) vd[j] = (double)v[j];
    orc_token_update(dk, dv, S, kd, vd, (double)a, (double)beta, NULL);
    orc_readout(dk, dv, S, qd, o);
    store_state(cfg, u, S);
    free(kd);
    free(vd);
  } else {
    buffer_append(cfg, u, u->m, k, v, a, beta);
    u->m += 1;
    replay(cfg, u, S);
    orc_readout(dk, dv, S, qd, o);
    if (u->m == cfg->dP) {
      store_state(cfg, u, S);
      u->m = 0;
    }
  }
  free(S);
  free(qd);
}

void orc_flush(const orc_cfg *cfg, orc_unit *u) {
  if (cfg->state_mode == ORC_STATE_BF16 || u->m == 0) return;
  double *S = (double *)malloc(sizeof(double) * (long)cfg->d_k * cfg->d_v);
  load_state(cfg, u, S);
  replay(cfg, u, S);
  store_state(cfg, u, S);
  u->m = 0;
  free(S);
}

/* One prefill chunk ([P1] 어떻게 동작하나: the chunk kernel writes the state once per chunk, so the  */
/* prefill period is the 256-token chunk length). Inputs are applied unbuffered, then rounded once. */
void orc_prefill(const orc_cfg *cfg, orc_unit *u, int n, const float *q, const float *k, const float *v,
                 const float *a, const float *beta, double *o) {
  const int dk = cfg->d_k, dv = cfg->d_v;
  if (n <= 0) return;
  orc_flush(cfg, u);
  double *S = (double *)malloc(sizeof(double) * (long)dk * dv);
  double *kd = (double *)malloc(sizeof(double) * dk);
  double *qd = (double *)malloc(sizeof(double) * dk);
  double *vd = (double *)malloc(sizeof(double) * dv);
  load_state(cfg, u, S);
  for (int t = 0; t < n; ++t) {
    for (int i = 0; i < dk; ++i) kd[i] = (double)k[(long)t * dk + i];
    for (int i = 0; i < dk; ++i) qd[i] = (double)q[(long)t * dk + i];
    for (int j = 0; j < dv; ++j) vd[j] = (double)v[(long)t * dv + j];
    orc_token_update(dk, dv, S, kd, vd, (double)a[t], (double)beta[t], NULL);
    orc_readout(dk, dv, S, qd, o + (long)t * dv);
  }
  store_state(cfg, u, S);
  free(S);
  free(kd);
  free(qd);
  free(vd);
}

/* ---------------------------------------------------------------------------------------------- */
/* Head precision allocation ([P1] 무엇과 다른가; [P2] 3. Method & Key Results).                    */
double orc_error_energy(const orc_cfg *cfg, const float *S32) {
  const long n = (long)cfg->d_k * cfg->d_v;
  const int ng = cfg->d_k / cfg->g;
  int32_t *code = (int32_t *)malloc(sizeof(int32_t) * n);
  float *scale = (float *)malloc(sizeof(float) * ng * cfg->d_v);
  int32_t *zp = (int32_t *)malloc(sizeof(int32_t) * ng * cfg->d_v);
  double *D = (double *)malloc(sizeof(double) * n);
  orc_quantize_state(cfg, S32, code, scale, zp);
  orc_dequantize_state(cfg, code, scale, zp, D);
  double e = 0.0;
  for (long i = 0; i < n; ++i) {
    double d = D[i] - (double)S32[i];
    e += d * d;
  }
  free(code);
  free(scale);
  free(zp);
  free(D);
  return e;
}

/* The baseline the pages contrast the key-axis groups with ([P1] 무엇과 다른가: the scale is shared   */
/* by g consecutive elements along the key axis of one column, so an outlier value channel does not */
/* widen the groups of the other channels): groups of g consecutive elements along the VALUE axis   */
/* of one key row. Those are exactly the key-axis groups of the transposed state, so the error is   */
/* orc_error_energy of S^T under the same quantizer (d_k and d_v swapped). axis 0: key axis.         */
double orc_error_energy_axis(const orc_cfg *cfg, const float *S32, int axis) {
  if (axis == 0) return orc_error_energy(cfg, S32);
  const int dk = cfg->d_k, dv = cfg->d_v;
  float *T = (float *)malloc(sizeof(float) * (long)dk * dv);
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) T[(long)j * dk + i] = S32[(long)i * dv + j];
  orc_cfg ct = *cfg;
  ct.d_k = dv;
  ct.d_v = dk;
  const double e = orc_error_energy(&ct, T);
  free(T);
  return e;
}

/* One rounding leaves e_h; it decays by a_h^(2 dP) in energy per period, so the error still held  */
/* is the geometric sum e_h (1 + a^(2dP) + a^(4dP) + ...) = e_h / (1 - a_h^(2 dP)).                  */
double orc_retained_error(double e_h, double a_h, int dP) {
  if (a_h >= 1.0) return INFINITY;
  return e_h / (1.0 - pow(a_h, 2.0 * dP));
}

void orc_assign_heads(const double *e_h, const double *a_h, int H, int dP, double frac, uint8_t *mask) {
  int k = (int)floor((double)H * frac);
  double *E = (double *)malloc(sizeof(double) * H);
  for (int h = 0; h < H; ++h) {
    E[h] = orc_retained_error(e_h[h], a_h[h], dP);
    mask[h] = 0;
  }
  /* Pick the largest remaining E k times; a strict '>' keeps the lower index on ties. */
  for (int r = 0; r < k; ++r) {
    int best = -1;
    for (int h = 0; h < H; ++h) {
      if (mask[h]) continue;
      if (best < 0 || E[h] > E[best]) best = h;
    }
    if (best >= 0) mask[best] = 1;
  }
  free(E);
}

/* ---------------------------------------------------------------------------------------------- */
/* Accounting ([P1] 어떻게 동작하나: buffer cost c dP, c = (b_k d_k/gamma + b_v d_v + 32)/(d_k d_v);  */
/* [P1] 무엇과 다른가: PACE-4/8 payload 5.66 bits per value).                                        */
double orc_payload_bits(int bits, int g, int zero_point) {
  return (double)bits + (16.0 + (zero_point ? (double)bits : 0.0)) / (double)g;
}

double orc_buffer_bits(int d_k, int d_v, int b_k, int b_v, double gamma, int scalar_bits, int dP) {
  double c = ((double)b_k * d_k / gamma + (double)b_v * d_v + (double)scalar_bits) / ((double)d_k * d_v);
  return c * dP;
}

/* ---------------------------------------------------------------------------------------------- */
void orc_decode_batch(const orc_cfg *cfg, orc_unit *units, int n_units, const float *q, const float *k,
                      const float *v, const float *a, const float *beta, double *o, int nthreads) {
  const int dk = cfg->d_k, dv = cfg->d_v;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int n = 0; n < n_units; ++n)
    orc_decode_step(cfg, &units[n], q + (long)n * dk, k + (long)n * dk, v + (long)n * dv, a[n], beta[n],
                    o + (long)n * dv);
  (void)nthreads;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
