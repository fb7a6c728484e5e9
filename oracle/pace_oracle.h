/*
 * pace_oracle.h -- plain CPU statement of the PACE decode path (TEST INFRASTRUCTURE ONLY).
 *
 * This is the oracle the CUDA library is checked against. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or helper with the CUDA library, and it never calls it.
 *
 * Sources (each page is cited by its title and the section a rule comes from):
 *   [P1] "PACE는 4비트 순환 상태를 주기적으로 반올림해 추론 메모리를 줄인다" (onedev.kr summary)
 *   [P2] "[논문리뷰] PACE: Periodic and Channel-Aligned Encoding of Four-Bit Recurrent States"
 *   [P3] "PACE сжимает состояние линейных LLM до 4 бит и экономит треть памяти" (news piece)
 *
 * Canonical layouts used by every oracle function (one unit = one (sequence, head)):
 *   state S          double [d_k][d_v]   S[i*d_v + j], row i = key index, column j = value channel
 *   codes            int32  [d_k][d_v]   same indexing; symmetric codes are signed,
 *                                         zero-point codes are unsigned 0..2^b-1
 *   scale, zp        float / int32 [d_k/g][d_v]   one entry per key-axis group of one column
 */
#ifndef PACE_ORACLE_H
#define PACE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BUF_INT8 = 0, ORC_BUF_MIXED = 1, ORC_BUF_FP32 = 2 };
/* ORC_STATE_BF16: per-token bf16 state, no buffer (the pages' comparison point).
 * ORC_STATE_BF16_BUF: bf16 state with PACE's decode buffer: rounded to bf16 once every dP tokens. */
enum { ORC_STATE_QUANT = 0, ORC_STATE_FP32 = 1, ORC_STATE_BF16 = 2, ORC_STATE_BF16_BUF = 3 };

typedef struct {
  int d_k, d_v;
  int g;           /* key-axis group size (elements) */
  int bits;        /* state code width: 4 or 8 */
  int zero_point;  /* 0: symmetric, 1: integer zero-point */
  int dP;          /* decode period */
  int buf_mode;    /* ORC_BUF_* */
  int state_mode;  /* ORC_STATE_* */
} orc_cfg;

/* One unit's resident data. Arrays are owned by the caller; unused arrays may be NULL. */
typedef struct {
  int32_t *code;   /* [d_k*d_v]          quantized mode */
  float   *scale;  /* [(d_k/g)*d_v]      quantized mode */
  int32_t *zp;     /* [(d_k/g)*d_v]      quantized mode, zero-point only */
  double  *S;      /* [d_k*d_v]          fp32 mode (kept exact, fp64); bf16 modes (bf16 values) */
  int      m;      /* tokens held in the decode buffer */
  /* decode buffer, dP slots */
  int32_t *bk;     /* [dP*d_k] key codes (int8 or int4 mode) */
  int32_t *bv;     /* [dP*d_v] value codes (int8 mode) */
  float   *bsk;    /* [dP] key scales */
  float   *bsv;    /* [dP] value scales (int8 mode) */
  float   *bkf;    /* [dP*d_k] fp32 keys (fp32 buffer mode) */
  float   *bvf;    /* [dP*d_v] values: bf16 values (mixed mode) or fp32 values (fp32 mode) */
  float   *ba;     /* [dP] decay a_t */
  float   *bb;     /* [dP] beta_t */
} orc_unit;

/* Rounding of an fp32 value to the nearest bf16 value, ties to even; returned as fp32. */
float orc_bf16_rn(float x);
void orc_bf16_rn_array(const float *x, float *y, long n);

/* State quantizers of one key-axis group: n values x[0], x[stride], ... */
void orc_quant_group_sym(const float *x, int n, int stride, int bits, float *s, int32_t *c, int cstride);
void orc_quant_group_zp(const float *x, int n, int stride, int bits, float *s, int32_t *z, int32_t *c,
                        int cstride);
/* Whole-state quantize / dequantize (all columns, all groups). */
void orc_quantize_state(const orc_cfg *cfg, const float *S32, int32_t *code, float *scale, int32_t *zp);
void orc_dequantize_state(const orc_cfg *cfg, const int32_t *code, const float *scale, const int32_t *zp,
                          double *S);
/* Per-token decode-buffer quantizer: symmetric, one fp32 scale for the vector, codes in [-qmax, qmax]. */
void orc_buffer_quant(const float *x, int n, int qmax, int32_t *c, float *s);

/* Gated delta rule for one token, in fp64:
 *   w = (a S)^T k,  u = beta (v - w),  S <- a S + k u^T.   u_out may be NULL. */
void orc_token_update(int d_k, int d_v, double *S, const double *k, const double *v, double a, double beta,
                      double *u_out);
/* o = S^T q */
void orc_readout(int d_k, int d_v, const double *S, const double *q, double *o);

/* One decode step of one unit (buffer append, replay, readout, flush when the buffer holds dP tokens). */
void orc_decode_step(const orc_cfg *cfg, orc_unit *u, const float *q, const float *k, const float *v, float a,
                     float beta, double *o);
/* Apply a pending buffer to the state and round once (no-op when m == 0). */
void orc_flush(const orc_cfg *cfg, orc_unit *u);
/* One prefill chunk of n tokens (flushes a pending buffer first), rounding the state once at its end. */
void orc_prefill(const orc_cfg *cfg, orc_unit *u, int n, const float *q, const float *k, const float *v,
                 const float *a, const float *beta, double *o);

/* Error energy of one rounding of an fp32 state: sum (deq(Q(S)) - S)^2. */
double orc_error_energy(const orc_cfg *cfg, const float *S32);
/* Same with the groups along the value axis of one key row (axis 1), the baseline grouping; axis 0 = key axis. */
double orc_error_energy_axis(const orc_cfg *cfg, const float *S32, int axis);
/* Head ranking by E_h = e_h / (1 - a_h^(2 dP)); marks the floor(H*frac) largest (ties: lower index). */
void orc_assign_heads(const double *e_h, const double *a_h, int H, int dP, double frac, uint8_t *mask);
/* Retained error E_h of one head (closed form; +inf when a_h >= 1). */
double orc_retained_error(double e_h, double a_h, int dP);

/* Accounting, bits per state value. */
double orc_payload_bits(int bits, int g, int zero_point);
double orc_buffer_bits(int d_k, int d_v, int b_k, int b_v, double gamma, int scalar_bits, int dP);

/* Batched decode over n units sharing one config (per-unit inputs at unit stride), OpenMP over units
 * with nthreads threads (<= 0: runtime default). Used only to time the oracle. */
void orc_decode_batch(const orc_cfg *cfg, orc_unit *units, int n_units, const float *q, const float *k,
                      const float *v, const float *a, const float *beta, double *o, int nthreads);
int orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
