/*
 * pace.h -- C ABI of libpace, the GB300 (sm_103a) implementation of the PACE decode hot path.
 *
 * PACE stores the recurrent state of a gated-delta linear-attention layer -- one d_k x d_v matrix per
 * (sequence, head) -- as int4 (int8 for a quarter of the heads in PACE-4/8) codes whose scales are
 * shared by g contiguous elements along the key axis of one column. The state is rounded once every
 * dP decoded tokens; the tokens in between wait in an int8 decode buffer and are replayed through the
 * gated delta rule at every step. Prefill runs in 256-token chunks and rounds once per chunk.
 *
 * Pages (cited by title and section):
 *   [P1] "PACE는 4비트 순환 상태를 주기적으로 반올림해 추론 메모리를 줄인다" (onedev.kr summary)
 *   [P2] "[논문리뷰] PACE: Periodic and Channel-Aligned Encoding of Four-Bit Recurrent States"
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller unless stated otherwise; the library
 *     never allocates device memory. `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Calls enqueue work on `stream` and return without synchronising. Argument errors are detected on
 *     the host and returned before anything is launched; a failed launch returns PACE_ERR_CUDA.
 *     pace_last_error() gives a message for the last failure of the calling thread.
 *   - q, k [B, H_k, d_k], v and o [B, H, d_v] (decode) or [B, H_k | H, n, d] (prefill) are dense row-major
 *     tensors of the configured I/O type (bf16 or fp32), H_k = key heads (= H unless configured); a and beta
 *     are fp32 [B, H] or [B, H, n].
 *   - The library does not L2-normalise k, does not scale q, and applies no output gate or norm.
 *   - Calls on one state must not overlap on the GPU (same stream, or ordered by events).
 */
#ifndef PACE_H
#define PACE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PACE_OK = 0,
  PACE_ERR_INVALID_ARG = 1,  /* bad pointer, size, shape or config field */
  PACE_ERR_UNSUPPORTED = 2,  /* valid request this library does not implement */
  PACE_ERR_STATE = 3,        /* state handle cannot take this call (e.g. wrong mode) */
  PACE_ERR_CUDA = 4,         /* a CUDA call failed; see pace_last_error() */
  PACE_ERR_TIMEOUT = 5       /* a bounded device wait gave up (pace_get_status) */
} pace_status;

/* Resident state format. */
enum {
  PACE_STATE_QUANT = 0,      /* PACE: int4/int8 codes + bf16 key-axis group scales (+ zero points) */
  PACE_STATE_FP32 = 1,       /* unquantized test mode: fp32 state, fp32 buffer, same periodic schedule */
  PACE_STATE_BF16 = 2,       /* comparison kernel: bf16 state read and written every token, no buffer */
  PACE_STATE_BF16_BUF = 3    /* bf16 state rounded once every dP tokens, with the int8 decode buffer: the
                                decode buffer without the 4-bit state ([P1] 전제와 한계: the pages attribute
                                most of the TPOT gain to the buffer with a bf16 state) */
};
/* Decode-buffer format ([P1] 어떻게 동작하나: int8 keys and values in the uniform configuration, 4-bit keys
 * and bf16 values in the mixed configuration). */
enum { PACE_BUF_INT8 = 0, PACE_BUF_MIXED = 1, PACE_BUF_FP32 = 2 };
enum { PACE_IO_BF16 = 0, PACE_IO_F32 = 1 };

#define PACE_MAX_HEADS 256
#define PACE_MAX_DP 32
#define PACE_GUARD_BYTES 256   /* guard region after every array of a state region (pace_validate_state) */
#define PACE_VALIDATE_N 6      /* counts pace_validate_state reports */

/* Immutable configuration of one state ([P1] 무엇과 다른가, 어떻게 동작하나). */
typedef struct {
  int n_heads;        /* H, 1..PACE_MAX_HEADS */
  int d_k, d_v;       /* head dims; this library: d_k == d_v, 64 or 128 */
  int max_batch;      /* sequences the device memory is sized for */
  int dP;             /* decode period, 1..PACE_MAX_DP (pages' default 8) */
  int group;          /* key-axis group size g: 32 or 64, divides d_k (PACE-4: 64, PACE-4/8: 32) */
  int zero_point;     /* 0: symmetric codes (PACE-4); 1: integer zero point (PACE-4/8) */
  int buf_mode;       /* PACE_BUF_*; PACE_STATE_FP32 requires PACE_BUF_FP32, PACE_STATE_BF16_BUF PACE_BUF_INT8 */
  int state_mode;     /* PACE_STATE_* */
  int prefill_chunk;  /* tokens rounded together in prefill; must be 256 ([P1] 어떻게 동작하나) */
  int io_dtype;       /* PACE_IO_* for q, k, v, o */
  int key_heads;      /* key heads H_k (0 = n_heads): gamma = n_heads / key_heads value heads share one key head,
                         its q and k, and one copy of its buffered key codes ([P1] 어떻게 동작하나: the buffer term
                         b_k d_k / gamma). gamma > 1 needs PACE_STATE_QUANT; value head h uses key head h / gamma */
} pace_config;

typedef struct pace_state pace_state;   /* opaque host handle */

/* Byte offsets (from the state's device base) and strides of the resident arrays, for checkpoint
 * tooling and tests. Unused arrays have offset (size_t)-1. Units are u = b*H + h.
 *   codes4  uint32 [B][H4][d_k*d_v/8]   int4 heads, in warp-level MMA fragment order. For column j let
 *                                      mt = j/16, r8 = j%8, hi = (j/8)%2; for key i let n = i/8,
 *                                      t = (i%8)/2, p = n/4, r = n%4. Key i of column j is the nibble at
 *                                      bit 4r + 16*(i%2) of word ((mt*(d_k/64) + p/2)*32 + r8*4 + t)*4
 *                                      + hi*2 + p%2
 *   codes8  uint32 [B][H8][2][d_k*d_v/8] int8 heads: plane 0 = low nibbles, plane 1 = high nibbles, each
 *                                      in the codes4 arrangement
 *           stored codes are unsigned: symmetric code c is stored as c+8 (int4) / c+128 (int8);
 *           zero-point codes are stored as they are
 *   scale   bf16   [B][H][d_k/g][d_v]   group scales
 *   zp      uint8  [B][H][d_k/g][d_v]   zero points (zero-point mode)
 *   buf_k   int8   [B][H_k][dP][d_k]    int8 buffer (one row per key head); mixed: uint8 [B][H_k][dP][d_k/2], key 2t in the low
 *                                      nibble of byte t, 2t+1 in the high one, stored as code+8;
 *                                      fp32 buffer: float [B][H][dP][d_k]
 *   buf_v   int8   [B][H][dP][d_v]      mixed: bf16 values; fp32 buffer: float
 *   buf_s   float  [B][H][dP][4]        a_t, beta_t, key scale, value scale
 *   m       int32  [B][H]               tokens in the buffer
 *   status  int32  [64]                 word 0, bit 0: a bounded device wait gave up (see pace_get_status);
 *                                      words 16..27: the counts of the last pace_validate_state
 * Every array is followed by a PACE_GUARD_BYTES guard region, filled with 0xA5 when the state is allocated;
 * pace_validate_state counts guard bytes that changed (a write past the end of an array).
 *   S       float/bf16 [B][H][d_k][d_v] state of PACE_STATE_FP32 / PACE_STATE_BF16 and PACE_STATE_BF16_BUF
 * head_slot[h] is the index of head h inside its pool (codes4 or codes8). */
typedef struct {
  size_t codes4, codes8, scale, zp, buf_k, buf_v, buf_s, m, S, status;
  size_t total_bytes;
  int H4, H8;
  int head_slot[PACE_MAX_HEADS];
  uint8_t head_is_int8[PACE_MAX_HEADS];
} pace_layout;

/* Device bytes a state for cfg->max_batch sequences needs. head_is_int8 is NULL (all heads int4) or
 * an H-byte host mask of heads kept at 8 bits (PACE-4/8, [P1] 무엇과 다른가). */
pace_status pace_state_bytes(const pace_config *cfg, const uint8_t *head_is_int8, size_t *bytes_out);

/* Bind a caller-owned device region of `bytes` (>= pace_state_bytes, 256-byte aligned) to a new state
 * handle for `batch` (1..max_batch) sequences, and enqueue its zeroing on `stream` (zero state,
 * empty buffers). The handle is host memory; release it with pace_state_free. A quantized state with
 * both int4 and int8 heads also gets its own non-blocking CUDA stream and two events (created on the
 * current device): decode steps run the int8-head pool there, forked from and joined back into the
 * caller's stream, so that the two pools share the SMs; every call stays ordered on its `stream`. */
pace_status pace_state_alloc(const pace_config *cfg, const uint8_t *head_is_int8, void *device_mem,
                             size_t bytes, int batch, void *stream, pace_state **out);
/* Frees the host handle (and the stream and events of a state with both int4 and int8 heads; work
 * already queued completes); the device region stays the caller's. NULL is accepted. */
void pace_state_free(pace_state *state);
pace_status pace_state_get_layout(const pace_state *state, pace_layout *out);

/* One prefill chunk of n_tokens (0..256) for every sequence ([P1] 어떻게 동작하나: the chunk kernel writes
 * the state once per chunk). Units with a pending decode buffer are flushed first. q, k [B,H,n,d_k],
 * v, o [B,H,n,d_v], a, beta [B,H,n]. The state is rounded once at the end of the chunk. */
pace_status pace_prefill_chunk(pace_state *state, int n_tokens, const void *q, const void *k, const void *v,
                               const float *a, const float *beta, void *o, void *stream);

/* One decode token for every sequence ([P1] 어떻게 동작하나; [P2] 1. Key Terms & Definitions): append
 * (k_t, v_t, a_t, beta_t) to the buffer, replay the buffered tokens from the rounded state through
 * S_t = a_t S_{t-1} + k_t u_t^T, u_t = beta_t (v_t - (a_t S_{t-1})^T k_t), emit o_t = S_t^T q_t, and
 * when the buffer holds dP tokens, round the state once and empty the buffer.
 * q, k [B,H,d_k], v, o [B,H,d_v], a, beta [B,H]. In PACE_STATE_BF16 mode: no buffer, the bf16 state
 * is read, updated and written every token (the pages' per-token comparison point, [P1] 전제와 한계).
 * A unit whose buffer counter is outside 0..dP-1 (e.g. after importing a corrupted region) is left
 * unchanged and its output is zero. q, k, v and o must be 16-byte aligned, a and beta 4-byte aligned
 * (PACE_ERR_INVALID_ARG otherwise, before any launch); the same holds for pace_prefill_chunk. */
pace_status pace_decode_step(pace_state *state, const void *q, const void *k, const void *v, const float *a,
                             const float *beta, void *o, void *stream);

/* Apply every pending buffer to its state, round once, and empty the buffers ([P1] 어떻게 동작하나:
 * buffered tokens are applied to the state together at the flush). */
pace_status pace_flush(pace_state *state, void *stream);

/* Host-only head ranking ([P1] 무엇과 다른가; [P2] 3. Method & Key Results): E_h = e_h / (1 - a_h^(2 dP))
 * (+inf for a_h >= 1); marks the floor(H*frac) heads with the largest E_h (ties: lower index).
 * e_h, a_h, mask_out are HOST arrays of H entries. Deterministic, no GPU needed.
 * e_h is the caller's per-head mean over calibration sequences of the per-unit energies that
 * pace_calib_error_energy writes (e_h = mean over b of e_out[b*H + h]; with the batch split over ranks, sum the
 * per-rank sums and counts first), and a_h the head's mean decay over its calibration tokens. */
pace_status pace_assign_heads(const float *e_h, const float *a_h, int H, int dP, float frac,
                              uint8_t *mask_out);

/* Set the resident state from fp32 states S [B,H,d_k,d_v] (device): quantize with the configured
 * key-axis quantizer (PACE_STATE_QUANT), copy (FP32) or round to bf16 (BF16); empties the buffers. */
pace_status pace_quantize_state(pace_state *state, const float *S, void *stream);
/* Write the resident state (without the pending buffer) as fp32 S_out [B,H,d_k,d_v] (device). */
pace_status pace_dequantize_state(const pace_state *state, float *S_out, void *stream);

/* Calibration for the head ranking: e_out[b*H+h] = || Q(S) - S ||_F^2 for the fp32 state of a
 * PACE_STATE_FP32 handle, with the key-axis quantizer (bits, group, zero_point). e_out: device, fp32. */
pace_status pace_calib_error_energy(const pace_state *fp32_state, int bits, int group, int zero_point,
                                    float *e_out, void *stream);
/* The same error energy with the groups along the key axis of one column (axis 0, PACE: the call above) or
 * along the value axis of one key row (axis 1): the grouping the pages contrast PACE's with ([P1] 무엇과
 * 다른가: sharing the scale along the key axis keeps an outlier value channel from widening the groups of the
 * other channels). Same arguments and errors as pace_calib_error_energy; axis outside {0, 1} is
 * PACE_ERR_INVALID_ARG. */
pace_status pace_calib_error_energy_axis(const pace_state *fp32_state, int bits, int group, int zero_point, int axis,
                                         float *e_out, void *stream);

/* Checkpoint / resume: copy the whole resident region (codes, scales, zero points, buffers, m) to or
 * from `bytes` bytes at dst/src, which may be host or device memory. Enqueued on `stream`. */
pace_status pace_state_export(const pace_state *state, void *dst, size_t bytes, void *stream);
pace_status pace_state_import(pace_state *state, const void *src, size_t bytes, void *stream);

/* Resident bits per state value ([P1] 어떻게 동작하나, 무엇과 다른가). literal_formula != 0: payload
 * b + (16 + zero-point bits)/g averaged over heads, plus the buffer cost c*dP with
 * c = (b_k d_k / gamma + b_v d_v + 32)/(d_k d_v), gamma = value heads per key head; literal_formula == 0: the bytes
 * this library actually keeps per state value (codes, scales, zero points, buffer, counters) * 8.
 * head_is_int8 as for pace_state_bytes. Returns a negative value for an invalid config. */
double pace_resident_bits(const pace_config *cfg, const uint8_t *head_is_int8, int literal_formula);

/* Device-side status of a state: *status_out = 0, or bit 0 set when a bounded wait inside a kernel gave up
 * (the unit involved was left unchanged). This call SYNCHRONISES `stream` to read the word; it returns
 * PACE_ERR_TIMEOUT when the bit is set, and clears it when `clear` is non-zero. */
pace_status pace_get_status(const pace_state *state, int clear, int *status_out, void *stream);

/* Failure-detection hook for tests (no fault, no hang): with ns > 0, every later tensor-core prefill launch of
 * this state (d_k = d_v = 128, bf16 I/O) first waits on an mbarrier that nothing signals, for at most ns
 * nanoseconds, gives up like any bounded wait that runs out: it issues no MMA, leaves every unit and its output
 * unchanged, sets bit 0 of the status word (pace_get_status then returns PACE_ERR_TIMEOUT) and releases its
 * tensor memory. ns = 0 turns the probe off. Host-only; PACE_ERR_INVALID_ARG for a NULL state. */
pace_status pace_test_wait_probe(pace_state *state, uint32_t ns);

/* Debug check of a state: no value of the state changes and nothing can fault. Counts, over all units, into
 * the HOST array counts_out[PACE_VALIDATE_N]:
 *   [0] buffer counters m outside 0..dP-1;
 *   [1] group scales that are negative, infinite or NaN (bf16 bits); in the fp32 and bf16 state modes, state
 *       values that are infinite or NaN;
 *   [2] zero points above the code range of their head (15 for an int4 head);
 *   [3] symmetric codes at the unused level -2^(b-1) (stored as 0);
 *   [4] values of pending buffer entries (slots below m) that no quantizer writes: an int8 code of -128, a
 *       mixed-buffer int4 key stored as 0, a non-finite bf16 value, a non-finite a, beta or scale (key rows
 *       shared by several value heads are not checked);
 *   [5] guard bytes that differ from 0xA5.
 * Launches one counting kernel on `stream` and SYNCHRONISES `stream` to read the counts. Returns
 * PACE_ERR_STATE when any count is non-zero (counts_out is filled either way). */
pace_status pace_validate_state(const pace_state *state, int64_t *counts_out, void *stream);

/* Message for the last non-OK status returned to the calling thread ("" if none). */
const char *pace_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int pace_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PACE_H */
