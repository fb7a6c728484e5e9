// Internal declarations shared by the host runtime and the kernels of libpace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pace.h"

// Device view of one state, passed by value to every kernel (fits in the kernel parameter space).
struct PaceDev {
  int B, H, D, G, NG, dP;
  int zero_point, buf_mode, state_mode, io;
  int H4, H8;
  int Hk, gamma;           // key heads; value heads per key head (value head h reads key head h / gamma)
  uint32_t *codes4;        // [B][H4][D/8][D]
  uint32_t *codes8;        // [B][H8][D/4][D]
  __nv_bfloat16 *scale;    // [B][H][NG][D]
  uint8_t *zp;             // [B][H][NG][D]
  void *buf_k;             // int8 [B][H][dP][D] | packed int4 [B][H][dP][D/2] | f32 [B][H][dP][D]
  void *buf_v;             // int8 [B][H][dP][D] | bf16 | f32
  float *buf_s;            // [B][H][dP][4]: a, beta, s_k, s_v
  int32_t *m;              // [B][H]
  int32_t *status;         // one word: bit 0 set when a bounded device wait gave up
  uint32_t probe_ns;       // failure-detection test: > 0 makes the tensor-core prefill wait this long on an
                           // mbarrier that nothing signals, give up and report (pace_test_wait_probe)
  void *S;                 // f32 / bf16 [B][H][D][D]
  // host-side: with int4 and int8 heads both present, the int8-head pool of a decode step runs on this state's own
  // stream, forked from the caller's stream and joined back into it (null otherwise)
  cudaStream_t side;
  cudaEvent_t ev_fork, ev_join;
  uint8_t head_is_int8[PACE_MAX_HEADS];
  int16_t head_slot[PACE_MAX_HEADS];
  int16_t pool_head[PACE_MAX_HEADS];   // heads of the int4 pool in slot order, then those of the int8 pool
};

constexpr int PACE_MAX_GUARDS = 16;

struct pace_state {
  pace_config cfg;
  int batch;
  pace_layout lay;
  char *base;
  size_t bytes;
  PaceDev dev;
  int n_guards;                   // guard regions (PACE_GUARD_BYTES each, 0xA5) after the arrays of the region
  size_t guard[PACE_MAX_GUARDS];  // their offsets
};

// Per-call pointers of one decode step / flush / prefill chunk.
struct PaceIO {
  const void *q, *k, *v;
  const float *a, *beta;
  void *o;
  int n;            // tokens (prefill) ; decode: 1 ; flush: 0
};

// Kernel launchers (each returns the launch status; nothing synchronises).
cudaError_t pace_launch_decode(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s);
cudaError_t pace_launch_decode_quant(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s);
cudaError_t pace_launch_decode_bf16(const PaceDev &d, const PaceIO &io, cudaStream_t s);
// The folded-readout kernel with 32-token tables (decode_fold_t32.cu): int4 symmetric, g = 64, int8 buffer, no int8
// heads, 8 < dP <= 32.
bool pace_fold32_supported(const PaceDev &d);
cudaError_t pace_launch_decode_fold32(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s);
// Buffered bf16 state with dP <= 8 on the folded-readout kernel (decode_fold.cuh).
cudaError_t pace_launch_decode_bf16buf_fold(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s);
cudaError_t pace_launch_prefill(const PaceDev &d, const PaceIO &io, cudaStream_t s);
// Tensor-core chunk prefill (d_k = d_v = 128, bf16 I/O); pace_prefill_tc_supported says whether it applies.
bool pace_prefill_tc_supported(const PaceDev &d);
cudaError_t pace_launch_prefill_tc(const PaceDev &d, const PaceIO &io, cudaStream_t s);
cudaError_t pace_launch_quantize_state(const PaceDev &d, const float *S, cudaStream_t s);
// Counting kernel of pace_validate_state: adds the PACE_VALIDATE_N counts into counts (device, zeroed by the caller).
cudaError_t pace_launch_validate(const PaceDev &d, const char *base, const size_t *guard, int n_guards,
                                 unsigned long long *counts, cudaStream_t s);
cudaError_t pace_launch_dequantize_state(const PaceDev &d, float *S, cudaStream_t s);
cudaError_t pace_launch_calib(const PaceDev &d, int bits, int group, int zero_point, int axis, float *e_out,
                              cudaStream_t s);
