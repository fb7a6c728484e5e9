// Host side of libpace: argument validation, resident layout, kernel dispatch, head ranking and
// accounting. Every entry point validates on the host and returns before any launch on error.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <string>
#include <vector>

#include "pace_internal.h"

namespace {

thread_local std::string g_last_error;

pace_status fail(pace_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

pace_status ok() {
  g_last_error.clear();
  return PACE_OK;
}

pace_status cuda_fail(cudaError_t e, const char *what) {
  return fail(PACE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

pace_status validate_config(const pace_config *c, const uint8_t *mask) {
  if (!c) return fail(PACE_ERR_INVALID_ARG, "config is NULL");
  if (c->n_heads < 1 || c->n_heads > PACE_MAX_HEADS)
    return fail(PACE_ERR_INVALID_ARG, "n_heads %d outside 1..%d", c->n_heads, PACE_MAX_HEADS);
  if (c->d_k != c->d_v) return fail(PACE_ERR_UNSUPPORTED, "d_k (%d) != d_v (%d) is not supported", c->d_k, c->d_v);
  if (c->d_k != 64 && c->d_k != 128) return fail(PACE_ERR_UNSUPPORTED, "d_k = %d: supported 64, 128", c->d_k);
  if (c->max_batch < 1) return fail(PACE_ERR_INVALID_ARG, "max_batch %d < 1", c->max_batch);
  if (c->dP < 1 || c->dP > PACE_MAX_DP) return fail(PACE_ERR_INVALID_ARG, "dP %d outside 1..%d", c->dP, PACE_MAX_DP);
  if (c->group != 32 && c->group != 64)
    return fail(PACE_ERR_UNSUPPORTED, "group %d: supported 32, 64", c->group);
  if (c->group > c->d_k || c->d_k % c->group) return fail(PACE_ERR_INVALID_ARG, "group %d does not divide d_k %d", c->group, c->d_k);
  if (c->zero_point != 0 && c->zero_point != 1) return fail(PACE_ERR_INVALID_ARG, "zero_point must be 0 or 1");
  if (c->prefill_chunk != 256)
    return fail(PACE_ERR_UNSUPPORTED, "prefill_chunk %d: the method fixes it to 256", c->prefill_chunk);
  if (c->io_dtype != PACE_IO_BF16 && c->io_dtype != PACE_IO_F32) return fail(PACE_ERR_INVALID_ARG, "bad io_dtype");
  if (c->key_heads < 0 || (c->key_heads > 0 && c->n_heads % c->key_heads))
    return fail(PACE_ERR_INVALID_ARG, "key_heads %d does not divide n_heads %d", c->key_heads, c->n_heads);
  if (c->key_heads > 0 && c->key_heads != c->n_heads && c->state_mode != PACE_STATE_QUANT)
    return fail(PACE_ERR_UNSUPPORTED, "shared key heads need the quantized state mode");
  switch (c->state_mode) {
    case PACE_STATE_QUANT:
      if (c->buf_mode != PACE_BUF_INT8 && c->buf_mode != PACE_BUF_MIXED)
        return fail(PACE_ERR_UNSUPPORTED, "quantized state needs an int8 or mixed buffer");
      break;
    case PACE_STATE_FP32:
      if (c->buf_mode != PACE_BUF_FP32) return fail(PACE_ERR_INVALID_ARG, "fp32 state needs the fp32 buffer");
      break;
    case PACE_STATE_BF16:
      break;
    case PACE_STATE_BF16_BUF:
      if (c->buf_mode != PACE_BUF_INT8) return fail(PACE_ERR_UNSUPPORTED, "buffered bf16 state needs the int8 buffer");
      break;
    default:
      return fail(PACE_ERR_INVALID_ARG, "bad state_mode %d", c->state_mode);
  }
  if (mask && c->state_mode != PACE_STATE_QUANT) {
    for (int h = 0; h < c->n_heads; ++h)
      if (mask[h]) return fail(PACE_ERR_INVALID_ARG, "8-bit heads need the quantized state mode");
  }
  return PACE_OK;
}

// Offsets of every resident array for `batch` sequences.
pace_layout make_layout(const pace_config *c, const uint8_t *mask, int batch, size_t *guard = nullptr,
                        int *n_guards = nullptr) {
  pace_layout L;
  memset(&L, 0, sizeof L);
  const size_t none = (size_t)-1;
  L.codes4 = L.codes8 = L.scale = L.zp = L.buf_k = L.buf_v = L.buf_s = L.m = L.S = L.status = none;
  const size_t B = (size_t)batch, H = (size_t)c->n_heads, D = (size_t)c->d_k, NG = D / (size_t)c->group;
  const size_t Hk = c->key_heads > 0 ? (size_t)c->key_heads : H;
  const size_t P = (size_t)c->dP;
  int h4 = 0, h8 = 0;
  for (int h = 0; h < c->n_heads; ++h) {
    const int is8 = (mask && mask[h]) ? 1 : 0;
    L.head_is_int8[h] = (uint8_t)is8;
    L.head_slot[h] = is8 ? h8++ : h4++;
  }
  L.H4 = h4;
  L.H8 = h8;
  size_t off = 0;
  int ng = 0;
  auto take = [&](size_t &field, size_t bytes) {   // the array, then its guard region
    field = off;
    off = align256(off + bytes);
    if (guard && ng < PACE_MAX_GUARDS) guard[ng] = off;
    ++ng;
    off += PACE_GUARD_BYTES;
  };
  if (c->state_mode == PACE_STATE_QUANT) {
    take(L.codes4, B * h4 * (D / 8) * D * 4);
    take(L.codes8, B * h8 * (D / 4) * D * 4);
    take(L.scale, B * H * NG * D * 2);
    if (c->zero_point) take(L.zp, B * H * NG * D);
    if (c->buf_mode == PACE_BUF_MIXED) {
      take(L.buf_k, B * Hk * P * (D / 2));
      take(L.buf_v, B * H * P * D * 2);
    } else {
      take(L.buf_k, B * Hk * P * D);
      take(L.buf_v, B * H * P * D);
    }
    take(L.buf_s, B * H * P * 16);
  } else if (c->state_mode == PACE_STATE_FP32) {
    take(L.S, B * H * D * D * 4);
    take(L.buf_k, B * H * P * D * 4);
    take(L.buf_v, B * H * P * D * 4);
    take(L.buf_s, B * H * P * 16);
  } else if (c->state_mode == PACE_STATE_BF16_BUF) {
    take(L.S, B * H * D * D * 2);
    take(L.buf_k, B * H * P * D);
    take(L.buf_v, B * H * P * D);
    take(L.buf_s, B * H * P * 16);
  } else {
    take(L.S, B * H * D * D * 2);
  }
  take(L.m, B * H * 4);
  take(L.status, 64 * 4);
  L.total_bytes = off;
  if (n_guards) *n_guards = ng;
  return L;
}

template <typename T>
T *at(char *base, size_t off) {
  return off == (size_t)-1 ? nullptr : reinterpret_cast<T *>(base + off);
}

pace_status check_state(const pace_state *s) {
  if (!s) return fail(PACE_ERR_INVALID_ARG, "state is NULL");
  return PACE_OK;
}

bool need(const void *p) { return p != nullptr; }

}  // namespace

extern "C" {

int pace_version(void) { return 100; }

const char *pace_last_error(void) { return g_last_error.c_str(); }

pace_status pace_state_bytes(const pace_config *cfg, const uint8_t *head_is_int8, size_t *bytes_out) {
  pace_status st = validate_config(cfg, head_is_int8);
  if (st != PACE_OK) return st;
  if (!bytes_out) return fail(PACE_ERR_INVALID_ARG, "bytes_out is NULL");
  *bytes_out = make_layout(cfg, head_is_int8, cfg->max_batch).total_bytes;
  return ok();
}

pace_status pace_state_alloc(const pace_config *cfg, const uint8_t *head_is_int8, void *device_mem, size_t bytes,
                             int batch, void *stream, pace_state **out) {
  pace_status st = validate_config(cfg, head_is_int8);
  if (st != PACE_OK) return st;
  if (!out) return fail(PACE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (batch < 1 || batch > cfg->max_batch)
    return fail(PACE_ERR_INVALID_ARG, "batch %d outside 1..max_batch (%d)", batch, cfg->max_batch);
  if (!device_mem) return fail(PACE_ERR_INVALID_ARG, "device_mem is NULL");
  if (reinterpret_cast<uintptr_t>(device_mem) % 256)
    return fail(PACE_ERR_INVALID_ARG, "device_mem must be 256-byte aligned");
  size_t guard[PACE_MAX_GUARDS];
  int n_guards = 0;
  const pace_layout L = make_layout(cfg, head_is_int8, batch, guard, &n_guards);
  if (bytes < L.total_bytes)
    return fail(PACE_ERR_INVALID_ARG, "device region of %zu bytes is smaller than the %zu the state needs", bytes,
                L.total_bytes);
  pace_state *s = new (std::nothrow) pace_state;
  if (!s) return fail(PACE_ERR_INVALID_ARG, "host allocation of the handle failed");
  s->cfg = *cfg;
  s->batch = batch;
  s->lay = L;
  s->base = static_cast<char *>(device_mem);
  s->bytes = bytes;
  s->n_guards = n_guards;
  for (int g = 0; g < n_guards; ++g) s->guard[g] = guard[g];
  PaceDev &d = s->dev;
  memset(&d, 0, sizeof d);
  d.B = batch;
  d.H = cfg->n_heads;
  d.D = cfg->d_k;
  d.G = cfg->group;
  d.NG = cfg->d_k / cfg->group;
  d.dP = cfg->dP;
  d.zero_point = cfg->zero_point;
  d.buf_mode = cfg->buf_mode;
  d.state_mode = cfg->state_mode;
  d.io = cfg->io_dtype;
  d.H4 = L.H4;
  d.H8 = L.H8;
  d.Hk = cfg->key_heads > 0 ? cfg->key_heads : cfg->n_heads;
  d.gamma = cfg->n_heads / d.Hk;
  d.codes4 = at<uint32_t>(s->base, L.codes4);
  d.codes8 = at<uint32_t>(s->base, L.codes8);
  d.scale = at<__nv_bfloat16>(s->base, L.scale);
  d.zp = at<uint8_t>(s->base, L.zp);
  d.buf_k = at<void>(s->base, L.buf_k);
  d.buf_v = at<void>(s->base, L.buf_v);
  d.buf_s = at<float>(s->base, L.buf_s);
  d.m = at<int32_t>(s->base, L.m);
  d.status = at<int32_t>(s->base, L.status);
  d.S = at<void>(s->base, L.S);
  for (int h = 0; h < cfg->n_heads; ++h) {
    d.head_is_int8[h] = L.head_is_int8[h];
    d.head_slot[h] = (int16_t)L.head_slot[h];
    d.pool_head[(L.head_is_int8[h] ? L.H4 : 0) + L.head_slot[h]] = (int16_t)h;
  }
  // zero state: every code stands for 0 (symmetric codes are stored offset by 2^(b-1))
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(s->base, 0, L.total_bytes, cs);
  if (e == cudaSuccess && cfg->state_mode == PACE_STATE_QUANT && !cfg->zero_point) {
    const size_t D = cfg->d_k;
    if (L.H4) e = cudaMemsetAsync(d.codes4, 0x88, (size_t)batch * L.H4 * (D / 8) * D * 4, cs);
    // int8 code 0 is stored as 128: low-nibble plane 0x0, high-nibble plane 0x8
    const size_t plane = (size_t)(D / 8) * D * 4;
    if (e == cudaSuccess && L.H8)
      e = cudaMemset2DAsync(reinterpret_cast<char *>(d.codes8) + plane, 2 * plane, 0x88, plane, (size_t)batch * L.H8, cs);
  }
  for (int g = 0; g < n_guards && e == cudaSuccess; ++g) e = cudaMemsetAsync(s->base + guard[g], 0xA5, PACE_GUARD_BYTES, cs);
  if (e != cudaSuccess) {
    delete s;
    return cuda_fail(e, "zeroing the state");
  }
  if (cfg->state_mode == PACE_STATE_QUANT && L.H4 > 0 && L.H8 > 0) {
    e = cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      pace_state_free(s);
      return cuda_fail(e, "creating the int8-pool stream");
    }
  }
  *out = s;
  return ok();
}

void pace_state_free(pace_state *state) {
  if (!state) return;
  const PaceDev &d = state->dev;
  if (d.ev_join) cudaEventDestroy(d.ev_join);
  if (d.ev_fork) cudaEventDestroy(d.ev_fork);
  if (d.side) cudaStreamDestroy(d.side);
  delete state;
}

pace_status pace_state_get_layout(const pace_state *state, pace_layout *out) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!out) return fail(PACE_ERR_INVALID_ARG, "out is NULL");
  *out = state->lay;
  return ok();
}

// The kernels read q, k, v and write o in 8- and 16-byte vectors.
static bool io_aligned(const void *q, const void *k, const void *v, const float *a, const float *beta, const void *o) {
  auto al = [](const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
  return al(q, 16) && al(k, 16) && al(v, 16) && al(o, 16) && al(a, 4) && al(beta, 4);
}

pace_status pace_decode_step(pace_state *state, const void *q, const void *k, const void *v, const float *a,
                             const float *beta, void *o, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!need(q) || !need(k) || !need(v) || !need(a) || !need(beta) || !need(o))
    return fail(PACE_ERR_INVALID_ARG, "decode_step: a tensor pointer is NULL");
  if (!io_aligned(q, k, v, a, beta, o))
    return fail(PACE_ERR_INVALID_ARG, "decode_step: q, k, v, o must be 16-byte aligned, a and beta 4-byte aligned");
  PaceIO io{q, k, v, a, beta, o, 1};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (state->cfg.state_mode == PACE_STATE_BF16)
    e = pace_launch_decode_bf16(state->dev, io, cs);
  else if (state->cfg.state_mode == PACE_STATE_QUANT)
    e = pace_launch_decode_quant(state->dev, io, 1, cs);
  else
    e = pace_launch_decode(state->dev, io, 1, cs);
  if (e != cudaSuccess) return cuda_fail(e, "decode_step launch");
  return ok();
}

pace_status pace_flush(pace_state *state, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (state->cfg.state_mode == PACE_STATE_BF16) return ok();   // no buffer
  PaceIO io{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = state->cfg.state_mode == PACE_STATE_QUANT ? pace_launch_decode_quant(state->dev, io, 0, cs)
                                                            : pace_launch_decode(state->dev, io, 0, cs);
  if (e != cudaSuccess) return cuda_fail(e, "flush launch");
  return ok();
}

pace_status pace_prefill_chunk(pace_state *state, int n_tokens, const void *q, const void *k, const void *v,
                               const float *a, const float *beta, void *o, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (n_tokens < 0 || n_tokens > state->cfg.prefill_chunk)
    return fail(PACE_ERR_INVALID_ARG, "n_tokens %d outside 0..%d", n_tokens, state->cfg.prefill_chunk);
  if (n_tokens == 0) return ok();
  if (!need(q) || !need(k) || !need(v) || !need(a) || !need(beta) || !need(o))
    return fail(PACE_ERR_INVALID_ARG, "prefill_chunk: a tensor pointer is NULL");
  if (!io_aligned(q, k, v, a, beta, o))
    return fail(PACE_ERR_INVALID_ARG, "prefill_chunk: q, k, v, o must be 16-byte aligned, a and beta 4-byte aligned");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (state->cfg.state_mode != PACE_STATE_BF16) {
    PaceIO fio{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    e = state->cfg.state_mode == PACE_STATE_QUANT ? pace_launch_decode_quant(state->dev, fio, 0, cs)
                                                  : pace_launch_decode(state->dev, fio, 0, cs);   // pending buffers first
    if (e != cudaSuccess) return cuda_fail(e, "prefill flush launch");
  }
  PaceIO io{q, k, v, a, beta, o, n_tokens};
  e = pace_prefill_tc_supported(state->dev) ? pace_launch_prefill_tc(state->dev, io, cs) : pace_launch_prefill(state->dev, io, cs);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return ok();
}

pace_status pace_quantize_state(pace_state *state, const float *S, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!S) return fail(PACE_ERR_INVALID_ARG, "S is NULL");
  cudaError_t e = pace_launch_quantize_state(state->dev, S, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize_state launch");
  return ok();
}

pace_status pace_dequantize_state(const pace_state *state, float *S_out, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!S_out) return fail(PACE_ERR_INVALID_ARG, "S_out is NULL");
  cudaError_t e = pace_launch_dequantize_state(state->dev, S_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dequantize_state launch");
  return ok();
}

pace_status pace_calib_error_energy(const pace_state *state, int bits, int group, int zero_point, float *e_out,
                                    void *stream) {
  return pace_calib_error_energy_axis(state, bits, group, zero_point, 0, e_out, stream);
}

pace_status pace_calib_error_energy_axis(const pace_state *state, int bits, int group, int zero_point, int axis,
                                         float *e_out, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (state->cfg.state_mode != PACE_STATE_FP32)
    return fail(PACE_ERR_STATE, "calibration reads an fp32 (unquantized) state");
  if (bits != 4 && bits != 8) return fail(PACE_ERR_INVALID_ARG, "bits must be 4 or 8");
  if ((group != 32 && group != 64) || state->cfg.d_k % group)
    return fail(PACE_ERR_INVALID_ARG, "group %d not supported for d_k %d", group, state->cfg.d_k);
  if (zero_point != 0 && zero_point != 1) return fail(PACE_ERR_INVALID_ARG, "zero_point must be 0 or 1");
  if (axis != 0 && axis != 1) return fail(PACE_ERR_INVALID_ARG, "axis must be 0 (key axis) or 1 (value axis)");
  if (!e_out) return fail(PACE_ERR_INVALID_ARG, "e_out is NULL");
  cudaError_t e = pace_launch_calib(state->dev, bits, group, zero_point, axis, e_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "calibration launch");
  return ok();
}

pace_status pace_state_export(const pace_state *state, void *dst, size_t bytes, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!dst) return fail(PACE_ERR_INVALID_ARG, "dst is NULL");
  if (bytes < state->lay.total_bytes)
    return fail(PACE_ERR_INVALID_ARG, "export needs %zu bytes, got %zu", state->lay.total_bytes, bytes);
  cudaError_t e = cudaMemcpyAsync(dst, state->base, state->lay.total_bytes, cudaMemcpyDefault,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "state export copy");
  return ok();
}

pace_status pace_state_import(pace_state *state, const void *src, size_t bytes, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!src) return fail(PACE_ERR_INVALID_ARG, "src is NULL");
  if (bytes != state->lay.total_bytes)
    return fail(PACE_ERR_INVALID_ARG, "import expects exactly %zu bytes, got %zu", state->lay.total_bytes, bytes);
  cudaError_t e = cudaMemcpyAsync(state->base, src, bytes, cudaMemcpyDefault, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "state import copy");
  return ok();
}

pace_status pace_test_wait_probe(pace_state *state, uint32_t ns) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  state->dev.probe_ns = ns;
  return ok();
}

pace_status pace_get_status(const pace_state *state, int clear, int *status_out, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!status_out) return fail(PACE_ERR_INVALID_ARG, "status_out is NULL");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, state->dev.status, 4, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess && clear && word) e = cudaMemsetAsync(state->dev.status, 0, 4, cs);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  *status_out = word;
  if (word & 1) return fail(PACE_ERR_TIMEOUT, "a bounded device wait gave up");
  return ok();
}

pace_status pace_validate_state(const pace_state *state, int64_t *counts_out, void *stream) {
  pace_status st = check_state(state);
  if (st != PACE_OK) return st;
  if (!counts_out) return fail(PACE_ERR_INVALID_ARG, "counts_out is NULL");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // the counts live in the status array (words 16..27) of the caller's region: the library allocates nothing
  unsigned long long *dev = reinterpret_cast<unsigned long long *>(state->base + state->lay.status + 64);
  unsigned long long host[PACE_VALIDATE_N] = {};
  cudaError_t e = cudaMemsetAsync(dev, 0, sizeof host, cs);
  if (e == cudaSuccess) e = pace_launch_validate(state->dev, state->base, state->guard, state->n_guards, dev, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, dev, sizeof host, cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e, "validating the state");
  unsigned long long any = 0;
  for (int k = 0; k < PACE_VALIDATE_N; ++k) {
    counts_out[k] = (int64_t)host[k];
    any |= host[k];
  }
  if (any)
    return fail(PACE_ERR_STATE, "state check: %llu counters, %llu scales/values, %llu zero points, %llu unused-level "
                "codes, %llu buffer values, %llu guard bytes out of range", host[0], host[1], host[2], host[3], host[4],
                host[5]);
  return ok();
}

pace_status pace_assign_heads(const float *e_h, const float *a_h, int H, int dP, float frac, uint8_t *mask_out) {
  if (!e_h || !a_h || !mask_out) return fail(PACE_ERR_INVALID_ARG, "assign_heads: NULL array");
  if (H < 1 || H > PACE_MAX_HEADS) return fail(PACE_ERR_INVALID_ARG, "H %d outside 1..%d", H, PACE_MAX_HEADS);
  if (dP < 1) return fail(PACE_ERR_INVALID_ARG, "dP %d < 1", dP);
  if (!(frac >= 0.0f && frac <= 1.0f)) return fail(PACE_ERR_INVALID_ARG, "frac must lie in [0, 1]");
  // E_h = e_h / (1 - a_h^(2 dP)): the rounding error still held after it decays for every period
  std::vector<double> E(H);
  for (int h = 0; h < H; ++h) {
    const double a = a_h[h], e = e_h[h];
    if (!(e >= 0.0) || !(a >= 0.0)) return fail(PACE_ERR_INVALID_ARG, "e_h and a_h must be finite, >= 0");
    E[h] = a >= 1.0 ? INFINITY : e / (1.0 - pow(a, 2.0 * dP));
  }
  std::vector<int> order(H);
  for (int h = 0; h < H; ++h) order[h] = h;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return E[x] > E[y]; });
  const int k = (int)floor((double)H * (double)frac);
  for (int h = 0; h < H; ++h) mask_out[h] = 0;
  for (int r = 0; r < k; ++r) mask_out[order[r]] = 1;
  return ok();
}

double pace_resident_bits(const pace_config *cfg, const uint8_t *head_is_int8, int literal_formula) {
  if (validate_config(cfg, head_is_int8) != PACE_OK) return -1.0;
  const double D = cfg->d_k, H = cfg->n_heads;
  const double values = (double)cfg->max_batch * H * D * D;
  if (!literal_formula) {
    int ng = 0;
    const pace_layout L = make_layout(cfg, head_is_int8, cfg->max_batch, nullptr, &ng);
    return 8.0 * (double)(L.total_bytes - (size_t)ng * PACE_GUARD_BYTES) / values;   // (guards are not state)
  }
  if (cfg->state_mode == PACE_STATE_FP32) return 32.0 + 0.0;
  if (cfg->state_mode == PACE_STATE_BF16) return 16.0;
  if (cfg->state_mode == PACE_STATE_BF16_BUF) return 16.0 + (8.0 * D + 8.0 * D + 32.0) / (D * D) * cfg->dP;
  int n8 = 0;
  for (int h = 0; h < cfg->n_heads; ++h) n8 += (head_is_int8 && head_is_int8[h]) ? 1 : 0;
  const double f8 = n8 / H;
  auto payload = [&](int bits) { return bits + (16.0 + (cfg->zero_point ? bits : 0)) / cfg->group; };
  const double bk = cfg->buf_mode == PACE_BUF_MIXED ? 4.0 : 8.0, bv = cfg->buf_mode == PACE_BUF_MIXED ? 16.0 : 8.0;
  const double gamma = cfg->key_heads > 0 ? H / cfg->key_heads : 1.0;
  const double c = (bk * D / gamma + bv * D + 32.0) / (D * D);
  return (1.0 - f8) * payload(4) + f8 * payload(8) + c * cfg->dP;
}

}  // extern "C"
