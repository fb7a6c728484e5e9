// State conversion hooks and the calibration statistic of the head ranking.
//   quantize_state:   fp32 S [B,H,D,D] -> resident format (key-axis group quantizer, [P1] 무엇과 다른가)
//   dequantize_state: resident format -> fp32 S
//   calib:            e[b,h] = || Q(S) - S ||_F^2 of an fp32 state, the error energy of one rounding that
//                     the ranking E_h = e_h / (1 - a_h^(2 dP)) uses ([P1] 무엇과 다른가).
//   validate:         counts of values no step of the method writes (a debug check, pace_validate_state).
// One CTA per unit, one thread per column; groups are thread-local.
#include "pace_common.cuh"

namespace pace {

template <int D, int BITS>
__device__ __forceinline__ uint32_t *unit_codes(const PaceDev &st, int b, int h) {
  return BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                   : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
}

template <int D, int G, int BITS>
__device__ void quantize_column(const PaceDev &st, long unit, int b, int h, const float *Sg) {
  constexpr int NG = D / G;
  const int j = threadIdx.x;
  uint32_t *codes = unit_codes<D, BITS>(st, b, h);
#pragma unroll 1
  for (int g = 0; g < NG; ++g) {
    float x[G];
#pragma unroll
    for (int ii = 0; ii < G; ++ii) x[ii] = Sg[(g * G + ii) * D + j];
    float s;
    int z;
    quant_store_group<G, BITS>(x, st.zero_point, codes, D, j, g, s, z);
    st.scale[(unit * NG + g) * D + j] = __float2bfloat16_rn(s);
    if (st.zero_point) st.zp[(unit * NG + g) * D + j] = (uint8_t)z;
  }
}

template <int D, int G, int BITS>
__device__ void dequantize_column(const PaceDev &st, long unit, int b, int h, float *So) {
  constexpr int NG = D / G;
  const int j = threadIdx.x;
  const uint32_t *codes = unit_codes<D, BITS>(st, b, h);
  for (int i = 0; i < D; ++i) {
    const int g = i / G;
    const float s = __bfloat162float(st.scale[(unit * NG + g) * D + j]);
    const int z = st.zero_point ? (int)st.zp[(unit * NG + g) * D + j] : (1 << (BITS - 1));
    So[i * D + j] = s * (float)((int)load_code<BITS>(codes, D, j, i) - z);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(D) quantize_state_kernel(const PaceDev st, const float *S) {
  const long unit = blockIdx.x;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int j = threadIdx.x;
  const float *Sg = S + unit * D * D;
  if (st.state_mode == PACE_STATE_QUANT) {
    if (st.head_is_int8[h]) quantize_column<D, G, 8>(st, unit, b, h, Sg);
    else quantize_column<D, G, 4>(st, unit, b, h, Sg);
  } else if (st.state_mode == PACE_STATE_FP32) {
    float *Sd = static_cast<float *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) Sd[i * D + j] = Sg[i * D + j];
  } else {
    __nv_bfloat16 *Sd = static_cast<__nv_bfloat16 *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) Sd[i * D + j] = __float2bfloat16_rn(Sg[i * D + j]);
  }
  if (j == 0) st.m[unit] = 0;
}

template <int D, int G>
__global__ void __launch_bounds__(D) dequantize_state_kernel(const PaceDev st, float *S) {
  const long unit = blockIdx.x;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int j = threadIdx.x;
  float *So = S + unit * D * D;
  if (st.state_mode == PACE_STATE_QUANT) {
    if (st.head_is_int8[h]) dequantize_column<D, G, 8>(st, unit, b, h, So);
    else dequantize_column<D, G, 4>(st, unit, b, h, So);
  } else if (st.state_mode == PACE_STATE_FP32) {
    const float *Ss = static_cast<const float *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) So[i * D + j] = Ss[i * D + j];
  } else {
    const __nv_bfloat16 *Ss = static_cast<const __nv_bfloat16 *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) So[i * D + j] = __bfloat162float(Ss[i * D + j]);
  }
}

template <int D, int G, int BITS, int AXIS>
__global__ void __launch_bounds__(D) calib_kernel(const PaceDev st, int zero_point, float *e_out) {
  // AXIS 0: thread j quantizes the key-axis groups of column j (PACE); AXIS 1: thread i quantizes the groups of
  // g consecutive elements along the value axis of key row i (the baseline grouping)
  constexpr int NG = D / G;
  __shared__ float red[32];
  const long unit = blockIdx.x;
  const int j = threadIdx.x;
  const float *Sg = static_cast<const float *>(st.S) + unit * D * D;
  float e = 0.0f;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float x[G];
#pragma unroll
    for (int ii = 0; ii < G; ++ii) x[ii] = AXIS == 0 ? Sg[(g * G + ii) * D + j] : Sg[j * D + g * G + ii];
    uint32_t uq[G];
    float s;
    int z;
    quant_group<G, BITS>(x, zero_point, uq, s, z);
#pragma unroll
    for (int ii = 0; ii < G; ++ii) {
      const float d = s * (float)((int)uq[ii] - z) - x[ii];
      e = fmaf(d, d, e);
    }
  }
  e = warp_sum(e);
  if ((j & 31) == 0) red[j >> 5] = e;
  __syncthreads();
  if (j == 0) {
    float t = 0.0f;
    for (int w = 0; w < D / 32; ++w) t += red[w];
    e_out[unit] = t;
  }
}

template <int D, int AXIS>
static cudaError_t launch_calib_t(const PaceDev &d, int bits, int group, int zp, float *e, cudaStream_t s) {
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  if (group == 64) {
    if (bits == 8) calib_kernel<D, 64, 8, AXIS><<<units, D, 0, s>>>(d, zp, e);
    else calib_kernel<D, 64, 4, AXIS><<<units, D, 0, s>>>(d, zp, e);
  } else {
    if (bits == 8) calib_kernel<D, 32, 8, AXIS><<<units, D, 0, s>>>(d, zp, e);
    else calib_kernel<D, 32, 4, AXIS><<<units, D, 0, s>>>(d, zp, e);
  }
  return cudaGetLastError();
}

}  // namespace pace

using namespace pace;

cudaError_t pace_launch_quantize_state(const PaceDev &d, const float *S, cudaStream_t s) {
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  if (d.D == 128) {
    if (d.G == 64) quantize_state_kernel<128, 64><<<units, 128, 0, s>>>(d, S);
    else quantize_state_kernel<128, 32><<<units, 128, 0, s>>>(d, S);
  } else {
    if (d.G == 64) quantize_state_kernel<64, 64><<<units, 64, 0, s>>>(d, S);
    else quantize_state_kernel<64, 32><<<units, 64, 0, s>>>(d, S);
  }
  return cudaGetLastError();
}

cudaError_t pace_launch_dequantize_state(const PaceDev &d, float *S, cudaStream_t s) {
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  if (d.D == 128) {
    if (d.G == 64) dequantize_state_kernel<128, 64><<<units, 128, 0, s>>>(d, S);
    else dequantize_state_kernel<128, 32><<<units, 128, 0, s>>>(d, S);
  } else {
    if (d.G == 64) dequantize_state_kernel<64, 64><<<units, 64, 0, s>>>(d, S);
    else dequantize_state_kernel<64, 32><<<units, 64, 0, s>>>(d, S);
  }
  return cudaGetLastError();
}

cudaError_t pace_launch_calib(const PaceDev &d, int bits, int group, int zero_point, int axis, float *e_out,
                              cudaStream_t s) {
  if (axis == 1)
    return d.D == 128 ? launch_calib_t<128, 1>(d, bits, group, zero_point, e_out, s)
                      : launch_calib_t<64, 1>(d, bits, group, zero_point, e_out, s);
  return d.D == 128 ? launch_calib_t<128, 0>(d, bits, group, zero_point, e_out, s)
                    : launch_calib_t<64, 0>(d, bits, group, zero_point, e_out, s);
}

// ---- pace_validate_state: every thread counts over grid-stride ranges, then one atomic add per warp and count
namespace pace {

struct ValidateArgs {
  const char *base;
  int n_guards;
  size_t guard[PACE_MAX_GUARDS];
  unsigned long long *counts;
};

__device__ __forceinline__ bool bf16_bits_nonfinite(uint32_t b) { return (b & 0x7F80u) == 0x7F80u; }

__global__ void __launch_bounds__(256) validate_kernel(const PaceDev d, const ValidateArgs a) {
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nth = (size_t)gridDim.x * blockDim.x;
  unsigned c[PACE_VALIDATE_N] = {};
  const size_t U = (size_t)d.B * d.H, D = d.D, NG = d.NG, P = d.dP;
  // [0] buffer counters
  for (size_t u = tid; u < U; u += nth) {
    const int m = d.m[u];
    if (m < 0 || m >= d.dP) ++c[0];
  }
  if (d.state_mode == PACE_STATE_QUANT) {
    // [1] scales: negative (non-zero), infinite or NaN
    const uint16_t *sc = reinterpret_cast<const uint16_t *>(d.scale);
    for (size_t i = tid; i < U * NG * D; i += nth) {
      const uint32_t b = sc[i];
      if (bf16_bits_nonfinite(b) || ((b & 0x8000u) && (b & 0x7FFFu))) ++c[1];
    }
    if (d.zero_point) {
      // [2] zero points above the head's code range
      for (size_t i = tid; i < U * NG * D; i += nth) {
        const int h = (int)((i / (NG * D)) % (size_t)d.H);
        if (d.zp[i] > (d.head_is_int8[h] ? 255 : 15)) ++c[2];
      }
    } else {
      // [3] symmetric codes at the unused level (stored 0): int4 nibbles; int8 where both planes hold 0
      const size_t W = D * D / 8;
      for (size_t i = tid; i < (size_t)d.B * d.H4 * W; i += nth) {
        const uint32_t w = d.codes4[i];
        for (int k = 0; k < 8; ++k) c[3] += ((w >> (4 * k)) & 0xFu) == 0u;
      }
      for (size_t i = tid; i < (size_t)d.B * d.H8 * W; i += nth) {
        const size_t u = i / W, r = i - u * W;
        const uint32_t lo = d.codes8[(2 * u) * W + r], hi = d.codes8[(2 * u + 1) * W + r];
        for (int k = 0; k < 8; ++k) c[3] += (((lo | hi) >> (4 * k)) & 0xFu) == 0u;
      }
    }
  } else if (d.S) {
    // [1] fp32 / bf16 state values that are infinite or NaN
    const size_t n = U * D * D;
    if (d.state_mode == PACE_STATE_FP32) {
      const float *S = static_cast<const float *>(d.S);
      for (size_t i = tid; i < n; i += nth) c[1] += !isfinite(S[i]);
    } else {
      const uint16_t *S = static_cast<const uint16_t *>(d.S);
      for (size_t i = tid; i < n; i += nth) c[1] += bf16_bits_nonfinite(S[i]);
    }
  }
  // [4] pending buffer entries (slots below m of units with a valid counter)
  if (d.buf_s && d.state_mode != PACE_STATE_BF16) {
    const bool keys = d.gamma == 1;
    for (size_t i = tid; i < U * P; i += nth) {
      const size_t u = i / P;
      const int t = (int)(i - u * P), m = d.m[u];
      if (m < 0 || m >= d.dP || t >= m) continue;
      for (int e = 0; e < 4; ++e) c[4] += !isfinite(d.buf_s[i * 4 + e]);
      if (d.buf_mode == PACE_BUF_FP32) {
        const float *kr = static_cast<const float *>(d.buf_k) + i * D, *vr = static_cast<const float *>(d.buf_v) + i * D;
        for (size_t j = 0; j < D; ++j) c[4] += (keys && !isfinite(kr[j])) + !isfinite(vr[j]);
      } else if (d.buf_mode == PACE_BUF_MIXED) {
        const uint8_t *kr = static_cast<const uint8_t *>(d.buf_k) + i * (D / 2);
        const uint16_t *vr = static_cast<const uint16_t *>(d.buf_v) + i * D;
        for (size_t j = 0; j < D / 2; ++j)
          c[4] += keys ? ((kr[j] & 0xFu) == 0u) + ((kr[j] >> 4) == 0u) : 0u;
        for (size_t j = 0; j < D; ++j) c[4] += bf16_bits_nonfinite(vr[j]);
      } else {
        const int8_t *kr = static_cast<const int8_t *>(d.buf_k) + i * D, *vr = static_cast<const int8_t *>(d.buf_v) + i * D;
        for (size_t j = 0; j < D; ++j) c[4] += (keys && kr[j] == -128) + (vr[j] == -128);
      }
    }
  }
  // [5] guard bytes
  for (int g = 0; g < a.n_guards; ++g)
    for (size_t i = tid; i < PACE_GUARD_BYTES; i += nth) c[5] += (uint8_t)a.base[a.guard[g] + i] != 0xA5u;
#pragma unroll
  for (int k = 0; k < PACE_VALIDATE_N; ++k) {
    unsigned v = c[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0 && v) atomicAdd(a.counts + k, (unsigned long long)v);
  }
}

}  // namespace pace

cudaError_t pace_launch_validate(const PaceDev &d, const char *base, const size_t *guard, int n_guards,
                                 unsigned long long *counts, cudaStream_t s) {
  pace::ValidateArgs a;
  a.base = base;
  a.n_guards = n_guards < PACE_MAX_GUARDS ? n_guards : PACE_MAX_GUARDS;
  for (int g = 0; g < PACE_MAX_GUARDS; ++g) a.guard[g] = g < a.n_guards ? guard[g] : 0;
  a.counts = counts;
  pace::validate_kernel<<<pace::device_sm_count() * 4, 256, 0, s>>>(d, a);
  return cudaGetLastError();
}
