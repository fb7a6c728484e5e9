// Device helpers shared by the libpace kernels: I/O conversion, integer dot products, block
// reductions and the key-axis group quantizers.
#pragma once

#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include "pace_internal.h"

namespace pace {

// Sequential carving of a dynamic shared-memory block (16-byte aligned pieces, or `align`).
__host__ __device__ inline size_t carve(size_t &off, size_t bytes, size_t align = 16) {
  const size_t o = (off + align - 1) & ~(align - 1);
  off = o + bytes;
  return o;
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float load_io(const void *p, long idx, int io) {
  if (io == PACE_IO_F32) return static_cast<const float *>(p)[idx];
  return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[idx]);
}

__device__ __forceinline__ void store_io(void *p, long idx, float v, int io) {
  if (io == PACE_IO_F32)
    static_cast<float *>(p)[idx] = v;
  else
    static_cast<__nv_bfloat16 *>(p)[idx] = __float2bfloat16_rn(v);
}

// Four-way byte dot product: unsigned bytes of a times signed bytes of b, added to c.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// Four-way byte dot product of signed bytes.
__device__ __forceinline__ int dp4a_ss(int a, int b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Max over the block; `red` holds >= 32 floats of shared scratch. Every thread gets the result.
__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = lane < nw ? red[lane] : 0.0f;
  return warp_max(r);
}

// Symmetric or zero-point quantization of one key-axis group of N values ([P1] 무엇과 다른가).
// Every fp32 operation rounds once (explicit _rn intrinsics, no contraction):
//   symmetric:  s = bf16(A / qmax), r = 1/s, c = clamp(rint(x*r), -qmax, qmax), stored u = c + 2^(b-1)
//   zero point: s = bf16((hi-lo)/(2^b-1)), z = clamp(rint(-lo*r)), u = clamp(rint(x*r) + z), lo <= 0 <= hi
// A zero or subnormal scale makes the whole group zero. Returns the stored unsigned codes u, the
// scale and the zero offset z_out (2^(b-1) for symmetric), so that the value is s * (u - z_out).
template <int N, int BITS>
__device__ __forceinline__ void quant_group(const float (&x)[N], int zero_point, uint32_t (&u)[N],
                                            float &s_out, int &z_out) {
  if (!zero_point) {
    constexpr int qmax = (1 << (BITS - 1)) - 1;
    constexpr int off = 1 << (BITS - 1);
    float A = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) A = fmaxf(A, fabsf(x[i]));
    float s = bf16_round(__fdiv_rn(A, (float)qmax));
    z_out = off;
    if (!(s >= FLT_MIN)) {
      s_out = 0.0f;
#pragma unroll
      for (int i = 0; i < N; ++i) u[i] = off;
      return;
    }
    const float r = __fdiv_rn(1.0f, s);
#pragma unroll
    for (int i = 0; i < N; ++i) {
      int c = __float2int_rn(__fmul_rn(x[i], r));
      c = min(max(c, -qmax), qmax);
      u[i] = (uint32_t)(c + off);
    }
    s_out = s;
  } else {
    constexpr int qm = (1 << BITS) - 1;
    float lo = 0.0f, hi = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      lo = fminf(lo, x[i]);
      hi = fmaxf(hi, x[i]);
    }
    const float span = __fsub_rn(hi, lo);
    const float s = bf16_round(__fdiv_rn(span, (float)qm));
    if (!(s >= FLT_MIN)) {
      s_out = 0.0f;
      z_out = 0;
#pragma unroll
      for (int i = 0; i < N; ++i) u[i] = 0;
      return;
    }
    const float r = __fdiv_rn(1.0f, s);
    const int z = min(max(__float2int_rn(__fmul_rn(-lo, r)), 0), qm);
#pragma unroll
    for (int i = 0; i < N; ++i) {
      int c = __float2int_rn(__fmul_rn(x[i], r)) + z;
      u[i] = (uint32_t)min(max(c, 0), qm);
    }
    s_out = s;
    z_out = z;
  }
}

// Per-token buffer quantizer ([P1] 어떻게 동작하나): one fp32 scale s = A/qmax for the vector,
// code = clamp(rint(x * (qmax/A)), -qmax, qmax); a zero (or subnormal) maximum gives zero codes.
__device__ __forceinline__ int buffer_code(float x, float A, int qmax) {
  if (!(A >= FLT_MIN)) return 0;
  const float r = __fdiv_rn((float)qmax, A);
  const int c = __float2int_rn(__fmul_rn(x, r));
  return min(max(c, -qmax), qmax);
}
__device__ __forceinline__ float buffer_scale(float A, int qmax) {
  if (!(A >= FLT_MIN)) return 0.0f;
  return __fdiv_rn(A, (float)qmax);
}

// Stored-code extraction from packed words (layouts in pace.h). An int4 word holds keys 8w..8w+7 of one
// column in order, key 8w+e in bits 4e..4e+3; masking with 0x0F0F0F0F leaves the even keys as bytes and
// 0xF0F0F0F0 the odd keys (times 16), the two planes the byte dot products use.
__device__ __forceinline__ int nibble_shift(int key_in_word) { return key_in_word << 2; }
__device__ __forceinline__ uint32_t nibble_of(uint32_t word, int key_in_word) {
  return (word >> nibble_shift(key_in_word)) & 0xFu;
}
// Pack 8 stored int4 codes (keys 0..7 of a word) / 4 stored int8 codes.
__device__ __forceinline__ uint32_t pack_nibbles(const uint32_t *u) {
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) w |= u[e] << nibble_shift(e);
  return w;
}
__device__ __forceinline__ uint32_t pack_bytes(const uint32_t *u) {
  return u[0] | (u[1] << 8) | (u[2] << 16) | (u[3] << 24);
}
__device__ __forceinline__ uint32_t byte_of(uint32_t word, int key_in_word) {
  return (word >> (key_in_word << 3)) & 0xFFu;
}

// Requantize one key-axis group of G values (the arithmetic of quant_group) and write its packed words
// to dst[0], dst[stride], ... as they are produced. Returns the bf16-exact scale and the zero point.
template <int G, int BITS>
__device__ __forceinline__ void quant_pack_group(const float (&x)[G], int zero_point, uint32_t *dst, int stride,
                                                 float &s_out, int &z_out) {
  constexpr int KPW = 32 / BITS;
  float s;
  int z;
  if (!zero_point) {
    constexpr int qmax = (1 << (BITS - 1)) - 1;
    float A = 0.0f;
#pragma unroll
    for (int i = 0; i < G; ++i) A = fmaxf(A, fabsf(x[i]));
    s = bf16_round(__fdiv_rn(A, (float)qmax));
    z = 1 << (BITS - 1);
    if (!(s >= FLT_MIN)) s = 0.0f;
  } else {
    constexpr int qm = (1 << BITS) - 1;
    float lo = 0.0f, hi = 0.0f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      lo = fminf(lo, x[i]);
      hi = fmaxf(hi, x[i]);
    }
    s = bf16_round(__fdiv_rn(__fsub_rn(hi, lo), (float)qm));
    z = 0;
    if (!(s >= FLT_MIN)) {
      s = 0.0f;
    } else {
      z = min(max(__float2int_rn(__fmul_rn(-lo, __fdiv_rn(1.0f, s))), 0), qm);
    }
  }
  const float r = s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
#pragma unroll
  for (int w = 0; w < G / KPW; ++w) {
    uint32_t u[KPW];
#pragma unroll
    for (int e = 0; e < KPW; ++e) {
      int c;
      if (s == 0.0f) {
        c = z;                                     // symmetric: the offset (code 0); zero point: 0
      } else if (!zero_point) {
        constexpr int qmax = (1 << (BITS - 1)) - 1;
        c = min(max(__float2int_rn(__fmul_rn(x[w * KPW + e], r)), -qmax), qmax) + z;
      } else {
        constexpr int qm = (1 << BITS) - 1;
        c = min(max(__float2int_rn(__fmul_rn(x[w * KPW + e], r)) + z, 0), qm);
      }
      u[e] = (uint32_t)c;
    }
    dst[(size_t)w * stride] = BITS == 4 ? pack_nibbles(u) : pack_bytes(u);
  }
  s_out = s;
  z_out = z;
}

}  // namespace pace
