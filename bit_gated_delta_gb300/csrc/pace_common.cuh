// Device helpers shared by the libpace kernels: I/O conversion, integer dot products, block
// reductions and the key-axis group quantizers.
#pragma once

#include <cuda_bf16.h>
#include <float.h>
#include <stdint.h>

#include <atomic>

#include "pace_internal.h"

namespace pace {

// ---- host-side launch set-up, per device: the library may drive several GPUs, from several host threads
constexpr int PACE_MAX_DEVICES = 64;
inline int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= PACE_MAX_DEVICES) d = 0;
  return d;
}
// SM count of the current device (queried once per device).
inline int device_sm_count() {
  static std::atomic<int> cache[PACE_MAX_DEVICES];
  const int dev = current_device();
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}
// Let kernel K use up to 227 KB of dynamic shared memory on the current device (once per kernel and device; a
// racing second caller repeats the idempotent attribute call).
template <auto K>
inline cudaError_t smem_opt_in(size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  if (bytes > 227 * 1024) return cudaErrorInvalidValue;
  static std::atomic<int> opted[PACE_MAX_DEVICES];
  const int dev = current_device();
  if (opted[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e == cudaSuccess) opted[dev].store(1, std::memory_order_release);
  return e;
}

// Blocks of kernel K (with `threads` threads and `smem` bytes of dynamic shared memory) resident per SM on the current
// device (queried once per kernel and device).
template <auto K>
inline int resident_blocks(int threads, size_t smem) {
  static std::atomic<int> cache[PACE_MAX_DEVICES];
  const int dev = current_device();
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, K, threads, smem) != cudaSuccess || v <= 0) v = 1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Sequential carving of a dynamic shared-memory block (16-byte aligned pieces, or `align`).
__host__ __device__ inline size_t carve(size_t &off, size_t bytes, size_t align = 16) {
  const size_t o = (off + align - 1) & ~(align - 1);
  off = o + bytes;
  return o;
}

// Programmatic dependent launch of the decode kernels: the next kernel of the stream may be scheduled as soon
// as every block of this one has started (its blocks take SMs as ours leave), and a kernel touches no global
// memory before every kernel it depends on has completed with its writes visible. Without the launch
// attribute both instructions are no-ops.
// Programmatic dependent launch in two halves: the trigger lets the next launch on the stream place its blocks, the
// wait holds until the previous launch has finished and its writes are visible.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Launch configuration with the programmatic-serialization attribute (attr must outlive the launch call).
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute *attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
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

// ---- Packed code layout (pace.h), in the order of the warp-level MMA fragments. Column j has
// mt = j/16, r8 = j%8, hi = (j/8)%2; key i has n = i/8, t = (i%8)/2, odd = i%2, p = n/4, r = n%4. Word
// (column j, lane r8*4+t, p) holds the keys 8n+2t, 8n+2t+1 of the four 8-key blocks n = 4p..4p+3: key
// 8n+2t in bits 4r..4r+3, key 8n+2t+1 in bits 16+4r..19+4r, so that (word >> 4r) & 0x000F000F is that
// pair in two 16-bit halves. Word index = ((mt*(D/64) + p/2)*32 + r8*4+t)*4 + hi*2 + p%2: one lane's
// four words of 64 keys are one 16-byte vector, and a warp reads 512 contiguous bytes per (mt, p/2).
// int8 codes are two such planes: plane 0 holds the low nibbles, plane 1 the high nibbles.
__host__ __device__ __forceinline__ uint32_t code_word(int D, int j, int i) {
  const int mt = j >> 4, r8 = j & 7, hi = (j >> 3) & 1, t = (i >> 1) & 3, p = i >> 5;
  return (uint32_t)((((mt * (D >> 6) + (p >> 1)) * 32 + r8 * 4 + t) << 2) + hi * 2 + (p & 1));
}
__host__ __device__ __forceinline__ uint32_t code_plane_words(int D) { return (uint32_t)(D * D / 8); }
__host__ __device__ __forceinline__ int nibble_shift(int i) { return (((i >> 3) & 3) << 2) | ((i & 1) << 4); }
// Stored code (unsigned) of key i of column j; BITS 4 or 8 (two nibble planes).
template <int BITS>
__device__ __forceinline__ uint32_t load_code(const uint32_t *unit_codes, int D, int j, int i) {
  const uint32_t wi = code_word(D, j, i);
  const int sh = nibble_shift(i);
  const uint32_t lo = (unit_codes[wi] >> sh) & 0xFu;
  if (BITS == 4) return lo;
  return lo | (((unit_codes[code_plane_words(D) + wi] >> sh) & 0xFu) << 4);
}

// Requantize one key-axis group of G values (keys g*G .. g*G+G-1 of column j) with the arithmetic of
// quant_group and store the packed codes of the group. Returns the bf16-exact scale and the zero point.
template <int G, int BITS>
__device__ __forceinline__ void quant_store_group(const float (&x)[G], int zero_point, uint32_t *unit_codes, int D,
                                                  int j, int g, float &s_out, int &z_out) {
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
  uint32_t u[G];
#pragma unroll
  for (int e = 0; e < G; ++e) {
    int c;
    if (s == 0.0f) {
      c = z;                                     // symmetric: the offset (code 0); zero point: 0
    } else if (!zero_point) {
      constexpr int qmax = (1 << (BITS - 1)) - 1;
      c = min(max(__float2int_rn(__fmul_rn(x[e], r)), -qmax), qmax) + z;
    } else {
      constexpr int qm = (1 << BITS) - 1;
      c = min(max(__float2int_rn(__fmul_rn(x[e], r)) + z, 0), qm);
    }
    u[e] = (uint32_t)c;
  }
  // the group covers whole words: G/32 spans of 32 keys, four words (t = 0..3) each
#pragma unroll
  for (int pw = 0; pw < G / 32; ++pw) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int e0 = pw * 32 + rr * 8 + 2 * t;      // key offset inside the group
        const int sh = 4 * rr;
        lo |= ((u[e0] & 0xFu) << sh) | ((u[e0 + 1] & 0xFu) << (16 + sh));
        hi |= (((u[e0] >> 4) & 0xFu) << sh) | (((u[e0 + 1] >> 4) & 0xFu) << (16 + sh));
      }
      const uint32_t wi = code_word(D, j, g * G + pw * 32 + 2 * t);
      unit_codes[wi] = lo;
      if (BITS == 8) unit_codes[code_plane_words(D) + wi] = hi;
    }
  }
  s_out = s;
  z_out = z;
}

}  // namespace pace
