// Chunked prefill ([P1] 어떻게 동작하나: the chunk kernel writes the state once per chunk, so PACE fixes
// the prefill rounding period to the 256-token chunk length).
//
// One CTA per unit, one thread per column j. The chunk-start state is decoded into shared memory as
// fp32, the n tokens of the chunk go through the gated delta rule token by token in fp32
// (S <- a S + k u^T, u = beta (v - (a S)^T k), o_t = S_t^T q_t), and the chunk-end state is rounded
// once: requantized with key-axis groups (thread-local per column), kept (fp32 mode) or rounded to
// bf16 (bf16 mode). Inputs are used as given, not buffered.
#include "pace_common.cuh"

namespace pace {

constexpr int PF_STAGE = 16;   // tokens staged in shared memory at a time

__host__ __device__ inline size_t prefill_smem_bytes(int D) {
  return (size_t)D * D * 4 + 2 * (size_t)PF_STAGE * D * 4 + 2 * PF_STAGE * 4;
}

// Resident codes of unit (b, h): int4 heads one plane, int8 heads two nibble planes (layout in pace.h).
template <int D, int BITS>
__device__ __forceinline__ uint32_t *unit_codes(const PaceDev &st, int b, int h) {
  return BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                   : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
}

// fp32 column j of the resident state into S_s[i][j].
template <int D, int G, int BITS>
__device__ void load_quant_column(const PaceDev &st, long unit, int b, int h, float *S_s) {
  constexpr int NG = D / G;
  const int j = threadIdx.x;
  const uint32_t *codes = unit_codes<D, BITS>(st, b, h);
#pragma unroll 1
  for (int g = 0; g < NG; ++g) {
    const float s = __bfloat162float(st.scale[(unit * NG + g) * D + j]);
    const int z = st.zero_point ? (int)st.zp[(unit * NG + g) * D + j] : (1 << (BITS - 1));
    for (int ii = 0; ii < G; ++ii) {
      const int i = g * G + ii;
      S_s[i * D + j] = s * (float)((int)load_code<BITS>(codes, D, j, i) - z);
    }
  }
}

// Round column j of S_s once and store it in the resident format.
template <int D, int G, int BITS>
__device__ void store_quant_column(const PaceDev &st, long unit, int b, int h, const float *S_s) {
  constexpr int NG = D / G;
  const int j = threadIdx.x;
  uint32_t *codes = unit_codes<D, BITS>(st, b, h);
#pragma unroll 1
  for (int g = 0; g < NG; ++g) {
    float x[G];
#pragma unroll
    for (int ii = 0; ii < G; ++ii) x[ii] = S_s[(g * G + ii) * D + j];
    float s;
    int z;
    quant_store_group<G, BITS>(x, st.zero_point, codes, D, j, g, s, z);
    st.scale[(unit * NG + g) * D + j] = __float2bfloat16_rn(s);
    if (st.zero_point) st.zp[(unit * NG + g) * D + j] = (uint8_t)z;
  }
}

template <int D, int G>
__global__ void __launch_bounds__(D) prefill_kernel(const PaceDev st, const PaceIO io) {
  extern __shared__ __align__(16) unsigned char smem[];
  float *S_s = reinterpret_cast<float *>(smem);
  float *k_s = S_s + D * D;
  float *q_s = k_s + PF_STAGE * D;
  float *a_s = q_s + PF_STAGE * D;
  float *b_s = a_s + PF_STAGE;
  const long unit = blockIdx.x;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int j = threadIdx.x;
  const int n = io.n;
  const int quant = st.state_mode == PACE_STATE_QUANT;
  const int is8 = st.head_is_int8[h];

  // chunk-start state
  if (quant) {
    if (is8) load_quant_column<D, G, 8>(st, unit, b, h, S_s);
    else load_quant_column<D, G, 4>(st, unit, b, h, S_s);
  } else if (st.state_mode == PACE_STATE_FP32) {
    const float *Sg = static_cast<const float *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) S_s[i * D + j] = Sg[i * D + j];
  } else {
    const __nv_bfloat16 *Sg = static_cast<const __nv_bfloat16 *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) S_s[i * D + j] = __bfloat162float(Sg[i * D + j]);
  }

  for (int t0 = 0; t0 < n; t0 += PF_STAGE) {
    const int nt = min(PF_STAGE, n - t0);
    __syncthreads();
    const long kunit = (unit / st.H) * st.Hk + (unit % st.H) / st.gamma;   // key head of this value head
    for (int tt = 0; tt < nt; ++tt) {
      const long row = (kunit * n + t0 + tt) * D + j;
      k_s[tt * D + j] = load_io(io.k, row, st.io);
      q_s[tt * D + j] = load_io(io.q, row, st.io);
    }
    if (j < nt) {
      a_s[j] = io.a[unit * n + t0 + j];
      b_s[j] = io.beta[unit * n + t0 + j];
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const float *kk = k_s + tt * D, *qq = q_s + tt * D;
      const float a = a_s[tt], beta = b_s[tt];
      const float v = load_io(io.v, (unit * n + t0 + tt) * D + j, st.io);
      float w = 0.0f;
      for (int i = 0; i < D; ++i) w = fmaf(S_s[i * D + j], kk[i], w);
      const float u = beta * (v - a * w);
      float o = 0.0f;
      for (int i = 0; i < D; ++i) {
        const float x = fmaf(a, S_s[i * D + j], kk[i] * u);
        S_s[i * D + j] = x;
        o = fmaf(x, qq[i], o);
      }
      store_io(io.o, (unit * n + t0 + tt) * D + j, o, st.io);
    }
  }

  // chunk-end rounding
  if (quant) {
    if (is8) store_quant_column<D, G, 8>(st, unit, b, h, S_s);
    else store_quant_column<D, G, 4>(st, unit, b, h, S_s);
  } else if (st.state_mode == PACE_STATE_FP32) {
    float *Sg = static_cast<float *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) Sg[i * D + j] = S_s[i * D + j];
  } else {
    __nv_bfloat16 *Sg = static_cast<__nv_bfloat16 *>(st.S) + unit * D * D;
    for (int i = 0; i < D; ++i) Sg[i * D + j] = __float2bfloat16_rn(S_s[i * D + j]);
  }
  if (j == 0) st.m[unit] = 0;
}

template <int D, int G>
static cudaError_t launch_prefill_t(const PaceDev &d, const PaceIO &io, cudaStream_t s) {
  const size_t smem = prefill_smem_bytes(D);
  auto kern = prefill_kernel<D, G>;
  const cudaError_t e = smem_opt_in<prefill_kernel<D, G>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0 || io.n == 0) return cudaSuccess;
  kern<<<units, D, smem, s>>>(d, io);
  return cudaGetLastError();
}

}  // namespace pace

cudaError_t pace_launch_prefill(const PaceDev &d, const PaceIO &io, cudaStream_t s) {
  using namespace pace;
  if (d.D == 128) return d.G == 64 ? launch_prefill_t<128, 64>(d, io, s) : launch_prefill_t<128, 32>(d, io, s);
  return d.G == 64 ? launch_prefill_t<64, 64>(d, io, s) : launch_prefill_t<64, 32>(d, io, s);
}
