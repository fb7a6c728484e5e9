// Chunked prefill on the 5th-generation tensor cores ([P1] 어떻게 동작하나: the chunk kernel writes the state
// once per chunk, so PACE rounds the prefill state once per 256-token chunk; [P2] 1. Key Terms & Definitions:
// the gated delta rule S_t = a_t S_{t-1} + k_t u_t^T, u_t = beta_t (v_t - (a_t S_{t-1})^T k_t)).
//
// One CTA of 128 threads per unit (sequence b, head h), d_k = d_v = 128, bf16 q/k/v/o. Thread j owns value
// column j, which is TMEM lane j of every accumulator. The fp32 state lives in TMEM as S^T (lane j, column i)
// for the whole chunk; it is rounded (or stored) once, at the end. The chunk is walked in sub-chunks of T = 32
// tokens. With G_t = a_0 .. a_t and R_{t,s} = a_{s+1} .. a_t inside a sub-chunk that starts from the state S:
//   w_t = S^T k_t,  p_t = S^T q_t                       (MMA: A = S^T as two bf16 parts, B = the k and q rows)
//   K_ts = k_s . k_t,  Q_ts = k_s . q_t                 (MMA: A = the k and q rows, B = the k rows)
//   u_t = beta_t (v_t - G_t w_t - sum_{s<t} R_ts K_ts u_s)        (per column, fp32, CUDA cores)
//   o_t = G_t p_t + sum_{s<=t} R_ts Q_ts u_s
//   S_end = G_T S + sum_t R_Tt k_t u_t^T                (MMA: A = (R_Tt u_t)^T as two bf16 parts, B = k^T)
// These equal the token-by-token rule exactly in real arithmetic (expand S_t = G_t S + sum_{s<=t} R_ts k_s u_s^T).
// k and q are bf16 and enter the MMAs exactly; the fp32 operands (S and the scaled u) are split into a bf16
// high part and a bf16 remainder, so every product carries about 16 significant bits and accumulates in fp32.
// Every mbarrier wait is bounded; on timeout the unit is left unchanged, the status word is set, and the
// kernel releases its TMEM and returns.
#include <cuda_bf16.h>

#include "pace_common.cuh"
#include "umma.cuh"

namespace pace {
using namespace umma;

namespace ptc {

constexpr int D = 128;           // d_k = d_v
constexpr int T = 32;            // tokens per sub-chunk
constexpr int NT = 128;          // threads
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_S = 0, COL_D1 = 128, COL_D2 = 192;   // S^T (128), [w | p] (64), [K | Q] Gram (32)

// Shared memory (bytes). X must be followed by at least 16 KB of shared memory: the Gram MMA reads 128 rows of
// X, of which rows 64-127 (ignored results) fall in the next region.
constexpr uint32_t OFF_X = 0;                      // [k_0..k_31 ; q_0..q_31] bf16, 64 x 128, K-major cores
constexpr uint32_t OFF_A = OFF_X + 64 * D * 2;     // S^T high / low parts, 2 x (128 x 128) bf16; later the
                                                   // update operands: (R u)^T parts 2 x (128 x 32), k^T 128 x 32
constexpr uint32_t A_PART = D * D * 2;
constexpr uint32_t OFF_A3 = OFF_A, A3_PART = D * T * 2, OFF_B3 = OFF_A + 2 * A3_PART;
constexpr uint32_t OFF_V = OFF_A + 2 * A_PART;     // v rows, bf16, T x 128 (row-major)
constexpr uint32_t OFF_WK = OFF_V + T * D * 2;     // R_ts K_ts, fp32 T x T (row t)
constexpr uint32_t OFF_WQ = OFF_WK + T * T * 4;    // R_ts Q_ts
constexpr uint32_t OFF_SC = OFF_WQ + T * T * 4;    // per token: a, beta, G_t, R_Tt (fp32 x 4T)
constexpr uint32_t OFF_BAR = OFF_SC + 4 * T * 4;   // mbarrier
constexpr uint32_t OFF_TB = OFF_BAR + 8;           // TMEM base address
constexpr uint32_t OFF_OK = OFF_TB + 4;            // 1 while every wait succeeded
constexpr uint32_t OFF_PROBE = OFF_OK + 4;         // mbarrier that nothing signals (failure-detection probe)
constexpr uint32_t SMEM = OFF_PROBE + 8;
static_assert(OFF_BAR % 8 == 0 && OFF_PROBE % 8 == 0, "mbarriers are 8-byte aligned");

// Byte offset of element (row r, k) in a K-major operand with kdim columns made of 8-row x 16-byte cores:
// cores adjacent along K (128 B apart), 8-row groups kdim/8 * 128 B apart.
__host__ __device__ constexpr uint32_t core_off(int r, int k, int kdim) {
  return (uint32_t)((r >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros (padding tokens).
__device__ __forceinline__ void cp16_zfill(void *dst_smem, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst_smem)),
               "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}
// x ~= hi + lo with hi = bf16(x), lo = bf16(x - hi), for a pair.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16(x0, x1);
  const float r0 = x0 - __uint_as_float(hi << 16), r1 = x1 - __uint_as_float(hi & 0xFFFF0000u);
  lo = pack_bf16(r0, r1);
}

// The 128 stored codes of column j, dequantized, as 16-value TMEM rows: s_g * (u - z).
template <int G, int BITS>
__device__ void load_quant_column(const PaceDev &st, long unit, int b, int h, int j, uint32_t taddr) {
  constexpr int NG = D / G;
  const uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                                    : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
  float s[NG];
  int z[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    s[g] = __bfloat162float(st.scale[(unit * NG + g) * D + j]);
    z[g] = st.zero_point ? (int)st.zp[(unit * NG + g) * D + j] : (1 << (BITS - 1));
  }
  // word (p, t) of column j holds keys 32p + 8r + 2t + e at bit 4r + 16e
#pragma unroll
  for (int p = 0; p < D / 32; ++p) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t wi = code_word(D, j, 32 * p + 2 * t);
      lo[t] = codes[wi];
      hi[t] = BITS == 8 ? codes[code_plane_words(D) + wi] : 0u;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {            // keys 32p + 16 half .. + 15
      uint32_t r[16];
#pragma unroll
      for (int e16 = 0; e16 < 16; ++e16) {
        const int kk = 16 * half + e16;                 // key offset inside the 32-key span: 8rr + 2t + e
        const int rr = kk >> 3, t = (kk >> 1) & 3, e = kk & 1;
        const int sh = 4 * rr + 16 * e;
        int u = (int)((lo[t] >> sh) & 0xFu);
        if (BITS == 8) u |= (int)((hi[t] >> sh) & 0xFu) << 4;
        const int g = (32 * p + kk) / G;
        r[e16] = __float_as_uint(s[g] * (float)(u - z[g]));
      }
      tmem_st16(taddr + 32 * p + 16 * half, r);
    }
  }
}

// Round column j (TMEM lane j) once and store it in the resident format.
template <int G, int BITS>
__device__ void store_quant_column(const PaceDev &st, long unit, int b, int h, int j, uint32_t taddr) {
  constexpr int NG = D / G;
  uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                              : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
#pragma unroll 1
  for (int g = 0; g < NG; ++g) {
    float x[G];
#pragma unroll
    for (int c = 0; c < G / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(taddr + g * G + 16 * c, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) x[16 * c + e] = __uint_as_float(r[e]);
    }
    float s;
    int z;
    quant_store_group<G, BITS>(x, st.zero_point, codes, D, j, g, s, z);
    st.scale[(unit * NG + g) * D + j] = __float2bfloat16_rn(s);
    if (st.zero_point) st.zp[(unit * NG + g) * D + j] = (uint8_t)z;
  }
}

}  // namespace ptc

template <int G>
__global__ void __launch_bounds__(ptc::NT, 1) prefill_tc_kernel(const PaceDev st, const PaceIO io) {
  using namespace ptc;
  extern __shared__ __align__(1024) unsigned char smem[];
  const long unit = blockIdx.x;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = tid;                                   // value column = TMEM lane
  const int n = io.n;
  const int quant = st.state_mode == PACE_STATE_QUANT;
  const int is8 = st.head_is_int8[h];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint32_t *tbase = reinterpret_cast<uint32_t *>(smem + OFF_TB);
  volatile int *okf = reinterpret_cast<volatile int *>(smem + OFF_OK);
  float *sc = reinterpret_cast<float *>(smem + OFF_SC);   // [0,T) a, [T,2T) beta, [2T,3T) G_t, [3T,4T) R_Tt
  const uint32_t sbase = smem_u32(smem);
  const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(io.q);
  const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(io.k);
  const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(io.v);
  __nv_bfloat16 *go = static_cast<__nv_bfloat16 *>(io.o);

  if (warp == 0) {
    tmem_alloc(tbase, TMEM_COLS);
    tmem_relinquish();
  }
  uint64_t *probe = reinterpret_cast<uint64_t *>(smem + OFF_PROBE);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(probe, 1);
    mbar_fence_init();
    *okf = 1;
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tbase;
  const uint32_t lanes = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem + lanes + COL_S;
  uint32_t phase = 0;

  // ---- chunk-start state S^T into TMEM (lane j = column j of S)
  if (quant) {
    if (is8) load_quant_column<G, 8>(st, unit, b, h, j, tS);
    else load_quant_column<G, 4>(st, unit, b, h, j, tS);
  } else {
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const long idx = (unit * D + 16 * c + e) * D + j;
        r[e] = __float_as_uint(st.state_mode == PACE_STATE_FP32 ? static_cast<const float *>(st.S)[idx]
                                                                : __bfloat162float(static_cast<const __nv_bfloat16 *>(st.S)[idx]));
      }
      tmem_st16(tS + 16 * c, r);
    }
  }
  tmem_wait_st();

  // the k, q rows (K-major cores) and v rows of the sub-chunk starting at token s0, as asynchronous copies;
  // padding tokens (s0 + t >= n) are zeros
  const long kunit = (unit / st.H) * st.Hk + (unit % st.H) / st.gamma;   // key head of this value head
  auto issue_rows = [&](int s0) {
    const int ns = min(T, n - s0);
#pragma unroll
    for (int it = 0; it < 8; ++it) {                    // 64 rows x 16 chunks of 16 bytes
      const int c = tid + NT * it, row = c >> 4, c8 = c & 15, t = row & (T - 1);
      const bool in = t < ns;
      const __nv_bfloat16 *src = (row < T ? gk : gq) + ((kunit * n + s0 + (in ? t : 0)) * D + 8 * c8);
      cp16_zfill(smem + OFF_X + core_off(row, 8 * c8, D), src, in ? 16u : 0u);
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {                    // 32 rows x 16 chunks
      const int c = tid + NT * it, t = c >> 4, c8 = c & 15;
      const bool in = t < ns;
      cp16_zfill(smem + OFF_V + (t * D + 8 * c8) * 2, gv + ((unit * n + s0 + (in ? t : 0)) * D + 8 * c8), in ? 16u : 0u);
    }
  };
  if (n > 0) issue_rows(0);

  bool ok = true;
  bool drain = false;                                   // an MMA group whose wait gave up is still in flight
  uint32_t pending = 0;                                 // its phase parity
  if (st.probe_ns) {                                    // failure-detection probe: a wait that runs out, no MMA issued
    if (tid == 0 && !mbar_wait(probe, 0, st.probe_ns)) *okf = 0;
    __syncthreads();
    if (!*okf) ok = false;
  }
#pragma unroll 1
  for (int t0 = 0; t0 < n && ok; t0 += T) {
    const int nt = min(T, n - t0);
    // ---- (a) the sub-chunk's rows (in flight since the previous sub-chunk's update), a and beta; padding tokens
    // are a = 1, beta = 0, k = q = v = 0, which leave the state unchanged.
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (warp == 0) {
      const float a = lane < nt ? io.a[unit * n + t0 + lane] : 1.0f;
      const float be = lane < nt ? io.beta[unit * n + t0 + lane] : 0.0f;
      float g = 1.0f, rho = 1.0f;                       // G_t = a_0..a_t ; R_Tt = a_{t+1}..a_{T-1}
#pragma unroll
      for (int r = 0; r < T; ++r) {
        const float ar = __shfl_sync(0xffffffffu, a, r);
        if (r <= lane) g *= ar;
        else rho *= ar;
      }
      sc[lane] = a;
      sc[T + lane] = be;
      sc[2 * T + lane] = g;
      sc[3 * T + lane] = rho;
    }
    __syncthreads();
    const float gT = sc[2 * T + T - 1];

    // ---- (c) S^T -> two bf16 parts (A of the dot MMA), and S <- G_T S in place for the update MMA
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(tS + 16 * c, r);
      tmem_wait_ld();
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) split2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]), hi[e], lo[e]);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {                  // keys 16c + 8hh .. +7
        const uint32_t off = core_off(j, 16 * c + 8 * hh, D);
        *reinterpret_cast<uint4 *>(smem + OFF_A + off) = make_uint4(hi[4 * hh], hi[4 * hh + 1], hi[4 * hh + 2], hi[4 * hh + 3]);
        *reinterpret_cast<uint4 *>(smem + OFF_A + A_PART + off) =
            make_uint4(lo[4 * hh], lo[4 * hh + 1], lo[4 * hh + 2], lo[4 * hh + 3]);
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(gT * __uint_as_float(r[e]));
      tmem_st16(tS + 16 * c, r);
    }
    tmem_wait_st();
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();

    // ---- (e) dots [w | p] = S^T [k | q]^T and the Gram products [K | Q] = [k | q] k^T
    if (tid == 0) {
      fence_after_sync();
      const uint32_t xb = sbase + OFF_X, ab = sbase + OFF_A;
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + COL_D1, smem_desc(ab + part * A_PART + kk * 256, 128, (D / 8) * 128),
                 smem_desc(xb + kk * 256, 128, (D / 8) * 128), idesc_bf16(128, 2 * T), (part | kk) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + COL_D2, smem_desc(xb + kk * 256, 128, (D / 8) * 128), smem_desc(xb + kk * 256, 128, (D / 8) * 128),
               idesc_bf16(128, T), kk ? 1u : 0u);
      commit(bar);
      if (!mbar_wait(bar, phase, WAIT_NS)) *okf = 0;
    }
    __syncthreads();
    phase ^= 1u;
    if (!*okf) {
      ok = false;
      pending = phase ^ 1u;
      drain = true;
      break;
    }
    fence_after_sync();

    // ---- (f) coefficient tables from the Gram rows: thread r < T is k_r, T <= r < 2T is q_{r-T}
    if (warp < 2) {
      const int t = tid & (T - 1), isq = tid >= T;
      uint32_t d0[16], d1[16];
      tmem_ld16(tmem + lanes + COL_D2, d0);
      tmem_ld16(tmem + lanes + COL_D2 + 16, d1);
      tmem_wait_ld();
      float out[T];
      float Rr = 1.0f;
#pragma unroll
      for (int s = T - 1; s >= 0; --s) {
        if (s < t) Rr *= sc[s + 1];                     // R_{t,s} = a_{s+1} .. a_t
        const float d = __uint_as_float(s < 16 ? d0[s] : d1[s - 16]);
        out[s] = (s < t || (isq && s == t)) ? Rr * d : 0.0f;
      }
      // stored transposed, [s][t]: the recurrence sweeps by s and reads row s four tokens per load
      float *tab = reinterpret_cast<float *>(smem + (isq ? OFF_WQ : OFF_WK));
#pragma unroll
      for (int s = 0; s < T; ++s) tab[s * T + t] = out[s];
    }
    float w[T], p[T];
    {
      uint32_t r[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld16(tmem + lanes + COL_D1 + 16 * c, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          if (c < 2) w[16 * c + e] = __uint_as_float(r[e]);
          else p[16 * (c - 2) + e] = __uint_as_float(r[e]);
        }
      }
    }
    __syncthreads();

    // ---- (h) the per-column recurrence and the outputs, swept by s (right-looking): once u_s is known it is
    // subtracted from every later token's residual R_t and added to every output O_t with t >= s, so the
    // dependent chain per token is one multiply-add and one multiply; the other updates are independent.
    float u[T];
    {
      const float *wkT = reinterpret_cast<const float *>(smem + OFF_WK);    // [s][t] = R_ts K_ts (t > s)
      const float *wqT = reinterpret_cast<const float *>(smem + OFF_WQ);    // [s][t] = R_ts Q_ts (t >= s)
      const __nv_bfloat16 *vs = reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_V);
      float *R = w, *O = p;                             // in place: R_t = v_t - G_t w_t, O_t = G_t p_t
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float gt = sc[2 * T + t];
        R[t] = fmaf(-gt, w[t], __bfloat162float(vs[t * D + j]));
        O[t] = gt * p[t];
      }
#pragma unroll
      for (int s = 0; s < T; ++s) {
        u[s] = sc[T + s] * R[s];
#pragma unroll
        for (int t4 = (s + 1) & ~3; t4 < T; t4 += 4) {
          const float4 c = *reinterpret_cast<const float4 *>(wkT + s * T + t4);
          if (t4 + 0 > s) R[t4 + 0] = fmaf(-c.x, u[s], R[t4 + 0]);
          if (t4 + 1 > s) R[t4 + 1] = fmaf(-c.y, u[s], R[t4 + 1]);
          if (t4 + 2 > s) R[t4 + 2] = fmaf(-c.z, u[s], R[t4 + 2]);
          if (t4 + 3 > s) R[t4 + 3] = fmaf(-c.w, u[s], R[t4 + 3]);
        }
#pragma unroll
        for (int t4 = s & ~3; t4 < T; t4 += 4) {
          const float4 c = *reinterpret_cast<const float4 *>(wqT + s * T + t4);
          if (t4 + 0 >= s) O[t4 + 0] = fmaf(c.x, u[s], O[t4 + 0]);
          if (t4 + 1 >= s) O[t4 + 1] = fmaf(c.y, u[s], O[t4 + 1]);
          if (t4 + 2 >= s) O[t4 + 2] = fmaf(c.z, u[s], O[t4 + 2]);
          if (t4 + 3 >= s) O[t4 + 3] = fmaf(c.w, u[s], O[t4 + 3]);
        }
      }
#pragma unroll
      for (int t = 0; t < T; ++t)
        if (t < nt) go[(unit * n + t0 + t) * D + j] = __float2bfloat16_rn(O[t]);
    }

    // ---- (i) update operands: (R_Tt u_t)^T parts (row j, K = tokens) and k^T (row i = tid, K = tokens)
#pragma unroll
    for (int t8 = 0; t8 < T; t8 += 8) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        split2(sc[3 * T + t8 + 2 * e] * u[t8 + 2 * e], sc[3 * T + t8 + 2 * e + 1] * u[t8 + 2 * e + 1], hi[e], lo[e]);
      const uint32_t off = core_off(j, t8, T);
      *reinterpret_cast<uint4 *>(smem + OFF_A3 + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4 *>(smem + OFF_A3 + A3_PART + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    {
      const int i = tid;
#pragma unroll
      for (int t8 = 0; t8 < T; t8 += 8) {
        uint32_t kw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t k0 = *reinterpret_cast<const uint16_t *>(smem + OFF_X + core_off(t8 + 2 * e, i, D));
          const uint32_t k1 = *reinterpret_cast<const uint16_t *>(smem + OFF_X + core_off(t8 + 2 * e + 1, i, D));
          kw[e] = k0 | (k1 << 16);
        }
        *reinterpret_cast<uint4 *>(smem + OFF_B3 + core_off(i, t8, T)) = make_uint4(kw[0], kw[1], kw[2], kw[3]);
      }
    }
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
    if (t0 + T < n) issue_rows(t0 + T);                 // the rows and keys of this sub-chunk are done with

    // ---- (j) S^T += (R u)^T k : M = columns, N = keys, K = tokens
    if (tid == 0) {
      fence_after_sync();
      const uint32_t a3 = sbase + OFF_A3, b3 = sbase + OFF_B3;
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < T / 16; ++kk)
          mma_ss(tmem + COL_S, smem_desc(a3 + part * A3_PART + kk * 256, 128, (T / 8) * 128),
                 smem_desc(b3 + kk * 256, 128, (T / 8) * 128), idesc_bf16(128, D), 1u);
      commit(bar);
      if (!mbar_wait(bar, phase, WAIT_NS)) *okf = 0;
    }
    __syncthreads();
    phase ^= 1u;
    if (!*okf) {
      ok = false;
      pending = phase ^ 1u;
      drain = true;
    }
    fence_after_sync();
  }

  if (ok) {
    // ---- chunk-end rounding (or store) of column j
    if (quant) {
      if (is8) store_quant_column<G, 8>(st, unit, b, h, j, tS);
      else store_quant_column<G, 4>(st, unit, b, h, j, tS);
    } else {
#pragma unroll 1
      for (int c = 0; c < D / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tS + 16 * c, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const long idx = (unit * D + 16 * c + e) * D + j;
          const float x = __uint_as_float(r[e]);
          if (st.state_mode == PACE_STATE_FP32) static_cast<float *>(st.S)[idx] = x;
          else static_cast<__nv_bfloat16 *>(st.S)[idx] = __float2bfloat16_rn(x);
        }
      }
    }
    if (j == 0) st.m[unit] = 0;
  } else if (tid == 0) {
    atomicOr(st.status, 1);
    if (drain) mbar_wait(bar, pending, WAIT_NS);        // let the MMAs in flight drain before TMEM is released
  }
  asm volatile("cp.async.wait_all;" ::: "memory");      // no copy may land after the CTA leaves
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

template <int G>
static cudaError_t launch_prefill_tc_t(const PaceDev &d, const PaceIO &io, cudaStream_t s) {
  const cudaError_t e = smem_opt_in<prefill_tc_kernel<G>>(ptc::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0 || io.n == 0) return cudaSuccess;
  prefill_tc_kernel<G><<<units, ptc::NT, ptc::SMEM, s>>>(d, io);
  return cudaGetLastError();
}

}  // namespace pace

// d_k = d_v = 128 with bf16 I/O runs the tensor-core chunk kernel; other shapes use the per-token kernel.
bool pace_prefill_tc_supported(const PaceDev &d) { return d.D == 128 && d.io == PACE_IO_BF16; }

cudaError_t pace_launch_prefill_tc(const PaceDev &d, const PaceIO &io, cudaStream_t s) {
  using namespace pace;
  return d.G == 64 ? launch_prefill_tc_t<64>(d, io, s) : launch_prefill_tc_t<32>(d, io, s);
}
