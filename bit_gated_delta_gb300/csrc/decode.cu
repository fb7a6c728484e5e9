// PACE decode step and flush ([P1] 어떻게 동작하나; [P2] 1. Key Terms & Definitions).
//
// One CTA per unit (sequence b, head h), one thread per state column j (value channel). Per call:
//   1. the buffered tokens 0..m-1 and (decode) the new token, quantized into slot m, are staged in
//      shared memory as int8 key codes, fp32 values and per-token scalars;
//   2. thread j reads its column's packed codes (int4 or int8) once, and forms the dot products
//      (S_hat^T k_tau)_j for every buffered key and (S_hat^T q)_j with dp4a on the integer codes:
//      codes x int8 keys are exact integers; q enters as a 16-bit fixed-point image split in two
//      int8 halves. Group scales and zero points are applied per group afterwards;
//   3. the buffered tokens are replayed through the gated delta rule in the reduced per-column form
//        u_t = beta_t (v_t - G_t (S_hat^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),  G_t = a_1..a_t,
//        o   = G_m (S_hat^T q) + sum_s (G_m/G_s)(k_s.q) u_s,
//      which is S_t = a_t S_{t-1} + k_t u_t^T applied m times to S_hat, without the d_k x d_v updates;
//   4. when the buffer holds dP tokens (or on an explicit flush) the column is rebuilt,
//        S_new = G_m S_hat + sum_s (G_m/G_s) k_s u_s^T,
//      requantized with its own key-axis groups (thread-local absmax / min-max), packed and stored.
#include <algorithm>

#include "pace_common.cuh"

namespace pace {

constexpr int VCHUNK = 8;   // dot-product vectors handled per pass over the codes

__host__ __device__ inline size_t carve(size_t &off, size_t bytes) {
  const size_t o = (off + 15) & ~size_t(15);
  off = o + bytes;
  return o;
}

struct DecodeSmem {
  size_t kq, keyf, vf, P, U, kf, csum, vscale, a, beta, gam, Dm, W, cq, ck, red, qf, total;
};

__host__ __device__ inline DecodeSmem decode_smem(int D, int dP, int fp32mode) {
  DecodeSmem L;
  size_t off = 0;
  L.kq = carve(off, (size_t)(dP + 2) * D);                     // int8 key codes (+ q halves)
  L.keyf = carve(off, fp32mode ? (size_t)(dP + 1) * D * 4 : 0); // fp32 keys (+ q), fp32 mode
  L.vf = carve(off, (size_t)dP * D * 4);                       // dequantized values
  L.P = carve(off, (size_t)(dP + 2) * D * 4);                  // S_hat^T k_tau, S_hat^T q
  L.U = carve(off, (size_t)dP * D * 4);                        // u_tau per column
  L.kf = carve(off, (size_t)dP * D * 4);                       // flush coefficients x keys
  L.csum = carve(off, (size_t)(dP + 2) * 4 * 4);               // per vector, per group code sums
  L.vscale = carve(off, (size_t)(dP + 2) * 4);
  L.a = carve(off, (size_t)dP * 4);
  L.beta = carve(off, (size_t)dP * 4);
  L.gam = carve(off, (size_t)dP * 4);
  L.Dm = carve(off, (size_t)dP * dP * 4);                      // Dm[s][t] = a_{s+1} .. a_t
  L.W = carve(off, (size_t)dP * dP * 4);                       // W[t][s] = Dm[s][t] k_s.k_t
  L.cq = carve(off, (size_t)dP * 4);
  L.ck = carve(off, (size_t)dP * 4);
  L.red = carve(off, 32 * 4);
  L.qf = carve(off, (size_t)D * 4);
  L.total = carve(off, 0);
  return L;
}

struct DecodeShared {
  int8_t *kq;
  float *keyf, *vf, *P, *U, *kf;
  int *csum;
  float *vscale, *a, *beta, *gam, *Dm, *W, *cq, *ck, *red, *qf;
};

__device__ inline DecodeShared decode_shared(unsigned char *base, const DecodeSmem &L) {
  DecodeShared s;
  s.kq = reinterpret_cast<int8_t *>(base + L.kq);
  s.keyf = reinterpret_cast<float *>(base + L.keyf);
  s.vf = reinterpret_cast<float *>(base + L.vf);
  s.P = reinterpret_cast<float *>(base + L.P);
  s.U = reinterpret_cast<float *>(base + L.U);
  s.kf = reinterpret_cast<float *>(base + L.kf);
  s.csum = reinterpret_cast<int *>(base + L.csum);
  s.vscale = reinterpret_cast<float *>(base + L.vscale);
  s.a = reinterpret_cast<float *>(base + L.a);
  s.beta = reinterpret_cast<float *>(base + L.beta);
  s.gam = reinterpret_cast<float *>(base + L.gam);
  s.Dm = reinterpret_cast<float *>(base + L.Dm);
  s.W = reinterpret_cast<float *>(base + L.W);
  s.cq = reinterpret_cast<float *>(base + L.cq);
  s.ck = reinterpret_cast<float *>(base + L.ck);
  s.red = reinterpret_cast<float *>(base + L.red);
  s.qf = reinterpret_cast<float *>(base + L.qf);
  return s;
}

// Stage buffered tokens 0..m0-1 of one unit into shared memory.
template <int D>
__device__ void load_buffer(const PaceDev &st, long unit, int m0, const DecodeShared &sh) {
  const int j = threadIdx.x;
  const int dP = st.dP;
  const float *bs = st.buf_s + unit * dP * 4;
  if (j < m0) {
    sh.a[j] = bs[j * 4 + 0];
    sh.beta[j] = bs[j * 4 + 1];
    sh.vscale[j] = bs[j * 4 + 2];
  }
  if (st.buf_mode == PACE_BUF_INT8) {
    const int8_t *bk = static_cast<const int8_t *>(st.buf_k) + unit * dP * D;
    const int8_t *bv = static_cast<const int8_t *>(st.buf_v) + unit * dP * D;
    for (int t = 0; t < m0; ++t) {
      sh.kq[t * D + j] = bk[t * D + j];
      sh.vf[t * D + j] = bs[t * 4 + 3] * (float)bv[t * D + j];
    }
  } else if (st.buf_mode == PACE_BUF_MIXED) {
    const uint8_t *bk = static_cast<const uint8_t *>(st.buf_k) + unit * dP * (D / 2);
    const __nv_bfloat16 *bv = static_cast<const __nv_bfloat16 *>(st.buf_v) + unit * dP * D;
    for (int t = 0; t < m0; ++t) {
      const uint32_t byte = bk[t * (D / 2) + (j >> 1)];
      sh.kq[t * D + j] = (int8_t)((int)((byte >> ((j & 1) * 4)) & 0xF) - 8);
      sh.vf[t * D + j] = __bfloat162float(bv[t * D + j]);
    }
  } else {
    const float *bk = static_cast<const float *>(st.buf_k) + unit * dP * D;
    const float *bv = static_cast<const float *>(st.buf_v) + unit * dP * D;
    for (int t = 0; t < m0; ++t) {
      sh.keyf[t * D + j] = bk[t * D + j];
      sh.vf[t * D + j] = bv[t * D + j];
    }
  }
}

// Quantize the new token into buffer slot m0 (shared and global), and stage q.
template <int D>
__device__ void append_token(const PaceDev &st, const PaceIO &io, long unit, int m0, const DecodeShared &sh) {
  const int j = threadIdx.x;
  const int dP = st.dP;
  const float kx = load_io(io.k, unit * D + j, st.io);
  const float vx = load_io(io.v, unit * D + j, st.io);
  const float qx = load_io(io.q, unit * D + j, st.io);
  sh.qf[j] = qx;
  float sk = 1.0f, sv = 1.0f;
  if (st.buf_mode == PACE_BUF_INT8) {
    const float Ak = block_max(fabsf(kx), sh.red);
    const float Av = block_max(fabsf(vx), sh.red);
    const int ck = buffer_code(kx, Ak, 127), cv = buffer_code(vx, Av, 127);
    sk = buffer_scale(Ak, 127);
    sv = buffer_scale(Av, 127);
    sh.kq[m0 * D + j] = (int8_t)ck;
    sh.vf[m0 * D + j] = sv * (float)cv;
    static_cast<int8_t *>(st.buf_k)[(unit * dP + m0) * D + j] = (int8_t)ck;
    static_cast<int8_t *>(st.buf_v)[(unit * dP + m0) * D + j] = (int8_t)cv;
  } else if (st.buf_mode == PACE_BUF_MIXED) {
    const float Ak = block_max(fabsf(kx), sh.red);
    const int ck = buffer_code(kx, Ak, 7);
    sk = buffer_scale(Ak, 7);
    const float vb = bf16_round(vx);
    sh.kq[m0 * D + j] = (int8_t)ck;
    sh.vf[m0 * D + j] = vb;
    const int nb = __shfl_down_sync(0xffffffffu, ck, 1);
    if ((j & 1) == 0)
      static_cast<uint8_t *>(st.buf_k)[(unit * dP + m0) * (D / 2) + (j >> 1)] =
          (uint8_t)((ck + 8) | ((nb + 8) << 4));
    static_cast<__nv_bfloat16 *>(st.buf_v)[(unit * dP + m0) * D + j] = __float2bfloat16_rn(vx);
  } else {
    sh.keyf[m0 * D + j] = kx;
    sh.vf[m0 * D + j] = vx;
    static_cast<float *>(st.buf_k)[(unit * dP + m0) * D + j] = kx;
    static_cast<float *>(st.buf_v)[(unit * dP + m0) * D + j] = vx;
  }
  if (j == 0) {
    const float ax = io.a[unit], bx = io.beta[unit];
    sh.a[m0] = ax;
    sh.beta[m0] = bx;
    sh.vscale[m0] = sk;
    float *bs = st.buf_s + (unit * dP + m0) * 4;
    bs[0] = ax;
    bs[1] = bx;
    bs[2] = sk;
    bs[3] = sv;
  }
  if (st.state_mode == PACE_STATE_FP32) {
    sh.keyf[(m0 + 1) * D + j] = qx;          // q follows the keys
  } else {
    // 16-bit fixed-point image of q: q ~= sigma * (256 hi + lo), |256 hi + lo| <= 32512
    const float Aq = block_max(fabsf(qx), sh.red);
    int hi = 0, lo = 0;
    float sigma = 0.0f;
    if (Aq >= FLT_MIN) {
      sigma = Aq / 32512.0f;
      int qi = __float2int_rn(qx * (32512.0f / Aq));
      qi = min(max(qi, -32512), 32512);
      hi = (qi + 128) >> 8;
      lo = qi - (hi << 8);
    }
    const int mt = m0 + 1;
    sh.kq[mt * D + j] = (int8_t)hi;
    sh.kq[(mt + 1) * D + j] = (int8_t)lo;
    if (j == 0) {
      sh.vscale[mt] = 256.0f * sigma;
      sh.vscale[mt + 1] = sigma;
    }
  }
}

// Per-vector group sums of the int8 key codes (for the zero-offset correction of the dot products).
template <int D, int G>
__device__ void code_sums(int nv, const DecodeShared &sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = D / 32;
  for (int v = wid; v < nv; v += nw) {
    int gs[D / G];
#pragma unroll
    for (int g = 0; g < D / G; ++g) gs[g] = 0;
#pragma unroll
    for (int r = 0; r < D / 32; ++r) {
      const int x = sh.kq[v * D + r * 32 + lane];
      gs[(r * 32) / G] += __reduce_add_sync(0xffffffffu, x);
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < D / G; ++g) sh.csum[v * 4 + g] = gs[g];
    }
  }
}

// Decay products, Gram coefficients, readout and flush coefficients shared by all columns.
template <int D>
__device__ void unit_tables(int mt, int has_token, int fp32mode, int dP, const DecodeShared &sh) {
  const int j = threadIdx.x, lane = j & 31, wid = j >> 5, nw = D / 32;
  if (j < mt) {                                   // row j of Dm: a_{j+1} .. a_t
    float p = 1.0f;
    sh.Dm[j * dP + j] = 1.0f;
    for (int t = j + 1; t < mt; ++t) {
      p *= sh.a[t];
      sh.Dm[j * dP + t] = p;
    }
  }
  if (j == 0) {
    float p = 1.0f;
    for (int t = 0; t < mt; ++t) {
      p *= sh.a[t];
      sh.gam[t] = p;
    }
  }
  __syncthreads();
  // Gram k_s . k_t (s < t) and, with a token, k_s . q
  int item = 0;
  for (int t = 1; t < mt; ++t) {
    for (int s = 0; s < t; ++s, ++item) {
      if (item % nw != wid) continue;
      float dot;
      if (fp32mode) {
        float acc = 0.0f;
#pragma unroll
        for (int r = 0; r < D / 32; ++r) acc += sh.keyf[s * D + r * 32 + lane] * sh.keyf[t * D + r * 32 + lane];
        dot = warp_sum(acc);
      } else {
        int acc = 0;
        if (lane < D / 4) {
          const int *ks = reinterpret_cast<const int *>(sh.kq + s * D);
          const int *kt = reinterpret_cast<const int *>(sh.kq + t * D);
          acc = dp4a_ss(ks[lane], kt[lane], 0);
        }
        dot = sh.vscale[s] * sh.vscale[t] * (float)__reduce_add_sync(0xffffffffu, acc);
      }
      if (lane == 0) sh.W[t * dP + s] = sh.Dm[s * dP + t] * dot;
    }
  }
  for (int s = wid; s < mt; s += nw) {
    float acc = 0.0f;
    if (has_token) {
#pragma unroll
      for (int r = 0; r < D / 32; ++r) {
        const int i = r * 32 + lane;
        const float kv = fp32mode ? sh.keyf[s * D + i] : (float)sh.kq[s * D + i];
        acc += kv * sh.qf[i];
      }
      acc = warp_sum(acc);
    }
    if (lane == 0) {
      const float ks = fp32mode ? 1.0f : sh.vscale[s];
      sh.cq[s] = sh.Dm[s * dP + (mt - 1)] * ks * acc;
      sh.ck[s] = sh.Dm[s * dP + (mt - 1)] * ks;
    }
  }
}

// Per-column replay of the buffered tokens (reduced form) and the readout o_j.
template <int D>
__device__ void recurrence(const PaceDev &st, const PaceIO &io, long unit, int nv, int mt, int has_token,
                           int fp32mode, const DecodeShared &sh) {
  const int j = threadIdx.x;
  const int dP = st.dP;
  for (int t = 0; t < mt; ++t) {
    float acc = sh.vf[t * D + j] - sh.gam[t] * sh.P[t * D + j];
    for (int s = 0; s < t; ++s) acc = fmaf(-sh.W[t * dP + s], sh.U[s * D + j], acc);
    sh.U[t * D + j] = sh.beta[t] * acc;
  }
  if (has_token) {
    const float R = fp32mode ? sh.P[mt * D + j] : sh.P[mt * D + j] + sh.P[(mt + 1) * D + j];
    float o = sh.gam[mt - 1] * R;
    for (int s = 0; s < mt; ++s) o = fmaf(sh.cq[s], sh.U[s * D + j], o);
    store_io(io.o, unit * D + j, o, st.io);
  }
  (void)nv;
}

// kf[s][i] = (G_m / G_s) k_s,i : coefficients of the rank-m flush update (thread j fills key j).
template <int D>
__device__ void flush_coeffs(int mt, int fp32mode, const DecodeShared &sh) {
  const int i = threadIdx.x;
  for (int s = 0; s < mt; ++s)
    sh.kf[s * D + i] = sh.ck[s] * (fp32mode ? sh.keyf[s * D + i] : (float)sh.kq[s * D + i]);
}

// Dot products of the packed column with every staged vector, then flush of the column.
template <int D, int G, int BITS>
__device__ void quant_column(const PaceDev &st, const PaceIO &io, long unit, int b, int h, int nv, int mt,
                             int has_token, int do_flush, const DecodeShared &sh) {
  constexpr int KPW = 32 / BITS;           // keys per 32-bit word
  constexpr int NWC = D / KPW;             // words per column
  constexpr int NG = D / G;
  constexpr int WPG = G / KPW;             // words per group
  const int j = threadIdx.x;
  const int slot = st.head_slot[h];
  uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + slot) * NWC * D
                              : st.codes8 + (size_t)(b * st.H8 + slot) * NWC * D;
  uint32_t wr[NWC];
#pragma unroll
  for (int w = 0; w < NWC; ++w) wr[w] = codes[w * D + j];
  float sg[NG];
  int zg[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    sg[g] = __bfloat162float(st.scale[(unit * NG + g) * D + j]);
    zg[g] = st.zero_point ? (int)st.zp[(unit * NG + g) * D + j] : (1 << (BITS - 1));
  }
  // ---- dot products: P[v][j] = vscale[v] * sum_g s_g (sum_i u_i c_v,i - z_g sum_i c_v,i)
  for (int c0 = 0; c0 < nv; c0 += VCHUNK) {
    float pf[VCHUNK];
#pragma unroll
    for (int t = 0; t < VCHUNK; ++t) pf[t] = 0.0f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      int acc[VCHUNK], acc16[VCHUNK];
#pragma unroll
      for (int t = 0; t < VCHUNK; ++t) acc[t] = acc16[t] = 0;
#pragma unroll
      for (int ww = 0; ww < WPG; ++ww) {
        const int w = g * WPG + ww;
        if (BITS == 4) {
          const uint32_t lo = wr[w] & 0x0F0F0F0Fu, hi = wr[w] & 0xF0F0F0F0u;
#pragma unroll
          for (int t = 0; t < VCHUNK; ++t) {
            if (c0 + t < nv) {
              const int2 kk = *reinterpret_cast<const int2 *>(sh.kq + (c0 + t) * D + 8 * w);
              acc[t] = dp4a_us(lo, kk.x, acc[t]);
              acc16[t] = dp4a_us(hi, kk.y, acc16[t]);
            }
          }
        } else {
#pragma unroll
          for (int t = 0; t < VCHUNK; ++t) {
            if (c0 + t < nv) {
              const int kk = *reinterpret_cast<const int *>(sh.kq + (c0 + t) * D + 4 * w);
              acc[t] = dp4a_us(wr[w], kk, acc[t]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < VCHUNK; ++t) {
        if (c0 + t < nv) {
          const int tot = acc[t] + (acc16[t] >> 4) - zg[g] * sh.csum[(c0 + t) * 4 + g];
          pf[t] = fmaf(sg[g], (float)tot, pf[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < VCHUNK; ++t)
      if (c0 + t < nv) sh.P[(c0 + t) * D + j] = pf[t] * sh.vscale[c0 + t];
  }
  recurrence<D>(st, io, unit, nv, mt, has_token, 0, sh);
  if (!do_flush) return;
  flush_coeffs<D>(mt, 0, sh);
  __syncthreads();
  // ---- flush: S_new = G_m S_hat + sum_s ck_s k_s u_s^T, requantized group by group
  const float gm = sh.gam[mt - 1];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    float x[G];
#pragma unroll
    for (int ii = 0; ii < G; ++ii) {
      const int i = g * G + ii;
      const uint32_t u = BITS == 4 ? nibble_of(wr[i / KPW], i % KPW) : byte_of(wr[i / KPW], i % KPW);
      x[ii] = gm * (sg[g] * (float)((int)u - zg[g]));
    }
    for (int s = 0; s < mt; ++s) {
      const float us = sh.U[s * D + j];
      const float4 *kf4 = reinterpret_cast<const float4 *>(sh.kf + s * D + g * G);
#pragma unroll
      for (int i4 = 0; i4 < G / 4; ++i4) {
        const float4 kk = kf4[i4];
        x[4 * i4 + 0] = fmaf(kk.x, us, x[4 * i4 + 0]);
        x[4 * i4 + 1] = fmaf(kk.y, us, x[4 * i4 + 1]);
        x[4 * i4 + 2] = fmaf(kk.z, us, x[4 * i4 + 2]);
        x[4 * i4 + 3] = fmaf(kk.w, us, x[4 * i4 + 3]);
      }
    }
    uint32_t uq[G];
    float s_new;
    int z_new;
    quant_group<G, BITS>(x, st.zero_point, uq, s_new, z_new);
#pragma unroll
    for (int ww = 0; ww < WPG; ++ww) {
      uint32_t word = 0;
      if (BITS == 4) {
#pragma unroll
        for (int t = 0; t < 4; ++t) word |= (uq[8 * ww + t] | (uq[8 * ww + 4 + t] << 4)) << (8 * t);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) word |= uq[4 * ww + t] << (8 * t);
      }
      codes[(g * WPG + ww) * D + j] = word;
    }
    st.scale[(unit * NG + g) * D + j] = __float2bfloat16_rn(s_new);
    if (st.zero_point) st.zp[(unit * NG + g) * D + j] = (uint8_t)z_new;
  }
}

// Unquantized test mode: fp32 state streamed from global memory.
template <int D>
__device__ void fp32_column(const PaceDev &st, const PaceIO &io, long unit, int nv, int mt, int has_token,
                            int do_flush, const DecodeShared &sh) {
  const int j = threadIdx.x;
  float *Sp = static_cast<float *>(st.S) + unit * D * D;
  for (int c0 = 0; c0 < nv; c0 += VCHUNK) {
    float pf[VCHUNK];
#pragma unroll
    for (int t = 0; t < VCHUNK; ++t) pf[t] = 0.0f;
    for (int i = 0; i < D; ++i) {
      const float s = Sp[i * D + j];
#pragma unroll
      for (int t = 0; t < VCHUNK; ++t)
        if (c0 + t < nv) pf[t] = fmaf(s, sh.keyf[(c0 + t) * D + i], pf[t]);
    }
#pragma unroll
    for (int t = 0; t < VCHUNK; ++t)
      if (c0 + t < nv) sh.P[(c0 + t) * D + j] = pf[t];
  }
  recurrence<D>(st, io, unit, nv, mt, has_token, 1, sh);
  if (!do_flush) return;
  flush_coeffs<D>(mt, 1, sh);
  __syncthreads();
  const float gm = sh.gam[mt - 1];
  for (int i = 0; i < D; ++i) {
    float x = gm * Sp[i * D + j];
    for (int s = 0; s < mt; ++s) x = fmaf(sh.kf[s * D + i], sh.U[s * D + j], x);
    Sp[i * D + j] = x;
  }
}

template <int D, int G>
__global__ void __launch_bounds__(D) decode_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(16) unsigned char smem[];
  const long unit = blockIdx.x;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int fp32mode = st.state_mode == PACE_STATE_FP32;
  const DecodeSmem L = decode_smem(D, st.dP, fp32mode);
  const DecodeShared sh = decode_shared(smem, L);

  const int m0 = st.m[unit];
  if (m0 < 0 || m0 >= st.dP) {                    // corrupted counter: leave the unit, emit zeros
    if (has_token) store_io(io.o, unit * D + threadIdx.x, 0.0f, st.io);
    return;
  }
  if (!has_token && m0 == 0) return;              // flush with nothing pending
  const int mt = m0 + has_token;                  // tokens replayed
  const int do_flush = !has_token || mt == st.dP;
  const int nv = mt + (has_token ? (fp32mode ? 1 : 2) : 0);

  load_buffer<D>(st, unit, m0, sh);
  if (has_token) append_token<D>(st, io, unit, m0, sh);
  __syncthreads();
  if (!fp32mode) code_sums<D, G>(nv, sh);
  unit_tables<D>(mt, has_token, fp32mode, st.dP, sh);
  __syncthreads();

  if (fp32mode)
    fp32_column<D>(st, io, unit, nv, mt, has_token, do_flush, sh);
  else if (st.head_is_int8[h])
    quant_column<D, G, 8>(st, io, unit, b, h, nv, mt, has_token, do_flush, sh);
  else
    quant_column<D, G, 4>(st, io, unit, b, h, nv, mt, has_token, do_flush, sh);

  if (threadIdx.x == 0) st.m[unit] = do_flush ? 0 : mt;
}

template <int D, int G>
static cudaError_t launch_decode_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  const int fp32mode = d.state_mode == PACE_STATE_FP32;
  const size_t smem = decode_smem(D, d.dP, fp32mode).total;
  auto kern = decode_kernel<D, G>;
  static size_t opted = 48 * 1024;                // dynamic shared memory allowed so far
  if (smem > opted) {
    const size_t most = decode_smem(D, PACE_MAX_DP, 1).total;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    opted = most;
  }
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  kern<<<units, D, smem, s>>>(d, io, has_token);
  return cudaGetLastError();
}

}  // namespace pace

cudaError_t pace_launch_decode(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.D == 128) return d.G == 64 ? launch_decode_t<128, 64>(d, io, has_token, s)
                                   : launch_decode_t<128, 32>(d, io, has_token, s);
  return d.G == 64 ? launch_decode_t<64, 64>(d, io, has_token, s) : launch_decode_t<64, 32>(d, io, has_token, s);
}
