// PACE decode step with fused flush, quantized state ([P1] 어떻게 동작하나: round once every dP tokens, the
// buffered tokens applied together at the flush; [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// One warp per unit (sequence b, head h); the warp walks the state in blocks of 32 columns. Both dense
// contractions of the step run on the tensor cores as warp-level bf16 MMAs (m16n8k16 / m16n8k8, fp32
// accumulation), with operands built in registers straight from the packed codes:
//   dots   D_g[v][j] = sum_{i in group g} B[v][i] (128 + u_ij)        M = vectors v, N = columns j, K = keys
//          The vectors are the int8 key codes of the buffered tokens and three int8 digits of a 24-bit
//          fixed-point image of q. The packed words are stored in fragment order (pace.h): the lane's
//          word gives its B fragment as (word >> 4r) & 0x000F000F | 0x43004300, the bf16 pair
//          (128 + u, 128 + u'). Every product and partial sum is an exact integer in fp32, so with the
//          group scale s_gj and zero point z_gj: (S_hat^T x)_j = sum_g s_gj (D_g[v][j] - (128 + z_gj) c_vg),
//          c_vg = sum_{i in g} B[v][i];
//   flush  S_new^T[j][i] = G_m s_gj (u_ij - z_gj) + sum_s (rho_s u_s,j) k_s,i  M = columns, N = keys,
//          K = (token, part): rho_s u_s,j is split into three bf16 parts (fp32-accurate) and the int8 keys
//          are exact in bf16. The accumulator starts from the dequantized state, and a lane's fragment
//          holds exactly the keys of its own packed words: each key-axis group is requantized by the lane
//          quad that holds it (two shuffles for the absmax or the min/max) and written back in place.
// Between the two, each lane replays one column in reduced form (fp32):
//   u_t = beta_t (v_t - G_t (S_hat^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),   G_t = a_1 .. a_t
//   o   = G_m (S_hat^T q) + sum_s (G_m/G_s)(k_s.q) u_s
#include "pace_common.cuh"

namespace pace {

constexpr int DM_WARPS = 4;   // units (warps) per block
constexpr int PB_STRIDE = 40; // floats per row of the per-block dot table (conflict-free fragment stores)
constexpr int UB_STRIDE = 36; // floats per row of the per-block replay table (conflict-free fragment loads)

__host__ __device__ inline int dm_dpp(int dP) { return 8 * ((dP + 7) / 8); }   // token slots per K part

struct MmaSmem {
  size_t krow, vrow, abf, kbf, pb, ub, W, a, gam, dmq, cq, ck, vsc, bt, sv, csum, total;
};
// Per-warp work area.
__host__ __device__ inline MmaSmem mma_smem(int D, int dP, int mixed) {
  MmaSmem L;
  size_t off = 0;
  const int nvmax = dP + 3, nvt = (nvmax + 15) / 16;
  L.krow = carve(off, (size_t)nvmax * D);                 // int8 key rows, then the three digits of q
  L.vrow = carve(off, (size_t)dP * D * (mixed ? 2 : 1));  // value codes (int8) or bf16 values
  L.abf = carve(off, (size_t)nvt * (D / 16) * 32 * 16);   // A fragments of the vectors (bf16)
  L.kbf = carve(off, (size_t)D * dm_dpp(dP) * 2);          // flush B operand: bf16 k_s,i as [i][s]
  L.pb = carve(off, (size_t)nvmax * PB_STRIDE * 4);       // dots of one 32-column block [v][j]
  L.ub = carve(off, (size_t)dP * UB_STRIDE * 4);          // replayed u of one block [s][j]
  L.W = carve(off, (size_t)dP * dP * 4);
  L.a = carve(off, (size_t)dP * 4);
  L.gam = carve(off, (size_t)dP * 4);
  L.dmq = carve(off, (size_t)dP * 4);
  L.cq = carve(off, (size_t)dP * 4);
  L.ck = carve(off, (size_t)dP * 4);
  L.vsc = carve(off, (size_t)nvmax * 4);
  L.bt = carve(off, (size_t)dP * 4);
  L.sv = carve(off, (size_t)dP * 4);
  L.csum = carve(off, (size_t)nvmax * 4 * 4);
  L.total = carve(off, 0, 16);
  return L;
}

struct MmaShared {
  int8_t *krow;
  unsigned char *vrow;
  uint4 *abf;
  uint32_t *kbf;
  float *pb, *ub, *W, *a, *gam, *dmq, *cq, *ck, *vsc, *bt, *sv;
  int *csum;
};
__device__ inline MmaShared mma_shared(unsigned char *base, const MmaSmem &L) {
  MmaShared s;
  s.krow = reinterpret_cast<int8_t *>(base + L.krow);
  s.vrow = base + L.vrow;
  s.abf = reinterpret_cast<uint4 *>(base + L.abf);
  s.kbf = reinterpret_cast<uint32_t *>(base + L.kbf);
  s.pb = reinterpret_cast<float *>(base + L.pb);
  s.ub = reinterpret_cast<float *>(base + L.ub);
  s.W = reinterpret_cast<float *>(base + L.W);
  s.a = reinterpret_cast<float *>(base + L.a);
  s.gam = reinterpret_cast<float *>(base + L.gam);
  s.dmq = reinterpret_cast<float *>(base + L.dmq);
  s.cq = reinterpret_cast<float *>(base + L.cq);
  s.ck = reinterpret_cast<float *>(base + L.ck);
  s.vsc = reinterpret_cast<float *>(base + L.vsc);
  s.bt = reinterpret_cast<float *>(base + L.bt);
  s.sv = reinterpret_cast<float *>(base + L.sv);
  s.csum = reinterpret_cast<int *>(base + L.csum);
  return s;
}

// D (4 fp32) += A (16x16 bf16, 4 regs) x B (16x8 bf16, 2 regs)
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D (4 fp32) += A (16x8 bf16, 2 regs) x B (8x8 bf16, 1 reg)
__device__ __forceinline__ void mma8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// bf16 pair (128 + u, 128 + u') of the nibbles at bits 4r and 16 + 4r of a packed word.
__device__ __forceinline__ uint32_t nib_pair(uint32_t word, int r) {
  return ((word >> (4 * r)) & 0x000F000Fu) | 0x43004300u;
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int D, int BITS>
__device__ __forceinline__ uint32_t *dm_unit_codes(const PaceDev &st, int b, int h) {
  return BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                   : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
}

template <int CPL>
__device__ __forceinline__ void dm_load_io(const void *p, long idx, int io, float (&x)[CPL]) {
  if (io == PACE_IO_F32) {
#pragma unroll
    for (int e = 0; e < CPL; e += 2) {
      const float2 v = *reinterpret_cast<const float2 *>(static_cast<const float *>(p) + idx + e);
      x[e] = v.x;
      x[e + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < CPL; e += 2) {
      const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(static_cast<const __nv_bfloat16 *>(p) + idx + e);
      x[e] = __low2float(v);
      x[e + 1] = __high2float(v);
    }
  }
}

template <int CPL>
__device__ __forceinline__ void dm_store_bytes(void *p, const int (&c)[CPL]) {
  if constexpr (CPL == 4)
    *reinterpret_cast<uint32_t *>(p) = (uint32_t)(c[0] & 0xFF) | ((uint32_t)(c[1] & 0xFF) << 8) |
                                       ((uint32_t)(c[2] & 0xFF) << 16) | ((uint32_t)(c[3] & 0xFF) << 24);
  else
    *reinterpret_cast<uint16_t *>(p) = (uint16_t)((c[0] & 0xFF) | ((c[1] & 0xFF) << 8));
}

// Stage the buffered tokens and the new one (written into buffer slot m0) and compute the per-unit tables:
// decay products, Gram coefficients W[t][s], readout coefficients cq / ck, group sums of every row.
template <int D, int G>
__device__ void dm_stage(const PaceDev &st, const PaceIO &io, long unit, int m0, int has_token, const MmaShared &sh) {
  constexpr int CPL = D / 32, NG = D / G;
  const int lane = threadIdx.x & 31;
  const int col0 = CPL * lane;
  const int dP = st.dP;
  const int mt = m0 + has_token;
  const int nv = mt + (has_token ? 3 : 0);
  const int mixed = st.buf_mode == PACE_BUF_MIXED;
  float sa = 0.0f, sb = 0.0f, ssk = 0.0f, ssv = 0.0f;
  if (lane < m0) {
    const float4 r = *reinterpret_cast<const float4 *>(st.buf_s + ((size_t)unit * dP + lane) * 4);
    sa = r.x; sb = r.y; ssk = r.z; ssv = r.w;
  }
  for (int t = 0; t < m0; ++t) {
    if (lane < D / 8) {                         // one 8-key run per lane, natural order
      uint2 x;
      if (mixed) {
        const uint32_t nb = *reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(st.buf_k) +
                                                                 ((size_t)unit * dP + t) * (D / 2) + 4 * lane);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          lo |= (uint32_t)(((int)((nb >> (8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
          hi |= (uint32_t)(((int)((nb >> (16 + 8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
        }
        x = make_uint2(lo, hi);
      } else {
        x = *reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(st.buf_k) + ((size_t)unit * dP + t) * D + 8 * lane);
      }
      *reinterpret_cast<uint2 *>(sh.krow + t * D + 8 * lane) = x;
    }
    if (mixed) {
      const uint32_t *src = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(st.buf_v) +
                                                               ((size_t)unit * dP + t) * D + col0);
      uint32_t *dst = reinterpret_cast<uint32_t *>(sh.vrow + ((size_t)t * D + col0) * 2);
#pragma unroll
      for (int e = 0; e < CPL / 2; ++e) dst[e] = src[e];
    } else {
      const int8_t *src = static_cast<const int8_t *>(st.buf_v) + ((size_t)unit * dP + t) * D + col0;
      if constexpr (CPL == 4)
        *reinterpret_cast<uint32_t *>(sh.vrow + t * D + col0) = *reinterpret_cast<const uint32_t *>(src);
      else
        *reinterpret_cast<uint16_t *>(sh.vrow + t * D + col0) = *reinterpret_cast<const uint16_t *>(src);
    }
  }
  float qx[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) qx[c] = 0.0f;
  if (has_token) {
    float kx[CPL], vx[CPL];
    dm_load_io<CPL>(io.k, unit * D + col0, st.io, kx);
    dm_load_io<CPL>(io.v, unit * D + col0, st.io, vx);
    dm_load_io<CPL>(io.q, unit * D + col0, st.io, qx);
    float mk = 0.0f, mv = 0.0f, mq = 0.0f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      mk = fmaxf(mk, fabsf(kx[c]));
      mv = fmaxf(mv, fabsf(vx[c]));
      mq = fmaxf(mq, fabsf(qx[c]));
    }
    const float Ak = warp_max(mk), Av = warp_max(mv), Aq = warp_max(mq);
    const int qk = mixed ? 7 : 127;
    const float sk = buffer_scale(Ak, qk);
    int ck[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) ck[c] = buffer_code(kx[c], Ak, qk);
    dm_store_bytes<CPL>(sh.krow + m0 * D + col0, ck);
    float sv = 0.0f;
    if (mixed) {
      uint8_t *bk = static_cast<uint8_t *>(st.buf_k) + ((size_t)unit * dP + m0) * (D / 2) + col0 / 2;
#pragma unroll
      for (int c = 0; c < CPL; c += 2) bk[c / 2] = (uint8_t)((ck[c] + 8) | ((ck[c + 1] + 8) << 4));
      __nv_bfloat16 *bv = static_cast<__nv_bfloat16 *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0;
      uint32_t *vr = reinterpret_cast<uint32_t *>(sh.vrow + ((size_t)m0 * D + col0) * 2);
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        const __nv_bfloat162 pv = __floats2bfloat162_rn(vx[c], vx[c + 1]);
        *reinterpret_cast<__nv_bfloat162 *>(bv + c) = pv;
        vr[c / 2] = *reinterpret_cast<const uint32_t *>(&pv);
      }
    } else {
      sv = buffer_scale(Av, 127);
      int cv[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) cv[c] = buffer_code(vx[c], Av, 127);
      dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_k) + ((size_t)unit * dP + m0) * D + col0, ck);
      dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0, cv);
      dm_store_bytes<CPL>(sh.vrow + m0 * D + col0, cv);
    }
    const float an = io.a[unit], bn = io.beta[unit];
    if (lane == m0) {
      sa = an; sb = bn; ssk = sk; ssv = sv;
    }
    if (lane == 0)
      *reinterpret_cast<float4 *>(st.buf_s + ((size_t)unit * dP + m0) * 4) = make_float4(an, bn, sk, sv);
    // q ~= sigma (65536 d2 + 256 d1 + d0), |qi| <= 127 * 65536, balanced base-256 digits in [-128, 127]
    const float QMAX = 8323072.0f;
    const float sigma = Aq >= FLT_MIN ? Aq / QMAX : 0.0f;
    int d2[CPL], d1[CPL], d0[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      int qi = 0;
      if (Aq >= FLT_MIN) qi = min(max(__float2int_rn(qx[c] * (QMAX / Aq)), -8323072), 8323072);
      const int q1 = (qi + 128) >> 8;
      d0[c] = qi - (q1 << 8);
      d2[c] = (q1 + 128) >> 8;
      d1[c] = q1 - (d2[c] << 8);
    }
    dm_store_bytes<CPL>(sh.krow + mt * D + col0, d2);
    dm_store_bytes<CPL>(sh.krow + (mt + 1) * D + col0, d1);
    dm_store_bytes<CPL>(sh.krow + (mt + 2) * D + col0, d0);
    if (lane == 0) {
      sh.vsc[mt] = 65536.0f * sigma;
      sh.vsc[mt + 1] = 256.0f * sigma;
      sh.vsc[mt + 2] = sigma;
    }
  }
  if (lane < mt) {
    sh.a[lane] = sa;
    sh.vsc[lane] = ssk;
    sh.bt[lane] = sb;
    sh.sv[lane] = ssv;
  }
  __syncwarp();
  // group sums of every staged row
  for (int p = lane; p < nv * NG; p += 32) {
    const int v = p / NG, g = p - v * NG;
    int s = 0;
#pragma unroll
    for (int i4 = 0; i4 < G / 4; ++i4) s = dp4a_ss(*reinterpret_cast<const int *>(sh.krow + v * D + g * G + 4 * i4), 0x01010101, s);
    sh.csum[v * 4 + g] = s;
  }
  // decay products, Gram coefficients, readout coefficients
  if (lane < mt) {
    float g = 1.0f, dm = 1.0f;
    for (int r = 0; r <= lane; ++r) g *= sh.a[r];
    for (int r = lane + 1; r < mt; ++r) dm *= sh.a[r];
    sh.gam[lane] = g;
    sh.dmq[lane] = dm;
  }
  const int npairs = mt * (mt - 1) / 2;
  for (int p = lane; p < npairs; p += 32) {
    int t = 1, base = 0;
    while (base + t <= p) {
      base += t;
      ++t;
    }
    const int s = p - base;
    float dm = 1.0f;
    for (int r = s + 1; r <= t; ++r) dm *= sh.a[r];
    int dot = 0;
#pragma unroll
    for (int i4 = 0; i4 < D / 4; ++i4)
      dot = dp4a_ss(*reinterpret_cast<const int *>(sh.krow + s * D + 4 * i4),
                    *reinterpret_cast<const int *>(sh.krow + t * D + 4 * i4), dot);
    sh.W[t * dP + s] = dm * sh.vsc[s] * sh.vsc[t] * (float)dot;
  }
  __syncwarp();
  for (int s = 0; s < mt; ++s) {
    float part = 0.0f;
    if (has_token) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) part += (float)sh.krow[s * D + col0 + c] * qx[c];
      part = warp_sum(part);
    }
    if (lane == 0) {
      const float dv = sh.dmq[s] * sh.vsc[s];
      sh.cq[s] = dv * part;
      sh.ck[s] = dv;
    }
  }
  __syncwarp();
}

// The MMA operand tables: A fragments of the staged vectors for the dots (rows >= nv are zero) and, for
// a flush, the bf16 key table kbf[i][s] (s >= mt zero).
template <int D>
__device__ void dm_tables(const MmaShared &sh, int nv, int mt, int dpp, int do_flush) {
  constexpr int KS = D / 16;
  const int lane = threadIdx.x & 31, g8 = lane >> 2, tq = lane & 3;
  const int nvt = (nv + 15) >> 4;
  for (int vt = 0; vt < nvt; ++vt) {
#pragma unroll 4
    for (int ks = 0; ks < KS; ++ks) {
      const int k0 = 16 * ks + 2 * tq;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = 16 * vt + g8 + 8 * (q & 1), key = k0 + 8 * (q >> 1);
        w[q] = 0u;
        if (row < nv) {
          const int8_t *p = sh.krow + row * D + key;
          w[q] = bf16x2_bits((float)p[0], (float)p[1]);
        }
      }
      sh.abf[(vt * KS + ks) * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (do_flush) {
    const int half = dpp >> 1;
    for (int idx = lane; idx < D * half; idx += 32) {
      const int i = idx / half, s = 2 * (idx - i * half);
      const float k0 = s < mt ? (float)sh.krow[s * D + i] : 0.0f;
      const float k1 = s + 1 < mt ? (float)sh.krow[(s + 1) * D + i] : 0.0f;
      sh.kbf[idx] = bf16x2_bits(k0, k1);
    }
  }
  __syncwarp();
}

// Requantize one key-axis group of one column from the lane quad that holds it (NV values per lane, the
// quad together holding the group), with the arithmetic of quant_group. Returns the stored codes.
template <int NV, int BITS>
__device__ __forceinline__ void quad_quant(const float (&x)[NV], int zero_point, uint32_t (&u)[NV], float &s_out,
                                           int &z_out) {
  float s;
  int z;
  if (!zero_point) {
    constexpr int qmax = (1 << (BITS - 1)) - 1;
    float A = 0.0f;
#pragma unroll
    for (int e = 0; e < NV; ++e) A = fmaxf(A, fabsf(x[e]));
    A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 1));
    A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 2));
    s = bf16_round(__fdiv_rn(A, (float)qmax));
    z = 1 << (BITS - 1);
    if (!(s >= FLT_MIN)) s = 0.0f;
  } else {
    constexpr int qm = (1 << BITS) - 1;
    float lo = 0.0f, hi = 0.0f;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      lo = fminf(lo, x[e]);
      hi = fmaxf(hi, x[e]);
    }
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 2));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, 2));
    s = bf16_round(__fdiv_rn(__fsub_rn(hi, lo), (float)qm));
    z = 0;
    if (!(s >= FLT_MIN))
      s = 0.0f;
    else
      z = min(max(__float2int_rn(__fmul_rn(-lo, __fdiv_rn(1.0f, s))), 0), qm);
  }
  const float r = s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    int c;
    if (s == 0.0f) {
      c = z;
    } else if (!zero_point) {
      constexpr int qmax = (1 << (BITS - 1)) - 1;
      c = min(max(__float2int_rn(__fmul_rn(x[e], r)), -qmax), qmax) + z;
    } else {
      constexpr int qm = (1 << BITS) - 1;
      c = min(max(__float2int_rn(__fmul_rn(x[e], r)) + z, 0), qm);
    }
    u[e] = (uint32_t)c;
  }
  s_out = s;
  z_out = z;
}

template <int D, int G, int BITS>
__device__ void dm_unit(const PaceDev &st, const PaceIO &io, long unit, int m0, int has_token, const MmaShared &sh) {
  constexpr int NG = D / G, NPP = D / 64, KS = D / 16, KSG = G / 16, PL = BITS / 4;
  constexpr int NKG = G / 8;            // key n-tiles (8 keys) per group
  constexpr int NH = BITS == 8 ? 2 : 1, NPN = 4 / NH;   // dot passes, column n-tiles per pass
  constexpr uint32_t PLANE = D * D / 8; // words per nibble plane
  const int lane = threadIdx.x & 31, g8 = lane >> 2, tq = lane & 3;
  const int dP = st.dP;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 3 : 0);
  const int nvt = (nv + 15) >> 4;
  const int dpp = dm_dpp(dP);
  const int mixed = st.buf_mode == PACE_BUF_MIXED;
  const int zpm = st.zero_point;
  uint32_t *codes = dm_unit_codes<D, BITS>(st, b, h);
  __nv_bfloat16 *scale = st.scale + (size_t)unit * NG * D;
  uint8_t *zpt = zpm ? st.zp + (size_t)unit * NG * D : nullptr;

  if (lane == 0) {                       // the unit's resident bytes start moving into L2 right away
    prefetch_l2(codes, PL * PLANE * 4);
    prefetch_l2(scale, NG * D * 2);
    if (zpm) prefetch_l2(zpt, NG * D);
    if (m0 > 0) {
      const uint32_t rk = mixed ? D / 2 : D, rv = mixed ? 2 * D : D;
      prefetch_l2(static_cast<const char *>(st.buf_k) + (size_t)unit * dP * rk, m0 * rk);
      prefetch_l2(static_cast<const char *>(st.buf_v) + (size_t)unit * dP * rv, m0 * rv);
    }
  }
  dm_stage<D, G>(st, io, unit, m0, has_token, sh);
  dm_tables<D>(sh, nv, mt, dpp, do_flush);
  const float gm = sh.gam[mt - 1];

#pragma unroll 1
  for (int cb = 0; cb < D / 32; ++cb) {
    // ---- the lane's packed words of this block: M-tiles 2cb, 2cb+1 (columns cb*32 + 16m + 8hi + g8)
    uint32_t cw[PL][2][NPP][4];
#pragma unroll
    for (int pl = 0; pl < PL; ++pl)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int pp = 0; pp < NPP; ++pp) {
          const uint4 v = *reinterpret_cast<const uint4 *>(codes + pl * PLANE + (((2 * cb + m) * NPP + pp) * 32 + lane) * 4);
          cw[pl][m][pp][0] = v.x;
          cw[pl][m][pp][1] = v.y;
          cw[pl][m][pp][2] = v.z;
          cw[pl][m][pp][3] = v.w;
        }

    // ---- dots: P[v][j] for the 32 columns of the block; n-tile n = columns cb*32 + 8n .. +7
#pragma unroll 1
    for (int vt = 0; vt < nvt; ++vt) {
      const int v0 = 16 * vt + g8;
      float pacc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) pacc[n][e] = 0.0f;
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)          // int8 heads: two passes of two n-tiles (register budget)
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          uint32_t sc[NPN], zz[NPN];
#pragma unroll
          for (int q = 0; q < NPN; ++q) {
            const int j = cb * 32 + 8 * (nh * NPN + q) + 2 * tq;
            sc[q] = *reinterpret_cast<const uint32_t *>(scale + gi * D + j);
            zz[q] = zpm ? (uint32_t)*reinterpret_cast<const uint16_t *>(zpt + gi * D + j) : 0u;
          }
          float dacc[PL][NPN][4];
#pragma unroll
          for (int pl = 0; pl < PL; ++pl)
#pragma unroll
            for (int q = 0; q < NPN; ++q)
#pragma unroll
              for (int e = 0; e < 4; ++e) dacc[pl][q][e] = 0.0f;
#pragma unroll
          for (int kk = 0; kk < KSG; ++kk) {
            const int ks = gi * KSG + kk;
            const uint4 av = sh.abf[(vt * KS + ks) * 32 + lane];
            const uint32_t a[4] = {av.x, av.y, av.z, av.w};
            const int r = 2 * (ks & 1);
#pragma unroll
            for (int q = 0; q < NPN; ++q)
#pragma unroll
              for (int pl = 0; pl < PL; ++pl) {
                const int n = nh * NPN + q;
                const uint32_t w = cw[pl][n >> 1][ks >> 2][(n & 1) * 2 + ((ks >> 1) & 1)];
                mma16(dacc[pl][q], a, nib_pair(w, r), nib_pair(w, r + 1));
              }
          }
          // fold the group: P += s_gj sum_i (u_ij - z_gj) B[v][i]
          const int cs0 = v0 < nv ? sh.csum[v0 * 4 + gi] : 0;
          const int cs1 = v0 + 8 < nv ? sh.csum[(v0 + 8) * 4 + gi] : 0;
#pragma unroll
          for (int q = 0; q < NPN; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int n = nh * NPN + q;
              const float s = (e & 1) ? bf16_hi(sc[q]) : bf16_lo(sc[q]);
              const int zj = zpm ? (int)((zz[q] >> (8 * (e & 1))) & 0xFFu) : (1 << (BITS - 1));
              const int cs = (e >> 1) ? cs1 : cs0;
              float tot;
              if (BITS == 4) {
                tot = fmaf(-(float)(128 + zj), (float)cs, dacc[0][q][e]);
              } else {
                tot = (float)(__float2int_rn(dacc[0][q][e]) + 16 * __float2int_rn(dacc[PL - 1][q][e]) - (2176 + zj) * cs);
              }
              pacc[n][e] = gi == 0 ? s * tot : fmaf(s, tot, pacc[n][e]);
            }
        }
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        if (v0 < nv) *reinterpret_cast<float2 *>(sh.pb + v0 * PB_STRIDE + 8 * n + 2 * tq) = make_float2(pacc[n][0], pacc[n][1]);
        if (v0 + 8 < nv)
          *reinterpret_cast<float2 *>(sh.pb + (v0 + 8) * PB_STRIDE + 8 * n + 2 * tq) = make_float2(pacc[n][2], pacc[n][3]);
      }
    }
    __syncwarp();

    // ---- replay and readout: lane = column cb*32 + lane
    {
      const int j = cb * 32 + lane;
      for (int t = 0; t < mt; ++t) {
        float vt;
        if (mixed)
          vt = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(sh.vrow)[t * D + j]);
        else
          vt = sh.sv[t] * (float)reinterpret_cast<const int8_t *>(sh.vrow)[t * D + j];
        float acc = vt - sh.gam[t] * (sh.vsc[t] * sh.pb[t * PB_STRIDE + lane]);
        for (int s = 0; s < t; ++s) acc = fmaf(-sh.W[t * dP + s], sh.ub[s * UB_STRIDE + lane], acc);
        sh.ub[t * UB_STRIDE + lane] = sh.bt[t] * acc;
      }
      if (has_token) {
        float o = gm * (sh.vsc[mt] * sh.pb[mt * PB_STRIDE + lane] +
                        (sh.vsc[mt + 1] * sh.pb[(mt + 1) * PB_STRIDE + lane] + sh.vsc[mt + 2] * sh.pb[(mt + 2) * PB_STRIDE + lane]));
        for (int s = 0; s < mt; ++s) o = fmaf(sh.cq[s], sh.ub[s * UB_STRIDE + lane], o);
        store_io(io.o, unit * D + j, o, st.io);
      }
    }
    __syncwarp();
    if (!do_flush) continue;

    // ---- flush: rebuild and requantize the block's columns, M-tile by M-tile
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int jl = 16 * m + g8;              // local columns jl (hi = 0) and jl + 8 (hi = 1)
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float fs[2];
        int fz[2];
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int j = cb * 32 + jl + 8 * hi;
          fs[hi] = gm * __bfloat162float(scale[gi * D + j]);
          fz[hi] = zpm ? (int)zpt[gi * D + j] : (1 << (BITS - 1));
        }
        __syncwarp();                          // the quad has read the old scale before lane 0 replaces it
        float c[NKG][4];
#pragma unroll
        for (int nn = 0; nn < NKG; ++nn) {
          const int nk = gi * NKG + nn;
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const int wi = hi * 2 + ((nk >> 2) & 1), r = nk & 3;
            uint32_t u0 = (cw[0][m][nk >> 3][wi] >> (4 * r)) & 0xFu;
            uint32_t u1 = (cw[0][m][nk >> 3][wi] >> (16 + 4 * r)) & 0xFu;
            if (BITS == 8) {
              u0 |= ((cw[PL - 1][m][nk >> 3][wi] >> (4 * r)) & 0xFu) << 4;
              u1 |= ((cw[PL - 1][m][nk >> 3][wi] >> (16 + 4 * r)) & 0xFu) << 4;
            }
            c[nn][2 * hi] = fs[hi] * (float)((int)u0 - fz[hi]);
            c[nn][2 * hi + 1] = fs[hi] * (float)((int)u1 - fz[hi]);
          }
        }
#pragma unroll 1
        for (int sb = 0; sb < (dpp >> 3); ++sb) {
          // A: the three bf16 parts of rho_s u_s,j for tokens s = 8sb + 2tq, +1 and columns jl, jl + 8
          uint32_t ap[3][2];
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const int s0 = 8 * sb + 2 * tq;
            const float x0 = s0 < mt ? sh.ck[s0] * sh.ub[s0 * UB_STRIDE + jl + 8 * hi] : 0.0f;
            const float x1 = s0 + 1 < mt ? sh.ck[s0 + 1] * sh.ub[(s0 + 1) * UB_STRIDE + jl + 8 * hi] : 0.0f;
            const uint32_t p0 = bf16x2_bits(x0, x1);
            const float r0 = x0 - bf16_lo(p0), r1 = x1 - bf16_hi(p0);
            const uint32_t p1 = bf16x2_bits(r0, r1);
            const uint32_t p2 = bf16x2_bits(r0 - bf16_lo(p1), r1 - bf16_hi(p1));
            ap[0][hi] = p0;
            ap[1][hi] = p1;
            ap[2][hi] = p2;
          }
          const uint32_t a16[4] = {ap[0][0], ap[0][1], ap[1][0], ap[1][1]};
#pragma unroll
          for (int nn = 0; nn < NKG; ++nn) {
            const int i = 8 * (gi * NKG + nn) + g8;
            const uint32_t bk = sh.kbf[i * (dpp >> 1) + 4 * sb + tq];
            mma16(c[nn], a16, bk, bk);
            mma8(c[nn], ap[2][0], ap[2][1], bk);
          }
        }
        // requantize the group for both columns; the lane's keys fill its own words
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          float x[2 * NKG];
#pragma unroll
          for (int nn = 0; nn < NKG; ++nn) {
            x[2 * nn] = c[nn][2 * hi];
            x[2 * nn + 1] = c[nn][2 * hi + 1];
          }
          uint32_t u[2 * NKG];
          float s_new;
          int z_new;
          quad_quant<2 * NKG, BITS>(x, zpm, u, s_new, z_new);
#pragma unroll
          for (int pw = 0; pw < G / 32; ++pw) {
            const int p = gi * (G / 32) + pw;  // 32-key span
            uint32_t lo = 0, hw = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int nn = 4 * pw + r;
              lo |= ((u[2 * nn] & 0xFu) << (4 * r)) | ((u[2 * nn + 1] & 0xFu) << (16 + 4 * r));
              hw |= (((u[2 * nn] >> 4) & 0xFu) << (4 * r)) | (((u[2 * nn + 1] >> 4) & 0xFu) << (16 + 4 * r));
            }
            cw[0][m][p >> 1][hi * 2 + (p & 1)] = lo;
            if (BITS == 8) cw[PL - 1][m][p >> 1][hi * 2 + (p & 1)] = hw;
          }
          if (tq == 0) {
            const int j = cb * 32 + jl + 8 * hi;
            scale[gi * D + j] = __float2bfloat16_rn(s_new);
            if (zpm) zpt[gi * D + j] = (uint8_t)z_new;
          }
        }
      }
    }
#pragma unroll
    for (int pl = 0; pl < PL; ++pl)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int pp = 0; pp < NPP; ++pp)
          *reinterpret_cast<uint4 *>(codes + pl * PLANE + (((2 * cb + m) * NPP + pp) * 32 + lane) * 4) =
              make_uint4(cw[pl][m][pp][0], cw[pl][m][pp][1], cw[pl][m][pp][2], cw[pl][m][pp][3]);
  }
}

// One launch per code pool (int4 heads, int8 heads), so that each path gets its own register allocation
// (int4: 16 warps per SM at <= 128 registers; int8, with twice the code words live: 12 warps per SM).
// Warp w of the launch handles pool unit w: sequence w / HP, the pool's head slot w % HP.
template <int D, int G, int BITS>
__global__ void __launch_bounds__(DM_WARPS * 32, BITS == 4 ? 4 : 3) decode_mma_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const MmaSmem L = mma_smem(D, st.dP, st.buf_mode == PACE_BUF_MIXED);
  const MmaShared sh = mma_shared(smem + (size_t)warp * L.total, L);
  const int HP = BITS == 4 ? st.H4 : st.H8;
  const long w = (long)blockIdx.x * DM_WARPS + warp;
  if (w >= (long)st.B * HP) return;
  const int b = (int)(w / HP), slot = (int)(w - (long)b * HP);
  const int h = st.pool_head[(BITS == 4 ? 0 : st.H4) + slot];
  const long u = (long)b * st.H + h;
  const int m0 = st.m[u];
  if (m0 < 0 || m0 >= st.dP) {                  // corrupted counter: leave the unit, emit zeros
    if (has_token)
      for (int c = lane; c < D; c += 32) store_io(io.o, u * D + c, 0.0f, st.io);
    return;
  }
  if (!has_token && m0 == 0) return;            // flush with nothing pending
  dm_unit<D, G, BITS>(st, io, u, m0, has_token, sh);
  __syncwarp();
  if (lane == 0) st.m[u] = (!has_token || m0 + 1 == st.dP) ? 0 : m0 + 1;
}

template <int D, int G, int BITS>
static cudaError_t launch_pool(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s, size_t smem) {
  auto kern = decode_mma_kernel<D, G, BITS>;
  static size_t opted = 0;
  if (smem > 48 * 1024 && smem > opted) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    opted = 227 * 1024;
  }
  const long units = (long)d.B * (BITS == 4 ? d.H4 : d.H8);
  if (units == 0) return cudaSuccess;
  const long blocks = (units + DM_WARPS - 1) / DM_WARPS;
  kern<<<(unsigned)blocks, DM_WARPS * 32, smem, s>>>(d, io, has_token);
  return cudaGetLastError();
}

template <int D, int G>
static cudaError_t launch_mma_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  const MmaSmem L = mma_smem(D, d.dP, d.buf_mode == PACE_BUF_MIXED);
  const size_t smem = (size_t)DM_WARPS * L.total;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = launch_pool<D, G, 4>(d, io, has_token, s, smem);
  if (e == cudaSuccess) e = launch_pool<D, G, 8>(d, io, has_token, s, smem);
  return e;
}

}  // namespace pace

cudaError_t pace_launch_decode_quant(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.D == 128) return d.G == 64 ? launch_mma_t<128, 64>(d, io, has_token, s) : launch_mma_t<128, 32>(d, io, has_token, s);
  return d.G == 64 ? launch_mma_t<64, 64>(d, io, has_token, s) : launch_mma_t<64, 32>(d, io, has_token, s);
}
