// PACE decode step with fused flush, quantized state ([P1] 어떻게 동작하나: round once every dP tokens, the
// buffered tokens applied together at the flush; [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// One warp per unit (sequence b, head h); lane l owns state columns CPL*l .. CPL*l+CPL-1 (CPL = d_v/32),
// so every per-column quantity -- the dot products, the replay recurrence, the output and the key-axis
// group requantization -- stays inside one lane; warp shuffles carry the per-unit reductions. Many
// independent units per SM hide memory latency. Per call:
//   1. the lane reads its columns' packed codes with 128-bit coalesced loads (a warp covers 512
//      contiguous bytes per row of 8 keys), its group scales / zero points, and stages the m buffered key
//      rows, value codes and scalars; the new token is quantized into buffer slot m (warp-shuffle absmax);
//      q enters as a 24-bit fixed-point image split into three int8 digit rows (fp32-grade);
//   2. byte dot products (dp4a) of the packed codes with every staged key row: the int4 word keeps key
//      8w+e in bits 4e, so `w & 0x0F0F0F0F` / `w & 0xF0F0F0F0` are the even / odd keys (the latter times
//      16) against key rows stored as (even quad, odd quad); integers are exact, the group scale and zero
//      point apply per group: (S_hat^T k)_j = s_k sum_g s_gj (sum_i u_ij k_i - z_gj sum_i k_i);
//   3. the replay in reduced per-column form (fp32):
//        u_t = beta_t (v_t - G_t (S_hat^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),   G_t = a_1 .. a_t
//        o   = G_m (S_hat^T q) + sum_s (G_m/G_s)(k_s.q) u_s
//   4. at a flush each lane rebuilds its columns, S_new = G_m S_hat + sum_s (G_m/G_s) k_s u_s^T, group by
//      group, and requantizes them in place (thread-local absmax / min-max).
#include "pace_common.cuh"
#include "umma.cuh"

namespace pace {
using umma::bulk_g2s;
using umma::mbar_arrive_expect_tx;
using umma::mbar_fence_init;
using umma::mbar_init;
using umma::mbar_wait;

constexpr int WU_WARPS = 2;                    // warps per block
constexpr uint64_t WU_WAIT_NS = 1000000000ull; // bound of every wait (1 s)

// A unit's bytes as they sit in global memory, staged by bulk asynchronous copies.
struct UnitStage {
  size_t codes, scales, zp, bk, bv, bs, q, k, v, bytes;
};
__host__ __device__ inline UnitStage unit_stage(int D, int G, int dP, int zp, int mixed, int io_f32, int any8) {
  UnitStage L;
  size_t off = 0;
  const size_t iob = io_f32 ? 4 : 2;
  L.codes = carve(off, (size_t)D * D / (any8 ? 1 : 2));
  L.scales = carve(off, (size_t)(D / G) * D * 2);
  L.zp = carve(off, zp ? (size_t)(D / G) * D : 0);
  L.bk = carve(off, (size_t)dP * (mixed ? D / 2 : D));
  L.bv = carve(off, (size_t)dP * (mixed ? 2 * D : D));
  L.bs = carve(off, (size_t)dP * 16);
  L.q = carve(off, D * iob);
  L.k = carve(off, D * iob);
  L.v = carve(off, D * iob);
  L.bytes = carve(off, 0);
  return L;
}

struct WarpSmem {
  size_t krow, vrow, P, U, W, a, gam, dmq, cq, ck, vsc, csum, total;
};
// Per-warp work area. P is lane-private (float4 / float2 per row); at a flush it is reused for the
// coefficient table kc[s][i] = (G_m/G_s) s_ks k_s,i read by every lane.
__host__ __device__ inline WarpSmem warp_smem(int D, int dP, int mixed) {
  WarpSmem L;
  size_t off = 0;
  L.krow = carve(off, (size_t)(dP + 3) * D);           // key code rows, then the three digits of q (int8)
  L.vrow = carve(off, (size_t)dP * D * (mixed ? 2 : 1)); // value codes (int8) or bf16 values, lane-private
  L.P = carve(off, (size_t)(dP + 3) * D * 4);
  L.U = carve(off, (size_t)dP * D * 4);
  L.W = carve(off, (size_t)dP * dP * 4);
  L.a = carve(off, (size_t)dP * 4);
  L.gam = carve(off, (size_t)dP * 4);
  L.dmq = carve(off, (size_t)dP * 4);
  L.cq = carve(off, (size_t)dP * 4);
  L.ck = carve(off, (size_t)dP * 4);
  L.vsc = carve(off, (size_t)(dP + 3) * 4);
  L.csum = carve(off, (size_t)(dP + 3) * 4 * 4);
  L.total = carve(off, 0, 16);
  return L;
}

struct WarpShared {
  int8_t *krow;
  unsigned char *vrow;
  float *P, *U, *W, *a, *gam, *dmq, *cq, *ck, *vsc;
  int *csum;
};
__device__ inline WarpShared warp_shared(unsigned char *base, const WarpSmem &L) {
  WarpShared s;
  s.krow = reinterpret_cast<int8_t *>(base + L.krow);
  s.vrow = base + L.vrow;
  s.P = reinterpret_cast<float *>(base + L.P);
  s.U = reinterpret_cast<float *>(base + L.U);
  s.W = reinterpret_cast<float *>(base + L.W);
  s.a = reinterpret_cast<float *>(base + L.a);
  s.gam = reinterpret_cast<float *>(base + L.gam);
  s.dmq = reinterpret_cast<float *>(base + L.dmq);
  s.cq = reinterpret_cast<float *>(base + L.cq);
  s.ck = reinterpret_cast<float *>(base + L.ck);
  s.vsc = reinterpret_cast<float *>(base + L.vsc);
  s.csum = reinterpret_cast<int *>(base + L.csum);
  return s;
}

// Position of natural key i in a staged key row of an int4 head: each 8-key word row holds the even keys
// (0,2,4,6) in its first 4 bytes and the odd keys (1,3,5,7) in the next 4.
__device__ __forceinline__ int perm_pos(int i) { return (i & ~7) | ((i & 1) << 2) | ((i & 7) >> 1); }

template <int CPL>
__device__ __forceinline__ void load_words(const uint32_t *p, uint32_t (&w)[CPL]) {
  if constexpr (CPL == 4) {
    const uint4 x = *reinterpret_cast<const uint4 *>(p);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    w[0] = x.x; w[1] = x.y;
  }
}

template <int CPL>
__device__ __forceinline__ void load_io_vec(const void *p, long idx, int io, float (&x)[CPL]) {
  if (io == PACE_IO_F32) {
    if constexpr (CPL == 4) {
      const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + idx);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2 *>(static_cast<const float *>(p) + idx);
      x[0] = v.x; x[1] = v.y;
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
__device__ __forceinline__ void store_io_vec(void *p, long idx, int io, const float (&x)[CPL]) {
  if (io == PACE_IO_F32) {
    if constexpr (CPL == 4)
      *reinterpret_cast<float4 *>(static_cast<float *>(p) + idx) = make_float4(x[0], x[1], x[2], x[3]);
    else
      *reinterpret_cast<float2 *>(static_cast<float *>(p) + idx) = make_float2(x[0], x[1]);
  } else {
#pragma unroll
    for (int e = 0; e < CPL; e += 2)
      *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p) + idx + e) = __floats2bfloat162_rn(x[e], x[e + 1]);
  }
}

__device__ __forceinline__ float stage_io_at(const unsigned char *p, int i, int io) {
  if (io == PACE_IO_F32) return reinterpret_cast<const float *>(p)[i];
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
}

// CPL consecutive bytes (int8 codes) stored / loaded as one 4- or 2-byte access.
template <int CPL>
__device__ __forceinline__ void store_bytes(void *p, const int (&c)[CPL]) {
  if constexpr (CPL == 4)
    *reinterpret_cast<uint32_t *>(p) = (uint32_t)(c[0] & 0xFF) | ((uint32_t)(c[1] & 0xFF) << 8) |
                                       ((uint32_t)(c[2] & 0xFF) << 16) | ((uint32_t)(c[3] & 0xFF) << 24);
  else
    *reinterpret_cast<uint16_t *>(p) = (uint16_t)((c[0] & 0xFF) | ((c[1] & 0xFF) << 8));
}

template <int D, int G, int BITS>
__device__ void warp_unit(const PaceDev &st, const PaceIO &io, long unit, int m0, int has_token, float an, float bn,
                          const unsigned char *stg, const UnitStage &SL, const WarpShared &sh) {
  constexpr int CPL = D / 32;           // columns per lane
  constexpr int KPW = 32 / BITS;        // keys per packed word
  constexpr int NWC = D / KPW;          // words per column
  constexpr int NG = D / G;
  constexpr int WPG = G / KPW;          // words per group
  constexpr int RC = WPG < 8 ? WPG : 8; // packed word rows held in registers at a time
  const int lane = threadIdx.x & 31;
  const int col0 = CPL * lane;
  const int dP = st.dP;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 3 : 0);
  const int mixed = st.buf_mode == PACE_BUF_MIXED;
  const int slot = st.head_slot[h];
  uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + slot) * NWC * D
                              : st.codes8 + (size_t)(b * st.H8 + slot) * NWC * D;
  const uint32_t *scodes = reinterpret_cast<const uint32_t *>(stg + SL.codes);
  const __nv_bfloat16 *sscale = reinterpret_cast<const __nv_bfloat16 *>(stg + SL.scales);
  const uint8_t *szp = stg + SL.zp;

  // ---- 1. the buffered tokens: scalars (lane t holds token t), key rows (natural order), value codes
  float sa = 0.0f, sb = 0.0f, ssk = 0.0f, ssv = 0.0f;
  if (lane < m0) {
    const float4 r = reinterpret_cast<const float4 *>(stg + SL.bs)[lane];
    sa = r.x; sb = r.y; ssk = r.z; ssv = r.w;
  }
  for (int t = 0; t < m0; ++t) {
    if (lane < D / 8) {                         // one 8-key word row per lane
      uint2 x;
      if (mixed) {
        const uint32_t nb = *reinterpret_cast<const uint32_t *>(stg + SL.bk + t * (D / 2) + 4 * lane);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          lo |= (uint32_t)(((int)((nb >> (8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
          hi |= (uint32_t)(((int)((nb >> (16 + 8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
        }
        x = make_uint2(lo, hi);
      } else {
        x = *reinterpret_cast<const uint2 *>(stg + SL.bk + t * D + 8 * lane);
      }
      *reinterpret_cast<uint2 *>(sh.krow + t * D + 8 * lane) = x;
    }
    if (mixed) {
      const uint32_t *src = reinterpret_cast<const uint32_t *>(stg + SL.bv + ((size_t)t * D + col0) * 2);
      uint32_t *dst = reinterpret_cast<uint32_t *>(sh.vrow + ((size_t)t * D + col0) * 2);
#pragma unroll
      for (int e = 0; e < CPL / 2; ++e) dst[e] = src[e];
    } else {
      if constexpr (CPL == 4)
        *reinterpret_cast<uint32_t *>(sh.vrow + t * D + col0) = *reinterpret_cast<const uint32_t *>(stg + SL.bv + t * D + col0);
      else
        *reinterpret_cast<uint16_t *>(sh.vrow + t * D + col0) = *reinterpret_cast<const uint16_t *>(stg + SL.bv + t * D + col0);
    }
  }

  // ---- the new token: buffer slot m0, and the fixed-point image of q
  float qx[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) qx[c] = 0.0f;
  if (has_token) {
    float kx[CPL], vx[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      kx[c] = stage_io_at(stg + SL.k, col0 + c, st.io);
      vx[c] = stage_io_at(stg + SL.v, col0 + c, st.io);
      qx[c] = stage_io_at(stg + SL.q, col0 + c, st.io);
    }
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
    store_bytes<CPL>(sh.krow + m0 * D + col0, ck);
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
      store_bytes<CPL>(static_cast<int8_t *>(st.buf_k) + ((size_t)unit * dP + m0) * D + col0, ck);
      store_bytes<CPL>(static_cast<int8_t *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0, cv);
      store_bytes<CPL>(sh.vrow + m0 * D + col0, cv);
    }
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
    store_bytes<CPL>(sh.krow + mt * D + col0, d2);
    store_bytes<CPL>(sh.krow + (mt + 1) * D + col0, d1);
    store_bytes<CPL>(sh.krow + (mt + 2) * D + col0, d0);
    if (lane == 0) {
      sh.vsc[mt] = 65536.0f * sigma;
      sh.vsc[mt + 1] = 256.0f * sigma;
      sh.vsc[mt + 2] = sigma;
    }
  }
  if (lane < mt) {
    sh.a[lane] = sa;
    sh.vsc[lane] = ssk;
  }
  __syncwarp();

  // ---- 2. per-row group sums (natural order), then even/odd key quads for int4 heads
  for (int p = lane; p < nv * NG; p += 32) {
    const int v = p / NG, g = p - v * NG;
    int s = 0;
#pragma unroll
    for (int i4 = 0; i4 < G / 4; ++i4) s = dp4a_ss(*reinterpret_cast<const int *>(sh.krow + v * D + g * G + 4 * i4), 0x01010101, s);
    sh.csum[v * 4 + g] = s;
  }
  __syncwarp();
  if (BITS == 4 && lane < D / 8) {
    for (int v = 0; v < nv; ++v) {
      uint2 *p = reinterpret_cast<uint2 *>(sh.krow + v * D + 8 * lane);
      const uint2 x = *p;
      *p = make_uint2(__byte_perm(x.x, x.y, 0x6420), __byte_perm(x.x, x.y, 0x7531));
    }
  }
  __syncwarp();
  // ---- tables: G_t, the readout coefficients, and the Gram coefficients W[t][s]
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
      for (int c = 0; c < CPL; ++c) {
        const int i = col0 + c;
        part += (float)sh.krow[s * D + (BITS == 4 ? perm_pos(i) : i)] * qx[c];
      }
      part = warp_sum(part);
    }
    if (lane == 0) {
      const float dv = sh.dmq[s] * sh.vsc[s];
      sh.cq[s] = dv * part;
      sh.ck[s] = dv;
    }
  }
  __syncwarp();

  // ---- 3. dot products: P[v][j] = sum_g s_gj (sum_i u_ij kv_i - z_gj sum_i kv_i)   (times vsc[v] at use)
#pragma unroll 1
  for (int g = 0; g < NG; ++g) {
    float sgc[CPL];
    int zgc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      sgc[c] = __bfloat162float(sscale[g * D + col0 + c]);
      zgc[c] = st.zero_point ? (int)szp[g * D + col0 + c] : (1 << (BITS - 1));
    }
#pragma unroll 1
    for (int c0 = 0; c0 < nv; c0 += 4) {
      int acc[CPL][4], acc16[CPL][4];
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[c][v] = acc16[c][v] = 0;
#pragma unroll
      for (int rc = 0; rc < WPG / RC; ++rc) {
        uint32_t cw[RC][CPL];
#pragma unroll
        for (int r = 0; r < RC; ++r) load_words<CPL>(scodes + (g * WPG + rc * RC + r) * D + col0, cw[r]);
#pragma unroll
        for (int r = 0; r < RC; ++r) {
          const int wrow = g * WPG + rc * RC + r;
          if (BITS == 4) {
            int2 kk[4];
#pragma unroll
            for (int v = 0; v < 4; ++v)
              kk[v] = c0 + v < nv ? *reinterpret_cast<const int2 *>(sh.krow + (c0 + v) * D + 8 * wrow) : make_int2(0, 0);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
              const uint32_t lo = cw[r][c] & 0x0F0F0F0Fu, hi = cw[r][c] & 0xF0F0F0F0u;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                acc[c][v] = dp4a_us(lo, kk[v].x, acc[c][v]);
                acc16[c][v] = dp4a_us(hi, kk[v].y, acc16[c][v]);
              }
            }
          } else {
            int kk[4];
#pragma unroll
            for (int v = 0; v < 4; ++v)
              kk[v] = c0 + v < nv ? *reinterpret_cast<const int *>(sh.krow + (c0 + v) * D + 4 * wrow) : 0;
#pragma unroll
            for (int c = 0; c < CPL; ++c)
#pragma unroll
              for (int v = 0; v < 4; ++v) acc[c][v] = dp4a_us(cw[r][c], kk[v], acc[c][v]);
          }
        }
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (c0 + v < nv) {
          const int cs = sh.csum[(c0 + v) * 4 + g];
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int tot = acc[c][v] + (acc16[c][v] >> 4) - zgc[c] * cs;
            float *pp = sh.P + (c0 + v) * D + col0 + c;
            *pp = fmaf(sgc[c], (float)tot, g == 0 ? 0.0f : *pp);
          }
        }
      }
    }
  }

  // ---- 4. replay recurrence and readout (this lane's columns)
  for (int t = 0; t < mt; ++t) {
    const float bt = __shfl_sync(0xffffffffu, sb, t);
    const float svt = __shfl_sync(0xffffffffu, ssv, t);
    const float gt = sh.gam[t], vs = sh.vsc[t];
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      float vt;
      if (mixed)
        vt = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(sh.vrow)[t * D + col0 + c]);
      else
        vt = svt * (float)reinterpret_cast<const int8_t *>(sh.vrow)[t * D + col0 + c];
      acc[c] = vt - gt * (vs * sh.P[t * D + col0 + c]);
    }
    for (int s = 0; s < t; ++s) {
      const float w = sh.W[t * dP + s];
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[c] = fmaf(-w, sh.U[s * D + col0 + c], acc[c]);
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) sh.U[t * D + col0 + c] = bt * acc[c];
  }
  if (has_token) {
    const float gm = sh.gam[mt - 1], v2 = sh.vsc[mt], v1 = sh.vsc[mt + 1], v0 = sh.vsc[mt + 2];
    float o[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
      o[c] = gm * (v2 * sh.P[mt * D + col0 + c] + (v1 * sh.P[(mt + 1) * D + col0 + c] + v0 * sh.P[(mt + 2) * D + col0 + c]));
    for (int s = 0; s < mt; ++s) {
      const float cq = sh.cq[s];
#pragma unroll
      for (int c = 0; c < CPL; ++c) o[c] = fmaf(cq, sh.U[s * D + col0 + c], o[c]);
    }
    store_io_vec<CPL>(io.o, unit * D + col0, st.io, o);
  }
  if (!do_flush) return;

  // ---- 5. flush: kc[s][i] = (G_m/G_s) s_ks k_s,i in the P area, then each column group is rebuilt and
  //         requantized in place
  __syncwarp();
  float *kc = sh.P;
  for (int s = 0; s < mt; ++s) {
    const float cks = sh.ck[s];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int i = col0 + c;
      kc[s * D + i] = cks * (float)sh.krow[s * D + (BITS == 4 ? perm_pos(i) : i)];
    }
  }
  __syncwarp();
  const float gm = sh.gam[mt - 1];
#pragma unroll 1
  for (int c = 0; c < CPL; ++c) {
    const int j = col0 + c;
#pragma unroll 1
    for (int g = 0; g < NG; ++g) {
      float x[G];
      const float gs = gm * __bfloat162float(sscale[g * D + j]);
      const int zz = st.zero_point ? (int)szp[g * D + j] : (1 << (BITS - 1));
#pragma unroll
      for (int ww = 0; ww < WPG; ++ww) {
        const uint32_t wd = scodes[(g * WPG + ww) * D + j];
#pragma unroll
        for (int e = 0; e < KPW; ++e) {
          const uint32_t u = BITS == 4 ? nibble_of(wd, e) : byte_of(wd, e);
          x[ww * KPW + e] = gs * (float)((int)u - zz);
        }
      }
      for (int s = 0; s < mt; ++s) {
        const float us = sh.U[s * D + j];
        const float4 *k4 = reinterpret_cast<const float4 *>(kc + s * D + g * G);
#pragma unroll
        for (int i4 = 0; i4 < G / 4; ++i4) {
          const float4 kk = k4[i4];
          x[4 * i4 + 0] = fmaf(kk.x, us, x[4 * i4 + 0]);
          x[4 * i4 + 1] = fmaf(kk.y, us, x[4 * i4 + 1]);
          x[4 * i4 + 2] = fmaf(kk.z, us, x[4 * i4 + 2]);
          x[4 * i4 + 3] = fmaf(kk.w, us, x[4 * i4 + 3]);
        }
      }
      float s_new;
      int z_new;
      quant_pack_group<G, BITS>(x, st.zero_point, codes + (size_t)g * WPG * D + j, D, s_new, z_new);
      st.scale[((size_t)unit * NG + g) * D + j] = __float2bfloat16_rn(s_new);
      if (st.zero_point) st.zp[((size_t)unit * NG + g) * D + j] = (uint8_t)z_new;
    }
  }
}

// Per-warp shared memory: two unit stages, the work area, two mbarriers.
struct WarpPlan {
  UnitStage S;
  WarpSmem W;
  size_t stage0, stage1, work, bars, total;
};
__host__ __device__ inline WarpPlan warp_plan(int D, int G, int dP, int zp, int mixed, int io_f32, int any8) {
  WarpPlan p;
  p.S = unit_stage(D, G, dP, zp, mixed, io_f32, any8);
  p.W = warp_smem(D, dP, mixed);
  size_t off = 0;
  p.stage0 = carve(off, p.S.bytes, 128);
  p.stage1 = carve(off, p.S.bytes, 128);
  p.work = carve(off, p.W.total, 16);
  p.bars = carve(off, 16, 8);
  p.total = carve(off, 0, 128);
  return p;
}

// Issue the bulk copies of one unit into a stage (lane 0); returns a_t and beta_t of the unit for lane 0.
template <int D, int G>
__device__ __forceinline__ void issue_unit(const PaceDev &st, const PaceIO &io, int has_token, long u, int m0,
                                           unsigned char *stg, const UnitStage &SL, uint64_t *bar, float &an, float &bn) {
  constexpr int NG = D / G;
  const int dP = st.dP;
  const int mixed = st.buf_mode == PACE_BUF_MIXED;
  const uint32_t iob = st.io == PACE_IO_F32 ? 4u : 2u;
  const uint32_t rowk = mixed ? D / 2 : D, rowv = mixed ? 2 * D : D;
  const bool work = (m0 >= 0 && m0 < dP) && (has_token || m0 > 0);
  const int b = (int)(u / st.H), h = (int)(u - (long)b * st.H);
  const int is8 = st.head_is_int8[h];
  const uint32_t cbytes = is8 ? D * D : D * D / 2;
  const uint32_t sbytes = NG * D * 2, zbytes = st.zero_point ? NG * D : 0;
  uint32_t tx = 0;
  if (work) tx = cbytes + sbytes + zbytes + (uint32_t)m0 * (rowk + rowv + 16) + (has_token ? 3 * D * iob : 0);
  umma::fence_smem_to_async();                     // earlier generic reads of this stage come first
  mbar_arrive_expect_tx(bar, tx);
  if (work) {
    const uint32_t *codes = is8 ? st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D / 4) * D
                                : st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D / 8) * D;
    bulk_g2s(stg + SL.codes, codes, cbytes, bar);
    bulk_g2s(stg + SL.scales, st.scale + (size_t)u * NG * D, sbytes, bar);
    if (zbytes) bulk_g2s(stg + SL.zp, st.zp + (size_t)u * NG * D, zbytes, bar);
    if (m0 > 0) {
      bulk_g2s(stg + SL.bk, static_cast<const char *>(st.buf_k) + (size_t)u * dP * rowk, m0 * rowk, bar);
      bulk_g2s(stg + SL.bv, static_cast<const char *>(st.buf_v) + (size_t)u * dP * rowv, m0 * rowv, bar);
      bulk_g2s(stg + SL.bs, st.buf_s + (size_t)u * dP * 4, m0 * 16, bar);
    }
    if (has_token) {
      bulk_g2s(stg + SL.q, static_cast<const char *>(io.q) + (size_t)u * D * iob, D * iob, bar);
      bulk_g2s(stg + SL.k, static_cast<const char *>(io.k) + (size_t)u * D * iob, D * iob, bar);
      bulk_g2s(stg + SL.v, static_cast<const char *>(io.v) + (size_t)u * D * iob, D * iob, bar);
    }
  }
  if (has_token) {
    an = io.a[u];
    bn = io.beta[u];
  }
}

// Persistent kernel: warp w of the grid handles units w, w + W, w + 2W, ... (W warps in all). The next
// unit's bytes are copied into the other stage while the current unit computes.
template <int D, int G>
__global__ void __launch_bounds__(WU_WARPS * 32) decode_warp_kernel(const PaceDev st, const PaceIO io,
                                                                    const int has_token, const int any8) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WarpPlan P = warp_plan(D, G, st.dP, st.zero_point, st.buf_mode == PACE_BUF_MIXED, st.io == PACE_IO_F32, any8);
  unsigned char *base = smem + (size_t)warp * P.total;
  unsigned char *stage[2] = {base + P.stage0, base + P.stage1};
  uint64_t *bar = reinterpret_cast<uint64_t *>(base + P.bars);
  const WarpShared sh = warp_shared(base + P.work, P.W);
  const long units = (long)st.B * st.H;
  const long gw = (long)blockIdx.x * WU_WARPS + warp, nw = (long)gridDim.x * WU_WARPS;
  if (gw >= units) return;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  __syncwarp();
  // buffer counts of this warp's units, 32 at a time (lane n holds unit n of the batch)
  int mcur = 0, mnext = 0;
  {
    const long u0 = gw + (long)lane * nw, u1 = gw + (long)(32 + lane) * nw;
    mcur = u0 < units ? st.m[u0] : 0;
    mnext = u1 < units ? st.m[u1] : 0;
  }
  float an = 0.0f, bn = 0.0f, an_next = 0.0f, bn_next = 0.0f;
  if (lane == 0) issue_unit<D, G>(st, io, has_token, gw, mcur, stage[0], P.S, &bar[0], an, bn);  // lane 0 holds unit 0
  int n = 0;
  bool failed = false;
  for (;; ++n) {
    const long u = gw + (long)n * nw;
    if (u >= units) break;
    if (n > 0 && (n & 31) == 0) {                 // next batch of buffer counts
      mcur = mnext;
      const long u1 = gw + (long)(n + 32 + lane) * nw;
      mnext = u1 < units ? st.m[u1] : 0;
    }
    const int m0 = __shfl_sync(0xffffffffu, mcur, n & 31);
    const long un = u + nw;
    const int mn = __shfl_sync(0xffffffffu, ((n + 1) & 31) ? mcur : mnext, (n + 1) & 31);
    if (lane == 0 && un < units)
      issue_unit<D, G>(st, io, has_token, un, mn, stage[(n + 1) & 1], P.S, &bar[(n + 1) & 1], an_next, bn_next);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar[n & 1], (n >> 1) & 1, WU_WAIT_NS));
    if (!ok) {
      if (lane == 0) atomicOr(st.status, 1);
      failed = true;
      break;
    }
    const float a_u = __shfl_sync(0xffffffffu, an, 0), b_u = __shfl_sync(0xffffffffu, bn, 0);
    an = an_next;
    bn = bn_next;
    if (m0 < 0 || m0 >= st.dP) {                  // corrupted counter: leave the unit, emit zeros
      if (has_token) {
        float z[D / 32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) z[c] = 0.0f;
        store_io_vec<D / 32>(io.o, u * D + (D / 32) * lane, st.io, z);
      }
      continue;
    }
    if (!has_token && m0 == 0) continue;          // flush with nothing pending
    const int h = (int)(u % st.H);
    if (st.head_is_int8[h])
      warp_unit<D, G, 8>(st, io, u, m0, has_token, a_u, b_u, stage[n & 1], P.S, sh);
    else
      warp_unit<D, G, 4>(st, io, u, m0, has_token, a_u, b_u, stage[n & 1], P.S, sh);
    __syncwarp();
    if (lane == 0) st.m[u] = (!has_token || m0 + 1 == st.dP) ? 0 : m0 + 1;
  }
  if (failed && lane == 0) {
    // copies already issued for the following unit must land before the warp leaves
    const long un = gw + (long)(n + 1) * nw;
    if (un < units) mbar_wait(&bar[(n + 1) & 1], ((n + 1) >> 1) & 1, WU_WAIT_NS);
  }
}

template <int D, int G>
static cudaError_t launch_warp_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  auto kern = decode_warp_kernel<D, G>;
  const int any8 = d.H8 > 0;
  const WarpPlan plan = warp_plan(D, G, d.dP, d.zero_point, d.buf_mode == PACE_BUF_MIXED, d.io == PACE_IO_F32, any8);
  const size_t smem = (size_t)WU_WARPS * plan.total;
  static size_t opted = 0;
  static int sms = 0;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (smem > opted) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    opted = 227 * 1024;
  }
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const long units = (long)d.B * d.H;
  if (units == 0) return cudaSuccess;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, WU_WARPS * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  long blocks = (long)sms * per_sm;
  const long need = (units + WU_WARPS - 1) / WU_WARPS;
  if (blocks > need) blocks = need;
  kern<<<(unsigned)blocks, WU_WARPS * 32, smem, s>>>(d, io, has_token, any8);
  return cudaGetLastError();
}

}  // namespace pace

cudaError_t pace_launch_decode_quant(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.D == 128) return d.G == 64 ? launch_warp_t<128, 64>(d, io, has_token, s) : launch_warp_t<128, 32>(d, io, has_token, s);
  return d.G == 64 ? launch_warp_t<64, 64>(d, io, has_token, s) : launch_warp_t<64, 32>(d, io, has_token, s);
}
