// PACE decode step with fused flush on the 5th-generation tensor cores (tcgen05) -- the quantized path
// ([P1] 어떻게 동작하나: round once every dP tokens, buffered tokens applied together at the flush;
// [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// One CTA of 128 threads per unit (sequence b, head h); thread j owns state column j, which is also TMEM
// lane j of every accumulator, so per-column work (the replay recurrence, the output, the key-axis group
// requantization) stays inside one thread. Per call:
//   1. the buffered tokens 0..m-1 and (decode) the new token, quantized into slot m, are staged in shared
//      memory: int8 key codes (bf16 rows of the MMA B operand and int8 rows for the Gram products),
//      dequantized values, per-token scalars; q enters as two bf16 rows q_hi + q_lo (fp32 precision);
//   2. thread j reads its column's packed codes once and writes c = u - z as exact bf16 into TMEM lane j:
//      the A operand (state transposed, M = 128 columns x K = d_k keys);
//   3. one MMA chain per key-axis group g: D_g[j][v] = sum_{i in g} c_ij B[v][i], exact integers for the
//      int8 keys; then (S_hat^T k_v)_j = s_kv sum_g s_gj D_g[j][v] and (S_hat^T q)_j likewise;
//   4. the replay in reduced per-column form (thread-local, fp32):
//        u_t = beta_t (v_t - G_t (S_hat^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),   G_t = a_1 .. a_t
//        o   = G_m (S_hat^T q) + sum_s (G_m/G_s)(k_s.q) u_s
//   5. at a flush, a 128 x d_k fp32 accumulator in TMEM is set to G_m S_hat^T and the rank-m update
//        S_new^T += (rho u)^T K,   rho_s = (G_m/G_s) s_ks,
//      runs as one MMA chain with rho u split into three bf16 parts (hi + mid + lo, fp32-accurate) and the
//      int8 key codes as the other operand; thread j then requantizes column j group by group.
// Every mbarrier wait is bounded (1 s); on timeout the status word is set, TMEM is released and the
// kernel returns.
#include "pace_common.cuh"
#include "umma.cuh"

namespace pace {
using namespace umma;

constexpr uint64_t TC_WAIT_NS = 1000000000ull;

__host__ __device__ inline int tc_ntile(int dP) { return 16 * ((dP + 2 + 15) / 16); }   // B rows: keys + q_hi/q_lo
__host__ __device__ inline int tc_kflush(int dP) { return 16 * ((3 * dP + 15) / 16); }  // K of the flush MMA
__host__ __device__ inline int tc_cols(int D, int G, int dP) {
  int need = D / 2 + (D / G) * tc_ntile(dP);
  if (need < D) need = D;
  int c = 32;
  while (c < need) c <<= 1;
  return c;
}

struct TcSmem {
  size_t bdots, bflush, aflush, kq8, vf, P, U, qf, vscale, a, beta, gam, Dm, W, cq, ck, red, bar, tbase, total;
};

__host__ __device__ inline TcSmem tc_smem(int D, int dP) {
  TcSmem L;
  size_t off = 0;
  const size_t nt = tc_ntile(dP), kf = tc_kflush(dP);
  L.bdots = carve(off, nt * D * 2, 128);       // B of the dot MMAs: nt rows x D keys (bf16, K-major cores)
  L.bflush = carve(off, (size_t)D * kf * 2, 128);  // B of the flush MMA: D keys x kf (bf16)
  L.aflush = carve(off, 128 * kf * 2, 128);    // A of the flush MMA: 128 columns x kf (bf16)
  L.kq8 = carve(off, (size_t)dP * D);          // int8 key codes
  L.vf = carve(off, (size_t)dP * D * 4);
  L.P = carve(off, nt * 128 * 4);
  L.U = carve(off, (size_t)dP * 128 * 4);
  L.qf = carve(off, (size_t)D * 4);
  L.vscale = carve(off, nt * 4);
  L.a = carve(off, (size_t)dP * 4);
  L.beta = carve(off, (size_t)dP * 4);
  L.gam = carve(off, (size_t)dP * 4);
  L.Dm = carve(off, (size_t)dP * dP * 4);
  L.W = carve(off, (size_t)dP * dP * 4);
  L.cq = carve(off, (size_t)dP * 4);
  L.ck = carve(off, (size_t)dP * 4);
  L.red = carve(off, 32 * 4);
  L.bar = carve(off, 8, 8);
  L.tbase = carve(off, 4);
  L.total = carve(off, 0);
  return L;
}

// Byte offset of element (row r, k) in a K-major operand of `kdim` columns made of 8 x 16-byte cores:
// cores along K are adjacent (128 B apart), 8-row groups are kdim/8 * 128 B apart.
__device__ __forceinline__ uint32_t core_off(int r, int k, int kdim) {
  return (uint32_t)((r >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

struct TcShared {
  unsigned char *bdots, *bflush, *aflush;
  int8_t *kq8;
  float *vf, *P, *U, *qf, *vscale, *a, *beta, *gam, *Dm, *W, *cq, *ck, *red;
  uint64_t *bar;
  uint32_t *tbase;
};

__device__ inline TcShared tc_shared(unsigned char *base, const TcSmem &L) {
  TcShared s;
  s.bdots = base + L.bdots;
  s.bflush = base + L.bflush;
  s.aflush = base + L.aflush;
  s.kq8 = reinterpret_cast<int8_t *>(base + L.kq8);
  s.vf = reinterpret_cast<float *>(base + L.vf);
  s.P = reinterpret_cast<float *>(base + L.P);
  s.U = reinterpret_cast<float *>(base + L.U);
  s.qf = reinterpret_cast<float *>(base + L.qf);
  s.vscale = reinterpret_cast<float *>(base + L.vscale);
  s.a = reinterpret_cast<float *>(base + L.a);
  s.beta = reinterpret_cast<float *>(base + L.beta);
  s.gam = reinterpret_cast<float *>(base + L.gam);
  s.Dm = reinterpret_cast<float *>(base + L.Dm);
  s.W = reinterpret_cast<float *>(base + L.W);
  s.cq = reinterpret_cast<float *>(base + L.cq);
  s.ck = reinterpret_cast<float *>(base + L.ck);
  s.red = reinterpret_cast<float *>(base + L.red);
  s.bar = reinterpret_cast<uint64_t *>(base + L.bar);
  s.tbase = reinterpret_cast<uint32_t *>(base + L.tbase);
  return s;
}

// Stage the buffered tokens 0..m0-1 and (decode) the new token into shared memory; thread i handles key
// (and value channel) i. B rows: 0..mt-1 keys, mt / mt+1 q_hi / q_lo (decode), zero up to nt.
template <int D>
__device__ void tc_stage(const PaceDev &st, const PaceIO &io, long unit, int m0, int has_token, int nt,
                         const TcShared &sh) {
  const int i = threadIdx.x;
  const int dP = st.dP;
  const float *bs = st.buf_s + unit * dP * 4;
  if (i < m0) {
    sh.a[i] = bs[i * 4 + 0];
    sh.beta[i] = bs[i * 4 + 1];
    sh.vscale[i] = bs[i * 4 + 2];
  }
  float kx = 0.0f, vx = 0.0f, qx = 0.0f;
  if (has_token && i < D) {
    kx = load_io(io.k, unit * D + i, st.io);
    vx = load_io(io.v, unit * D + i, st.io);
    qx = load_io(io.q, unit * D + i, st.io);
  }
  if (i < D) {
    if (st.buf_mode == PACE_BUF_MIXED) {
      const uint8_t *bk = static_cast<const uint8_t *>(st.buf_k) + unit * dP * (D / 2);
      const __nv_bfloat16 *bv = static_cast<const __nv_bfloat16 *>(st.buf_v) + unit * dP * D;
      for (int t = 0; t < m0; ++t) {
        const uint32_t byte = bk[t * (D / 2) + (i >> 1)];
        sh.kq8[t * D + i] = (int8_t)((int)((byte >> ((i & 1) * 4)) & 0xF) - 8);
        sh.vf[t * D + i] = __bfloat162float(bv[t * D + i]);
      }
    } else {
      const int8_t *bk = static_cast<const int8_t *>(st.buf_k) + unit * dP * D;
      const int8_t *bv = static_cast<const int8_t *>(st.buf_v) + unit * dP * D;
      for (int t = 0; t < m0; ++t) {
        sh.kq8[t * D + i] = bk[t * D + i];
        sh.vf[t * D + i] = bs[t * 4 + 3] * (float)bv[t * D + i];
      }
    }
  }
  if (has_token) {
    float sk, sv = 0.0f;
    int ck;
    if (st.buf_mode == PACE_BUF_MIXED) {
      const float Ak = block_max(fabsf(kx), sh.red);
      ck = buffer_code(kx, Ak, 7);
      sk = buffer_scale(Ak, 7);
      const int nb = __shfl_down_sync(0xffffffffu, ck, 1);
      if (i < D) {
        sh.kq8[m0 * D + i] = (int8_t)ck;
        sh.vf[m0 * D + i] = bf16_round(vx);
        if ((i & 1) == 0)
          static_cast<uint8_t *>(st.buf_k)[(unit * dP + m0) * (D / 2) + (i >> 1)] =
              (uint8_t)((ck + 8) | ((nb + 8) << 4));
        static_cast<__nv_bfloat16 *>(st.buf_v)[(unit * dP + m0) * D + i] = __float2bfloat16_rn(vx);
      }
    } else {
      const float Ak = block_max(fabsf(kx), sh.red);
      const float Av = block_max(fabsf(vx), sh.red);
      ck = buffer_code(kx, Ak, 127);
      const int cv = buffer_code(vx, Av, 127);
      sk = buffer_scale(Ak, 127);
      sv = buffer_scale(Av, 127);
      if (i < D) {
        sh.kq8[m0 * D + i] = (int8_t)ck;
        sh.vf[m0 * D + i] = sv * (float)cv;
        static_cast<int8_t *>(st.buf_k)[(unit * dP + m0) * D + i] = (int8_t)ck;
        static_cast<int8_t *>(st.buf_v)[(unit * dP + m0) * D + i] = (int8_t)cv;
      }
    }
    if (i == 0) {
      const float ax = io.a[unit], bx = io.beta[unit];
      sh.a[m0] = ax;
      sh.beta[m0] = bx;
      sh.vscale[m0] = sk;
      float *bw = st.buf_s + (unit * dP + m0) * 4;
      bw[0] = ax;
      bw[1] = bx;
      bw[2] = sk;
      bw[3] = sv;
      sh.vscale[m0 + 1] = 1.0f;
      sh.vscale[m0 + 2] = 1.0f;
    }
    if (i < D) sh.qf[i] = qx;
  }
  __syncthreads();
  // bf16 B rows of the dot MMAs (column i of every row)
  if (i < D) {
    const int mt = m0 + has_token;
    for (int r = 0; r < nt; ++r) {
      float x = 0.0f;
      if (r < mt) {
        x = (float)sh.kq8[r * D + i];
      } else if (has_token && r == mt) {
        x = bf16_round(qx);
      } else if (has_token && r == mt + 1) {
        x = qx - bf16_round(qx);
      }
      *reinterpret_cast<uint16_t *>(sh.bdots + core_off(r, i, D)) = bf16_bits(x);
    }
  }
}

// Decay products, Gram coefficients, readout and flush coefficients shared by all columns (4 warps).
template <int D>
__device__ void tc_tables(int mt, int has_token, int dP, const TcShared &sh) {
  const int j = threadIdx.x, lane = j & 31, wid = j >> 5;
  constexpr int NW = 4;
  if (j < mt) {                                   // Dm[j][t] = a_{j+1} .. a_t
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
  int item = 0;
  for (int t = 1; t < mt; ++t) {
    for (int s = 0; s < t; ++s, ++item) {
      if ((item & (NW - 1)) != wid) continue;
      int acc = 0;
      if (lane < D / 4) {
        const int *ks = reinterpret_cast<const int *>(sh.kq8 + s * D);
        const int *kt = reinterpret_cast<const int *>(sh.kq8 + t * D);
        acc = dp4a_ss(ks[lane], kt[lane], 0);
      }
      const float dot = sh.vscale[s] * sh.vscale[t] * (float)__reduce_add_sync(0xffffffffu, acc);
      if (lane == 0) sh.W[t * dP + s] = sh.Dm[s * dP + t] * dot;
    }
  }
  for (int s = wid; s < mt; s += NW) {
    float acc = 0.0f;
    if (has_token) {
#pragma unroll
      for (int r = 0; r < D / 32; ++r) {
        const int i = r * 32 + lane;
        acc += (float)sh.kq8[s * D + i] * sh.qf[i];
      }
      acc = warp_sum(acc);
    }
    if (lane == 0) {
      sh.cq[s] = sh.Dm[s * dP + (mt - 1)] * sh.vscale[s] * acc;
      sh.ck[s] = sh.Dm[s * dP + (mt - 1)] * sh.vscale[s];
    }
  }
}

// A operand (column j of the state, transposed) into TMEM lane j: c = u - z as exact bf16, keys in order.
template <int D, int G, int BITS>
__device__ __forceinline__ void tc_write_A(uint32_t taddr, const uint32_t *wr, const int *zg, bool col) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {              // 16 TMEM columns = 32 keys per chunk
    uint32_t r[16];
    if (BITS == 4) {
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        const int w = 4 * c + ww;
        const uint32_t wd = col ? wr[w] : 0u;
        const int z = col ? zg[(8 * w) / G] : 0;
        const __nv_bfloat162 zz = __floats2bfloat162_rn(128.0f + z, 128.0f + z);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t x = ((wd >> (4 * s)) & 0x000F000Fu) | 0x43004300u;   // bf16 pair (128 + u, 128 + u')
          __nv_bfloat162 xb = *reinterpret_cast<__nv_bfloat162 *>(&x);
          __nv_bfloat162 cb = __hsub2(xb, zz);
          r[4 * ww + s] = col ? *reinterpret_cast<uint32_t *>(&cb) : 0u;
        }
      }
    } else {
#pragma unroll
      for (int ww = 0; ww < 8; ++ww) {
        const int w = 8 * c + ww;
        const uint32_t wd = col ? wr[w] : 0u;
        const int z = col ? zg[(4 * w) / G] : 0;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float c0 = (float)((int)byte_of(wd, 2 * p) - z);
          const float c1 = (float)((int)byte_of(wd, 2 * p + 1) - z);
          __nv_bfloat162 cb = __floats2bfloat162_rn(c0, c1);
          r[2 * ww + p] = col ? *reinterpret_cast<uint32_t *>(&cb) : 0u;
        }
      }
    }
    tmem_st16(taddr + 16 * c, r);
  }
}

// Flush accumulator init: G_m * s_g * (u - z) for every key of column j, fp32, keys in order.
template <int D, int G, int BITS>
__device__ __forceinline__ void tc_write_init(uint32_t taddr, const uint32_t *wr, const float *sg, const int *zg,
                                              float gm, bool col) {
  constexpr int KPW = 32 / BITS;
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    uint32_t r[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int i = 16 * c + t;
      const int g = i / G;
      float x = 0.0f;
      if (col) {
        const uint32_t wd = wr[i / KPW];
        const uint32_t u = BITS == 4 ? nibble_of(wd, i % KPW) : byte_of(wd, i % KPW);
        x = gm * (sg[g] * (float)((int)u - zg[g]));
      }
      r[t] = __float_as_uint(x);
    }
    tmem_st16(taddr + 16 * c, r);
  }
}

template <int D, int G, int BITS>
__device__ void tc_unit(const PaceDev &st, const PaceIO &io, long unit, int b, int h, int m0, int has_token,
                        const TcShared &sh) {
  constexpr int KPW = 32 / BITS, NWC = D / KPW, NG = D / G, WPG = G / KPW;
  const int j = threadIdx.x, warp = j >> 5;
  const bool col = j < D;
  const int dP = st.dP, nt = tc_ntile(dP), kf = tc_kflush(dP), ncols = tc_cols(D, G, dP);
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 2 : 0);

  // packed codes of column j (issued first; consumed after staging)
  const int slot = st.head_slot[h];
  uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + slot) * NWC * D
                              : st.codes8 + (size_t)(b * st.H8 + slot) * NWC * D;
  uint32_t wr[NWC];
  float sg[NG];
  int zg[NG];
#pragma unroll
  for (int w = 0; w < NWC; ++w) wr[w] = col ? codes[w * D + j] : 0u;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    sg[g] = col ? __bfloat162float(st.scale[(unit * NG + g) * D + j]) : 0.0f;
    zg[g] = (col && st.zero_point) ? (int)st.zp[(unit * NG + g) * D + j] : (1 << (BITS - 1));
  }

  if (warp == 0) {
    tmem_alloc(sh.tbase, (uint32_t)ncols);
    tmem_relinquish();
  }
  if (j == 0) {
    mbar_init(sh.bar, 1);
    mbar_fence_init();
  }
  tc_stage<D>(st, io, unit, m0, has_token, nt, sh);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *sh.tbase;
  const uint32_t lanes = (uint32_t)(warp * 32) << 16;

  // ---- A operand, then the dot-product MMAs (one chain per key-axis group)
  tc_write_A<D, G, BITS>(tmem + lanes, wr, zg, col);
  tmem_wait_st();
  fence_smem_to_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (j == 0) {
    const uint32_t idesc = idesc_bf16(128, nt);
    const uint32_t bbase = smem_u32(sh.bdots);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int s = 0; s < G / 16; ++s) {
        const int kk = g * (G / 16) + s;
        mma_ts(tmem + D / 2 + g * nt, tmem + kk * 8, smem_desc(bbase + kk * 256, 128, (D / 8) * 128), idesc,
               s > 0 ? 1u : 0u);
      }
    commit(sh.bar);
  }
  tc_tables<D>(mt, has_token, dP, sh);
  __syncthreads();
  uint32_t waiting = 0;                           // mbarrier phase being waited for
  bool ok = mbar_wait(sh.bar, waiting, TC_WAIT_NS);
  fence_after_sync();

  if (ok) {
    // ---- P[v][j] = vscale_v * sum_g s_g D_g[j][v]
    for (int c = 0; c * 16 < nv; ++c) {
      float acc[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[t] = 0.0f;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        uint32_t r[16];
        tmem_ld16(tmem + lanes + D / 2 + g * nt + 16 * c, r);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[t] = fmaf(sg[g], __uint_as_float(r[t]), acc[t]);
      }
      if (col) {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const int v = 16 * c + t;
          if (v < nv) sh.P[v * 128 + j] = acc[t] * sh.vscale[v];
        }
      }
    }
    // ---- replay recurrence and readout (thread-local per column)
    if (col) {
      for (int t = 0; t < mt; ++t) {
        float acc = sh.vf[t * D + j] - sh.gam[t] * sh.P[t * 128 + j];
        for (int s = 0; s < t; ++s) acc = fmaf(-sh.W[t * dP + s], sh.U[s * 128 + j], acc);
        sh.U[t * 128 + j] = sh.beta[t] * acc;
      }
      if (has_token) {
        const float R = sh.P[mt * 128 + j] + sh.P[(mt + 1) * 128 + j];
        float o = sh.gam[mt - 1] * R;
        for (int s = 0; s < mt; ++s) o = fmaf(sh.cq[s], sh.U[s * 128 + j], o);
        store_io(io.o, unit * D + j, o, st.io);
      }
    }
  }

  if (ok && do_flush) {
    // ---- flush operands: A[j][3s+p] = part p of rho_s u_s,j ; B[i][3s+p] = key code k_s,i
    for (int kk = 0; kk < kf; ++kk) {
      const int s = kk / 3, p = kk - 3 * s;
      float x = 0.0f;
      if (col && s < mt) {
        const float y = sh.ck[s] * sh.U[s * 128 + j];
        const float hi = bf16_round(y);
        const float mid = bf16_round(y - hi);
        x = p == 0 ? hi : (p == 1 ? mid : bf16_round(y - hi - mid));
      }
      *reinterpret_cast<uint16_t *>(sh.aflush + core_off(j, kk, kf)) = bf16_bits(x);
      if (col) {
        const float kc = s < mt ? (float)sh.kq8[s * D + j] : 0.0f;
        *reinterpret_cast<uint16_t *>(sh.bflush + core_off(j, kk, kf)) = bf16_bits(kc);
      }
    }
    // accumulator init G_m S_hat^T (TMEM columns 0..D-1; the dot operands there are consumed)
    tc_write_init<D, G, BITS>(tmem + lanes, wr, sg, zg, sh.gam[mt - 1], col);
    tmem_wait_st();
    fence_smem_to_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (j == 0) {
      const uint32_t idesc = idesc_bf16(128, D);
      const uint32_t abase = smem_u32(sh.aflush), bbase = smem_u32(sh.bflush);
      for (int s = 0; s < kf / 16; ++s)
        mma_ss(tmem, smem_desc(abase + s * 256, 128, (kf / 8) * 128), smem_desc(bbase + s * 256, 128, (kf / 8) * 128),
               idesc, 1u);
      commit(sh.bar);
    }
    __syncwarp();
    waiting = 1;
    ok = mbar_wait(sh.bar, waiting, TC_WAIT_NS);
    fence_after_sync();
    if (ok && col) {
      // ---- requantize column j, group by group
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        float x[G];
#pragma unroll
        for (int cc = 0; cc < G / 16; ++cc) {
          uint32_t r[16];
          tmem_ld16(tmem + lanes + g * G + 16 * cc, r);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 16; ++t) x[16 * cc + t] = __uint_as_float(r[t]);
        }
        uint32_t uq[G];
        float s_new;
        int z_new;
        quant_group<G, BITS>(x, st.zero_point, uq, s_new, z_new);
#pragma unroll
        for (int ww = 0; ww < WPG; ++ww)
          codes[(g * WPG + ww) * D + j] = BITS == 4 ? pack_nibbles(uq + 8 * ww) : pack_bytes(uq + 4 * ww);
        st.scale[(unit * NG + g) * D + j] = __float2bfloat16_rn(s_new);
        if (st.zero_point) st.zp[(unit * NG + g) * D + j] = (uint8_t)z_new;
      }
    }
  }
  if (!ok) {
    if (j == 0) atomicOr(st.status, 1);
    mbar_wait(sh.bar, waiting, TC_WAIT_NS);       // let in-flight MMAs drain before releasing TMEM
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)ncols);
  if (j == 0 && ok) st.m[unit] = do_flush ? 0 : mt;
}

template <int D, int G>
__global__ void __launch_bounds__(128) decode_tc_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const TcShared sh = tc_shared(smem, tc_smem(D, st.dP));
  const long unit = blockIdx.x;
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const int m0 = st.m[unit];
  if (m0 < 0 || m0 >= st.dP) {                    // corrupted counter: leave the unit, emit zeros
    if (has_token && threadIdx.x < D) store_io(io.o, unit * D + threadIdx.x, 0.0f, st.io);
    return;
  }
  if (!has_token && m0 == 0) return;              // flush with nothing pending
  if (st.head_is_int8[h])
    tc_unit<D, G, 8>(st, io, unit, b, h, m0, has_token, sh);
  else
    tc_unit<D, G, 4>(st, io, unit, b, h, m0, has_token, sh);
}

// Dynamic shared memory per CTA: what the kernel uses, raised so that no more CTAs fit on an SM than
// its 512 TMEM columns can serve (a CTA beyond that would wait inside the allocation).
inline size_t tc_launch_smem(int D, int G, int dP) {
  const size_t need = tc_smem(D, dP).total;
  const int per_sm = 512 / tc_cols(D, G, dP);
  const size_t floor_bytes = (size_t)(228 * 1024) / (size_t)(per_sm + 1) + 1024;
  return need > floor_bytes ? need : floor_bytes;
}

template <int D, int G>
static cudaError_t launch_tc_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  auto kern = decode_tc_kernel<D, G>;
  const size_t smem = tc_launch_smem(D, G, d.dP);
  static size_t opted = 0;
  if (smem > opted) {
    const size_t most = 200 * 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    opted = most;
  }
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  kern<<<units, 128, smem, s>>>(d, io, has_token);
  return cudaGetLastError();
}

}  // namespace pace

cudaError_t pace_launch_decode_tc(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.D == 128) return d.G == 64 ? launch_tc_t<128, 64>(d, io, has_token, s) : launch_tc_t<128, 32>(d, io, has_token, s);
  return d.G == 64 ? launch_tc_t<64, 64>(d, io, has_token, s) : launch_tc_t<64, 32>(d, io, has_token, s);
}
