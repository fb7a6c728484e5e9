// Decode step and flush of the two states kept in plain floating point, on PACE's periodic schedule
// ([P1] 어떻게 동작하나):
//   - the unquantized test mode (fp32 state, fp32 decode buffer): the rounding left out, to check the replay
//     arithmetic to 1e-4 against the exact recurrence;
//   - the buffered bf16 state ([P1] 전제와 한계: most of the TPOT gain of periodic rounding comes from the decode
//     buffer with a bf16 state): bf16 state rounded once every dP tokens, int8 decode buffer as in PACE-4.
// One CTA per unit, one thread per column j; the state is streamed from global memory. The buffered tokens
// are replayed in the reduced per-column form
//   u_t = beta_t (v_t - G_t (S^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),  G_t = a_1 .. a_t,
//   o   = G_m (S^T q) + sum_s (G_m/G_s)(k_s.q) u_s,
// and a flush writes S_new = G_m S + sum_s (G_m/G_s) k_s u_s^T.
#include <algorithm>

#include "pace_common.cuh"

namespace pace {

constexpr int VCHUNK = 8;   // dot-product vectors handled per pass over the codes


struct DecodeSmem {
  size_t kq, keyf, vf, P, U, kf, csum, vscale, a, beta, gam, Dm, W, cq, ck, red, qf, ah, Ss, total;
};

// Rows of the tensor-core dot products of the buffered bf16 state: the mt key codes, then q as three bf16
// parts, padded to whole 16-row tiles.
__host__ __device__ inline int dec_arows(int dP) { return 16 * ((dP + 3 + 15) / 16); }

__host__ __device__ inline DecodeSmem decode_smem(int D, int dP, int fp32mode) {
  DecodeSmem L;
  size_t off = 0;
  L.kq = carve(off, (size_t)(dP + 2) * D);                     // int8 key codes (+ q halves)
  L.keyf = carve(off, fp32mode ? (size_t)(dP + 1) * D * 4 : 0); // fp32 keys (+ q), fp32 mode
  L.vf = carve(off, (size_t)dP * D * 4);                       // dequantized values
  L.P = carve(off, (size_t)(dP + 3) * D * 4);                  // S^T k_tau, S^T q (bf16 state: 3 q parts)
  // u_tau per column; the bf16 state's bf16 rows (keys, q parts) share it, being done with before the replay
  const size_t ub = (size_t)dP * D * 4, ab = (size_t)dec_arows(dP) * D * 2;
  L.U = carve(off, fp32mode || ub >= ab ? ub : ab);
  L.kf = carve(off, fp32mode ? (size_t)dP * D * 4 : 0);         // fp32 mode: flush coefficients x keys
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
  L.ah = fp32mode ? carve(off, 0) : L.U;                       // bf16 state: bf16 rows (keys, q parts)
  L.Ss = carve(off, fp32mode ? 0 : (size_t)D * D * 2, 128);           // bf16 state: the unit's state, staged
  L.total = carve(off, 0);
  return L;
}

struct DecodeShared {
  int8_t *kq;
  float *keyf, *vf, *P, *U, *kf;
  int *csum;
  float *vscale, *a, *beta, *gam, *Dm, *W, *cq, *ck, *red, *qf;
  __nv_bfloat16 *ah, *Ss;
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
  s.ah = reinterpret_cast<__nv_bfloat16 *>(base + L.ah);
  s.Ss = reinterpret_cast<__nv_bfloat16 *>(base + L.Ss);
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
  {
    const float *bk = static_cast<const float *>(st.buf_k) + unit * dP * D;
    const float *bv = static_cast<const float *>(st.buf_v) + unit * dP * D;
    for (int t = 0; t < m0; ++t) {
      sh.keyf[t * D + j] = bk[t * D + j];
      sh.vf[t * D + j] = bv[t * D + j];
    }
  }
}

// Store the new token in buffer slot m0 (shared and global), and stage q.
template <int D>
__device__ void append_token(const PaceDev &st, const PaceIO &io, long unit, int m0, const DecodeShared &sh) {
  const int j = threadIdx.x;
  const int dP = st.dP;
  const float kx = load_io(io.k, unit * D + j, st.io);
  const float vx = load_io(io.v, unit * D + j, st.io);
  const float qx = load_io(io.q, unit * D + j, st.io);
  sh.qf[j] = qx;
  const float sk = 1.0f, sv = 1.0f;
  {
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
  sh.keyf[(m0 + 1) * D + j] = qx;            // q follows the keys
}

// Buffered bf16 state: the copies of buffered tokens 0..m0-1 in flight at once (int8 key codes straight into
// their rows, value codes into a byte staging area), and their scalars (a, beta, key scale; the value scale
// parked in cq until the values are converted).
template <int D>
__device__ void issue_buffer_i8(const PaceDev &st, long unit, int m0, const DecodeShared &sh, int8_t *vstage) {
  const int j = threadIdx.x, dP = st.dP;
  const char *bk = static_cast<const char *>(st.buf_k) + unit * dP * D;
  const char *bv = static_cast<const char *>(st.buf_v) + unit * dP * D;
  for (int c = j; c < m0 * D / 16; c += D) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(sh.kq + 16 * c)),
                 "l"(bk + 16 * c) : "memory");
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(vstage + 16 * c)),
                 "l"(bv + 16 * c) : "memory");
  }
  if (j < m0) {
    const float4 r = *reinterpret_cast<const float4 *>(st.buf_s + (unit * dP + j) * 4);
    sh.a[j] = r.x;
    sh.beta[j] = r.y;
    sh.vscale[j] = r.z;
    sh.cq[j] = r.w;
  }
}

// Buffered bf16 state: quantize the new token into slot m0 ([P1] 어떻게 동작하나: int8 keys and values, one
// fp32 scale each), in shared and global memory, and stage q.
template <int D>
__device__ void append_token_i8(const PaceDev &st, const PaceIO &io, long unit, int m0, const DecodeShared &sh,
                                float kx, float vx, float qx) {
  const int j = threadIdx.x;
  const int dP = st.dP;
  sh.qf[j] = qx;
  const float Ak = block_max(fabsf(kx), sh.red);
  const float Av = block_max(fabsf(vx), sh.red + 32 - D / 32);
  const int kc = buffer_code(kx, Ak, 127), vc = buffer_code(vx, Av, 127);
  const float sk = buffer_scale(Ak, 127), sv = buffer_scale(Av, 127);
  sh.kq[m0 * D + j] = (int8_t)kc;
  sh.vf[m0 * D + j] = sv * (float)vc;
  static_cast<int8_t *>(st.buf_k)[(unit * dP + m0) * D + j] = (int8_t)kc;
  static_cast<int8_t *>(st.buf_v)[(unit * dP + m0) * D + j] = (int8_t)vc;
  if (j == 0) {
    const float ax = io.a[unit], bx = io.beta[unit];
    sh.a[m0] = ax;
    sh.beta[m0] = bx;
    sh.vscale[m0] = sk;
    *reinterpret_cast<float4 *>(st.buf_s + (unit * dP + m0) * 4) = make_float4(ax, bx, sk, sv);
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
                           int qrows, const DecodeShared &sh) {
  const int j = threadIdx.x;
  const int dP = st.dP;
  for (int t = 0; t < mt; ++t) {
    float acc = sh.vf[t * D + j] - sh.gam[t] * sh.P[t * D + j];
    for (int s = 0; s < t; ++s) acc = fmaf(-sh.W[t * dP + s], sh.U[s * D + j], acc);
    sh.U[t * D + j] = sh.beta[t] * acc;
  }
  if (has_token) {
    const float R = qrows == 1 ? sh.P[mt * D + j] : sh.P[mt * D + j] + (sh.P[(mt + 1) * D + j] + sh.P[(mt + 2) * D + j]);
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

// Element (i, j) of the staged bf16 state: rows of D values, 16-byte chunks XOR-swizzled by the row, so that
// the eight rows of an ldmatrix tile fall in distinct banks.
template <int D>
__device__ __forceinline__ int ss_off(int i, int j) { return i * D + ((((j >> 3) ^ (i & 7)) << 3) | (j & 7)); }

__device__ __forceinline__ void bb_ldsm_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"((uint32_t)__cvta_generic_to_shared(p)) : "memory");
}
__device__ __forceinline__ void bb_ldsm_x4_trans(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"((uint32_t)__cvta_generic_to_shared(p)) : "memory");
}
__device__ __forceinline__ void bb_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Buffered bf16 state: the dot products P[v][j] = sum_i A[v][i] S[i][j] on the tensor cores (bf16 MMA, fp32
// accumulation) with A = the key codes of the mt buffered tokens (exact in bf16) and q as three bf16 parts
// (q0 + q1 + q2 = q to 24 bits), B = the unit's state staged in shared memory (ldmatrix.trans); warp w takes
// the 32 columns 32w.., one 16-row tile of A at a time. Then the replay and, at a rounding,
// S_new = G_m S + sum_s (G_m/G_s) k_s u_s^T written back to global memory as bf16.
template <int D>
__device__ void bf16_column(const PaceDev &st, const PaceIO &io, long unit, int mt, int has_token, int do_flush,
                            const DecodeShared &sh) {
  const int j = threadIdx.x, lane = j & 31, w = j >> 5;
  const int g8 = lane >> 2, tq = lane & 3;
  __nv_bfloat16 *Sp = static_cast<__nv_bfloat16 *>(st.S) + unit * D * D;
  const __nv_bfloat16 *Ss = sh.Ss;
  const int nr = mt + (has_token ? 3 : 0);       // rows of A in use
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = lane >> 4;   // ldmatrix x4: A row, 8-key chunk
  const int bkey = (lane & 7) + 8 * ((lane >> 3) & 1), bchk = lane >> 4;   // ldmatrix x4.trans: key, column chunk
  for (int vt = 0; vt < (nr + 15) / 16; ++vt) {
    float acc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[n][e] = 0.0f;
#pragma unroll 4
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      bb_ldsm_x4(a, sh.ah + ss_off<D>(16 * vt + arow, 16 * ks + 8 * acol));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t b[4];
        bb_ldsm_x4_trans(b, Ss + ss_off<D>(16 * ks + bkey, 32 * w + 16 * h + 8 * bchk));
        bb_mma(acc[2 * h], a, b[0], b[1]);
        bb_mma(acc[2 * h + 1], a, b[2], b[3]);
      }
    }
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int col = 32 * w + 8 * n + 2 * tq;
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int v = 16 * vt + g8 + 8 * hi;
        if (v < nr) {
          const float sc = v < mt ? sh.vscale[v] : 1.0f;   // key codes times the key scale; q parts as they are
          *reinterpret_cast<float2 *>(sh.P + v * D + col) = make_float2(sc * acc[n][2 * hi], sc * acc[n][2 * hi + 1]);
        }
      }
    }
  }
  __syncthreads();
  recurrence<D>(st, io, unit, nr, mt, has_token, 3, sh);
  if (!do_flush) return;
  const float gm = sh.gam[mt - 1];
  for (int i = 0; i < D; ++i) {                   // (G_m/G_s) s_ks k_s,i formed on the fly: one rounding, as stored
    float x = gm * __bfloat162float(Ss[ss_off<D>(i, j)]);
    for (int s2 = 0; s2 < mt; ++s2) x = fmaf(sh.ck[s2] * (float)sh.kq[s2 * D + i], sh.U[s2 * D + j], x);
    Sp[i * D + j] = __float2bfloat16_rn(x);
  }
}

// Buffered bf16 state: one decode step (or a flush) of one unit.
template <int D>
__global__ void __launch_bounds__(D) decode_bf16buf_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_enter();
  const long unit = blockIdx.x;
  const DecodeSmem L = decode_smem(D, st.dP, 0);
  const DecodeShared sh = decode_shared(smem, L);
  const int j = threadIdx.x;
  {                                               // the unit's bf16 state, all copies in flight at once
    const char *src = reinterpret_cast<const char *>(static_cast<const __nv_bfloat16 *>(st.S) + unit * D * D);
    char *dst = reinterpret_cast<char *>(sh.Ss);
    for (int c = j; c < D * D * 2 / 16; c += D) {  // 16-byte chunk c = (row i, chunk cc), swizzled
      const int i = c / (D / 8), cc = c - i * (D / 8);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                   ::"r"((uint32_t)__cvta_generic_to_shared(dst + 16 * (i * (D / 8) + (cc ^ (i & 7))))),
                   "l"(src + 16 * c) : "memory");
    }
  }
  const int m0 = st.m[unit];
  float kx = 0.0f, vx = 0.0f, qx = 0.0f;          // the new token, in flight with the count
  if (has_token) {
    kx = load_io(io.k, unit * D + j, st.io);
    vx = load_io(io.v, unit * D + j, st.io);
    qx = load_io(io.q, unit * D + j, st.io);
  }
  if (m0 < 0 || m0 >= st.dP || (!has_token && m0 == 0)) {
    asm volatile("cp.async.wait_all;" ::: "memory");   // nothing may land in shared memory after the CTA leaves
    if (has_token && m0 != 0) store_io(io.o, unit * D + j, 0.0f, st.io);   // corrupted counter: emit zeros
    return;                                       // (or a flush with nothing pending)
  }
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == st.dP;
  int8_t *vstage = reinterpret_cast<int8_t *>(sh.U);    // (the bf16 rows and the replay use it later)
  issue_buffer_i8<D>(st, unit, m0, sh, vstage);
  if (has_token) append_token_i8<D>(st, io, unit, m0, sh, kx, vx, qx);
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  for (int t = 0; t < m0; ++t) sh.vf[t * D + j] = sh.cq[t] * (float)vstage[t * D + j];
  __syncthreads();                                // the staged value codes are read before the rows overwrite them
  {                                               // bf16 rows of A: key codes, q in three parts, zeros
    const int rows = dec_arows(st.dP);
    for (int item = j; item < rows * (D / 8); item += D) {
      const int v = item / (D / 8), k8 = 8 * (item - v * (D / 8));
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x0 = 0.0f, x1 = 0.0f;
        if (v < mt) {
          x0 = (float)sh.kq[v * D + k8 + 2 * e];
          x1 = (float)sh.kq[v * D + k8 + 2 * e + 1];
        } else if (has_token && v < mt + 3) {
          float q0 = sh.qf[k8 + 2 * e], q1 = sh.qf[k8 + 2 * e + 1];
          for (int p = 0; p < v - mt; ++p) {           // the part's remainder: q - (earlier parts)
            q0 -= bf16_round(q0);
            q1 -= bf16_round(q1);
          }
          x0 = q0;
          x1 = q1;
        }
        const __nv_bfloat162 pr = __floats2bfloat162_rn(x0, x1);
        wv[e] = *reinterpret_cast<const uint32_t *>(&pr);
      }
      *reinterpret_cast<uint4 *>(sh.ah + ss_off<D>(v, k8)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  }
  unit_tables<D>(mt, has_token, 0, st.dP, sh);
  __syncthreads();
  bf16_column<D>(st, io, unit, mt, has_token, do_flush, sh);
  if (j == 0) st.m[unit] = do_flush ? 0 : mt;
}

template <int D>
__global__ void __launch_bounds__(D) decode_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(16) unsigned char smem[];
  pdl_enter();
  const long unit = blockIdx.x;
  const DecodeSmem L = decode_smem(D, st.dP, 1);
  const DecodeShared sh = decode_shared(smem, L);

  const int m0 = st.m[unit];
  if (m0 < 0 || m0 >= st.dP) {                    // corrupted counter: leave the unit, emit zeros
    if (has_token) store_io(io.o, unit * D + threadIdx.x, 0.0f, st.io);
    return;
  }
  if (!has_token && m0 == 0) return;              // flush with nothing pending
  const int mt = m0 + has_token;                  // tokens replayed
  const int do_flush = !has_token || mt == st.dP;
  const int nv = mt + has_token;                  // keys, then q

  load_buffer<D>(st, unit, m0, sh);
  if (has_token) append_token<D>(st, io, unit, m0, sh);
  __syncthreads();
  unit_tables<D>(mt, has_token, 1, st.dP, sh);
  __syncthreads();
  fp32_column<D>(st, io, unit, nv, mt, has_token, do_flush, sh);
  if (threadIdx.x == 0) st.m[unit] = do_flush ? 0 : mt;
}

template <int D>
static cudaError_t launch_decode_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  const size_t smem = decode_smem(D, d.dP, 1).total;
  auto kern = decode_kernel<D>;
  const cudaError_t e = smem_opt_in<decode_kernel<D>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(units), dim3(D), smem, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, d, io, has_token);
}

template <int D>
static cudaError_t launch_bf16buf_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  const size_t smem = decode_smem(D, d.dP, 0).total;
  auto kern = decode_bf16buf_kernel<D>;
  const cudaError_t e = smem_opt_in<decode_bf16buf_kernel<D>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(units), dim3(D), smem, s, attr);
  return cudaLaunchKernelEx(&cfg, kern, d, io, has_token);
}

}  // namespace pace

cudaError_t pace_launch_decode(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.state_mode == PACE_STATE_BF16_BUF) {
    if (d.dP <= 8) return pace_launch_decode_bf16buf_fold(d, io, has_token, s);   // periods of up to 8 tokens
    return d.D == 128 ? launch_bf16buf_t<128>(d, io, has_token, s) : launch_bf16buf_t<64>(d, io, has_token, s);
  }
  return d.D == 128 ? launch_decode_t<128>(d, io, has_token, s) : launch_decode_t<64>(d, io, has_token, s);
}
