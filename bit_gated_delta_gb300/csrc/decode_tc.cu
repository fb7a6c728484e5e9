// PACE decode step with fused flush on the 5th-generation tensor cores (tcgen05) -- the quantized path
// ([P1] 어떻게 동작하나: round once every dP tokens, buffered tokens applied together at the flush;
// [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// Persistent kernel: each CTA loops over units (sequence b, head h). Warp 4 is a producer that streams
// every unit's bytes -- packed codes, group scales (and zero points), the m buffered entries, scalars,
// q/k/v -- into a ring of shared-memory stages with bulk asynchronous copies completing on an mbarrier,
// running several units ahead. Warps 0-3 (128 threads) compute; thread j owns state column j, which is
// also TMEM lane j of every accumulator, so the replay recurrence, the output and the key-axis group
// requantization of a column stay inside one thread. Per unit:
//   1. stage: the new token is quantized into buffer slot m; int8 key codes become the bf16 rows of the
//      MMA B operand (q enters as two rows q_hi + q_lo, fp32 precision); the stage is released early;
//   2. thread j writes c = u - z of its column as exact bf16 into TMEM lane j: the A operand (the state
//      transposed, M = 128 columns x K = d_k keys);
//   3. one MMA chain per key-axis group g: D_g[j][v] = sum_{i in g} c_ij B[v][i] (exact integers for the
//      int8 keys), then (S_hat^T k_v)_j = s_kv sum_g s_gj D_g[j][v] and (S_hat^T q)_j likewise;
//   4. the replay in reduced per-column form (thread-local, fp32):
//        u_t = beta_t (v_t - G_t (S_hat^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),   G_t = a_1 .. a_t
//        o   = G_m (S_hat^T q) + sum_s (G_m/G_s)(k_s.q) u_s
//   5. at a flush, a 128 x d_k fp32 accumulator in TMEM is set to G_m S_hat^T and the rank-m update
//        S_new^T += (rho u)^T K,   rho_s = (G_m/G_s) s_ks,
//      runs as one MMA chain with rho u split into three bf16 parts (hi + mid + lo, fp32-accurate) and the
//      int8 key codes as the other operand; thread j then requantizes column j group by group.
// Every mbarrier wait is bounded (1 s); on timeout the status word is set and the CTA stops after
// draining its tensor-core work and releasing its TMEM.
#include "pace_common.cuh"
#include "umma.cuh"

namespace pace {
using namespace umma;

constexpr uint64_t TC_WAIT_NS = 1000000000ull;
constexpr int TC_STAGES = 3;
constexpr int TC_COMPUTE = 128;            // compute threads (4 warps); warp 4 produces
constexpr int TC_THREADS = TC_COMPUTE + 32;

__host__ __device__ inline int tc_ntile(int dP) { return 16 * ((dP + 2 + 15) / 16); }   // B rows: keys + q_hi/q_lo
__host__ __device__ inline int tc_kflush(int dP) { return 16 * ((3 * dP + 15) / 16); }  // K of the flush MMA
__host__ __device__ inline int tc_cols(int D, int G, int dP) {
  int need = D / 2 + (D / G) * tc_ntile(dP);
  if (need < D) need = D;
  int c = 32;
  while (c < need) c <<= 1;
  return c;
}

// One stage of the ring: a unit's bytes as they sit in global memory.
struct StageLayout {
  size_t codes, scales, zp, bk, bv, bs, q, k, v, ab, bytes;
};
__host__ __device__ inline StageLayout stage_layout(int D, int G, int dP, int zp, int mixed, int io_f32, int any8) {
  StageLayout L;
  size_t off = 0;
  const size_t iob = io_f32 ? 4 : 2;
  L.codes = carve(off, (size_t)D * D / (any8 ? 1 : 2), 128);
  L.scales = carve(off, (size_t)(D / G) * D * 2);
  L.zp = carve(off, zp ? (size_t)(D / G) * D : 0);
  L.bk = carve(off, (size_t)dP * (mixed ? D / 2 : D));
  L.bv = carve(off, (size_t)dP * (mixed ? 2 * D : D));
  L.bs = carve(off, (size_t)dP * 16);
  L.q = carve(off, D * iob);
  L.k = carve(off, D * iob);
  L.v = carve(off, D * iob);
  L.ab = carve(off, 16);                    // a, beta, m (written by the producer)
  L.bytes = carve(off, 0, 128);
  return L;
}

// Work area of the compute warps.
struct TcSmem {
  size_t bdots, bflush, aflush, kq8, vf, P, U, qf, vscale, a, beta, gam, Dm, W, cq, ck, red, total;
};
__host__ __device__ inline TcSmem tc_smem(int D, int dP) {
  TcSmem L;
  size_t off = 0;
  const size_t nt = tc_ntile(dP), kf = tc_kflush(dP);
  L.bdots = carve(off, nt * D * 2, 128);           // B of the dot MMAs: nt rows x D keys (bf16, K-major cores)
  L.bflush = carve(off, (size_t)D * kf * 2, 128);  // B of the flush MMA: D keys x kf (bf16)
  L.aflush = carve(off, 128 * kf * 2, 128);        // A of the flush MMA: 128 columns x kf (bf16)
  L.kq8 = carve(off, (size_t)dP * D);              // int8 key codes
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
  L.total = carve(off, 0, 128);
  return L;
}

struct TcPlan {
  StageLayout S;
  TcSmem W;
  size_t stages, work, bars, total;
};
__host__ __device__ inline TcPlan tc_plan(int D, int G, int dP, int zp, int mixed, int io_f32, int any8) {
  TcPlan p;
  p.S = stage_layout(D, G, dP, zp, mixed, io_f32, any8);
  p.W = tc_smem(D, dP);
  size_t off = 0;
  p.stages = carve(off, TC_STAGES * p.S.bytes, 128);
  p.work = carve(off, p.W.total, 128);
  p.bars = carve(off, (2 * TC_STAGES + 1) * 8 + 16, 8);   // full[], empty[], mma, tmem base, flags
  p.total = carve(off, 0, 128);
  return p;
}

// Byte offset of element (row r, k) in a K-major operand of `kdim` columns made of 8 x 16-byte cores:
// cores along K are adjacent (128 B apart), 8-row groups are kdim/8 * 128 B apart.
__device__ __forceinline__ uint32_t core_off(int r, int k, int kdim) {
  return (uint32_t)((r >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

__device__ __forceinline__ float stage_io(const unsigned char *p, int i, int io) {
  if (io == PACE_IO_F32) return reinterpret_cast<const float *>(p)[i];
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
}

// Max over the 128 compute threads (named barrier 1; the producer warp does not take part).
__device__ __forceinline__ float compute_max(float v, float *red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_max(v);
  bar_sync_1(TC_COMPUTE);
  if (lane == 0) red[wid] = v;
  bar_sync_1(TC_COMPUTE);
  return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

struct TcShared {
  unsigned char *bdots, *bflush, *aflush;
  int8_t *kq8;
  float *vf, *P, *U, *qf, *vscale, *a, *beta, *gam, *Dm, *W, *cq, *ck, *red;
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
  return s;
}

// Decision shared by all 128 compute threads: true only if every one of them passes `ok`.
__device__ __forceinline__ bool compute_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, rr;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred rr, 1, 128, q;\n\tselp.u32 %0, 1, 0, rr;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

// Producer warp: streams unit n of this CTA into stage n % TC_STAGES. Lane 0 records the buffer count and
// issues the bulk copies (expected bytes on full[s]); lane 1 stores a_t, beta_t. Returns the number of
// stages it filled.
template <int D, int G>
__device__ int tc_produce(const PaceDev &st, const PaceIO &io, int has_token, long units, const TcPlan &P,
                          unsigned char *stages, uint64_t *full, uint64_t *empty, volatile int *stop) {
  constexpr int NG = D / G;
  const int lane = threadIdx.x & 31;
  const int dP = st.dP;
  const int mixed = st.buf_mode == PACE_BUF_MIXED;
  const uint32_t iob = st.io == PACE_IO_F32 ? 4u : 2u;
  const uint32_t rowk = mixed ? D / 2 : D, rowv = mixed ? 2 * D : D;
  int mreg = 0;
  int n = 0;
  for (;; ++n) {
    const long u = blockIdx.x + (long)n * gridDim.x;
    if (u >= units || *stop) break;
    const int s = n % TC_STAGES;
    if (n >= TC_STAGES) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ((n / TC_STAGES) - 1) & 1, TC_WAIT_NS));
      if (!ok) {
        if (lane == 0) {
          atomicOr(st.status, 1);
          *stop = 1;
        }
        break;
      }
    }
    if ((n & 31) == 0) {                          // buffer counts of the next 32 units, one load per lane
      const long uu = blockIdx.x + (long)(n + lane) * gridDim.x;
      mreg = uu < units ? st.m[uu] : 0;
    }
    const int m0 = __shfl_sync(0xffffffffu, mreg, n & 31);
    unsigned char *stg = stages + (size_t)s * P.S.bytes;
    if (lane == 0) {
      reinterpret_cast<int *>(stg + P.S.ab)[2] = m0;
      const bool work = (m0 >= 0 && m0 < dP) && (has_token || m0 > 0);
      const int b = (int)(u / st.H), h = (int)(u - (long)b * st.H);
      const int is8 = st.head_is_int8[h];
      const uint32_t cbytes = is8 ? D * D : D * D / 2;
      const uint32_t sbytes = NG * D * 2, zbytes = st.zero_point ? NG * D : 0;
      uint32_t tx = 0;
      if (work) tx = cbytes + sbytes + zbytes + (uint32_t)m0 * (rowk + rowv + 16) + (has_token ? 3 * D * iob : 0);
      mbar_arrive_expect_tx(&full[s], tx);
      if (work) {
        const uint32_t *codes = is8 ? st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D / 4) * D
                                    : st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D / 8) * D;
        bulk_g2s(stg + P.S.codes, codes, cbytes, &full[s]);
        bulk_g2s(stg + P.S.scales, st.scale + (size_t)u * NG * D, sbytes, &full[s]);
        if (zbytes) bulk_g2s(stg + P.S.zp, st.zp + (size_t)u * NG * D, zbytes, &full[s]);
        if (m0 > 0) {
          bulk_g2s(stg + P.S.bk, static_cast<const char *>(st.buf_k) + (size_t)u * dP * rowk, m0 * rowk, &full[s]);
          bulk_g2s(stg + P.S.bv, static_cast<const char *>(st.buf_v) + (size_t)u * dP * rowv, m0 * rowv, &full[s]);
          bulk_g2s(stg + P.S.bs, st.buf_s + (size_t)u * dP * 4, m0 * 16, &full[s]);
        }
        if (has_token) {
          bulk_g2s(stg + P.S.q, static_cast<const char *>(io.q) + (size_t)u * D * iob, D * iob, &full[s]);
          bulk_g2s(stg + P.S.k, static_cast<const char *>(io.k) + (size_t)u * D * iob, D * iob, &full[s]);
          bulk_g2s(stg + P.S.v, static_cast<const char *>(io.v) + (size_t)u * D * iob, D * iob, &full[s]);
        }
      }
    }
    if (lane == 1) {
      float *abf = reinterpret_cast<float *>(stg + P.S.ab);
      if (has_token) {
        abf[0] = io.a[u];
        abf[1] = io.beta[u];
      }
      mbar_arrive(&full[s]);
    }
    __syncwarp();
  }
  return n;
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
  bar_sync_1(TC_COMPUTE);
  // Gram k_s . k_t for s < t (pair index walks the strictly lower triangle), one warp per pair
  const int npairs = mt * (mt - 1) / 2;
  for (int item = wid; item < npairs; item += NW) {
    int t = 1, base = 0;
    while (base + t <= item) {
      base += t;
      ++t;
    }
    const int s = item - base;
    int acc = 0;
    if (lane < D / 4) {
      const int *ks = reinterpret_cast<const int *>(sh.kq8 + s * D);
      const int *kt = reinterpret_cast<const int *>(sh.kq8 + t * D);
      acc = dp4a_ss(ks[lane], kt[lane], 0);
    }
    const float dot = sh.vscale[s] * sh.vscale[t] * (float)__reduce_add_sync(0xffffffffu, acc);
    if (lane == 0) sh.W[t * dP + s] = sh.Dm[s * dP + t] * dot;
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
        const float zf = col ? 128.0f + (float)zg[(8 * w) / G] : 0.0f;
        const __nv_bfloat162 zz = __floats2bfloat162_rn(zf, zf);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t x = ((wd >> (4 * s)) & 0x000F000Fu) | 0x43004300u;   // bf16 pair (128 + u, 128 + u')
          __nv_bfloat162 cb = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&x), zz);
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
          __nv_bfloat162 cb = __floats2bfloat162_rn((float)((int)byte_of(wd, 2 * p) - z),
                                                    (float)((int)byte_of(wd, 2 * p + 1) - z));
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

// Requantize one group of G values and write its packed words (same arithmetic as quant_group, with the
// codes packed as they are produced).
template <int G, int BITS>
__device__ __forceinline__ void quant_pack_group(const float (&x)[G], int zero_point, uint32_t *dst, int stride,
                                                 float &s_out, int &z_out) {
  constexpr int KPW = 32 / BITS;
  float s, r;
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
    if (!(s >= FLT_MIN)) {
      s = 0.0f;
      z = 0;
    } else {
      r = __fdiv_rn(1.0f, s);
      z = min(max(__float2int_rn(__fmul_rn(-lo, r)), 0), qm);
    }
  }
  r = s > 0.0f ? __fdiv_rn(1.0f, s) : 0.0f;
#pragma unroll
  for (int w = 0; w < G / KPW; ++w) {
    uint32_t u[KPW];
#pragma unroll
    for (int e = 0; e < KPW; ++e) {
      int c;
      if (s == 0.0f) {
        c = zero_point ? 0 : z;
      } else if (!zero_point) {
        constexpr int qmax = (1 << (BITS - 1)) - 1;
        c = min(max(__float2int_rn(__fmul_rn(x[w * KPW + e], r)), -qmax), qmax) + z;
      } else {
        constexpr int qm = (1 << BITS) - 1;
        c = min(max(__float2int_rn(__fmul_rn(x[w * KPW + e], r)) + z, 0), qm);
      }
      u[e] = (uint32_t)c;
    }
    dst[w * stride] = BITS == 4 ? pack_nibbles(u) : pack_bytes(u);
  }
  s_out = s;
  z_out = zero_point ? z : 0;
}

// One unit on the 128 compute threads. Returns false if a bounded wait gave up (decided jointly).
template <int D, int G, int BITS>
__device__ bool tc_compute_unit(const PaceDev &st, const PaceIO &io, long unit, int has_token, int m0,
                                const unsigned char *stg, const StageLayout &SL, uint64_t *empty_s, uint64_t *mma_bar,
                                uint32_t &mma_phase, uint32_t tmem, const TcShared &sh) {
  constexpr int KPW = 32 / BITS, NWC = D / KPW, NG = D / G, WPG = G / KPW;
  const int j = threadIdx.x, warp = j >> 5;
  const bool col = j < D;
  const int dP = st.dP, nt = tc_ntile(dP), kf = tc_kflush(dP);
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 2 : 0);
  const int b = (int)(unit / st.H), h = (int)(unit - (long)b * st.H);
  const uint32_t lanes = (uint32_t)(warp * 32) << 16;

  // ---- the unit's packed column, scales and zero points from the stage
  const uint32_t *scodes = reinterpret_cast<const uint32_t *>(stg + SL.codes);
  const __nv_bfloat16 *sscale = reinterpret_cast<const __nv_bfloat16 *>(stg + SL.scales);
  uint32_t wr[NWC];
  float sg[NG];
  int zg[NG];
#pragma unroll
  for (int w = 0; w < NWC; ++w) wr[w] = col ? scodes[w * D + j] : 0u;
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    sg[g] = col ? __bfloat162float(sscale[g * D + j]) : 0.0f;
    zg[g] = (col && st.zero_point) ? (int)stg[SL.zp + g * D + j] : (1 << (BITS - 1));
  }

  // ---- buffered tokens and the new one into the work area
  const float *sbs = reinterpret_cast<const float *>(stg + SL.bs);
  if (j < m0) {
    sh.a[j] = sbs[j * 4 + 0];
    sh.beta[j] = sbs[j * 4 + 1];
    sh.vscale[j] = sbs[j * 4 + 2];
  }
  const int mixed = st.buf_mode == PACE_BUF_MIXED;
  if (col) {
    for (int t = 0; t < m0; ++t) {
      if (mixed) {
        const uint32_t byte = stg[SL.bk + t * (D / 2) + (j >> 1)];
        sh.kq8[t * D + j] = (int8_t)((int)((byte >> ((j & 1) * 4)) & 0xF) - 8);
        sh.vf[t * D + j] = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(stg + SL.bv)[t * D + j]);
      } else {
        sh.kq8[t * D + j] = reinterpret_cast<const int8_t *>(stg + SL.bk)[t * D + j];
        sh.vf[t * D + j] = sbs[t * 4 + 3] * (float)reinterpret_cast<const int8_t *>(stg + SL.bv)[t * D + j];
      }
    }
  }
  float qx = 0.0f;
  if (has_token) {
    float kx = 0.0f, vx = 0.0f;
    if (col) {
      kx = stage_io(stg + SL.k, j, st.io);
      vx = stage_io(stg + SL.v, j, st.io);
      qx = stage_io(stg + SL.q, j, st.io);
    }
    const int qmax = mixed ? 7 : 127;
    const float Ak = compute_max(fabsf(kx), sh.red);
    const float Av = mixed ? 0.0f : compute_max(fabsf(vx), sh.red + 4);
    const int ck = buffer_code(kx, Ak, qmax);
    const float sk = buffer_scale(Ak, qmax);
    const int nb = __shfl_down_sync(0xffffffffu, ck, 1);
    float sv = 0.0f;
    if (col) {
      sh.kq8[m0 * D + j] = (int8_t)ck;
      sh.qf[j] = qx;
      if (mixed) {
        sh.vf[m0 * D + j] = bf16_round(vx);
        if ((j & 1) == 0)
          static_cast<uint8_t *>(st.buf_k)[(unit * dP + m0) * (D / 2) + (j >> 1)] = (uint8_t)((ck + 8) | ((nb + 8) << 4));
        static_cast<__nv_bfloat16 *>(st.buf_v)[(unit * dP + m0) * D + j] = __float2bfloat16_rn(vx);
      } else {
        const int cv = buffer_code(vx, Av, 127);
        sv = buffer_scale(Av, 127);
        sh.vf[m0 * D + j] = sv * (float)cv;
        static_cast<int8_t *>(st.buf_k)[(unit * dP + m0) * D + j] = (int8_t)ck;
        static_cast<int8_t *>(st.buf_v)[(unit * dP + m0) * D + j] = (int8_t)cv;
      }
    }
    if (j == 0) {
      const float *ab = reinterpret_cast<const float *>(stg + SL.ab);
      const float ax = ab[0], bx = ab[1];
      sv = mixed ? 0.0f : buffer_scale(Av, 127);
      sh.a[m0] = ax;
      sh.beta[m0] = bx;
      sh.vscale[m0] = sk;
      sh.vscale[mt] = 1.0f;
      sh.vscale[mt + 1] = 1.0f;
      float *bw = st.buf_s + (unit * dP + m0) * 4;
      bw[0] = ax;
      bw[1] = bx;
      bw[2] = sk;
      bw[3] = sv;
    }
  }
  bar_sync_1(TC_COMPUTE);
  if (j == 0) mbar_arrive(empty_s);              // every read of the stage is done: hand it back
  // bf16 rows of the dot MMAs' B operand (rows >= nv are never read back)
  if (col) {
    for (int r = 0; r < nv; ++r) {
      float x;
      if (r < mt) x = (float)sh.kq8[r * D + j];
      else if (r == mt) x = bf16_round(qx);
      else x = qx - bf16_round(qx);
      *reinterpret_cast<uint16_t *>(sh.bdots + core_off(r, j, D)) = bf16_bits(x);
    }
  }

  // ---- A operand, then the dot-product MMAs (one chain per key-axis group)
  tc_write_A<D, G, BITS>(tmem + lanes, wr, zg, col);
  tmem_wait_st();
  fence_smem_to_async();
  fence_before_sync();
  bar_sync_1(TC_COMPUTE);
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
    commit(mma_bar);
  }
  tc_tables<D>(mt, has_token, dP, sh);
  bar_sync_1(TC_COMPUTE);
  bool ok = compute_all(mbar_wait(mma_bar, mma_phase, TC_WAIT_NS));
  mma_phase ^= 1u;
  fence_after_sync();
  if (!ok) return false;

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
  if (!do_flush) return true;

  // ---- flush operands: A[j][3s+p] = part p of rho_s u_s,j ; B[i][3s+p] = key code k_s,i
  for (int kk = 0; kk < kf; ++kk) {
    const int s = kk / 3, p = kk - 3 * s;
    float x = 0.0f;
    if (col && s < mt) {
      const float y = sh.ck[s] * sh.U[s * 128 + j];
      const float hi = bf16_round(y);
      const float mid = bf16_round(y - hi);
      x = p == 0 ? hi : (p == 1 ? mid : y - hi - mid);
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
  bar_sync_1(TC_COMPUTE);
  fence_after_sync();
  if (j == 0) {
    const uint32_t idesc = idesc_bf16(128, D);
    const uint32_t abase = smem_u32(sh.aflush), bbase = smem_u32(sh.bflush);
    for (int s = 0; s < kf / 16; ++s)
      mma_ss(tmem, smem_desc(abase + s * 256, 128, (kf / 8) * 128), smem_desc(bbase + s * 256, 128, (kf / 8) * 128),
             idesc, 1u);
    commit(mma_bar);
  }
  ok = compute_all(mbar_wait(mma_bar, mma_phase, TC_WAIT_NS));
  mma_phase ^= 1u;
  fence_after_sync();
  if (!ok) return false;
  if (col) {
    const int slot = st.head_slot[h];
    uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + slot) * NWC * D
                                : st.codes8 + (size_t)(b * st.H8 + slot) * NWC * D;
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
      float s_new;
      int z_new;
      quant_pack_group<G, BITS>(x, st.zero_point, codes + (size_t)g * WPG * D + j, D, s_new, z_new);
      st.scale[(unit * NG + g) * D + j] = __float2bfloat16_rn(s_new);
      if (st.zero_point) st.zp[(unit * NG + g) * D + j] = (uint8_t)z_new;
    }
  }
  return true;
}

template <int D, int G>
__global__ void __launch_bounds__(TC_THREADS, 3) decode_tc_kernel(const PaceDev st, const PaceIO io, const int has_token,
                                                                  const int any8) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const TcPlan P = tc_plan(D, G, st.dP, st.zero_point, st.buf_mode == PACE_BUF_MIXED, st.io == PACE_IO_F32, any8);
  unsigned char *stages = smem + P.stages;
  const TcShared sh = tc_shared(smem + P.work, P.W);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + P.bars);
  uint64_t *empty = full + TC_STAGES;
  uint64_t *mma_bar = empty + TC_STAGES;
  uint32_t *tbase = reinterpret_cast<uint32_t *>(mma_bar + 1);
  volatile int *stop = reinterpret_cast<volatile int *>(tbase + 1);
  int *consumed = const_cast<int *>(stop + 1);
  const long units = (long)st.B * st.H;
  const int ncols = tc_cols(D, G, st.dP);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 2);
      mbar_init(&empty[s], 1);
    }
    mbar_init(mma_bar, 1);
    *stop = 0;
    *consumed = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tbase, (uint32_t)ncols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tbase;

  int produced = 0;
  if (warp == 4) {
    produced = tc_produce<D, G>(st, io, has_token, units, P, stages, full, empty, stop);
  } else {
    const int j = threadIdx.x;
    uint32_t mma_phase = 0;
    int n = 0;
    for (;; ++n) {
      const long u = blockIdx.x + (long)n * gridDim.x;
      if (u >= units) break;
      const int s = n % TC_STAGES;
      const bool ready = compute_all(mbar_wait(&full[s], (n / TC_STAGES) & 1, TC_WAIT_NS));
      if (!ready) {
        if (j == 0) {
          atomicOr(st.status, 1);
          *stop = 1;
        }
        break;
      }
      const unsigned char *stg = stages + (size_t)s * P.S.bytes;
      const int m0 = reinterpret_cast<const int *>(stg + P.S.ab)[2];
      if (m0 < 0 || m0 >= st.dP || (!has_token && m0 == 0)) {
        if (has_token && j < D && (m0 < 0 || m0 >= st.dP)) store_io(io.o, u * D + j, 0.0f, st.io);
        bar_sync_1(TC_COMPUTE);
        if (j == 0) mbar_arrive(&empty[s]);
        continue;
      }
      const int h = (int)(u % st.H);
      bool ok;
      if (st.head_is_int8[h])
        ok = tc_compute_unit<D, G, 8>(st, io, u, has_token, m0, stg, P.S, &empty[s], mma_bar, mma_phase, tmem, sh);
      else
        ok = tc_compute_unit<D, G, 4>(st, io, u, has_token, m0, stg, P.S, &empty[s], mma_bar, mma_phase, tmem, sh);
      if (!ok) {
        if (j == 0) {
          atomicOr(st.status, 1);
          *stop = 1;
        }
        mbar_wait(mma_bar, mma_phase ^ 1u, TC_WAIT_NS);   // let the pending MMAs drain before TMEM goes
        ++n;
        break;
      }
      if (j == 0) st.m[u] = (!has_token || m0 + 1 == st.dP) ? 0 : m0 + 1;
      bar_sync_1(TC_COMPUTE);                    // the work area is reused by the next unit
    }
    if (j == 0) *consumed = n;
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 4 && (threadIdx.x & 31) == 0) {
    // stages filled but never consumed (only after a timeout): wait for their copies before exiting
    for (int n = *consumed; n < produced; ++n) mbar_wait(&full[n % TC_STAGES], (n / TC_STAGES) & 1, TC_WAIT_NS);
  }
  if (warp == 0) tmem_dealloc(tmem, (uint32_t)ncols);
}

template <int D, int G>
static cudaError_t launch_tc_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  auto kern = decode_tc_kernel<D, G>;
  const int any8 = d.H8 > 0;
  const TcPlan plan = tc_plan(D, G, d.dP, d.zero_point, d.buf_mode == PACE_BUF_MIXED, d.io == PACE_IO_F32, any8);
  const size_t smem = plan.total;
  static size_t opted = 0;
  static int sms = 0;
  if (smem > opted) {
    const size_t most = 227 * 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    if (e != cudaSuccess) return e;
    opted = most;
  }
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const long units = (long)d.B * d.H;
  if (units == 0) return cudaSuccess;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, TC_THREADS, smem);
  if (e != cudaSuccess) return e;
  const int tmem_per_sm = 512 / tc_cols(D, G, d.dP);
  if (per_sm > tmem_per_sm) per_sm = tmem_per_sm;
  if (per_sm < 1) per_sm = 1;
  long grid = (long)sms * per_sm;
  if (grid > units) grid = units;
  kern<<<(unsigned)grid, TC_THREADS, smem, s>>>(d, io, has_token, any8);
  return cudaGetLastError();
}

}  // namespace pace

cudaError_t pace_launch_decode_tc(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.D == 128) return d.G == 64 ? launch_tc_t<128, 64>(d, io, has_token, s) : launch_tc_t<128, 32>(d, io, has_token, s);
  return d.G == 64 ? launch_tc_t<64, 64>(d, io, has_token, s) : launch_tc_t<64, 32>(d, io, has_token, s);
}
