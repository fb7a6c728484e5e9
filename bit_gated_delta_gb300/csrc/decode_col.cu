// PACE decode step with fused flush on the 5th-generation tensor cores, one thread per state column
// ([P1] 어떻게 동작하나: round once every dP tokens, the buffered tokens applied together at the flush;
// [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// Int4 heads, d_k = d_v = 128, int8 decode buffer, dP <= 8. One CTA of 128 threads per unit; thread j owns value
// column j, which is also TMEM lane j. Per step:
//   1. the unit's loads are issued before the buffer count is read; thread j loads the 16 code words of its
//      column and its group scales; the buffered rows arrive by async copies;
//   2. the new token is quantized into buffer slot m (block maxima), q becomes three int8 digit rows;
//   3. the vectors (buffered keys, new key, q digits) become the fp16 B operand, K-major cores, in a key order
//      that matches the A operand; thread j turns its code words into the A operand in TMEM: the word of keys
//      32p+8r+2t+e (r = 0..3, e = 0, 1) gives (w>>0 & 0x000F000F)|0x6400... = the pair 1024+u for r = 0, the
//      mask 0x00F000F0 = 1024+16u for r = 1 (those B values pre-scaled by 1/16), and the same after a shift by 8
//      for r = 2, 3. One thread issues the MMAs, one accumulator per key-axis group:
//        D_g[j][v] = sum_{i in g} (1024 + u_ij or 1024 + 16 u_ij) B[v][i]        (exact integers, fp32)
//      meanwhile two warps build the group sums (T1, T2), the Gram and digit products with warp-level MMAs;
//   4. thread j folds its column, P[v] = sum_g s_gj (D_g[v] - T1_gv - z_gj T2_gv), replays the buffered tokens
//      u_t = beta_t (v_t - G_t P_t - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s) and emits o = G_m (S^T q) + sum_s ...;
//   5. at a rounding, one bf16 MMA (A = three bf16 parts of (G_m/G_s) s_ks u_s,j per column, B = the int8 keys)
//      gives the rank-m update of every element in TMEM; thread j adds G_m s_gj (u_ij - z_gj), requantizes its
//      column group by group (no shuffles) with the quantizer's exact arithmetic and writes its code words.
// Every mbarrier wait is bounded; on timeout the unit is left unchanged, the status word is set and the kernel
// drains its MMAs and releases its TMEM.
#include "decode_mma.cuh"
#include "umma.cuh"

namespace pace {

namespace dcol {
constexpr int D = 128, NT = 128;
constexpr int MAXP = 8;                 // largest decode period handled
constexpr int NVR = 16;                 // vector rows: N of the dot MMA
constexpr uint32_t TCOLS = 128;         // TMEM columns: A (64) + D_g (16 per group) ; flush D (128)
constexpr uint64_t WAIT_NS = 1000000000ull;
// shared memory (bytes)
constexpr uint32_t OFF_BV = 0;                          // fp16 [16][128] K-major cores (4 KB)
constexpr uint32_t OFF_A3 = OFF_BV + NVR * D * 2;       // bf16 [128][32] flush A: parts of rho u (8 KB)
constexpr uint32_t OFF_B3 = OFF_A3 + D * 32 * 2;        // bf16 [128][32] flush B: keys (8 KB)
constexpr uint32_t OFF_KROW = OFF_B3 + D * 32 * 2;      // int8 [MAXP + 3][128]
constexpr uint32_t OFF_VROW = OFF_KROW + (MAXP + 3) * D;// int8 [MAXP][128]
constexpr uint32_t OFF_F = OFF_VROW + MAXP * D;         // float tables
// float table offsets (in floats, from OFF_F)
constexpr int T_A = 0, T_BET = 8, T_SVT = 16, T_VSC = 24, T_GAM = 40, T_DMQ = 48, T_DMT = 56, T_W = 120, T_E3 = 184,
              T_TK = 208, T_CK = 240, T_RED = 248, T_CF = 264, T_END = T_CF + NVR * 4 * 2;
constexpr uint32_t OFF_SSC = OFF_F + T_END * 4;          // bf16 [4][128] group scales
constexpr uint32_t OFF_SZP = OFF_SSC + 4 * D * 2;        // u8 [4][128] zero points
constexpr uint32_t OFF_BAR = OFF_SZP + 4 * D;
constexpr uint32_t OFF_TB = OFF_BAR + 8;
constexpr uint32_t OFF_OK = OFF_TB + 4;
constexpr uint32_t SMEM = OFF_OK + 4;

__host__ __device__ constexpr uint32_t core_off(int r, int k, int kdim) {
  return (uint32_t)((r >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
// K index of key i in the dot operands: i = 32p + 8r + 2t + e -> column pair c = 16p + 4r + t, index 2c + e.
__device__ __forceinline__ int kappa(int i) {
  const int p = i >> 5, r = (i >> 3) & 3, t = (i >> 1) & 3, e = i & 1;
  return 2 * (16 * p + 4 * r + t) + e;
}
// Instruction descriptor of kind::f16 with fp16 A and B (K-major), fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
}  // namespace dcol

template <int G, int ZP>
__global__ void __launch_bounds__(dcol::NT, 4) decode_col_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  using namespace dcol;
  using namespace umma;
  constexpr int NG = D / G, KSG = G / 16;
  constexpr int OFF = 8;                              // symmetric int4 offset
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, j = tid;
  const int g8 = lane >> 2, tq = lane & 3;
  const int HP = st.H4;
  const int w = blockIdx.x;
  if (w >= st.B * HP) return;
  const int b = w / HP, slot = w - b * HP;
  const int h = st.pool_head[slot];
  const int unit = b * st.H + h;
  const int dP = st.dP;
  float *F = reinterpret_cast<float *>(smem + OFF_F);
  int8_t *krow = reinterpret_cast<int8_t *>(smem + OFF_KROW);
  int8_t *vrow = reinterpret_cast<int8_t *>(smem + OFF_VROW);
  __half *Bv = reinterpret_cast<__half *>(smem + OFF_BV);
  uint32_t *codes = st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8);
  const uint32_t sbase = smem_u32(smem);

  // ---- 1. loads that do not depend on the buffer count
  uint32_t cw[4][4];                                  // [p][t]: keys 32p + 8r + 2t + e of column j
#pragma unroll
  for (int p2 = 0; p2 < 2; ++p2)
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint2 v2 = *reinterpret_cast<const uint2 *>(codes + code_word(D, j, 64 * p2 + 2 * t));
      cw[2 * p2][t] = v2.x;
      cw[2 * p2 + 1][t] = v2.y;
    }
  float sg[NG];
  int zg[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    sg[g] = __bfloat162float(st.scale[((size_t)unit * NG + g) * D + j]);
    zg[g] = ZP ? (int)st.zp[((size_t)unit * NG + g) * D + j] : OFF;
  }
  {                                                   // every buffered row, before the count is known
    const char *gk = static_cast<const char *>(st.buf_k) + (size_t)unit * dP * D;
    const char *gv = static_cast<const char *>(st.buf_v) + (size_t)unit * dP * D;
    for (int c = tid; c < 2 * dP * (D / 16); c += NT) {
      if (c < dP * (D / 16)) cp_async16(krow + 16 * c, gk + 16 * c);
      else cp_async16(vrow + 16 * (c - dP * (D / 16)), gv + 16 * (c - dP * (D / 16)));
    }
  }
  float kx = 0.0f, vx = 0.0f, qx = 0.0f, an = 0.0f, bn = 0.0f;
  if (has_token) {
    kx = load_io(io.k, (long)unit * D + j, st.io);
    vx = load_io(io.v, (long)unit * D + j, st.io);
    qx = load_io(io.q, (long)unit * D + j, st.io);
    an = io.a[unit];
    bn = io.beta[unit];
  }
  float4 bs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (warp == 3 && lane < dP) bs = *reinterpret_cast<const float4 *>(st.buf_s + ((size_t)unit * dP + lane) * 4);
  const int m0 = st.m[unit];
  if (m0 < 0 || m0 >= dP || (!has_token && m0 == 0)) {
    cp_async_wait_all();                               // nothing may land in shared memory after the CTA leaves
    if (has_token && m0 != 0) store_io(io.o, (long)unit * D + j, 0.0f, st.io);   // corrupted counter: zeros
    return;
  }
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 3 : 0);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint32_t *tbase = reinterpret_cast<uint32_t *>(smem + OFF_TB);
  volatile int *okf = reinterpret_cast<volatile int *>(smem + OFF_OK);
  if (warp == 0) {
    tmem_alloc(tbase, TCOLS);
    tmem_relinquish();
  }
  fence_before_sync();
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
    *okf = 1;
  }
  {                                                   // scales and zero points of the unit, for the flush
    __nv_bfloat16 *ssc = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_SSC);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      ssc[g * D + j] = __float2bfloat16_rn(sg[g]);
      if (ZP) smem[OFF_SZP + g * D + j] = (unsigned char)zg[g];
    }
  }

  // ---- 2. the new token: block maxima of |k|, |v|, |q|
  float Ak = 0.0f, Av = 0.0f, Aq = 0.0f;
  if (has_token) {
    const float mk = warp_max(fabsf(kx)), mv = warp_max(fabsf(vx)), mq = warp_max(fabsf(qx));
    if (lane == 0) {
      F[T_RED + warp] = mk;
      F[T_RED + 4 + warp] = mv;
      F[T_RED + 8 + warp] = mq;
    }
  }
  cp_async_wait_all();
  __syncthreads();
  float sk = 0.0f, sv = 0.0f;
  if (has_token) {
    Ak = fmaxf(fmaxf(F[T_RED + 0], F[T_RED + 1]), fmaxf(F[T_RED + 2], F[T_RED + 3]));
    Av = fmaxf(fmaxf(F[T_RED + 4], F[T_RED + 5]), fmaxf(F[T_RED + 6], F[T_RED + 7]));
    Aq = fmaxf(fmaxf(F[T_RED + 8], F[T_RED + 9]), fmaxf(F[T_RED + 10], F[T_RED + 11]));
    const int kc = buffer_code(kx, Ak, 127), vc = buffer_code(vx, Av, 127);
    sk = buffer_scale(Ak, 127);
    sv = buffer_scale(Av, 127);
    krow[m0 * D + j] = (int8_t)kc;
    vrow[m0 * D + j] = (int8_t)vc;
    static_cast<int8_t *>(st.buf_k)[((size_t)unit * dP + m0) * D + j] = (int8_t)kc;
    static_cast<int8_t *>(st.buf_v)[((size_t)unit * dP + m0) * D + j] = (int8_t)vc;
    if (tid == 0) *reinterpret_cast<float4 *>(st.buf_s + ((size_t)unit * dP + m0) * 4) = make_float4(an, bn, sk, sv);
    // q ~= sigma (65536 d2 + 256 d1 + d0), balanced base-256 digits
    const float QMAX = 8323072.0f;
    const bool qz = !(Aq >= FLT_MIN);
    const float sigma = qz ? 0.0f : __fdiv_rn(Aq, QMAX);
    const float rq = qz ? 0.0f : __fdiv_rn(QMAX, Aq);
    const int qi = min(max(__float2int_rn(qx * rq), -8323072), 8323072);
    const int q1 = (qi + 128) >> 8;
    const int d0 = qi - (q1 << 8), d2 = (q1 + 128) >> 8, d1 = q1 - (d2 << 8);
    krow[mt * D + j] = (int8_t)d2;
    krow[(mt + 1) * D + j] = (int8_t)d1;
    krow[(mt + 2) * D + j] = (int8_t)d0;
    if (tid == 0) {
      F[T_VSC + mt] = 65536.0f * sigma;
      F[T_VSC + mt + 1] = 256.0f * sigma;
      F[T_VSC + mt + 2] = sigma;
    }
  }
  if (warp == 3 && lane < mt) {
    F[T_A + lane] = lane < m0 ? bs.x : an;
    F[T_BET + lane] = lane < m0 ? bs.y : bn;
    F[T_VSC + lane] = lane < m0 ? bs.z : sk;
    F[T_SVT + lane] = lane < m0 ? bs.w : sv;
  }
  __syncthreads();

  // ---- 3a. B operand (vectors) in the A operand's key order; the decay products
  {
    const int kap = kappa(j);
    const float sc = ((j >> 3) & 1) ? 0.0625f : 1.0f;   // r odd: the A values are 1024 + 16u
#pragma unroll
    for (int v = 0; v < NVR; ++v) {
      const float x = v < nv ? (float)krow[v * D + j] * sc : 0.0f;
      Bv[core_off(v, kap, D) / 2] = __float2half_rn(x);
    }
  }
  if (warp == 3 && lane < mt) {
    float gg = 1.0f, dm = 1.0f;
    for (int r = 0; r <= lane; ++r) gg *= F[T_A + r];
    for (int r = lane + 1; r < mt; ++r) dm *= F[T_A + r];
    F[T_GAM + lane] = gg;
    F[T_DMQ + lane] = dm;
    float p = 1.0f;                                   // G_t/G_s = a_{s+1} .. a_t for t = lane, s < t
    for (int s2 = lane - 1; s2 >= 0; --s2) {
      p *= F[T_A + s2 + 1];
      F[T_DMT + lane * 8 + s2] = p;
    }
  }
  // ---- 3b. A operand: this column's codes as fp16 pairs in TMEM lane j (columns 16p + 4r + t)
  fence_after_sync();
  const uint32_t tmem = *tbase;
  const uint32_t lanes = (uint32_t)(warp * 32) << 16;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t r16[16];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t x = cw[p][t], y = x >> 8;
      r16[0 + t] = (x & 0x000F000Fu) | 0x64006400u;
      r16[4 + t] = (x & 0x00F000F0u) | 0x64006400u;
      r16[8 + t] = (y & 0x000F000Fu) | 0x64006400u;
      r16[12 + t] = (y & 0x00F000F0u) | 0x64006400u;
    }
    tmem_st16(tmem + lanes + 16 * p, r16);
  }
  tmem_wait_st();
  fence_smem_to_async();
  fence_before_sync();
  __syncthreads();

  // ---- 3c. the dot MMAs (one thread), and the tables on warps 0 and 1 meanwhile
  if (tid == 0) {
    fence_after_sync();
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int kk = 0; kk < KSG; ++kk) {
        const int ks = g * KSG + kk;
        mma_ts(tmem + 64 + 16 * g, tmem + 8 * ks, smem_desc(sbase + OFF_BV + ks * 256, 128, (D / 8) * 128),
               idesc_f16(128, NVR), kk ? 1u : 0u);
      }
    commit(bar);
  }
  {
    const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = lane >> 4;
    const int brow = lane & 7, bcol = (lane >> 3) & 1;
    if (warp == 0) {                                  // group sums: column 2gi = first halves, 2gi + 1 = second
      float cs[4];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, smem + OFF_BV + core_off(arow, 16 * ks + 8 * acol, D));
        const int gi = ks / KSG;
        const uint32_t o0 = g8 == 2 * gi ? 0x3C003C00u : 0u, o1 = g8 == 2 * gi + 1 ? 0x3C003C00u : 0u;
        if (ks == 0) mma_f16_z(cs, a, o0, o1); else mma_f16(cs, a, o0, o1);
      }
      if (tq < NG) {
        float2 *cf = reinterpret_cast<float2 *>(F + T_CF);
        cf[g8 * 4 + tq] = make_float2(1024.0f * (cs[0] + cs[1]), cs[0] + 16.0f * cs[1]);
        cf[(g8 + 8) * 4 + tq] = make_float2(1024.0f * (cs[2] + cs[3]), cs[2] + 16.0f * cs[3]);
      }
    } else if (warp == 1) {                           // Gram k_s.k_t and digit products k_s.(q digit)
      float gr[4];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4], bb[2];
        ldsm_x4(a, smem + OFF_BV + core_off(arow, 16 * ks + 8 * acol, D));
        ldsm_x2(bb, smem + OFF_BV + core_off(brow, 16 * ks + 8 * bcol, D));
        const uint32_t b1 = f16x2_scale(bb[1], 256.0f);
        if (ks == 0) mma_f16_z(gr, a, bb[0], b1); else mma_f16(gr, a, bb[0], b1);
      }
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = g8 + 8 * (e >> 1), s2 = 2 * tq + (e & 1);
        if (s2 >= mt) continue;
        if (v < mt && s2 < v)
          F[T_W + v * 8 + s2] = F[T_DMT + v * 8 + s2] * F[T_VSC + s2] * F[T_VSC + v] * gr[e];
        else if (v >= mt && v < nv)
          F[T_E3 + (v - mt) * 8 + s2] = gr[e];
      }
      __syncwarp();
      if (lane < mt) {
        const float dv = F[T_DMQ + lane] * F[T_VSC + lane];
        const float cq = has_token ? dv * (F[T_VSC + mt] * F[T_E3 + lane] +
                                           (F[T_VSC + mt + 1] * F[T_E3 + 8 + lane] + F[T_VSC + mt + 2] * F[T_E3 + 16 + lane]))
                                   : 0.0f;
        F[T_CK + lane] = dv;
        reinterpret_cast<float4 *>(F + T_TK)[lane] =
            make_float4(F[T_GAM + lane] * F[T_VSC + lane], F[T_BET + lane], F[T_SVT + lane], cq);
      }
    }
  }
  if (tid == 0 && !mbar_wait(bar, 0, WAIT_NS)) *okf = 0;
  __syncthreads();
  bool ok = *okf != 0;
  uint32_t pending = 0;
  fence_after_sync();

  float u[MAXP];
#pragma unroll
  for (int t = 0; t < MAXP; ++t) u[t] = 0.0f;
  if (ok) {
    // ---- 4. fold, replay and readout of column j
    float P[NVR];
#pragma unroll
    for (int v = 0; v < NVR; ++v) P[v] = 0.0f;
    const float2 *cf = reinterpret_cast<const float2 *>(F + T_CF);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      uint32_t d[16];
      tmem_ld16(tmem + lanes + 64 + 16 * g, d);
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < NVR; ++v) {
        const float2 c = cf[v * 4 + g];
        const float tot = __uint_as_float(d[v]) - fmaf((float)zg[g], c.y, c.x);
        P[v] = fmaf(sg[g], tot, P[v]);
      }
    }
    const float gm = F[T_GAM + mt - 1];
    float o = 0.0f;
    if (has_token) {
      float pq = 0.0f;
#pragma unroll
      for (int v = 0; v < NVR; ++v)
        if (v >= mt && v < mt + 3) pq = fmaf(F[T_VSC + v], P[v], pq);
      o = gm * pq;
    }
    const float4 *tk4 = reinterpret_cast<const float4 *>(F + T_TK);
#pragma unroll
    for (int t = 0; t < MAXP; ++t) {
      if (t < mt) {
        const float4 tk = tk4[t];                       // G_t s_kt, beta_t, s_vt, readout coefficient
        float acc = fmaf(-tk.x, P[t], tk.z * (float)vrow[t * D + j]);
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-F[T_W + t * 8 + s2], u[s2], acc);
        u[t] = tk.y * acc;
        o = fmaf(tk.w, u[t], o);
      }
    }
    if (has_token) store_io(io.o, (long)unit * D + j, o, st.io);

    if (do_flush) {
      // ---- 5. the rounding: A3 row j = three bf16 parts of ck_s u_s,j (K = part*8 + s), B3 row i = keys k_s,i
      {
        uint32_t pw[3][4];
#pragma unroll
        for (int s2 = 0; s2 < MAXP; s2 += 2) {
          const float x0 = s2 < mt ? F[T_CK + s2] * u[s2] : 0.0f;
          const float x1 = s2 + 1 < mt ? F[T_CK + s2 + 1] * u[s2 + 1] : 0.0f;
          const uint32_t p0 = bf16x2_bits(x0, x1);
          const float r0 = x0 - bf16_lo(p0), r1 = x1 - bf16_hi(p0);
          const uint32_t p1 = bf16x2_bits(r0, r1);
          pw[0][s2 / 2] = p0;
          pw[1][s2 / 2] = p1;
          pw[2][s2 / 2] = bf16x2_bits(r0 - bf16_lo(p1), r1 - bf16_hi(p1));
        }
#pragma unroll
        for (int part = 0; part < 3; ++part)
          *reinterpret_cast<uint4 *>(smem + OFF_A3 + core_off(j, 8 * part, 32)) =
              make_uint4(pw[part][0], pw[part][1], pw[part][2], pw[part][3]);
        *reinterpret_cast<uint4 *>(smem + OFF_A3 + core_off(j, 24, 32)) = make_uint4(0u, 0u, 0u, 0u);
        uint32_t kw[4];
#pragma unroll
        for (int s2 = 0; s2 < MAXP; s2 += 2) {
          const float k0 = s2 < mt ? (float)krow[s2 * D + j] : 0.0f;
          const float k1 = s2 + 1 < mt ? (float)krow[(s2 + 1) * D + j] : 0.0f;
          kw[s2 / 2] = bf16x2_bits(k0, k1);
        }
#pragma unroll
        for (int part = 0; part < 3; ++part)
          *reinterpret_cast<uint4 *>(smem + OFF_B3 + core_off(j, 8 * part, 32)) = make_uint4(kw[0], kw[1], kw[2], kw[3]);
        *reinterpret_cast<uint4 *>(smem + OFF_B3 + core_off(j, 24, 32)) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_smem_to_async();
      fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_ss(tmem, smem_desc(sbase + OFF_A3 + kk * 256, 128, 4 * 128), smem_desc(sbase + OFF_B3 + kk * 256, 128, 4 * 128),
                 idesc_bf16(128, D), kk ? 1u : 0u);
        commit(bar);
        if (!mbar_wait(bar, 1, WAIT_NS)) *okf = 0;
      }
      __syncthreads();
      ok = *okf != 0;
      pending = 1;
      fence_after_sync();
      if (ok) {
        __nv_bfloat16 *scale = st.scale + (size_t)unit * NG * D;
        uint8_t *zpt = ZP ? st.zp + (size_t)unit * NG * D : nullptr;
#pragma unroll
        for (int g = 0; g < NG; ++g) {               // unrolled: the code words are indexed by group
          float x[G];
#pragma unroll
          for (int c = 0; c < G / 16; ++c) {
            uint32_t r16[16];
            tmem_ld16(tmem + lanes + g * G + 16 * c, r16);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) x[16 * c + e] = __uint_as_float(r16[e]);
          }
          // the old state G_m s_gj (u_ij - z_gj), added in fp32 pairs (u - z exact)
          const float fs = gm * sg[g];
          const float fz = -(8388608.0f + (float)zg[g]);
#pragma unroll
          for (int k2 = 0; k2 < G / 2; ++k2) {
            const int i = g * G + 2 * k2;             // keys i, i + 1: word (p, t), nibble row r
            const int p = i >> 5, r = (i >> 3) & 3, t = (i >> 1) & 3;
            const uint32_t m16 = (cw[p][t] >> (4 * r)) & 0x000F000Fu;
            const float2 f = make_float2(__uint_as_float(__byte_perm(m16, 0x4B000000u, 0x7610)),
                                         __uint_as_float(__byte_perm(m16, 0x4B000000u, 0x7632)));
            const float2 dd = __fadd2_rn(f, make_float2(fz, fz));
            const float2 y = __ffma2_rn(make_float2(fs, fs), dd, make_float2(x[2 * k2], x[2 * k2 + 1]));
            x[2 * k2] = y.x;
            x[2 * k2 + 1] = y.y;
          }
          // requantize the group with the quantizer's arithmetic
          float s;
          int z;
          if (!ZP) {
            float A = 0.0f;
#pragma unroll
            for (int e = 0; e < G; e += 2) A = fmax3(A, fabsf(x[e]), fabsf(x[e + 1]));
            s = bf16_quot(A, 7.0f, 1.0f / 7.0f);
            z = OFF;
          } else {
            float lo = 0.0f, hi = 0.0f;
#pragma unroll
            for (int e = 0; e < G; e += 2) {
              lo = fmin3(lo, x[e], x[e + 1]);
              hi = fmax3(hi, x[e], x[e + 1]);
            }
            s = bf16_quot(__fsub_rn(hi, lo), 15.0f, 1.0f / 15.0f);
            z = 0;
            if (s >= FLT_MIN) z = min(max(__float2int_rn(__fmul_rn(-lo, rcp_bf16(s))), 0), 15);
          }
          if (!(s >= FLT_MIN)) s = 0.0f;
          const float rr = s > 0.0f ? rcp_bf16(s) : 0.0f;
          const float2 r2 = make_float2(rr, rr);
          const float mg = ZP ? 12582912.0f : 12582912.0f + (float)OFF;
          const float2 mg2 = make_float2(mg, mg);
#pragma unroll
          for (int pw2 = 0; pw2 < G / 32; ++pw2) {
            const int p = g * (G / 32) + pw2;           // 32-key span of the column
            uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int rq2 = 0; rq2 < 4; ++rq2)
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int e0 = pw2 * 32 + 8 * rq2 + 2 * t;   // key offset inside the group
                const float2 y = __fadd2_rn(__fmul2_rn(make_float2(x[e0], x[e0 + 1]), r2), mg2);
                uint32_t pair;
                if (!ZP) {
                  pair = __byte_perm(__float_as_uint(y.x), __float_as_uint(y.y), 0x5410);   // code + 8 in 1..15
                } else {
                  const int c0 = min(max((int)(__float_as_uint(y.x) - 0x4B400000u) + z, 0), 15);
                  const int c1 = min(max((int)(__float_as_uint(y.y) - 0x4B400000u) + z, 0), 15);
                  pair = __byte_perm((uint32_t)c0, (uint32_t)c1, 0x5410);
                }
                wd[t] = rq2 == 0 ? pair : wd[t] + (pair << (4 * rq2));
              }
#pragma unroll
            for (int t = 0; t < 4; ++t) codes[code_word(D, j, 32 * p + 2 * t)] = wd[t];
          }
          scale[g * D + j] = __float2bfloat16_rn(s);
          if (ZP) zpt[g * D + j] = (uint8_t)z;
        }
      }
    }
  }
  if (ok) {
    if (tid == 0) st.m[unit] = do_flush ? 0 : mt;
  } else if (tid == 0) {
    atomicOr(st.status, 1);
    mbar_wait(bar, pending, WAIT_NS);                 // let the MMAs in flight drain before TMEM is released
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TCOLS);
}

template <int G, int ZP>
static cudaError_t launch_col_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  static bool opted = false;
  if (!opted) {
    cudaError_t e = cudaFuncSetAttribute(decode_col_kernel<G, ZP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dcol::SMEM);
    if (e != cudaSuccess) return e;
    opted = true;
  }
  const unsigned units = (unsigned)(d.B * d.H4);
  if (units == 0) return cudaSuccess;
  decode_col_kernel<G, ZP><<<units, dcol::NT, dcol::SMEM, s>>>(d, io, has_token);
  return cudaGetLastError();
}

}  // namespace pace

// The int4 pool of a state with d = 128, an int8 buffer and dP <= 8 (the PACE-4 and PACE-4/8 int4 heads).
bool pace_decode_col_supported(const PaceDev &d) {
  return d.D == 128 && d.buf_mode == PACE_BUF_INT8 && d.dP <= pace::dcol::MAXP && d.state_mode == PACE_STATE_QUANT &&
         d.gamma == 1;
}

cudaError_t pace_launch_decode_col(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  if (d.zero_point) return d.G == 64 ? launch_col_t<64, 1>(d, io, has_token, s) : launch_col_t<32, 1>(d, io, has_token, s);
  return d.G == 64 ? launch_col_t<64, 0>(d, io, has_token, s) : launch_col_t<32, 0>(d, io, has_token, s);
}
