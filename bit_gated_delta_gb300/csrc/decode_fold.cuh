// PACE decode step with fused flush, on the folded readout ([P1] 어떻게 동작하나: round once every dP tokens,
// the buffered tokens applied together at the flush; [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// Between two roundings the state of a unit is S_t = G_t S_hat + sum_{s<=t} (G_t/G_s) k_s u_s^T, G_t = a_1 .. a_t,
// so replaying the m buffered tokens is one unit lower-triangular system per column j, shared by all columns:
//   (I + L) u_j = diag(beta) r_j,   r_tj = v_tj - G_t (S_hat^T k_t)_j,   L_ts = beta_t (G_t/G_s) k_s.k_t  (s < t).
// The output of the step does not need u. With cq_s = (G_m/G_s) k_s.q and c = diag(beta) (I + L)^-T cq,
//   o = S_m^T q = G_m S_hat^T q + sum_s cq_s u_s = S_hat^T y + V^T c,   y = G_m q - sum_t c_t G_t k_t,
// so a step without a rounding reads the packed state once against a single vector y. The per-unit work is an
// m x m Gram matrix of the buffered int8 keys (fp16 tensor-core MMAs, 16 keys each, exact in fp32), a back
// substitution across lanes, and y; the state is then contracted with y's three int8 digits (a 24-bit fixed-point
// image) on the tensor cores, straight from the packed nibbles:
//   M = state columns (A: the lane's own packed words as fp16 1024 + u, or 1024 + 16u for the second 8 keys of a
//   16-key step), N = the digit rows of y (B: fp16, second-half keys scaled by 1/16), K = keys.
// Every product and partial sum is an exact integer in fp32; each key-axis group's accumulator starts at minus the
// contribution of the zero level (computed by the same MMA from a constant operand), so the group fold is one
// paired multiply-add by the group scale. The rounding step adds the buffered keys as a second N tile, replays
// each column (four columns per lane) and requantizes the state per key-axis group as in decode_mma.cuh.
//
// The same kernel with BITS = 16 serves the buffered bf16 state (int8 decode buffer, bf16 state rounded to bf16
// once every dP tokens): the prologue (token quantization, Gram, solve, y in fp32) is shared; the state is then read
// on the CUDA cores, a row of D bf16 values per warp load, against y (and, at a rounding, against the buffered keys).
// With TK = 32 the tables hold up to 32 buffered tokens (int4 symmetric state, periods of 9 to 32): the Gram
// matrix over token tiles, a 32-lane solve, and a rounding that passes over the state once per group of 8 tokens.
#pragma once

#include <type_traits>

#include "decode_mma.cuh"

namespace pace {

constexpr int DF_TOK = 8;   // buffered tokens the tables hold by default (dP <= 8; 32-token tables: decode_fold_t32.cu)

// Four warps per unit share the token quantization and the Gram products (int4, int8 buffer, 8-token tables).
template <int WU, int BITS, int MX, int TK>
__host__ __device__ constexpr bool fold_coop() {
  return WU == 4 && BITS == 4 && !MX && TK == DF_TOK;
}
constexpr size_t FOLD_COOP_BYTES = 2048 + 16;   // 4 warps x 32 lanes x float4 partial Gram, 3 shared scales

struct FoldSmem {
  size_t krow, vrow, ydig, ssc, szp, po, pb, kbf, csx, kf, gram, qk, Lm, tk, ck, total;
};
// Per-warp work area. int8 rows use a stride of D + 16 bytes and fp16 digit rows D + 8 halves, so that the
// fragment loads of the eight rows of a tile fall in distinct banks.
__host__ __device__ inline FoldSmem fold_smem(int D, int G, int mixed, int zp, int bf = 0, int tk = DF_TOK) {
  FoldSmem L;
  size_t off = 0;
  L.krow = carve(off, (size_t)(tk + 3) * (D + 16));         // key codes of tokens 0..tk-1, then the 3 digits of q
  L.vrow = carve(off, (size_t)tk * D * (mixed ? 2 : 1));     // value codes (int8) or bf16 values
  // 32-token tables: the Gram matrix and then L share one area, and the rounding step's key table is built after
  // the replay over the values and that area (both dead by then), so that six units fit on an SM
  if (tk > DF_TOK) L.gram = L.Lm = carve(off, (size_t)tk * tk * 4);
  L.ydig = carve(off, (size_t)3 * (D + 8) * 2);              // fp16 digit rows of y; packed int4 keys of the
                                                             // mixed buffer while staging
  L.ssc = carve(off, bf ? 0 : (size_t)(D / G) * D * 2);      // group scales (bf16), as resident
  L.szp = carve(off, zp ? (size_t)(D / G) * D : 0);          // zero points
  L.po = carve(off, (size_t)D * 4);                          // S_hat^T y per column
  L.pb = carve(off, (size_t)tk * D * 4);                     // rounding step: P_t then u_t [t][j]
  if (tk > DF_TOK) {
    L.kbf = L.vrow;                                          // fp16 key pairs [i][tk/2], after the replay
    L.csx = carve(off, 0);                                   // (pb alone holds the staged code words)
  } else {
    L.kbf = carve(off, (size_t)D * 4 * 4 * (bf ? 2 : 1));    // flush B operand: fp16 pairs of int8 keys [i][pair];
                                                             // bf16 state: the keys as fp32 [i][t] (kf)
    // steps without a rounding: the unit's int4 code words are staged over pb, kbf and this spare area
    L.csx = carve(off, !bf && (size_t)D * D / 2 > (L.kbf - L.pb) + (size_t)D * 16
                           ? (size_t)D * D / 2 - (L.kbf - L.pb) - (size_t)D * 16 : 0);
  }
  L.kf = L.kbf;
  if (tk <= DF_TOK) L.gram = carve(off, 64 * 4);             // k_s.k_t (integers)
  L.qk = carve(off, 3 * (size_t)tk * 4);                     // (q digit d).k_t (integers)
  if (tk <= DF_TOK) L.Lm = carve(off, 64 * 4);               // L[t][s]
  L.tk = carve(off, (size_t)tk * 16);                        // per token: G_t s_kt, beta_t, s_vt, 0
  L.ck = carve(off, (size_t)tk * 4);                         // flush coefficient (G_m/G_s) s_ks
  L.total = carve(off, 0, 16);
  return L;
}

__device__ __forceinline__ void imma_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds32(const void *p) { return *reinterpret_cast<const uint32_t *>(p); }
// Signed byte e of x as a float.
__device__ __forceinline__ float sbyte(uint32_t x, int e) { return (float)(int)(int8_t)(x >> (8 * e)); }
// N consecutive outputs from element idx (N = 1, 2 or 4; the output pointer is 16-byte aligned, idx a multiple of N).
template <int N>
__device__ __forceinline__ void store_io_vec(void *p, size_t idx, const float (&x)[N], int io) {
  if (io == PACE_IO_F32) {
    float *f = static_cast<float *>(p) + idx;
    if constexpr (N == 4) *reinterpret_cast<float4 *>(f) = make_float4(x[0], x[1], x[2], x[3]);
    else if constexpr (N == 2) *reinterpret_cast<float2 *>(f) = make_float2(x[0], x[1]);
    else f[0] = x[0];
  } else {
    __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(p) + idx;
    if constexpr (N == 4) *reinterpret_cast<uint2 *>(h) = make_uint2(bf16x2_bits(x[0], x[1]), bf16x2_bits(x[2], x[3]));
    else if constexpr (N == 2) *reinterpret_cast<uint32_t *>(h) = bf16x2_bits(x[0], x[1]);
    else h[0] = __float2bfloat16_rn(x[0]);
  }
}

// N consecutive bf16 values of the bf16 state as floats (N = 1, 2 or 4; 2N-byte aligned).
template <int N>
__device__ __forceinline__ void df_load_bf16(const __nv_bfloat16 *p, float (&x)[N]) {
  if constexpr (N == 4) {
    const uint2 v = ldg_v2(p);
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  } else if constexpr (N == 2) {
    const uint32_t v = ldg_u32(p);
    x[0] = bf16_lo(v); x[1] = bf16_hi(v);
  } else {
    x[0] = __bfloat162float(*p);
  }
}
// Raw N-element bf16 rows (N = 1, 2, 4): load and unpack, so that loads can run ahead of their use.
template <int N> struct Bf16Raw { uint32_t w[(N + 1) / 2]; };
template <int N>
__device__ __forceinline__ Bf16Raw<N> df_ldraw(const __nv_bfloat16 *p) {
  Bf16Raw<N> r;
  if constexpr (N == 4) {
    const uint2 v = ldg_v2(p);
    r.w[0] = v.x;
    r.w[1] = v.y;
  } else if constexpr (N == 2) {
    r.w[0] = ldg_u32(p);
  } else {
    r.w[0] = (uint32_t)*reinterpret_cast<const uint16_t *>(p);
  }
  return r;
}
template <int N>
__device__ __forceinline__ float df_raw_at(const Bf16Raw<N> &r, int c) {
  return (c & 1) ? bf16_hi(r.w[c >> 1]) : bf16_lo(r.w[c >> 1]);
}

// N floats rounded to bf16 (nearest, ties to even) into the bf16 state.
template <int N>
__device__ __forceinline__ void df_store_bf16(__nv_bfloat16 *p, const float (&x)[N]) {
  if constexpr (N == 4) *reinterpret_cast<uint2 *>(p) = make_uint2(bf16x2_bits(x[0], x[1]), bf16x2_bits(x[2], x[3]));
  else if constexpr (N == 2) *reinterpret_cast<uint32_t *>(p) = bf16x2_bits(x[0], x[1]);
  else *p = __float2bfloat16_rn(x[0]);
}

// The lane's packed words of M-tile mt (columns 16 mt .. 16 mt + 15), one 16-byte vector per 64 keys and plane.
template <int D, int PL>
__device__ __forceinline__ void df_load_tile(const uint32_t *codes, int mt, int lane, uint32_t (&cw)[PL][D / 64][4]) {
  constexpr int NPP = D / 64;
#pragma unroll
  for (int pl = 0; pl < PL; ++pl)
#pragma unroll
    for (int pp = 0; pp < NPP; ++pp) {
      const uint4 v = ldg_v4(codes + pl * (D * D / 8) + ((mt * NPP + pp) * 32 + lane) * 4);
      cw[pl][pp][0] = v.x;
      cw[pl][pp][1] = v.y;
      cw[pl][pp][2] = v.z;
      cw[pl][pp][3] = v.w;
    }
}

// A fragment (M = columns 16mt + g8 and + 8, K = the 16 keys of step ks) from the lane's words of that M-tile.
template <int D, int PL>
__device__ __forceinline__ void df_afrag(const uint32_t (&cw)[PL][D / 64][4], int pl, int ks, uint32_t (&a)[4]) {
  const int p = ks >> 1;
  uint32_t w0 = cw[pl][p >> 1][p & 1], w1 = cw[pl][p >> 1][2 + (p & 1)];
  if (ks & 1) {
    w0 >>= 8;
    w1 >>= 8;
  }
  a[0] = (w0 & 0x000F000Fu) | 0x64006400u;
  a[1] = (w1 & 0x000F000Fu) | 0x64006400u;
  a[2] = (w0 & 0x00F000F0u) | 0x64006400u;
  a[3] = (w1 & 0x00F000F0u) | 0x64006400u;
}
// The A fragment of a constant word (every code of the tile equal).
__device__ __forceinline__ void df_afrag_const(uint32_t w, uint32_t (&a)[4]) {
  a[0] = a[1] = (w & 0x000F000Fu) | 0x64006400u;
  a[2] = a[3] = (w & 0x00F000F0u) | 0x64006400u;
}

// Offsets of one group for the B operand b (the fragments of its G/16 key steps): the MMA of a constant code word.
// off[e] = sum_i A_w[i] B[i][n] for the lane's two N columns n = 2tq, 2tq + 1 (every row of the tile is equal).
template <int KSG>
__device__ __forceinline__ void df_offset(uint32_t w, const uint32_t (*b)[2], float (&off)[2]) {
  uint32_t a[4];
  df_afrag_const(w, a);
  float d[4];
  mma_f16_z(d, a, b[0][0], b[0][1]);
#pragma unroll
  for (int kk = 1; kk < KSG; ++kk) mma_f16(d, a, b[kk][0], b[kk][1]);
  off[0] = d[0];
  off[1] = d[1];
}
// The pattern whose MMA is the plain sum of the B values of a group (second-half keys, stored / 16, count 16x).
__device__ __forceinline__ void df_afrag_ones(uint32_t (&a)[4]) {
  a[0] = a[1] = 0x3C003C00u;   // 1.0
  a[2] = a[3] = 0x4C004C00u;   // 16.0
}
template <int KSG>
__device__ __forceinline__ void df_sum(const uint32_t (*b)[2], float (&t2)[2]) {
  uint32_t a[4];
  df_afrag_ones(a);
  float d[4];
  mma_f16_z(d, a, b[0][0], b[0][1]);
#pragma unroll
  for (int kk = 1; kk < KSG; ++kk) mma_f16(d, a, b[kk][0], b[kk][1]);
  t2[0] = d[0];
  t2[1] = d[1];
}

// One unit: staging, tables, the folded readout and (at m = dP) the rounding. WU warps share the unit: each
// stages it on its own and takes D/16/WU of its M-tiles.
template <int D, int G, int BITS, int ZP, int MX, int WU, int TK = DF_TOK>
__device__ void df_unit(const PaceDev &st, const PaceIO &io, int b, int h, int unit, int has_token,
                        unsigned char *wsm, int part) {
  // BITS 4 or 8: the packed int4 / int8 state (PACE); BITS 16: the bf16 state of the buffered bf16 mode (row-major,
  // rounded to bf16 once every dP tokens, the same int8 decode buffer), contracted on the CUDA cores
  constexpr bool BF = BITS == 16;
  constexpr int CPL = D / 32, NG = D / G, MT = D / 16, NPP = D / 64, PL = BF ? 1 : BITS / 4, KS = D / 16, KSG = G / 16;
  constexpr int RS = D + 16, YS = D + 8, MTW = MT / WU, CW = D / WU, CPW = CW / 32;
  // the dot loop over M-tiles stays rolled except for the smallest tile body (int4, symmetric, two groups, int8
  // buffer): the larger bodies, fully unrolled, overflow the instruction cache
  constexpr bool DF_ROLL = !(BITS == 4 && NG <= 2 && !ZP && !MX);
  // four warps per unit (small launches): the warps share the new token's quantization and the Gram products
  // instead of each staging them, through a shared area after the block's work areas
  constexpr bool COOP = fold_coop<WU, BITS, MX, TK>();
  unsigned char *shared_area = wsm + (size_t)(WU - part) * fold_smem(D, G, MX, ZP, BF, TK).total;
  constexpr int OFF = BF ? 0 : 1 << (BITS - 1);
  constexpr int NKG = G / 8;
  static_assert(MTW >= 1 && CPW >= 1, "warps per unit");
  // TK: buffered tokens the tables hold (8, or 32 for the longer periods of the int4 symmetric state)
  static_assert(TK == DF_TOK || (TK == 32 && BITS == 4 && !ZP && !MX), "32-token tables: int4 symmetric only");
  constexpr int QR = TK;                           // first of the three q digit rows in krow
  const int lane = threadIdx.x & 31, g8 = lane >> 2, tq = lane & 3;
  const int dP = st.dP;
  const FoldSmem L = fold_smem(D, G, MX, ZP, BF, TK);
  int8_t *krow = reinterpret_cast<int8_t *>(wsm + L.krow);
  unsigned char *vrow = wsm + L.vrow;
  __half *ydig = reinterpret_cast<__half *>(wsm + L.ydig);
  __nv_bfloat16 *ssc = reinterpret_cast<__nv_bfloat16 *>(wsm + L.ssc);
  uint8_t *szp = wsm + L.szp;
  float *po = reinterpret_cast<float *>(wsm + L.po);
  float *pb = reinterpret_cast<float *>(wsm + L.pb);
  uint32_t *kbf = reinterpret_cast<uint32_t *>(wsm + L.kbf);
  float *gram = reinterpret_cast<float *>(wsm + L.gram);
  float *qk = reinterpret_cast<float *>(wsm + L.qk);
  float *Lm = reinterpret_cast<float *>(wsm + L.Lm);
  float4 *tk = reinterpret_cast<float4 *>(wsm + L.tk);
  float *ckf = reinterpret_cast<float *>(wsm + L.ck);

  uint32_t *codes = BF ? nullptr
                      : BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                                  : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
  __nv_bfloat16 *scale = BF ? nullptr : st.scale + (size_t)unit * NG * D;
  uint8_t *zpt = ZP ? st.zp + (size_t)unit * NG * D : nullptr;
  __nv_bfloat16 *Sbf = BF ? static_cast<__nv_bfloat16 *>(st.S) + (size_t)unit * D * D : nullptr;   // [i][j]
  float *kf = reinterpret_cast<float *>(wsm + L.kf);

  // ---- loads, in the order the step needs them: the count and the new token; then the buffered rows, their
  // scalars, the scales; the first code tiles once the new token is in
  const int m0 = (int)ldg_u32(st.m + unit);
  TokenIn<CPL> tin;
  dm_load_token<D>(st, io, unit, has_token, tin);
  if (m0 < 0 || m0 >= dP || (!has_token && m0 == 0)) {
    if (part == 0 && has_token && m0 != 0)       // corrupted counter: leave the unit, emit zeros
      for (int c = lane; c < D; c += 32) store_io(io.o, (long)unit * D + c, 0.0f, st.io);
    return;                                      // (or a flush with nothing pending)
  }
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const size_t ku = key_unit(st, unit);
  const int mt0 = part * MTW;
  float4 bs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);   // lane t < mt: token t's a, beta, key scale, value scale
  if (m0 > 0) {
    constexpr int rk = MX ? D / 2 : D, rv = MX ? 2 * D : D;
    const char *gk = static_cast<const char *>(st.buf_k) + ku * dP * rk;
    const char *gv = static_cast<const char *>(st.buf_v) + (size_t)unit * dP * rv;
    if (MX) {
      unsigned char *scr = reinterpret_cast<unsigned char *>(ydig);
      for (int c = lane; c < m0 * rk / 16; c += 32) cp_async16(scr + 16 * c, gk + 16 * c);
    } else {
      for (int c = lane; c < m0 * (D / 16); c += 32) {
        const int t = c / (D / 16), q = c - t * (D / 16);
        cp_async16(krow + t * RS + 16 * q, gk + 16 * c);
      }
    }
    for (int c = lane; c < m0 * rv / 16; c += 32) cp_async16(vrow + 16 * c, gv + 16 * c);
    if (lane < m0) bs = *reinterpret_cast<const float4 *>(st.buf_s + ((size_t)unit * dP + lane) * 4);
  }
  if constexpr (!BF) {
    const char *gs = reinterpret_cast<const char *>(scale);
    for (int c = lane; c < NG * D * 2 / 16; c += 32) cp_async16(reinterpret_cast<char *>(ssc) + 16 * c, gs + 16 * c);
    if (ZP) {
      const char *gz = reinterpret_cast<const char *>(zpt);
      for (int c = lane; c < NG * D / 16; c += 32) cp_async16(szp + 16 * c, gz + 16 * c);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  // steps without a rounding stage the warp's int4 code words in shared memory (issued after the new token, below);
  // the rounding step, whose work areas cover that space, keeps them in registers, two tiles ahead
  const bool smem_codes = BITS == 4 && !do_flush;
  const uint32_t *cs = reinterpret_cast<const uint32_t *>(pb);

  // ---- the new token: buffer slot m0 (global and shared), its scalars; q as three int8 digit rows
  float sq = 0.0f;                                 // scale of the q digits
  if constexpr (COOP) {
    // warp 0 quantizes k, warp 1 v, warp 2 q: each writes its rows into every warp's work area and its scale into
    // the shared slots; the buffer entry's scalars follow the barrier
    float *shs = reinterpret_cast<float *>(shared_area + 2048);
    if (has_token) {
      const int col0 = CPL * lane;
      if (part == 0) {
        float mk = 0.0f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) mk = fmaxf(mk, fabsf(tin.kx[c]));
        const float Ak = warp_max(mk);
        const bool kz = !(Ak >= FLT_MIN);
        const float rkk = kz ? 0.0f : __fdiv_rn(127.0f, Ak);
        const float sk = kz ? 0.0f : __fdiv_rn(Ak, 127.0f);
        int ck[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) ck[c] = min(max(__float2int_rn(__fmul_rn(tin.kx[c], rkk)), -127), 127);
#pragma unroll
        for (int w = 0; w < WU; ++w)
          dm_store_bytes<CPL>(reinterpret_cast<int8_t *>(wsm + (w - part) * (long)L.total + L.krow) + m0 * RS + col0, ck);
        if (key_writer(st, unit)) dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_k) + (ku * dP + m0) * D + col0, ck);
        if (lane == 0) shs[0] = sk;
      } else if (part == 1) {
        float mv = 0.0f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) mv = fmaxf(mv, fabsf(tin.vx[c]));
        const float Av = warp_max(mv);
        const bool vz = !(Av >= FLT_MIN);
        const float rvv = vz ? 0.0f : __fdiv_rn(127.0f, Av);
        const float sv = vz ? 0.0f : __fdiv_rn(Av, 127.0f);
        int cv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) cv[c] = min(max(__float2int_rn(__fmul_rn(tin.vx[c], rvv)), -127), 127);
#pragma unroll
        for (int w = 0; w < WU; ++w) dm_store_bytes<CPL>(wsm + (w - part) * (long)L.total + L.vrow + m0 * D + col0, cv);
        dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0, cv);
        if (lane == 0) shs[1] = sv;
      } else if (part == 2) {
        float mq = 0.0f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) mq = fmaxf(mq, fabsf(tin.qx[c]));
        const float Aq = warp_max(mq);
        const float QMAX = 8323072.0f;
        const bool qz = !(Aq >= FLT_MIN);
        const float sqw = qz ? 0.0f : __fdividef(Aq, QMAX);
        const float rq = qz ? 0.0f : __fdividef(QMAX, Aq);
        int d2[CPL], d1[CPL], d0[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int qi = min(max(__float2int_rn(tin.qx[c] * rq), -8323072), 8323072);
          const int q1 = (qi + 128) >> 8;
          d0[c] = qi - (q1 << 8);
          d2[c] = (q1 + 128) >> 8;
          d1[c] = q1 - (d2[c] << 8);
        }
#pragma unroll
        for (int w = 0; w < WU; ++w) {
          int8_t *kr = reinterpret_cast<int8_t *>(wsm + (w - part) * (long)L.total + L.krow);
          dm_store_bytes<CPL>(kr + QR * RS + col0, d2);
          dm_store_bytes<CPL>(kr + (QR + 1) * RS + col0, d1);
          dm_store_bytes<CPL>(kr + (QR + 2) * RS + col0, d0);
        }
        if (lane == 0) shs[2] = sqw;
      }
    }
    __syncthreads();
    if (has_token) {
      const float sk = shs[0], sv = shs[1];
      sq = shs[2];
      if (lane == m0) bs = make_float4(tin.an, tin.bn, sk, sv);
      if (part == 0 && lane == 0)
        *reinterpret_cast<float4 *>(st.buf_s + ((size_t)unit * dP + m0) * 4) = make_float4(tin.an, tin.bn, sk, sv);
    }
  } else
  if (has_token) {
    const int col0 = CPL * lane;
    float mk = 0.0f, mv = 0.0f, mq = 0.0f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      mk = fmaxf(mk, fabsf(tin.kx[c]));
      mv = fmaxf(mv, fabsf(tin.vx[c]));
      mq = fmaxf(mq, fabsf(tin.qx[c]));
    }
    const float Ak = warp_max(mk), Av = warp_max(mv), Aq = warp_max(mq);
    const int qkm = MX ? 7 : 127;
    const bool kz = !(Ak >= FLT_MIN);
    const float rkk = kz ? 0.0f : __fdiv_rn((float)qkm, Ak);
    const float sk = kz ? 0.0f : __fdiv_rn(Ak, (float)qkm);
    int ck[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) ck[c] = min(max(__float2int_rn(__fmul_rn(tin.kx[c], rkk)), -qkm), qkm);
    dm_store_bytes<CPL>(krow + m0 * RS + col0, ck);
    float sv = 0.0f;
    const bool kw = part == 0 && key_writer(st, unit);
    if (MX) {
      uint8_t *bk = static_cast<uint8_t *>(st.buf_k) + (ku * dP + m0) * (D / 2) + col0 / 2;
      if (kw) {
#pragma unroll
        for (int c = 0; c < CPL; c += 2) bk[c / 2] = (uint8_t)((ck[c] + 8) | ((ck[c + 1] + 8) << 4));
      }
      __nv_bfloat16 *bv = static_cast<__nv_bfloat16 *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0;
      uint32_t *vr = reinterpret_cast<uint32_t *>(vrow + ((size_t)m0 * D + col0) * 2);
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        const __nv_bfloat162 pv = __floats2bfloat162_rn(tin.vx[c], tin.vx[c + 1]);
        if (part == 0) *reinterpret_cast<__nv_bfloat162 *>(bv + c) = pv;
        vr[c / 2] = *reinterpret_cast<const uint32_t *>(&pv);
      }
    } else {
      const bool vz = !(Av >= FLT_MIN);
      const float rvv = vz ? 0.0f : __fdiv_rn(127.0f, Av);
      sv = vz ? 0.0f : __fdiv_rn(Av, 127.0f);
      int cv[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) cv[c] = min(max(__float2int_rn(__fmul_rn(tin.vx[c], rvv)), -127), 127);
      if (kw) dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_k) + (ku * dP + m0) * D + col0, ck);
      if (part == 0) dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0, cv);
      dm_store_bytes<CPL>(vrow + m0 * D + col0, cv);
    }
    if (lane == m0) bs = make_float4(tin.an, tin.bn, sk, sv);
    if (part == 0 && lane == 0)
      *reinterpret_cast<float4 *>(st.buf_s + ((size_t)unit * dP + m0) * 4) = make_float4(tin.an, tin.bn, sk, sv);
    // q ~= sq (65536 d2 + 256 d1 + d0), balanced base-256 digits in [-128, 127] (rows 8, 9, 10)
    const float QMAX = 8323072.0f;
    const bool qz = !(Aq >= FLT_MIN);
    sq = qz ? 0.0f : __fdividef(Aq, QMAX);       // internal digit scale: any sq ~ Aq/QMAX with rq ~ 1/sq works
    const float rq = qz ? 0.0f : __fdividef(QMAX, Aq);
    int d2[CPL], d1[CPL], d0[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int qi = min(max(__float2int_rn(tin.qx[c] * rq), -8323072), 8323072);
      const int q1 = (qi + 128) >> 8;
      d0[c] = qi - (q1 << 8);
      d2[c] = (q1 + 128) >> 8;
      d1[c] = q1 - (d2[c] << 8);
    }
    dm_store_bytes<CPL>(krow + QR * RS + col0, d2);
    dm_store_bytes<CPL>(krow + (QR + 1) * RS + col0, d1);
    dm_store_bytes<CPL>(krow + (QR + 2) * RS + col0, d0);
  }
  // the warp's first two code tiles, once the new token is in
  uint32_t cwA[PL][NPP][4], cwB[PL][NPP][4];
  if (smem_codes) {
#pragma unroll
    for (int k = 0; k < MTW * NPP; ++k)
      cp_async16(pb + (k * 32 + lane) * 4, codes + ((mt0 * NPP + k) * 32 + lane) * 4);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");    // the staging group (the codes may still land)
  } else {
    if constexpr (!BF) {
      df_load_tile<D, PL>(codes, mt0, lane, cwA);
      if (MTW > 1) df_load_tile<D, PL>(codes, mt0 + 1, lane, cwB);
    }
    cp_async_wait_all();
  }
  __syncwarp();
  if (MX) {                                        // packed int4 keys (code + 8) -> int8 rows
    const unsigned char *scr = reinterpret_cast<const unsigned char *>(ydig);
    for (int t = 0; t < m0; ++t) {
      if (lane < D / 8) {
        const uint32_t nb = *reinterpret_cast<const uint32_t *>(scr + t * (D / 2) + 4 * lane);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          lo |= (uint32_t)(((int)((nb >> (8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
          hi |= (uint32_t)(((int)((nb >> (16 + 8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
        }
        *reinterpret_cast<uint2 *>(krow + t * RS + 8 * lane) = make_uint2(lo, hi);
      }
    }
    __syncwarp();
  }

  // ---- Gram products k_s.k_t and (q digit).k_t: fp16 MMA (the int8 codes and digits are exact in fp16, every sum
  // an exact integer below 2^24), A = [keys 0..7 | q digits] (M), B = keys (N). (An int8 MMA would take the codes as
  // they are, but on this chip it runs at an eighth of the fp16 rate.)
  if constexpr (COOP) {
    // each warp two of the eight K steps; the partial fragments are summed (exact integers) by every warp
    float gacc[2][4] = {};
    const uint32_t sel = (tq & 1) ? 0x4342u : 0x4140u;
#pragma unroll
    for (int j = 0; j < KS / WU; ++j) {
      const int ks = part * (KS / WU) + j;
      const int off = 16 * ks + 4 * (tq >> 1);
      uint32_t a[4];
      a[0] = i8pair_f16(lds32(krow + g8 * RS + off), sel, false);
      a[2] = i8pair_f16(lds32(krow + g8 * RS + off + 8), sel, false);
      a[1] = g8 < 3 ? i8pair_f16(lds32(krow + (QR + g8) * RS + off), sel, false) : 0u;
      a[3] = g8 < 3 ? i8pair_f16(lds32(krow + (QR + g8) * RS + off + 8), sel, false) : 0u;
      mma_f16(gacc[j & 1], a, a[0], a[2]);
    }
    float4 *gp = reinterpret_cast<float4 *>(shared_area);
    gp[part * 32 + lane] = make_float4(gacc[0][0] + gacc[1][0], gacc[0][1] + gacc[1][1], gacc[0][2] + gacc[1][2],
                                       gacc[0][3] + gacc[1][3]);
    __syncthreads();
    float4 t = gp[lane];
#pragma unroll
    for (int w = 1; w < WU; ++w) {
      const float4 u = gp[w * 32 + lane];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    *reinterpret_cast<float2 *>(gram + g8 * 8 + 2 * tq) = make_float2(t.x, t.y);
    if (g8 < 3) *reinterpret_cast<float2 *>(qk + g8 * 8 + 2 * tq) = make_float2(t.z, t.w);
  } else if constexpr (TK == DF_TOK) {
    float gacc[4][4] = {};   // four independent chains of the K steps
    const uint32_t sel = (tq & 1) ? 0x4342u : 0x4140u;   // the lane's key pair inside its 4-byte load
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int off = 16 * ks + 4 * (tq >> 1);
      uint32_t a[4];
      a[0] = i8pair_f16(lds32(krow + g8 * RS + off), sel, false);
      a[2] = i8pair_f16(lds32(krow + g8 * RS + off + 8), sel, false);
      a[1] = g8 < 3 ? i8pair_f16(lds32(krow + (QR + g8) * RS + off), sel, false) : 0u;
      a[3] = g8 < 3 ? i8pair_f16(lds32(krow + (QR + g8) * RS + off + 8), sel, false) : 0u;
      mma_f16(gacc[ks & 3], a, a[0], a[2]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) gacc[0][e] = (gacc[0][e] + gacc[1][e]) + (gacc[2][e] + gacc[3][e]);
    *reinterpret_cast<float2 *>(gram + g8 * 8 + 2 * tq) = make_float2(gacc[0][0], gacc[0][1]);
    if (g8 < 3) *reinterpret_cast<float2 *>(qk + g8 * 8 + 2 * tq) = make_float2(gacc[0][2], gacc[0][3]);
  } else {
    // 32 tokens: M tiles = tokens 0-15, tokens 16-31, the q digits; N tiles = 8 tokens each (only those in use)
    const uint32_t sel = (tq & 1) ? 0x4342u : 0x4140u;
    const int nt = (mt + 7) >> 3;
#pragma unroll 1
    for (int nb = 0; nb < nt; ++nb) {
      float gacc[3][4] = {};
#pragma unroll 2
      for (int ks = 0; ks < KS; ++ks) {
        const int off = 16 * ks + 4 * (tq >> 1);
        const int8_t *rb = krow + (8 * nb + g8) * RS + off;
        const uint32_t b0 = i8pair_f16(lds32(rb), sel, false), b1 = i8pair_f16(lds32(rb + 8), sel, false);
#pragma unroll
        for (int ma = 0; ma < 3; ++ma) {
          if (ma < 2 && 16 * ma >= mt) continue;
          const int r0 = ma < 2 ? 16 * ma + g8 : QR + g8, r1 = 16 * ma + 8 + g8;
          const bool v0 = ma < 2 || g8 < 3, v1 = ma < 2;
          uint32_t a[4];
          a[0] = v0 ? i8pair_f16(lds32(krow + r0 * RS + off), sel, false) : 0u;
          a[2] = v0 ? i8pair_f16(lds32(krow + r0 * RS + off + 8), sel, false) : 0u;
          a[1] = v1 ? i8pair_f16(lds32(krow + r1 * RS + off), sel, false) : 0u;
          a[3] = v1 ? i8pair_f16(lds32(krow + r1 * RS + off + 8), sel, false) : 0u;
          mma_f16(gacc[ma], a, b0, b1);
        }
      }
      const int cn = 8 * nb + 2 * tq;              // the fragment's two token columns
#pragma unroll
      for (int ma = 0; ma < 2; ++ma) {
        if (16 * ma >= mt) continue;
        *reinterpret_cast<float2 *>(gram + (16 * ma + g8) * TK + cn) = make_float2(gacc[ma][0], gacc[ma][1]);
        *reinterpret_cast<float2 *>(gram + (16 * ma + 8 + g8) * TK + cn) = make_float2(gacc[ma][2], gacc[ma][3]);
      }
      if (g8 < 3) *reinterpret_cast<float2 *>(qk + g8 * TK + cn) = make_float2(gacc[2][0], gacc[2][1]);
    }
  }
  __syncwarp();

  // the next launch on the stream may place its blocks from here (programmatic dependent launch): at entry they
  // would crowd the SMs of a small launch while its units stage (measured on the 16-head layer shape, per launch
  // at 48 / 128 / 256 units: trigger at entry 6.57 / 6.69 / 6.78 us, at the end of the unit 5.17 / 5.37 / 5.65, here
  // 4.88 / 5.06 / 5.38; at 512-4096 units here and at entry are within 1%)
  pdl_trigger();
  // ---- per-token tables (lane s = token s): decay products, L's column s, the flush coefficient
  const int s = lane;
  const float a_s = bs.x, beta_s = bs.y, sk_s = bs.z, sv_s = bs.w;
  float Gs = 1.0f, gmr = 1.0f;                     // G_s = a_1 .. a_s ; G_m / G_s
  float Lc[TK];                                    // L_ts = beta_t (G_t/G_s) s_ks s_kt (k_s.k_t), t > s
  {
    float grow[TK];
    if constexpr (TK == DF_TOK) {
      *reinterpret_cast<float4 *>(grow) = *reinterpret_cast<const float4 *>(gram + (s & 7) * 8);
      *reinterpret_cast<float4 *>(grow + 4) = *reinterpret_cast<const float4 *>(gram + (s & 7) * 8 + 4);
    } else {
#pragma unroll
      for (int q4 = 0; q4 < TK / 4; ++q4)
        *reinterpret_cast<float4 *>(grow + 4 * q4) = *reinterpret_cast<const float4 *>(gram + s * TK + 4 * q4);
    }
    const float bsk = beta_s * sk_s;
    float p = 1.0f;                                // a_{s+1} .. a_t
#pragma unroll
    for (int t = 0; t < TK; ++t) {
      const float at = __shfl_sync(0xffffffffu, a_s, t);
      const float bt = __shfl_sync(0xffffffffu, bsk, t);
      if (t <= s) Gs *= at;
      if (t > s && t < mt) p *= at;
      if (t == mt - 1) gmr = p;
      Lc[t] = (t > s && t < mt) ? bt * p * sk_s * grow[t] : 0.0f;
    }
  }
  const float Gm = __shfl_sync(0xffffffffu, Gs, mt - 1);
  if constexpr (TK > DF_TOK) __syncwarp();         // every Gram row is read before L takes its place
  if (do_flush) {
    if (s < mt) {
      tk[s] = make_float4(Gs * sk_s, beta_s, MX ? 1.0f : sv_s, 0.0f);
      ckf[s] = gmr * sk_s;
#pragma unroll
      for (int t = 0; t < TK; ++t) Lm[t * TK + s] = Lc[t];
    }
    // the flush B operand: kbf[i][p] = fp16 pair (k_{2p,i}, k_{2p+1,i}), zero for tokens >= mt (32-token
    // tables: built after the replay, below)
    if constexpr (!BF && TK == DF_TOK) {
      const int p = lane & 3, t0 = 2 * p;
      const bool z0 = t0 >= mt, z1 = t0 + 1 >= mt;
#pragma unroll
      for (int it = 0; it < D / 32; ++it) {
        const int i0 = 4 * ((lane >> 2) + 8 * it);
        const uint32_t r0 = z0 ? 0u : lds32(krow + t0 * RS + i0);
        const uint32_t r1 = z1 ? 0u : lds32(krow + (t0 + 1) * RS + i0);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 hk = __floats2half2_rn(sbyte(r0, e), sbyte(r1, e));
          kbf[(i0 + e) * 4 + p] = *reinterpret_cast<const uint32_t *>(&hk);
        }
      }
    }
  }

  // ---- the folded readout: c = diag(beta) (I + L)^-T cq, y = G_m q - sum_t c_t G_t s_kt k_t, its digits
  uint32_t yb[KS][2];                              // B fragments of the y digit rows (lanes g8 < 3)
  float cvs = 0.0f;                                // c_s times the value scale (value coefficient of token s)
  float wd0 = 0.0f, wd1 = 0.0f;                    // weights of the lane's two digit columns
  if (has_token) {
    const int sq8 = TK == DF_TOK ? (s & 7) : s;
    const float kq = (65536.0f * qk[sq8] + 256.0f * qk[TK + sq8] + qk[2 * TK + sq8]) * sq;
    float z = s < mt ? gmr * sk_s * kq : 0.0f;     // cq_s, then z_s of (I + L)^T z = cq
#pragma unroll
    for (int t = TK - 1; t >= 0; --t) {
      if (t < mt) {
        const float zt = __shfl_sync(0xffffffffu, z, t);
        if (s < t) z = fmaf(-Lc[t], zt, z);
      }
    }
    const float c_s = s < mt ? beta_s * z : 0.0f;
    cvs = MX ? c_s : c_s * sv_s;
    const float al = -c_s * Gs * sk_s;             // y = G_m q + sum_s al_s k_s (int8 codes)
    float y[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) y[c] = Gm * tin.qx[c];
#pragma unroll
    for (int t = 0; t < TK; ++t) {
      if (t < mt) {
        const float at = __shfl_sync(0xffffffffu, al, t);
        uint32_t kw;
        if (CPL == 4) kw = lds32(krow + t * RS + 4 * lane);
        else kw = *reinterpret_cast<const uint16_t *>(krow + t * RS + 2 * lane);
#pragma unroll
        for (int c = 0; c < CPL; ++c) y[c] = fmaf(at, sbyte(kw, c), y[c]);
      }
    }
    if constexpr (BF) {                            // the bf16 state: y in fp32 (ydig area), read by every lane
      float *yf = reinterpret_cast<float *>(ydig);
#pragma unroll
      for (int c = 0; c < CPL; ++c) yf[CPL * lane + c] = y[c];
    } else {
    float my = 0.0f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) my = fmaxf(my, fabsf(y[c]));
    const float Ay = warp_max(my);
    const float QMAX = 8323072.0f;
    const bool yz = !(Ay >= FLT_MIN);
    const float sy = yz ? 0.0f : __fdividef(Ay, QMAX);
    const float ry = yz ? 0.0f : __fdividef(QMAX, Ay);
    // keys of the lane: CPL*lane .. ; all in the first or all in the second half of a 16-key step
    const float hs = ((CPL * lane) & 8) ? 0.0625f : 1.0f;
    float dg[3][CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int yi = min(max(__float2int_rn(y[c] * ry), -8323072), 8323072);
      const int y1 = (yi + 128) >> 8;
      const int e2 = (y1 + 128) >> 8;
      dg[0][c] = (float)e2 * hs;
      dg[1][c] = (float)(y1 - (e2 << 8)) * hs;
      dg[2][c] = (float)(yi - (y1 << 8)) * hs;
    }
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      __half *row = ydig + d * YS + CPL * lane;
      if constexpr (CPL == 4) {
        const __half2 h0 = __floats2half2_rn(dg[d][0], dg[d][1]), h1 = __floats2half2_rn(dg[d][2], dg[d][3]);
        *reinterpret_cast<uint2 *>(row) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
      } else {
        const __half2 h0 = __floats2half2_rn(dg[d][0], dg[d][1]);
        *reinterpret_cast<__half2 *>(row) = h0;
      }
    }
    wd0 = tq == 0 ? 65536.0f * sy : (tq == 1 ? sy : 0.0f);
    wd1 = tq == 0 ? 256.0f * sy : 0.0f;
    __syncwarp();
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      yb[ks][0] = g8 < 3 ? lds32(ydig + g8 * YS + 16 * ks + 2 * tq) : 0u;
      yb[ks][1] = g8 < 3 ? lds32(ydig + g8 * YS + 16 * ks + 8 + 2 * tq) : 0u;
    }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) yb[ks][0] = yb[ks][1] = 0u;
  }
  // B fragments of the buffered keys (rounding step): token tok0 + g8's keys as fp16, second halves / 16 (32-token
  // tables: one group of 8 tokens at a time, tok0 = 0, 8, 16, 24)
  uint32_t kb[KS][2];
  int tok0 = 0;
  auto load_kb = [&]() {
    const int tg = tok0 + g8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t x0 = tg < mt ? lds32(krow + tg * RS + 16 * ks + 4 * (tq >> 1)) : 0u;
      const uint32_t x1 = tg < mt ? lds32(krow + tg * RS + 16 * ks + 8 + 4 * (tq >> 1)) : 0u;
      const uint32_t sel = (tq & 1) ? 0x4342u : 0x4140u;
      kb[ks][0] = i8pair_f16(x0, sel, false);
      kb[ks][1] = i8pair_f16(x1, sel, true);
    }
  };
  if (!BF && do_flush) load_kb();

  // ---- group offsets: the contribution of the zero level (symmetric: code offset; zero point: 0) and, for zero
  // points and int8 planes, the plain sums T2
  float offy[NG][PL][2] = {}, t2y[NG][2] = {}, offk[NG][PL][2] = {}, t2k[NG][2] = {};
#pragma unroll
  for (int g = 0; g < (BF ? 0 : NG); ++g) {
#pragma unroll
    for (int pl = 0; pl < PL; ++pl) {
      // int4 symmetric: every code at 8 -> -(T1 + 8 T2); int8 symmetric: low plane 0, high plane 8; zero point: 0
      const uint32_t w = (!ZP && (BITS == 4 || pl == 1)) ? 0x88888888u : 0u;
      if (has_token) df_offset<KSG>(w, yb + g * KSG, offy[g][pl]);
      if (do_flush) df_offset<KSG>(w, kb + g * KSG, offk[g][pl]);
    }
    if (ZP) {
      if (has_token) df_sum<KSG>(yb + g * KSG, t2y[g]);
      if (do_flush) df_sum<KSG>(kb + g * KSG, t2k[g]);
    }
  }
  auto key_offsets = [&]() {                       // the key operand's offsets again (next token group)
#pragma unroll
    for (int g = 0; g < (BF ? 0 : NG); ++g) {
#pragma unroll
      for (int pl = 0; pl < PL; ++pl) {
        const uint32_t w = (!ZP && (BITS == 4 || pl == 1)) ? 0x88888888u : 0u;
        offk[g][pl][0] = offk[g][pl][1] = 0.0f;
        df_offset<KSG>(w, kb + g * KSG, offk[g][pl]);
      }
    }
  };

  // the L2 prefetch of the warp's other tiles, after the tables (requested earlier, it delays the staging loads)
  if (smem_codes) {
    cp_async_wait_all();
    __syncwarp();
  } else if (!BF && MTW > 2 && lane < PL) {
    constexpr uint32_t TW = NPP * 128;             // words of one M-tile in a plane
    prefetch_l2(codes + lane * (D * D / 8) + (mt0 + 2) * TW, (MTW - 2) * TW * 4);
  }

  // ---- dots over the warp's M-tiles: o part (y digits) and, at a rounding, P_t (keys). Two instantiations of the
  // loop, so that a step without a rounding carries none of the rounding step's work.
  auto dots = [&](auto with_keys) {
    constexpr bool WK = decltype(with_keys)::value;
    const bool wy = WK ? has_token != 0 && tok0 == 0 : true;   // (steps without a rounding always have a token)
    // TP tiles at a time (two on steps without a rounding, from registers cwA, cwB): their accumulators of every
    // group are independent chains, issued interleaved so that the tensor pipe always has work from this warp (the
    // rounding step, with twice the accumulators, takes one tile at a time)
    constexpr int TP = 1;
    static_assert(MTW % 2 == 0, "tiles are loaded in pairs");
    // one M-tile; PAR = the tile's parity, which selects its register buffer (cwA even, cwB odd)
    auto tile = [&](const int mi, auto par) {
      constexpr int PAR = decltype(par)::value;
      float ay[TP][NG][PL][4], ak[TP][NG][PL][4];
#pragma unroll
      for (int tt = 0; tt < TP; ++tt)
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
          for (int pl = 0; pl < PL; ++pl) {
            ay[tt][g][pl][0] = ay[tt][g][pl][2] = -offy[g][pl][0];
            ay[tt][g][pl][1] = ay[tt][g][pl][3] = -offy[g][pl][1];
            if (WK) {
              ak[tt][g][pl][0] = ak[tt][g][pl][2] = -offk[g][pl][0];
              ak[tt][g][pl][1] = ak[tt][g][pl][3] = -offk[g][pl][1];
            }
          }
      constexpr bool SM = !WK && BITS == 4;        // words from shared memory
      if (SM) {
#pragma unroll
        for (int tt = 0; tt < TP; ++tt)
#pragma unroll
          for (int pp = 0; pp < NPP; ++pp) {
            const uint4 v = *reinterpret_cast<const uint4 *>(cs + (((mi + tt) * NPP + pp) * 32 + lane) * 4);
            uint32_t(&w)[PL][NPP][4] = (PAR ^ (tt & 1)) ? cwB : cwA;
            w[0][pp][0] = v.x;
            w[0][pp][1] = v.y;
            w[0][pp][2] = v.z;
            w[0][pp][3] = v.w;
          }
      }
#pragma unroll
      for (int kk = 0; kk < KSG; ++kk)
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
          for (int tt = 0; tt < TP; ++tt) {
            const int ks = g * KSG + kk;
#pragma unroll
            for (int pl = 0; pl < PL; ++pl) {
              uint32_t a[4];
              df_afrag<D, PL>((PAR ^ (tt & 1)) ? cwB : cwA, pl, ks, a);
              mma_f16(ay[tt][g][pl], a, yb[ks][0], yb[ks][1]);
              if (WK) mma_f16(ak[tt][g][pl], a, kb[ks][0], kb[ks][1]);
            }
          }
      // these tiles' words are done with (the rounding reloads them from L2): the tiles two ahead take their registers
      if (!SM) {
#pragma unroll
        for (int tt = 0; tt < TP; ++tt)
          if (mi + tt + 2 < MTW) df_load_tile<D, PL>(codes, mt0 + mi + tt + 2, lane, (PAR ^ (tt & 1)) ? cwB : cwA);
      }
#pragma unroll
      for (int tt = 0; tt < TP; ++tt) {
        const int mtile = mt0 + mi + tt;
        const int j0 = 16 * mtile + g8, j1 = j0 + 8;
        float oc[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};   // [column][digit] folded over groups
        float pk[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};   // [column][token]
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          // fold the group: exact integer level sums, times the group scale
          const float s0 = __bfloat162float(ssc[g * D + j0]), s1 = __bfloat162float(ssc[g * D + j1]);
          float z0 = 0.0f, z1 = 0.0f;
          if (ZP) {
            z0 = (float)szp[g * D + j0];
            z1 = (float)szp[g * D + j1];
          }
          auto level = [&](const float (&x)[PL][4], int e, float zc, const float (&t2)[2]) -> float {
            float v = PL == 2 ? fmaf(16.0f, x[PL - 1][e], x[0][e]) : x[0][e];
            if (ZP) v = fmaf(-zc, t2[e & 1], v);
            return v;
          };
          oc[0][0] = fmaf(s0, level(ay[tt][g], 0, z0, t2y[g]), oc[0][0]);
          oc[0][1] = fmaf(s0, level(ay[tt][g], 1, z0, t2y[g]), oc[0][1]);
          oc[1][0] = fmaf(s1, level(ay[tt][g], 2, z1, t2y[g]), oc[1][0]);
          oc[1][1] = fmaf(s1, level(ay[tt][g], 3, z1, t2y[g]), oc[1][1]);
          if (WK) {
            pk[0][0] = fmaf(s0, level(ak[tt][g], 0, z0, t2k[g]), pk[0][0]);
            pk[0][1] = fmaf(s0, level(ak[tt][g], 1, z0, t2k[g]), pk[0][1]);
            pk[1][0] = fmaf(s1, level(ak[tt][g], 2, z1, t2k[g]), pk[1][0]);
            pk[1][1] = fmaf(s1, level(ak[tt][g], 3, z1, t2k[g]), pk[1][1]);
          }
        }
        if (wy) {
          float o0 = fmaf(wd1, oc[0][1], wd0 * oc[0][0]), o1 = fmaf(wd1, oc[1][1], wd0 * oc[1][0]);
          o0 += __shfl_xor_sync(0xffffffffu, o0, 1);
          o1 += __shfl_xor_sync(0xffffffffu, o1, 1);
          if (tq == 0) po[j0] = o0;
          else if (tq == 1) po[j1] = o1;
        }
        if (WK) {
          const int t0 = tok0 + 2 * tq;
          if (t0 < mt) {
            pb[t0 * D + j0] = pk[0][0];
            pb[t0 * D + j1] = pk[1][0];
          }
          if (t0 + 1 < mt) {
            pb[(t0 + 1) * D + j0] = pk[0][1];
            pb[(t0 + 1) * D + j1] = pk[1][1];
          }
        }
      }
    };
    // the tiles in pairs; a rolled loop where the unrolled one would overflow the instruction cache (more groups,
    // zero points, the mixed buffer or int8 planes make the tile body several times larger)
    if constexpr (DF_ROLL) {
#pragma unroll 1
      for (int mi = 0; mi < MTW; mi += 2) {
        tile(mi, std::integral_constant<int, 0>{});
        tile(mi + 1, std::integral_constant<int, 1>{});
      }
    } else {
#pragma unroll
      for (int mi = 0; mi < MTW; mi += 2) {
        tile(mi, std::integral_constant<int, 0>{});
        tile(mi + 1, std::integral_constant<int, 1>{});
      }
    }
  };
  if constexpr (BF) {
    // ---- the bf16 state on the CUDA cores: lane = CPW consecutive columns (8-, 4- or 2-byte loads, coalesced
    // across the warp), rows streamed through a window of loads in flight (32 rows on a step without a rounding, 8
    // at a rounding, where the registers also hold the eight key dots); S_hat^T y into po, and at a rounding
    // S_hat^T k_t (key codes) into pb
    const float *yf = reinterpret_cast<const float *>(ydig);
    const int jb = part * CW + CPW * lane;
    __syncwarp();                                  // y, written by every lane, is read by every lane
    if (do_flush) {                                // the keys as fp32 [i][t] (zero for t >= mt)
      for (int idx = lane; idx < D * DF_TOK; idx += 32) {
        const int i = idx >> 3, t = idx & 7;
        kf[idx] = t < mt ? (float)krow[t * RS + i] : 0.0f;
      }
      __syncwarp();
    }
    float acc[CPW] = {};
    if (!do_flush) {
      // rows streamed through a window of PD loads in flight (row r + PD requested as row r is used)
      constexpr int PD = 32;
      Bf16Raw<CPW> win[PD];
#pragma unroll
      for (int r = 0; r < PD; ++r) win[r] = df_ldraw<CPW>(Sbf + (size_t)r * D + jb);
#pragma unroll 1
      for (int i0 = 0; i0 < D; i0 += PD) {
#pragma unroll
        for (int rr = 0; rr < PD; ++rr) {
          const Bf16Raw<CPW> v = win[rr];
          if (i0 + PD < D) win[rr] = df_ldraw<CPW>(Sbf + (size_t)(i0 + PD + rr) * D + jb);
          const float yi = yf[i0 + rr];
#pragma unroll
          for (int c = 0; c < CPW; ++c) acc[c] = fmaf(yi, df_raw_at<CPW>(v, c), acc[c]);
        }
      }
    } else {
      float pk[DF_TOK][CPW] = {};
      constexpr int PD = 8;
      Bf16Raw<CPW> win[PD];
#pragma unroll
      for (int r = 0; r < PD; ++r) win[r] = df_ldraw<CPW>(Sbf + (size_t)r * D + jb);
#pragma unroll 1
      for (int i0 = 0; i0 < D; i0 += PD) {
#pragma unroll
        for (int rr = 0; rr < PD; ++rr) {
          const Bf16Raw<CPW> v = win[rr];
          if (i0 + PD < D) win[rr] = df_ldraw<CPW>(Sbf + (size_t)(i0 + PD + rr) * D + jb);
          const float yi = has_token ? yf[i0 + rr] : 0.0f;
          const float4 ka = *reinterpret_cast<const float4 *>(kf + (i0 + rr) * DF_TOK);
          const float4 kb4 = *reinterpret_cast<const float4 *>(kf + (i0 + rr) * DF_TOK + 4);
          const float kr[8] = {ka.x, ka.y, ka.z, ka.w, kb4.x, kb4.y, kb4.z, kb4.w};
#pragma unroll
          for (int c = 0; c < CPW; ++c) {
            const float x = df_raw_at<CPW>(v, c);
            acc[c] = fmaf(yi, x, acc[c]);
#pragma unroll
            for (int t = 0; t < DF_TOK; ++t) pk[t][c] = fmaf(kr[t], x, pk[t][c]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < DF_TOK; ++t)
        if (t < mt) {
#pragma unroll
          for (int c = 0; c < CPW; ++c) pb[t * D + jb + c] = pk[t][c];
        }
    }
    if (has_token) {
#pragma unroll
      for (int c = 0; c < CPW; ++c) po[jb + c] = acc[c];
    }
  } else {
    if (!do_flush) {
      dots(std::false_type{});
    } else if constexpr (TK == DF_TOK) {
      dots(std::true_type{});
    } else {
      // 32-token tables: one pass over the warp's tiles per group of 8 buffered tokens (the first pass also
      // contracts y); each later pass reloads its first two tiles (from L2) and the key fragments
#pragma unroll 1
      for (tok0 = 0; tok0 == 0 || tok0 < mt; tok0 += 8) {
        if (tok0 > 0) {
          load_kb();
          key_offsets();
          df_load_tile<D, PL>(codes, mt0, lane, cwA);
          if (MTW > 1) df_load_tile<D, PL>(codes, mt0 + 1, lane, cwB);
        }
        dots(std::true_type{});
      }
    }
  }
  __syncwarp();

  // ---- output (lane: CPW consecutive columns of the warp's range): o = S_hat^T y + V^T c
  const int jc = part * CW + CPW * lane;
  if (has_token) {
    float o[CPW];
#pragma unroll
    for (int c = 0; c < CPW; ++c) o[c] = po[jc + c];
#pragma unroll
    for (int t = 0; t < TK; ++t) {
      if (t < mt) {
        const float cv = __shfl_sync(0xffffffffu, cvs, t);
        if (MX) {
          const __nv_bfloat16 *vr = reinterpret_cast<const __nv_bfloat16 *>(vrow) + t * D + jc;
#pragma unroll
          for (int c = 0; c < CPW; ++c) o[c] = fmaf(cv, __bfloat162float(vr[c]), o[c]);
        } else {
          const int8_t *vr = reinterpret_cast<const int8_t *>(vrow) + t * D + jc;
#pragma unroll
          for (int c = 0; c < CPW; ++c) o[c] = fmaf(cv, (float)vr[c], o[c]);
        }
      }
    }
    store_io_vec<CPW>(io.o, (size_t)unit * D + jc, o, st.io);
  }

  if (do_flush) {
    // ---- replay of the lane's columns: u_t = beta_t r_t - sum_{s<t} L_ts u_s, r_t = v_t - G_t s_kt P_t
    float u[DF_TOK][CPW];
    if constexpr (TK > DF_TOK) {
      // 32-token tables: u_t replaces P_t in pb as it is found (the lane's own columns, so no barrier)
      const int8_t *v8 = reinterpret_cast<const int8_t *>(vrow);
#pragma unroll 1
      for (int t = 0; t < mt; ++t) {
        const float4 tt = tk[t];
        float acc[CPW];
#pragma unroll
        for (int c = 0; c < CPW; ++c) acc[c] = tt.y * fmaf(-tt.x, pb[t * D + jc + c], tt.z * (float)v8[t * D + jc + c]);
#pragma unroll 4
        for (int s2 = 0; s2 < t; ++s2) {
          const float l = Lm[t * TK + s2];
#pragma unroll
          for (int c = 0; c < CPW; ++c) acc[c] = fmaf(-l, pb[s2 * D + jc + c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < CPW; ++c) pb[t * D + jc + c] = acc[c];
      }
      __syncwarp();
      // the rounding's key table over the values and L (both read for the last time above): kbf[i][p] = fp16
      // pair (k_{2p,i}, k_{2p+1,i}), p < TK/2, zero for tokens >= mt
      for (int idx = lane; idx < D * (TK / 2); idx += 32) {
        const int i = idx / (TK / 2), t0 = 2 * (idx - i * (TK / 2));
        const float k0 = t0 < mt ? (float)krow[t0 * RS + i] : 0.0f;
        const float k1 = t0 + 1 < mt ? (float)krow[(t0 + 1) * RS + i] : 0.0f;
        const __half2 hk = __floats2half2_rn(k0, k1);
        kbf[idx] = *reinterpret_cast<const uint32_t *>(&hk);
      }
    } else {
#pragma unroll
    for (int t = 0; t < DF_TOK; ++t) {
      if (t < mt) {
        const float4 tt = tk[t];
        float acc[CPW];
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
          const float v = MX ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(vrow)[t * D + jc + c])
                             : tt.z * (float)reinterpret_cast<const int8_t *>(vrow)[t * D + jc + c];
          acc[c] = tt.y * fmaf(-tt.x, pb[t * D + jc + c], v);
        }
#pragma unroll
        for (int s2 = 0; s2 < t; ++s2) {
          const float l = Lm[t * TK + s2];
#pragma unroll
          for (int c = 0; c < CPW; ++c) acc[c] = fmaf(-l, u[s2][c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
          u[t][c] = acc[c];
          pb[t * D + jc + c] = acc[c];
        }
      } else {
#pragma unroll
        for (int c = 0; c < CPW; ++c) u[t][c] = 0.0f;
      }
    }
    }
    __syncwarp();

    if constexpr (BF) {
      // ---- rounding of the bf16 state: S_new[i][j] = bf16(G_m S[i][j] + sum_s k_si (rho_s u_sj)), the lane's columns
      float w[DF_TOK][CPW];
#pragma unroll
      for (int t = 0; t < DF_TOK; ++t)
#pragma unroll
        for (int c = 0; c < CPW; ++c) w[t][c] = t < mt ? ckf[t] * u[t][c] : 0.0f;
      constexpr int PD = 8;
      Bf16Raw<CPW> win[PD];
#pragma unroll
      for (int r = 0; r < PD; ++r) win[r] = df_ldraw<CPW>(Sbf + (size_t)r * D + jc);
#pragma unroll 1
      for (int i0 = 0; i0 < D; i0 += PD) {
#pragma unroll
        for (int rr = 0; rr < PD; ++rr) {
          const Bf16Raw<CPW> v = win[rr];
          if (i0 + PD < D) win[rr] = df_ldraw<CPW>(Sbf + (size_t)(i0 + PD + rr) * D + jc);
          const float4 ka = *reinterpret_cast<const float4 *>(kf + (i0 + rr) * DF_TOK);
          const float4 kb4 = *reinterpret_cast<const float4 *>(kf + (i0 + rr) * DF_TOK + 4);
          const float kr[8] = {ka.x, ka.y, ka.z, ka.w, kb4.x, kb4.y, kb4.z, kb4.w};
          float x[CPW];
#pragma unroll
          for (int c = 0; c < CPW; ++c) {
            float vv = Gm * df_raw_at<CPW>(v, c);
#pragma unroll
            for (int t = 0; t < DF_TOK; ++t) vv = fmaf(kr[t], w[t][c], vv);
            x[c] = vv;
          }
          df_store_bf16<CPW>(Sbf + (size_t)(i0 + rr) * D + jc, x);
        }
      }
    } else {
    // ---- rounding of the warp's M-tiles: S_new^T[j][i] = sum_s rho_s u_sj k_si + G_m s_gj (u_ij - z_gj)
    constexpr int KP = TK / 2;                     // token pairs in a row of the key table kbf
    uint32_t cwn[PL][NPP][4];                      // the next tile's words, requested one tile ahead
    df_load_tile<D, PL>(codes, mt0, lane, cwn);
#pragma unroll 1
    for (int mi = 0; mi < MTW; ++mi) {
      const int mtile = mt0 + mi;
      uint32_t cw[PL][NPP][4];
#pragma unroll
      for (int pl = 0; pl < PL; ++pl)
#pragma unroll
        for (int pp = 0; pp < NPP; ++pp)
#pragma unroll
          for (int e = 0; e < 4; ++e) cw[pl][pp][e] = cwn[pl][pp][e];
      if (mi + 1 < MTW) df_load_tile<D, PL>(codes, mtile + 1, lane, cwn);
      // A: rho_s u_s,j for tokens 2tq, 2tq + 1 and columns 16 mtile + g8, + 8, times a power of two 2^e_j per column
      // that puts the column's largest |rho_s u_s,j| in [2^8, 2^9), as two fp16 parts (about 22 significant bits;
      // K = 16 = 8 tokens x 2 parts, one MMA per key tile). The old state is scaled by the same 2^e_j, so the
      // accumulator holds 2^e_j x; scales and codes are invariant under it (the scale found is divided back).
      uint32_t a16[TK / 8][4];                     // one A fragment per group of 8 tokens
      float pw2[2], pw2i[2];
      if constexpr (TK == DF_TOK) {
        uint32_t ap[2][2];
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int j = 16 * mtile + g8 + 8 * hi, s0 = 2 * tq;
          float x0 = s0 < mt ? ckf[s0] * pb[s0 * D + j] : 0.0f;
          float x1 = s0 + 1 < mt ? ckf[s0 + 1] * pb[(s0 + 1) * D + j] : 0.0f;
          float mx = fmaxf(fabsf(x0), fabsf(x1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const int e = min(max(135 - (int)((__float_as_uint(mx) >> 23) & 0xFFu), -60), 60);
          pw2[hi] = __uint_as_float((uint32_t)(e + 127) << 23);
          pw2i[hi] = __uint_as_float((uint32_t)(127 - e) << 23);
          x0 *= pw2[hi];
          x1 *= pw2[hi];
          const __half2 p0 = __floats2half2_rn(x0, x1);
          const float2 f0 = __half22float2(p0);
          const __half2 p1 = __floats2half2_rn(x0 - f0.x, x1 - f0.y);
          ap[0][hi] = *reinterpret_cast<const uint32_t *>(&p0);
          ap[1][hi] = *reinterpret_cast<const uint32_t *>(&p1);
        }
        a16[0][0] = ap[0][0];
        a16[0][1] = ap[0][1];
        a16[0][2] = ap[1][0];
        a16[0][3] = ap[1][1];
      } else {
        // 32 tokens: the column's exponent from all of its tokens, then one fragment per group of 8
        float xs[TK / 8][2][2], mxh[2] = {0.0f, 0.0f};
#pragma unroll
        for (int q = 0; q < TK / 8; ++q)
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const int j = 16 * mtile + g8 + 8 * hi, s0 = 8 * q + 2 * tq;
            xs[q][hi][0] = s0 < mt ? ckf[s0] * pb[s0 * D + j] : 0.0f;
            xs[q][hi][1] = s0 + 1 < mt ? ckf[s0 + 1] * pb[(s0 + 1) * D + j] : 0.0f;
            mxh[hi] = fmax3(mxh[hi], fabsf(xs[q][hi][0]), fabsf(xs[q][hi][1]));
          }
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          float mx = mxh[hi];
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const int e = min(max(135 - (int)((__float_as_uint(mx) >> 23) & 0xFFu), -60), 60);
          pw2[hi] = __uint_as_float((uint32_t)(e + 127) << 23);
          pw2i[hi] = __uint_as_float((uint32_t)(127 - e) << 23);
        }
#pragma unroll
        for (int q = 0; q < TK / 8; ++q)
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const float x0 = xs[q][hi][0] * pw2[hi], x1 = xs[q][hi][1] * pw2[hi];
            const __half2 p0 = __floats2half2_rn(x0, x1);
            const float2 f0 = __half22float2(p0);
            const __half2 p1 = __floats2half2_rn(x0 - f0.x, x1 - f0.y);
            a16[q][hi] = *reinterpret_cast<const uint32_t *>(&p0);
            a16[q][2 + hi] = *reinterpret_cast<const uint32_t *>(&p1);
          }
      }
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float fs[2], fz[2];
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int j = 16 * mtile + g8 + 8 * hi;
          fs[hi] = Gm * __bfloat162float(ssc[gi * D + j]) * pw2[hi];
          fz[hi] = -(8388608.0f + (float)(ZP ? (int)szp[gi * D + j] : OFF));
        }
        float c[NKG][4];
#pragma unroll
        for (int nn = 0; nn < NKG; ++nn) {
          const uint32_t *kr = kbf + (8 * (gi * NKG + nn) + g8) * KP + tq;
          mma_f16_z(c[nn], a16[0], kr[0], kr[0]);
#pragma unroll
          for (int q = 1; q < TK / 8; ++q)
            if (8 * q < mt) mma_f16(c[nn], a16[q], kr[4 * q], kr[4 * q]);
        }
        // the old state: 2^e_j x = 2^e_j G_m s_gj (u_ij - z_gj) + replay term, fp32 pairs (u - z exact)
#pragma unroll
        for (int nn = 0; nn < NKG; ++nn) {
          const int nk = gi * NKG + nn, r = nk & 3;
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const int wi = hi * 2 + ((nk >> 2) & 1);
            uint32_t m16 = (cw[0][nk >> 3][wi] >> (4 * r)) & 0x000F000Fu;
            if (BITS == 8) m16 |= ((cw[PL - 1][nk >> 3][wi] >> (4 * r)) & 0x000F000Fu) << 4;
            const float2 f = make_float2(__uint_as_float(__byte_perm(m16, 0x4B000000u, 0x7610)),
                                         __uint_as_float(__byte_perm(m16, 0x4B000000u, 0x7632)));
            const float2 d = __fadd2_rn(f, make_float2(fz[hi], fz[hi]));
            const float2 x = __ffma2_rn(make_float2(fs[hi], fs[hi]), d, make_float2(c[nn][2 * hi], c[nn][2 * hi + 1]));
            c[nn][2 * hi] = x.x;
            c[nn][2 * hi + 1] = x.y;
          }
        }
        // requantize the group for both columns; the lane's keys fill its own words
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          float sc;
          int z;
          if (!ZP) {
            float A = 0.0f;
#pragma unroll
            for (int nn = 0; nn < NKG; ++nn) A = fmax3(A, fabsf(c[nn][2 * hi]), fabsf(c[nn][2 * hi + 1]));
            A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 1));
            A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 2));
            constexpr float QMAX = (float)(OFF - 1);
            sc = bf16_quot(A, QMAX, 1.0f / QMAX);
            z = OFF;
          } else {
            float lo = 0.0f, hi_ = 0.0f;
#pragma unroll
            for (int nn = 0; nn < NKG; ++nn) {
              lo = fmin3(lo, c[nn][2 * hi], c[nn][2 * hi + 1]);
              hi_ = fmax3(hi_, c[nn][2 * hi], c[nn][2 * hi + 1]);
            }
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
            hi_ = fmaxf(hi_, __shfl_xor_sync(0xffffffffu, hi_, 1));
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 2));
            hi_ = fmaxf(hi_, __shfl_xor_sync(0xffffffffu, hi_, 2));
            constexpr float QM = (float)((1 << BITS) - 1);
            sc = bf16_quot(__fsub_rn(hi_, lo), QM, 1.0f / QM);
            z = 0;
            if (sc * pw2i[hi] >= FLT_MIN) z = min(max(__float2int_rn(__fmul_rn(-lo, rcp_bf16(sc))), 0), (1 << BITS) - 1);
          }
          // sc is 2^e_j times the scale (bf16-exact either way); a zero or subnormal scale makes the group zero
          float st = sc * pw2i[hi];
          if (!(st >= FLT_MIN)) st = sc = 0.0f;
          const float rr = sc > 0.0f ? rcp_bf16(sc) : 0.0f;
          // codes: rint(x r) by the 1.5 * 2^23 rounding constant, one fused multiply-add (the product is not
          // rounded first; it differs from rint(fl(x r)) only within 2^-24 of a half-integer) (symmetric: the clamp
          // to +-qmax never binds, since s = bf16(A / qmax) puts |x r| below qmax + 1/2); zero point: + z, clamp
          // to [0, 2^b - 1]
          const float2 r2 = make_float2(rr, rr);
          const float mg = ZP ? 12582912.0f : 12582912.0f + (float)OFF;
          const float2 mg2 = make_float2(mg, mg);
#pragma unroll
          for (int pw = 0; pw < G / 32; ++pw) {
            const int p = gi * (G / 32) + pw;      // 32-key span
            uint32_t w0 = 0, w1 = 0;
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4) {
              const int nn = 4 * pw + r4;
              const float2 yv = __ffma2_rn(make_float2(c[nn][2 * hi], c[nn][2 * hi + 1]), r2, mg2);
              uint32_t pair;
              if (!ZP) {
                pair = __byte_perm(__float_as_uint(yv.x), __float_as_uint(yv.y), 0x5410);   // bytes 1, 3 are 0
                if (BITS == 4) {                   // each half is code + 8 in 1..15: no other bit is set
                  w0 = r4 == 0 ? pair : w0 + (pair << (4 * r4));
                  continue;
                }
              } else {
                const int c0 = min(max((int)(__float_as_uint(yv.x) - 0x4B400000u) + z, 0), (1 << BITS) - 1);
                const int c1 = min(max((int)(__float_as_uint(yv.y) - 0x4B400000u) + z, 0), (1 << BITS) - 1);
                pair = __byte_perm((uint32_t)c0, (uint32_t)c1, 0x5410);
              }
              w0 += (pair & 0x000F000Fu) << (4 * r4);
              if (BITS == 8) w1 += ((pair >> 4) & 0x000F000Fu) << (4 * r4);
            }
            cw[0][p >> 1][hi * 2 + (p & 1)] = w0;
            if (BITS == 8) cw[PL - 1][p >> 1][hi * 2 + (p & 1)] = w1;
          }
          if (tq == 0) {
            const int j = 16 * mtile + g8 + 8 * hi;
            scale[gi * D + j] = __float2bfloat16_rn(st);
            if (ZP) zpt[gi * D + j] = (uint8_t)z;
          }
        }
      }
#pragma unroll
      for (int pl = 0; pl < PL; ++pl)
#pragma unroll
        for (int pp = 0; pp < NPP; ++pp)
          *reinterpret_cast<uint4 *>(codes + pl * (D * D / 8) + ((mtile * NPP + pp) * 32 + lane) * 4) =
              make_uint4(cw[pl][pp][0], cw[pl][pp][1], cw[pl][pp][2], cw[pl][pp][3]);
    }
  }
  }
  // every warp of the unit has read the count before it moves on
  if (WU > 1) __syncthreads(); else __syncwarp();
  if (threadIdx.x == 0) st.m[unit] = do_flush ? 0 : mt;
}

// One unit per block of WU warps; one launch per code pool (int4 heads, int8 heads).
template <int D, int G, int BITS, int ZP, int MX, int WU, int TK = DF_TOK>
__global__ void __launch_bounds__(WU * 32, (TK > DF_TOK ? 8 : BITS == 4 ? PACE_DM_MIN_WARPS : BITS == 16 ? 16 : 12) / WU)
    decode_fold_kernel(const PaceDev st, const PaceIO io, const int has_token, const int one_wave) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int HP = BITS == 8 ? st.H8 : st.H4;   // (the bf16 state: every head, in the first pool)
  const int w = blockIdx.x;
  if (w >= st.B * HP) {
    pdl_wait();
    return;
  }
  const int b = w / HP, slot = w - b * HP;
  const int h = st.pool_head[(BITS == 8 ? st.H4 : 0) + slot];
  // Before the wait on the previous launch: L2 prefetches of the unit's first loads (its count and the new token),
  // for a launch whose blocks are all resident at once (they may be placed while the previous launch drains). L2 is
  // where device memory is coherent, so a line the previous launch writes afterwards is still read current.
  // (Measured: -1.8% per step at 2,048 units, -2% at 48 and 1,024; with two waves, +1.6%, so not there.)
  if (one_wave && warp == 0 && has_token) {
    const int lane = threadIdx.x & 31, unit = b * st.H + h;
    const size_t ku = (size_t)key_unit(st, unit);
    const int es = st.io == PACE_IO_F32 ? 4 : 2;
    const size_t c16 = (size_t)unit * 4 & ~(size_t)15;         // the 16 bytes holding the unit's word
    const bool in16 = c16 + 16 <= (size_t)st.B * st.H * 4;       // (only where they lie inside the array)
    if (lane == 0 && in16) prefetch_l2(reinterpret_cast<const char *>(st.m) + c16, 16);
    else if (lane == 1) prefetch_l2(static_cast<const char *>(io.q) + ku * D * es, D * es);
    else if (lane == 2) prefetch_l2(static_cast<const char *>(io.k) + ku * D * es, D * es);
    else if (lane == 3) prefetch_l2(static_cast<const char *>(io.v) + (size_t)unit * D * es, D * es);
    else if (lane == 4 && in16) prefetch_l2(reinterpret_cast<const char *>(io.a) + c16, 16);
    else if (lane == 5 && in16) prefetch_l2(reinterpret_cast<const char *>(io.beta) + c16, 16);
  }
  pdl_wait();                                      // (the trigger follows the unit's Gram products, in df_unit)
  const FoldSmem L = fold_smem(D, G, MX, ZP, BITS == 16, TK);
  df_unit<D, G, BITS, ZP, MX, WU, TK>(st, io, b, h, b * st.H + h, has_token, smem + (size_t)warp * L.total, warp);
}

template <int D, int G, int BITS, int ZP, int MX, int WU, int TK = DF_TOK>
static cudaError_t launch_fold_w(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s, long units) {
  const FoldSmem L = fold_smem(D, G, MX, ZP, BITS == 16, TK);
  const size_t smem = (size_t)WU * L.total + (fold_coop<WU, BITS, MX, TK>() ? FOLD_COOP_BYTES : 0);
  cudaError_t e = smem_opt_in<decode_fold_kernel<D, G, BITS, ZP, MX, WU, TK>>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)units), dim3(WU * 32), smem, s, attr);
  const int one_wave =
      units <= (long)device_sm_count() * resident_blocks<decode_fold_kernel<D, G, BITS, ZP, MX, WU, TK>>(WU * 32, smem);
  return cudaLaunchKernelEx(&cfg, decode_fold_kernel<D, G, BITS, ZP, MX, WU, TK>, d, io, has_token, one_wave);
}

// Warps per unit by the size of the pool: while the units fill fewer than a half (a quarter) of the SMs' warp
// slots, two (four) warps share each unit and split its M-tiles, which shortens the per-unit chain.
template <int D, int G, int BITS, int ZP, int MX>
static cudaError_t launch_fold_pool(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  const long units = (long)d.B * (BITS == 8 ? d.H8 : d.H4);
  if (units == 0) return cudaSuccess;
  const long slots = (long)device_sm_count() * 16;
  if constexpr (D >= 128) {                      // (at least 32 columns per warp)
    if (units * 4 <= slots) return launch_fold_w<D, G, BITS, ZP, MX, 4>(d, io, has_token, s, units);
  }
  if (units * 2 <= slots) return launch_fold_w<D, G, BITS, ZP, MX, 2>(d, io, has_token, s, units);
  return launch_fold_w<D, G, BITS, ZP, MX, 1>(d, io, has_token, s, units);
}

// The int4 and int8 pools touch disjoint units: with both present, the int8 pool runs on the state's side stream,
// forked from s after everything already queued there and joined back before anything queued later, so the two
// launches share the SMs (each pool alone leaves part of a wave idle).
template <int D, int G, int ZP, int MX>
static cudaError_t launch_fold_pools(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  if (!d.side || d.H4 == 0 || d.H8 == 0) {
    cudaError_t e = launch_fold_pool<D, G, 4, ZP, MX>(d, io, has_token, s);
    if (e == cudaSuccess) e = launch_fold_pool<D, G, 8, ZP, MX>(d, io, has_token, s);
    return e;
  }
  cudaError_t e = cudaEventRecord(d.ev_fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d.side, d.ev_fork, 0);
  if (e == cudaSuccess) e = launch_fold_pool<D, G, 8, ZP, MX>(d, io, has_token, d.side);
  if (e == cudaSuccess) e = cudaEventRecord(d.ev_join, d.side);
  if (e == cudaSuccess) e = launch_fold_pool<D, G, 4, ZP, MX>(d, io, has_token, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, d.ev_join, 0);
  return e;
}

template <int ZP, int MX>
cudaError_t launch_fold_zm(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  if (d.D == 128)
    return d.G == 64 ? launch_fold_pools<128, 64, ZP, MX>(d, io, has_token, s)
                     : launch_fold_pools<128, 32, ZP, MX>(d, io, has_token, s);
  return d.G == 64 ? launch_fold_pools<64, 64, ZP, MX>(d, io, has_token, s)
                   : launch_fold_pools<64, 32, ZP, MX>(d, io, has_token, s);
}
extern template cudaError_t launch_fold_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
extern template cudaError_t launch_fold_zm<0, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t);
extern template cudaError_t launch_fold_zm<1, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
extern template cudaError_t launch_fold_zm<1, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t);

}  // namespace pace
