// PACE decode step with fused flush, quantized state ([P1] 어떻게 동작하나: round once every dP tokens, the
// buffered tokens applied together at the flush; [P2] 1. Key Terms & Definitions: the gated delta rule).
//
// One warp per unit (sequence b, head h); the warp walks the state in blocks of 32 columns. Every dense
// contraction of the step runs on the tensor cores as a warp-level MMA (fp32 accumulation), with operands
// built in registers straight from the packed codes:
//   dots   D_g[v][j] = sum_{i in group g} A[v][i] B[i][j]        M = vectors v, N = columns j, K = keys
//          fp16 operands. The vectors are the int8 key codes of the buffered tokens and three int8 digits
//          of a 24-bit fixed-point image of q, kept as swizzled fp16 rows read with ldmatrix. The packed
//          words are stored in fragment order (pace.h): a lane's word w gives its B fragment of a 16-key
//          step as (w & 0x000F000F) | 0x64006400 (the pair 1024 + u) for the first 8 keys and
//          (w & 0x00F000F0) | 0x64006400 (1024 + 16u) for the last 8, whose A values are pre-scaled by
//          1/16. Every product and partial sum is an exact integer or sixteenth in fp32, so with the group
//          scale s_gj and zero point z_gj:
//            (S_hat^T x)_j = sum_g s_gj (D_g[v][j] - T1_vg - z_gj T2_vg),
//            T1 = 1024 (sum of the first-half A) + 1024 (sum of the second-half A), T2 = sum of x over g;
//   tables the Gram products k_s.k_t, the products k_s.(q digits) and the group sums T1, T2 are MMAs of
//          the same fp16 rows;
//   flush  S_new^T[j][i] = sum_s (rho_s u_s,j) k_s,i + G_m s_gj (u_ij - z_gj)   M = columns, N = keys,
//          K = (token, part): rho_s u_s,j is split into three bf16 parts (fp32-accurate) and the int8 keys
//          are exact in bf16. A lane's accumulator fragment holds exactly the keys of its own packed
//          words: the old state is added in fp32 pairs, each key-axis group is requantized by the lane
//          quad that holds it (two shuffles for the absmax or the min/max) and written back in place.
// Between the two, each lane replays one column in reduced form (fp32):
//   u_t = beta_t (v_t - G_t (S_hat^T k_t) - sum_{s<t} (G_t/G_s)(k_s.k_t) u_s),   G_t = a_1 .. a_t
//   o   = G_m (S_hat^T q) + sum_s (G_m/G_s)(k_s.q) u_s
#pragma once

#include <cuda_fp16.h>

#include "pace_common.cuh"

namespace pace {

constexpr int DM_WARPS = 4;   // units (warps) per block
#ifndef PACE_DM_CTA_PER_UNIT
#define PACE_DM_CTA_PER_UNIT 0  // 1: the CTA-per-unit kernel at every batch size
#endif
#ifndef PACE_DM_WARPS_PER_UNIT
#define PACE_DM_WARPS_PER_UNIT 0   // warps per unit of the warp-level kernel: 1, 2, or 0 = by batch size
#endif
#ifndef PACE_DM_MIN_WARPS
#define PACE_DM_MIN_WARPS 16  // resident warps per SM the int4 kernels are compiled for (register cap)
#endif
static_assert(PACE_DM_MIN_WARPS % 2 == 0, "the warp-level kernel is compiled for blocks of one and two warps");
constexpr int PB_STRIDE = 40; // floats per row of the per-block dot table (conflict-free fragment stores)
constexpr int UB_STRIDE = 36; // floats per row of the per-block replay table (conflict-free fragment loads)

// RN(1/(1 + i/128)), i < 128: the reciprocals of the 8-bit significands of bf16 scales. Each entry is the
// correctly rounded double quotient rounded to float; no quotient 128/(128+i) lies within 2^-53 of a float
// rounding tie, so the double rounding is exact.
struct RcpTable {
  float v[128];
};
constexpr RcpTable make_rcp_table() {
  RcpTable t{};
  for (int i = 0; i < 128; ++i) t.v[i] = (float)(128.0 / (128 + i));
  return t;
}
static __device__ const RcpTable g_rcp = make_rcp_table();

__host__ __device__ inline int dm_dpp(int dP) { return 8 * ((dP + 7) / 8); }   // token slots per K part
__host__ __device__ inline int dm_wstride(int dP) { return dP <= 8 ? 8 : dP; }
__host__ __device__ inline int dm_nvt(int dP) { return (dP + 3 + 15) / 16; }   // 16-vector tiles

struct MmaSmem {
  size_t krow, vrow, ah, kbf, pb, ub, W, tk, ck, cf, a, vsc, gam, dmq, bet, svt, ssc, szp, total;
};
// Per-warp work area.
__host__ __device__ inline MmaSmem mma_smem(int D, int G, int dP, int mixed, int zp) {
  MmaSmem L;
  size_t off = 0;
  const int nvmax = dP + 3, nrow = 16 * dm_nvt(dP), ws = dm_wstride(dP);
  L.krow = carve(off, (size_t)nvmax * D);                 // int8 key rows, then the three digits of q
  L.vrow = carve(off, (size_t)dP * D * (mixed ? 2 : 1));  // value codes (int8) or bf16 values
  L.ah = carve(off, (size_t)nrow * D * 2);                // fp16 rows of the vectors, 16-byte chunks
                                                          // XOR-swizzled by row (also staging)
  L.kbf = carve(off, (size_t)D * dm_dpp(dP) * 2);          // flush B operand: bf16 k_s,i as [i][s]
  L.pb = carve(off, (size_t)nvmax * PB_STRIDE * 4);       // dots of one 32-column block [v][j]; while the
                                                          // tables are built: G_t/G_s, then k_s.(q digit d)
  L.ub = carve(off, (size_t)dP * UB_STRIDE * 4);          // replayed u of one block [s][j]
  L.W = carve(off, (size_t)ws * dP * 4);                  // (G_t/G_s) s_ks s_kt (k_s.k_t)
  L.tk = carve(off, (size_t)dP * 16);                     // per token: G_t s_kt, beta_t, s_vt, readout coef
  L.ck = carve(off, (size_t)dP * 4);                      // flush coefficient (G_m/G_s) s_ks
  L.cf = carve(off, (size_t)nrow * 4 * 8);                // (T1, T2) per vector and group
  L.a = carve(off, (size_t)dP * 4);
  L.vsc = carve(off, (size_t)nvmax * 4);
  L.gam = carve(off, (size_t)dP * 4);
  L.dmq = carve(off, (size_t)dP * 4);
  L.bet = carve(off, (size_t)dP * 4);                     // beta_t and the value scale s_vt (cooperative
  L.svt = carve(off, (size_t)dP * 4);                     // staging hands them over in shared memory)
  L.ssc = carve(off, (size_t)(D / G) * D * 2);            // the unit's group scales (bf16), as resident
  L.szp = carve(off, zp ? (size_t)(D / G) * D : 0);       // and zero points
  L.total = carve(off, 0, 16);
  return L;
}

struct MmaShared {
  int8_t *krow;
  unsigned char *vrow;
  __half *ah;
  uint32_t *kbf;
  float *pb, *ub, *W, *dmt;
  float4 *tk;
  float *ck;
  float2 *cf;
  float *e3, *a, *vsc, *gam, *dmq, *bet, *svt;
  __nv_bfloat16 *ssc;
  uint8_t *szp;
};
__device__ inline MmaShared mma_shared(unsigned char *base, const MmaSmem &L, int dP) {
  MmaShared s;
  s.krow = reinterpret_cast<int8_t *>(base + L.krow);
  s.vrow = base + L.vrow;
  s.ah = reinterpret_cast<__half *>(base + L.ah);
  s.kbf = reinterpret_cast<uint32_t *>(base + L.kbf);
  s.pb = reinterpret_cast<float *>(base + L.pb);
  s.ub = reinterpret_cast<float *>(base + L.ub);
  s.W = reinterpret_cast<float *>(base + L.W);
  s.dmt = s.pb;                                           // G_t/G_s, while the tables are built
  s.e3 = s.pb + dm_wstride(dP) * dP;                      // k_s . (q digit d), likewise
  s.tk = reinterpret_cast<float4 *>(base + L.tk);
  s.ck = reinterpret_cast<float *>(base + L.ck);
  s.cf = reinterpret_cast<float2 *>(base + L.cf);
  s.a = reinterpret_cast<float *>(base + L.a);
  s.vsc = reinterpret_cast<float *>(base + L.vsc);
  s.gam = reinterpret_cast<float *>(base + L.gam);
  s.dmq = reinterpret_cast<float *>(base + L.dmq);
  s.bet = reinterpret_cast<float *>(base + L.bet);
  s.svt = reinterpret_cast<float *>(base + L.svt);
  s.ssc = reinterpret_cast<__nv_bfloat16 *>(base + L.ssc);
  s.szp = base + L.szp;
  return s;
}

// ---- warp-level MMAs (fp32 accumulators) ----------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D = A x B + C
__device__ __forceinline__ void mma_f16_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float c0,
                                          float c1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%11,%11};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
// D = A x B (zero accumulator)
__device__ __forceinline__ void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma8_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}
// Fragments of 8x8 b16 tiles from shared memory (row addresses from lanes 0-7, 8-15, 16-23, 24-31).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"((uint32_t)__cvta_generic_to_shared(p))
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"((uint32_t)__cvta_generic_to_shared(p))
               : "memory");
}

// Element offset of 16-byte chunk c of fp16 row r (D halves per row): chunks are XOR-swizzled by r mod 8
// so that the 8 row addresses of one ldmatrix tile fall in distinct banks.
template <int D>
__device__ __forceinline__ int ah_off(int r, int c) { return r * D + ((c ^ (r & 7)) << 3); }

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// fp16 pair of two signed int8 codes (bytes selected from x by `sel`), times 1 or 1/16; exact.
// (code + 128) | 0x6400 is the fp16 number 1152 + code.
__device__ __forceinline__ uint32_t i8pair_f16(uint32_t x, uint32_t sel, bool sixteenth) {
  const uint32_t h = (__byte_perm(x, 0u, sel) ^ 0x00800080u) | 0x64006400u;
  const __half2 v = *reinterpret_cast<const __half2 *>(&h);
  const __half2 r = sixteenth ? __hfma2(v, __float2half2_rn(0.0625f), __float2half2_rn(-72.0f))
                              : __hsub2(v, __float2half2_rn(1152.0f));
  return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t f16x2_scale(uint32_t p, float f) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&p), __float2half2_rn(f));
  return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// bf16(fl(num / den)) for num >= 0: a product with rc = fl(1/den) is within two ulps of the quotient, so it
// rounds to the same bf16 unless it lies within three ulps of a bf16 rounding tie; then the exact quotient.
__device__ __forceinline__ float bf16_quot(float num, float den, float rc) {
  float q = __fmul_rn(num, rc);
  if ((__float_as_uint(q) & 0xFFFFu) - 0x7FFDu <= 6u) q = __fdiv_rn(num, den);
  return bf16_round(q);
}
// RN(1/s) for a positive normal s with an 8-bit significand: the table entry of the significand, with the
// power of two applied exactly to the exponent (far out of range: the division itself).
__device__ __forceinline__ float rcp_bf16(float s) {
  const uint32_t b = __float_as_uint(s), e = b >> 23;
  if (e > 252u) return __fdiv_rn(1.0f, s);
  return __uint_as_float(__float_as_uint(__ldg(&g_rcp.v[(b >> 16) & 0x7Fu])) + ((127u - e) << 23));
}

// Key head of unit u = b*H + h: value head h reads key head h / gamma (q, k and the buffered key codes); the first
// value head of each key head writes the shared buffer row (all of them compute the same codes).
__device__ __forceinline__ int key_unit(const PaceDev &st, int unit) {
  if (st.gamma == 1) return unit;
  const int b = unit / st.H;
  return b * st.Hk + (unit - b * st.H) / st.gamma;
}
__device__ __forceinline__ bool key_writer(const PaceDev &st, int unit) {
  return st.gamma == 1 || (unit % st.H) % st.gamma == 0;
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Global loads issued exactly where they stand in the program (volatile: the compiler neither sinks them past
// a branch to their first use nor merges them), so that a unit's loads leave in the order the step needs them.
__device__ __forceinline__ uint32_t ldg_u32(const void *p) {
  uint32_t r;
  asm volatile("ld.global.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ldg_v2(const void *p) {
  uint2 r;
  asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ldg_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// CPL consecutive elements (CPL = 2 or 4; the I/O pointers are 16-byte aligned) in one vector load.
template <int CPL>
__device__ __forceinline__ void dm_load_io(const void *p, size_t idx, int io, float (&x)[CPL]) {
  static_assert(CPL == 2 || CPL == 4, "two or four elements per lane");
  if (io == PACE_IO_F32) {
    const float *f = static_cast<const float *>(p) + idx;
    if constexpr (CPL == 4) {
      const uint4 v = ldg_v4(f);
      x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y); x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    } else {
      const uint2 v = ldg_v2(f);
      x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    }
  } else {
    const __nv_bfloat16 *h = static_cast<const __nv_bfloat16 *>(p) + idx;
    uint32_t w[CPL / 2];
    if constexpr (CPL == 4) {
      const uint2 v = ldg_v2(h);
      w[0] = v.x; w[1] = v.y;
    } else {
      w[0] = ldg_u32(h);
    }
#pragma unroll
    for (int e = 0; e < CPL / 2; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
}

template <int CPL>
__device__ __forceinline__ void dm_store_bytes(void *p, const int (&c)[CPL]) {
  if constexpr (CPL == 4)
    *reinterpret_cast<uint32_t *>(p) = __byte_perm(__byte_perm((uint32_t)c[0], (uint32_t)c[1], 0x0040),
                                                   __byte_perm((uint32_t)c[2], (uint32_t)c[3], 0x0040), 0x5410);
  else
    *reinterpret_cast<uint16_t *>(p) = (uint16_t)((c[0] & 0xFF) | ((c[1] & 0xFF) << 8));
}

// The lane's packed words of column block cb: M-tiles 2cb, 2cb+1 (columns cb*32 + 16m + 8hi + lane/4), one
// 16-byte vector per 64 keys and plane.
template <int D, int PL>
__device__ __forceinline__ void dm_load_block(const uint32_t *codes, int cb, int lane, uint32_t (&cw)[PL][2][D / 64][4]) {
  constexpr int NPP = D / 64;
#pragma unroll
  for (int pl = 0; pl < PL; ++pl)
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int pp = 0; pp < NPP; ++pp) {
        const uint4 v = ldg_v4(codes + pl * (D * D / 8) + (((2 * cb + m) * NPP + pp) * 32 + lane) * 4);
        cw[pl][m][pp][0] = v.x;
        cw[pl][m][pp][1] = v.y;
        cw[pl][m][pp][2] = v.z;
        cw[pl][m][pp][3] = v.w;
      }
}

// The new token of the step as loaded (lane l holds elements CPL*l .. CPL*l + CPL-1), with a_t and beta_t.
template <int CPL>
struct TokenIn {
  float kx[CPL], vx[CPL], qx[CPL], an, bn;
  float4 bs;   // buffered token `lane`: a, beta, key scale, value scale (when prefetched)
  int pre;     // buffered rows already in flight (0: the staging issues the count's rows itself)
};

// Asynchronous copies of buffered rows 0 .. n-1 of a unit into shared memory: int8 keys straight into their
// rows, packed int4 keys of the mixed buffer into a scratch area (the fp16 row area, built later).
template <int D, int MX>
__device__ __forceinline__ void dm_issue_rows(const PaceDev &st, int unit, int n, const MmaShared &sh) {
  constexpr int mixed = MX;
  const int lane = threadIdx.x & 31, dP = st.dP;
  const int rk = mixed ? D / 2 : D, rv = mixed ? 2 * D : D;
  unsigned char *kdst = mixed ? reinterpret_cast<unsigned char *>(sh.ah) : reinterpret_cast<unsigned char *>(sh.krow);
  const char *gk = static_cast<const char *>(st.buf_k) + (size_t)key_unit(st, unit) * dP * rk;
  const char *gv = static_cast<const char *>(st.buf_v) + (size_t)unit * dP * rv;
  for (int c = lane; c < n * rk / 16; c += 32) cp_async16(kdst + 16 * c, gk + 16 * c);
  for (int c = lane; c < n * rv / 16; c += 32) cp_async16(sh.vrow + 16 * c, gv + 16 * c);
}

// The unit's group scales and zero points, as asynchronous copies into shared memory.
template <int D, int G, int ZP>
__device__ __forceinline__ void dm_issue_scales(const PaceDev &st, int unit, const MmaShared &sh) {
  constexpr int NG = D / G;
  const int lane = threadIdx.x & 31;
  const char *gs = reinterpret_cast<const char *>(st.scale + (size_t)unit * NG * D);
  for (int c = lane; c < NG * D * 2 / 16; c += 32) cp_async16(reinterpret_cast<char *>(sh.ssc) + 16 * c, gs + 16 * c);
  if (ZP) {
    const char *gz = reinterpret_cast<const char *>(st.zp + (size_t)unit * NG * D);
    for (int c = lane; c < NG * D / 16; c += 32) cp_async16(sh.szp + 16 * c, gz + 16 * c);
  }
}

// The new token of the step into registers (zeros without one).
template <int D>
__device__ __forceinline__ void dm_load_token(const PaceDev &st, const PaceIO &io, int unit, int has_token,
                                              TokenIn<D / 32> &tin) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < CPL; ++c) tin.kx[c] = tin.vx[c] = tin.qx[c] = 0.0f;
  tin.an = tin.bn = 0.0f;
  if (has_token) {
    const size_t e0 = (size_t)unit * D + CPL * lane, ek = (size_t)key_unit(st, unit) * D + CPL * lane;
    dm_load_io<CPL>(io.k, ek, st.io, tin.kx);
    dm_load_io<CPL>(io.v, e0, st.io, tin.vx);
    dm_load_io<CPL>(io.q, ek, st.io, tin.qx);
    tin.an = __uint_as_float(ldg_u32(io.a + unit));
    tin.bn = __uint_as_float(ldg_u32(io.beta + unit));
  }
  tin.pre = 0;
  tin.bs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// Stage the unit: the buffered tokens (asynchronous copies, all in flight at once: int8 keys straight into
// their rows, packed int4 keys of the mixed buffer into a scratch area first) and the new one (written into
// buffer slot m0). Leaves in shared memory the key rows (then the q digits), the values, a_t, the key
// scales and the digit weights (vsc), G_t and G_m/G_t. Returns beta_t and the value scale of token t = lane.
template <int D, int G, int MX, class AfterToken>
__device__ void dm_stage(const PaceDev &st, int unit, int m0, int has_token, const TokenIn<D / 32> &tin,
                         const MmaShared &sh, float &bt, float &sv_out, AfterToken &&after_token) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int col0 = CPL * lane;
  const int dP = st.dP;
  const int mt = m0 + has_token;
  constexpr int mixed = MX;
  unsigned char *kdst = mixed ? reinterpret_cast<unsigned char *>(sh.ah) : reinterpret_cast<unsigned char *>(sh.krow);
  float sa = 0.0f, sb = 0.0f, ssk = 0.0f, ssv = 0.0f;
  if (lane < m0) {
    const float4 r = tin.pre ? tin.bs : *reinterpret_cast<const float4 *>(st.buf_s + ((size_t)unit * dP + lane) * 4);
    sa = r.x; sb = r.y; ssk = r.z; ssv = r.w;
  }
  const float *kx = tin.kx, *vx = tin.vx, *qx = tin.qx;
  const float an = tin.an, bn = tin.bn;
  if (has_token) {
    float mk = 0.0f, mv = 0.0f, mq = 0.0f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      mk = fmaxf(mk, fabsf(kx[c]));
      mv = fmaxf(mv, fabsf(vx[c]));
      mq = fmaxf(mq, fabsf(qx[c]));
    }
    const float Ak = warp_max(mk), Av = warp_max(mv), Aq = warp_max(mq);
    // per-token buffer quantizer: s = A/qmax, code = clamp(rint(x * fl(qmax/A))), zero codes for A = 0
    const int qk = mixed ? 7 : 127;
    const bool kz = !(Ak >= FLT_MIN);
    const float rkk = kz ? 0.0f : __fdiv_rn((float)qk, Ak);
    const float sk = kz ? 0.0f : __fdiv_rn(Ak, (float)qk);
    int ck[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) ck[c] = min(max(__float2int_rn(__fmul_rn(kx[c], rkk)), -qk), qk);
    dm_store_bytes<CPL>(sh.krow + m0 * D + col0, ck);
    float sv = 0.0f;
    const size_t ku = key_unit(st, unit);
    const bool kw = key_writer(st, unit);
    if (mixed) {
      uint8_t *bk = static_cast<uint8_t *>(st.buf_k) + (ku * dP + m0) * (D / 2) + col0 / 2;
      if (kw) {
#pragma unroll
        for (int c = 0; c < CPL; c += 2) bk[c / 2] = (uint8_t)((ck[c] + 8) | ((ck[c + 1] + 8) << 4));
      }
      __nv_bfloat16 *bv = static_cast<__nv_bfloat16 *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0;
      uint32_t *vr = reinterpret_cast<uint32_t *>(sh.vrow + ((size_t)m0 * D + col0) * 2);
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        const __nv_bfloat162 pv = __floats2bfloat162_rn(vx[c], vx[c + 1]);
        *reinterpret_cast<__nv_bfloat162 *>(bv + c) = pv;
        vr[c / 2] = *reinterpret_cast<const uint32_t *>(&pv);
      }
    } else {
      const bool vz = !(Av >= FLT_MIN);
      const float rvv = vz ? 0.0f : __fdiv_rn(127.0f, Av);
      sv = vz ? 0.0f : __fdiv_rn(Av, 127.0f);
      int cv[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) cv[c] = min(max(__float2int_rn(__fmul_rn(vx[c], rvv)), -127), 127);
      if (kw) dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_k) + (ku * dP + m0) * D + col0, ck);
      dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0, cv);
      dm_store_bytes<CPL>(sh.vrow + m0 * D + col0, cv);
    }
    if (lane == m0) {
      sa = an; sb = bn; ssk = sk; ssv = sv;
    }
    if (lane == 0)
      *reinterpret_cast<float4 *>(st.buf_s + ((size_t)unit * dP + m0) * 4) = make_float4(an, bn, sk, sv);
    // q ~= sigma (65536 d2 + 256 d1 + d0), |qi| <= 127 * 65536, balanced base-256 digits in [-128, 127]
    const float QMAX = 8323072.0f;
    const bool qz = !(Aq >= FLT_MIN);
    const float sigma = qz ? 0.0f : __fdiv_rn(Aq, QMAX);
    const float rq = qz ? 0.0f : __fdiv_rn(QMAX, Aq);
    int d2[CPL], d1[CPL], d0[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int qi = min(max(__float2int_rn(qx[c] * rq), -8323072), 8323072);
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
  after_token();
  // the buffered rows have landed (the new token's rows above are other slots)
  cp_async_wait_all();
  __syncwarp();
  if (mixed) {
    for (int t = 0; t < m0; ++t) {
      if (lane < D / 8) {                       // one 8-key run per lane: nibble code + 8 -> int8
        const uint32_t nb = *reinterpret_cast<const uint32_t *>(kdst + t * (D / 2) + 4 * lane);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          lo |= (uint32_t)(((int)((nb >> (8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
          hi |= (uint32_t)(((int)((nb >> (16 + 8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
        }
        *reinterpret_cast<uint2 *>(sh.krow + t * D + 8 * lane) = make_uint2(lo, hi);
      }
    }
  }
  if (lane < mt) {
    sh.a[lane] = sa;
    sh.vsc[lane] = ssk;
  }
  bt = sb;
  sv_out = ssv;
  const int ws = dm_wstride(dP);
  if (dP <= 8) {                                // a_t of every token in registers: fixed-length products
    float ar[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) ar[r] = __shfl_sync(0xffffffffu, sa, r);
    if (lane < mt) {
      float g = 1.0f, dm = 1.0f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r <= lane) g *= ar[r];
        if (r > lane && r < mt) dm *= ar[r];
      }
      sh.gam[lane] = g;
      sh.dmq[lane] = dm;
      float p = 1.0f;                           // G_t/G_s = a_{s+1} .. a_t for t = lane, s < t
#pragma unroll
      for (int s = 6; s >= 0; --s) {
        if (s < lane) {
          p *= ar[s + 1];
          sh.dmt[lane * ws + s] = p;
        }
      }
    }
    __syncwarp();
  } else {
    __syncwarp();
    if (lane < mt) {
      float g = 1.0f, dm = 1.0f;
      for (int r = 0; r <= lane; ++r) g *= sh.a[r];
      for (int r = lane + 1; r < mt; ++r) dm *= sh.a[r];
      sh.gam[lane] = g;
      sh.dmq[lane] = dm;
      float p = 1.0f;
      for (int s = lane - 1; s >= 0; --s) {
        p *= sh.a[s + 1];
        sh.dmt[lane * ws + s] = p;
      }
    }
  }
}

// Unit tables: the fp16 rows of the staged vectors (rows >= nv zero; keys 8..15 of every 16-key step
// scaled by 1/16); then, by MMAs of those rows, the group sums (T1, T2), the Gram coefficients W and the
// digit products k_s.q; the per-token replay table; for a flush the bf16 key table kbf[i][s].
template <int D, int G>
__device__ void dm_tables(const MmaShared &sh, int nv, int mt, int dP, int dpp, int has_token, int do_flush,
                          float bt, float sv) {
  constexpr int KS = D / 16, KSG = G / 16, NG = D / G;
  const int lane = threadIdx.x & 31, g8 = lane >> 2, tq = lane & 3;
  const int nvt = (nv + 15) >> 4;
  const int ws = dm_wstride(dP);
  auto row_f16 = [&](int idx, uint2 x) {                 // 8 keys per item
    const int row = idx / (D / 8), k8 = 8 * (idx - row * (D / 8));
    const bool sx = (k8 & 8) != 0;
    const uint4 h = row < nv ? make_uint4(i8pair_f16(x.x, 0x4140, sx), i8pair_f16(x.x, 0x4342, sx),
                                          i8pair_f16(x.y, 0x4140, sx), i8pair_f16(x.y, 0x4342, sx))
                             : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(sh.ah + ah_off<D>(row, k8 >> 3)) = h;
  };
  {                                                      // the first 16 rows: all loads, then all stores
    constexpr int NIT = 16 * (D / 8) / 32;
    uint2 x[NIT];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int idx = lane + 32 * it, row = idx / (D / 8);
      x[it] = row < nv ? *reinterpret_cast<const uint2 *>(sh.krow + row * D + 8 * (idx - row * (D / 8)))
                       : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < NIT; ++it) row_f16(lane + 32 * it, x[it]);
  }
  for (int idx = 16 * (D / 8) + lane; idx < 16 * nvt * (D / 8); idx += 32) {
    const int row = idx / (D / 8);
    row_f16(idx, row < nv ? *reinterpret_cast<const uint2 *>(sh.krow + row * D + 8 * (idx - row * (D / 8)))
                          : make_uint2(0u, 0u));
  }
  __syncwarp();
  const int ntg = (mt + 7) >> 3;                 // 8-token tiles of the Gram columns
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = lane >> 4;   // ldmatrix x4: row, chunk
  const int brow = lane & 7, bcol = (lane >> 3) & 1;                       // ldmatrix x2: row, chunk
  for (int vt = 0; vt < nvt; ++vt) {
    float cs[4], gr[4][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, sh.ah + ah_off<D>(16 * vt + arow, 2 * ks + acol));
      const int gi = ks / KSG;                   // sums: column 2gi (first halves), 2gi + 1 (second halves)
      const uint32_t o0 = g8 == 2 * gi ? 0x3C003C00u : 0u, o1 = g8 == 2 * gi + 1 ? 0x3C003C00u : 0u;
      if (ks == 0) mma_f16_z(cs, a, o0, o1); else mma_f16(cs, a, o0, o1);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        if (n < ntg) {
          uint32_t bb[2];
          ldsm_x2(bb, sh.ah + ah_off<D>(8 * n + brow, 2 * ks + bcol));
          const uint32_t b1 = f16x2_scale(bb[1], 256.0f);
          if (ks == 0) mma_f16_z(gr[n], a, bb[0], b1); else mma_f16(gr[n], a, bb[0], b1);
        }
      }
    }
    const int v0 = 16 * vt + g8;
    if (tq < NG) {
      sh.cf[v0 * 4 + tq] = make_float2(1024.0f * (cs[0] + cs[1]), cs[0] + 16.0f * cs[1]);
      sh.cf[(v0 + 8) * 4 + tq] = make_float2(1024.0f * (cs[2] + cs[3]), cs[2] + 16.0f * cs[3]);
    }
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      if (n >= ntg) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = v0 + 8 * (e >> 1), s = 8 * n + 2 * tq + (e & 1);
        if (s >= mt) continue;
        if (v < mt && s < v)
          sh.W[v * ws + s] = sh.dmt[v * ws + s] * sh.vsc[s] * sh.vsc[v] * gr[n][e];
        else if (v >= mt && v < nv)
          sh.e3[(v - mt) * dP + s] = gr[n][e];
      }
    }
  }
  __syncwarp();
  if (lane < mt) {
    const float dv = sh.dmq[lane] * sh.vsc[lane];
    const float cq = has_token ? dv * (sh.vsc[mt] * sh.e3[lane] + (sh.vsc[mt + 1] * sh.e3[dP + lane] +
                                                                   sh.vsc[mt + 2] * sh.e3[2 * dP + lane]))
                               : 0.0f;
    sh.ck[lane] = dv;
    sh.tk[lane] = make_float4(sh.gam[lane] * sh.vsc[lane], bt, sv, cq);
  }
  if (do_flush) {
    const int half = dpp >> 1;
    if (half == 4) {                             // dP <= 8: lane = (token pair p, key quads), 4-byte row loads
      const int p = lane & 3, s = 2 * p;
      const bool z0 = s >= mt, z1 = s + 1 >= mt;
#pragma unroll
      for (int it = 0; it < D / 32; ++it) {
        const int i0 = 4 * ((lane >> 2) + 8 * it);   // keys i0 .. i0 + 3
        const uint32_t r0 = z0 ? 0u : *reinterpret_cast<const uint32_t *>(sh.krow + s * D + i0);
        const uint32_t r1 = z1 ? 0u : *reinterpret_cast<const uint32_t *>(sh.krow + (s + 1) * D + i0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sh.kbf[(i0 + e) * 4 + p] = bf16x2_bits((float)(int8_t)(r0 >> (8 * e)), (float)(int8_t)(r1 >> (8 * e)));
      }
    } else {
      for (int idx = lane; idx < D * half; idx += 32) {
        const int i = idx / half, s = 2 * (idx - i * half);
        const float k0 = s < mt ? (float)sh.krow[s * D + i] : 0.0f;
        const float k1 = s + 1 < mt ? (float)sh.krow[(s + 1) * D + i] : 0.0f;
        sh.kbf[idx] = bf16x2_bits(k0, k1);
      }
    }
  }
  __syncwarp();
}

// One 32-column block cb of a unit: the dots, the replay and readout of its columns and, at a rounding step,
// their requantization. sh holds the unit's tables; its pb and ub are the calling warp's own. With next_block
// set, the words of block cb + 1 are loaded into cw as soon as this block's dots are done with them (steps
// without rounding).
template <int D, int G, int BITS, int ZP, int MX>
__device__ __forceinline__ void dm_block(const PaceDev &st, const PaceIO &io, int unit, int cb, int m0, int has_token,
                                         uint32_t *codes, __nv_bfloat16 *scale, uint8_t *zpt, const MmaShared &sh,
                                         uint32_t (&cw)[BITS / 4][2][D / 64][4], bool next_block) {
  constexpr int NG = D / G, NPP = D / 64, KSG = G / 16, PL = BITS / 4;
  constexpr int NKG = G / 8;            // key n-tiles (8 keys) per group
  constexpr int NH = BITS == 8 ? 2 : 1, NPN = 4 / NH;   // dot passes, column n-tiles per pass
  constexpr uint32_t PLANE = D * D / 8; // words per nibble plane
  constexpr int OFF = 1 << (BITS - 1);  // symmetric code offset
  const int lane = threadIdx.x & 31, g8 = lane >> 2, tq = lane & 3;
  const int dP = st.dP;
  constexpr int zpm = ZP;
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 3 : 0);
  const int nvt = (nv + 15) >> 4;
  const int dpp = dm_dpp(dP);
  constexpr int mixed = MX;
  const float gm = sh.gam[mt - 1];
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = lane >> 4;

  // ---- dots: P[v][j] for the 32 columns of the block; n-tile n = columns cb*32 + 8n .. +7
#pragma unroll 1
  for (int vt = 0; vt < nvt; ++vt) {
    const int v0 = 16 * vt + g8;
    const int ar = 16 * vt + arow;
    if constexpr (BITS == 4) {
      // int4: each group's accumulator starts at -(T1 + z T2) (symmetric: z = 8 for every column, so the whole
      // offset goes in; zero point: -T1, and -z_gj T2 per column after the MMAs). All partial sums are exact
      // integers below 2^24, so the fold is one rounding per group: P += s_gj * (D_g - T1 - z_gj T2).
      float2 pacc2[4][2];
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        const float2 c0 = sh.cf[v0 * 4 + gi], c1 = sh.cf[(v0 + 8) * 4 + gi];
        const float i0 = ZP ? -c0.x : -fmaf((float)OFF, c0.y, c0.x);
        const float i1 = ZP ? -c1.x : -fmaf((float)OFF, c1.y, c1.x);
        float dacc[4][4];
#pragma unroll
        for (int kk = 0; kk < KSG; ++kk) {
          const int ks = gi * KSG + kk;
          uint32_t a[4];
          ldsm_x4(a, sh.ah + ah_off<D>(ar, 2 * ks + acol));
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w = cw[0][q >> 1][ks >> 2][(q & 1) * 2 + ((ks >> 1) & 1)];
            if (ks & 1) w >>= 8;
            const uint32_t b0 = (w & 0x000F000Fu) | 0x64006400u, b1 = (w & 0x00F000F0u) | 0x64006400u;
            if (kk == 0) mma_f16_c(dacc[q], a, b0, b1, i0, i1); else mma_f16(dacc[q], a, b0, b1);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = cb * 32 + 8 * q + 2 * tq;
          const uint32_t sp = *reinterpret_cast<const uint32_t *>(sh.ssc + gi * D + j);
          const float2 s2 = make_float2(bf16_lo(sp), bf16_hi(sp));
          float2 t0 = make_float2(dacc[q][0], dacc[q][1]), t1 = make_float2(dacc[q][2], dacc[q][3]);
          if (ZP) {
            const uint32_t zw = *reinterpret_cast<const uint16_t *>(sh.szp + gi * D + j);
            const float2 z2 = make_float2((float)(zw & 0xFFu), (float)(zw >> 8));
            t0 = __ffma2_rn(z2, make_float2(-c0.y, -c0.y), t0);
            t1 = __ffma2_rn(z2, make_float2(-c1.y, -c1.y), t1);
          }
          if (gi == 0) {
            pacc2[q][0] = __fmul2_rn(s2, t0);
            pacc2[q][1] = __fmul2_rn(s2, t1);
          } else {
            pacc2[q][0] = __ffma2_rn(s2, t0, pacc2[q][0]);
            pacc2[q][1] = __ffma2_rn(s2, t1, pacc2[q][1]);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        if (v0 < nv) *reinterpret_cast<float2 *>(sh.pb + v0 * PB_STRIDE + 8 * n + 2 * tq) = pacc2[n][0];
        if (v0 + 8 < nv) *reinterpret_cast<float2 *>(sh.pb + (v0 + 8) * PB_STRIDE + 8 * n + 2 * tq) = pacc2[n][1];
      }
    } else {
    float pacc[4][4];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)          // int8 heads: two passes of two n-tiles (register budget)
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        uint32_t sc[NPN], zz[NPN];
#pragma unroll
        for (int q = 0; q < NPN; ++q) {
          const int j = cb * 32 + 8 * (nh * NPN + q) + 2 * tq;
          sc[q] = *reinterpret_cast<const uint32_t *>(sh.ssc + gi * D + j);
          zz[q] = zpm ? (uint32_t)*reinterpret_cast<const uint16_t *>(sh.szp + gi * D + j) : 0u;
        }
        float dacc[PL][NPN][4];
#pragma unroll
        for (int kk = 0; kk < KSG; ++kk) {
          const int ks = gi * KSG + kk;
          uint32_t a[4];
          ldsm_x4(a, sh.ah + ah_off<D>(ar, 2 * ks + acol));
#pragma unroll
          for (int q = 0; q < NPN; ++q)
#pragma unroll
            for (int pl = 0; pl < PL; ++pl) {
              const int n = nh * NPN + q;
              uint32_t w = cw[pl][n >> 1][ks >> 2][(n & 1) * 2 + ((ks >> 1) & 1)];
              if (ks & 1) w >>= 8;
              const uint32_t b0 = (w & 0x000F000Fu) | 0x64006400u, b1 = (w & 0x00F000F0u) | 0x64006400u;
              if (kk == 0) mma_f16_z(dacc[pl][q], a, b0, b1); else mma_f16(dacc[pl][q], a, b0, b1);
            }
        }
        // fold the group: P += s_gj (D - T1 - z_gj T2)
        const float2 c0 = sh.cf[v0 * 4 + gi], c1 = sh.cf[(v0 + 8) * 4 + gi];
        const float k0 = fmaf((float)OFF, c0.y, c0.x), k1 = fmaf((float)OFF, c1.y, c1.x);
#pragma unroll
        for (int q = 0; q < NPN; ++q) {
          const int n = nh * NPN + q;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float s = (e & 1) ? bf16_hi(sc[q]) : bf16_lo(sc[q]);
            const float2 c = (e >> 1) ? c1 : c0;
            float tot;
            if (BITS == 4) {
              if (!zpm)
                tot = dacc[0][q][e] - ((e >> 1) ? k1 : k0);
              else
                tot = dacc[0][q][e] - fmaf((float)((zz[q] >> (8 * (e & 1))) & 0xFFu), c.y, c.x);
            } else {
              const int zj = zpm ? (int)((zz[q] >> (8 * (e & 1))) & 0xFFu) : OFF;
              tot = (float)(__float2int_rn(dacc[0][q][e]) + 16 * __float2int_rn(dacc[PL - 1][q][e]) -
                            17 * __float2int_rn(c.x) - zj * __float2int_rn(c.y));
            }
            pacc[n][e] = gi == 0 ? s * tot : fmaf(s, tot, pacc[n][e]);
          }
        }
      }
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      if (v0 < nv) *reinterpret_cast<float2 *>(sh.pb + v0 * PB_STRIDE + 8 * n + 2 * tq) = make_float2(pacc[n][0], pacc[n][1]);
      if (v0 + 8 < nv)
        *reinterpret_cast<float2 *>(sh.pb + (v0 + 8) * PB_STRIDE + 8 * n + 2 * tq) = make_float2(pacc[n][2], pacc[n][3]);
    }
    }
  }
  // without a flush the block's words are done with: the next block's load overlaps the replay
  if (next_block && !do_flush && cb + 1 < D / 32) dm_load_block<D, PL>(codes, cb + 1, lane, cw);
  __syncwarp();

  // ---- replay and readout: lane = column cb*32 + lane
  {
    const int j = cb * 32 + lane;
    auto value = [&](int t, float svt) -> float {
      if (mixed) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(sh.vrow)[t * D + j]);
      return svt * (float)reinterpret_cast<const int8_t *>(sh.vrow)[t * D + j];
    };
    float o = 0.0f;
    if (has_token)
      o = gm * (sh.vsc[mt] * sh.pb[mt * PB_STRIDE + lane] +
                (sh.vsc[mt + 1] * sh.pb[(mt + 1) * PB_STRIDE + lane] + sh.vsc[mt + 2] * sh.pb[(mt + 2) * PB_STRIDE + lane]));
    if (dP <= 8) {                           // u in registers
      // the per-token operands of every token first (slot min(t, mt - 1) for the unused ones), so that the
      // chain below waits for shared memory once rather than once per token
      float pv[8], vv[8], bt[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int tt = min(t, mt - 1);
        const float4 tk = sh.tk[tt];           // G_t s_kt, beta_t, s_vt, readout coefficient
        vv[t] = fmaf(-tk.x, sh.pb[tt * PB_STRIDE + lane], value(tt, tk.z));
        bt[t] = tk.y;
        pv[t] = tk.w;
      }
      float u[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        u[t] = 0.0f;
        if (t < mt) {
          float acc = vv[t];
#pragma unroll
          for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-sh.W[t * 8 + s2], u[s2], acc);
          u[t] = bt[t] * acc;
          o = fmaf(pv[t], u[t], o);
          if (do_flush) sh.ub[t * UB_STRIDE + lane] = u[t];
        }
      }
    } else {
      for (int t = 0; t < mt; ++t) {
        const float4 tk = sh.tk[t];
        float acc = fmaf(-tk.x, sh.pb[t * PB_STRIDE + lane], value(t, tk.z));
        for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-sh.W[t * dP + s2], sh.ub[s2 * UB_STRIDE + lane], acc);
        const float ut = tk.y * acc;
        sh.ub[t * UB_STRIDE + lane] = ut;
        o = fmaf(tk.w, ut, o);
      }
    }
    if (has_token) store_io(io.o, (long)unit * D + j, o, st.io);
  }
  __syncwarp();
  if (!do_flush) return;

  // ---- flush: rebuild and requantize the block's columns, M-tile by M-tile, group by group
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int jl = 16 * m + g8;              // local columns jl (hi = 0) and jl + 8 (hi = 1)
    // A: the three bf16 parts of rho_s u_s,j for tokens s = 8sb + 2tq, +1 and columns jl, jl + 8
    auto parts = [&](int sb, uint32_t (&ap)[3][2]) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int s0 = 8 * sb + 2 * tq;
        const float x0 = s0 < mt ? sh.ck[s0] * sh.ub[s0 * UB_STRIDE + jl + 8 * hi] : 0.0f;
        const float x1 = s0 + 1 < mt ? sh.ck[s0 + 1] * sh.ub[(s0 + 1) * UB_STRIDE + jl + 8 * hi] : 0.0f;
        const uint32_t p0 = bf16x2_bits(x0, x1);
        const float r0 = x0 - bf16_lo(p0), r1 = x1 - bf16_hi(p0);
        const uint32_t p1 = bf16x2_bits(r0, r1);
        ap[0][hi] = p0;
        ap[1][hi] = p1;
        ap[2][hi] = bf16x2_bits(r0 - bf16_lo(p1), r1 - bf16_hi(p1));
      }
    };
    uint32_t ap0[3][2];                      // tokens 0..7: shared by the groups of the M-tile
    parts(0, ap0);
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float fs[2], fz[2];
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int j = cb * 32 + jl + 8 * hi;
        fs[hi] = gm * __bfloat162float(sh.ssc[gi * D + j]);
        fz[hi] = -(8388608.0f + (float)(zpm ? (int)sh.szp[gi * D + j] : OFF));
      }
      float c[NKG][4];
      {
        const uint32_t(&ap)[3][2] = ap0;
        const uint32_t a16[4] = {ap[0][0], ap[0][1], ap[1][0], ap[1][1]};
#pragma unroll
        for (int nn = 0; nn < NKG; ++nn) {
          const uint32_t bk = sh.kbf[(8 * (gi * NKG + nn) + g8) * (dpp >> 1) + tq];
          mma_bf16_z(c[nn], a16, bk, bk);
          mma8_bf16(c[nn], ap[2][0], ap[2][1], bk);
        }
      }
#pragma unroll 1
      for (int sb = 1; sb < (dpp >> 3); ++sb) {
        uint32_t ap[3][2];
        parts(sb, ap);
        const uint32_t a16[4] = {ap[0][0], ap[0][1], ap[1][0], ap[1][1]};
#pragma unroll
        for (int nn = 0; nn < NKG; ++nn) {
          const uint32_t bk = sh.kbf[(8 * (gi * NKG + nn) + g8) * (dpp >> 1) + 4 * sb + tq];
          mma_bf16(c[nn], a16, bk, bk);
          mma8_bf16(c[nn], ap[2][0], ap[2][1], bk);
        }
      }
      // the old state: x = G_m s_gj (u_ij - z_gj) + replay term, fp32 pairs (u - z exact)
#pragma unroll
      for (int nn = 0; nn < NKG; ++nn) {
        const int nk = gi * NKG + nn, r = nk & 3;
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int wi = hi * 2 + ((nk >> 2) & 1);
          uint32_t m16 = (cw[0][m][nk >> 3][wi] >> (4 * r)) & 0x000F000Fu;
          if (BITS == 8) m16 |= ((cw[PL - 1][m][nk >> 3][wi] >> (4 * r)) & 0x000F000Fu) << 4;
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
        float s;
        int z;
        if (!zpm) {
          float A = 0.0f;
#pragma unroll
          for (int nn = 0; nn < NKG; ++nn) A = fmax3(A, fabsf(c[nn][2 * hi]), fabsf(c[nn][2 * hi + 1]));
          A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 1));
          A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, 2));
          constexpr float QMAX = (float)(OFF - 1);
          s = bf16_quot(A, QMAX, 1.0f / QMAX);
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
          s = bf16_quot(__fsub_rn(hi_, lo), QM, 1.0f / QM);
          z = 0;
          if (s >= FLT_MIN) z = min(max(__float2int_rn(__fmul_rn(-lo, rcp_bf16(s))), 0), (1 << BITS) - 1);
        }
        if (!(s >= FLT_MIN)) s = 0.0f;
        const float r = s > 0.0f ? rcp_bf16(s) : 0.0f;
        // codes: rint(x r) by the 1.5 * 2^23 rounding constant (symmetric: the clamp to +-qmax never binds,
        // since s = bf16(A / qmax) puts |x r| below qmax + 1/2); zero point: + z, clamp to [0, 2^b - 1]
        const float2 r2 = make_float2(r, r);
        const float mg = zpm ? 12582912.0f : 12582912.0f + (float)OFF;
        const float2 mg2 = make_float2(mg, mg);
#pragma unroll
        for (int pw = 0; pw < G / 32; ++pw) {
          const int p = gi * (G / 32) + pw;  // 32-key span
          uint32_t w0 = 0, w1 = 0;
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int nn = 4 * pw + rr;
            const float2 y = __fadd2_rn(__fmul2_rn(make_float2(c[nn][2 * hi], c[nn][2 * hi + 1]), r2), mg2);
            uint32_t pair;
            if (!zpm) {
              pair = __byte_perm(__float_as_uint(y.x), __float_as_uint(y.y), 0x5410);   // bytes 1, 3 are 0
              if (BITS == 4) {                 // each half is code + 8 in 1..15: no other bit is set
                w0 = rr == 0 ? pair : w0 + (pair << (4 * rr));
                continue;
              }
            } else {
              const int c0 = min(max((int)(__float_as_uint(y.x) - 0x4B400000u) + z, 0), (1 << BITS) - 1);
              const int c1 = min(max((int)(__float_as_uint(y.y) - 0x4B400000u) + z, 0), (1 << BITS) - 1);
              pair = __byte_perm((uint32_t)c0, (uint32_t)c1, 0x5410);
            }
            w0 += (pair & 0x000F000Fu) << (4 * rr);
            if (BITS == 8) w1 += ((pair >> 4) & 0x000F000Fu) << (4 * rr);
          }
          cw[0][m][p >> 1][hi * 2 + (p & 1)] = w0;
          if (BITS == 8) cw[PL - 1][m][p >> 1][hi * 2 + (p & 1)] = w1;
        }
        if (tq == 0) {
          const int j = cb * 32 + jl + 8 * hi;
          scale[gi * D + j] = __float2bfloat16_rn(s);
          if (zpm) zpt[gi * D + j] = (uint8_t)z;
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

template <int D, int G, int BITS, int ZP, int MX, int WU>
__device__ void dm_unit(const PaceDev &st, const PaceIO &io, int b, int h, int unit, int has_token,
                        const MmaShared &sh, int part) {
  // WU warps per unit: warp `part` runs the column blocks [cb0, cb1)
  const int cb0 = WU == 1 ? 0 : part * (D / 32) / WU, cb1 = WU == 1 ? D / 32 : (part + 1) * (D / 32) / WU;
  constexpr int NG = D / G, NPP = D / 64, PL = BITS / 4;
  constexpr uint32_t PLANE = D * D / 8; // words per nibble plane
  const int lane = threadIdx.x & 31;
  const int dP = st.dP;
  constexpr int zpm = ZP;
  uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                              : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
  __nv_bfloat16 *scale = st.scale + (size_t)unit * NG * D;
  uint8_t *zpt = zpm ? st.zp + (size_t)unit * NG * D : nullptr;

  // The loads go out in the order the step needs them: the buffer count (it gates the buffered rows) and the
  // new token; once the count is known, the buffered rows, then the scales and zero points; the first column
  // block's words once the new token has arrived; the L2 prefetch of the other blocks only after the tables.
  // All units start together, so whatever is requested early delays the loads the staging waits for.
  const int m0 = (int)ldg_u32(st.m + unit);
  TokenIn<D / 32> tin;
  dm_load_token<D>(st, io, unit, has_token, tin);
  if (m0 < 0 || m0 >= dP || (!has_token && m0 == 0)) {
    if (has_token && m0 != 0)                    // corrupted counter: leave the unit, emit zeros
      for (int c = lane; c < D; c += 32) store_io(io.o, (long)unit * D + c, 0.0f, st.io);
    return;                                      // (or a flush with nothing pending)
  }
  if (m0 > 0) {
    dm_issue_rows<D, MX>(st, unit, m0, sh);
    if (lane < m0) tin.bs = *reinterpret_cast<const float4 *>(st.buf_s + ((size_t)unit * dP + lane) * 4);
    tin.pre = m0;
  }
  dm_issue_scales<D, G, ZP>(st, unit, sh);
  uint32_t cw[PL][2][NPP][4];

  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 3 : 0);
  const int dpp = dm_dpp(dP);
  float bt, sv;
  // the first column block's words once the new token is in (they are first needed by the dots)
  dm_stage<D, G, MX>(st, unit, m0, has_token, tin, sh, bt, sv, [&]() { dm_load_block<D, PL>(codes, cb0, lane, cw); });
  dm_tables<D, G>(sh, nv, mt, dP, dpp, has_token, do_flush, bt, sv);
  if (cb1 - cb0 > 1) {                           // the warp's other blocks into L2, ahead of their loads
    constexpr uint32_t BLK = 2 * NPP * 128;      // words of one 32-column block in a plane
    if (lane < PL) prefetch_l2(codes + lane * PLANE + (cb0 + 1) * BLK, (cb1 - cb0 - 1) * BLK * 4);
  }

#pragma unroll 1
  for (int cb = cb0; cb < cb1; ++cb) {
    if (cb > cb0 && do_flush) dm_load_block<D, PL>(codes, cb, lane, cw);
    dm_block<D, G, BITS, ZP, MX>(st, io, unit, cb, m0, has_token, codes, scale, zpt, sh, cw, cb + 1 < cb1);
  }
  // every warp of the unit has read the count before it moves on
  if (WU > 1) __syncthreads(); else __syncwarp();
  if (threadIdx.x == 0) st.m[unit] = do_flush ? 0 : mt;
}

// One launch per code pool (int4 heads, int8 heads), so that each path gets its own register allocation
// (int4: 16 warps per SM at <= 128 registers; int8, with twice the code words live: 12 warps per SM).
// Warp w of the launch handles pool unit w: sequence w / HP, the pool's head slot w % HP.
template <int D, int G, int BITS, int ZP, int MX, int WU>
__global__ void __launch_bounds__(WU * 32, (BITS == 4 ? PACE_DM_MIN_WARPS : 12) / WU) decode_mma_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_enter();
  const int warp = threadIdx.x >> 5;
  const int HP = BITS == 4 ? st.H4 : st.H8;
  const int w = blockIdx.x;                      // one unit per block, W warps per unit
  if (w >= st.B * HP) return;                    // (the whole block)
  const int b = w / HP, slot = w - b * HP;
  const int h = st.pool_head[(BITS == 4 ? 0 : st.H4) + slot];
  const MmaSmem L = mma_smem(D, G, st.dP, MX, ZP);
  const MmaShared sh = mma_shared(smem + (size_t)warp * L.total, L, st.dP);
  dm_unit<D, G, BITS, ZP, MX, WU>(st, io, b, h, b * st.H + h, has_token, sh, warp);
}

// ---- cooperative form: the four warps of a CTA stage one unit together ---------------------------------------
// Named barrier among the CTA's warps (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void dc_bar() { asm volatile("bar.sync 1, %0;" ::"r"(DM_WARPS * 32) : "memory"); }

// Loads that do not depend on the buffer count, split by role: warp 0 the key side (new k and q, every buffered
// key row, the per-token scalars), warp 1 the value side (new v, every buffered value row), warp 3 the per-token
// scalars; the group scales and zero points by all four. Every buffered row is fetched before the count is known
// (at most dP rows), so the count read and the row copies are in flight together. The q digit rows share the
// key-row area with those copies, so the warp that issues the copies also writes the digits, after its wait.
template <int D, int G, int ZP, int MX>
__device__ __forceinline__ void dc_issue(const PaceDev &st, const PaceIO &io, int unit, int has_token, const MmaShared &sh,
                                         int warp, float (&x)[D / 32], float (&xq)[D / 32], float4 &bs, float &an,
                                         float &bn) {
  constexpr int CPL = D / 32, NG = D / G;
  const int lane = threadIdx.x & 31, dP = st.dP, tid = threadIdx.x;
  const char *gs = reinterpret_cast<const char *>(st.scale + (size_t)unit * NG * D);
  for (int c = tid; c < NG * D * 2 / 16; c += DM_WARPS * 32) cp_async16(reinterpret_cast<char *>(sh.ssc) + 16 * c, gs + 16 * c);
  if (ZP) {
    const char *gz = reinterpret_cast<const char *>(st.zp + (size_t)unit * NG * D);
    for (int c = tid; c < NG * D / 16; c += DM_WARPS * 32) cp_async16(sh.szp + 16 * c, gz + 16 * c);
  }
  const int rk = MX ? D / 2 : D, rv = MX ? 2 * D : D;
  if (warp == 0) {
    unsigned char *kdst = MX ? reinterpret_cast<unsigned char *>(sh.ah) : reinterpret_cast<unsigned char *>(sh.krow);
    const char *gk = static_cast<const char *>(st.buf_k) + (size_t)key_unit(st, unit) * dP * rk;
    for (int c = lane; c < dP * rk / 16; c += 32) cp_async16(kdst + 16 * c, gk + 16 * c);
  } else if (warp == 1) {
    const char *gv = static_cast<const char *>(st.buf_v) + (size_t)unit * dP * rv;
    for (int c = lane; c < dP * rv / 16; c += 32) cp_async16(sh.vrow + 16 * c, gv + 16 * c);
  }
#pragma unroll
  for (int c = 0; c < CPL; ++c) x[c] = xq[c] = 0.0f;
  an = bn = 0.0f;
  bs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (has_token) {
    const size_t e0 = (size_t)unit * D + CPL * lane, ek = (size_t)key_unit(st, unit) * D + CPL * lane;
    if (warp < 2) dm_load_io<CPL>(warp == 0 ? io.k : io.v, warp == 0 ? ek : e0, st.io, x);
    if (warp == 0) dm_load_io<CPL>(io.q, ek, st.io, xq);
    an = io.a[unit];
    bn = io.beta[unit];
  }
  if ((warp == 0 || warp == 3) && lane < dP) bs = *reinterpret_cast<const float4 *>(st.buf_s + ((size_t)unit * dP + lane) * 4);
}

// Stage the new token and the tables that need no MMA, by role (see dc_issue). Leaves in shared memory what the
// single-warp staging leaves, plus beta_t (bet) and the value scales s_vt (svt).
template <int D, int G, int MX>
__device__ void dc_stage(const PaceDev &st, int unit, int m0, int has_token, const MmaShared &sh, int warp,
                         const float (&x)[D / 32], const float (&xq)[D / 32], float4 bs, float an, float bn) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31, col0 = CPL * lane, dP = st.dP, mt = m0 + has_token;
  cp_async_wait_all();
  __syncwarp();
  if (warp == 0) {                                      // key side
    if (MX) {
      const unsigned char *kp = reinterpret_cast<const unsigned char *>(sh.ah);
      for (int t = 0; t < m0; ++t) {
        if (lane < D / 8) {                             // one 8-key run per lane: nibble code + 8 -> int8
          const uint32_t nb = *reinterpret_cast<const uint32_t *>(kp + t * (D / 2) + 4 * lane);
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            lo |= (uint32_t)(((int)((nb >> (8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
            hi |= (uint32_t)(((int)((nb >> (16 + 8 * (e >> 1) + 4 * (e & 1))) & 0xF) - 8) & 0xFF) << (8 * e);
          }
          *reinterpret_cast<uint2 *>(sh.krow + t * D + 8 * lane) = make_uint2(lo, hi);
        }
      }
    }
    float sk = 0.0f;
    if (has_token) {
      float mk = 0.0f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) mk = fmaxf(mk, fabsf(x[c]));
      const float Ak = warp_max(mk);
      const int qk = MX ? 7 : 127;
      const bool kz = !(Ak >= FLT_MIN);
      const float rkk = kz ? 0.0f : __fdiv_rn((float)qk, Ak);
      sk = kz ? 0.0f : __fdiv_rn(Ak, (float)qk);
      int ck[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) ck[c] = min(max(__float2int_rn(__fmul_rn(x[c], rkk)), -qk), qk);
      dm_store_bytes<CPL>(sh.krow + m0 * D + col0, ck);
      const size_t ku = key_unit(st, unit);
      if (key_writer(st, unit)) {
        if (MX) {
          uint8_t *bk = static_cast<uint8_t *>(st.buf_k) + (ku * dP + m0) * (D / 2) + col0 / 2;
#pragma unroll
          for (int c = 0; c < CPL; c += 2) bk[c / 2] = (uint8_t)((ck[c] + 8) | ((ck[c + 1] + 8) << 4));
        } else {
          dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_k) + (ku * dP + m0) * D + col0, ck);
        }
      }
      if (lane == 0) {
        float *e = st.buf_s + ((size_t)unit * dP + m0) * 4;
        *reinterpret_cast<float2 *>(e) = make_float2(an, bn);
        e[2] = sk;
      }
    }
    if (lane < mt) sh.vsc[lane] = lane < m0 ? bs.z : sk;
    // q as three balanced base-256 digits
    if (has_token) {
      float mq = 0.0f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) mq = fmaxf(mq, fabsf(xq[c]));
      const float Aq = warp_max(mq);
      const float QMAX = 8323072.0f;
      const bool qz = !(Aq >= FLT_MIN);
      const float sigma = qz ? 0.0f : __fdiv_rn(Aq, QMAX);
      const float rq = qz ? 0.0f : __fdiv_rn(QMAX, Aq);
      int d2[CPL], d1[CPL], d0[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int qi = min(max(__float2int_rn(xq[c] * rq), -8323072), 8323072);
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
  } else if (warp == 1) {                               // value side
    float sv = 0.0f;
    if (has_token) {
      if (MX) {
        __nv_bfloat16 *bv = static_cast<__nv_bfloat16 *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0;
        uint32_t *vr = reinterpret_cast<uint32_t *>(sh.vrow + ((size_t)m0 * D + col0) * 2);
#pragma unroll
        for (int c = 0; c < CPL; c += 2) {
          const __nv_bfloat162 pv = __floats2bfloat162_rn(x[c], x[c + 1]);
          *reinterpret_cast<__nv_bfloat162 *>(bv + c) = pv;
          vr[c / 2] = *reinterpret_cast<const uint32_t *>(&pv);
        }
      } else {
        float mv = 0.0f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) mv = fmaxf(mv, fabsf(x[c]));
        const float Av = warp_max(mv);
        const bool vz = !(Av >= FLT_MIN);
        const float rvv = vz ? 0.0f : __fdiv_rn(127.0f, Av);
        sv = vz ? 0.0f : __fdiv_rn(Av, 127.0f);
        int cv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) cv[c] = min(max(__float2int_rn(__fmul_rn(x[c], rvv)), -127), 127);
        dm_store_bytes<CPL>(static_cast<int8_t *>(st.buf_v) + ((size_t)unit * dP + m0) * D + col0, cv);
        dm_store_bytes<CPL>(sh.vrow + m0 * D + col0, cv);
      }
      if (lane == 0) st.buf_s[((size_t)unit * dP + m0) * 4 + 3] = sv;
    }
    // value scales of the buffered tokens: read back from global (written by the earlier steps)
    if (lane < m0) sh.svt[lane] = st.buf_s[((size_t)unit * dP + lane) * 4 + 3];
    if (lane == m0 && has_token) sh.svt[lane] = sv;
  } else if (warp == 3) {                              // decays: G_t, G_m/G_t and the ratios G_t/G_s
    if (lane < mt) {
      sh.a[lane] = lane < m0 ? bs.x : an;
      sh.bet[lane] = lane < m0 ? bs.y : bn;
    }
    __syncwarp();
    if (lane < mt) {
      const int ws = dm_wstride(dP);
      float g = 1.0f, dm = 1.0f;
      for (int r = 0; r <= lane; ++r) g *= sh.a[r];
      for (int r = lane + 1; r < mt; ++r) dm *= sh.a[r];
      sh.gam[lane] = g;
      sh.dmq[lane] = dm;
      float p = 1.0f;                                   // G_t/G_s = a_{s+1} .. a_t for t = lane, s < t
      for (int s2 = lane - 1; s2 >= 0; --s2) {
        p *= sh.a[s2 + 1];
        sh.dmt[lane * ws + s2] = p;
      }
    }
  }
}

// The fp16 rows of the vectors (rows >= nv zero; keys 8..15 of every 16-key step scaled by 1/16) and, for a
// flush, the bf16 key table kbf[i][s]: split over the CTA's threads.
template <int D>
__device__ void dc_rows(const MmaShared &sh, int nv, int mt, int dpp, int do_flush) {
  const int tid = threadIdx.x;
  const int nvt = (nv + 15) >> 4;
  for (int idx = tid; idx < 16 * nvt * (D / 8); idx += DM_WARPS * 32) {
    const int row = idx / (D / 8), k8 = 8 * (idx - row * (D / 8));
    uint4 h = make_uint4(0u, 0u, 0u, 0u);
    if (row < nv) {
      const uint2 x = *reinterpret_cast<const uint2 *>(sh.krow + row * D + k8);
      const bool sx = (k8 & 8) != 0;
      h = make_uint4(i8pair_f16(x.x, 0x4140, sx), i8pair_f16(x.x, 0x4342, sx), i8pair_f16(x.y, 0x4140, sx),
                     i8pair_f16(x.y, 0x4342, sx));
    }
    *reinterpret_cast<uint4 *>(sh.ah + ah_off<D>(row, k8 >> 3)) = h;
  }
  if (do_flush) {
    const int half = dpp >> 1;
    for (int idx = tid; idx < D * half; idx += DM_WARPS * 32) {
      const int i = idx / half, s2 = 2 * (idx - i * half);
      const float k0 = s2 < mt ? (float)sh.krow[s2 * D + i] : 0.0f;
      const float k1 = s2 + 1 < mt ? (float)sh.krow[(s2 + 1) * D + i] : 0.0f;
      sh.kbf[idx] = bf16x2_bits(k0, k1);
    }
  }
}

// Tables by MMA of the fp16 rows, split over two warps: warp 0 the group sums (T1, T2), warp 1 the Gram
// coefficients W and the digit products k_s.q, then the per-token replay table tk and the flush coefficients ck.
template <int D, int G>
__device__ void dc_tables(const MmaShared &sh, int nv, int mt, int dP, int has_token, int warp) {
  constexpr int KS = D / 16, KSG = G / 16, NG = D / G;
  const int lane = threadIdx.x & 31, g8 = lane >> 2, tq = lane & 3;
  const int nvt = (nv + 15) >> 4;
  const int ws = dm_wstride(dP);
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), acol = lane >> 4;
  const int brow = lane & 7, bcol = (lane >> 3) & 1;
  if (warp == 0) {
    for (int vt = 0; vt < nvt; ++vt) {
      float cs[4];
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, sh.ah + ah_off<D>(16 * vt + arow, 2 * ks + acol));
        const int gi = ks / KSG;                        // sums: column 2gi (first halves), 2gi + 1 (second halves)
        const uint32_t o0 = g8 == 2 * gi ? 0x3C003C00u : 0u, o1 = g8 == 2 * gi + 1 ? 0x3C003C00u : 0u;
        if (ks == 0) mma_f16_z(cs, a, o0, o1); else mma_f16(cs, a, o0, o1);
      }
      const int v0 = 16 * vt + g8;
      if (tq < NG) {
        sh.cf[v0 * 4 + tq] = make_float2(1024.0f * (cs[0] + cs[1]), cs[0] + 16.0f * cs[1]);
        sh.cf[(v0 + 8) * 4 + tq] = make_float2(1024.0f * (cs[2] + cs[3]), cs[2] + 16.0f * cs[3]);
      }
    }
  } else if (warp == 1) {
    const int ntg = (mt + 7) >> 3;                      // 8-token tiles of the Gram columns
    for (int vt = 0; vt < nvt; ++vt) {
      float gr[4][4];
#pragma unroll 2
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, sh.ah + ah_off<D>(16 * vt + arow, 2 * ks + acol));
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          if (n < ntg) {
            uint32_t bb[2];
            ldsm_x2(bb, sh.ah + ah_off<D>(8 * n + brow, 2 * ks + bcol));
            const uint32_t b1 = f16x2_scale(bb[1], 256.0f);
            if (ks == 0) mma_f16_z(gr[n], a, bb[0], b1); else mma_f16(gr[n], a, bb[0], b1);
          }
        }
      }
      const int v0 = 16 * vt + g8;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        if (n >= ntg) continue;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = v0 + 8 * (e >> 1), s2 = 8 * n + 2 * tq + (e & 1);
          if (s2 >= mt) continue;
          if (v < mt && s2 < v)
            sh.W[v * ws + s2] = sh.dmt[v * ws + s2] * sh.vsc[s2] * sh.vsc[v] * gr[n][e];
          else if (v >= mt && v < nv)
            sh.e3[(v - mt) * dP + s2] = gr[n][e];
        }
      }
    }
    __syncwarp();
    if (lane < mt) {
      const float dv = sh.dmq[lane] * sh.vsc[lane];
      const float cq = has_token ? dv * (sh.vsc[mt] * sh.e3[lane] + (sh.vsc[mt + 1] * sh.e3[dP + lane] +
                                                                     sh.vsc[mt + 2] * sh.e3[2 * dP + lane]))
                                 : 0.0f;
      sh.ck[lane] = dv;
      sh.tk[lane] = make_float4(sh.gam[lane] * sh.vsc[lane], sh.bet[lane], sh.svt[lane], cq);
    }
  }
}

// One CTA per unit. The four warps stage the unit and build its tables together (dc_issue, dc_stage, dc_rows,
// dc_tables, three barriers), in the first work area; then warp w runs column block w with its own dot and
// replay tables. The chain of dependent work per warp is about a quarter of the one-warp-per-unit kernel's.
template <int D, int G, int BITS, int ZP, int MX>
__global__ void __launch_bounds__(DM_WARPS * 32, BITS == 4 ? 4 : 3) decode_split_kernel(const PaceDev st, const PaceIO io, const int has_token) {
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_enter();
  constexpr int NG = D / G, NPP = D / 64, PL = BITS / 4, NB = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HP = BITS == 4 ? st.H4 : st.H8;
  const int w = blockIdx.x;
  if (w >= st.B * HP) return;                   // the whole CTA
  const int b = w / HP, slot = w - b * HP;
  const int h = st.pool_head[(BITS == 4 ? 0 : st.H4) + slot];
  const int unit = b * st.H + h;
  const int dP = st.dP;
  constexpr int zpm = ZP;
  const MmaSmem L = mma_smem(D, G, dP, MX, zpm);
  const MmaShared sh0 = mma_shared(smem, L, dP);
  MmaShared shw = sh0;
  {
    const MmaShared own = mma_shared(smem + (size_t)warp * L.total, L, dP);
    shw.pb = own.pb;
    shw.ub = own.ub;
  }
  uint32_t *codes = BITS == 4 ? st.codes4 + (size_t)(b * st.H4 + st.head_slot[h]) * (D * D / 8)
                              : st.codes8 + (size_t)(b * st.H8 + st.head_slot[h]) * (D * D / 4);
  __nv_bfloat16 *scale = st.scale + (size_t)unit * NG * D;
  uint8_t *zpt = zpm ? st.zp + (size_t)unit * NG * D : nullptr;
  const bool active = warp < NB;
  const int m0 = (int)ldg_u32(st.m + unit);      // first: every warp's first wait is on the count
  uint32_t cw[PL][2][NPP][4];
  if (active) dm_load_block<D, PL>(codes, warp, lane, cw);
  float x[D / 32], xq[D / 32], an, bn;
  float4 bs;
  dc_issue<D, G, ZP, MX>(st, io, unit, has_token, sh0, warp, x, xq, bs, an, bn);
  if (m0 < 0 || m0 >= dP || (!has_token && m0 == 0)) {
    cp_async_wait_all();                         // nothing may land in shared memory after the CTA leaves
    if (warp == 0 && has_token && m0 != 0)       // corrupted counter: leave the unit, emit zeros
      for (int c = lane; c < D; c += 32) store_io(io.o, (long)unit * D + c, 0.0f, st.io);
    return;
  }
  const int mt = m0 + has_token;
  const int do_flush = !has_token || mt == dP;
  const int nv = mt + (has_token ? 3 : 0);
  dc_stage<D, G, MX>(st, unit, m0, has_token, sh0, warp, x, xq, bs, an, bn);
  dc_bar();
  dc_rows<D>(sh0, nv, mt, dm_dpp(dP), do_flush);
  dc_bar();
  dc_tables<D, G>(sh0, nv, mt, dP, has_token, warp);
  dc_bar();
  if (active) dm_block<D, G, BITS, ZP, MX>(st, io, unit, warp, m0, has_token, codes, scale, zpt, shw, cw, false);
  __syncthreads();
  if (threadIdx.x == 0) st.m[unit] = do_flush ? 0 : mt;
}

template <int D, int G, int BITS, int ZP, int MX>
static cudaError_t launch_pool(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s, size_t unit_smem) {
  const size_t smem = (size_t)DM_WARPS * unit_smem;   // the larger of the two launch shapes
  cudaError_t e = smem_opt_in<decode_mma_kernel<D, G, BITS, ZP, MX, 1>>(smem);
  if (e == cudaSuccess) e = smem_opt_in<decode_mma_kernel<D, G, BITS, ZP, MX, 2>>(smem);
  if (e == cudaSuccess) e = smem_opt_in<decode_split_kernel<D, G, BITS, ZP, MX>>(smem);
  if (e != cudaSuccess) return e;
  const long units = (long)d.B * (BITS == 4 ? d.H4 : d.H8);
  if (units == 0) return cudaSuccess;
  // one warp per unit while every SM holds 16 units' warps or more; below that, a CTA per unit
  cudaLaunchAttribute attr[1];
  const long slots = (long)device_sm_count() * 16;   // resident warps of the warp-level kernel
  if (PACE_DM_CTA_PER_UNIT || (PACE_DM_WARPS_PER_UNIT == 0 && units * DM_WARPS <= slots)) {
    const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)units), dim3(DM_WARPS * 32), smem, s, attr);
    return cudaLaunchKernelEx(&cfg, decode_split_kernel<D, G, BITS, ZP, MX>, d, io, has_token);
  }
  // One unit per block. Each unit's warps stage it on their own and split its column blocks: while the units
  // fill fewer than half the warp slots, two warps per unit halve the per-unit chain; otherwise one warp, and
  // one-warp blocks spread the units evenly over the SMs (the slowest SM sets the step time).
  const int W = PACE_DM_WARPS_PER_UNIT ? PACE_DM_WARPS_PER_UNIT : (units * 2 <= slots ? 2 : 1);
  const cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)units), dim3(W * 32), (size_t)W * unit_smem, s, attr);
  return W == 2 ? cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, G, BITS, ZP, MX, 2>, d, io, has_token)
                : cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, G, BITS, ZP, MX, 1>, d, io, has_token);
}

template <int D, int G, int ZP, int MX>
static cudaError_t launch_mma_t(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s, bool int4_pool = true) {
  const MmaSmem L = mma_smem(D, G, d.dP, MX, ZP);
  if ((size_t)DM_WARPS * L.total > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = int4_pool ? launch_pool<D, G, 4, ZP, MX>(d, io, has_token, s, L.total) : cudaSuccess;
  if (e == cudaSuccess) e = launch_pool<D, G, 8, ZP, MX>(d, io, has_token, s, L.total);
  return e;
}

// Every (D, G) of one zero-point mode and buffer format; each combination is instantiated in a translation
// unit of its own so that they compile in parallel.
template <int ZP, int MX>
cudaError_t launch_quant_zm(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s, bool int4_pool = true) {
  if (d.D == 128)
    return d.G == 64 ? launch_mma_t<128, 64, ZP, MX>(d, io, has_token, s, int4_pool)
                     : launch_mma_t<128, 32, ZP, MX>(d, io, has_token, s, int4_pool);
  return d.G == 64 ? launch_mma_t<64, 64, ZP, MX>(d, io, has_token, s) : launch_mma_t<64, 32, ZP, MX>(d, io, has_token, s);
}
extern template cudaError_t launch_quant_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
extern template cudaError_t launch_quant_zm<0, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
extern template cudaError_t launch_quant_zm<1, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
extern template cudaError_t launch_quant_zm<1, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);

}  // namespace pace
