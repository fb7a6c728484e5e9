// Per-token bf16-state decode: the comparison point of the pages' throughput study
// ([P1] 전제와 한계: periodic INT4 decoding against per-token bf16 decoding; [P2] 3. Method & Key Results,
// Figure 6). Every token reads the bf16 state, applies S = a S + k u^T with u = beta (v - (a S)^T k) in
// fp32, emits o = S^T q from the fp32 result, and writes the state back rounded to bf16.
//
// One CTA per unit: 4 row blocks x D/2 column pairs; each thread keeps D/4 rows x 2 columns in
// registers, so the state is read once and written once per token (bf16x2, coalesced rows).
#include "pace_common.cuh"

namespace pace {

template <int D>
__global__ void __launch_bounds__(2 * D) decode_bf16_kernel(const PaceDev st, const PaceIO io, const int late_trigger) {
  constexpr int NCP = D / 2;          // column pairs
  constexpr int RB = D / 4;           // rows per row block
  __shared__ float ks[D], qs[D], vs[D], us[D];
  __shared__ float part[4][D];
  // the next launch's blocks: placed as this launch finishes when it has 33 units to one per SM, else from the start
  // (measured on the 16-head layer shape: at 48 and 128 units the early trigger cost 16% and 12% per launch; at 16
  // units the late one 6%; at 256 units the two measured equal, above it the early one is ahead)
  if (!late_trigger) pdl_trigger();
  pdl_wait();
  const long unit = blockIdx.x;
  const int tid = threadIdx.x;
  const int cp = tid % NCP, rb = tid / NCP;
  if (tid < D) {
    ks[tid] = load_io(io.k, unit * D + tid, st.io);
    qs[tid] = load_io(io.q, unit * D + tid, st.io);
    vs[tid] = load_io(io.v, unit * D + tid, st.io);
  }
  const float a = io.a[unit], beta = io.beta[unit];
  __nv_bfloat162 *Sp = reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(st.S) + unit * D * D);
  float2 s[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) s[r] = __bfloat1622float2(Sp[(rb * RB + r) * NCP + cp]);
  __syncthreads();
  // w = (a S)^T k, partial over this row block
  float w0 = 0.0f, w1 = 0.0f;
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    const float kk = ks[rb * RB + r];
    w0 = fmaf(s[r].x, kk, w0);
    w1 = fmaf(s[r].y, kk, w1);
  }
  part[rb][2 * cp] = w0;
  part[rb][2 * cp + 1] = w1;
  __syncthreads();
  if (tid < D) {
    const float w = a * (part[0][tid] + part[1][tid] + part[2][tid] + part[3][tid]);
    us[tid] = beta * (vs[tid] - w);
  }
  __syncthreads();
  const float u0 = us[2 * cp], u1 = us[2 * cp + 1];
  float o0 = 0.0f, o1 = 0.0f;
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    const int i = rb * RB + r;
    const float kk = ks[i], qq = qs[i];
    const float x0 = fmaf(a, s[r].x, kk * u0);
    const float x1 = fmaf(a, s[r].y, kk * u1);
    o0 = fmaf(x0, qq, o0);
    o1 = fmaf(x1, qq, o1);
    Sp[i * NCP + cp] = __floats2bfloat162_rn(x0, x1);
  }
  __syncthreads();
  part[rb][2 * cp] = o0;
  part[rb][2 * cp + 1] = o1;
  __syncthreads();
  if (tid < D) store_io(io.o, unit * D + tid, part[0][tid] + part[1][tid] + part[2][tid] + part[3][tid], st.io);
}

}  // namespace pace

cudaError_t pace_launch_decode_bf16(const PaceDev &d, const PaceIO &io, cudaStream_t s) {
  using namespace pace;
  const unsigned units = (unsigned)(d.B * d.H);
  if (units == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = pdl_config(dim3(units), dim3(2 * d.D), 0, s, attr);
  const int late = units > 32 && units <= (unsigned)device_sm_count();
  return d.D == 128 ? cudaLaunchKernelEx(&cfg, decode_bf16_kernel<128>, d, io, late)
                    : cudaLaunchKernelEx(&cfg, decode_bf16_kernel<64>, d, io, late);
}
