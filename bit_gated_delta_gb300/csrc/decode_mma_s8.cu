// Instantiation of the quantized decode kernels for symmetric codes, int8 decode buffer (PACE-4).
#include "decode_mma.cuh"

namespace pace {
template cudaError_t launch_quant_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
}  // namespace pace

#ifndef PACE_DECODE_COL
#define PACE_DECODE_COL 0   // 1: int4 pools of d = 128, int8-buffer, dP <= 8 states on the column kernel
#endif

cudaError_t pace_launch_decode_quant(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  const int mx = d.buf_mode == PACE_BUF_MIXED;
  // int4 heads of d = 128 states with an int8 buffer and dP <= 8: the column kernel (tcgen05); the int8 pool and
  // every other shape: the warp-level kernels
  const bool col = PACE_DECODE_COL && pace_decode_col_supported(d);
  if (col) {
    cudaError_t e = pace_launch_decode_col(d, io, has_token, s);
    if (e != cudaSuccess) return e;
  }
  if (d.zero_point) return mx ? launch_quant_zm<1, 1>(d, io, has_token, s, !col) : launch_quant_zm<1, 0>(d, io, has_token, s, !col);
  return mx ? launch_quant_zm<0, 1>(d, io, has_token, s, !col) : launch_quant_zm<0, 0>(d, io, has_token, s, !col);
}
