// Instantiation of the quantized decode kernels for symmetric codes, int8 decode buffer (PACE-4).
#include "decode_mma.cuh"

namespace pace {
template cudaError_t launch_quant_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
}  // namespace pace

cudaError_t pace_launch_decode_quant(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  const int mx = d.buf_mode == PACE_BUF_MIXED;
  if (d.zero_point) return mx ? launch_quant_zm<1, 1>(d, io, has_token, s) : launch_quant_zm<1, 0>(d, io, has_token, s);
  return mx ? launch_quant_zm<0, 1>(d, io, has_token, s) : launch_quant_zm<0, 0>(d, io, has_token, s);
}
