// Instantiation of the quantized decode kernels for symmetric codes, int8 decode buffer (PACE-4).
#include "decode_mma.cuh"

namespace pace {
template cudaError_t launch_quant_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
}  // namespace pace

constexpr int DF_TOK_MAX = 8;   // the folded-readout kernels handle decode periods of up to 8 tokens

namespace pace {
template <int ZP, int MX>
cudaError_t launch_fold_zm(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s);
extern template cudaError_t launch_fold_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
extern template cudaError_t launch_fold_zm<0, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t);
extern template cudaError_t launch_fold_zm<1, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
extern template cudaError_t launch_fold_zm<1, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t);
}  // namespace pace

cudaError_t pace_launch_decode_quant(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  const int mx = d.buf_mode == PACE_BUF_MIXED;
  // periods of up to 8 tokens: the folded-readout kernels (decode_fold.cuh); longer periods: decode_mma.cuh, except
  // the int4 symmetric case below
  if (d.dP <= DF_TOK_MAX) {
    if (d.zero_point) return mx ? launch_fold_zm<1, 1>(d, io, has_token, s) : launch_fold_zm<1, 0>(d, io, has_token, s);
    return mx ? launch_fold_zm<0, 1>(d, io, has_token, s) : launch_fold_zm<0, 0>(d, io, has_token, s);
  }
  // up to 32 tokens, int4 symmetric g = 64 with the int8 buffer: the folded readout with 32-token tables
  if (pace_fold32_supported(d)) return pace_launch_decode_fold32(d, io, has_token, s);
  if (d.zero_point) return mx ? launch_quant_zm<1, 1>(d, io, has_token, s) : launch_quant_zm<1, 0>(d, io, has_token, s);
  return mx ? launch_quant_zm<0, 1>(d, io, has_token, s) : launch_quant_zm<0, 0>(d, io, has_token, s);
}
