// Instantiation of the folded-readout decode kernel with 32-token tables: int4 symmetric state, g = 64, int8
// decode buffer, every head at 4 bits, periods of 9..32 tokens (the long-context rounding periods).
#include "decode_fold.cuh"

bool pace_fold32_supported(const PaceDev &d) {
  return d.state_mode == PACE_STATE_QUANT && d.dP > pace::DF_TOK && d.dP <= 32 && d.G == 64 && !d.zero_point &&
         d.buf_mode == PACE_BUF_INT8 && d.H8 == 0 && (d.D == 128 || d.D == 64);
}

// One warp per unit (each warp of a block would need its own 33 KB work area).
cudaError_t pace_launch_decode_fold32(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  const long units = (long)d.B * d.H4;
  if (units == 0) return cudaSuccess;
  return d.D == 128 ? launch_fold_w<128, 64, 4, 0, 0, 1, 32>(d, io, has_token, s, units)
                    : launch_fold_w<64, 64, 4, 0, 0, 1, 32>(d, io, has_token, s, units);
}
