// Instantiation of the folded-readout decode kernels for the buffered bf16 state (int8 decode buffer, bf16 state
// rounded once every dP tokens).
#include "decode_fold.cuh"

cudaError_t pace_launch_decode_bf16buf_fold(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  using namespace pace;
  return d.D == 128 ? launch_fold_pool<128, 64, 16, 0, 0>(d, io, has_token, s)
                    : launch_fold_pool<64, 64, 16, 0, 0>(d, io, has_token, s);
}
