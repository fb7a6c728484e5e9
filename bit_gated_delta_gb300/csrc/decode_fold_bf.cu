// Instantiation of the folded-readout decode kernels for the buffered bf16 state (int8 decode buffer, bf16 state
// rounded once every dP tokens).
#include "decode_fold.cuh"

cudaError_t pace_launch_decode_bf16buf_fold(const PaceDev &d, const PaceIO &io, int has_token, cudaStream_t s) {
  return pace::launch_fold_bf16buf(d, io, has_token, s);
}
