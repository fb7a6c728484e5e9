// Instantiation of the folded-readout decode kernels for zero-point codes, int8 decode buffer.
#include "decode_fold.cuh"

namespace pace {
template cudaError_t launch_fold_zm<1, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
}  // namespace pace
