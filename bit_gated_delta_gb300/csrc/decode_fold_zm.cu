// Instantiation of the folded-readout decode kernels for zero-point codes, mixed decode buffer (PACE-4/8).
#include "decode_fold.cuh"

namespace pace {
template cudaError_t launch_fold_zm<1, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t);
}  // namespace pace
