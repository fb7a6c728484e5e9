// Instantiation of the folded-readout decode kernels for symmetric codes, mixed decode buffer.
#include "decode_fold.cuh"

namespace pace {
template cudaError_t launch_fold_zm<0, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t);
}  // namespace pace
