// Instantiation of the folded-readout decode kernels for symmetric codes, int8 decode buffer (PACE-4).
#include "decode_fold.cuh"

namespace pace {
template cudaError_t launch_fold_zm<0, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t);
}  // namespace pace
