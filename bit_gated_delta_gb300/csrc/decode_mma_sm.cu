// Instantiation of the quantized decode kernels for symmetric codes, mixed decode buffer.
#include "decode_mma.cuh"

namespace pace {
template cudaError_t launch_quant_zm<0, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
}  // namespace pace
