// Instantiation of the quantized decode kernels for zero-point codes, int8 decode buffer.
#include "decode_mma.cuh"

namespace pace {
template cudaError_t launch_quant_zm<1, 0>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
}  // namespace pace
