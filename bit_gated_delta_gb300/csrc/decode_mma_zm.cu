// Instantiation of the quantized decode kernels for zero-point codes, mixed decode buffer (PACE-4/8).
#include "decode_mma.cuh"

namespace pace {
template cudaError_t launch_quant_zm<1, 1>(const PaceDev &, const PaceIO &, int, cudaStream_t, bool);
}  // namespace pace
