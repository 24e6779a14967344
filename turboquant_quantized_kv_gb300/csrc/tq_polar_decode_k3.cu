// Polar decode kernels with 3-bit key angles (see tq_polar.cu).
#include "tq_polar.cuh"

namespace tq {
template cudaError_t polar_decode_bk<3>(const PolarDecodeArgs&, int, int, cudaStream_t);
}  // namespace tq
