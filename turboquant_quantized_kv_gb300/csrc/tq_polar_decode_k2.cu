// Polar decode kernels with 2-bit key angles (see tq_polar.cu).
#include "tq_polar.cuh"

namespace tq {
template cudaError_t polar_decode_bk<2>(const PolarDecodeArgs&, int, int, cudaStream_t);
}  // namespace tq
