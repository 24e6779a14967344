// Polar decode kernels with 4-bit key angles (see tq_polar.cu).
#include "tq_polar.cuh"

namespace tq {
template cudaError_t polar_decode_bk<4>(const PolarDecodeArgs&, int, int, cudaStream_t);
}  // namespace tq
