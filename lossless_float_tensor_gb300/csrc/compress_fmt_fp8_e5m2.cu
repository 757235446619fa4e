// Compressor kernels for one element format (fp8_e5m2).
#include "compress_ws.cuh"

namespace uzip {
template cudaError_t launch_mode<UZIP_FP8_E5M2>(CompressArgs, int, bool, cudaStream_t);
}  // namespace uzip
