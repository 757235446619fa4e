// Compressor kernels for one element format (fp8_e4m3).
#include "compress_ws.cuh"

namespace uzip {
template cudaError_t launch_mode<UZIP_FP8_E4M3>(CompressArgs, int, bool, cudaStream_t);
}  // namespace uzip
