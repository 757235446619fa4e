// Compressor kernels for one element format (fp32).
#include "compress_ws.cuh"

namespace uzip {
template cudaError_t launch_mode<UZIP_FP32>(CompressArgs, int, bool, cudaStream_t);
}  // namespace uzip
