// Compressor kernels for one element format (bf16).
#include "compress_ws.cuh"

namespace uzip {
template cudaError_t launch_mode<UZIP_BF16>(CompressArgs, int, bool, cudaStream_t);
}  // namespace uzip
