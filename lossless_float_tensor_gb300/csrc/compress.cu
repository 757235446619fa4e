// Compressor host side: the launch entry points used by the C ABI and the
// allocation-free work area.  The device code lives in compress_kernels.cuh
// and is compiled once per element format (compress_fmt_*.cu).
#include <cuda.h>

#include <cmath>

#include <mutex>

#include "compress_kernels.cuh"

namespace uzip {

// tuning of the warp-specialised compressor (see CompressArgs::jit_blocks)
uint32_t g_ws_jit_blocks = 32;

extern template cudaError_t launch_mode<UZIP_BF16>(CompressArgs, int, bool, cudaStream_t);
extern template cudaError_t launch_mode<UZIP_FP32>(CompressArgs, int, bool, cudaStream_t);
extern template cudaError_t launch_mode<UZIP_FP16>(CompressArgs, int, bool, cudaStream_t);
extern template cudaError_t launch_mode<UZIP_FP8_E4M3>(CompressArgs, int, bool, cudaStream_t);
extern template cudaError_t launch_mode<UZIP_FP8_E5M2>(CompressArgs, int, bool, cudaStream_t);

// ---------------------------------------------------------------------------
// host launchers (called by the C ABI after argument checks)

// Launches the compressor with its work area (status, ticket, done counter,
// look-back descriptors: scratch_bytes(n) bytes) at `scratch`, which is
// zeroed on `s` first (mode 1, whole-message RAW, needs no work area: only
// the container's bytes of d_out are written).
cudaError_t launch_compress_with_scratch(int dtype, const void* d_in, uint64_t n, void* d_out, uint64_t* d_out_size,
                                         int32_t* d_status, uint32_t first_ticket, void* scratch_area, void* stash,
                                         cudaStream_t s, int mode, uint64_t* progress, const uint32_t* model) {
    const uint64_t C = num_chunks(n);
    uint8_t* out = static_cast<uint8_t*>(d_out);
    Scratch* scratch = static_cast<Scratch*>(scratch_area);
    if (mode != 1) {  // the whole-message RAW kernel uses no work area
        const cudaError_t err = cudaMemsetAsync(scratch, 0, scratch_bytes(n), s);
        if (err != cudaSuccess) return err;
    }
    CompressArgs a;
    a.in = static_cast<const uint8_t*>(d_in);
    a.n = n;
    a.out = out;
    a.scratch = scratch;
    a.desc = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(scratch) + kScratchHead);
    a.out_size = d_out_size;
    a.status_out = d_status;
    a.first_ticket = C > 0 ? (first_ticket < C ? first_ticket : uint32_t(C - 1)) : 0;
    a.num_chunks = uint32_t(C);
    a.stash = static_cast<uint8_t*>(stash);
    a.gated = 0;
    a.progress = progress;
    a.jit_blocks = g_ws_jit_blocks;
    a.model_total = 0;
    for (int e = 0; e < 256; ++e) {
        a.model[e] = model ? model[e] : 0u;
        a.model_total += a.model[e];
    }
    const bool has_stash = stash != nullptr;
    switch (dtype) {
        case UZIP_BF16: return launch_mode<UZIP_BF16>(a, mode, has_stash, s);
        case UZIP_FP32: return launch_mode<UZIP_FP32>(a, mode, has_stash, s);
        case UZIP_FP16: return launch_mode<UZIP_FP16>(a, mode, has_stash, s);
        case UZIP_FP8_E4M3: return launch_mode<UZIP_FP8_E4M3>(a, mode, has_stash, s);
        default: return launch_mode<UZIP_FP8_E5M2>(a, mode, has_stash, s);
    }
}

// The regular path: the work area (counters, descriptors, slots) sits in the
// caller's output buffer, behind the largest possible container.
cudaError_t launch_compress(int dtype, const void* d_in, uint64_t n, void* d_out, uint64_t* d_out_size,
                            int32_t* d_status, uint32_t first_ticket, cudaStream_t s, int mode, uint64_t* progress,
                            const uint32_t* model) {
    uint8_t* work = static_cast<uint8_t*>(d_out) + scratch_offset(dtype, n);
    const uintptr_t st = (reinterpret_cast<uintptr_t>(work) + scratch_bytes(n) + 4095) & ~uintptr_t(4095);
    return launch_compress_with_scratch(dtype, d_in, n, d_out, d_out_size, d_status, first_ticket, work,
                                        reinterpret_cast<void*>(st), s, mode, progress, model);
}

// Counts of the Gaussian-model table (ZipCCL abstract: the exponent coding
// follows from the values' Gaussian shape, no statistics gathered online)
// for values ~ N(0, sigma^2).  Exponent field e of a format with bias b holds
// the magnitudes [2^(e-b), 2^(e-b+1)) (e >= 1) or [0, 2^(1-b)) (e = 0); with
// the normal distribution's tail erfc(t / sqrt 2), the binade's probability
// is erfc(x) - erfc(2x) for x = 2^(e-b) / (sigma sqrt 2), and 1 - erfc(2x)
// for e = 0.  Each probability becomes a count out of 65536 rounded to
// nearest, and every value of the field counts at least 1, so that any
// tensor stays codable.  Returns false for a sigma that is not finite and
// positive.
bool model_counts(int dtype, double sigma, uint32_t counts[256]) {
    for (int e = 0; e < 256; ++e) counts[e] = 0;
    if (!(sigma > 0.0) || !std::isfinite(sigma)) return false;
    int ebits = 0;
    switch (dtype) {
        case UZIP_BF16: ebits = Fmt<UZIP_BF16>::kEbits; break;
        case UZIP_FP32: ebits = Fmt<UZIP_FP32>::kEbits; break;
        case UZIP_FP16: ebits = Fmt<UZIP_FP16>::kEbits; break;
        case UZIP_FP8_E4M3: ebits = Fmt<UZIP_FP8_E4M3>::kEbits; break;
        case UZIP_FP8_E5M2: ebits = Fmt<UZIP_FP8_E5M2>::kEbits; break;
        default: return false;
    }
    const int b = (1 << (ebits - 1)) - 1;
    const double unit = sigma * std::sqrt(2.0);  // sigma sqrt 2
    for (int e = 0; e < (1 << ebits); ++e) {
        const double x = std::ldexp(1.0, e - b) / unit;
        const double tail_lo = std::erfc(x), tail_hi = std::erfc(2.0 * x);
        const double p = e == 0 ? 1.0 - tail_hi : tail_lo - tail_hi;
        const double c = std::floor(65536.0 * p + 0.5);
        counts[e] = c < 1.0 ? 1u : uint32_t(c);
    }
    return true;
}

// ---------------------------------------------------------------------------
// Work area for callers that may not allocate device memory (see
// uzip_compress_noalloc).  It lives in the library's own module memory, one
// copy per GPU that loads the library, held until the process exits, and is
// sized for kNoAllocMaxElems elements.  Every call shares it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchHead + 8 * (kNoAllocMaxElems / kChunk)];

namespace {
std::mutex g_noalloc_mutex;
struct NoallocEntry {
    unsigned long long ctx_id;  // CUDA context the address belongs to (0: unknown)
    void* ptr;
};
NoallocEntry g_noalloc[kNoAllocMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the current CUDA context (unique for the life of the process), or 0
// if the driver cannot tell.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
    return 0;
}
}  // namespace

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name only stands in for the symbol, so the address is asked of
// the runtime (with that device current) the first time a device is used and
// kept; it is asked again when the device's CUDA context has changed since
// (a cudaDeviceReset reloads the library's module, and the old address is
// gone), which the context id tells.
cudaError_t noalloc_scratch_address(void** ptr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= int(kNoAllocMaxDevices)) return cudaErrorInvalidDevice;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocEntry& e = g_noalloc[dev];
    if (e.ptr == nullptr || e.ctx_id != id) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        e.ptr = p;
        e.ctx_id = id;
    }
    *ptr = e.ptr;
    return cudaSuccess;
}

}  // namespace uzip
