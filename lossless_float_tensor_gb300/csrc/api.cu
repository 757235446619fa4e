// C ABI of the uzip library: argument checks, work-area layout and launches.
// Every check that can be made on the host is made before anything is
// enqueued, so that no kernel is ever launched on a buffer it would overrun.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "uzip_internal.cuh"
#include "../../include/uzip_debug.h"

namespace {

using namespace uzip;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

typedef CUresult (*AddrRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);

AddrRangeFn addr_range_fn() {
    static AddrRangeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddrRangeFn>(p);
        tried = true;
    }
    return fn;
}

// [p, p + bytes) must be device-accessible memory.  Device allocations are
// checked against the allocation that holds p; mapped host memory is accepted
// by type (its extent is not known to the driver query).
bool device_range_ok(const void* p, uint64_t bytes) {
    if (bytes == 0) return true;
    if (p == nullptr) return false;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type == cudaMemoryTypeHost) return attr.devicePointer != nullptr;
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return false;
    AddrRangeFn fn = addr_range_fn();
    if (!fn) return true;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fn(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return true;  // not a plain allocation
    const uint64_t start = reinterpret_cast<uint64_t>(p) - uint64_t(base);
    return start <= size && bytes <= size - start;
}

}  // namespace

namespace uzip {
namespace {
struct ShapeEntry {
    int dev;
    const void* kern;
    int threads;
    size_t smem;
    int sms, per_sm;
};
std::mutex g_shape_mutex;
ShapeEntry g_shapes[64];
int g_num_shapes = 0;
}  // namespace

cudaError_t launch_shape(const void* kern, int threads, size_t smem, int* sms, int* per_sm) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_shape_mutex);
    for (int i = 0; i < g_num_shapes; ++i) {
        const ShapeEntry& e = g_shapes[i];
        if (e.dev == dev && e.kern == kern && e.threads == threads && e.smem == smem) {
            *sms = e.sms;
            *per_sm = e.per_sm;
            return cudaSuccess;
        }
    }
    int n_sms = 0, blocks = 0;
    if ((err = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, threads, smem)) != cudaSuccess) return err;
    if (blocks < 1) blocks = 1;
    if (g_num_shapes < 64) g_shapes[g_num_shapes++] = ShapeEntry{dev, kern, threads, smem, n_sms, blocks};
    *sms = n_sms;
    *per_sm = blocks;
    return cudaSuccess;
}
}  // namespace uzip

extern "C" {

uint64_t uzip_max_compressed_size(uzip_dtype dtype, uint64_t n) {
    if (!valid_dtype(dtype) || n > UZIP_MAX_ELEMS) return 0;
    return scratch_offset(dtype, n) + work_area_bytes(n);
}

uzip_status uzip_compress_ex(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out, uint64_t out_capacity,
                             uint64_t* d_out_size, int32_t* d_status, uint32_t flags, cudaStream_t s) {
    if (!valid_dtype(dtype)) return UZIP_ERR_UNSUPPORTED_DTYPE;
    if (n > UZIP_MAX_ELEMS) return UZIP_ERR_INVALID_ARG;
    if (n > 0 && (d_in == nullptr || !aligned(d_in, 16))) return UZIP_ERR_INVALID_ARG;
    if (d_out == nullptr || !aligned(d_out, 16)) return UZIP_ERR_INVALID_ARG;
    if (d_out_size && !aligned(d_out_size, 8)) return UZIP_ERR_INVALID_ARG;
    if (d_status && !aligned(d_status, 4)) return UZIP_ERR_INVALID_ARG;
    if ((flags & ~(UZIP_TESTFLAG_SKIP_CHUNK0 | UZIP_FLAG_SAMPLED_TABLES)) != 0) return UZIP_ERR_INVALID_ARG;
    const uint64_t need = uzip_max_compressed_size(dtype, n);
    if (out_capacity < need) return UZIP_ERR_CAPACITY;
    if (!device_range_ok(d_in, n * elem_bytes(dtype)) || !device_range_ok(d_out, need) ||
        (d_out_size && !device_range_ok(d_out_size, 8)) || (d_status && !device_range_ok(d_status, 4)))
        return UZIP_ERR_INVALID_ARG;
    const uint32_t first = (flags & UZIP_TESTFLAG_SKIP_CHUNK0) ? 1u : 0u;
    const int mode = (flags & UZIP_FLAG_SAMPLED_TABLES) ? 3 : 0;
    if (launch_compress(dtype, d_in, n, d_out, d_out_size, d_status, first, s, mode) != cudaSuccess) {
        cudaGetLastError();
        return UZIP_ERR_CUDA;
    }
    return UZIP_OK;
}

uzip_status uzip_compress(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out, uint64_t out_capacity,
                          uint64_t* d_out_size, cudaStream_t s) {
    return uzip_compress_ex(d_in, dtype, n, d_out, out_capacity, d_out_size, nullptr, 0, s);
}

uzip_status uzip_compress_parametric(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out,
                                     uint64_t out_capacity, uint64_t* d_out_size, int32_t* d_status, double sigma,
                                     cudaStream_t s) {
    if (!valid_dtype(dtype)) return UZIP_ERR_UNSUPPORTED_DTYPE;
    if (n > UZIP_MAX_ELEMS) return UZIP_ERR_INVALID_ARG;
    if (n > 0 && (d_in == nullptr || !aligned(d_in, 16))) return UZIP_ERR_INVALID_ARG;
    if (d_out == nullptr || !aligned(d_out, 16)) return UZIP_ERR_INVALID_ARG;
    if (d_out_size && !aligned(d_out_size, 8)) return UZIP_ERR_INVALID_ARG;
    if (d_status && !aligned(d_status, 4)) return UZIP_ERR_INVALID_ARG;
    uint32_t model[256];
    if (!model_counts(dtype, sigma, model)) return UZIP_ERR_INVALID_ARG;
    const uint64_t need = uzip_max_compressed_size(dtype, n);
    if (out_capacity < need) return UZIP_ERR_CAPACITY;
    if (!device_range_ok(d_in, n * elem_bytes(dtype)) || !device_range_ok(d_out, need) ||
        (d_out_size && !device_range_ok(d_out_size, 8)) || (d_status && !device_range_ok(d_status, 4)))
        return UZIP_ERR_INVALID_ARG;
    if (launch_compress(dtype, d_in, n, d_out, d_out_size, d_status, 0, s, 4, nullptr, model) != cudaSuccess) {
        cudaGetLastError();
        return UZIP_ERR_CUDA;
    }
    return UZIP_OK;
}

uzip_status uzip_compress_gated(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out, uint64_t out_capacity,
                                uint64_t* d_out_size, int32_t* d_status, uint64_t raw_below_bytes, cudaStream_t s) {
    if (!valid_dtype(dtype)) return UZIP_ERR_UNSUPPORTED_DTYPE;
    if (n > UZIP_MAX_ELEMS) return UZIP_ERR_INVALID_ARG;
    if (n > 0 && (d_in == nullptr || !aligned(d_in, 16))) return UZIP_ERR_INVALID_ARG;
    if (d_out == nullptr || !aligned(d_out, 16)) return UZIP_ERR_INVALID_ARG;
    if (d_out_size && !aligned(d_out_size, 8)) return UZIP_ERR_INVALID_ARG;
    if (d_status && !aligned(d_status, 4)) return UZIP_ERR_INVALID_ARG;
    const uint64_t need = uzip_max_compressed_size(dtype, n);
    if (out_capacity < need) return UZIP_ERR_CAPACITY;
    if (!device_range_ok(d_in, n * elem_bytes(dtype)) || !device_range_ok(d_out, need) ||
        (d_out_size && !device_range_ok(d_out_size, 8)) || (d_status && !device_range_ok(d_status, 4)))
        return UZIP_ERR_INVALID_ARG;
    const int mode = n * elem_bytes(dtype) < raw_below_bytes ? 1 : 2;
    if (launch_compress(dtype, d_in, n, d_out, d_out_size, d_status, 0, s, mode) != cudaSuccess) {
        cudaGetLastError();
        return UZIP_ERR_CUDA;
    }
    return UZIP_OK;
}

uzip_status uzip_compress_noalloc(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out, uint64_t out_capacity,
                                  uint64_t* d_out_size, int32_t* d_status, cudaStream_t s) {
    if (!valid_dtype(dtype)) return UZIP_ERR_UNSUPPORTED_DTYPE;
    if (n > UZIP_NOALLOC_MAX_ELEMS) return UZIP_ERR_TOO_LARGE;
    if (n > 0 && (d_in == nullptr || !aligned(d_in, 16))) return UZIP_ERR_INVALID_ARG;
    if (d_out == nullptr || !aligned(d_out, 16)) return UZIP_ERR_INVALID_ARG;
    if (d_out_size && !aligned(d_out_size, 8)) return UZIP_ERR_INVALID_ARG;
    if (d_status && !aligned(d_status, 4)) return UZIP_ERR_INVALID_ARG;
    const uint64_t need = container_bound(dtype, n);
    if (out_capacity < need) return UZIP_ERR_CAPACITY;
    if (!device_range_ok(d_in, n * elem_bytes(dtype)) || !device_range_ok(d_out, need) ||
        (d_out_size && !device_range_ok(d_out_size, 8)) || (d_status && !device_range_ok(d_status, 4)))
        return UZIP_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (noalloc_scratch_address(&scratch) != cudaSuccess ||
        launch_compress_with_scratch(dtype, d_in, n, d_out, d_out_size, d_status, 0, scratch, nullptr, s) !=
            cudaSuccess) {
        cudaGetLastError();
        return UZIP_ERR_CUDA;
    }
    return UZIP_OK;
}

uzip_status uzip_decompress(const void* d_comp, uint64_t comp_capacity, void* d_out, uzip_dtype dtype, uint64_t n,
                            int32_t* d_status, cudaStream_t s) {
    if (!valid_dtype(dtype)) return UZIP_ERR_UNSUPPORTED_DTYPE;
    if (n > UZIP_MAX_ELEMS) return UZIP_ERR_INVALID_ARG;
    if (d_comp == nullptr || !aligned(d_comp, 16)) return UZIP_ERR_INVALID_ARG;
    if (n > 0 && (d_out == nullptr || !aligned(d_out, 16))) return UZIP_ERR_INVALID_ARG;
    if (d_status && !aligned(d_status, 4)) return UZIP_ERR_INVALID_ARG;
    if (comp_capacity < kHeader) return UZIP_ERR_CORRUPT;
    if (!device_range_ok(d_comp, comp_capacity) || !device_range_ok(d_out, n * elem_bytes(dtype)) ||
        (d_status && !device_range_ok(d_status, 4)))
        return UZIP_ERR_INVALID_ARG;
    if (launch_decompress(dtype, d_comp, comp_capacity, d_out, n, d_status, s) != cudaSuccess) {
        cudaGetLastError();
        return UZIP_ERR_CUDA;
    }
    return UZIP_OK;
}

uzip_status uzip_query_size(const void* d_comp, uint64_t* h_total_bytes, uzip_dtype* h_dtype, uint64_t* h_n,
                            cudaStream_t s) {
    if (d_comp == nullptr || !aligned(d_comp, 16)) return UZIP_ERR_INVALID_ARG;
    if (!device_range_ok(d_comp, kHeader)) return UZIP_ERR_INVALID_ARG;
    uint8_t h[kHeader];
    if (cudaMemcpyAsync(h, d_comp, kHeader, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return UZIP_ERR_CUDA;
    }
    uint32_t magic, chunk, c;
    uint16_t version;
    uint64_t n, roff, eoff, total;
    std::memcpy(&magic, h, 4);
    std::memcpy(&version, h + 4, 2);
    std::memcpy(&n, h + 8, 8);
    std::memcpy(&chunk, h + 16, 4);
    std::memcpy(&c, h + 20, 4);
    std::memcpy(&roff, h + 24, 8);
    std::memcpy(&eoff, h + 32, 8);
    std::memcpy(&total, h + 40, 8);
    const int dt = h[6];
    if (magic != 0x31505A55u || version != 1 || !valid_dtype(dt) || h[7] != 0 || chunk != kChunk ||
        n > UZIP_MAX_ELEMS || c != num_chunks(n) || roff != rem_offset(n) || eoff != exp_offset(dt, n) ||
        total < eoff || total == 0)
        return UZIP_ERR_CORRUPT;
    if (h_total_bytes) *h_total_bytes = total;
    if (h_dtype) *h_dtype = static_cast<uzip_dtype>(dt);
    if (h_n) *h_n = n;
    return UZIP_OK;
}

const char* uzip_status_string(uzip_status st) {
    switch (st) {
        case UZIP_OK: return "ok";
        case UZIP_ERR_INVALID_ARG: return "invalid argument";
        case UZIP_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case UZIP_ERR_CAPACITY: return "output buffer too small";
        case UZIP_ERR_CORRUPT: return "corrupt container";
        case UZIP_ERR_TIMEOUT: return "device-side wait timed out";
        case UZIP_ERR_CUDA: return "CUDA error";
        case UZIP_ERR_TOO_LARGE: return "tensor larger than the allocation-free limit";
    }
    return "unknown status";
}

int uzip_debug_div_magic(uint32_t f, uint32_t* m, uint32_t* add, uint32_t* shift) {
    const DivMagic d = div_magic(f);
    if (m) *m = d.m;
    if (add) *add = d.add;
    if (shift) *shift = d.sh + 32;
    return int(d.ok);
}

int uzip_debug_div_magic33(uint32_t f, uint32_t* m_lo, uint32_t* shift) {
    if (f == 0 || f > kM) return 0;
    const Magic33 d = magic33(f);
    if (m_lo) *m_lo = d.m_lo;
    if (shift) *shift = d.sh;
    return 1;
}

void uzip_debug_set_ws_jit_blocks(uint32_t blocks) { g_ws_jit_blocks = blocks; }

int uzip_debug_model_counts(int dtype, double sigma, uint32_t* counts) {
    if (!counts || !valid_dtype(dtype)) return 0;
    return model_counts(dtype, sigma, counts) ? 1 : 0;
}

uint64_t uzip_debug_scratch_offset(uzip_dtype dtype, uint64_t n) {
    if (!valid_dtype(dtype) || n > UZIP_MAX_ELEMS) return 0;
    return scratch_offset(dtype, n);
}

}  // extern "C"
