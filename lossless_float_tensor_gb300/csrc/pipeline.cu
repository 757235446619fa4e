// Split-send pipeline on one GPU (UCCL-Zip Fig. 1 b and Fig. 4 d: expose
// transmissible data early and overlap the transfer with the remaining
// compression; NCCLZ Sec. IV-D4: two ping-pong staging banks, batch i+1 is
// encoded into one bank while batch i is in flight from the other).  The
// device-to-host copy into pinned memory stands in for the wire.
#include "uzip_internal.cuh"

namespace uzip {

// Copies exactly total_bytes (read from the container header on the device)
// into mapped host memory with 16-byte stores.  total_bytes is a multiple of
// 16 for every container the compressor writes; a failed compression has
// total_bytes = 0 and copies nothing.
__global__ void copy_exact_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst) {
    const uint64_t total = *reinterpret_cast<const volatile uint64_t*>(src + 40);
    const uint64_t nvec = total / 16;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride)
        reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
}

cudaError_t launch_copy_exact(const void* d_container, void* h_dst_mapped, cudaStream_t s) {
    int sms = 0, per_sm = 0;
    cudaError_t err;
    if ((err = launch_shape(reinterpret_cast<const void*>(copy_exact_kernel), 512, 0, &sms, &per_sm)) != cudaSuccess)
        return err;
    copy_exact_kernel<<<dim3(uint32_t(sms) * 2), dim3(512), 0, s>>>(static_cast<const uint8_t*>(d_container),
                                                                      static_cast<uint8_t*>(h_dst_mapped));
    return cudaGetLastError();
}

}  // namespace uzip

namespace {
bool host_mapped(const void* p, void** dev) {
    cudaPointerAttributes attr;
    if (p == nullptr || cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return false;
    if (dev) *dev = attr.devicePointer;
    return true;
}
}  // namespace

namespace {
// Copies one message's container to the host while its compression runs:
// the remainder plane in runs of finished chunks (their split posted), the
// exponent section in runs of placed chunks (their stream end posted), then,
// once the kernel is done, the header and chunk table.  Progress words are
// read from the host bank at prog_off (mapped memory the kernel writes).
cudaError_t stream_out(int dtype, uint64_t n, const uint8_t* db, uint8_t* hb, uint64_t prog_off, cudaEvent_t done,
                       cudaStream_t sx) {
    using namespace uzip;
    const uint64_t C = num_chunks(n);
    const uint64_t rem_off = rem_offset(n), exp_off = exp_offset(dtype, n);
    const uint64_t rem_end = rem_off + rem_plane_bytes(dtype, n);
    const uint64_t rem_chunk = uint64_t(kChunk) / 8 * rem_bits(dtype);
    const volatile uint64_t* prog = reinterpret_cast<const volatile uint64_t*>(hb + prog_off);
    constexpr uint64_t kRun = 64;  // chunks per copy while the kernel runs
    uint64_t rem_done = 0, exp_done = 0, exp_end = 0;
    bool kernel_done = false;
    cudaError_t err = cudaSuccess;
    while (err == cudaSuccess) {
        uint64_t p = rem_done;
        while (p < C && prog[2 * p] != 0) ++p;
        if (p > rem_done && (p - rem_done >= kRun || p == C || kernel_done)) {
            const uint64_t lo = rem_off + rem_done * rem_chunk, hi = p == C ? rem_end : rem_off + p * rem_chunk;
            err = cudaMemcpyAsync(hb + lo, db + lo, hi - lo, cudaMemcpyDeviceToHost, sx);
            rem_done = p;
        }
        uint64_t q = exp_done, end = exp_end;
        while (q < C) {
            const uint64_t v = prog[2 * q + 1];
            if (!(v >> 63)) break;
            end = v & ~(1ull << 63);
            ++q;
        }
        if (err == cudaSuccess && q > exp_done && (q - exp_done >= kRun || q == C || kernel_done)) {
            if (end > exp_end)
                err = cudaMemcpyAsync(hb + exp_off + exp_end, db + exp_off + exp_end, end - exp_end,
                                      cudaMemcpyDeviceToHost, sx);
            exp_done = q;
            exp_end = end;
        }
        if ((rem_done == C && exp_done == C) || kernel_done) break;
        const cudaError_t qs = cudaEventQuery(done);
        if (qs == cudaSuccess) kernel_done = true;  // one more pass picks up the last posts
        else if (qs != cudaErrorNotReady) err = qs;
    }
    if (err == cudaSuccess) err = cudaEventSynchronize(done);
    // header, chunk table and padding, final once the kernel is done
    if (err == cudaSuccess) err = cudaMemcpyAsync(hb, db, rem_off, cudaMemcpyDeviceToHost, sx);
    return err;
}
}  // namespace

extern "C" uzip_status uzip_pipeline_send_ex(uzip_dtype dtype, const void* const* d_msgs, const uint64_t* msg_elems,
                                             uint32_t n_msgs, void* const* d_bank, uint64_t bank_capacity,
                                             void* const* h_bank, uint32_t n_hbanks, uint64_t h_capacity,
                                             uint64_t* h_sizes, uzip_pipe_mode mode, uint64_t raw_below_bytes,
                                             cudaStream_t s_compress, cudaStream_t s_copy) {
    using namespace uzip;
    if (!valid_dtype(dtype)) return UZIP_ERR_UNSUPPORTED_DTYPE;
    if (n_msgs == 0 || !d_msgs || !msg_elems || !d_bank || !h_bank || !h_sizes || n_hbanks < 2)
        return UZIP_ERR_INVALID_ARG;
    if (mode != UZIP_PIPE_EXACT && mode != UZIP_PIPE_BOUND && mode != UZIP_PIPE_SERIAL && mode != UZIP_PIPE_SIZED &&
        mode != UZIP_PIPE_STREAMED)
        return UZIP_ERR_INVALID_ARG;
    uint64_t largest = 0;
    for (uint32_t k = 0; k < n_msgs; ++k) {
        if (msg_elems[k] > UZIP_MAX_ELEMS) return UZIP_ERR_INVALID_ARG;
        if (msg_elems[k] > largest) largest = msg_elems[k];
    }
    if (bank_capacity < uzip_max_compressed_size(dtype, largest)) return UZIP_ERR_CAPACITY;
    if (h_capacity < container_bound(dtype, largest)) return UZIP_ERR_CAPACITY;
    // streamed: the host banks also hold 16 bytes of progress per chunk
    const uint64_t prog_off = round16(container_bound(dtype, largest));
    if (mode == UZIP_PIPE_STREAMED && h_capacity < prog_off + 16 * num_chunks(largest)) return UZIP_ERR_CAPACITY;
    void* sizes_dev = nullptr;
    for (int b = 0; b < 2; ++b)
        if (!d_bank[b] || (reinterpret_cast<uintptr_t>(d_bank[b]) & 15)) return UZIP_ERR_INVALID_ARG;
    for (uint32_t b = 0; b < n_hbanks; ++b) {
        void* hd = nullptr;
        if (!host_mapped(h_bank[b], &hd) || (reinterpret_cast<uintptr_t>(hd) & 15)) return UZIP_ERR_INVALID_ARG;
        for (uint32_t b2 = 0; b2 < b; ++b2)
            if (h_bank[b2] == h_bank[b]) return UZIP_ERR_INVALID_ARG;
    }
    if (d_bank[0] == d_bank[1]) return UZIP_ERR_INVALID_ARG;
    if (!host_mapped(h_sizes, &sizes_dev) || (reinterpret_cast<uintptr_t>(sizes_dev) & 7)) return UZIP_ERR_INVALID_ARG;

    const bool serial = mode == UZIP_PIPE_SERIAL;
    cudaStream_t sc = s_compress;
    cudaStream_t sx = serial ? s_compress : s_copy;
    // whole-message RAW below the threshold (NCCLZ Sec. IV-C: a message whose
    // coding does not pay travels RAW).  A RAW container needs only its own
    // bytes in a device bank, so when every message travels RAW each bank
    // holds up to kSubSlots of them and up to 2 kSubSlots messages are in
    // flight instead of two (small messages are bound by the latency of the
    // hand-over between the streams, not by the copy engine).
    constexpr uint32_t kSubSlots = 8;
    bool all_raw = true;
    uint64_t raw_need = 0;
    for (uint32_t k = 0; k < n_msgs; ++k) {
        if (msg_elems[k] * elem_bytes(dtype) >= raw_below_bytes) all_raw = false;
        const uint64_t need = (container_bound(dtype, msg_elems[k]) + 255) & ~uint64_t(255);
        if (need > raw_need) raw_need = need;
    }
    uint32_t sub = 1;
    if (all_raw && !serial && raw_need > 0) {
        const uint64_t fit = bank_capacity / raw_need;
        sub = fit < kSubSlots ? uint32_t(fit) : kSubSlots;
        if (sub < 1) sub = 1;
    }
    const uint32_t nslots = 2 * sub;  // slot v: bank v % 2, at (v / 2) * raw_need in it
    cudaEvent_t compressed[2 * kSubSlots] = {}, copied[2 * kSubSlots] = {};
    uzip_status result = UZIP_OK;
    for (uint32_t v = 0; v < nslots && result == UZIP_OK; ++v) {
        if (cudaEventCreateWithFlags(&compressed[v], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&copied[v], cudaEventDisableTiming) != cudaSuccess)
            result = UZIP_ERR_CUDA;
    }
    for (uint32_t k = 0; k < n_msgs && result == UZIP_OK; ++k) {
        const uint32_t b = k % nslots;      // device slot
        void* dbank = static_cast<uint8_t*>(d_bank[b % 2]) + uint64_t(b / 2) * raw_need;
        void* hb = h_bank[k % n_hbanks];    // host bank
        void* hd = nullptr;                 // its device-side address
        host_mapped(hb, &hd);
        // a RAW message asked to stream is copied with the sized scheme
        const bool raw_msg = msg_elems[k] * elem_bytes(dtype) < raw_below_bytes;
        const uzip_pipe_mode mk = (raw_msg && mode == UZIP_PIPE_STREAMED) ? UZIP_PIPE_SIZED : mode;
        // slot b still holds message k - nslots until its copy has finished
        if (k >= nslots && !serial && cudaStreamWaitEvent(sc, copied[b], 0) != cudaSuccess) {
            result = UZIP_ERR_CUDA;
            break;
        }
        if (raw_msg) {
            if (msg_elems[k] > 0 && (!d_msgs[k] || (reinterpret_cast<uintptr_t>(d_msgs[k]) & 15))) {
                result = UZIP_ERR_INVALID_ARG;
                break;
            }
            if (launch_compress(dtype, d_msgs[k], msg_elems[k], dbank, static_cast<uint64_t*>(sizes_dev) + k, nullptr,
                                0, sc, 1) != cudaSuccess) {
                result = UZIP_ERR_CUDA;
                break;
            }
        } else if (mk == UZIP_PIPE_STREAMED) {
            // progress words live past the container in the host bank
            volatile uint64_t* prog = reinterpret_cast<volatile uint64_t*>(static_cast<uint8_t*>(hb) + prog_off);
            for (uint64_t i = 0; i < 2 * num_chunks(msg_elems[k]); ++i) prog[i] = 0;
            if (msg_elems[k] > 0 && (!d_msgs[k] || (reinterpret_cast<uintptr_t>(d_msgs[k]) & 15))) {
                result = UZIP_ERR_INVALID_ARG;
                break;
            }
            uint64_t* prog_dev = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(hd) + prog_off);
            if (launch_compress(dtype, d_msgs[k], msg_elems[k], dbank, static_cast<uint64_t*>(sizes_dev) + k, nullptr,
                                0, sc, 0, prog_dev) != cudaSuccess) {
                result = UZIP_ERR_CUDA;
                break;
            }
        } else {
            result = uzip_compress(d_msgs[k], dtype, msg_elems[k], dbank, bank_capacity,
                                   static_cast<uint64_t*>(sizes_dev) + k, sc);
            if (result != UZIP_OK) break;
        }
        // streamed copies run while the kernel does: only they skip the wait
        if (!serial && (cudaEventRecord(compressed[b], sc) != cudaSuccess ||
                        (mk != UZIP_PIPE_STREAMED && cudaStreamWaitEvent(sx, compressed[b], 0) != cudaSuccess))) {
            result = UZIP_ERR_CUDA;
            break;
        }
        cudaError_t err = cudaSuccess;
        if (mk == UZIP_PIPE_STREAMED) {
            err = stream_out(dtype, msg_elems[k], static_cast<const uint8_t*>(dbank), static_cast<uint8_t*>(hb),
                             prog_off, compressed[b], sx);
        } else if (mk == UZIP_PIPE_BOUND || (mk == UZIP_PIPE_SIZED && raw_msg)) {
            // a whole-message RAW container is exactly the bound: its size is
            // known on the host without waiting for the compression
            err = cudaMemcpyAsync(hb, dbank, container_bound(dtype, msg_elems[k]), cudaMemcpyDeviceToHost, sx);
        } else if (mk == UZIP_PIPE_SIZED) {
            // the size is known once this compression is done; message k-1's
            // copy keeps running on s_copy meanwhile
            err = cudaEventSynchronize(compressed[b]);
            const uint64_t total = *reinterpret_cast<volatile const uint64_t*>(h_sizes + k);
            if (err == cudaSuccess && total > 0)
                err = cudaMemcpyAsync(hb, dbank, total, cudaMemcpyDeviceToHost, sx);
        } else {
            err = launch_copy_exact(dbank, hd, sx);
        }
        if (err == cudaSuccess && !serial) err = cudaEventRecord(copied[b], sx);
        if (err != cudaSuccess) result = UZIP_ERR_CUDA;
    }
    for (uint32_t v = 0; v < 2 * kSubSlots; ++v) {
        if (compressed[v]) cudaEventDestroy(compressed[v]);
        if (copied[v]) cudaEventDestroy(copied[v]);
    }
    if (result == UZIP_ERR_CUDA) cudaGetLastError();
    return result;
}

extern "C" uzip_status uzip_pipeline_send(uzip_dtype dtype, const void* const* d_msgs, const uint64_t* msg_elems,
                                          uint32_t n_msgs, void* const* d_bank, uint64_t bank_capacity,
                                          void* const* h_bank, uint64_t h_capacity, uint64_t* h_sizes,
                                          uzip_pipe_mode mode, cudaStream_t s_compress, cudaStream_t s_copy) {
    return uzip_pipeline_send_ex(dtype, d_msgs, msg_elems, n_msgs, d_bank, bank_capacity, h_bank, 2, h_capacity,
                                 h_sizes, mode, UZIP_PIPE_RAW_BELOW_DEFAULT, s_compress, s_copy);
}
