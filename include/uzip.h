/*
 * uzip -- lossless compression of bf16 / fp16 / fp32 / fp8 GPU tensors (C ABI).
 *
 * What it computes.  Each value is split into its exponent field and the
 * remaining sign and fraction bits; only the exponent field is entropy coded
 * (with ANS), the remainder is stored raw (UCCL-Zip, arXiv 2604.17172,
 * Fig. 2 caption).  Every chunk of work builds its own frequency table, so no
 * global table or cross-block synchronisation is needed for the statistics
 * (UCCL-Zip, Fig. 5 caption).  A chunk that coding does not shrink is stored
 * RAW (NCCLZ, arXiv 2605.12396, Sec. IV-B/IV-C, Alg. 1), and the result is a
 * self-describing frame, header plus payload (NCCLZ Sec. IV-B, IV-D2).
 *
 * Container (little endian):
 *   [0,64)          header: "UZP1", u16 version = 1, u8 dtype, u8 flags = 0,
 *                   u64 n, u32 chunk_elems = 65536, u32 num_chunks C,
 *                   u64 rem_offset, u64 exp_offset, u64 total_bytes,
 *                   16 zero bytes
 *   [64, 64+8C)     u64 offset of chunk c's stream, relative to exp_offset
 *   [64+8C, 64+12C) u32 length of chunk c's stream, bit 31 = stored RAW
 *   rem_offset = round16(64 + 12C): the remainder plane.  Each element
 *                   contributes a w-bit field, its sign placed just above
 *                   its fraction: bf16 w = 8 (sign<<7 | fraction),
 *                   fp32 w = 24 (sign<<23 | fraction), fp16 w = 11
 *                   (sign<<10 | fraction), fp8 e4m3fn w = 4 (sign<<3 |
 *                   fraction), fp8 e5m2 w = 3 (sign<<2 | fraction).  The
 *                   fields are packed back to back, least significant bit
 *                   first: element i occupies bits [w*i, w*i + w) of the
 *                   plane, where bit k of the plane is bit k % 8 of byte
 *                   k / 8; bits past the last field are zero.  For bf16 this
 *                   is one byte per element and for fp32 three little-endian
 *                   bytes.  P = ceil(n * w / 8) bytes.
 *   exp_offset = round16(rem_offset + P): one stream per chunk, each
 *                   starting 16-byte aligned and zero padded to 16 bytes.
 *   The exponent field (8 bits for bf16 and fp32, 5 for fp16 and e5m2, 4
 *   for e4m3fn) is the symbol, one byte per element.
 *   A coded stream is u32 state[32], u8 bitmap[32] of present exponent
 *   bytes, u16 freq[K] (present bytes ascending, summing to 4096) and
 *   u16 words[W]: 32 interleaved rANS states (32-bit, 16-bit renormalisation,
 *   element i on lane i mod 32), the words listed in decoding order.  A RAW
 *   stream is the chunk's exponent bytes.  Chunks hold 65536 elements (the
 *   last may hold fewer).
 *
 * Conventions.
 *   - Device pointers must be 16-byte aligned; the library never allocates:
 *     the caller owns every buffer.
 *   - Calls are stream ordered and asynchronous, except uzip_query_size,
 *     which synchronises its stream.
 *   - A call keeps all its working state in the buffers it is given (the
 *     compressors' counters and staging in d_out, past the container), so
 *     calls on different streams, from any host threads, may run on the GPU
 *     at the same time as long as they share no buffer.  The one exception
 *     is uzip_compress_noalloc, whose scratch array is shared by all its
 *     calls on a device.
 *   - The return value reports argument and launch errors.  Data-dependent
 *     errors (a corrupt container, a device-side wait that ran out) are
 *     written to device memory (*d_status, *d_out_size = 0) and never trap.
 *   - The input is never modified.
 */
#ifndef UZIP_H
#define UZIP_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* UZIP_FP16 is IEEE binary16; UZIP_FP8_E4M3 and UZIP_FP8_E5M2 are the OCP
 * 8-bit formats float8_e4m3fn and float8_e5m2 (UCCL-Zip Fig. 12 runs its
 * codec on all five). */
typedef enum {
    UZIP_BF16 = 0,
    UZIP_FP32 = 1,
    UZIP_FP16 = 2,
    UZIP_FP8_E4M3 = 3,
    UZIP_FP8_E5M2 = 4
} uzip_dtype;

typedef enum {
    UZIP_OK = 0,
    UZIP_ERR_INVALID_ARG = 1,       /* null or misaligned pointer, n too large */
    UZIP_ERR_UNSUPPORTED_DTYPE = 2, /* dtype is not one of the five uzip_dtype values */
    UZIP_ERR_CAPACITY = 3,          /* output buffer smaller than required */
    UZIP_ERR_CORRUPT = 4,           /* container failed validation */
    UZIP_ERR_TIMEOUT = 5,           /* a bounded device-side wait ran out */
    UZIP_ERR_CUDA = 6,              /* a CUDA runtime call or launch failed */
    UZIP_ERR_TOO_LARGE = 7          /* n above UZIP_NOALLOC_MAX_ELEMS (uzip_compress_noalloc) */
} uzip_status;

/* Largest number of elements one call accepts (2^40). */
#define UZIP_MAX_ELEMS (1ull << 40)

/* Bytes the output buffer of uzip_compress must hold for (dtype, n).  The
 * container itself is a self-describing frame whose header states its size
 * (NCCLZ, arXiv 2605.12396, Sec. IV-B and IV-D2: a frame header carrying the
 * payload byte count ahead of the payload); the buffer also holds the
 * compressor's work area behind the largest frame.  In detail: the
 * largest possible container (every chunk stored RAW, rounded up to 16) plus
 * the compressor's work area behind it: 16 + 8*C bytes of counters and chunk
 * descriptors, 4096 bytes of alignment slack and, for C > 0,
 * min(ceil(C / 4), 160) blocks x 8 encoding warps x 2 slots of 69,632 bytes
 * (each encoding warp uses its two slots in turn, for a chunk's exponent bytes
 * and then for its finished stream while that waits for its offset).  For
 * 2^29 bf16 values (C = 8192) that is 1,073,840,192 + 178,327,568 bytes.  Pure
 * host function;
 * returns 0 for an unsupported dtype or n > UZIP_MAX_ELEMS. */
uint64_t uzip_max_compressed_size(uzip_dtype dtype, uint64_t n);

/* Compress n elements at d_in into the container at d_out.
 *   d_in          device, 16-byte aligned, n * element bytes (2 for bf16
 *                 and fp16, 4 for fp32, 1 for fp8); may be NULL
 *                 when n == 0.
 *   d_out         device, 16-byte aligned, out_capacity bytes; must be at
 *                 least uzip_max_compressed_size(dtype, n) (else
 *                 UZIP_ERR_CAPACITY).  On completion [0, total_bytes) is the
 *                 container; the rest of the buffer is scratch.
 *   d_out_size    device u64 (nullable): receives total_bytes, or 0 if a
 *                 device-side wait ran out.
 *   s             CUDA stream (0 = legacy default stream).
 * Output bytes are a pure function of the input: the same input always gives
 * the same container, equal byte for byte to the reference implementation. */
uzip_status uzip_compress(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out,
                          uint64_t out_capacity, uint64_t* d_out_size, cudaStream_t s);

/* As uzip_compress, plus:
 *   d_status  device i32 (nullable): 0 on success, else a uzip_status
 *             (UZIP_ERR_TIMEOUT when a chunk's offset wait ran out).
 *   flags     0 for normal use.  UZIP_FLAG_SAMPLED_TABLES builds each
 *             chunk's table from a sample of the chunk instead of its full
 *             histogram (UCCL-Zip Fig. 5: every block samples and builds its
 *             own table): the elements at positions 0, 16, 32, ... of the
 *             chunk; a symbol seen s times counts 16 s, every unseen symbol
 *             of the format's exponent range counts 1 (so all stay codable);
 *             the container format is unchanged, the containers are a little
 *             larger.  UZIP_TESTFLAG_SKIP_CHUNK0 makes the chunk counter
 *             start at 1, so chunk 0 never publishes its length and every
 *             wait on it runs out (about a second): it exists only to test
 *             the timeout path; the container is then invalid. */
#define UZIP_TESTFLAG_SKIP_CHUNK0 1u
#define UZIP_FLAG_SAMPLED_TABLES 2u
uzip_status uzip_compress_ex(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out,
                             uint64_t out_capacity, uint64_t* d_out_size, int32_t* d_status,
                             uint32_t flags, cudaStream_t s);

/* Allocation-free compression.  The pages have no counterpart: this entry
 * point serves callers that hold only the user's input and output buffers and
 * must not allocate device memory of their own -- for instance a transport or
 * plugin hook that runs once per message inside someone else's memory plan,
 * where a cudaMalloc could stall the whole device and would take memory the
 * application has budgeted elsewhere.  uzip_compress needs a work area at the
 * tail of its output buffer (counters, chunk descriptors and per-warp slots
 * for exponent bytes and finished streams); this variant keeps the counters
 * and descriptors in the library's own device memory instead -- a fixed array
 * in the library, one per GPU that loads it, kept until the process exits --
 * and does without the slots: each chunk is encoded twice from the input
 * (counting, then writing in place), so it is slower than uzip_compress.
 *
 *   d_in, n, dtype   as uzip_compress; n <= UZIP_NOALLOC_MAX_ELEMS (2^30,
 *                    so the array is 131,088 bytes), else UZIP_ERR_TOO_LARGE.
 *   d_out            device, 16-byte aligned; out_capacity must be at least
 *                    the largest container (every chunk stored RAW):
 *                    round16(round16(64 + 12 C) + P) + (C - 1) * 65536
 *                    + round16(n - (C - 1) * 65536) bytes for C > 0 chunks,
 *                    64 for n = 0, with P the remainder plane's size (n,
 *                    2n, 3n or ceil(n/2) bytes, see above) (else
 *                    UZIP_ERR_CAPACITY).
 *   d_out_size, d_status  as uzip_compress_ex (both nullable).
 * The result is byte for byte the container uzip_compress writes.  The call
 * allocates nothing: it clears the work area with cudaMemsetAsync on s and
 * launches the same kernel.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is kept per device and
 * CUDA context: after a cudaDeviceReset the next call on that device looks it
 * up again (so that call too must come before any capture).  Every call
 * shares the one array, so two calls whose work overlaps on the GPU (different streams, or different
 * host threads without ordering) race and corrupt each other's output: order
 * them on one stream or synchronise between them. */
#define UZIP_NOALLOC_MAX_ELEMS (1ull << 30)
uzip_status uzip_compress_noalloc(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out,
                                  uint64_t out_capacity, uint64_t* d_out_size, int32_t* d_status,
                                  cudaStream_t s);

/* Decompress the container at d_comp into n elements at d_out.
 *   d_comp         device, 16-byte aligned; comp_capacity = readable bytes
 *                  (at least the container's total_bytes).
 *   d_out          device, 16-byte aligned, n * element bytes (1, 2 or 4).
 *   d_status       device i32 (nullable): set to 0, then to UZIP_ERR_CORRUPT
 *                  if any check fails: header fields against (dtype, n),
 *                  chunk offsets and lengths in range, frequency table sums
 *                  to 4096 with every present entry >= 1, word reads stay in
 *                  the stream, every lane ends in state 2^16 having used every
 *                  word (NCCLZ Alg. 2 validates a frame before use).  On
 *                  CORRUPT the contents of d_out are unspecified.
 * Returns UZIP_ERR_CORRUPT at once (without a launch) if comp_capacity < 64. */
uzip_status uzip_decompress(const void* d_comp, uint64_t comp_capacity, void* d_out,
                            uzip_dtype dtype, uint64_t n, int32_t* d_status, cudaStream_t s);

/* Compression with one Gaussian-model table for every chunk (ZipCCL abstract:
 * exponent coding that follows from the Gaussian shape of LLM tensors, with
 * no statistics gathered online), for values ~ N(0, sigma^2):
 *   sigma         finite and > 0 (else UZIP_ERR_INVALID_ARG, nothing
 *                 enqueued), e.g. a weight initialisation's standard
 *                 deviation.  For exponent field e >= 1 of a format with bias
 *                 b the model's probability is erfc(x) - erfc(2x), x =
 *                 2^(e-b) / (sigma sqrt 2) (the binade [2^(e-b), 2^(e-b+1))
 *                 on both sides of zero), for e = 0 it is 1 - erfc(2x); each
 *                 becomes a count out of 65536 (rounded to nearest, at least
 *                 1 for every value of the field) and the counts are
 *                 normalised to 4096 like a chunk's histogram.
 * The helper warps then count nothing: every chunk is coded with that one
 * table, or stored RAW where coding does not shrink it.  Every value stays
 * codable whatever sigma is; a sigma far from the data's only costs size.
 * The container format is unchanged (each coded chunk lists all 2^ebits
 * symbols), so uzip_decompress reads it.  Other arguments and errors as for
 * uzip_compress_ex. */
uzip_status uzip_compress_parametric(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out,
                                     uint64_t out_capacity, uint64_t* d_out_size, int32_t* d_status, double sigma,
                                     cudaStream_t s);

/* Compression with a whole-message choice (NCCLZ Sec. IV-C and Alg. 1: a
 * message whose coding would not pay travels RAW; it samples at most 64 KiB).
 * The container format is the one above; only the choice differs:
 *   - n * element bytes < raw_below_bytes: every chunk is stored RAW (no
 *     statistics or coding; chunk c's RAW stream at offset 65536 c);
 *   - otherwise the first min(n, 65536 / element bytes) elements (64 KiB of
 *     input) are a sample: their exponent bytes are counted, normalised and
 *     coded as one chunk on the device; if that chunk would be stored RAW
 *     under the per-chunk rule, every chunk of the message is stored RAW,
 *     else each chunk is coded or RAW as in uzip_compress.
 * raw_below_bytes = 0 leaves the choice to the sample; UINT64_MAX forces RAW.
 * Arguments, capacity (uzip_max_compressed_size), d_out_size and d_status
 * are as for uzip_compress_ex; the decision never leaves the device. */
uzip_status uzip_compress_gated(const void* d_in, uzip_dtype dtype, uint64_t n, void* d_out,
                                uint64_t out_capacity, uint64_t* d_out_size, int32_t* d_status,
                                uint64_t raw_below_bytes, cudaStream_t s);

/* Read the 64-byte header of the container at d_comp (device) and return
 * its total size, dtype and element count (NCCLZ Sec. IV-B and IV-D2: the
 * receiver learns the payload size and codec from the frame header before it
 * touches the payload).  Synchronises s.  Returns
 * UZIP_ERR_CORRUPT if the magic, version or layout fields do not check out,
 * or total_bytes == 0 (a failed compression). Any output pointer may be NULL. */
uzip_status uzip_query_size(const void* d_comp, uint64_t* h_total_bytes, uzip_dtype* h_dtype,
                            uint64_t* h_n, cudaStream_t s);

/* Static description of a status code. */
const char* uzip_status_string(uzip_status st);

/* ---------------------------------------------------------------------------
 * Split-send pipeline on one GPU (UCCL-Zip Fig. 1 b and Fig. 4 d; NCCLZ
 * Sec. IV-D4 ping-pong staging banks): message k is compressed on s_compress
 * into device bank k % 2 while message k-1's container is copied to the host
 * on s_copy.  The device-to-host copy stands in for the wire.
 *
 *   d_msgs[k], msg_elems[k]  device input of message k (16-byte aligned).
 *   d_bank[2]                device banks, each bank_capacity bytes, at least
 *                            uzip_max_compressed_size of the largest message.
 *                            When every message travels RAW (below the
 *                            threshold), each bank is used as up to 8 slots
 *                            of the largest RAW container (256-byte aligned),
 *                            so up to 16 messages are in flight.
 *   h_bank[2]                pinned host banks (cudaHostAlloc / page-locked),
 *                            h_capacity bytes each; message k's container
 *                            lands in h_bank[k % 2] (a later message reuses
 *                            the bank, as a sender's staging buffer would).
 *                            A message of fewer than
 *                            UZIP_PIPE_RAW_BELOW_DEFAULT input bytes travels
 *                            as a whole-message RAW container (see
 *                            uzip_pipeline_send_ex).
 *   h_sizes                  pinned host u64[n_msgs]: container size of each
 *                            message, written by the device (0 on failure).
 *   mode                     UZIP_PIPE_EXACT: a copy kernel reads the size on
 *                            the device and writes exactly total_bytes into
 *                            the mapped host bank.  UZIP_PIPE_BOUND: one
 *                            cudaMemcpyAsync of the size bound per message.
 *                            UZIP_PIPE_SERIAL: compress then copy on one
 *                            stream, no overlap (the naive design of UCCL-Zip
 *                            Fig. 1 a), for comparison.  UZIP_PIPE_SIZED:
 *                            the host waits for each message's compression
 *                            to finish, reads its size from h_sizes and
 *                            issues one cudaMemcpyAsync of exactly that many
 *                            bytes (the copy engine instead of SM stores; the
 *                            call then blocks until the last compression has
 *                            finished, while the copies still overlap it).  A
 *                            whole-message RAW container's size is the bound,
 *                            known up front, so its copy is issued at once.
 *                            UZIP_PIPE_STREAMED: each message's container
 *                            travels while it is being compressed (UCCL-Zip
 *                            Fig. 4 d, split-send at plane and chunk grain):
 *                            the kernel posts, in mapped memory, when each
 *                            chunk's remainder bytes are written and where
 *                            each chunk's stream ends once placed; the host
 *                            copies finished runs of 64 chunks of either
 *                            with cudaMemcpyAsync as they appear, and the
 *                            header and chunk table when the kernel is done.
 *                            The host banks must then hold round16(container
 *                            bound of the largest message) + 16 bytes per
 *                            chunk of it (the progress words sit after the
 *                            container); the call returns once every copy of
 *                            the last message is enqueued.
 * Returns once all work is enqueued; the work ends when both streams drain.
 * The caller must not reuse the banks until then. */
typedef enum {
    UZIP_PIPE_EXACT = 0,
    UZIP_PIPE_BOUND = 1,
    UZIP_PIPE_SERIAL = 2,
    UZIP_PIPE_SIZED = 3,
    UZIP_PIPE_STREAMED = 4
} uzip_pipe_mode;

uzip_status uzip_pipeline_send(uzip_dtype dtype, const void* const* d_msgs, const uint64_t* msg_elems,
                               uint32_t n_msgs, void* const* d_bank, uint64_t bank_capacity,
                               void* const* h_bank, uint64_t h_capacity, uint64_t* h_sizes,
                               uzip_pipe_mode mode, cudaStream_t s_compress, cudaStream_t s_copy);

/* uzip_pipeline_send sends a message smaller than this many input bytes as a
 * whole-message RAW container (every chunk stored RAW, no statistics or
 * coding; NCCLZ Sec. IV-C: a message whose coding would not pay travels RAW):
 * below it, coding one message takes longer than copying its raw bytes. */
#define UZIP_PIPE_RAW_BELOW_DEFAULT (32ull << 20)

/* The split-send pipeline with every choice explicit:
 *   h_bank[n_hbanks]  n_hbanks >= 2 pinned host banks; message k's container
 *                     lands in h_bank[k % n_hbanks] (with n_hbanks = n_msgs
 *                     every container stays on the host); the device banks
 *                     stay two.
 *   raw_below_bytes   a message of fewer input bytes travels as a
 *                     whole-message RAW container (its streamed mode falls
 *                     back to the sized copy); 0 codes every message.
 * Everything else is as for uzip_pipeline_send, which is this call with
 * n_hbanks = 2 and raw_below_bytes = UZIP_PIPE_RAW_BELOW_DEFAULT. */
uzip_status uzip_pipeline_send_ex(uzip_dtype dtype, const void* const* d_msgs, const uint64_t* msg_elems,
                                  uint32_t n_msgs, void* const* d_bank, uint64_t bank_capacity,
                                  void* const* h_bank, uint32_t n_hbanks, uint64_t h_capacity,
                                  uint64_t* h_sizes, uzip_pipe_mode mode, uint64_t raw_below_bytes,
                                  cudaStream_t s_compress, cudaStream_t s_copy);

#ifdef __cplusplus
}
#endif
#endif /* UZIP_H */
