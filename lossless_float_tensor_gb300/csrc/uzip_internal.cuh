// Internal definitions shared by the uzip CUDA sources: container layout,
// launch constants and small inline-PTX helpers.  Nothing here is exported.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/uzip.h"

namespace uzip {

// ---- container format (see include/uzip.h) --------------------------------
constexpr uint32_t kChunk = 65536;        // elements per chunk
constexpr uint32_t kLanes = 32;           // interleaved rANS states
constexpr uint32_t kSteps = kChunk / kLanes;
constexpr uint32_t kProbBits = 12;
constexpr uint32_t kM = 1u << kProbBits;  // frequency total 4096
constexpr uint32_t kRansL = 1u << 16;     // state interval [2^16, 2^32)
constexpr uint32_t kHeader = 64;
constexpr uint32_t kRawFlag = 0x80000000u;
constexpr uint32_t kStreamHead = 160;     // 32 states + 32-byte bitmap

__host__ __device__ inline uint64_t round16(uint64_t v) { return (v + 15) & ~uint64_t(15); }
__host__ __device__ inline bool valid_dtype(int d) { return d >= UZIP_BF16 && d <= UZIP_FP8_E5M2; }
__host__ __device__ inline uint32_t elem_bytes(int dtype) {
    return dtype == UZIP_FP32 ? 4u : (dtype == UZIP_BF16 || dtype == UZIP_FP16) ? 2u : 1u;
}
// width of an element's sign|fraction field: 8 (bf16), 24 (fp32), 11 (fp16),
// 4 (fp8 e4m3fn), 3 (fp8 e5m2)
__host__ __device__ inline uint32_t rem_bits(int dtype) {
    switch (dtype) {
        case UZIP_BF16: return 8;
        case UZIP_FP32: return 24;
        case UZIP_FP16: return 11;
        case UZIP_FP8_E4M3: return 4;
        default: return 3;
    }
}
// remainder plane bytes of n elements: the fields packed least significant
// bit first
__host__ __device__ inline uint64_t rem_plane_bytes(int dtype, uint64_t n) { return (n * rem_bits(dtype) + 7) / 8; }
__host__ __device__ inline uint64_t num_chunks(uint64_t n) { return (n + kChunk - 1) / kChunk; }
__host__ __device__ inline uint64_t rem_offset(uint64_t n) { return round16(kHeader + 12 * num_chunks(n)); }
__host__ __device__ inline uint64_t exp_offset(int dtype, uint64_t n) {
    return round16(rem_offset(n) + rem_plane_bytes(dtype, n));
}

// Element format: bytes per element, exponent and fraction bit widths, the
// remainder field width (sign + fraction) and a full chunk's share of the
// remainder plane in bytes.
template <int DT>
struct Fmt;
template <int ES, int EB, int MB>
struct FmtOf {
    static constexpr uint32_t kEs = ES, kEbits = EB, kMbits = MB, kRbits = MB + 1;
    static constexpr uint32_t kRemChunk = kChunk / 8 * kRbits;
    // formats whose fields are not whole bytes: packed 32 elements at a time
    static constexpr bool kPacked = (kRbits % 8) != 0;
};
template <>
struct Fmt<UZIP_BF16> : FmtOf<2, 8, 7> {};
template <>
struct Fmt<UZIP_FP32> : FmtOf<4, 8, 23> {};
template <>
struct Fmt<UZIP_FP16> : FmtOf<2, 5, 10> {};
template <>
struct Fmt<UZIP_FP8_E4M3> : FmtOf<1, 4, 3> {};
template <>
struct Fmt<UZIP_FP8_E5M2> : FmtOf<1, 5, 2> {};
// Largest container: every chunk stored RAW (round16 of each chunk length).
__host__ __device__ inline uint64_t container_bound(int dtype, uint64_t n) {
    uint64_t c = num_chunks(n);
    uint64_t body = 0;
    if (c > 0) body = (c - 1) * uint64_t(kChunk) + round16(n - (c - 1) * uint64_t(kChunk));
    return exp_offset(dtype, n) + body;
}

// ---- compressor work area, placed at round16(container_bound) in d_out ----
struct Scratch {
    uint32_t status;      // 0 or a uzip_status set by the first failing chunk
    uint32_t ticket;      // next chunk to take
    uint32_t done;        // chunks finished
    uint32_t pad;
    // followed by uint64_t desc[C]: decoupled look-back descriptors
};
constexpr uint64_t kScratchHead = 16;
__host__ __device__ inline uint64_t scratch_offset(int dtype, uint64_t n) { return round16(container_bound(dtype, n)); }
// status, ticket, done counter and look-back descriptors (zeroed before each launch)
__host__ __device__ inline uint64_t scratch_bytes(uint64_t n) { return kScratchHead + 8 * num_chunks(n); }
// Slot area, at the first 4 KiB-aligned address (absolute) after the
// descriptors (4 KiB of slack cover the alignment), in slots of kSlotBytes: a
// chunk's exponent bytes fill the first 64 KiB of a slot and its rANS words
// grow down from the slot's end over exponent bytes already read (the 4 KiB
// beyond the exponent bytes keep the first words clear of bytes not yet
// read); the finished record waits there for its offset.  The
// warp-specialised compressor gives each of its kWsEnc encoders per block two
// slots (contexts), used in turn; the one-warp compressor (sampled tables)
// gives each warp two.  Slots are never read before they are written.
constexpr uint32_t kWsEnc = 8;                   // encoder warps per block of the warp-specialised compressor
constexpr uint32_t kWsFirst = kWsEnc / 2;        // chunks a block starts on at once: one per helper warp
constexpr uint64_t kWsMaxCtas = 160;             // blocks the slot area is sized for
constexpr uint32_t kSlotBytes = 65536 + 4096;
// Blocks of the warp-specialised compressor for n values: one per kWsFirst
// chunks (a helper splits its two encoders' first chunks one after the
// other, so a small tensor spread over more blocks starts every chunk at
// once), at most kWsMaxCtas.
__host__ __device__ inline uint64_t ws_ctas(uint64_t n) {
    const uint64_t c = (num_chunks(n) + kWsFirst - 1) / kWsFirst;
    return c < kWsMaxCtas ? c : kWsMaxCtas;
}
__host__ __device__ inline uint64_t slot_area_bytes(uint64_t n) { return ws_ctas(n) * kWsEnc * 2 * uint64_t(kSlotBytes); }
// one-warp compressor: warps whose two slots fit the area
__host__ __device__ inline uint64_t stash_warps(uint64_t n) { return slot_area_bytes(n) / (2 * uint64_t(kSlotBytes)); }
__host__ __device__ inline uint64_t work_area_bytes(uint64_t n) { return scratch_bytes(n) + 4096 + slot_area_bytes(n); }

// look-back descriptor: flag in bits 62..63, byte count in bits 0..61
constexpr uint64_t kDescAggregate = 1ull << 62;
constexpr uint64_t kDescInclusive = 2ull << 62;
constexpr uint64_t kDescValue = (1ull << 62) - 1;

// ---- compressor shared-memory plan (one warp per CTA) ---------------------
// region A (16 KiB): lane-private histogram u32[256][16], then the encode
//                    table (4 KiB: {m, add} rows at 0, {bound, packed} at 2 KiB)
// region B (2 KiB) : frequencies, sort keys, bitmap, present-symbol list.
constexpr uint32_t kRegionA = 16384;
constexpr uint32_t kEncTable = 4096;
constexpr uint32_t kRegionB = 2048;
constexpr uint32_t kCompressSmem = kRegionA + kRegionB;

// spin limit of a look-back wait: iterations with a growing back-off (about a
// second of waiting in total)
constexpr uint32_t kSpinLimit = 1u << 20;

// ---- decompressor shared-memory plan (per warp) ---------------------------
constexpr uint32_t kDecWarps = 1;
constexpr uint32_t kDecSlotTable = 4096;    // slot -> symbol, u8[4096]
constexpr uint32_t kDecSymTable = 2048;     // symbol -> {f - 4096, -cum}, u32 pairs[256]
constexpr uint32_t kDecList = 1024;         // present symbols, u32[256]: cum << 8 | symbol
constexpr uint32_t kDecWarpSmem = kDecSlotTable + kDecSymTable + kDecList;

// ---- inline PTX helpers ----------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_v4_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_u16_hint(const void* p, uint64_t pol) {
    unsigned short v;
    asm volatile("ld.global.nc.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_u32_hint(const void* p, uint64_t pol) {
    uint32_t v;
    asm volatile("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_v2_hint(void* p, uint32_t a, uint32_t b, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;" ::"l"(p), "r"(a), "r"(b), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_v4_hint(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_u32_hint(void* p, uint32_t a, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(a), "l"(pol) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---- asynchronous copies and barriers (inline PTX) --------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// bulk copy global -> shared, completing `bytes` of transaction on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// bulk copy shared -> global, tracked by bulk groups
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void l2_discard_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Exact floor(x / f) for x in [16 f, f * 2^20) as (x * m + add) >> (32 + sh)
// (Robison, "N-bit unsigned division via N-bit multiply-add", ARITH 2005).
// With p = max(32, 31 + ceil(log2 f)) the reciprocal fits 32 bits; either the
// round-up reciprocal (add = 0) or the round-down reciprocal with increment
// (add = m) is exact over the whole range.  Exactness reduces to the worst
// points x = k f - 1 (round-up: (f 2^20 - 1) e < 2^p, e = m f - 2^p) and
// x = k f (round-down: ((2^20 - 1) f + 1) d <= 2^p, d = 2^p - m f); one of the
// two holds for every f in [1, 4096] (checked exhaustively by the tests
// through uzip_debug_div_magic).
struct DivMagic {
    uint32_t m, add, sh, ok;
};
__host__ __device__ constexpr inline DivMagic div_magic(uint32_t f) {
    DivMagic r{0u, 0u, 0u, 0u};
    if (f == 0 || f > kM) return r;
    uint32_t lg = 0;
    while ((1u << lg) < f) ++lg;  // ceil(log2 f)
    const uint32_t p = lg + 31 < 32 ? 32 : lg + 31;
    const uint64_t two_p = 1ull << p;
    const uint64_t md = (two_p - 1) / f;  // floor((2^p - 1) / f)
    const uint64_t mu = md + 1;           // ceil(2^p / f)
    const uint64_t xmax = (uint64_t(f) << 20) - 1;
    r.sh = p - 32;
    if (mu < (1ull << 32)) {
        const uint64_t e = mu * f - two_p;
        if (xmax * e < two_p) {
            r.m = uint32_t(mu);
            r.add = 0;
            r.ok = 1;
            return r;
        }
    }
    const uint64_t d = two_p - md * f;
    if (md < (1ull << 32) && (((1ull << 20) - 1) * f + 1) * d <= two_p) {
        r.m = uint32_t(md);
        r.add = uint32_t(md);
        r.ok = 1;
    }
    return r;
}

// div_magic of every f in [1, 4096], evaluated at compile time: {m, sh |
// (add != 0) << 8} (add is 0 or m)
struct MagicEntry {
    uint32_t m, add_sh;
};
struct MagicTable {
    MagicEntry e[kM + 1];
};
constexpr MagicTable make_magic_table() {
    MagicTable t{};
    for (uint32_t f = 1; f <= kM; ++f) {
        const DivMagic d = div_magic(f);
        t.e[f] = MagicEntry{d.m, d.sh | (d.add ? 256u : 0u)};
    }
    return t;
}

// Exact floor(x / f) for x in [0, f * 2^20) with a 33-bit reciprocal:
// sh = ceil(log2 f) and m = ceil(2^(32 + sh) / f), which lies in [2^32, 2^33),
// so m = 2^32 + m_lo and x m = x m_lo + x 2^32 is one 32 x 32 -> 64-bit
// multiply-add.  With e = m f - 2^(32 + sh) < f, the error term x e / (f 2^(32
// + sh)) stays below 1/f as long as x e < 2^(32 + sh); x < f 2^20 and
// e < f <= 2^sh give x e < 2^(2 sh + 20) <= 2^(32 + sh) for sh <= 12, so
// floor(x m / 2^(32 + sh)) = floor(x / f) for every f in [1, 4096] (Granlund
// and Montgomery, "Division by invariant integers using multiplication",
// PLDI 1994, with the extra multiplier bit folded into the addend).  The
// product also stays below 2^64: x m < 2^(52 + sh) + f 2^20 <= 2^64.
struct Magic33 {
    uint32_t m_lo, sh;
};
__host__ __device__ constexpr inline Magic33 magic33(uint32_t f) {
    Magic33 r{0u, 0u};
    if (f == 0 || f > kM) return r;
    uint32_t sh = 0;
    while ((1u << sh) < f) ++sh;
    const uint64_t two = 1ull << (32 + sh);
    const uint64_t m = (two + f - 1) / f;
    r.m_lo = uint32_t(m - (1ull << 32));
    r.sh = sh;
    return r;
}
struct Magic33Table {
    Magic33 e[kM + 1];
};
constexpr Magic33Table make_magic33_table() {
    Magic33Table t{};
    for (uint32_t f = 1; f <= kM; ++f) t.e[f] = magic33(f);
    return t;
}

// SM count and resident blocks per SM of `kern` on the current device, looked
// up once per (device, kernel, block shape) and cached (api.cu).
cudaError_t launch_shape(const void* kern, int threads, size_t smem, int* sms, int* per_sm);

// launchers (compress.cu, decompress.cu, pipeline.cu)
// mode: 0 per-chunk choice, 1 whole message RAW, 2 gated (a one-warp kernel
// decides from the first 64 KiB of input), 3 per-chunk choice with sampled
// tables, 4 per-chunk choice with the one table of the model counts `model`
// (256 u32, see model_counts)
// progress (nullable, mapped host memory, 2 u64 per chunk): see CompressArgs
cudaError_t launch_compress(int dtype, const void* d_in, uint64_t n, void* d_out, uint64_t* d_out_size,
                            int32_t* d_status, uint32_t first_ticket, cudaStream_t s, int mode = 0,
                            uint64_t* progress = nullptr, const uint32_t* model = nullptr);
cudaError_t launch_compress_with_scratch(int dtype, const void* d_in, uint64_t n, void* d_out, uint64_t* d_out_size,
                                         int32_t* d_status, uint32_t first_ticket, void* scratch_area, void* stash,
                                         cudaStream_t s, int mode = 0, uint64_t* progress = nullptr,
                                         const uint32_t* model = nullptr);
// Gaussian-model counts (mode 4) for values ~ N(0, sigma^2) (compress.cu);
// false for a sigma that is not finite and positive
bool model_counts(int dtype, double sigma, uint32_t counts[256]);

// warp-specialised compressor: blocks of its encoder's current chunk left when
// a helper starts splitting the next one (compress.cu; a test hook sets it)
extern uint32_t g_ws_jit_blocks;

// allocation-free compression: largest tensor and device count served by the
// library's own work area
constexpr uint64_t kNoAllocMaxElems = 1ull << 30;
constexpr uint32_t kNoAllocMaxDevices = 64;
cudaError_t noalloc_scratch_address(void** ptr);
cudaError_t launch_decompress(int dtype, const void* d_comp, uint64_t cap, void* d_out, uint64_t n, int32_t* d_status,
                              cudaStream_t s);
cudaError_t launch_copy_exact(const void* d_container, void* h_dst_mapped, cudaStream_t s);

}  // namespace uzip
