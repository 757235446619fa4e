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
// Slots: two slots of kSlotBytes per resident warp (at most kStashWarps
// warps), used in turn.  A full chunk's exponent bytes fill the first 64 KiB
// of a slot; its rANS words grow downwards from the slot's end, so the 4 KiB
// beyond the exponent bytes keep the first words clear of bytes not yet read.
// The finished stream then waits at the slot's end for its offset while the
// warp counts its next chunk in the other slot.  Slots are never read before
// they are written.
constexpr uint64_t kStashWarps = 1536;
constexpr uint32_t kSlotBytes = 65536 + 4096;
__host__ __device__ inline uint64_t stash_warps(uint64_t n) {
    const uint64_t c = num_chunks(n);
    return c < kStashWarps ? c : kStashWarps;
}
// The slots start at the first 256-byte aligned address (absolute) after the
// descriptors; 256 bytes of slack cover the alignment.
__host__ __device__ inline uint64_t work_area_bytes(uint64_t n) {
    return scratch_bytes(n) + 256 + stash_warps(n) * 2 * uint64_t(kSlotBytes);
}

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

// SM count and resident blocks per SM of `kern` on the current device, looked
// up once per (device, kernel, block shape) and cached (api.cu).
cudaError_t launch_shape(const void* kern, int threads, size_t smem, int* sms, int* per_sm);

// launchers (compress.cu, decompress.cu, pipeline.cu)
// mode: 0 per-chunk choice, 1 whole message RAW, 2 gated (a one-warp kernel
// decides from the first 64 KiB of input), 3 per-chunk choice with sampled
// tables
// progress (nullable, mapped host memory, 2 u64 per chunk): see CompressArgs
cudaError_t launch_compress(int dtype, const void* d_in, uint64_t n, void* d_out, uint64_t* d_out_size,
                            int32_t* d_status, uint32_t first_ticket, cudaStream_t s, int mode = 0,
                            uint64_t* progress = nullptr);
cudaError_t launch_compress_with_scratch(int dtype, const void* d_in, uint64_t n, void* d_out, uint64_t* d_out_size,
                                         int32_t* d_status, uint32_t first_ticket, void* scratch_area, void* stash,
                                         cudaStream_t s, int mode = 0, uint64_t* progress = nullptr);

// allocation-free compression: largest tensor and device count served by the
// library's own work area
constexpr uint64_t kNoAllocMaxElems = 1ull << 30;
constexpr uint32_t kNoAllocMaxDevices = 64;
cudaError_t noalloc_scratch_address(void** ptr);
cudaError_t launch_decompress(int dtype, const void* d_comp, uint64_t cap, void* d_out, uint64_t n, int32_t* d_status,
                              cudaStream_t s);
cudaError_t launch_copy_exact(const void* d_container, void* h_dst_mapped, cudaStream_t s);

}  // namespace uzip
