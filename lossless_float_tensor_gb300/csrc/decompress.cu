// Decompressor: one warp per chunk, chunks strided over a persistent grid.
// Per chunk the warp validates the chunk-table entry and the stream head,
// builds the 4096-slot symbol table in shared memory, runs the 32 interleaved
// rANS decoders forward, and merges each decoded exponent byte with its
// sign|fraction bits from the remainder plane into the output value (the
// receive side of UCCL-Zip's split-send and of NCCLZ Alg. 2, which validates a
// frame before using it).
#include "uzip_internal.cuh"

namespace uzip {

struct DecompressArgs {
    const uint8_t* comp;
    uint64_t cap;
    uint8_t* out;
    uint64_t n;
    int32_t* status;  // nullable
};

__device__ __forceinline__ void flag_corrupt(int32_t* status) {
    if (status) atomicCAS(reinterpret_cast<int*>(status), 0, int(UZIP_ERR_CORRUPT));
}

__device__ __forceinline__ uint32_t warp_excl_scan_d(uint32_t v, uint32_t lane, uint32_t* total) {
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= uint32_t(o)) inc += t;
    }
    *total = __shfl_sync(0xFFFFFFFFu, inc, 31);
    return inc - v;
}

// element bits from exponent field e and sign|fraction field r
template <int DT>
__device__ __forceinline__ uint32_t merge_bits(uint32_t e, uint32_t r) {
    constexpr uint32_t mb = Fmt<DT>::kMbits, top = 8 * Fmt<DT>::kEs - 1;
    return ((r >> mb) << top) | (e << mb) | (r & ((1u << mb) - 1u));
}
// The same merge for the decode loop, with fewer logic-unit instructions: for
// bf16, r * 257 puts the remainder byte at bits 0..7 and again at 8..15, so
// one mask keeps the fraction (bits 0..6) and the sign (bit 15).
template <int DT>
__device__ __forceinline__ uint32_t merge_fast(uint32_t e, uint32_t r) {
    if (DT == UZIP_BF16) return ((r * 257u) & 0x807Fu) | (e << 7);
    if (DT == UZIP_FP32) return ((r & 0x7FFFFFu) | (e << 23)) | ((r << 8) & 0x80000000u);
    return merge_bits<DT>(e, r);
}
// sign|fraction field of element i of a chunk's remainder plane (W-bit
// fields packed least significant bit first; only the bytes holding the
// field are read)
template <int DT>
__device__ __forceinline__ uint32_t rem_field(const uint8_t* __restrict__ rem, uint32_t i) {
    if constexpr (DT == UZIP_BF16) return __ldg(rem + i);
    if constexpr (DT == UZIP_FP32)
        return uint32_t(__ldg(rem + 3 * i)) | uint32_t(__ldg(rem + 3 * i + 1)) << 8 | uint32_t(__ldg(rem + 3 * i + 2)) << 16;
    constexpr uint32_t W = Fmt<DT>::kRbits;
    const uint32_t bit = W * i, b0 = bit >> 3, sh = bit & 7;
    uint32_t v = __ldg(rem + b0);
    if (sh + W > 8) v |= uint32_t(__ldg(rem + b0 + 1)) << 8;
    if (sh + W > 16) v |= uint32_t(__ldg(rem + b0 + 2)) << 16;
    return (v >> sh) & ((1u << W) - 1u);
}

// RAW chunk of a byte-field format (bf16, fp32): 16 values per lane at a time
template <int DT>
__device__ void merge_raw_bytes(const uint8_t* __restrict__ ex, const uint8_t* __restrict__ rem, uint8_t* __restrict__ out,
                          uint32_t n_c, uint32_t lane) {
    constexpr uint32_t rb = DT == UZIP_BF16 ? 1 : 3;
    constexpr uint32_t es = DT == UZIP_BF16 ? 2 : 4;
    const uint32_t nfull = n_c / 16;
    for (uint32_t b = lane; b < nfull; b += 32) {
        const uint4 eq = *reinterpret_cast<const uint4*>(ex + 16 * uint64_t(b));
        const uint32_t ew[4] = {eq.x, eq.y, eq.z, eq.w};
        uint32_t rw[12];
        if (DT == UZIP_BF16) {
            const uint4 rq = *reinterpret_cast<const uint4*>(rem + 16 * uint64_t(b));
            rw[0] = rq.x, rw[1] = rq.y, rw[2] = rq.z, rw[3] = rq.w;
        } else {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const uint4 rq = *reinterpret_cast<const uint4*>(rem + 48 * uint64_t(b) + 16 * j);
                rw[4 * j] = rq.x, rw[4 * j + 1] = rq.y, rw[4 * j + 2] = rq.z, rw[4 * j + 3] = rq.w;
            }
        }
        uint32_t o[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t e = (ew[k >> 2] >> (8 * (k & 3))) & 0xFFu;
            uint32_t r;
            if (DT == UZIP_BF16) {
                r = (rw[k >> 2] >> (8 * (k & 3))) & 0xFFu;
            } else {
                const uint32_t byte0 = 3 * k;
                r = 0;
#pragma unroll
                for (int q = 0; q < 3; ++q) r |= ((rw[(byte0 + q) >> 2] >> (8 * ((byte0 + q) & 3))) & 0xFFu) << (8 * q);
            }
            o[k] = merge_bits<DT>(e, r);
        }
        if (DT == UZIP_BF16) {
            uint4* d = reinterpret_cast<uint4*>(out + 32 * uint64_t(b));
            d[0] = make_uint4(o[0] | o[1] << 16, o[2] | o[3] << 16, o[4] | o[5] << 16, o[6] | o[7] << 16);
            d[1] = make_uint4(o[8] | o[9] << 16, o[10] | o[11] << 16, o[12] | o[13] << 16, o[14] | o[15] << 16);
        } else {
            uint4* d = reinterpret_cast<uint4*>(out + 64 * uint64_t(b));
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        }
    }
    for (uint32_t i = nfull * 16 + lane; i < n_c; i += 32) {
        uint32_t r = rem[rb * uint64_t(i)];
        if (DT == UZIP_FP32) r |= uint32_t(rem[3 * uint64_t(i) + 1]) << 8 | uint32_t(rem[3 * uint64_t(i) + 2]) << 16;
        const uint32_t v = merge_bits<DT>(ex[i], r);
        if (es == 2) reinterpret_cast<uint16_t*>(out)[i] = uint16_t(v);
        else reinterpret_cast<uint32_t*>(out)[i] = v;
    }
}

// RAW chunk of a packed-field format (fp16, fp8): element by element
template <int DT>
__device__ void merge_raw_packed(const uint8_t* __restrict__ ex, const uint8_t* __restrict__ rem,
                                 uint8_t* __restrict__ out, uint32_t n_c, uint32_t lane) {
    constexpr uint32_t es = Fmt<DT>::kEs;
    for (uint32_t i = lane; i < n_c; i += 32) {
        const uint32_t v = merge_bits<DT>(ex[i], rem_field<DT>(rem, i));
        if (es == 2) reinterpret_cast<uint16_t*>(out)[i] = uint16_t(v);
        else out[i] = uint8_t(v);
    }
}

// Coded chunk.  Returns false if the stream is invalid.  RING: the caller has
// checked that the stream padded to 16 bytes lies inside the readable buffer,
// so full chunks may stage the word stream through shared memory in 16-byte
// lines; otherwise every word window is read from global memory.
template <int DT, bool RING>
__device__ bool decode_coded(const uint8_t* __restrict__ src, uint32_t len, const uint8_t* __restrict__ rem,
                             uint8_t* __restrict__ out, uint32_t n_c, uint32_t lane, uint8_t* wsm) {
    constexpr uint32_t es = Fmt<DT>::kEs;
    uint8_t* slot_sym = wsm;                                                   // u8[4096]
    uint2* sym_gc = reinterpret_cast<uint2*>(wsm + kDecSlotTable);                  // {f - 4096, -cum}
    uint32_t* plist = reinterpret_cast<uint32_t*>(wsm + kDecSlotTable + kDecSymTable); // u32[256]: cum << 8 | s
    if (len < kStreamHead) return false;
    uint32_t x = reinterpret_cast<const uint32_t*>(src)[lane];
    const uint32_t bm = src[128 + lane];  // present symbols 8*lane .. 8*lane+7
    uint32_t k_total;
    const uint32_t prefix = warp_excl_scan_d(__popc(bm), lane, &k_total);
    if (len < kStreamHead + 2 * k_total || ((len - kStreamHead - 2 * k_total) & 1u)) return false;
    const uint32_t W = (len - kStreamHead - 2 * k_total) / 2;
    uint32_t f[8];
    uint32_t lsum = 0;
    bool bad = x < kRansL;
    {
        uint32_t idx = prefix;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            f[k] = 0;
            if (bm & (1u << k)) {
                f[k] = reinterpret_cast<const uint16_t*>(src + kStreamHead)[idx++];
                if (f[k] == 0 || f[k] > kM) bad = true;
            }
            lsum += f[k];
        }
    }
    uint32_t fsum;
    uint32_t cum = warp_excl_scan_d(lsum, lane, &fsum);
    if (__any_sync(0xFFFFFFFFu, bad) || fsum != kM) return false;
    {
        uint32_t idx = prefix;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (bm & (1u << k)) {
                sym_gc[8 * lane + k] = make_uint2(f[k] - kM, 0u - cum);
                plist[idx++] = (cum << 8) | (8 * lane + k);
            }
            cum += f[k];
        }
    }
    __syncwarp();
    // slot table in 16-slot pieces: lane l fills slots [512 g + 16 l, +16)
    // for g = 0..7, so each 16-byte store of the warp covers 512 contiguous
    // bytes (a lane filling one contiguous quarter-kilobyte would put all 32
    // lanes' stores in one bank).  Each piece's first symbol comes from a
    // branchless binary search over the sorted list (the eight searches are
    // independent, so their loads overlap), then the piece walks forward.
    {
        const uint32_t first = 16 * lane;
        uint32_t jg[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) jg[g] = 0;  // cum_0 = 0 <= every slot
#pragma unroll
        for (uint32_t step = 128; step > 0; step >>= 1) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint32_t t = jg[g] + step;
                if (t < k_total && (plist[t] >> 8) <= 512 * uint32_t(g) + first) jg[g] = t;
            }
        }
        const uint32_t slot_base = static_cast<uint32_t>(__cvta_generic_to_shared(slot_sym));
#pragma unroll 1
        for (uint32_t g = 0; g < 8; ++g) {
            const uint32_t p0 = 512 * g + first;
            uint32_t j = jg[0];
#pragma unroll
            for (int k = 1; k < 8; ++k) j = g == uint32_t(k) ? jg[k] : j;
            uint32_t cur = plist[j] & 0xFFu;
            uint32_t next_cum = j + 1 < k_total ? (plist[j + 1] >> 8) : kM;
            uint32_t wq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t i0 = p0 + 4 * q;
                uint32_t word;
                if (next_cum > i0 + 3) {
                    word = cur * 0x01010101u;
                } else {
                    word = 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        while (next_cum <= i0 + b) {
                            ++j;
                            cur = plist[j] & 0xFFu;
                            next_cum = j + 1 < k_total ? (plist[j + 1] >> 8) : kM;
                        }
                        word |= cur << (8 * b);
                    }
                }
                wq[q] = word;
            }
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(slot_base + p0), "r"(wq[0]), "r"(wq[1]),
                         "r"(wq[2]), "r"(wq[3])
                         : "memory");
        }
    }
    __syncwarp();

    // W == 0: any word request is an error, caught by the final pos == W
    // test; point the (never needed) reads at the stream head, which is
    // always inside the container.
    const uint16_t* words =
        W ? reinterpret_cast<const uint16_t*>(src + kStreamHead + 2 * k_total) : reinterpret_cast<const uint16_t*>(src);
    const uint32_t wlast = W ? W - 1 : 0;
    const uint32_t lt = lanemask_lt();
    const uint32_t slot_s = static_cast<uint32_t>(__cvta_generic_to_shared(slot_sym));
    const uint32_t gc_s = static_cast<uint32_t>(__cvta_generic_to_shared(sym_gc));
    uint32_t pos = 0;
    // One decode step (rule R6, read side).  At most 32 words are consumed
    // per step, so every lane first fetches the word at pos + lane (pos is
    // known from the previous step, so the fetch is off the state's dependency
    // chain) and a lane that renormalises takes its word from lane
    // popc(ballot & lanes below) with one shuffle.  Reads past the stream
    // return some other word and leave pos > W, which fails the check after
    // the loop.  The state update f (x >> 12) + (x mod 4096) - cum is computed
    // as (x >> 12)(f - 4096) + x - cum (exact modulo 2^32, and the result is
    // below 2^32), so one table entry {f - 4096, -cum} feeds it directly.
    // `cur` advances by scale words per consumed word.  This form serves
    // partial chunks and streams read from global memory; full chunks staged
    // in the shared-memory ring take rstep below, which saves the shuffle.
    auto step = [&](uint32_t t, uint32_t r, bool active, uint32_t win, uint32_t& cur, uint32_t scale) {
        const uint32_t slot = x & (kM - 1);
        uint32_t s, g, nc;
        asm("ld.shared.u8 %0, [%1];" : "=r"(s) : "r"(slot_s + slot));
        asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(g), "=r"(nc) : "r"(gc_s + 8 * s));
        const uint32_t xn = (x >> kProbBits) * g + x + nc;
        const bool need = active && xn < kRansL;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, need);
        const uint32_t w = __shfl_sync(0xFFFFFFFFu, win, __popc(b & lt));
        cur += scale * __popc(b);
        if (active) {
            x = need ? ((xn << 16) | w) : xn;
            const uint32_t v = merge_fast<DT>(s, r);
            const uint64_t i = 32 * uint64_t(t) + lane;
            if (es == 2) reinterpret_cast<uint16_t*>(out)[i] = uint16_t(v);
            else if (es == 4) reinterpret_cast<uint32_t*>(out)[i] = v;
            else out[i] = uint8_t(v);
        }
    };
    auto gwin = [&]() -> uint32_t {
        const uint32_t widx = pos + lane;
        return __ldg(words + (widx < wlast ? widx : wlast));
    };
    // A step's 32 fields are RB consecutive words (RB = field bits); this
    // lane's field starts at bit RB lane of them and may run into the next
    // word.
    constexpr uint32_t RB = Fmt<DT>::kRbits;
    const uint32_t lword = (RB * lane) >> 5, lsh = (RB * lane) & 31;
    const bool lstraddle = lsh + RB > 32;
    auto load_rem_full = [&](uint32_t t) -> uint32_t {  // t < 2048 of a full chunk
        if constexpr (DT == UZIP_BF16) {
            return rem_field<DT>(rem, 32 * t + lane);
        } else {  // two word loads at most and a funnel shift (fp32's 3-byte fields too)
            const uint32_t* p = reinterpret_cast<const uint32_t*>(rem) + RB * t + lword;
            const uint32_t lo = __ldg(p);
            const uint32_t hi = lstraddle ? __ldg(p + 1) : 0u;
            return __funnelshift_r(lo, hi, lsh) & ((1u << RB) - 1u);
        }
    };
    auto load_rem = [&](uint32_t t) -> uint32_t {
        const uint32_t i = 32 * t + lane;
        if (i >= n_c) return 0;
        return load_rem_full(t);
    };
    if (n_c == kChunk && RING) {
        // Word stream staged in a 1 KiB ring (the present-symbol list is no
        // longer needed): four 256-byte pieces of the stream record, piece p in
        // slot p % 4.  Every 8 steps the ring is topped up so that it holds the
        // worst case of the next 8 steps (8 * 32 words = 512 bytes) past pos;
        // the piece after that is loaded into registers one period early and
        // stored at the next top-up.
        const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(plist));
        const uint32_t wb0 = kStreamHead + 2 * k_total;  // byte offset of word 0 in the record
        const uint32_t nlines = (len + 15) / 16;
        const uint32_t npieces = (nlines + 15) / 16;
        const bool half = lane < 16;                      // a piece is 16 lines: lanes 0..15
        // steps between top-ups: their worst case plus a partly read piece and
        // the piece in flight fill the four slots exactly
        constexpr int kPeriod = 8;
        static_assert(2 * kPeriod * kLanes + 2 * 256 <= 1024, "the ring holds one period past pos");
        auto load_piece = [&](uint32_t piece) -> uint4 {
            const uint32_t line = piece * 16 + (lane & 15);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (half && line < nlines) v = __ldg(reinterpret_cast<const uint4*>(src) + line);
            return v;
        };
        auto store_piece = [&](uint32_t piece, uint4 v) {
            if (half)
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(ring_s + (piece & 3) * 256 + 16 * lane),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
        };
        uint32_t next_piece = 0;  // first piece not yet in the ring or in flight
        uint4 pend = make_uint4(0, 0, 0, 0);
        uint32_t pend_piece = 0;
        bool has_pend = false;
        uint32_t rq = wb0;  // byte offset in the record of word pos (the same in every lane)
        auto top_up = [&]() {
            if (has_pend) store_piece(pend_piece, pend);
            has_pend = false;
            pos = (rq - wb0) >> 1;
            const uint32_t cur = (wb0 + 2 * pos) >> 8;
            uint32_t need_end = ((wb0 + 2 * (pos + kPeriod * kLanes)) >> 8) + 1;
            need_end = need_end < npieces ? need_end : npieces;
            while (next_piece < need_end) {  // behind: bring pieces in now
                store_piece(next_piece, load_piece(next_piece));
                ++next_piece;
            }
            __syncwarp();
            if (next_piece < npieces && next_piece < cur + 4) {
                pend = load_piece(next_piece);
                pend_piece = next_piece;
                has_pend = true;
                ++next_piece;
            }
        };
        // A ring step: a renormalising lane reads its word straight from the
        // ring, at pos plus its rank among the renormalising lanes (one
        // shared load on the state's chain instead of a window load plus a
        // shuffle; the ring holds words pos .. pos + 31 at every step).
        auto rstep = [&](uint32_t t, uint32_t r) {
            const uint32_t slot = x & (kM - 1);
            uint32_t s, g, nc;
            asm("ld.shared.u8 %0, [%1];" : "=r"(s) : "r"(slot_s + slot));
            asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(g), "=r"(nc) : "r"(gc_s + 8 * s));
            const uint32_t xn = (x >> kProbBits) * g + x + nc;
            const bool need = xn < kRansL;
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, need);
            uint32_t w;
            asm volatile("ld.shared.u16 %0, [%1];" : "=r"(w) : "r"(ring_s + ((rq + 2 * __popc(b & lt)) & 1023u)) : "memory");
            rq += 2 * __popc(b);
            x = need ? ((xn << 16) | w) : xn;
            const uint32_t v = merge_fast<DT>(s, r);
            const uint64_t i = 32 * uint64_t(t) + lane;
            if (es == 2) reinterpret_cast<uint16_t*>(out)[i] = uint16_t(v);
            else if (es == 4) reinterpret_cast<uint32_t*>(out)[i] = v;
            else out[i] = uint8_t(v);
        };
        // Both streams are cold in L2 when decompression starts: pull the
        // remainder bytes of the steps 64 ahead and the stream bytes ~1 KiB
        // past the read position into L2 (one instruction each per 16 steps).
        constexpr uint32_t kRemStep = Fmt<DT>::kRemChunk / kSteps;  // remainder bytes per step
        constexpr uint32_t kRemLines = 16 * kRemStep / 128;
        auto prefetch_l2 = [&](uint32_t t_ahead) {
            if (lane < kRemLines && t_ahead + 16 <= kSteps)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(rem + uint64_t(t_ahead) * kRemStep + 128 * lane));
            if (lane >= 30) {
                const uint32_t at = rq + 1024 + 128 * (lane - 30);
                if (at < nlines * 16) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + at));
            }
        };
        constexpr int PF = kPeriod;  // one remainder field per step and top-up period in flight
        static_assert(kSteps % (2 * PF) == 0, "the remainder prefetch walks whole pairs of PF steps");
        uint32_t ra[PF], rbk[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) ra[j] = load_rem_full(j);
        prefetch_l2(16);
        prefetch_l2(32);
        prefetch_l2(48);
        for (uint32_t t0 = 0; t0 < kSteps; t0 += 2 * PF) {
            prefetch_l2(t0 + 64);
#pragma unroll
            for (int j = 0; j < PF; ++j) rbk[j] = load_rem_full(t0 + PF + j);
            top_up();
#pragma unroll
            for (int j = 0; j < PF; ++j) rstep(t0 + j, ra[j]);
            if (t0 + 2 * PF < kSteps) {
#pragma unroll
                for (int j = 0; j < PF; ++j) ra[j] = load_rem_full(t0 + 2 * PF + j);
            }
            top_up();
#pragma unroll
            for (int j = 0; j < PF; ++j) rstep(t0 + PF + j, rbk[j]);
        }
        pos = (rq - wb0) >> 1;
    } else if (n_c == kChunk) {
        // The word stream is read sequentially, ~11 bytes per step: pull the
        // lines about 40 steps ahead into L1 so a step never waits on a first
        // touch.
        const uint8_t* wbytes = reinterpret_cast<const uint8_t*>(words);
        const uint32_t wbytes_last = 2 * wlast;
        auto prefetch_words = [&]() {
            if (lane < 2) {
                uint32_t at = 2 * pos + 384 + 128 * lane;
                at = at < wbytes_last ? at : wbytes_last;
                asm volatile("prefetch.global.L1 [%0];" ::"l"(wbytes + at));
            }
        };
        constexpr int PF = DT == UZIP_BF16 ? 16 : 8;
        static_assert(kSteps % (2 * PF) == 0, "the remainder prefetch walks whole pairs of PF steps");
        uint32_t ra[PF], rbk[PF];
#pragma unroll
        for (int j = 0; j < PF; ++j) ra[j] = load_rem_full(j);
        for (uint32_t t0 = 0; t0 < kSteps; t0 += 2 * PF) {
            prefetch_words();
#pragma unroll
            for (int j = 0; j < PF; ++j) rbk[j] = load_rem_full(t0 + PF + j);
#pragma unroll
            for (int j = 0; j < PF; ++j) step(t0 + j, ra[j], true, gwin(), pos, 1);
            if (DT == UZIP_BF16) prefetch_words();
            if (t0 + 2 * PF < kSteps) {
#pragma unroll
                for (int j = 0; j < PF; ++j) ra[j] = load_rem_full(t0 + 2 * PF + j);
            }
#pragma unroll
            for (int j = 0; j < PF; ++j) step(t0 + PF + j, rbk[j], true, gwin(), pos, 1);
        }
    } else {
        const uint32_t T = (n_c + 31) / 32;
        for (uint32_t t = 0; t < T; ++t) step(t, load_rem(t), 32 * t + lane < n_c, gwin(), pos, 1);
    }
    const bool fail = bad || x != kRansL || pos != W;
    return !__any_sync(0xFFFFFFFFu, fail);
}

template <int DT>
__global__ void __launch_bounds__(kDecWarps * 32, 28 / kDecWarps) decompress_kernel(DecompressArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t wid = threadIdx.x >> 5;
    uint8_t* wsm = smem + wid * kDecWarpSmem;
    constexpr uint32_t es = Fmt<DT>::kEs;
    const uint8_t* h = a.comp;
    const uint64_t n = a.n;
    const uint64_t C = num_chunks(n);
    const uint64_t rem_off = rem_offset(n);
    const uint64_t exp_off = exp_offset(DT, n);
    // header checks (every warp, broadcast loads)
    const uint64_t total = *reinterpret_cast<const uint64_t*>(h + 40);
    bool ok = *reinterpret_cast<const uint32_t*>(h) == 0x31505A55u && *reinterpret_cast<const uint16_t*>(h + 4) == 1 &&
              h[6] == uint8_t(DT) && h[7] == 0 && *reinterpret_cast<const uint64_t*>(h + 8) == n &&
              *reinterpret_cast<const uint32_t*>(h + 16) == kChunk && *reinterpret_cast<const uint32_t*>(h + 20) == C &&
              *reinterpret_cast<const uint64_t*>(h + 24) == rem_off &&
              *reinterpret_cast<const uint64_t*>(h + 32) == exp_off && total <= a.cap && total >= exp_off;
    if (!ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_corrupt(a.status);
        return;
    }
    const uint64_t section = total - exp_off;
    const uint64_t nwarps = uint64_t(gridDim.x) * kDecWarps;
    for (uint64_t c = uint64_t(blockIdx.x) * kDecWarps + wid; c < C; c += nwarps) {
        const uint64_t off = reinterpret_cast<const uint64_t*>(h + kHeader)[c];
        const uint32_t lw = reinterpret_cast<const uint32_t*>(h + kHeader + 8 * C)[c];
        const bool raw = (lw & kRawFlag) != 0;
        const uint32_t len = lw & ~kRawFlag;
        const uint64_t left = n - c * kChunk;
        const uint32_t n_c = uint32_t(left < kChunk ? left : kChunk);
        bool good = (off & 15u) == 0 && off <= section && len <= section - off;
        if (good) {
            const uint8_t* src = h + exp_off + off;
            const uint8_t* rem = h + rem_off + c * Fmt<DT>::kRemChunk;
            uint8_t* out = a.out + c * kChunk * es;
            if (raw) {
                if (len == n_c) {
                    if constexpr (Fmt<DT>::kPacked) merge_raw_packed<DT>(src, rem, out, n_c, lane);
                    else merge_raw_bytes<DT>(src, rem, out, n_c, lane);
                }
                else good = false;
            } else {
                // the ring reads the stream in whole 16-byte lines
                if (exp_off + off + ((uint64_t(len) + 15) & ~uint64_t(15)) <= a.cap)
                    good = decode_coded<DT, true>(src, len, rem, out, n_c, lane, wsm);
                else
                    good = decode_coded<DT, false>(src, len, rem, out, n_c, lane, wsm);
            }
        }
        if (!good && lane == 0) flag_corrupt(a.status);
        __syncwarp();
    }
}

cudaError_t launch_decompress(int dtype, const void* d_comp, uint64_t cap, void* d_out, uint64_t n, int32_t* d_status,
                              cudaStream_t s) {
    cudaError_t err;
    if (d_status && (err = cudaMemsetAsync(d_status, 0, sizeof(int32_t), s)) != cudaSuccess) return err;
    DecompressArgs a{static_cast<const uint8_t*>(d_comp), cap, static_cast<uint8_t*>(d_out), n, d_status};
    const uint64_t C = num_chunks(n);  // C == 0 still launches one block to validate the header
    void (*kern)(DecompressArgs) = dtype == UZIP_BF16       ? decompress_kernel<UZIP_BF16>
                                   : dtype == UZIP_FP32     ? decompress_kernel<UZIP_FP32>
                                   : dtype == UZIP_FP16     ? decompress_kernel<UZIP_FP16>
                                   : dtype == UZIP_FP8_E4M3 ? decompress_kernel<UZIP_FP8_E4M3>
                                                            : decompress_kernel<UZIP_FP8_E5M2>;
    const uint32_t smem = kDecWarps * kDecWarpSmem;
    int sms = 0, per_sm = 0;
    if ((err = launch_shape(reinterpret_cast<const void*>(kern), kDecWarps * 32, smem, &sms, &per_sm)) != cudaSuccess)
        return err;
    uint64_t grid = uint64_t(per_sm) * uint64_t(sms);
    const uint64_t need = (C + kDecWarps - 1) / kDecWarps;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    // as few warps as give the same number of rounds (8192 chunks: 2 rounds
    // of 4096 warps rather than 1.9 of 4256); C == 0 keeps its one block
    if (need > 0) {
        const uint64_t rounds = (need + grid - 1) / grid;
        grid = (need + rounds - 1) / rounds;
    }
    kern<<<dim3(uint32_t(grid)), dim3(kDecWarps * 32), smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace uzip
