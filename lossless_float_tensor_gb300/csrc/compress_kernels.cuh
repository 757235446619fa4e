// Compressor device code (included by compress_fmt_*.cu, one element format
// each, so the formats compile in parallel).
//
// Fused compressor: one warp per chunk of 65536 elements, one kernel for the
// whole tensor (UCCL-Zip Fig. 5: local tables let the statistics, the coding
// and the output placement run in one pass without cross-block
// synchronisation).  Per chunk the warp
//   1. streams the chunk once, writes its sign|fraction bytes straight to the
//      remainder plane, writes its exponent bytes to the warp's slot in the
//      work area and counts them in a lane-private histogram;
//   2. normalises the histogram to 4096 (largest remainder) and builds the
//      encode table;
//   3. runs the 32-state interleaved rANS encoder backwards over the exponent
//      bytes of the slot, writing the words backwards from the slot's end;
//   4. publishes its stream length for the decoupled look-back over the chunks
//      before it (Merrill and Garland, "Single-pass parallel prefix scan with
//      decoupled look-back", 2016) and, after its next chunk, copies the
//      stream to its offset with 16-byte stores.
// Each warp owns two 68 KiB slots used in turn, so a finished stream can wait
// for its offset while the next chunk is counted.  A chunk whose words would
// reach exponent bytes not yet read, and every chunk when no slots are given
// (the allocation-free entry point), is encoded twice from the input instead:
// once counting, once writing in place.  A chunk that coding does not shrink
// is stored RAW (NCCLZ Sec. IV-C).
#pragma once

#include "uzip_internal.cuh"

namespace uzip {
struct CompressArgs {
    const uint8_t* in;
    uint64_t n;
    uint8_t* out;
    Scratch* scratch;
    uint64_t* desc;
    uint64_t* out_size;   // nullable
    int32_t* status_out;  // nullable
    uint8_t* stash;       // nullable: two slots of kSlotBytes per warp (exponent bytes, then the stream)
    uint32_t first_ticket;
    uint32_t num_chunks;
    uint32_t gated;  // 1: a gate kernel ran first; scratch->pad = 1 means the whole message goes RAW
    // nullable, mapped host memory: per chunk c, progress[2c] = 1 once its
    // remainder plane is written and progress[2c + 1] = 2^63 | (end of its
    // stream in the exponent section) once the stream is in place
    uint64_t* progress;
    // warp-specialised compressor: a helper starts splitting its next chunk
    // once its encoder has at most this many blocks of 32 steps left of the
    // current one (64 or more: at once)
    uint32_t jit_blocks;
    // mode 4 (parametric tables): the model counts of every exponent field
    // value and their total, the same for every chunk
    uint32_t model_total;
    uint32_t model[256];
};

// element traits --------------------------------------------------------------
template <int DT>
struct Traits {
    static constexpr uint32_t kEs = Fmt<DT>::kEs;
    static constexpr uint32_t kEmask = (1u << Fmt<DT>::kEbits) - 1u;
    __device__ static uint32_t exp_of(uint32_t b) { return (b >> Fmt<DT>::kMbits) & kEmask; }
    __device__ static uint32_t table_off(uint32_t b) { return exp_of(b) << 3; }  // exponent * 8
    // sign|fraction field of one element (sign just above the fraction)
    __device__ static uint32_t rem_of(uint32_t b) {
        constexpr uint32_t mb = Fmt<DT>::kMbits, top = 8 * kEs - 1;
        return ((b >> (top - mb)) & (1u << mb)) | (b & ((1u << mb) - 1u));
    }
    // load element i
    __device__ static uint32_t load(const uint8_t* p, uint64_t i) {
        if (kEs == 1) return p[i];
        if (kEs == 2) return reinterpret_cast<const uint16_t*>(p)[i];
        return reinterpret_cast<const uint32_t*>(p)[i];
    }
};

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, uint32_t lane, uint32_t* total) {
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= uint32_t(o)) inc += t;
    }
    *total = __shfl_sync(0xFFFFFFFFu, inc, 31);
    return inc - v;
}

// ---------------------------------------------------------------------------
// phase 1: plane split + exponent bytes + lane-private histogram
// hist layout: u32 [256 exponent values][16 columns]; lane l counts in column
// l mod 16 (16 KiB in all).  Lanes l and l + 16 share a column, so the atomic
// increments stay exact; within one instruction they meet only when both see
// exponents of equal parity.
// CM: which exponents are counted: 1 all, 2 those at positions 0, 16, 32, ...
// of the chunk (a sampled table), 0 none (a whole-message RAW container).
template <int DT, int CM = 1>
__device__ void split_and_count(const uint8_t* __restrict__ cin, uint32_t n_c, uint8_t* __restrict__ rem_dst,
                                uint8_t* __restrict__ ex_dst, uint8_t* hist, uint32_t lane, uint64_t pol_stream) {
    if constexpr (CM != 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 8
        for (uint32_t i = lane; i < kRegionA / 16; i += 32) reinterpret_cast<uint4*>(hist)[i] = z;
    }
    __syncwarp();
    uint8_t* hl = hist + 4 * (lane & 15);
    // e64 = exponent * 64; pos = the value's position in its 16-value unit
    auto count = [&](uint32_t e64, uint32_t pos) {
        if constexpr (CM == 1) atomicAdd(reinterpret_cast<uint32_t*>(hl + e64), 1u);
        if constexpr (CM == 2)
            if (pos == 0) atomicAdd(reinterpret_cast<uint32_t*>(hl + e64), 1u);
    };
    // A unit is 16 consecutive values (32 bytes of bf16, 64 of fp32) handled by
    // one lane: its remainder bytes (16 or 48) and exponent bytes (16) leave as
    // full 16-byte stores.
    static_assert(!Fmt<DT>::kPacked, "byte-field formats only");
    constexpr uint32_t es = Fmt<DT>::kEs, mb = Fmt<DT>::kMbits;
    constexpr uint32_t PV = es == 4 ? 4 : 2;  // 16-byte vectors per unit
    const uint32_t nunits = n_c / 16;
    auto process = [&](const uint4 (&q)[PV], uint32_t unit) {
        uint32_t ex[4];
        if constexpr (es == 2) {
            // two values per word; exponent field of both at bytes 0 and 2
            constexpr uint32_t em2 = Traits<DT>::kEmask * 0x10001u;
            constexpr uint32_t sgn = (1u << mb) * 0x10001u, frac = ((1u << mb) - 1u) * 0x10001u;
            uint32_t r[8];
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const uint32_t w[4] = {q[v].x, q[v].y, q[v].z, q[v].w};
                uint32_t eb[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    r[4 * v + j] = ((w[j] >> (15 - mb)) & sgn) | (w[j] & frac);
                    eb[j] = (w[j] >> mb) & em2;
                    count((eb[j] << 6) & 0x3FC0u, 8 * v + 2 * j);
                    count((eb[j] >> 10) & 0x3FC0u, 8 * v + 2 * j + 1);
                }
                ex[2 * v] = __byte_perm(eb[0], eb[1], 0x6420);
                ex[2 * v + 1] = __byte_perm(eb[2], eb[3], 0x6420);
            }
            st_v4_hint(rem_dst + uint64_t(unit) * 16,
                       make_uint4(__byte_perm(r[0], r[1], 0x6420), __byte_perm(r[2], r[3], 0x6420),
                                  __byte_perm(r[4], r[5], 0x6420), __byte_perm(r[6], r[7], 0x6420)),
                       pol_stream);
        } else {
            uint32_t r[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint32_t w[4] = {q[v].x, q[v].y, q[v].z, q[v].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    r[4 * v + j] = (w[j] & 0x7FFFFFu) | ((w[j] >> 8) & 0x800000u);
                    count((w[j] >> 17) & 0x3FC0u, 4 * v + j);
                }
                ex[v] = ((w[0] >> 23) & 0xFFu) | ((w[1] >> 15) & 0xFF00u) | ((w[2] >> 7) & 0xFF0000u) |
                        ((w[3] << 1) & 0xFF000000u);
            }
            uint32_t o[12];
#pragma unroll
            for (int g = 0; g < 4; ++g) {  // 4 values -> 12 bytes
                o[3 * g] = r[4 * g] | (r[4 * g + 1] << 24);
                o[3 * g + 1] = (r[4 * g + 1] >> 8) | (r[4 * g + 2] << 16);
                o[3 * g + 2] = (r[4 * g + 2] >> 16) | (r[4 * g + 3] << 8);
            }
            uint8_t* d = rem_dst + uint64_t(unit) * 48;
#pragma unroll
            for (int k = 0; k < 3; ++k)
                st_v4_hint(d + 16 * k, make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]), pol_stream);
        }
        if (ex_dst) *reinterpret_cast<uint4*>(ex_dst + 16 * uint64_t(unit)) = make_uint4(ex[0], ex[1], ex[2], ex[3]);
    };
    auto load_unit = [&](uint4 (&q)[PV], uint32_t unit) {
#pragma unroll
        for (int v = 0; v < int(PV); ++v) q[v] = ld_v4_hint(cin + (uint64_t(unit) * PV + v) * 16, pol_stream);
    };
    // Batches of U units per lane.  A unit's registers are refilled with the
    // same unit of the next batch as soon as it has been processed, so the
    // next batch's loads are in flight while this one is processed (one set
    // of registers, one copy of the loop body).
    constexpr int U = es == 4 ? 4 : 8;
    const uint32_t nb = nunits / (32 * U);
    const uint32_t head = nunits - nb * 32 * U;
    for (uint32_t u = lane; u < head; u += 32) {
        uint4 q[PV];
        load_unit(q, u);
        process(q, u);
    }
    uint4 qa[U][PV];
    auto unit_of = [&](uint32_t k, int u) -> uint32_t { return head + k * 32 * U + 32 * u + lane; };
    auto load = [&](uint4 (&q)[U][PV], uint32_t k) {
#pragma unroll
        for (int u = 0; u < U; ++u) load_unit(q[u], unit_of(k, u));
    };
    if (nb > 0) load(qa, 0);
#pragma unroll 1
    for (uint32_t k = 0; k < nb; ++k) {
        const bool more = k + 1 < nb;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            process(qa[u], unit_of(k, u));
            if (more) load_unit(qa[u], unit_of(k + 1, u));
        }
    }
    // ragged tail (n_c not a multiple of 16): element by element
    for (uint32_t i = nunits * 16 + lane; i < n_c; i += 32) {
        const uint32_t b = Traits<DT>::load(cin, i);
        const uint32_t r = Traits<DT>::rem_of(b);
        const uint32_t e = Traits<DT>::exp_of(b);
#pragma unroll
        for (uint32_t k = 0; k < es - 1; ++k) rem_dst[(es - 1) * uint64_t(i) + k] = uint8_t(r >> (8 * k));
        count(e << 6, i & 15u);
        if (ex_dst) ex_dst[i] = uint8_t(e);
    }
    __syncwarp();
}

// The same pass for formats whose sign|fraction field is not a whole number
// of bytes (fp16: 11 bits, fp8 e4m3fn: 4, e5m2: 3): a unit is 32 values, whose
// W-bit fields pack into exactly W 32-bit words, least significant bit first.
template <int DT, int CM = 1>
__device__ void split_and_count_packed(const uint8_t* __restrict__ cin, uint32_t n_c, uint8_t* __restrict__ rem_dst,
                                       uint8_t* __restrict__ ex_dst, uint8_t* hist, uint32_t lane,
                                       uint64_t pol_stream) {
    static_assert(Fmt<DT>::kPacked, "packed-field formats only");
    constexpr uint32_t es = Fmt<DT>::kEs, mb = Fmt<DT>::kMbits, W = Fmt<DT>::kRbits;
    if constexpr (CM != 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 8
        for (uint32_t i = lane; i < kRegionA / 16; i += 32) reinterpret_cast<uint4*>(hist)[i] = z;
    }
    __syncwarp();
    uint8_t* hl = hist + 4 * (lane & 15);
    auto count = [&](uint32_t e64, uint32_t pos) {  // pos: position in the 32-value unit, mod 16
        if constexpr (CM == 1) atomicAdd(reinterpret_cast<uint32_t*>(hl + e64), 1u);
        if constexpr (CM == 2)
            if (pos == 0) atomicAdd(reinterpret_cast<uint32_t*>(hl + e64), 1u);
    };
    constexpr uint32_t PV = 2 * es;  // 16-byte vectors per 32-value unit
    const uint32_t nunits = n_c / 32;
    auto process = [&](const uint4 (&q)[PV], uint32_t unit) {
        uint32_t w[4 * PV];
#pragma unroll
        for (int v = 0; v < int(PV); ++v) w[4 * v] = q[v].x, w[4 * v + 1] = q[v].y, w[4 * v + 2] = q[v].z, w[4 * v + 3] = q[v].w;
        uint32_t f[32];  // sign|fraction field of each value
        uint32_t ex[8];  // exponent symbols, four per word
        if constexpr (es == 2) {
            constexpr uint32_t em2 = Traits<DT>::kEmask * 0x10001u;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t eb = (w[j] >> mb) & em2;  // both exponents, bytes 0 and 2
                count((eb << 6) & 0x3FC0u, (2 * j) & 15);
                count((eb >> 10) & 0x3FC0u, (2 * j + 1) & 15);
                f[2 * j] = Traits<DT>::rem_of(w[j] & 0xFFFFu);
                f[2 * j + 1] = Traits<DT>::rem_of(w[j] >> 16);
                if (j & 1) ex[j >> 1] = __byte_perm((w[j - 1] >> mb) & em2, eb, 0x6420);
            }
        } else {
            constexpr uint32_t em4 = Traits<DT>::kEmask * 0x01010101u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                ex[j] = (w[j] >> mb) & em4;
                count((ex[j] << 6) & 0x3FC0u, (4 * j) & 15);
                count((ex[j] >> 2) & 0x3FC0u, (4 * j + 1) & 15);
                count((ex[j] >> 10) & 0x3FC0u, (4 * j + 2) & 15);
                count((ex[j] >> 18) & 0x3FC0u, (4 * j + 3) & 15);
#pragma unroll
                for (int k = 0; k < 4; ++k) f[4 * j + k] = Traits<DT>::rem_of((w[j] >> (8 * k)) & 0xFFu);
            }
        }
        uint32_t o[W];
#pragma unroll
        for (uint32_t k = 0; k < W; ++k) o[k] = 0;
#pragma unroll
        for (uint32_t k = 0; k < 32; ++k) {  // field k at bit W k
            const uint32_t bit = W * k, wd = bit >> 5, sh = bit & 31;
            o[wd] |= f[k] << sh;
            if (sh + W > 32) o[wd + 1] |= f[k] >> (32 - sh);
        }
        uint32_t* rd = reinterpret_cast<uint32_t*>(rem_dst + uint64_t(unit) * 4 * W);
#pragma unroll
        for (uint32_t k = 0; k < W; ++k) st_u32_hint(rd + k, o[k], pol_stream);
        if (ex_dst) {
            reinterpret_cast<uint4*>(ex_dst + 32 * uint64_t(unit))[0] = make_uint4(ex[0], ex[1], ex[2], ex[3]);
            reinterpret_cast<uint4*>(ex_dst + 32 * uint64_t(unit))[1] = make_uint4(ex[4], ex[5], ex[6], ex[7]);
        }
    };
    auto load_unit = [&](uint4 (&q)[PV], uint32_t unit) {
#pragma unroll
        for (int v = 0; v < int(PV); ++v) q[v] = ld_v4_hint(cin + (uint64_t(unit) * PV + v) * 16, pol_stream);
    };
    // batches of U units per lane, refilled unit by unit as above
    constexpr int U = es == 2 ? 2 : 4;
    const uint32_t nb = nunits / (32 * U);
    const uint32_t head = nunits - nb * 32 * U;
    for (uint32_t u = lane; u < head; u += 32) {
        uint4 q[PV];
        load_unit(q, u);
        process(q, u);
    }
    uint4 qa[U][PV];
    auto unit_of = [&](uint32_t k, int u) -> uint32_t { return head + k * 32 * U + 32 * u + lane; };
    auto load = [&](uint4 (&q)[U][PV], uint32_t k) {
#pragma unroll
        for (int u = 0; u < U; ++u) load_unit(q[u], unit_of(k, u));
    };
    if (nb > 0) load(qa, 0);
#pragma unroll 1
    for (uint32_t k = 0; k < nb; ++k) {
        const bool more = k + 1 < nb;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            process(qa[u], unit_of(k, u));
            if (more) load_unit(qa[u], unit_of(k + 1, u));
        }
    }
    // ragged tail (fewer than 32 values): its fields start byte aligned
    // (32 W bits per unit); lane 0 packs them, the lanes count and copy the
    // exponents
    const uint32_t i0 = nunits * 32;
    if (i0 < n_c) {
        if (lane == 0) {
            uint64_t acc = 0;
            uint32_t nacc = 0, out = i0 / 8 * W;
            for (uint32_t i = i0; i < n_c; ++i) {
                acc |= uint64_t(Traits<DT>::rem_of(Traits<DT>::load(cin, i))) << nacc;
                nacc += W;
                while (nacc >= 8) {
                    rem_dst[out++] = uint8_t(acc);
                    acc >>= 8;
                    nacc -= 8;
                }
            }
            if (nacc) rem_dst[out] = uint8_t(acc);
        }
        for (uint32_t i = i0 + lane; i < n_c; i += 32) {
            const uint32_t e = Traits<DT>::exp_of(Traits<DT>::load(cin, i));
            count(e << 6, i & 15u);
            if (ex_dst) ex_dst[i] = uint8_t(e);
        }
    }
    __syncwarp();
}

// counts of symbols 8*lane .. 8*lane+7: the 16 columns of each row, read as
// 4 x 16 bytes in a lane-staggered order
inline __device__ void reduce_hist(const uint8_t* hist, uint32_t lane, uint32_t c[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint8_t* row = hist + (8 * lane + k) * 64;
        uint32_t s = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 q = *reinterpret_cast<const uint4*>(row + ((j + lane) & 3) * 16);
            s += q.x + q.y + q.z + q.w;
        }
        c[k] = s;
    }
}

// ---------------------------------------------------------------------------
// phase 2: largest-remainder normalisation (rule R5) -- lane owns symbols
// 8*lane + k.  Leaves f in registers and in freq[] (shared), returns K.
struct Norm {
    uint32_t f[8];
    uint32_t present;  // 8-bit mask of present symbols of this lane
    uint32_t prefix;   // present symbols of lower lanes
    uint32_t k_total;  // present symbols overall
};

// CLOSED: the excess step of R5 in closed form (many boosted symbols, as in a
// sampled table); otherwise one unit at a time.  Both give the same table.
template <bool CLOSED = false>
__device__ void normalise(const uint32_t c[8], uint32_t n_c, uint32_t lane, uint8_t* regB, Norm& nm) {
    uint16_t* freq = reinterpret_cast<uint16_t*>(regB);          // u16[256]
    uint32_t* keys = reinterpret_cast<uint32_t*>(regB + 512);    // u32[256]
    uint32_t r[8];
    uint32_t boosted = 0, present = 0, fsum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t f, rr;
        if (n_c == kChunk) {
            f = c[k] >> 4;
            rr = (c[k] & 15u) << 12;
        } else {
            const uint32_t scaled = c[k] * kM;
            f = scaled / n_c;
            rr = scaled - f * n_c;
        }
        if (c[k]) {
            present |= 1u << k;
            if (f == 0) {
                f = 1;
                boosted |= 1u << k;
            }
        }
        nm.f[k] = f;
        r[k] = rr;
        fsum += f;
    }
    const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, fsum);
    if (total < kM) {
        // candidates: present, not boosted; key orders by (remainder desc, symbol asc)
        const uint32_t cand = present & ~boosted;
        uint32_t nc_total;
        const uint32_t base = warp_excl_scan(__popc(cand), lane, &nc_total);
        uint32_t idx = base;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (cand & (1u << k)) keys[idx++] = (r[k] << 8) | (255u - (8 * lane + k));
        __syncwarp();
        const uint32_t need = kM - total;
        // candidate i is ranked by lane i % 32
        for (uint32_t i = lane; i < nc_total; i += 32) {
            const uint32_t key = keys[i];
            uint32_t rank = 0;
            for (uint32_t j = 0; j < nc_total; ++j) rank += keys[j] > key ? 1u : 0u;
            // freq[] doubles as a winner flag for candidates until it is rewritten below
            freq[255u - (key & 0xFFu)] = rank < need ? 1 : 0;
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (cand & (1u << k)) nm.f[k] += freq[8 * lane + k];
        __syncwarp();
    } else if (total > kM) {
        if constexpr (CLOSED) {
            // R5 takes the excess one at a time from the largest f (ties: the
            // smaller symbol).  Its end state in closed form: with D(L) = sum over
            // symbols of max(0, f - L), the smallest level L with D(L) <= excess
            // caps every f at L, and the r = excess - D(L) smallest symbols at
            // level L lose one more.
            const uint32_t excess = total - kM;
            auto drop = [&](uint32_t level) {
                uint32_t d = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) d += nm.f[k] > level ? nm.f[k] - level : 0u;
                return __reduce_add_sync(0xFFFFFFFFu, d);
            };
            uint32_t lo = 1, hi = kM;  // D(kM) = 0 <= excess < D(0) = total
            while (lo < hi) {
                const uint32_t mid = (lo + hi) / 2;
                if (drop(mid) <= excess) hi = mid;
                else lo = mid + 1;
            }
            const uint32_t level = lo, r = excess - drop(lo);
            uint32_t at = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) at += nm.f[k] >= level ? 1u : 0u;
            uint32_t dummy;
            uint32_t idx = warp_excl_scan(at, lane, &dummy);  // symbols at the level, ascending
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (nm.f[k] >= level) {
                    nm.f[k] = level - (idx < r ? 1u : 0u);
                    ++idx;
                }
            }
        } else {
            // the same, one step at a time
            uint32_t excess = total - kM;
            while (excess--) {
                uint32_t best = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t key = (nm.f[k] << 8) | (255u - (8 * lane + k));
                    best = key > best ? key : best;
                }
                const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, best);
                const uint32_t s = 255u - (top & 0xFFu);
                if ((s >> 3) == lane) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (uint32_t(k) == (s & 7u)) nm.f[k] -= 1;
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) freq[8 * lane + k] = uint16_t(nm.f[k]);
    nm.present = present;
    uint32_t ktot;
    nm.prefix = warp_excl_scan(__popc(present), lane, &ktot);
    nm.k_total = ktot;
    regB[1536 + lane] = uint8_t(present);  // bitmap byte `lane` = symbols 8*lane..8*lane+7
    __syncwarp();
}

// division magic of every frequency, built at compile time
__device__ const MagicTable g_magic = make_magic_table();

// encode table row for each present symbol: {m, add} and {(f << 20) - 1, sh | cum << 5 | (M - f) << 20}
inline __device__ void build_enc_table(const Norm& nm, uint32_t lane, uint8_t* table, uint8_t* regB) {
    uint32_t lsum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) lsum += nm.f[k];
    uint32_t dummy;
    uint32_t cum = warp_excl_scan(lsum, lane, &dummy);
    // present symbol list (u8) in shared memory, then one symbol per lane
    uint8_t* plist = regB + 1600;  // 256 bytes
    uint32_t* cums = reinterpret_cast<uint32_t*>(regB + 512);  // reuse the key area: u32 cum per symbol
    uint32_t idx = nm.prefix;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (nm.present & (1u << k)) {
            plist[idx++] = uint8_t(8 * lane + k);
            cums[8 * lane + k] = cum;
        }
        cum += nm.f[k];
    }
    __syncwarp();
    const uint16_t* freq = reinterpret_cast<const uint16_t*>(regB);
    for (uint32_t i = lane; i < nm.k_total; i += 32) {
        const uint32_t s = plist[i];
        const uint32_t f = freq[s];
        const MagicEntry me = g_magic.e[f];
        const DivMagic dm{me.m, (me.add_sh >> 8) ? me.m : 0u, me.add_sh & 0xFFu, 1u};
        uint4 e;
        e.x = dm.m;
        e.y = dm.add;
        e.z = uint32_t((uint64_t(f) << 20) - 1);
        e.w = dm.sh | (cums[s] << 5) | ((kM - f) << 20);
        *reinterpret_cast<uint2*>(table + 8 * s) = make_uint2(e.x, e.y);
        *reinterpret_cast<uint2*>(table + 2048 + 8 * s) = make_uint2(e.z, e.w);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// rANS encode (rule R6).  The table entry of a symbol is
// {m, add, (f << 20) - 1, sh | cum << 5 | (M - f) << 20}: sh sits in the
// low 5 bits so that a wrapping funnel shift by the packed word shifts by sh,
// and M - f in the top 12 bits comes out with one shift.

// Table loads are written as side-effect-free asm: the table does not change
// while a chunk is encoded, so the compiler may issue them as early as it likes
// (ahead of the staging stores of earlier steps).
// The table is split in two arrays of 8-byte rows, {m, add} at [0, 2 KiB) and
// {(f << 20) - 1, packed} at [2 KiB, 4 KiB): a 64-bit load is served per half
// warp, and any 16 consecutive exponent values fall in distinct banks, so the
// usual ~20-value exponent window costs few bank conflicts (a 16-byte row would
// put values s and s + 8 in the same banks of every quarter warp).
__device__ __forceinline__ uint4 lds_table(uint32_t saddr) {
    uint4 v;
    asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(saddr));
    asm("ld.shared.v2.u32 {%0,%1}, [%2+2048];" : "=r"(v.z), "=r"(v.w) : "r"(saddr));
    return v;
}
__device__ __forceinline__ void sts_u16(uint32_t saddr, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(saddr), "h"(static_cast<unsigned short>(v)));
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t rans_update(uint32_t x, const uint4 e, bool emit) {
    const uint32_t xr = emit ? (x >> 16) : x;
    const uint64_t t = uint64_t(xr) * e.x + e.y;
    const uint32_t q = __funnelshift_r(uint32_t(t >> 32), 0u, e.w);  // shift by e.w mod 32 = sh
    const uint32_t mmf = e.w >> 20;
    const uint32_t cum = (e.w >> 5) & 0xFFFu;
    return q * mmf + (xr + cum);
}

enum class Sink { Count, Global };

struct EncState {
    uint32_t x;     // this lane's rANS state
    int32_t pos;    // Count: -words so far; Global / slot: u16 index below which the next words go
};

// One encode step for one lane (symbol from an input value).
template <int DT, Sink S>
__device__ __forceinline__ void enc_step(EncState& st, uint32_t bits, bool active, uint32_t table_s, uint8_t* gwords,
                                         uint32_t lt) {
    const uint4 e = lds_table(table_s + Traits<DT>::table_off(bits));
    const bool emit = active && (st.x > e.z);
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, emit);
    const int32_t nt = __popc(b);
    if (S == Sink::Global && emit)
        *reinterpret_cast<uint16_t*>(gwords + 2 * uint64_t(uint32_t(st.pos - nt) + __popc(b & lt))) = uint16_t(st.x);
    st.pos -= nt;
    const uint32_t xn = rans_update(st.x, e, emit);
    st.x = active ? xn : st.x;
}

// Symbol loads: 32 steps (t, t-1, ..., t-31) of this lane, most recent step
// first.  volatile keeps them ahead of the steps that consume them.
template <int DT>
__device__ __forceinline__ void load_block(uint32_t (&v)[32], const uint8_t* cin, int32_t t, uint32_t lane,
                                           uint64_t pol) {
    constexpr uint32_t es = Traits<DT>::kEs;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint8_t* p = cin + es * (uint64_t(uint32_t(t - j)) * 32 + lane);
        v[j] = es == 1 ? uint32_t(*p) : es == 2 ? ld_u16_hint(p, pol) : ld_u32_hint(p, pol);
    }
}

// Encoder over the input values, used when the fast path cannot run.
//   Sink::Count  only counts words (st.pos = -count) and returns false as soon
//                as hdr_bytes + 2 * count reaches n_c (the chunk goes RAW);
//   Sink::Global writes each word in place at gwords, st.pos counting down
//                from the word total.
template <int DT, Sink S>
__device__ bool encode_chunk(const uint8_t* __restrict__ cin, uint32_t n_c, uint32_t table_s, uint32_t lane,
                             EncState& st, uint8_t* gwords, uint32_t hdr_bytes, uint64_t pol) {
    const uint32_t lt = lanemask_lt();
    constexpr uint32_t es = Traits<DT>::kEs;
    st.x = kRansL;
    if (n_c == kChunk) {
        uint32_t va[32], vb[32];
        auto run_block = [&](const uint32_t (&v)[32]) -> bool {
#pragma unroll
            for (int j = 0; j < 32; ++j) enc_step<DT, S>(st, v[j], true, table_s, gwords, lt);
            return !(S == Sink::Count && hdr_bytes + 2u * uint32_t(-st.pos) >= n_c);
        };
        load_block<DT>(va, cin, int32_t(kSteps) - 1, lane, pol);
        for (int32_t t0 = int32_t(kSteps) - 1;; t0 -= 64) {
            load_block<DT>(vb, cin, t0 - 32, lane, pol);
            if (!run_block(va)) return false;
            const bool last = t0 == 63;
            if (!last) load_block<DT>(va, cin, t0 - 64, lane, pol);
            if (!run_block(vb)) return false;
            if (last) break;
        }
        return true;
    }
    const uint32_t T = (n_c + 31) / 32;
    for (int32_t t = int32_t(T) - 1; t >= 0; --t) {
        const uint32_t i = 32 * uint32_t(t) + lane;
        const bool active = i < n_c;
        uint32_t bits = 0;
        if (active)
            bits = es == 1   ? uint32_t(cin[i])
                   : es == 2 ? ld_u16_hint(cin + 2 * uint64_t(i), pol)
                             : ld_u32_hint(cin + 4 * uint64_t(i), pol);
        enc_step<DT, S>(st, bits, active, table_s, gwords, lt);
        if (S == Sink::Count && hdr_bytes + 2u * uint32_t(-st.pos) >= n_c) return false;
    }
    return true;
}

// Fast path: exponent bytes from the warp's slot, words written backwards
// from the slot's end (st.pos: u16 index, counting down).
// The word store of step j is issued after the state update of step j + 2:
// its address depends on the ballots of all earlier steps, and a warp issues
// in order, so storing at once would hold back every later step.  Returns
// false, before any word could overwrite an exponent byte not yet read, if the
// stream grows faster than the exponents are consumed.
__device__ __forceinline__ uint32_t ld_slot_u8(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.global.cg.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_slot_u16(uint8_t* p, uint32_t v) {
    asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(static_cast<unsigned short>(v)) : "memory");
}

inline __device__ bool encode_slot(uint8_t* slot, uint32_t n_c, uint32_t table_s, uint32_t lane, EncState& st) {
    const uint32_t lt = lanemask_lt();
    st.x = kRansL;
    st.pos = int32_t(kSlotBytes / 2);
    const int32_t T = int32_t((n_c + 31) / 32);  // steps
    const int32_t T0 = int32_t(n_c / 32) & ~31;  // steps in whole 32-step blocks of full steps
    // Steps above the whole blocks (a partial chunk only), one at a time: the
    // top step may have lanes past the chunk's end, which neither update nor
    // emit.  Their words go straight to the slot.
    for (int32_t t = T - 1; t >= T0; --t) {
        const bool active = uint32_t(t) * 32 + lane < n_c;
        const uint32_t v = ld_slot_u8(slot + (uint32_t(t) * 32 + lane));
        const uint4 e = lds_table(table_s + 8 * v);
        const bool emit = active && st.x > e.z;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, emit);
        const int32_t nt = __popc(b);
        if (emit) st_slot_u16(slot + 2u * uint32_t(st.pos - nt + __popc(b & lt)), st.x);
        st.pos -= nt;
        const uint32_t xn = rans_update(st.x, e, emit);
        st.x = active ? xn : st.x;
    }
    if (T0 == 0) return true;
    uint32_t va[32];
    auto load_ex = [&](uint32_t (&v)[32], int32_t t) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = ld_slot_u8(slot + (uint32_t(t - j) * 32 + lane));
    };
    // exponent bytes of the block three ahead are pulled into L2 (8 lines)
    auto prefetch_block = [&](int32_t t_top) {
        const int32_t t_low = t_top - 31;
        if (t_low >= 0 && lane < 8) asm volatile("prefetch.global.L2 [%0];" ::"l"(slot + uint32_t(t_low) * 32 + 128 * lane));
    };
    uint32_t w1 = 0, w2 = 0, b1 = 0, b2 = 0;
    bool e1 = false, e2 = false;
    auto flush_one = [&](uint32_t w, bool emit, uint32_t b) {
        const int32_t nt = __popc(b);
        if (emit) st_slot_u16(slot + 2u * uint32_t(st.pos - nt + __popc(b & lt)), w);
        st.pos -= nt;
    };
    // Words stored during the block starting at step t0 (the two delayed
    // steps of the last block and 30 of this one: at most 1024 words) must
    // land on exponent bytes whose loads have surely completed.  Each store's
    // address depends on the states of all steps before the previous block, so
    // the bytes of steps above t0 + 32 qualify: u16 index 16 (t0 + 33) and up.
    // Loads of later steps are in flight or not yet issued, and nothing orders
    // them against another lane's store.
    auto run_block = [&](uint32_t (&v)[32], int32_t t0, bool load_next) -> bool {
        if (st.pos - 32 * 32 < 16 * (t0 + 33)) return false;
        // byte of step t0 - 32 - j (the next block) at nxt - 32 j
        const uint8_t* nxt = slot + (uint32_t(load_next ? t0 - 32 : 0) * 32 + lane);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint4 e = lds_table(table_s + 8 * v[j]);
            if (load_next) v[j] = ld_slot_u8(nxt - 32 * j);
            const bool emit = st.x > e.z;
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, emit);
            const uint32_t w = st.x;
            st.x = rans_update(st.x, e, emit);
            flush_one(w2, e2, b2);  // step j - 2
            w2 = w1, e2 = e1, b2 = b1;
            w1 = w, e1 = emit, b1 = b;
        }
        return true;
    };
    // whole blocks from step T0 - 1 down.  Once step j of a block has read
    // its table entry, v[j] is refilled with the exponent byte of step j of
    // the next block, so that block's loads run during this one (one set of
    // 32 registers, one copy of the block's code).
    load_ex(va, T0 - 1);
    prefetch_block(T0 - 65);
#pragma unroll 1
    for (int32_t t0 = T0 - 1;; t0 -= 32) {
        const bool has_next = t0 >= 63;
        prefetch_block(t0 - 96);
        if (!run_block(va, t0, has_next)) return false;
        if (!has_next) break;
    }
    flush_one(w2, e2, b2);
    flush_one(w1, e1, b1);
    return true;
}

// ---------------------------------------------------------------------------
// output helpers

// header of a coded stream, written to global memory (2-byte aligned): 32
// states, bitmap, present frequencies ascending
inline __device__ void write_stream_head(uint8_t* dst, uint32_t x, const Norm& nm, uint32_t lane, const uint8_t* regB) {
    uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
    d16[2 * lane] = uint16_t(x);
    d16[2 * lane + 1] = uint16_t(x >> 16);
    if (lane < 16) d16[64 + lane] = uint16_t(regB[1536 + 2 * lane] | (regB[1536 + 2 * lane + 1] << 8));
    uint32_t idx = nm.prefix;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (nm.present & (1u << k)) d16[80 + idx++] = uint16_t(nm.f[k]);
}

// Copies the record [start, end) of a slot (start 2-byte aligned, end 4-byte
// aligned) to dst (16-byte aligned) in 16-byte blocks, zero padding the last
// block; 4 blocks in flight per lane.
inline __device__ void copy_record_from_slot(const uint8_t* slot, uint32_t start, uint8_t* dst, uint32_t lane,
                                      uint64_t pol, uint32_t end = kSlotBytes) {
    const uint32_t len = end - start;
    const uint32_t nb = (len + 15) / 16;
    const uint32_t mis = start & 2u;  // start mod 4 is 0 or 2
    const uint32_t* wbase = reinterpret_cast<const uint32_t*>(slot + (start & ~3u));
    const uint32_t nwords = (end - (start & ~3u)) / 4;  // words of the slot from wbase on
    for (uint32_t b0 = 0; b0 < nb; b0 += 4 * 32) {
        uint32_t w[4][5];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t b = b0 + 32 * k + lane;
#pragma unroll
            for (int j = 0; j < 5; ++j) {
                const uint32_t wi = 4 * b + j;
                w[k][j] = (b < nb && wi < nwords) ? __ldcg(wbase + wi) : 0u;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t b = b0 + 32 * k + lane;
            if (b >= nb) continue;
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = mis ? __byte_perm(w[k][j], w[k][j + 1], 0x5432) : w[k][j];
            const uint32_t valid = len - 16 * b;
            if (valid < 16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t lo = 4 * j;
                    if (valid <= lo) o[j] = 0;
                    else if (valid < lo + 4) o[j] &= (1u << (8 * (valid - lo))) - 1u;
                }
            }
            st_v4_hint(dst + 16 * b, make_uint4(o[0], o[1], o[2], o[3]), pol);
        }
    }
}

__device__ __forceinline__ void discard_l2_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
// drop the slot's L2 lines [first_byte, last_byte) (128-byte granularity,
// lines partly outside the range are kept)
inline __device__ void discard_slot(uint8_t* slot, uint32_t first_byte, uint32_t last_byte, uint32_t lane) {
    const uint32_t l0 = (first_byte + 127) / 128, l1 = last_byte / 128;
    for (uint32_t l = l0 + lane; l < l1; l += 32) discard_l2_line(slot + 128 * l);
}

// RAW chunk: the n_c exponent bytes, zero padded to 16
template <int DT>
__device__ void write_raw(const uint8_t* __restrict__ cin, uint32_t n_c, uint8_t* dst, uint32_t lane) {
    constexpr uint32_t es = Fmt<DT>::kEs, mb = Fmt<DT>::kMbits;
    const uint32_t nb = (n_c + 15) / 16;
    for (uint32_t b = lane; b < nb; b += 32) {
        const uint32_t i0 = 16 * b;
        uint32_t o[4] = {0, 0, 0, 0};
        if (i0 + 16 <= n_c) {
            if (es == 2) {
                constexpr uint32_t em2 = Traits<DT>::kEmask * 0x10001u;
                const uint4 q0 = *reinterpret_cast<const uint4*>(cin + 2 * uint64_t(i0));
                const uint4 q1 = *reinterpret_cast<const uint4*>(cin + 2 * uint64_t(i0) + 16);
                const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = __byte_perm((w[2 * j] >> mb) & em2, (w[2 * j + 1] >> mb) & em2, 0x6420);
            } else if (es == 1) {
                constexpr uint32_t em4 = Traits<DT>::kEmask * 0x01010101u;
                const uint4 q = *reinterpret_cast<const uint4*>(cin + uint64_t(i0));
                o[0] = (q.x >> mb) & em4, o[1] = (q.y >> mb) & em4, o[2] = (q.z >> mb) & em4, o[3] = (q.w >> mb) & em4;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 q = *reinterpret_cast<const uint4*>(cin + 4 * uint64_t(i0) + 16 * j);
                    o[j] = (q.x >> 23 & 0xFFu) | ((q.y >> 23 & 0xFFu) << 8) | ((q.z >> 23 & 0xFFu) << 16) |
                           ((q.w >> 23 & 0xFFu) << 24);
                }
            }
        } else {
            for (uint32_t k = 0; k < 16 && i0 + k < n_c; ++k)
                o[k >> 2] |= Traits<DT>::exp_of(Traits<DT>::load(cin, i0 + k)) << (8 * (k & 3));
        }
        *reinterpret_cast<uint4*>(dst + 16 * uint64_t(b)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Decoupled look-back.  publish_length makes chunk c's padded length visible
// (as its inclusive prefix for chunk 0, else as an aggregate);
// resolve_offset waits for the exclusive prefix before chunk c and publishes
// chunk c's inclusive prefix.
inline __device__ void publish_length(uint64_t* desc, uint32_t c, uint64_t padded, uint32_t lane) {
    if (lane == 0) st_release_u64(desc + c, (c == 0 ? kDescInclusive : kDescAggregate) | padded);
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// The walk reads 128 descriptors per round trip (4 per lane, nearest first):
// with placement deferred, the nearest published inclusive prefix can lie
// hundreds of chunks back.  A descriptor is one 64-bit word (flag and value),
// so a relaxed load sees both consistently.
inline __device__ bool resolve_offset(uint64_t* desc, uint32_t c, uint64_t padded, uint32_t lane, uint64_t& excl_out) {
    if (c == 0) {
        excl_out = 0;
        return true;
    }
    uint64_t excl = 0;
    int64_t top = int64_t(c) - 1;
    uint32_t spins = 0;
    uint32_t backoff = 32;
    bool ok = true;
    uint64_t d0[4] = {0, 0, 0, 0};  // the nearest window, kept for helping
    uint32_t first0 = 0, kin0 = 0;
    bool first_round = true;
    while (true) {
        // lane l holds descriptors top - 4l .. top - 4l - 3 (k = 0 nearest)
        uint64_t d[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t idx = top - 4 * int64_t(lane) - k;
            d[k] = idx >= 0 ? ld_relaxed_u64(desc + idx) : kDescInclusive;  // before chunk 0: inclusive 0
        }
        // first inclusive within the lane, and whether an empty one precedes it
        uint32_t kin = 4;
        bool empty_before = false;
#pragma unroll
        for (int k = 3; k >= 0; --k) {
            if ((d[k] >> 62) == 2) kin = uint32_t(k);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (uint32_t(k) < kin && (d[k] >> 62) == 0) empty_before = true;
        const uint32_t incl = __ballot_sync(0xFFFFFFFFu, kin < 4);
        const uint32_t first = incl ? uint32_t(__ffs(incl) - 1) : 32u;  // lane holding the nearest inclusive
        // any empty descriptor nearer than that inclusive?
        const bool my_empty = lane < first ? (d[0] >> 62 == 0 || d[1] >> 62 == 0 || d[2] >> 62 == 0 || d[3] >> 62 == 0)
                                           : (lane == first && empty_before);
        if (__any_sync(0xFFFFFFFFu, my_empty)) {
            if (++spins > kSpinLimit) {
                ok = false;
                break;
            }
            __nanosleep(backoff);
            backoff = backoff < 1024 ? backoff * 2 : 1024;
            continue;
        }
        if (first_round) {
#pragma unroll
            for (int k = 0; k < 4; ++k) d0[k] = d[k];
            first0 = first;
            kin0 = kin;
            first_round = false;
        }
        uint64_t val = 0;
        if (lane < first) {
#pragma unroll
            for (int k = 0; k < 4; ++k) val += d[k] & kDescValue;
        } else if (lane == first) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (uint32_t(k) <= kin) val += d[k] & kDescValue;
        }
        excl += warp_sum_u64(val);
        if (first < 32) break;
        top -= 128;
    }
    if (lane == 0) st_release_u64(desc + c, kDescInclusive | ((excl + padded) & kDescValue));
    // Help the chunks of the nearest window that had only aggregates: their
    // inclusive prefixes follow from this one (excl minus the aggregates of
    // the chunks between), and publishing them lets the next walks stop
    // within one round trip.  A prefix is unique, so a chunk's own warp or
    // another helper writing it too stores the same value.
    if (ok && first0 > 0) {
        const uint32_t nk = lane < first0 ? 4u : (lane == first0 ? kin0 : 0u);
        uint64_t v[4], tot = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = uint32_t(k) < nk ? (d0[k] & kDescValue) : 0;
            tot += v[k];
        }
        uint64_t inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= uint32_t(o)) inc += t;
        }
        uint64_t between = inc - tot;  // aggregates of the chunks nearer than this lane's
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (uint32_t(k) < nk) {
                const uint64_t idx = uint64_t(c) - 1 - 4 * lane - k;
                st_relaxed_u64(desc + idx, kDescInclusive | ((excl - between) & kDescValue));
            }
            between += v[k];
        }
    }
    excl_out = excl;
    return ok;
}

// ---------------------------------------------------------------------------
// Header (R11) and the zero padding around the remainder plane; total = 0
// marks a failed compression.  One thread.
// Progress for a host that copies finished parts while the kernel runs: every
// lane's writes are made visible system-wide before lane 0 posts the word.
__device__ __forceinline__ void post_progress(uint64_t* p, uint64_t v, uint32_t lane) {
    __threadfence_system();
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile uint64_t*>(p) = v;
}

template <int DT>
__device__ void write_header(const CompressArgs& a, uint64_t total, uint32_t st) {
    const uint64_t n = a.n, C = a.num_chunks;
    const uint64_t rem_off = C ? rem_offset(n) : kHeader, exp_off = C ? exp_offset(DT, n) : kHeader;
    uint8_t* h = a.out;
    *reinterpret_cast<uint32_t*>(h) = 0x31505A55u;  // "UZP1"
    *reinterpret_cast<uint16_t*>(h + 4) = 1;
    h[6] = uint8_t(DT);
    h[7] = 0;
    *reinterpret_cast<uint64_t*>(h + 8) = n;
    *reinterpret_cast<uint32_t*>(h + 16) = kChunk;
    *reinterpret_cast<uint32_t*>(h + 20) = uint32_t(C);
    *reinterpret_cast<uint64_t*>(h + 24) = rem_off;
    *reinterpret_cast<uint64_t*>(h + 32) = exp_off;
    *reinterpret_cast<uint64_t*>(h + 40) = total;
    *reinterpret_cast<uint64_t*>(h + 48) = 0;
    *reinterpret_cast<uint64_t*>(h + 56) = 0;
    for (uint64_t i = kHeader + 12 * C; i < rem_off; ++i) h[i] = 0;
    for (uint64_t i = rem_off + rem_plane_bytes(DT, n); i < exp_off; ++i) h[i] = 0;
    if (a.out_size) *a.out_size = total;
    if (a.status_out) *a.status_out = int32_t(st ? st : (total ? 0u : uint32_t(UZIP_ERR_TIMEOUT)));
}

// SAMPLED: each chunk's table from a sample of it (positions 0, 16, 32, ...;
// a seen symbol counts 16 x its sample count, an unseen one of the format's
// exponent range counts 1; UCCL-Zip Fig. 5), without the full histogram.
template <int DT, bool SAMPLED = false>
__global__ void __launch_bounds__(32) compress_kernel(CompressArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* regA = smem;
    uint8_t* regB = smem + kRegionA;
    const uint32_t lane = threadIdx.x;
    const uint64_t n = a.n;
    const uint32_t C = a.num_chunks;
    const uint64_t rem_off = rem_offset(n);
    const uint64_t exp_off = exp_offset(DT, n);
    constexpr uint32_t es = Traits<DT>::kEs;
    const uint64_t pol_stream = policy_evict_first();
    const uint32_t processed = C - a.first_ticket;
    const uint32_t table_s = smem_addr(regA);
    // this warp's two slots (one warp per block)
    uint8_t* slots = a.stash ? a.stash + uint64_t(blockIdx.x) * 2 * kSlotBytes : nullptr;
    uint32_t which = 0;
    if (a.gated && *reinterpret_cast<volatile uint32_t*>(&a.scratch->pad) != 0) return;  // the RAW kernel has it

    // Chunk c is placed: table entries, done counter; the warp that completes
    // the last chunk writes the header.  Returns true for that warp.
    auto complete = [&](uint32_t c, uint32_t len, bool raw, uint64_t excl, bool ok) -> bool {
        if (!ok && lane == 0) atomicCAS(&a.scratch->status, 0u, uint32_t(UZIP_ERR_TIMEOUT));
        if (ok && lane == 0) {
            reinterpret_cast<uint64_t*>(a.out + kHeader)[c] = excl;
            reinterpret_cast<uint32_t*>(a.out + kHeader + 8 * uint64_t(C))[c] = len | (raw ? kRawFlag : 0u);
        }
        if (a.progress && ok) post_progress(a.progress + 2 * uint64_t(c) + 1, (1ull << 63) | (excl + round16(len)), lane);
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) {
            __threadfence();
            prev = atomicAdd(&a.scratch->done, 1u);
        }
        prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
        if (prev + 1 != processed) return false;
        __threadfence();
        if (lane == 0) {
            const uint32_t st = *reinterpret_cast<volatile uint32_t*>(&a.scratch->status);
            const uint64_t last = ld_acquire_u64(a.desc + (C - 1));
            uint64_t total = exp_off + (last & kDescValue);
            if (st != 0 || (last >> 62) != 2) total = 0;
            write_header<DT>(a, total, st);
        }
        return true;
    };

    // A pending chunk: its record [p_start, kSlotBytes) waits in slot p_slot until
    // its offset is known; then it is copied out and the slot's lines dropped.
    bool pend = false;
    uint32_t p_c = 0, p_start = 0;
    uint8_t* p_slot = nullptr;
    auto place_pending = [&]() -> bool {
        const uint32_t len = kSlotBytes - p_start;
        uint64_t excl = 0;
        const bool ok = resolve_offset(a.desc, p_c, round16(len), lane, excl);
        if (ok) copy_record_from_slot(p_slot, p_start, a.out + exp_off + excl, lane, pol_stream);
        __syncwarp();
        discard_slot(p_slot, 0, kSlotBytes, lane);
        __syncwarp();
        pend = false;
        return complete(p_c, len, false, excl, ok);
    };

    uint32_t* ticket = &a.scratch->ticket;
    while (C > 0) {
        uint32_t c = 0;
        if (lane == 0) c = atomicAdd(ticket, 1u) + a.first_ticket;
        c = __shfl_sync(0xFFFFFFFFu, c, 0);
        if (c >= C) break;
        const uint64_t left = n - uint64_t(c) * kChunk;
        const uint32_t n_c = uint32_t(left < kChunk ? left : kChunk);
        const uint8_t* cin = a.in + uint64_t(c) * kChunk * es;
        uint8_t* slot = slots ? slots + which * kSlotBytes : nullptr;

        // 1. plane split + exponent bytes + histogram
        if constexpr (Fmt<DT>::kPacked)
            split_and_count_packed<DT, SAMPLED ? 2 : 1>(cin, n_c, a.out + rem_off + uint64_t(c) * Fmt<DT>::kRemChunk, slot,
                                                 regA, lane, pol_stream);
        else
            split_and_count<DT, SAMPLED ? 2 : 1>(cin, n_c, a.out + rem_off + uint64_t(c) * Fmt<DT>::kRemChunk, slot, regA,
                                          lane, pol_stream);
        if (a.progress) post_progress(a.progress + 2 * uint64_t(c), 1, lane);
        uint32_t total = n_c;  // counts' total
        uint32_t cnt[8];
        reduce_hist(regA, lane, cnt);
        __syncwarp();
        if constexpr (SAMPLED) {
            uint32_t part = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t sym = 8 * lane + k;
                cnt[k] = cnt[k] ? 16 * cnt[k] : (sym < (1u << Fmt<DT>::kEbits) ? 1u : 0u);
                part += cnt[k];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
            total = part;
        }
        // 2. normalise + encode table
        Norm nm;
        normalise<SAMPLED>(cnt, total, lane, regB, nm);
        build_enc_table(nm, lane, regA, regB);
        const uint32_t hdr = kStreamHead + 2 * nm.k_total;

        // 3. encode: fast path from the slot, else count from the input
        EncState st{kRansL, 0};
        bool fast = slot != nullptr && encode_slot(slot, n_c, table_s, lane, st);
        uint32_t len = 0, w_total = 0;
        bool raw = false;
        if (fast) {
            w_total = kSlotBytes / 2 - uint32_t(st.pos);
            len = hdr + 2 * w_total;
            raw = len >= n_c;
        } else {
            EncState cs{kRansL, 0};
            const bool coded = encode_chunk<DT, Sink::Count>(cin, n_c, table_s, lane, cs, nullptr, hdr, pol_stream);
            w_total = uint32_t(-cs.pos);
            len = hdr + 2 * w_total;
            raw = !coded || len >= n_c;
        }
        if (raw) len = n_c;

        // 4. publish the length; place the previous pending chunk, whose
        //    predecessors have had a whole chunk's time to finish
        publish_length(a.desc, c, round16(len), lane);
        if (pend && place_pending()) return;
        if (fast && !raw) {
            const uint32_t start = kSlotBytes - len;  // record = head + words, ending at the slot's end
            write_stream_head(slot + start, st.x, nm, lane, regB);
            __syncwarp();
            discard_slot(slot, 0, start, lane);  // exponent bytes below the record are spent
            pend = true;
            p_c = c;
            p_start = start;
            p_slot = slot;
            which ^= 1;
            continue;
        }
        // 5. otherwise place this chunk now
        uint64_t excl = 0;
        const bool ok = resolve_offset(a.desc, c, round16(len), lane, excl);
        if (ok) {
            uint8_t* dst = a.out + exp_off + excl;
            if (raw) {
                write_raw<DT>(cin, n_c, dst, lane);
            } else {
                // encode again from the input, writing the words in place
                EncState gs{kRansL, int32_t(w_total)};
                encode_chunk<DT, Sink::Global>(cin, n_c, table_s, lane, gs, dst + hdr, hdr, pol_stream);
                write_stream_head(dst, gs.x, nm, lane, regB);
                for (uint32_t i = len + lane; i < round16(len); i += 32) dst[i] = 0;
            }
        }
        __syncwarp();
        if (slot) discard_slot(slot, 0, kSlotBytes, lane);
        if (complete(c, len, raw, excl, ok)) return;
    }
    if (pend && place_pending()) return;
    // empty tensor: header only, written by the single launched warp
    if (C == 0 && blockIdx.x == 0 && lane == 0) write_header<DT>(a, kHeader, 0);
}

// ---------------------------------------------------------------------------
// Whole-message modes (NCCLZ Sec. IV-C, Alg. 1: a message whose coding would
// not pay travels RAW).
//
// gate_kernel: one warp decides from the message's first 64 KiB of input --
// the sample's exponent bytes counted, normalised and coded as one chunk --
// and sets scratch->pad = 1 when that chunk would be stored RAW under the
// per-chunk rule.  It writes the sample's share of the remainder plane as a
// side effect, with the bytes the main pass writes again, and codes through
// the first slot of the work area (free until the main pass starts).
template <int DT>
__global__ void __launch_bounds__(32) gate_kernel(CompressArgs a, uint32_t n_s) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* regA = smem;
    uint8_t* regB = smem + kRegionA;
    const uint32_t lane = threadIdx.x;
    const uint64_t pol = policy_evict_first();
    uint8_t* rem = a.out + rem_offset(a.n);
    uint8_t* slot = a.stash;  // nullable
    if constexpr (Fmt<DT>::kPacked)
        split_and_count_packed<DT>(a.in, n_s, rem, slot, regA, lane, pol);
    else
        split_and_count<DT>(a.in, n_s, rem, slot, regA, lane, pol);
    uint32_t cnt[8];
    reduce_hist(regA, lane, cnt);
    __syncwarp();
    Norm nm;
    normalise(cnt, n_s, lane, regB, nm);
    build_enc_table(nm, lane, regA, regB);
    const uint32_t hdr = kStreamHead + 2 * nm.k_total;
    EncState cs{kRansL, 0};
    bool raw;
    if (slot && encode_slot(slot, n_s, smem_addr(regA), lane, cs)) {
        raw = hdr + 2 * (kSlotBytes / 2 - uint32_t(cs.pos)) >= n_s;
    } else {
        cs = EncState{kRansL, 0};
        const bool coded = encode_chunk<DT, Sink::Count>(a.in, n_s, smem_addr(regA), lane, cs, nullptr, hdr, pol);
        raw = !coded || hdr + 2 * uint32_t(-cs.pos) >= n_s;
    }
    if (lane == 0) a.scratch->pad = raw ? 1u : 0u;
}

// raw_kernel: every chunk RAW.  Offsets need no look-back: chunk c's RAW
// stream (its exponent bytes) starts at 65536 c of the exponent section.  The
// work is cut into pieces of kRawPiece elements, one warp each, so that a
// message of a few chunks still spreads over the GPU (the remainder fields of
// a piece start on a byte: kRawPiece * W / 8 is whole for every format).
// Exits at once when a gate ran and chose coding.
constexpr uint32_t kRawPiece = 4096;
template <int DT>
__global__ void __launch_bounds__(32) raw_kernel(CompressArgs a) {
    if (a.gated && *reinterpret_cast<volatile uint32_t*>(&a.scratch->pad) == 0) return;
    const uint32_t lane = threadIdx.x;
    const uint64_t n = a.n, C = a.num_chunks;
    const uint64_t rem_off = rem_offset(n), exp_off = exp_offset(DT, n);
    const uint64_t pol = policy_evict_first();
    constexpr uint32_t kPer = kChunk / kRawPiece;  // pieces per chunk
    const uint64_t P = (n + kRawPiece - 1) / kRawPiece;
    for (uint64_t p = blockIdx.x; p < P; p += gridDim.x) {
        const uint64_t c = p / kPer, sub = p % kPer;
        const uint64_t left = n - c * kChunk;
        const uint32_t n_c = uint32_t(left < kChunk ? left : kChunk);
        const uint32_t first = uint32_t(sub) * kRawPiece;
        const uint32_t n_p = n_c - first < kRawPiece ? n_c - first : kRawPiece;
        const uint8_t* cin = a.in + (c * kChunk + first) * Fmt<DT>::kEs;
        uint8_t* rem = a.out + rem_off + c * Fmt<DT>::kRemChunk + uint64_t(first) / 8 * Fmt<DT>::kRbits;
        uint8_t* dst = a.out + exp_off + c * kChunk;
        if constexpr (Fmt<DT>::kPacked)
            split_and_count_packed<DT, 0>(cin, n_p, rem, dst + first, nullptr, lane, pol);
        else
            split_and_count<DT, 0>(cin, n_p, rem, dst + first, nullptr, lane, pol);
        if (first + n_p == n_c) {  // the chunk's last piece: padding and table entries
            for (uint32_t i = n_c + lane; i < round16(n_c); i += 32) dst[i] = 0;
            if (lane == 0) {
                reinterpret_cast<uint64_t*>(a.out + kHeader)[c] = c * kChunk;
                reinterpret_cast<uint32_t*>(a.out + kHeader + 8 * C)[c] = n_c | kRawFlag;
            }
        }
    }
    if (blockIdx.x == 0 && lane == 0) write_header<DT>(a, container_bound(DT, n), 0);
}

// ---------------------------------------------------------------------------
// launcher of one format and mode (instantiated in compress_fmt_*.cu)

// the warp-specialised compressor (compress_ws.cuh)
// TM, the table of each chunk: 0 its histogram, 1 a sample of it, 2 the
// caller's Gaussian model
template <int DT, int TM>
cudaError_t launch_ws(const CompressArgs& a, cudaStream_t s);

// Launches the kernels of one compression mode (0: per-chunk choice, 1: whole
// message RAW, 2: gated, 3: sampled tables, 4: parametric tables) for
// element format DT.  With a slot area, modes 0, 2, 3 and 4 code with the
// warp-specialised compressor; without one (the allocation-free entry point,
// modes 0 to 3 only) the one-warp compressor codes.
template <int DT>
cudaError_t launch_mode(CompressArgs a, int mode, bool stash, cudaStream_t s) {
    cudaError_t err;
    const uint64_t n = a.n, C = a.num_chunks;
    int sms = 0, per_sm = 0;
    a.gated = mode == 2 ? 1u : 0u;
    if (mode == 2 && n > 0) {
        const uint64_t ns_max = 65536 / Fmt<DT>::kEs;  // 64 KiB of input
        gate_kernel<DT><<<1, 32, kCompressSmem, s>>>(a, uint32_t(n < ns_max ? n : ns_max));
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (mode == 1 || (mode == 2 && n > 0)) {
        if ((err = launch_shape(reinterpret_cast<const void*>(raw_kernel<DT>), 32, 0, &sms, &per_sm)) != cudaSuccess)
            return err;
        uint64_t grid = uint64_t(per_sm) * uint64_t(sms);
        const uint64_t pieces = (n + kRawPiece - 1) / kRawPiece;
        if (grid > pieces) grid = pieces;
        if (grid < 1) grid = 1;
        raw_kernel<DT><<<dim3(uint32_t(grid)), dim3(32), 0, s>>>(a);
        if ((err = cudaGetLastError()) != cudaSuccess || mode == 1) return err;
    }
    if ((mode == 0 || mode == 2) && stash && C > 0) return launch_ws<DT, 0>(a, s);
    if (mode == 3 && stash && C > 0) return launch_ws<DT, 1>(a, s);
    if (mode == 4) {
        if (C == 0) mode = 0;  // no chunk: the header alone
        else if (stash) return launch_ws<DT, 2>(a, s);
        else return cudaErrorInvalidValue;
    }
    void (*kern)(CompressArgs) = mode == 3 ? compress_kernel<DT, true> : compress_kernel<DT, false>;
    if ((err = launch_shape(reinterpret_cast<const void*>(kern), 32, kCompressSmem, &sms, &per_sm)) != cudaSuccess)
        return err;
    uint64_t grid = uint64_t(per_sm) * uint64_t(sms);
    const uint64_t work = C > a.first_ticket ? C - a.first_ticket : 1;
    if (grid > work) grid = work;
    if (stash && grid > stash_warps(n)) grid = stash_warps(n);  // two slots per warp
    if (grid < 1) grid = 1;
    // As few warps as give the same number of rounds of chunks, so that the
    // last round is (nearly) full: 8192 chunks take 7 rounds of 1171 warps
    // rather than 6.7 of 1216.
    const uint64_t rounds = (work + grid - 1) / grid;  // work >= 1, grid >= 1
    grid = (work + rounds - 1) / rounds;
    kern<<<dim3(uint32_t(grid)), dim3(32), kCompressSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace uzip
