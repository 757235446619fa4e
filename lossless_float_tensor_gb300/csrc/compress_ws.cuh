// Warp-specialised compressor (included by compress_fmt_*.cu after
// compress_kernels.cuh, one element format each).
//
// One block per SM: kWsEnc encoder warps (two per scheduler) and kWsHelp
// helper warps, helper h serving encoders h and h + 4.  A helper splits a
// chunk (UCCL-Zip Fig. 2: exponent field vs sign and fraction): it writes the
// sign|fraction fields straight to the remainder plane, the exponent bytes to
// one of its encoder's two contexts in the slot area, counts them in a
// lane-column histogram, normalises the counts (largest remainder, M = 4096)
// and builds the encode table (UCCL-Zip Fig. 5: every block builds its own
// table, so no statistics cross blocks).  The encoder only runs the 32-state
// interleaved rANS coder: exponent bytes come back from the context into a
// shared-memory ring through bulk copies (cp.async.bulk, mbarrier completion),
// the 16-bit words go to a shared-memory ring and leave through bulk stores
// into the same context, from its end down, over exponent bytes already read.
// When a chunk is coded the encoder publishes its length for the decoupled
// look-back (Merrill and Garland, "Single-pass parallel prefix scan with
// decoupled look-back", 2016); the helper, while the encoder codes its other
// context, resolves the chunk's offset and copies the record to its place.  A
// chunk that coding does not shrink is written RAW from the input (NCCLZ
// Sec. IV-C).  A helper starts splitting an encoder's next chunk only once the
// encoder is well into its current one, so few contexts are held in L2 at a
// time.
//
// Table modes (template parameter TM): 0 counts every exponent of the chunk;
// 1 counts those at positions 0, 16, 32, ... and normalises 16 x the sample
// counts, every unseen symbol of the format's range counting 1; 2 counts
// nothing and normalises the caller's Gaussian-model counts (ZipCCL
// abstract), the same for every chunk.
#pragma once

#include "compress_kernels.cuh"

namespace uzip {

// ---- block layout -------------------------------------------------------------
// per encoder (kWsTeamSmem bytes):
//   [0, 4 KiB)        exponent-byte ring: 4 blocks of 32 steps x 32 lanes
//   [4 KiB, 8 KiB)    word ring: the record's tail, bytes at (offset in the
//                     context) mod 4096
//   [8 KiB, 12 KiB)   encode tables of the two contexts, 8 bytes per symbol:
//                     {m_lo, (4096 - f) << 20 | cum << 8 | sh}
//   [12 KiB, +1152)   per-context chunk description (kWsMeta*)
//   [13440, +64)      mbarriers: ring blocks 0..3, ready[2], coded[2]
//   [13504]           encoder progress (iteration << 16 | block); [13508]
//                     sink for the word stores of lanes that do not emit
// per helper (kWsHelperSmem bytes): histogram u32[256][16] (16 KiB, column =
// lane mod 16; lanes l and l + 16 share a column, the increments are atomic),
// normalisation scratch (2 KiB)
constexpr uint32_t kWsHelp = kWsEnc / 2;
constexpr uint32_t kWsRing = 4096;
constexpr uint32_t kWsWordRing = 4096;
constexpr uint32_t kWsTables = kWsRing + kWsWordRing;
constexpr uint32_t kWsFlushAt = 2032;  // unflushed word bytes that start a flush
// a block writes at most 2 KiB of words; with no flush pending the ring must
// hold them beside the words not yet flushed (under kWsFlushAt + 16 bytes)
static_assert(kWsFlushAt + 16 + 2048 <= kWsWordRing, "word ring too small for the flush threshold");
constexpr uint32_t kWsTableBytes = 2048;  // one context's table
constexpr uint32_t kWsMeta = kWsTables + 2 * kWsTableBytes;
constexpr uint32_t kWsMetaBytes = 576;
constexpr uint32_t kWsBars = kWsMeta + 2 * kWsMetaBytes;
constexpr uint32_t kWsProgress = kWsBars + 64;
constexpr uint32_t kWsTeamSmem = kWsProgress + 64;
constexpr uint32_t kWsHist = kRegionA;
constexpr uint32_t kWsHelperSmem = kWsHist + kRegionB;
constexpr uint32_t kWsSmem = kWsEnc * kWsTeamSmem + kWsHelp * kWsHelperSmem;
constexpr uint32_t kWsThreads = (kWsEnc + kWsHelp) * 32;
// chunk description fields (byte offsets in a context's kWsMetaBytes)
constexpr uint32_t kMetaChunk = 0, kMetaNc = 4, kMetaK = 8, kMetaFlags = 12, kMetaLen = 16, kMetaRaw = 20,
                   kMetaErr = 24, kMetaSlow = 28, kMetaBitmap = 32, kMetaFreq = 64;
constexpr uint32_t kMetaStop = 1;

__device__ const Magic33Table g_magic33 = make_magic33_table();

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ void red_shared_inc(uint32_t addr) {
    asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr) : "memory");
}
// The encoder's shared-memory accesses are inline asm whose order the
// compiler may change: loads are side-effect free (not volatile), so the
// loads of later steps can be issued ahead of the stores of earlier ones (the
// step chain would otherwise wait for two dependent load latencies per step),
// and the word store is volatile but has no memory clobber.  What they must
// not cross is made explicit: every base address they use comes out of
// opaque() after the wait that made its data valid, and the waits, warp syncs
// and bulk copies around them are volatile asm, which keep their order.
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts_u16_s(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(static_cast<unsigned short>(v)));
}
__device__ __forceinline__ uint32_t opaque(uint32_t v) {
    asm volatile("mov.b32 %0, %1;" : "=r"(v) : "r"(v));
    return v;
}
__device__ __forceinline__ void warp_sync_asm() { asm volatile("bar.warp.sync 0xffffffff;" ::: "memory"); }

// Bounded wait on an mbarrier phase (every lane polls); false if it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------------------
// helper: plane split + exponent bytes + histogram (column = lane)

// The pass over one chunk for formats with whole-byte fields.  A unit is 16
// consecutive values of one lane: its remainder bytes and its 16 exponent
// bytes leave as 16-byte stores; every exponent increments row e, column
// lane mod 16 of the histogram (red.shared).  CM 2 (sampled tables): only the
// exponents at positions 0, 16, 32, ... of the chunk are counted, i.e. each
// unit's first; CM 0 (parametric tables): none.
// bring [p, p + bytes) into L2 (p and bytes multiples of 16; a hint, no data returned)
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// batches of the fp32 split's loads pulled into L2 ahead of the batch being
// read (1, 2 and 3 measured alike on c3; 4: 1 % slower, 8: 5 %)
constexpr uint32_t kWsSplitAhead = 2;
template <int DT, int CM = 1>
__device__ void ws_split_bytes(const uint8_t* __restrict__ cin, uint32_t n_c, uint8_t* __restrict__ rem_dst,
                               uint8_t* __restrict__ ex_dst, uint32_t hist_s, uint32_t lane, uint64_t pol) {
    constexpr uint32_t es = Fmt<DT>::kEs;
    constexpr uint32_t PV = es == 4 ? 4 : 2;  // 16-byte vectors per unit
    const uint32_t lane4 = 4 * (lane & 15u);  // histogram column
    const uint32_t nunits = n_c / 16;
    auto process = [&](const uint4 (&q)[PV], uint32_t unit) {
        uint32_t r[4 * (es - 1)], ex[4];
        if constexpr (es == 2) {
            // two bf16 values per word: low byte of each value = exponent bit 0
            // | fraction, high byte = sign | exponent >> 1
            const uint32_t w[8] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w};
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t a = w[2 * g], b = w[2 * g + 1];
                const uint32_t lo = prmt(a, b, 0x6420);  // low bytes of the four values
                const uint32_t sg = prmt(a, b, 0xFDB9);  // high bytes, sign replicated
                r[g] = (lo & 0x7F7F7F7Fu) | (sg & 0x80808080u);
                ex[g] = prmt(a << 1, b << 1, 0x7531);
                if (CM == 1 || (CM == 2 && g == 0)) red_shared_inc(hist_s + (((a >> 1) & 0x3FC0u) | lane4));
                if (CM == 1) {
                    red_shared_inc(hist_s + (((a >> 17) & 0x3FC0u) | lane4));
                    red_shared_inc(hist_s + (((b >> 1) & 0x3FC0u) | lane4));
                    red_shared_inc(hist_s + (((b >> 17) & 0x3FC0u) | lane4));
                }
            }
            st_v4_hint(rem_dst + uint64_t(unit) * 16, make_uint4(r[0], r[1], r[2], r[3]), pol);
        } else {
            // fp32: bytes 0, 1 pass through; byte 2 keeps its low 7 bits and
            // takes the sign; the exponent is byte 3 << 1 | byte 2 >> 7
            const uint32_t w[16] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w,
                                    q[2].x, q[2].y, q[2].z, q[2].w, q[3].x, q[3].y, q[3].z, q[3].w};
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t a = w[4 * g], b = w[4 * g + 1], c = w[4 * g + 2], d = w[4 * g + 3];
                const uint32_t b2 = prmt(prmt(a, b, 0x0062), prmt(c, d, 0x0062), 0x5410);
                const uint32_t b3 = prmt(prmt(a, b, 0x0073), prmt(c, d, 0x0073), 0x5410);
                const uint32_t t = (b2 & 0x7F7F7F7Fu) | (b3 & 0x80808080u);
                ex[g] = ((b3 << 1) & 0xFEFEFEFEu) | ((b2 >> 7) & 0x01010101u);
                r[3 * g] = prmt(prmt(a, t, 0x0410), b, 0x4210);      // a0 a1 t0 b0
                r[3 * g + 1] = prmt(prmt(b, t, 0x0051), c, 0x5410);  // b1 t1 c0 c1
                r[3 * g + 2] = prmt(d, t, 0x7106);                   // t2 d0 d1 t3
                if (CM == 1 || (CM == 2 && g == 0)) red_shared_inc(hist_s + (((a >> 17) & 0x3FC0u) | lane4));
                if (CM == 1) {
                    red_shared_inc(hist_s + (((b >> 17) & 0x3FC0u) | lane4));
                    red_shared_inc(hist_s + (((c >> 17) & 0x3FC0u) | lane4));
                    red_shared_inc(hist_s + (((d >> 17) & 0x3FC0u) | lane4));
                }
            }
            uint8_t* dr = rem_dst + uint64_t(unit) * 48;
#pragma unroll
            for (int k = 0; k < 3; ++k)
                st_v4_hint(dr + 16 * k, make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]), pol);
        }
        *reinterpret_cast<uint4*>(ex_dst + 16 * uint64_t(unit)) = make_uint4(ex[0], ex[1], ex[2], ex[3]);
    };
    auto load_unit = [&](uint4 (&q)[PV], uint32_t unit) {
#pragma unroll
        for (int v = 0; v < int(PV); ++v) q[v] = ld_v4_hint(cin + (uint64_t(unit) * PV + v) * 16, pol);
    };
    // batches of U units per lane, each unit's registers refilled with the
    // next batch's unit as soon as it is processed
    constexpr int U = es == 4 ? 4 : 8;  // 8 KiB of loads in flight per warp
    const uint32_t nb = nunits / (32 * U);
    const uint32_t head = nunits - nb * 32 * U;
    for (uint32_t u = lane; u < head; u += 32) {
        uint4 q[PV];
        load_unit(q, u);
        process(q, u);
    }
    uint4 qa[U][PV];
    auto unit_of = [&](uint32_t k, int u) -> uint32_t { return head + k * 32 * U + 32 * u + lane; };
    // fp32: a chunk is 256 KiB of input read with only 8 KiB in flight, so
    // the split, not the encoder, bounds the kernel; batches kWsSplitAhead
    // ahead are pulled into L2 by one bulk prefetch each (for bf16 and the
    // packed formats the same prefetch measured slower: their helpers keep
    // up, and it only adds to the DRAM traffic the encoders wait on)
    constexpr uint32_t kBatchBytes = 32 * U * PV * 16;
    auto prefetch_batch = [&](uint32_t k) {
        if (es == 4 && lane == 0 && k < nb)
            prefetch_l2_bulk(cin + (uint64_t(head) * PV + uint64_t(k) * 32 * U * PV) * 16, kBatchBytes);
    };
    for (uint32_t k = 1; k < kWsSplitAhead; ++k) prefetch_batch(k);
    if (nb > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) load_unit(qa[u], unit_of(0, u));
    }
#pragma unroll 1
    for (uint32_t k = 0; k < nb; ++k) {
        prefetch_batch(k + kWsSplitAhead);
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
        if (CM == 1 || (CM == 2 && (i & 15u) == 0)) red_shared_inc(hist_s + ((e << 6) | lane4));
        ex_dst[i] = uint8_t(e);
    }
}

// The same pass for formats whose sign|fraction field is not a whole number
// of bytes (fp16: 11 bits, fp8 e4m3fn: 4, e5m2: 3): a unit is 32 values, whose
// W-bit fields pack into exactly W 32-bit words, least significant bit first.
// CM 2: only the unit's values 0 and 16 are counted; CM 0: none.
template <int DT, int CM = 1>
__device__ void ws_split_packed(const uint8_t* __restrict__ cin, uint32_t n_c, uint8_t* __restrict__ rem_dst,
                                uint8_t* __restrict__ ex_dst, uint32_t hist_s, uint32_t lane, uint64_t pol) {
    constexpr uint32_t es = Fmt<DT>::kEs, mb = Fmt<DT>::kMbits, W = Fmt<DT>::kRbits;
    const uint32_t lane4 = 4 * (lane & 15u);  // histogram column
    constexpr uint32_t PV = 2 * es;  // 16-byte vectors per 32-value unit
    const uint32_t nunits = n_c / 32;
    auto count = [&](uint32_t e64) { red_shared_inc(hist_s + (e64 | lane4)); };
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
                if (CM == 1 || (CM == 2 && (j == 0 || j == 8))) count((eb << 6) & 0x3FC0u);
                if (CM == 1) count((eb >> 10) & 0x3FC0u);
                f[2 * j] = Traits<DT>::rem_of(w[j] & 0xFFFFu);
                f[2 * j + 1] = Traits<DT>::rem_of(w[j] >> 16);
                if (j & 1) ex[j >> 1] = __byte_perm((w[j - 1] >> mb) & em2, eb, 0x6420);
            }
        } else {
            constexpr uint32_t em4 = Traits<DT>::kEmask * 0x01010101u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                ex[j] = (w[j] >> mb) & em4;
                if (CM == 1 || (CM == 2 && (j == 0 || j == 4))) count((ex[j] << 6) & 0x3FC0u);
                if (CM == 1) {
                    count((ex[j] >> 2) & 0x3FC0u);
                    count((ex[j] >> 10) & 0x3FC0u);
                    count((ex[j] >> 18) & 0x3FC0u);
                }
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
        for (uint32_t k = 0; k < W; ++k) st_u32_hint(rd + k, o[k], pol);
        reinterpret_cast<uint4*>(ex_dst + 32 * uint64_t(unit))[0] = make_uint4(ex[0], ex[1], ex[2], ex[3]);
        reinterpret_cast<uint4*>(ex_dst + 32 * uint64_t(unit))[1] = make_uint4(ex[4], ex[5], ex[6], ex[7]);
    };
    auto load_unit = [&](uint4 (&q)[PV], uint32_t unit) {
#pragma unroll
        for (int v = 0; v < int(PV); ++v) q[v] = ld_v4_hint(cin + (uint64_t(unit) * PV + v) * 16, pol);
    };
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
    if (nb > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) load_unit(qa[u], unit_of(0, u));
    }
#pragma unroll 1
    for (uint32_t k = 0; k < nb; ++k) {
        const bool more = k + 1 < nb;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            process(qa[u], unit_of(k, u));
            if (more) load_unit(qa[u], unit_of(k + 1, u));
        }
    }
    // ragged tail (fewer than 32 values): its fields start byte aligned; lane
    // 0 packs them, the lanes count and copy the exponents
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
            if (CM == 1 || (CM == 2 && (i & 15u) == 0)) count(e << 6);
            ex_dst[i] = uint8_t(e);
        }
    }
}

// Encode table of one context (8 bytes per present symbol) and the chunk
// description's bitmap and frequency list.
inline __device__ void ws_build_table(const Norm& nm, uint32_t lane, uint32_t table_s, uint8_t* meta) {
    uint32_t lsum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) lsum += nm.f[k];
    uint32_t dummy;
    uint32_t cum = warp_excl_scan(lsum, lane, &dummy);
    uint16_t* fl = reinterpret_cast<uint16_t*>(meta + kMetaFreq);
    uint32_t idx = nm.prefix;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t f = nm.f[k];
        if (nm.present & (1u << k)) {
            const Magic33 mg = g_magic33.e[f];
            const uint32_t pk = ((kM - f) << 20) | (cum << 8) | mg.sh;
            asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(table_s + 8 * (8 * lane + k)), "r"(mg.m_lo), "r"(pk)
                         : "memory");
            fl[idx++] = uint16_t(f);
        }
        cum += f;
    }
    meta[kMetaBitmap + lane] = uint8_t(nm.present);
    if (lane == 0) *reinterpret_cast<uint32_t*>(meta + kMetaK) = nm.k_total;
}

// ---------------------------------------------------------------------------
// chunk placed: chunk-table entries, progress, done counter; the warp that
// completes the last chunk writes the header.  Returns true for that warp.
template <int DT>
__device__ bool ws_complete(const CompressArgs& a, uint32_t c, uint32_t len, bool raw, uint64_t excl, bool ok,
                            uint32_t lane, uint32_t processed) {
    const uint64_t C = a.num_chunks;
    if (!ok && lane == 0) atomicCAS(&a.scratch->status, 0u, uint32_t(UZIP_ERR_TIMEOUT));
    if (ok && lane == 0) {
        reinterpret_cast<uint64_t*>(a.out + kHeader)[c] = excl;
        reinterpret_cast<uint32_t*>(a.out + kHeader + 8 * C)[c] = len | (raw ? kRawFlag : 0u);
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
        uint64_t total = exp_offset(DT, a.n) + (last & kDescValue);
        if (st != 0 || (last >> 62) != 2) total = 0;
        write_header<DT>(a, total, st);
    }
    return true;
}

// In-place coding of a chunk straight from the input, by one warp: a first
// pass (the encoder's) only counts the words, stopping as soon as the chunk
// would be stored RAW; once the offset is known a second pass (the
// helper's) writes each word at its place in the record.  Used for the rare chunk whose words would have
// reached exponent bytes not yet read back.  Returns the word count W (or
// kRawFlag for RAW); WRITE writes the words to `words` (u16, W of them) and
// leaves the final states in x.
template <int DT, bool WRITE>
__device__ uint32_t ws_direct(const uint8_t* __restrict__ cin, uint32_t n_c, uint32_t table_s, uint32_t hdr,
                              uint32_t lane, uint16_t* words, uint32_t W, uint32_t& x) {
    const uint32_t lt = lanemask_lt();
    x = kRansL;
    uint32_t cnt = 0;
    int32_t pos = int32_t(W);
    auto step = [&](int32_t t, uint32_t e) {
        const bool active = 32 * uint32_t(t) + lane < n_c;
        uint32_t mlo, pk;
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(mlo), "=r"(pk) : "r"(table_s + 8 * e));
        const bool emit = active && x > (~pk | 0xFFFFFu);
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, emit);
        const uint32_t nt = __popc(b);
        if (WRITE && emit) words[pos - int32_t(nt) + int32_t(__popc(b & lt))] = uint16_t(x);
        pos -= int32_t(nt);
        cnt += nt;
        const uint32_t xr = emit ? x >> 16 : x;
        const uint32_t q = __funnelshift_r(__umulhi(xr, mlo) + xr, 0u, pk);
        const uint32_t xn = q * (pk >> 20) + xr + ((pk >> 8) & 0xFFFu);
        x = active ? xn : x;
    };
    auto exp_at = [&](int32_t t) -> uint32_t {
        const uint32_t i = 32 * uint32_t(t) + lane;
        return t >= 0 && i < n_c ? Traits<DT>::exp_of(Traits<DT>::load(cin, i)) : 0u;
    };
    // groups of 8 steps whose input loads are issued first; the count only
    // grows, so testing for RAW after each group decides as testing after
    // each step would
    constexpr int G = 8;
    for (int32_t t0 = int32_t((n_c + 31) / 32) - 1; t0 >= 0; t0 -= G) {
        uint32_t e[G];
#pragma unroll
        for (int k = 0; k < G; ++k) e[k] = exp_at(t0 - k);
#pragma unroll
        for (int k = 0; k < G; ++k)
            if (t0 - k >= 0) step(t0 - k, e[k]);
        if (!WRITE && hdr + 2 * cnt >= n_c) return kRawFlag;
    }
    return cnt;
}

// Places the chunk of one context: offset from the look-back, then the record
// (or, for a RAW chunk, the exponent bytes from the input) copied to it.
template <int DT>
__device__ void ws_place(const CompressArgs& a, uint8_t* meta, uint8_t* ctx, uint32_t table_s, uint32_t lane,
                         uint32_t processed, uint64_t pol) {
    const uint32_t c = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaChunk);
    const uint32_t n_c = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaNc);
    uint32_t len = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaLen);
    bool raw = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaRaw) != 0;
    const bool err = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaErr) != 0;
    const bool slow = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaSlow) != 0;
    const uint8_t* cin = a.in + uint64_t(c) * kChunk * Fmt<DT>::kEs;
    const uint32_t K = *reinterpret_cast<const volatile uint32_t*>(meta + kMetaK);
    const uint32_t hdr = kStreamHead + 2 * K;
    const uint32_t W = (len - hdr) / 2;  // a slow chunk's word count (the encoder counted it)
    uint32_t x = kRansL;
    uint64_t excl = 0;
    bool ok = resolve_offset(a.desc, c, round16(len), lane, excl) && !err;
    if (ok) {
        uint8_t* dst = a.out + exp_offset(DT, a.n) + excl;
        if (raw) {
            write_raw<DT>(cin, n_c, dst, lane);
        } else if (slow) {  // write the words in place from the input
            ws_direct<DT, true>(cin, n_c, table_s, hdr, lane, reinterpret_cast<uint16_t*>(dst + hdr), W, x);
            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
            d16[2 * lane] = uint16_t(x);
            d16[2 * lane + 1] = uint16_t(x >> 16);
            if (lane < 16) d16[64 + lane] = uint16_t(meta[kMetaBitmap + 2 * lane] | (meta[kMetaBitmap + 2 * lane + 1] << 8));
            const uint16_t* fl = reinterpret_cast<const uint16_t*>(meta + kMetaFreq);
            for (uint32_t i = lane; i < K; i += 32) d16[80 + i] = fl[i];
            for (uint32_t i = len + lane; i < round16(len); i += 32) dst[i] = 0;
        } else {
            copy_record_from_slot(ctx, kSlotBytes - len, dst, lane, pol, kSlotBytes);
        }
    }
    __syncwarp();
    if (!raw && !slow) {  // the record's lines are spent
        for (uint32_t l = (kSlotBytes - len) / 128 + lane; l < kSlotBytes / 128; l += 32) l2_discard_line(ctx + 128 * l);
    }
    __syncwarp();
    ws_complete<DT>(a, c, len, raw, excl, ok, lane, processed);
}

// Helper h serves encoders h and h + kWsHelp in turn: for each of its
// encoders' contexts in order, place the chunk the context held, wait until
// the encoder is far enough into its other context, take the next chunk,
// split it into the context and mark it ready.
template <int DT, int TM>
__device__ void ws_helper(const CompressArgs& a, uint8_t* smem, uint32_t h, uint32_t lane) {
    const uint32_t C = a.num_chunks;
    const uint32_t processed = C - a.first_ticket;
    const uint64_t pol = policy_evict_first();
    const uint64_t rem_off = rem_offset(a.n);
    uint8_t* hsm = smem + kWsEnc * kWsTeamSmem + h * kWsHelperSmem;
    const uint32_t hist_s = smem_u32(hsm);
    uint8_t* regB = hsm + kWsHist;
    bool stopped[2] = {false, false};
    for (uint32_t k = 0; !(stopped[0] && stopped[1]); ++k) {
        const uint32_t side = k & 1u;
        if (stopped[side]) continue;
        const uint32_t e = h + side * kWsHelp;  // encoder
        const uint32_t it = k >> 1;             // that encoder's iteration
        const uint32_t cx = it & 1u;
        uint8_t* team = smem + e * kWsTeamSmem;
        const uint32_t bars = smem_u32(team + kWsBars);
        uint8_t* ctx0 = a.stash + (uint64_t(blockIdx.x) * kWsEnc + e) * 2 * kSlotBytes;
        uint8_t* meta = team + kWsMeta + cx * kWsMetaBytes;
        uint8_t* ctx = ctx0 + uint64_t(cx) * kSlotBytes;
        const uint32_t table_s = smem_u32(team + kWsTables + cx * kWsTableBytes);
        if (it >= 2) {  // the context's previous chunk: coded, then placed
            if (!mbar_wait(bars + 48 + 8 * cx, ((it - 2) >> 1) & 1u)) {
                if (lane == 0) atomicCAS(&a.scratch->status, 0u, uint32_t(UZIP_ERR_TIMEOUT));
                return;
            }
            ws_place<DT>(a, meta, ctx, table_s, lane, processed, pol);
        }
        if (it >= 1 && a.jit_blocks < 64) {  // wait until the encoder is far enough into chunk it - 1
            const volatile uint32_t* progress = reinterpret_cast<const volatile uint32_t*>(team + kWsProgress);
            for (uint32_t i = 0; i < kSpinLimit; ++i) {
                const uint32_t p = *progress;
                if ((p >> 16) > it - 1 || ((p >> 16) == it - 1 && (p & 0xFFFFu) <= a.jit_blocks)) break;
                __nanosleep(200);
            }
        }
        uint32_t c = 0;
        if (lane == 0) c = atomicAdd(&a.scratch->ticket, 1u) + a.first_ticket;
        c = __shfl_sync(0xFFFFFFFFu, c, 0);
        if (c >= C) {
            if (lane == 0) *reinterpret_cast<volatile uint32_t*>(meta + kMetaFlags) = kMetaStop;
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 32 + 8 * cx);
            stopped[side] = true;
            if (it >= 1) {  // the other context's chunk is still to be placed
                const uint32_t ox = cx ^ 1u;
                if (!mbar_wait(bars + 48 + 8 * ox, ((it - 1) >> 1) & 1u)) {
                    if (lane == 0) atomicCAS(&a.scratch->status, 0u, uint32_t(UZIP_ERR_TIMEOUT));
                    return;
                }
                ws_place<DT>(a, team + kWsMeta + ox * kWsMetaBytes, ctx0 + uint64_t(ox) * kSlotBytes,
                             smem_u32(team + kWsTables + ox * kWsTableBytes), lane, processed, pol);
            }
            continue;
        }
        const uint64_t left = a.n - uint64_t(c) * kChunk;
        const uint32_t n_c = uint32_t(left < kChunk ? left : kChunk);
        const uint8_t* cin = a.in + uint64_t(c) * kChunk * Fmt<DT>::kEs;
        if constexpr (TM != 2) {  // the histogram the split counts into
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 8
            for (uint32_t i = lane; i < kWsHist / 16; i += 32) reinterpret_cast<uint4*>(hsm)[i] = z;
        }
        __syncwarp();
        uint8_t* rem_dst = a.out + rem_off + uint64_t(c) * Fmt<DT>::kRemChunk;
        constexpr int CM = TM == 0 ? 1 : (TM == 1 ? 2 : 0);  // which exponents the histogram counts
        if constexpr (Fmt<DT>::kPacked) ws_split_packed<DT, CM>(cin, n_c, rem_dst, ctx, hist_s, lane, pol);
        else ws_split_bytes<DT, CM>(cin, n_c, rem_dst, ctx, hist_s, lane, pol);
        __syncwarp();
        if (a.progress) post_progress(a.progress + 2 * uint64_t(c), 1, lane);
        uint32_t cnt[8];
        if constexpr (TM != 2) reduce_hist(hsm, lane, cnt);
        Norm nm;
        uint32_t total = n_c;  // the counts' total
        if constexpr (TM == 2) {  // the model's counts, the same for every chunk
#pragma unroll
            for (int k = 0; k < 8; ++k) cnt[k] = a.model[8 * lane + k];
            total = a.model_total;
        }
        if constexpr (TM == 1) {  // a seen symbol counts 16 x, an unseen one of the format's range 1
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
        normalise<TM != 0>(cnt, total, lane, regB, nm);
        ws_build_table(nm, lane, table_s, meta);
        if (lane == 0) {
            *reinterpret_cast<volatile uint32_t*>(meta + kMetaChunk) = c;
            *reinterpret_cast<volatile uint32_t*>(meta + kMetaNc) = n_c;
            *reinterpret_cast<volatile uint32_t*>(meta + kMetaFlags) = 0;
        }
        fence_async_global();  // the exponent bytes are read back by bulk copies
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 32 + 8 * cx);
    }
}

// ---------------------------------------------------------------------------
// encoder

// One rANS encode step (rule R6) of one lane: the table entry of its symbol is
// {m_lo, pk = (4096 - f) << 20 | cum << 8 | sh}.  It renormalises when x
// exceeds f << 20 - 1 = ~pk | 0xFFFFF; the quotient floor(x / f) is
// (umulhi(x, m_lo) + x) >> sh (magic33); the new state is
// q (4096 - f) + x + cum.  A renormalising lane
// puts its word at dp + 2 * (its rank among the renormalising lanes), dp
// having moved down by 2 per renormalising lane, so each step's words sit in
// ascending lane order and the steps below the later ones (decoder order).
//
// A warp issues in order, and the word's address needs the step's ballot, so
// storing it at once would hold back everything after it: the words of step
// j are placed two steps later (ws_words), when the ballot is long known.
struct WsEnc {
    uint32_t x;        // this lane's state
    uint32_t dp;       // context offset of the lowest word written so far (same in every lane)
    uint32_t ring_s;   // word ring
    uint32_t lt;       // lanes below this one
    uint32_t sink_s;   // a word no one reads: the store target of lanes that do not renormalise
};
// the words of an earlier step: its ballot, this lane's old state, whether it renormalised
struct WsPending {
    uint32_t b, w;
    bool e;
};
__device__ __forceinline__ void ws_words(WsEnc& st, const WsPending& p) {
    st.dp -= 2 * __popc(p.b);
    const uint32_t wa = st.ring_s + ((st.dp + 2 * __popc(p.b & st.lt)) & (kWsWordRing - 1));
    sts_u16_s(p.e ? wa : st.sink_s, p.w);  // every lane stores: a store under `if` is a divergent branch
}
__device__ __forceinline__ uint2 ws_entry(uint32_t ex_s, uint32_t table_s) {
    const uint32_t e = lds_u8(ex_s);
    uint2 t;
    asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(t.x), "=r"(t.y) : "r"(table_s + 8 * e));
    return t;
}
// The state update of one step given its table entry; returns the words to
// place later.
__device__ __forceinline__ WsPending ws_update(WsEnc& st, const uint2 t, bool active) {
    const bool emit = active && st.x > (~t.y | 0xFFFFFu);
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, emit);
    const uint32_t w = st.x;
    const uint32_t xr = emit ? st.x >> 16 : st.x;
    uint32_t th;  // high word of xr (2^32 + m_lo): umulhi(xr, m_lo) + xr
    asm("mad.hi.u32 %0, %1, %2, %1;" : "=r"(th) : "r"(xr), "r"(t.x));
    const uint32_t q = __funnelshift_r(th, 0u, t.y);  // >> sh (low 5 bits of pk)
    const uint32_t xn = q * (t.y >> 20) + xr + ((t.y >> 8) & 0xFFFu);
    st.x = active ? xn : st.x;
    return WsPending{b, w, emit};
}
// one step, words placed at once (the partial top block of a short chunk)
__device__ __forceinline__ void ws_step(WsEnc& st, uint32_t ex_s, uint32_t table_s, bool active) {
    ws_words(st, ws_update(st, ws_entry(ex_s, table_s), active));
}
// 32 full steps of one block (step 31 - j of the block at j).  A step's word
// store would keep the shared loads of the steps after it from being issued
// earlier (the compiler cannot tell the addresses apart), so the entries are
// loaded kWsAhead steps ahead in program order, before the stores they would
// otherwise wait for.  12 measured best on c4 (0.877 ms; 4: 0.896, 8: 0.882,
// 16: 0.880).
constexpr int kWsAhead = 12;
__device__ __forceinline__ void ws_block(WsEnc& st, uint32_t ex0, uint32_t table_s) {
    uint2 t[kWsAhead];
#pragma unroll
    for (int k = 0; k < kWsAhead; ++k) t[k] = ws_entry(ex0 + 32 * (31 - k), table_s);
    WsPending p1{0, 0, false}, p2{0, 0, false};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint2 cur = t[j % kWsAhead];
        if (j + kWsAhead < 32) t[j % kWsAhead] = ws_entry(ex0 + 32 * (31 - (j + kWsAhead)), table_s);
        const WsPending p = ws_update(st, cur, true);
        if (j >= 2) ws_words(st, p2);
        p2 = p1;
        p1 = p;
    }
    ws_words(st, p2);
    ws_words(st, p1);
}

// Codes the chunk of one context.  Writes len, raw, slow and err into its
// description and publishes the padded length.  The words go to the context
// from its end (kSlotBytes) down, over exponent bytes already read back; a
// flush that would reach bytes still to be read (a stream growing faster
// than 8 bits per value for a while) stops the encoder instead: it counts
// that chunk's words from the input, and the helper writes them in place.
template <int DT>
__device__ void ws_encode(const CompressArgs& a, uint8_t* team, uint32_t cx, uint32_t it, uint8_t* ctx, uint32_t lane,
                          uint32_t& ring_ph) {
    uint8_t* meta = team + kWsMeta + cx * kWsMetaBytes;
    const uint32_t c = *reinterpret_cast<volatile uint32_t*>(meta + kMetaChunk);
    const uint32_t n_c = *reinterpret_cast<volatile uint32_t*>(meta + kMetaNc);
    const uint32_t K = *reinterpret_cast<volatile uint32_t*>(meta + kMetaK);
    const uint32_t hdr = kStreamHead + 2 * K;
    const uint32_t ring_s = smem_u32(team);
    const uint32_t table_s = opaque(smem_u32(team + kWsTables + cx * kWsTableBytes));  // built before the ready wait
    const uint32_t bars = smem_u32(team + kWsBars);
    volatile uint32_t* progress = reinterpret_cast<volatile uint32_t*>(team + kWsProgress);
    const int32_t T = int32_t((n_c + 31) / 32);
    const int32_t bt = (T - 1) / 32;               // top block
    const bool partial_top = (n_c & 1023u) != 0;  // the top block has fewer than 32 full steps
    auto issue = [&](int32_t b) {                  // block b's 1 KiB of exponent bytes into ring slot b & 3
        if (lane == 0) {
            const uint32_t bar = bars + 8 * (uint32_t(b) & 3u);
            mbar_expect_tx(bar, 1024);
            bulk_g2s(ring_s + (uint32_t(b) & 3u) * 1024, ctx + 1024 * uint32_t(b), 1024, bar);
        }
    };
    for (int32_t i = 0; i < 3 && bt - i >= 0; ++i) issue(bt - i);
    int32_t issued_lo = bt - 2 > 0 ? bt - 2 : 0;  // lowest block issued
    WsEnc st{kRansL, kSlotBytes, smem_u32(team + kWsRing), lanemask_lt(), smem_u32(team + kWsProgress + 4)};
    uint32_t flushed = kSlotBytes;  // context bytes at and above this offset hold flushed (or flushing) words
    uint32_t pend = 0;              // bytes of the last flush, whose reads of the ring may not be done
    bool raw = false, err = false, slow = false;
    auto flush = [&](uint32_t lo) {  // ring lines [lo, flushed) to the context
        warp_sync_asm();
        pend = flushed > lo ? flushed - lo : 0u;
        if (lane == 0 && lo < flushed) {
            fence_async_shared();
            for (uint32_t p = lo; p < flushed;) {
                const uint32_t ro = p & (kWsWordRing - 1);
                uint32_t seg = flushed - p;
                seg = seg < kWsWordRing - ro ? seg : kWsWordRing - ro;
                bulk_s2g(ctx + p, st.ring_s + ro, seg);
                p += seg;
            }
            bulk_commit();
        }
        flushed = lo < flushed ? lo : flushed;
    };
    int32_t b = bt;
    for (; b >= 0; --b) {
        if (lane == 0) *progress = (it << 16) | uint32_t(b);
        const uint32_t rs = uint32_t(b) & 3u;
        if (!mbar_wait(bars + 8 * rs, (ring_ph >> rs) & 1u)) {
            err = true;
            break;
        }
        ring_ph ^= 1u << rs;
        // block b + 1 has been read back; its lines are dropped from L2 unless
        // flushed words may already sit in them (a stream that grows faster
        // than 8 bits a value reaches the block just read: words above
        // `flushed` are in the context, and a discarded line loses them).  A
        // later flush may write a dropped line again; it is issued at the end
        // of a block, thousands of cycles after the drop, which reaches L2
        // first.
        if (b + 1 <= bt && lane < 8) {
            const uint32_t line = 1024 * uint32_t(b + 1) + 128 * lane;
            if (line + 128 <= flushed) l2_discard_line(ctx + line);
        }
        if (b >= 3) {  // block b - 3 goes into the slot block b + 1 has left (its reads are done)
            warp_sync_asm();
            issue(b - 3);
            issued_lo = b - 3;
        }
        // the word ring holds the last flush while its reads are pending
        // (pend bytes, above `flushed`), the words not yet flushed (under
        // kWsFlushAt + 16) and this block's words (at most 2 KiB): every
        // earlier flush must have been read, and the last one too unless all
        // three fit (with kWsFlushAt <= 2032 the last two always do)
        const bool fits = pend + (flushed - st.dp) + 2048 <= kWsWordRing;
        if (lane == 0) {
            if (fits) bulk_wait_read<1>();
            else bulk_wait_read<0>();
        }
        if (!fits) pend = 0;
        warp_sync_asm();
        const uint32_t ex0 = opaque(ring_s + rs * 1024 + lane);  // valid once block b's wait is over
        if (b == bt && partial_top) {
            for (int32_t t = T - 1; t >= 32 * b; --t)
                ws_step(st, ex0 + 32 * uint32_t(t - 32 * b), table_s, uint32_t(t) * 32 + lane < n_c);
        } else {
            ws_block(st, ex0, table_s);
        }
        if (hdr + (kSlotBytes - st.dp) >= n_c) {  // coding does not pay: RAW
            raw = true;
            break;
        }
        const uint32_t lo = (st.dp + 15) & ~15u;
        if (lo < 1024 * uint32_t(b)) {  // the words would overwrite blocks still to be read
            slow = true;
            break;
        }
        if (flushed - lo >= kWsFlushAt) flush(lo);  // fewer, larger flushes: each costs a proxy fence
    }
    // ring blocks issued but not waited for (a chunk cut short) complete first
    for (int32_t bb = (err ? b : b - 1); bb >= issued_lo && bb >= 0; --bb) {
        const uint32_t rs = uint32_t(bb) & 3u;
        if (!mbar_wait(bars + 8 * rs, (ring_ph >> rs) & 1u)) err = true;
        ring_ph ^= 1u << rs;
    }
    uint32_t len = n_c;
    if (!raw && !err && !slow) {
        // stream head below the words: states, bitmap, present frequencies
        const uint32_t rs0 = st.dp - hdr;
        if (lane == 0) bulk_wait_read<0>();
        warp_sync_asm();
        const uint32_t m = kWsWordRing - 1;
        sts_u16_s(st.ring_s + ((rs0 + 4 * lane) & m), st.x & 0xFFFFu);
        sts_u16_s(st.ring_s + ((rs0 + 4 * lane + 2) & m), st.x >> 16);
        if (lane < 16)
            sts_u16_s(st.ring_s + ((rs0 + 128 + 2 * lane) & m),
                      uint32_t(meta[kMetaBitmap + 2 * lane]) | (uint32_t(meta[kMetaBitmap + 2 * lane + 1]) << 8));
        const uint16_t* fl = reinterpret_cast<const uint16_t*>(meta + kMetaFreq);
        for (uint32_t i = lane; i < K; i += 32) sts_u16_s(st.ring_s + ((rs0 + 160 + 2 * i) & m), fl[i]);
        flush(rs0 & ~15u);
        len = kSlotBytes - rs0;
    }
    if (lane == 0) {
        bulk_wait<0>();
        fence_async_global();
    }
    warp_sync_asm();
    // exponent bytes not yet dropped from L2 (a RAW or slow chunk reads its
    // input again instead)
    const uint32_t lines = (raw || err || slow) ? 8 * uint32_t(b + 1) : 8;  // blocks 0..b, or block 0
    for (uint32_t l = lane; l < lines; l += 32) l2_discard_line(ctx + 128 * l);
    if (slow && !err) {  // count the words from the input (the helper writes them in place)
        uint32_t xs;
        const uint32_t W = ws_direct<DT, false>(a.in + uint64_t(c) * kChunk * Fmt<DT>::kEs, n_c, table_s, hdr, lane,
                                                nullptr, 0, xs);
        raw = W == kRawFlag;
        len = raw ? n_c : hdr + 2 * W;
    }
    if (err && lane == 0) atomicCAS(&a.scratch->status, 0u, uint32_t(UZIP_ERR_TIMEOUT));
    publish_length(a.desc, c, round16(len), lane);
    if (lane == 0) {
        *reinterpret_cast<volatile uint32_t*>(meta + kMetaLen) = len;
        *reinterpret_cast<volatile uint32_t*>(meta + kMetaRaw) = raw ? 1u : 0u;
        *reinterpret_cast<volatile uint32_t*>(meta + kMetaErr) = err ? 1u : 0u;
        *reinterpret_cast<volatile uint32_t*>(meta + kMetaSlow) = slow ? 1u : 0u;
    }
}

template <int DT>
__device__ void ws_encoder(const CompressArgs& a, uint8_t* smem, uint32_t e, uint32_t lane) {
    uint8_t* team = smem + e * kWsTeamSmem;
    uint8_t* ctx0 = a.stash + (uint64_t(blockIdx.x) * kWsEnc + e) * 2 * kSlotBytes;
    const uint32_t bars = smem_u32(team + kWsBars);
    volatile uint32_t* progress = reinterpret_cast<volatile uint32_t*>(team + kWsProgress);
    uint32_t ring_ph = 0;
    for (uint32_t it = 0;; ++it) {
        const uint32_t cx = it & 1u;
        if (!mbar_wait(bars + 32 + 8 * cx, (it >> 1) & 1u)) {
            if (lane == 0) atomicCAS(&a.scratch->status, 0u, uint32_t(UZIP_ERR_TIMEOUT));
            return;
        }
        const uint8_t* meta = team + kWsMeta + cx * kWsMetaBytes;
        if (*reinterpret_cast<const volatile uint32_t*>(meta + kMetaFlags) & kMetaStop) return;
        ws_encode<DT>(a, team, cx, it, ctx0 + uint64_t(cx) * kSlotBytes, lane, ring_ph);
        __syncwarp();
        if (lane == 0) {
            *progress = ((it + 1) << 16) | 0xFFFFu;
            mbar_arrive(bars + 48 + 8 * cx);
        }
    }
}

template <int DT, int TM>
__global__ void __launch_bounds__(kWsThreads, 1) compress_ws_kernel(CompressArgs a) {
    extern __shared__ __align__(128) uint8_t ws_smem[];
    uint8_t* smem = ws_smem;
    if (a.gated && *reinterpret_cast<volatile uint32_t*>(&a.scratch->pad) != 0) return;  // the RAW kernel has it
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < kWsEnc && lane == 0) {
        uint8_t* team = smem + warp * kWsTeamSmem;
        const uint32_t bars = smem_u32(team + kWsBars);
        for (uint32_t i = 0; i < 8; ++i) mbar_init(bars + 8 * i, 1);
        *reinterpret_cast<volatile uint32_t*>(team + kWsProgress) = 0xFFFFu;  // iteration 0, not started
        fence_mbar_init();
    }
    __syncthreads();
    if (warp < kWsEnc) ws_encoder<DT>(a, smem, warp, lane);
    else ws_helper<DT, TM>(a, smem, warp - kWsEnc, lane);
}

template <int DT, int TM>
cudaError_t launch_ws(const CompressArgs& a, cudaStream_t s) {
    void (*kern)(CompressArgs) = compress_ws_kernel<DT, TM>;
    cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(kWsSmem));
    if (err != cudaSuccess) return err;
    int sms = 0, per_sm = 0;
    if ((err = launch_shape(reinterpret_cast<const void*>(kern), kWsThreads, kWsSmem, &sms, &per_sm)) != cudaSuccess)
        return err;
    const uint64_t work = a.num_chunks - a.first_ticket;
    uint64_t grid = uint64_t(sms) * uint64_t(per_sm);
    const uint64_t need = (work + kWsFirst - 1) / kWsFirst;
    if (grid > need) grid = need;
    if (grid > ws_ctas(a.n)) grid = ws_ctas(a.n);  // contexts in the slot area
    if (grid < 1) grid = 1;
    kern<<<dim3(uint32_t(grid)), dim3(kWsThreads), kWsSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace uzip
