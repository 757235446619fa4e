/*
 * uzip oracle -- plain single-threaded C implementation of the container.
 *
 * TEST INFRASTRUCTURE ONLY: called by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the library.  It is written for
 * reading, not for speed: every step runs in the order the format states,
 * with plain integer division, and no blocking, vectorisation or fusion.
 *
 * Sources for each step (the pages, then the format readings R1..R20 of the
 * design notes where the pages are silent):
 *   split / merge ........ UCCL-Zip Fig. 2 caption (exponent field vs sign and
 *                          fraction); R1 byte layout of the remainder.
 *   local tables ......... UCCL-Zip Fig. 5 caption (each block builds its own
 *                          table); R3 chunking, R4 histogram, R5 normalisation.
 *   parametric tables .... ZipCCL abstract (exponent coding from the
 *                          Gaussian shape of the values, without online
 *                          statistics); R25 model counts.
 *   entropy coder ........ UCCL-Zip Fig. 2 caption ("ANS"); R6 rANS constants,
 *                          R7 lane interleaving and word order, R8 stream.
 *   RAW fallback ......... NCCLZ Sec. IV-B and IV-C, Alg. 1 (store RAW when
 *                          coding does not pay); R9 threshold.
 *   frame header ......... NCCLZ Sec. IV-B and IV-D2 (self-describing header
 *                          plus payload); R10 padding, R11 header fields.
 *   receiver validation .. NCCLZ Alg. 2 (validate before use); R12 checks.
 */
#include "uzip_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* little-endian helpers (the container is little endian on every host)     */

static uint64_t rd_le(const uint8_t* p, int nbytes) {
    uint64_t v = 0;
    for (int i = nbytes - 1; i >= 0; --i) v = (v << 8) | p[i];
    return v;
}

static void wr_le(uint8_t* p, uint64_t v, int nbytes) {
    for (int i = 0; i < nbytes; ++i) {
        p[i] = (uint8_t)(v & 0xFF);
        v >>= 8;
    }
}

static uint64_t round16(uint64_t v) { return (v + 15u) / 16u * 16u; }

/* ------------------------------------------------------------------------ */
/* R1, R21, R22: split each value into its exponent field and its           */
/* sign|fraction bits, the sign placed just above the fraction.             */
/* bf16    = s | e(8) | m(7):  rem = s<<7 | m    (8-bit field)              */
/* fp32    = s | e(8) | m(23): rem = s<<23 | m   (24-bit field)             */
/* fp16    = s | e(5) | m(10): rem = s<<10 | m   (11-bit field)             */
/* e4m3fn  = s | e(4) | m(3):  rem = s<<3 | m    (4-bit field)              */
/* e5m2    = s | e(5) | m(2):  rem = s<<2 | m    (3-bit field)              */
/* The remainder plane packs the w-bit fields back to back, least          */
/* significant bit first: element i occupies bits [w*i, w*i + w) of the    */
/* plane, bit k of the plane being bit k%8 of byte k/8.  For bf16 and fp32 */
/* this is one byte / three little-endian bytes per element; bits past the */
/* last field are zero.                                                     */

/* (exponent bits, fraction bits, element bytes) of each dtype */
static int layout(int dtype, int* ebits, int* mbits, int* es) {
    switch (dtype) {
        case ORC_BF16: *ebits = 8; *mbits = 7; *es = 2; return 1;
        case ORC_FP32: *ebits = 8; *mbits = 23; *es = 4; return 1;
        case ORC_FP16: *ebits = 5; *mbits = 10; *es = 2; return 1;
        case ORC_FP8_E4M3: *ebits = 4; *mbits = 3; *es = 1; return 1;
        case ORC_FP8_E5M2: *ebits = 5; *mbits = 2; *es = 1; return 1;
        default: return 0;
    }
}

static int dtype_ok(int dtype) {
    int eb, mb, es;
    return layout(dtype, &eb, &mb, &es);
}

/* width of the remainder field: the sign bit and the fraction bits */
static int field_bits(int dtype) {
    int ebits, mbits, es;
    return layout(dtype, &ebits, &mbits, &es) ? 1 + mbits : 0;
}

uint64_t orc_remainder_plane_bytes(int dtype, uint64_t n) {
    return (n * (uint64_t)field_bits(dtype) + 7) / 8;
}

/* remainder field of element i: read / write, bit by bit */
static uint32_t get_rem(int dtype, const uint8_t* rem, uint64_t i) {
    int w = field_bits(dtype);
    uint32_t r = 0;
    for (int k = 0; k < w; ++k) {
        uint64_t bit = (uint64_t)w * i + (uint64_t)k;
        r |= (uint32_t)((rem[bit / 8] >> (bit % 8)) & 1u) << k;
    }
    return r;
}

/* the plane must be zeroed first: fields are ORed in */
static void put_rem(int dtype, uint8_t* rem, uint64_t i, uint32_t r) {
    int w = field_bits(dtype);
    for (int k = 0; k < w; ++k) {
        uint64_t bit = (uint64_t)w * i + (uint64_t)k;
        rem[bit / 8] = (uint8_t)(rem[bit / 8] | (((r >> k) & 1u) << (bit % 8)));
    }
}

int orc_split(int dtype, const void* in, uint64_t n, uint8_t* exps, uint8_t* rem) {
    int ebits, mbits, es;
    if (!layout(dtype, &ebits, &mbits, &es)) return ORC_ERR_UNSUPPORTED_DTYPE;
    const uint8_t* src = (const uint8_t*)in;
    const int width = 8 * es;
    memset(rem, 0, (size_t)orc_remainder_plane_bytes(dtype, n));
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t bits = (uint32_t)rd_le(src + (uint64_t)es * i, es);
        uint32_t sign = (bits >> (width - 1)) & 1u;
        uint32_t e = (bits >> mbits) & ((1u << ebits) - 1u);
        uint32_t m = bits & ((1u << mbits) - 1u);
        exps[i] = (uint8_t)e;
        put_rem(dtype, rem, i, (sign << mbits) | m);
    }
    return ORC_OK;
}

int orc_merge(int dtype, const uint8_t* exps, const uint8_t* rem, uint64_t n, void* out) {
    int ebits, mbits, es;
    if (!layout(dtype, &ebits, &mbits, &es)) return ORC_ERR_UNSUPPORTED_DTYPE;
    uint8_t* dst = (uint8_t*)out;
    const int width = 8 * es;
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t r = get_rem(dtype, rem, i);
        uint32_t sign = (r >> mbits) & 1u;
        uint32_t m = r & ((1u << mbits) - 1u);
        uint32_t bits = (sign << (width - 1)) | ((uint32_t)exps[i] << mbits) | m;
        wr_le(dst + (uint64_t)es * i, bits, es);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* R4: 256-bin histogram of one chunk's exponent bytes.                     */

void orc_histogram(const uint8_t* exps, uint32_t n_c, uint32_t counts[256]) {
    for (int s = 0; s < 256; ++s) counts[s] = 0;
    for (uint32_t i = 0; i < n_c; ++i) counts[exps[i]] += 1;
}

/* ------------------------------------------------------------------------ */
/* R5: deterministic largest-remainder normalisation to M = 4096.           */
/*  1. f_s = floor(c_s*M/N), r_s = (c_s*M) mod N for each present s;        */
/*     a present s with f_s = 0 is raised to 1 and marked boosted.          */
/*  2. S = sum f.  If S < M: +1 to each of the first M-S non-boosted        */
/*     present symbols ordered by (r_s descending, s ascending).            */
/*  3. If S > M: S-M times, -1 to the symbol with the largest f (ties: the  */
/*     smallest s).                                                         */

int orc_normalise(const uint32_t counts[256], uint32_t n_c, uint16_t freq[256]) {
    uint64_t total = 0;
    for (int s = 0; s < 256; ++s) total += counts[s];
    if (n_c == 0 || total != n_c) return ORC_ERR_INVALID_ARG;

    uint32_t f[256];
    uint64_t r[256];
    int boosted[256];
    for (int s = 0; s < 256; ++s) {
        f[s] = 0;
        r[s] = 0;
        boosted[s] = 0;
        if (counts[s] == 0) continue;
        uint64_t scaled = (uint64_t)counts[s] * ORC_M;
        f[s] = (uint32_t)(scaled / n_c);
        r[s] = scaled % n_c;
        if (f[s] == 0) {
            f[s] = 1;
            boosted[s] = 1;
        }
    }
    uint32_t sum = 0;
    for (int s = 0; s < 256; ++s) sum += f[s];

    if (sum < ORC_M) {
        int taken[256];
        for (int s = 0; s < 256; ++s) taken[s] = 0;
        uint32_t need = ORC_M - sum;
        for (uint32_t k = 0; k < need; ++k) {
            int best = -1;
            for (int s = 0; s < 256; ++s) {
                if (counts[s] == 0 || boosted[s] || taken[s]) continue;
                if (best < 0 || r[s] > r[best]) best = s; /* ascending s keeps the first of ties */
            }
            if (best < 0) return ORC_ERR_INVALID_ARG; /* cannot happen: M-S < #non-boosted */
            f[best] += 1;
            taken[best] = 1;
        }
    } else if (sum > ORC_M) {
        uint32_t excess = sum - ORC_M;
        for (uint32_t k = 0; k < excess; ++k) {
            int best = 0;
            for (int s = 1; s < 256; ++s)
                if (f[s] > f[best]) best = s;
            f[best] -= 1; /* f[best] >= 2 here, since S > M >= 256 >= #present */
        }
    }
    for (int s = 0; s < 256; ++s) freq[s] = (uint16_t)f[s];
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* R6/R7: interleaved rANS, 32 lanes, x in [2^16, 2^32), 16-bit words.      */
/* Symbol i belongs to lane i mod 32 and to step i / 32.  The encoder runs  */
/* steps from last to first; the stream lists, step by step from the first, */
/* the words each step's renormalising lanes need, in ascending lane order. */

static void cumulative(const uint16_t freq[256], uint32_t cum[257]) {
    cum[0] = 0;
    for (int s = 0; s < 256; ++s) cum[s + 1] = cum[s] + freq[s];
}

int orc_rans_encode(const uint8_t* syms, uint32_t n_c, const uint16_t freq[256],
                    uint32_t states[32], uint16_t* words, uint32_t* n_words) {
    uint32_t cum[257];
    cumulative(freq, cum);
    if (cum[256] != ORC_M) return ORC_ERR_INVALID_ARG;

    uint8_t* emitted = (uint8_t*)calloc(n_c ? n_c : 1, 1);
    uint16_t* word_of = (uint16_t*)calloc(n_c ? n_c : 1, sizeof(uint16_t));
    if (!emitted || !word_of) {
        free(emitted);
        free(word_of);
        return ORC_ERR_INVALID_ARG;
    }
    uint32_t x[32];
    for (int j = 0; j < 32; ++j) x[j] = ORC_RANS_L;

    uint32_t steps = (n_c + ORC_LANES - 1) / ORC_LANES;
    int status = ORC_OK;
    for (uint32_t t = steps; t-- > 0 && status == ORC_OK;) {
        for (uint32_t j = 0; j < ORC_LANES; ++j) {
            uint32_t i = t * ORC_LANES + j;
            if (i >= n_c) continue;
            uint32_t s = syms[i];
            uint32_t f = freq[s];
            if (f == 0) {
                status = ORC_ERR_INVALID_ARG;
                break;
            }
            uint64_t x_max = (uint64_t)f << (32 - ORC_PROB_BITS); /* f * 2^20 */
            if ((uint64_t)x[j] >= x_max) {
                word_of[i] = (uint16_t)(x[j] & 0xFFFFu);
                emitted[i] = 1;
                x[j] >>= 16;
            }
            x[j] = (x[j] / f) * ORC_M + (x[j] % f) + cum[s];
        }
    }
    if (status == ORC_OK) {
        uint32_t w = 0;
        for (uint32_t i = 0; i < n_c; ++i)
            if (emitted[i]) words[w++] = word_of[i];
        *n_words = w;
        for (int j = 0; j < 32; ++j) states[j] = x[j];
    }
    free(emitted);
    free(word_of);
    return status;
}

int orc_rans_decode(const uint32_t states_in[32], const uint16_t* words, uint32_t n_words,
                    const uint16_t freq[256], uint32_t n_c, uint8_t* syms) {
    uint32_t cum[257];
    cumulative(freq, cum);
    if (cum[256] != ORC_M) return ORC_ERR_CORRUPT;

    /* slot -> symbol: slots [cum_s, cum_s + f_s) belong to s (R14) */
    uint8_t sym_of_slot[ORC_M];
    for (int s = 0; s < 256; ++s)
        for (uint32_t k = cum[s]; k < cum[s + 1]; ++k) sym_of_slot[k] = (uint8_t)s;

    uint32_t x[32];
    for (int j = 0; j < 32; ++j) {
        if (states_in[j] < ORC_RANS_L) return ORC_ERR_CORRUPT;
        x[j] = states_in[j];
    }
    uint32_t pos = 0;
    uint32_t steps = (n_c + ORC_LANES - 1) / ORC_LANES;
    for (uint32_t t = 0; t < steps; ++t) {
        for (uint32_t j = 0; j < ORC_LANES; ++j) {
            uint32_t i = t * ORC_LANES + j;
            if (i >= n_c) continue;
            uint32_t slot = x[j] & (ORC_M - 1);
            uint32_t s = sym_of_slot[slot];
            x[j] = freq[s] * (x[j] >> ORC_PROB_BITS) + slot - cum[s];
            if (x[j] < ORC_RANS_L) {
                if (pos >= n_words) return ORC_ERR_CORRUPT;
                x[j] = (x[j] << 16) | words[pos];
                pos += 1;
            }
            syms[i] = (uint8_t)s;
        }
    }
    for (int j = 0; j < 32; ++j)
        if (x[j] != ORC_RANS_L) return ORC_ERR_CORRUPT;
    if (pos != n_words) return ORC_ERR_CORRUPT;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* R8/R9: one chunk stream.                                                  */
/*   coded: u32 state[32] | u8 bitmap[32] | u16 f[K] (present s ascending)   */
/*          | u16 words[W];  len = 160 + 2K + 2W                             */
/*   raw:   the n_c exponent bytes; len = n_c                                */
/* Coded iff len_coded < n_c.                                                */

int orc_encode_chunk(const uint8_t* exps, uint32_t n_c, int force_coded,
                     uint8_t* out, uint32_t* len, int* raw) {
    if (n_c == 0 || n_c > ORC_CHUNK_ELEMS) return ORC_ERR_INVALID_ARG;
    uint32_t counts[256];
    uint16_t freq[256];
    orc_histogram(exps, n_c, counts);
    int st = orc_normalise(counts, n_c, freq);
    if (st != ORC_OK) return st;
    return orc_encode_chunk_freq(exps, n_c, freq, force_coded, out, len, raw);
}

/* R24: counts for a table built from a sample of the chunk (UCCL-Zip Fig. 5:
 * each block samples and builds its own table): the chunk's elements at
 * positions 0, 16, 32, ...; a symbol seen s times in the sample counts 16 s,
 * and every symbol of the format's exponent range [0, 2^ebits) not seen
 * counts 1, so that it can still be coded.  Returns the counts' total. */
uint32_t orc_sampled_counts(const uint8_t* exps, uint32_t n_c, int ebits, uint32_t counts[256]) {
    uint32_t seen[256];
    for (int s = 0; s < 256; ++s) seen[s] = 0;
    for (uint32_t i = 0; i < n_c; i += 16) seen[exps[i]] += 1;
    uint32_t total = 0;
    for (int s = 0; s < 256; ++s) {
        if (seen[s] > 0) counts[s] = 16u * seen[s];
        else counts[s] = s < (1 << ebits) ? 1u : 0u;
        total += counts[s];
    }
    return total;
}

/* R25: counts of the parametric table for values ~ N(0, sigma^2) (ZipCCL
 * abstract: the exponent coding follows from the Gaussian shape, with no
 * statistics gathered online).  With bias b = 2^(ebits-1) - 1, exponent field
 * e >= 1 holds the magnitudes [2^(e-b), 2^(e-b+1)), whose probability is
 * erfc(x_e) - erfc(2 x_e) for x_e = 2^(e-b) / (sigma sqrt 2); e = 0 holds
 * zero and the subnormals, |x| < 2^(1-b): probability 1 - erfc(2 x_0).  Each
 * probability becomes a count out of 65536, rounded to nearest, and every
 * symbol of [0, 2^ebits) counts at least 1 so that any value stays codable.
 * Returns the counts' total, or 0 for an unknown dtype or a sigma that is
 * not finite and positive. */
uint32_t orc_parametric_counts(int dtype, double sigma, uint32_t counts[256]) {
    int ebits, mbits, es;
    for (int s = 0; s < 256; ++s) counts[s] = 0;
    if (!layout(dtype, &ebits, &mbits, &es) || !(sigma > 0.0) || !isfinite(sigma)) return 0;
    const int bias = (1 << (ebits - 1)) - 1;
    const double scale = sigma * sqrt(2.0);
    uint32_t total = 0;
    for (int e = 0; e < (1 << ebits); ++e) {
        const double x = ldexp(1.0, e - bias) / scale;
        const double p = e == 0 ? 1.0 - erfc(2.0 * x) : erfc(x) - erfc(2.0 * x);
        double c = floor(65536.0 * p + 0.5);
        if (c < 1.0) c = 1.0;
        counts[e] = (uint32_t)c;
        total += counts[e];
    }
    return total;
}

int orc_encode_chunk_freq(const uint8_t* exps, uint32_t n_c, const uint16_t freq[256], int force_coded,
                          uint8_t* out, uint32_t* len, int* raw) {
    if (n_c == 0 || n_c > ORC_CHUNK_ELEMS) return ORC_ERR_INVALID_ARG;
    int st;
    uint32_t states[32];
    uint32_t n_words = 0;
    uint16_t* words = (uint16_t*)malloc((size_t)n_c * sizeof(uint16_t));
    if (!words) return ORC_ERR_INVALID_ARG;
    st = orc_rans_encode(exps, n_c, freq, states, words, &n_words);
    if (st != ORC_OK) {
        free(words);
        return st;
    }
    uint32_t k = 0;
    for (int s = 0; s < 256; ++s)
        if (freq[s] > 0) k += 1;
    uint64_t len_coded = 160u + 2u * (uint64_t)k + 2u * (uint64_t)n_words;

    if (force_coded || len_coded < n_c) {
        uint8_t* p = out;
        for (int j = 0; j < 32; ++j) wr_le(p + 4 * j, states[j], 4);
        p += 128;
        memset(p, 0, 32);
        for (int s = 0; s < 256; ++s)
            if (freq[s] > 0) p[s >> 3] |= (uint8_t)(1u << (s & 7));
        p += 32;
        for (int s = 0; s < 256; ++s)
            if (freq[s] > 0) {
                wr_le(p, freq[s], 2);
                p += 2;
            }
        for (uint32_t w = 0; w < n_words; ++w) {
            wr_le(p, words[w], 2);
            p += 2;
        }
        *len = (uint32_t)len_coded;
        *raw = 0;
    } else {
        memcpy(out, exps, n_c);
        *len = n_c;
        *raw = 1;
    }
    free(words);
    return ORC_OK;
}

int orc_decode_chunk(const uint8_t* stream, uint32_t len, int raw, uint32_t n_c, uint8_t* exps) {
    if (n_c == 0 || n_c > ORC_CHUNK_ELEMS) return ORC_ERR_CORRUPT;
    if (raw) {
        if (len != n_c) return ORC_ERR_CORRUPT;
        memcpy(exps, stream, n_c);
        return ORC_OK;
    }
    if (len < 160) return ORC_ERR_CORRUPT;
    uint32_t states[32];
    for (int j = 0; j < 32; ++j) states[j] = (uint32_t)rd_le(stream + 4 * j, 4);
    const uint8_t* bitmap = stream + 128;
    uint16_t freq[256];
    uint32_t k = 0;
    for (int s = 0; s < 256; ++s) {
        freq[s] = 0;
        if (bitmap[s >> 3] & (1u << (s & 7))) k += 1;
    }
    if ((uint64_t)len < 160u + 2u * (uint64_t)k) return ORC_ERR_CORRUPT;
    if ((len - 160u - 2u * k) % 2u != 0) return ORC_ERR_CORRUPT;
    uint32_t n_words = (len - 160u - 2u * k) / 2u;
    const uint8_t* fp = stream + 160;
    uint32_t sum = 0;
    for (int s = 0; s < 256; ++s) {
        if (!(bitmap[s >> 3] & (1u << (s & 7)))) continue;
        uint32_t f = (uint32_t)rd_le(fp, 2);
        fp += 2;
        if (f == 0 || f > ORC_M) return ORC_ERR_CORRUPT;
        freq[s] = (uint16_t)f;
        sum += f;
    }
    if (sum != ORC_M) return ORC_ERR_CORRUPT;
    uint16_t* words = (uint16_t*)malloc((size_t)(n_words ? n_words : 1) * sizeof(uint16_t));
    if (!words) return ORC_ERR_CORRUPT;
    for (uint32_t w = 0; w < n_words; ++w) words[w] = (uint16_t)rd_le(fp + 2 * w, 2);
    int st = orc_rans_decode(states, words, n_words, freq, n_c, exps);
    free(words);
    return st;
}

/* ------------------------------------------------------------------------ */
/* R3/R10/R11: the container.                                                */
/*   [0,64)         header: "UZP1" | u16 version=1 | u8 dtype | u8 flags=0 |  */
/*                  u64 n | u32 chunk_elems | u32 C | u64 rem_offset |        */
/*                  u64 exp_offset | u64 total_bytes | 16 zero bytes          */
/*   [64,64+8C)     u64 offset of chunk c's stream from exp_offset            */
/*   [64+8C,64+12C) u32 length of chunk c (bit 31 = RAW)                      */
/*   rem_offset = round16(64+12C):      remainder plane (R1, R21, R22)        */
/*   exp_offset = round16(rem_offset + plane bytes): chunk streams, each      */
/*                padded to 16 bytes; every padding byte is zero.             */

static uint64_t num_chunks(uint64_t n) { return (n + ORC_CHUNK_ELEMS - 1) / ORC_CHUNK_ELEMS; }

static uint32_t chunk_elems(uint64_t n, uint64_t c) {
    uint64_t start = c * ORC_CHUNK_ELEMS;
    uint64_t left = n - start;
    return (uint32_t)(left < ORC_CHUNK_ELEMS ? left : ORC_CHUNK_ELEMS);
}

static uint64_t rem_offset_of(uint64_t n) { return round16(ORC_HEADER_BYTES + 12u * num_chunks(n)); }

static uint64_t exp_offset_of(int dtype, uint64_t n) {
    return round16(rem_offset_of(n) + orc_remainder_plane_bytes(dtype, n));
}

uint64_t orc_container_bound(int dtype, uint64_t n) {
    uint64_t bound = exp_offset_of(dtype, n);
    uint64_t c_count = num_chunks(n);
    for (uint64_t c = 0; c < c_count; ++c) bound += round16(chunk_elems(n, c));
    return bound;
}

/* R23: the gate's sample is the first min(n, 65536 / element bytes)
 * elements (at most 64 KiB of input); the message goes RAW when that sample,
 * coded as one chunk, would be stored RAW under R9. */
uint64_t orc_gate_sample_elems(int dtype, uint64_t n) {
    int ebits, mbits, es;
    if (!layout(dtype, &ebits, &mbits, &es)) return 0;
    uint64_t s = 65536u / (uint64_t)es;
    return n < s ? n : s;
}

int orc_gate_says_raw(const uint8_t* exps, uint32_t n_s) {
    if (n_s == 0) return 0;
    uint8_t* tmp = (uint8_t*)malloc((size_t)n_s + 672u + 2u * (size_t)n_s);
    if (!tmp) return -1;
    uint32_t len = 0;
    int raw = 0;
    int st = orc_encode_chunk(exps, n_s, 0, tmp, &len, &raw);
    free(tmp);
    return st == ORC_OK ? raw : -1;
}

int orc_compress(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap,
                 uint64_t* total) {
    return orc_compress_mode(dtype, in, n, out, cap, total, ORC_MODE_CHUNK);
}

/* The container of every mode; model (R25) is the one table of every chunk,
 * or NULL. */
static int compress_impl(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap, uint64_t* total,
                         int mode, const uint16_t* model) {
    if (!dtype_ok(dtype)) return ORC_ERR_UNSUPPORTED_DTYPE;
    if (num_chunks(n) > 0xFFFFFFFFull) return ORC_ERR_INVALID_ARG;
    if ((n > 0 && in == NULL) || out == NULL) return ORC_ERR_INVALID_ARG;
    uint64_t bound = orc_container_bound(dtype, n);
    if (cap < bound) return ORC_ERR_CAPACITY;

    uint64_t c_count = num_chunks(n);
    uint64_t rem_offset = rem_offset_of(n);
    uint64_t exp_offset = exp_offset_of(dtype, n);
    memset(out, 0, bound); /* R10: every padding byte is zero */

    uint8_t* exps = (uint8_t*)malloc(n ? n : 1);
    if (!exps) return ORC_ERR_INVALID_ARG;
    orc_split(dtype, in, n, exps, out + rem_offset);

    int all_raw = mode == ORC_MODE_RAW;
    if (mode == ORC_MODE_GATE) {
        all_raw = orc_gate_says_raw(exps, (uint32_t)orc_gate_sample_elems(dtype, n));
        if (all_raw < 0) {
            free(exps);
            return ORC_ERR_INVALID_ARG;
        }
    }
    uint64_t off = 0;
    for (uint64_t c = 0; c < c_count; ++c) {
        uint32_t n_c = chunk_elems(n, c);
        uint32_t len = 0;
        int raw = 0;
        int st = ORC_OK;
        if (all_raw) { /* the chunk's exponent bytes, as R9 stores a RAW chunk */
            memcpy(out + exp_offset + off, exps + c * ORC_CHUNK_ELEMS, n_c);
            len = n_c;
            raw = 1;
        } else if (model != NULL) {
            st = orc_encode_chunk_freq(exps + c * ORC_CHUNK_ELEMS, n_c, model, 0, out + exp_offset + off, &len, &raw);
        } else if (mode == ORC_MODE_SAMPLED) {
            int ebits, mbits, es;
            layout(dtype, &ebits, &mbits, &es);
            uint32_t counts[256];
            uint16_t freq[256];
            const uint8_t* ce = exps + c * ORC_CHUNK_ELEMS;
            uint32_t total = orc_sampled_counts(ce, n_c, ebits, counts);
            st = orc_normalise(counts, total, freq);
            if (st == ORC_OK) st = orc_encode_chunk_freq(ce, n_c, freq, 0, out + exp_offset + off, &len, &raw);
        } else {
            st = orc_encode_chunk(exps + c * ORC_CHUNK_ELEMS, n_c, 0, out + exp_offset + off, &len, &raw);
        }
        if (st != ORC_OK) {
            free(exps);
            return st;
        }
        wr_le(out + ORC_HEADER_BYTES + 8u * c, off, 8);
        wr_le(out + ORC_HEADER_BYTES + 8u * c_count + 4u * c, len | (raw ? ORC_RAW_FLAG : 0u), 4);
        off += round16(len);
    }
    free(exps);

    uint8_t* h = out;
    h[0] = 'U';
    h[1] = 'Z';
    h[2] = 'P';
    h[3] = '1';
    wr_le(h + 4, 1, 2);
    h[6] = (uint8_t)dtype;
    h[7] = 0;
    wr_le(h + 8, n, 8);
    wr_le(h + 16, ORC_CHUNK_ELEMS, 4);
    wr_le(h + 20, c_count, 4);
    wr_le(h + 24, rem_offset, 8);
    wr_le(h + 32, exp_offset, 8);
    wr_le(h + 40, exp_offset + off, 8);
    *total = exp_offset + off;
    return ORC_OK;
}

int orc_compress_mode(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap,
                      uint64_t* total, int mode) {
    if (mode != ORC_MODE_CHUNK && mode != ORC_MODE_RAW && mode != ORC_MODE_GATE && mode != ORC_MODE_SAMPLED)
        return ORC_ERR_INVALID_ARG;
    return compress_impl(dtype, in, n, out, cap, total, mode, NULL);
}

/* R25: every chunk coded (or stored RAW, R9) with the one table R5 makes of
 * orc_parametric_counts(dtype, sigma). */
int orc_compress_parametric(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap,
                            uint64_t* total, double sigma) {
    if (!dtype_ok(dtype)) return ORC_ERR_UNSUPPORTED_DTYPE;
    uint32_t counts[256];
    uint16_t freq[256];
    const uint32_t sum = orc_parametric_counts(dtype, sigma, counts);
    if (sum == 0) return ORC_ERR_INVALID_ARG;
    const int st = orc_normalise(counts, sum, freq);
    if (st != ORC_OK) return st;
    return compress_impl(dtype, in, n, out, cap, total, ORC_MODE_CHUNK, freq);
}

/* R12: the receiver checks the header and every chunk before trusting it. */
int orc_decompress(const uint8_t* comp, uint64_t comp_bytes, int dtype, uint64_t n, void* out) {
    if (!dtype_ok(dtype)) return ORC_ERR_UNSUPPORTED_DTYPE;
    if (comp == NULL || (n > 0 && out == NULL)) return ORC_ERR_INVALID_ARG;
    if (comp_bytes < ORC_HEADER_BYTES) return ORC_ERR_CORRUPT;
    const uint8_t* h = comp;
    if (h[0] != 'U' || h[1] != 'Z' || h[2] != 'P' || h[3] != '1') return ORC_ERR_CORRUPT;
    if (rd_le(h + 4, 2) != 1) return ORC_ERR_CORRUPT;
    if (h[6] != (uint8_t)dtype || h[7] != 0) return ORC_ERR_CORRUPT;
    if (rd_le(h + 8, 8) != n) return ORC_ERR_CORRUPT;
    if (rd_le(h + 16, 4) != ORC_CHUNK_ELEMS) return ORC_ERR_CORRUPT;
    uint64_t c_count = num_chunks(n);
    if (rd_le(h + 20, 4) != c_count) return ORC_ERR_CORRUPT;
    uint64_t rem_offset = rem_offset_of(n);
    uint64_t exp_offset = exp_offset_of(dtype, n);
    if (rd_le(h + 24, 8) != rem_offset) return ORC_ERR_CORRUPT;
    if (rd_le(h + 32, 8) != exp_offset) return ORC_ERR_CORRUPT;
    uint64_t total = rd_le(h + 40, 8);
    if (total > comp_bytes || total < exp_offset) return ORC_ERR_CORRUPT;

    uint8_t* exps = (uint8_t*)malloc(n ? n : 1);
    if (!exps) return ORC_ERR_INVALID_ARG;
    uint64_t section = total - exp_offset;
    for (uint64_t c = 0; c < c_count; ++c) {
        uint64_t off = rd_le(comp + ORC_HEADER_BYTES + 8u * c, 8);
        uint32_t lw = (uint32_t)rd_le(comp + ORC_HEADER_BYTES + 8u * c_count + 4u * c, 4);
        int raw = (lw & ORC_RAW_FLAG) != 0;
        uint32_t len = lw & ~ORC_RAW_FLAG;
        if (off % 16u != 0 || off > section || len > section - off) {
            free(exps);
            return ORC_ERR_CORRUPT;
        }
        int st = orc_decode_chunk(comp + exp_offset + off, len, raw, chunk_elems(n, c),
                                  exps + c * ORC_CHUNK_ELEMS);
        if (st != ORC_OK) {
            free(exps);
            return st;
        }
    }
    int st = orc_merge(dtype, exps, comp + rem_offset, n, out);
    free(exps);
    return st;
}
