/*
 * uzip oracle: plain, slow, single-threaded CPU implementation of the
 * exponent-plane rANS container.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may
 * include, link or call this code; it exists so that tests, the smoke check
 * and the benchmark's CPU baseline can check the GPU path against an
 * independent implementation.  It shares no source with the CUDA library.
 *
 * What the method computes (the pages):
 *   - UCCL-Zip (arXiv 2604.17172), Fig. 2 caption: each float is split into
 *     its exponent field and the remaining sign+fraction bits; only the
 *     exponent field is entropy coded with ANS, the rest is kept raw.
 *   - UCCL-Zip, Fig. 5 caption: every block of work builds its own local
 *     frequency table, so there is no global table.
 *   - NCCLZ (arXiv 2605.12396), Sec. IV-B/IV-C and Alg. 1: a frame is a
 *     self-describing header plus payload, and a payload that coding does not
 *     shrink is stored RAW.
 * Container constants that the pages leave open (chunk of 65536 elements,
 * 256-bin histogram normalised to 4096 by largest remainder, 32 interleaved
 * 32-bit rANS states, 16-bit renormalisation, per-chunk raw store, chunk
 * table, raw sign|mantissa plane) follow the project's format specification;
 * every reading taken where the pages are silent is listed in the design
 * notes as R1..R20.
 */
#ifndef UZIP_ORACLE_H
#define UZIP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_CHUNK_ELEMS 65536u
#define ORC_PROB_BITS 12u
#define ORC_M 4096u
#define ORC_LANES 32u
#define ORC_RANS_L 65536u /* lower bound of the state interval [2^16, 2^32) */
#define ORC_HEADER_BYTES 64u
#define ORC_RAW_FLAG 0x80000000u

/* dtype codes, identical in value to the library's public enum */
#define ORC_BF16 0
#define ORC_FP32 1
#define ORC_FP16 2
#define ORC_FP8_E4M3 3
#define ORC_FP8_E5M2 4

/* status codes, identical in value to the library's public enum */
#define ORC_OK 0
#define ORC_ERR_INVALID_ARG 1
#define ORC_ERR_UNSUPPORTED_DTYPE 2
#define ORC_ERR_CAPACITY 3
#define ORC_ERR_CORRUPT 4

/* --- element split / merge (R1, R21, R22) -------------------------------- */
/* Bytes of the remainder plane of n elements: the sign|fraction fields of
 * w = 1 + fraction bits each (8 bf16, 24 fp32, 11 fp16, 4 e4m3fn, 3 e5m2),
 * packed least significant bit first, ceil(n*w/8) bytes.  0 for an unknown
 * dtype. */
uint64_t orc_remainder_plane_bytes(int dtype, uint64_t n);
/* Split n elements into exponent bytes (exps[n]) and the remainder plane
 * (rem[orc_remainder_plane_bytes(dtype, n)]). */
int orc_split(int dtype, const void* in, uint64_t n, uint8_t* exps, uint8_t* rem);
/* Inverse of orc_split. */
int orc_merge(int dtype, const uint8_t* exps, const uint8_t* rem, uint64_t n, void* out);

/* --- statistics (R4, R5) --------------------------------------------------- */
void orc_histogram(const uint8_t* exps, uint32_t n_c, uint32_t counts[256]);
/* Largest-remainder normalisation of counts (sum n_c) to sum 4096.
 * Returns ORC_OK, or ORC_ERR_INVALID_ARG if the counts do not sum to n_c or
 * n_c == 0. */
int orc_normalise(const uint32_t counts[256], uint32_t n_c, uint16_t freq[256]);

/* --- interleaved rANS over one chunk (R6, R7) ------------------------------ */
/* Encode n_c symbols with the given table (freq sums to 4096, every symbol
 * that occurs has freq >= 1).  Writes the 32 final states and the word stream
 * in decoder order; *n_words receives its length.  words must have room for
 * n_c entries.  Returns ORC_OK or ORC_ERR_INVALID_ARG. */
int orc_rans_encode(const uint8_t* syms, uint32_t n_c, const uint16_t freq[256],
                    uint32_t states[32], uint16_t* words, uint32_t* n_words);
/* Decode n_c symbols.  Returns ORC_OK, or ORC_ERR_CORRUPT if a word read
 * would pass n_words, a slot has no symbol, the final states are not all
 * 2^16 or not every word was consumed. */
int orc_rans_decode(const uint32_t states_in[32], const uint16_t* words, uint32_t n_words,
                    const uint16_t freq[256], uint32_t n_c, uint8_t* syms);

/* --- one chunk stream (R8, R9) --------------------------------------------- */
/* Encode one chunk of exponent bytes into out (room for max(n_c, 672 + 2*n_c)
 * bytes).  *len receives the stream length, *raw 1 if stored raw.
 * force_coded = 1 keeps the coded form even when it is not shorter (test
 * use only; a container never holds such a chunk). */
int orc_encode_chunk(const uint8_t* exps, uint32_t n_c, int force_coded,
                     uint8_t* out, uint32_t* len, int* raw);
int orc_decode_chunk(const uint8_t* stream, uint32_t len, int raw, uint32_t n_c, uint8_t* exps);

/* --- whole container (R3, R10, R11, R12) ----------------------------------- */
/* Bytes of the largest container for (dtype, n): every chunk stored raw. */
uint64_t orc_container_bound(int dtype, uint64_t n);
/* Compress; *total receives the container size.  cap must be at least
 * orc_container_bound(dtype, n). */
int orc_compress(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap,
                 uint64_t* total);
/* Whole-message modes (R23; survey next row 4, NCCLZ Sec. IV-C and Alg. 1:
 * a message whose coding would not pay travels RAW):
 *   ORC_MODE_CHUNK  coded or RAW per chunk (R9), as orc_compress
 *   ORC_MODE_RAW    every chunk stored RAW
 *   ORC_MODE_GATE   every chunk RAW if the gate's sample would be stored RAW
 *                   (orc_gate_says_raw), else as ORC_MODE_CHUNK */
#define ORC_MODE_CHUNK 0
#define ORC_MODE_RAW 1
#define ORC_MODE_GATE 2
#define ORC_MODE_SAMPLED 3 /* R24: each chunk's table from a sample of it */
int orc_compress_mode(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap,
                      uint64_t* total, int mode);
/* R24 sampled-table counts of one chunk (positions 0, 16, 32, ...; a seen
 * symbol counts 16 x its sample count, an unseen one of [0, 2^ebits) counts
 * 1); returns their total. */
uint32_t orc_sampled_counts(const uint8_t* exps, uint32_t n_c, int ebits, uint32_t counts[256]);
/* R25 parametric-table counts for values ~ N(0, sigma^2): for each exponent
 * field value of the format, the probability of its binade as a count out of
 * 65536 (rounded to nearest, at least 1); returns their total, 0 for an
 * unknown dtype or a sigma that is not finite and positive. */
uint32_t orc_parametric_counts(int dtype, double sigma, uint32_t counts[256]);
/* R25: every chunk coded with the one table normalised (R5) from
 * orc_parametric_counts, or stored RAW where that is not shorter (R9). */
int orc_compress_parametric(int dtype, const void* in, uint64_t n, uint8_t* out, uint64_t cap,
                            uint64_t* total, double sigma);
/* One chunk stream coded with the given table (every symbol of exps must have
 * freq > 0); RAW unless shorter, as orc_encode_chunk. */
int orc_encode_chunk_freq(const uint8_t* exps, uint32_t n_c, const uint16_t freq[256], int force_coded,
                          uint8_t* out, uint32_t* len, int* raw);
/* The gate's sample: the first min(n, 65536 / element bytes) elements. */
uint64_t orc_gate_sample_elems(int dtype, uint64_t n);
/* 1 if these n_s exponent bytes, coded as one chunk, would be stored RAW
 * (R9), 0 if coded, -1 on error. */
int orc_gate_says_raw(const uint8_t* exps, uint32_t n_s);
/* Decompress and validate (R12). */
int orc_decompress(const uint8_t* comp, uint64_t comp_bytes, int dtype, uint64_t n, void* out);

#ifdef __cplusplus
}
#endif
#endif
