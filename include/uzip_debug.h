/*
 * uzip test hooks: host-only helpers that expose internal arithmetic of the
 * library to its test-suite.  No GPU work; safe to call without a device.
 * The pages have no counterpart: these exist to check the library's own
 * implementation choices.
 */
#ifndef UZIP_DEBUG_H
#define UZIP_DEBUG_H

#include <stdint.h>

#include "uzip.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The encoder replaces x / f (x in [16 f, f * 2^20), f in [1, 4096]) by
 * (x * m + add) >> shift.  Returns 1 and the constants for a valid f, 0 for
 * f outside [1, 4096]. */
int uzip_debug_div_magic(uint32_t f, uint32_t* m, uint32_t* add, uint32_t* shift);

/* The warp-specialised encoder replaces x / f (x in [0, f * 2^20), f in
 * [1, 4096]) by (x * (2^32 + m_lo)) >> (32 + shift).  Returns 1 and the
 * constants for a valid f, 0 for f outside [1, 4096]. */
int uzip_debug_div_magic33(uint32_t f, uint32_t* m_lo, uint32_t* shift);

/* The counts uzip_compress_parametric normalises into its table, for values
 * ~ N(0, sigma^2) of format dtype (counts[256]; values beyond the format's
 * exponent field are 0).  Returns 1, or 0 for an unknown dtype or a sigma
 * that is not finite and positive. */
int uzip_debug_model_counts(int dtype, double sigma, uint32_t* counts);

/* Tuning of the warp-specialised compressor: a helper warp starts splitting
 * its encoder's next chunk once the encoder has at most `blocks` blocks of 32
 * steps left of its current chunk (64: at once).  Default 32.  Affects speed
 * and the L2 working set only, never the output. */
void uzip_debug_set_ws_jit_blocks(uint32_t blocks);

/* Byte offset of the compressor's work area inside the output buffer (the
 * area is 16 + 8*C bytes long and follows the largest possible container). */
uint64_t uzip_debug_scratch_offset(uzip_dtype dtype, uint64_t n);

#ifdef __cplusplus
}
#endif
#endif
