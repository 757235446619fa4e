/*
 * Test driver: runs the oracle's compressor and decompressor on cases that
 * tests/test_oracle_sanitizers.py writes as files, in a binary built with
 * AddressSanitizer and UndefinedBehaviorSanitizer (any report aborts).
 *
 * A case file is a 24-byte header, then its payload:
 *   [0]      'C': the payload is n values to compress and decompress back
 *            'D': the payload is a container (possibly damaged) to decode
 *   [1]      dtype, [2] mode (0 chunk, 1 RAW, 2 gate, 3 sampled tables,
 *            4 Gaussian model with the sigma below), [3, 8) zero
 *   [8, 16)  n, little endian
 *   [16, 24) sigma (a double), for mode 4
 * Every buffer is allocated at its exact size, so a read past a container's
 * end or a value array's end is caught.  Exit status 0 when every round trip
 * is exact and every decode ends in OK or CORRUPT.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../oracle/uzip_oracle.h"

static size_t elem_bytes(int dtype) { return dtype == 1 ? 4u : (dtype == 0 || dtype == 2) ? 2u : 1u; }

static uint8_t* read_file(const char* path, size_t* size) {
    FILE* f = fopen(path, "rb");
    if (!f) return NULL;
    fseek(f, 0, SEEK_END);
    long len = ftell(f);
    fseek(f, 0, SEEK_SET);
    uint8_t* buf = (uint8_t*)malloc(len > 0 ? (size_t)len : 1u);
    size_t got = len > 0 ? fread(buf, 1, (size_t)len, f) : 0;
    fclose(f);
    if (got != (size_t)(len > 0 ? len : 0)) {
        free(buf);
        return NULL;
    }
    *size = (size_t)len;
    return buf;
}

static uint8_t* exact_copy(const uint8_t* src, size_t size) {
    uint8_t* p = (uint8_t*)malloc(size ? size : 1u);
    if (size) memcpy(p, src, size);
    return p;
}

static int run_case(const char* path) {
    size_t size = 0;
    uint8_t* file = read_file(path, &size);
    if (!file || size < 24) {
        fprintf(stderr, "%s: unreadable case\n", path);
        free(file);
        return 1;
    }
    const int kind = file[0], dtype = file[1], mode = file[2];
    uint64_t n = 0;
    for (int i = 7; i >= 0; --i) n = (n << 8) | file[8 + i];
    double sigma;
    memcpy(&sigma, file + 16, sizeof sigma);
    const size_t payload = size - 24, es = elem_bytes(dtype);
    int bad = 0;
    if (kind == 'C') {
        if (payload != n * es) {
            fprintf(stderr, "%s: payload of %zu bytes for n = %llu\n", path, payload, (unsigned long long)n);
            free(file);
            return 1;
        }
        uint8_t* in = exact_copy(file + 24, payload);
        const uint64_t cap = orc_container_bound(dtype, n);
        uint8_t* out = (uint8_t*)malloc(cap ? cap : 1u);
        uint64_t total = 0;
        int st = mode == 4 ? orc_compress_parametric(dtype, in, n, out, cap, &total, sigma)
                           : orc_compress_mode(dtype, in, n, out, cap, &total, mode);
        if (st != ORC_OK || total > cap) {
            fprintf(stderr, "%s: compress status %d\n", path, st);
            bad = 1;
        } else {
            uint8_t* comp = exact_copy(out, total);  // exactly the container's bytes
            uint8_t* back = (uint8_t*)malloc(payload ? payload : 1u);
            st = orc_decompress(comp, total, dtype, n, back);
            if (st != ORC_OK || (payload && memcmp(back, in, payload) != 0)) {
                fprintf(stderr, "%s: round trip failed (status %d)\n", path, st);
                bad = 1;
            }
            free(back);
            free(comp);
        }
        free(out);
        free(in);
    } else if (kind == 'D') {
        uint8_t* comp = exact_copy(file + 24, payload);
        uint8_t* back = (uint8_t*)malloc(n * es ? n * es : 1u);
        const int st = orc_decompress(comp, payload, dtype, n, back);
        if (st != ORC_OK && st != ORC_ERR_CORRUPT) {
            fprintf(stderr, "%s: decode status %d\n", path, st);
            bad = 1;
        }
        free(back);
        free(comp);
    } else {
        fprintf(stderr, "%s: unknown case kind\n", path);
        bad = 1;
    }
    free(file);
    return bad;
}

int main(int argc, char** argv) {
    int failures = 0;
    for (int i = 1; i < argc; ++i) failures += run_case(argv[i]);
    printf("%d cases, %d failed\n", argc - 1, failures);
    return failures ? 1 : 0;
}
