"""Seeded random corruptions of a container, sorted by the region they hit.

The regions follow the container layout as the public header documents it
(64-byte header, chunk table, remainder plane, 16-byte aligned chunk
streams); this module reads a container's own header and chunk table and
does none of the codec's arithmetic.
"""
import numpy as np

CHUNK = 65536
HEADER = 64
# per format: (element bits, exponent bits, remainder field bits)
FORMATS = {0: (16, 8, 8), 1: (32, 8, 24), 2: (16, 5, 11), 3: (8, 4, 4), 4: (8, 5, 3)}


def _u64(b, o):
    return int(np.frombuffer(b[o:o + 8].tobytes(), np.uint64)[0])


def _u32(b, o):
    return int(np.frombuffer(b[o:o + 4].tobytes(), np.uint32)[0])


def _r16(v):
    return (v + 15) & ~15


def layout(comp, dtype, n):
    """Byte ranges [lo, hi) of each region of a well-formed container."""
    C = -(-n // CHUNK)
    _, _, w = FORMATS[dtype]
    rem_off, exp_off, total = _u64(comp, 24), _u64(comp, 32), _u64(comp, 40)
    plane = -(-n * w // 8)
    reg = {"header": [(0, 40)], "total": [(40, 48)], "reserved": [(48, 64)], "table": [(64, 64 + 12 * C)],
           "gap": [(64 + 12 * C, rem_off), (rem_off + plane, exp_off)], "plane": [(rem_off, rem_off + plane)],
           "raw": [], "coded": [], "stream_pad": []}
    for c in range(C):
        off = _u64(comp, HEADER + 8 * c)
        lw = _u32(comp, HEADER + 8 * C + 4 * c)
        ln = lw & 0x7FFFFFFF
        lo = exp_off + off
        reg["raw" if lw >> 31 else "coded"].append((lo, lo + ln))
        reg["stream_pad"].append((lo + ln, lo + _r16(ln)))
    assert max(hi for rs in reg.values() for _, hi in rs) <= total
    return {k: [(lo, hi) for lo, hi in v if hi > lo] for k, v in reg.items()}


def _pick(rng, ranges):
    sizes = np.array([hi - lo for lo, hi in ranges], np.float64)
    r = ranges[rng.choice(len(ranges), p=sizes / sizes.sum())]
    return int(rng.integers(r[0], r[1]))


def corruptions(comp, dtype, n, count, seed):
    """count cases (kind, bytes, detail): a flipped bit in a region, a byte
    set to a random value anywhere, or the container cut short.  detail is
    (byte, bit) for flips, else None."""
    rng = np.random.default_rng(seed)
    reg = layout(comp, dtype, n)
    kinds = [k for k, v in reg.items() if v] + ["byte", "truncate"]
    out = []
    for _ in range(count):
        kind = kinds[int(rng.integers(len(kinds)))]
        b = comp.copy()
        if kind == "truncate":
            out.append((kind, b[: int(rng.integers(0, comp.size))].copy(), None))
            continue
        if kind == "byte":
            at = int(rng.integers(0, comp.size))
            b[at] = np.uint8((int(b[at]) + 1 + int(rng.integers(0, 255))) & 0xFF)
            out.append((kind, b, None))
            continue
        at = _pick(rng, reg[kind])
        bit = int(rng.integers(0, 8))
        if kind == "raw":  # stay inside the exponent field, so the merged value changes in one bit
            bit = int(rng.integers(0, FORMATS[dtype][1]))
        b[at] ^= np.uint8(1 << bit)
        out.append((kind, b, (at, bit)))
    return out


def expected_flip(comp, dtype, n, at, bit, kind):
    """For a flip that decoding cannot detect: (element index, output bit)
    that changes, or None when no output bit changes."""
    width, ebits, w = FORMATS[dtype]
    mbits = w - 1
    if kind == "plane":
        k = 8 * (at - _u64(comp, 24)) + bit
        i, j = divmod(k, w)
        if i >= n:
            return None
        return i, (j if j < mbits else width - 1)
    if kind == "raw":
        C = -(-n // CHUNK)
        exp_off = _u64(comp, 32)
        for c in range(C):
            lo = exp_off + _u64(comp, HEADER + 8 * c)
            ln = _u32(comp, HEADER + 8 * C + 4 * c) & 0x7FFFFFFF
            if lo <= at < lo + ln:
                return c * CHUNK + (at - lo), mbits + bit
    raise ValueError(kind)


def fuzz_input(case):
    """(bits as unsigned integers, dtype) of the fuzzed containers: several
    chunks and a ragged tail in every format; the bf16 case has a chunk of
    random bit patterns, which is stored RAW."""
    import synth

    if case == 0:
        bits = synth.normal_bf16(3 * CHUNK + 777, 0.02, 8, 3)
        bits[CHUNK:2 * CHUNK] = np.random.default_rng(5).integers(0, 1 << 16, CHUNK, dtype=np.uint16)
        return bits, 0
    if case == 1:
        return synth.normal_fp32(2 * CHUNK + 100, 0.02, tensor=3), 1
    if case == 2:
        return synth.normal_fp16(2 * CHUNK + 5, 0.02, tensor=3).view(np.uint16), 2
    if case == 3:
        return synth.normal_fp8(CHUNK + 33, "e4m3", 0.02, tensor=3), 3
    return synth.normal_fp8(2 * CHUNK + 1, "e5m2", 0.02, tensor=3), 4
