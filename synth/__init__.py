"""Seeded synthetic tensors shaped like the pages' workloads.

This module only draws numbers: it holds none of the codec's arithmetic and
is shared by the oracle-side and the GPU-side tests and by the benchmark.

Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Draw k of element i in stream
(cfg, tensor) is mix64(key + (i*D + k + 1) * golden_gamma), with
key = mix64(seed << 40 ^ cfg << 32 ^ tensor).  Uniforms are
((z >> 11) + 0.5) * 2^-53, which lie strictly inside (0, 1).  Normals come from
Box-Muller in float64 (one cosine branch), then float64 -> float32 -> bf16 by
round-to-nearest-even.  Every element depends only on its index, so any block
split or thread count gives the same bytes.

Workloads (the pages measure real weights, gradients and KV caches, which are
not available; these stand in for them with the same shapes and value
distributions; the distribution of LLM tensors is near-Gaussian per the
ZipCCL abstract):
  c1  1,048,576 bf16 ~ N(0, 0.02)
  c2  one Llama-3-8B-shaped decoder layer of bf16 weights, per-row std
      U[0.5, 2] * 0.02, row = first index
  c3  268,435,456 fp32 gradients: 95% N(0, 1e-3), 5% Laplace(0, 1e-2),
      0.1% +0.0, plus 4096 each of -0.0, subnormals, +inf, -inf and NaN with
      random payloads
  c4  [8, 8192, 8192] bf16 activations ~ 0.5 * Student-t(4), 82 outlier
      channels x50, elements [2^28, 2^28 + 65536) replaced by random bits
  c5  Llama-3-8B-shaped parameter set (8,030,261,248 bf16 ~ N(0, 0.02)),
      cut into 1 GiB messages
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

SEED = 0
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
BLOCK = 1 << 22

_THREADS = max(1, min(16, os.cpu_count() or 1))


def mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(cfg: int, tensor: int, seed: int = SEED) -> np.uint64:
    k = np.array([((seed << 40) ^ (cfg << 32) ^ tensor) & 0xFFFFFFFFFFFFFFFF], np.uint64)
    return mix64(k)[0]


def raw64(key: np.uint64, idx: np.ndarray, ndraw: int, k: int) -> np.ndarray:
    """64 random bits for draw k of each element index in idx."""
    ctr = idx.astype(np.uint64) * np.uint64(ndraw) + np.uint64(k + 1)
    return mix64(key + ctr * GAMMA)


def uniform(key, idx, ndraw, k) -> np.ndarray:
    z = raw64(key, idx, ndraw, k)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(key, idx, ndraw, k0) -> np.ndarray:
    u0 = uniform(key, idx, ndraw, k0)
    u1 = uniform(key, idx, ndraw, k0 + 1)
    return np.sqrt(-2.0 * np.log(u0)) * np.cos(2.0 * math.pi * u1)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _parallel_fill(out: np.ndarray, n: int, fn, threads: int | None = None):
    """fn(lo, hi) -> values for flat indices [lo, hi); runs blocks on threads."""
    blocks = [(lo, min(n, lo + BLOCK)) for lo in range(0, n, BLOCK)]

    def work(b):
        lo, hi = b
        out[lo:hi] = fn(lo, hi)

    with ThreadPoolExecutor(threads or _THREADS) as ex:
        list(ex.map(work, blocks))
    return out


# --------------------------------------------------------------------------
# c1: 1,048,576 bf16 ~ N(0, 0.02)

def c1(n: int = 1 << 20, std: float = 0.02, cfg: int = 1, tensor: int = 0) -> np.ndarray:
    key = stream_key(cfg, tensor)

    def fn(lo, hi):
        idx = np.arange(lo, hi, dtype=np.uint64)
        return f32_to_bf16_bits((normal(key, idx, 2, 0) * std).astype(np.float32))

    return _parallel_fill(np.empty(n, np.uint16), n, fn)


def normal_bf16(n: int, std: float, cfg: int, tensor: int, start: int = 0) -> np.ndarray:
    """n bf16 ~ N(0, std) of stream (cfg, tensor), elements [start, start+n)."""
    key = stream_key(cfg, tensor)

    def fn(lo, hi):
        idx = np.arange(start + lo, start + hi, dtype=np.uint64)
        return f32_to_bf16_bits((normal(key, idx, 2, 0) * std).astype(np.float32))

    return _parallel_fill(np.empty(n, np.uint16), n, fn)


# --------------------------------------------------------------------------
# c2: one Llama-3-8B-shaped decoder layer, per-row std U[0.5, 2] * 0.02

C2_TENSORS = [
    ("q", (4096, 4096)),
    ("k", (4096, 1024)),
    ("v", (4096, 1024)),
    ("o", (4096, 4096)),
    ("gate", (4096, 14336)),
    ("up", (4096, 14336)),
    ("down", (14336, 4096)),
]


def c2_tensor(t: int, rows: int | None = None) -> np.ndarray:
    """Tensor t of the layer (flattened, row-major); rows limits the row count."""
    name, (r, cols) = C2_TENSORS[t]
    r = r if rows is None else min(r, rows)
    n = r * cols
    key = stream_key(2, t)
    row_key = stream_key(2, 100 + t)

    def fn(lo, hi):
        idx = np.arange(lo, hi, dtype=np.uint64)
        row = idx // np.uint64(cols)
        std = (0.5 + 1.5 * uniform(row_key, row, 1, 0)) * 0.02
        return f32_to_bf16_bits((normal(key, idx, 2, 0) * std).astype(np.float32))

    return _parallel_fill(np.empty(n, np.uint16), n, fn)


# --------------------------------------------------------------------------
# c3: fp32 gradient buffer with special values

C3_N = 268435456
C3_SPECIALS = 4096


def c3(n: int = C3_N, specials: int = C3_SPECIALS) -> np.ndarray:
    key = stream_key(3, 0)

    def fn(lo, hi):
        idx = np.arange(lo, hi, dtype=np.uint64)
        sel = uniform(key, idx, 5, 0)
        g = normal(key, idx, 5, 1) * 1e-3
        u = uniform(key, idx, 5, 3) - 0.5
        lap = -1e-2 * np.sign(u) * np.log1p(-2.0 * np.abs(u))
        v = np.where(sel < 0.95, g, lap).astype(np.float32)
        zero = uniform(key, idx, 5, 4) < 0.001
        v[zero] = np.float32(0.0)
        return v.view(np.uint32)

    out = _parallel_fill(np.empty(n, np.uint32), n, fn)
    # special values at uniformly drawn positions, kinds applied in this order
    j = np.arange(specials, dtype=np.uint64)
    for kind in range(5):
        k = stream_key(3, 10 + kind)
        pos = (uniform(k, j, 3, 0) * n).astype(np.int64)
        pos = np.minimum(pos, n - 1)
        bits = raw64(k, j, 3, 1)
        sign = ((bits >> np.uint64(63)) & np.uint64(1)).astype(np.uint32) << np.uint32(31)
        mant = (bits & np.uint64(0x7FFFFF)).astype(np.uint32)
        mant = np.where(mant == 0, np.uint32(1), mant)  # payload never zero
        if kind == 0:
            vals = np.full(specials, 0x80000000, np.uint32)  # -0.0
        elif kind == 1:
            vals = sign | mant  # subnormal: exponent 0, mantissa != 0
        elif kind == 2:
            vals = np.full(specials, 0x7F800000, np.uint32)  # +inf
        elif kind == 3:
            vals = np.full(specials, 0xFF800000, np.uint32)  # -inf
        else:
            vals = sign | np.uint32(0x7F800000) | mant  # NaN, quiet or signalling
        out[pos] = vals
    return out


# --------------------------------------------------------------------------
# c4: [8, 8192, 8192] bf16 activations ~ 0.5 * t(4) with outlier channels

C4_SHAPE = (8, 8192, 8192)
C4_OUTLIERS = 82  # round(1% of 8192)
C4_RANDOM_CHUNK = 4096  # elements [2^28, 2^28 + 65536) become random bits


def c4_outlier_channels(hidden: int = 8192, count: int = C4_OUTLIERS) -> np.ndarray:
    key = stream_key(4, 1)
    u = uniform(key, np.arange(hidden, dtype=np.uint64), 1, 0)
    return np.sort(np.argsort(u, kind="stable")[:count])


def c4(n: int | None = None, hidden: int = 8192) -> np.ndarray:
    total = C4_SHAPE[0] * C4_SHAPE[1] * C4_SHAPE[2]
    n = total if n is None else n
    key = stream_key(4, 0)
    is_out = np.zeros(hidden, bool)
    is_out[c4_outlier_channels(hidden)] = True

    def fn(lo, hi):
        idx = np.arange(lo, hi, dtype=np.uint64)
        z = normal(key, idx, 4, 0)
        chi2 = -2.0 * np.log(uniform(key, idx, 4, 2) * uniform(key, idx, 4, 3))
        t = z / np.sqrt(chi2 / 4.0)
        v = 0.5 * t
        v = np.where(is_out[(idx % np.uint64(hidden)).astype(np.int64)], v * 50.0, v)
        return f32_to_bf16_bits(v.astype(np.float32))

    out = _parallel_fill(np.empty(n, np.uint16), n, fn)
    lo = C4_RANDOM_CHUNK * 65536
    if n > lo:
        hi = min(n, lo + 65536)
        rk = stream_key(4, 2)
        out[lo:hi] = (raw64(rk, np.arange(lo, hi, dtype=np.uint64), 1, 0) & np.uint64(0xFFFF)).astype(np.uint16)
    return out


# --------------------------------------------------------------------------
# c5: Llama-3-8B-shaped parameter set, all ~ N(0, 0.02), cut into 1 GiB messages

def c5_layout():
    """(name, numel) in order: embed, 32 layers, final norm, lm_head."""
    d, ff, kv, vocab = 4096, 14336, 1024, 128256
    items = [("embed", vocab * d)]
    for layer in range(32):
        items += [
            (f"l{layer}.q", d * d), (f"l{layer}.k", kv * d), (f"l{layer}.v", kv * d), (f"l{layer}.o", d * d),
            (f"l{layer}.gate", ff * d), (f"l{layer}.up", ff * d), (f"l{layer}.down", d * ff),
            (f"l{layer}.input_norm", d), (f"l{layer}.post_norm", d),
        ]
    items += [("final_norm", d), ("lm_head", vocab * d)]
    return items


C5_TOTAL = 8030261248
C5_MESSAGE = 1 << 29  # 1 GiB of bf16


def c5_message_sizes():
    sizes = []
    left = C5_TOTAL
    while left > 0:
        sizes.append(min(C5_MESSAGE, left))
        left -= sizes[-1]
    return sizes


def c5_message(k: int, n: int | None = None) -> np.ndarray:
    """Message k of the flattened parameter set (its first n values if given)."""
    sizes = c5_message_sizes()
    start = k * C5_MESSAGE
    n = sizes[k] if n is None else min(n, sizes[k])
    return normal_bf16(n, 0.02, 5, 0, start=start)


def uniform_pm1_bf16(n: int, cfg: int = 9, tensor: int = 0) -> np.ndarray:
    """bf16 uniform in [-1, 1): the synthetic input of UCCL-Zip Fig. 8."""
    key = stream_key(cfg, tensor)

    def fn(lo, hi):
        idx = np.arange(lo, hi, dtype=np.uint64)
        return f32_to_bf16_bits((2.0 * uniform(key, idx, 1, 0) - 1.0).astype(np.float32))

    return _parallel_fill(np.empty(n, np.uint16), n, fn)


# --------------------------------------------------------------------------
# fp16 and the two fp8 formats (the dtype sweep of UCCL-Zip Fig. 12): the
# same N(0, std) stream, rounded to each element format

def normal_fp16(n: int, std: float = 0.02, cfg: int = 10, tensor: int = 0, start: int = 0) -> np.ndarray:
    """n fp16 ~ N(0, std) (numpy's round-to-nearest-even), as float16."""
    key = stream_key(cfg, tensor)

    def fn(lo, hi):
        idx = np.arange(start + lo, start + hi, dtype=np.uint64)
        return (normal(key, idx, 2, 0) * std).astype(np.float16).view(np.uint16)

    return _parallel_fill(np.empty(n, np.uint16), n, fn).view(np.float16)


FP8_FORMATS = {"e4m3": (4, 3, 7), "e5m2": (5, 2, 15)}  # exponent bits, fraction bits, bias


def _fp8_positive_codes(fmt: str):
    """Finite non-negative fp8 codes of a format, sorted by value."""
    eb, mb, bias = FP8_FORMATS[fmt]
    codes, vals = [], []
    for c in range(128):
        e, m = c >> mb, c & ((1 << mb) - 1)
        if fmt == "e4m3" and e == 15 and m == (1 << mb) - 1:
            continue  # NaN (e4m3fn has no infinities)
        if fmt == "e5m2" and e == 31:
            continue  # infinities and NaNs
        v = (m / (1 << mb)) * 2.0 ** (1 - bias) if e == 0 else (1 + m / (1 << mb)) * 2.0 ** (e - bias)
        codes.append(c)
        vals.append(v)
    order = np.argsort(vals, kind="stable")
    return np.array(vals)[order], np.array(codes, np.uint8)[order]


def round_to_fp8(x: np.ndarray, fmt: str) -> np.ndarray:
    """Nearest finite fp8 code of each value (magnitudes beyond the largest
    finite value saturate; ties go to the smaller magnitude), as uint8 bits."""
    vals, codes = _fp8_positive_codes(fmt)
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(vals, a), 1, vals.size - 1)
    lo = hi - 1
    pick = np.where(a - vals[lo] <= vals[hi] - a, lo, hi)
    pick = np.where(a >= vals[-1], vals.size - 1, pick)
    return (codes[pick] | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))).astype(np.uint8)


def normal_fp8(n: int, fmt: str, std: float = 0.02, cfg: int = 11, tensor: int = 0, start: int = 0) -> np.ndarray:
    """n fp8 (fmt 'e4m3' or 'e5m2') ~ N(0, std), as uint8 bit patterns."""
    key = stream_key(cfg, tensor)

    def fn(lo, hi):
        idx = np.arange(start + lo, start + hi, dtype=np.uint64)
        return round_to_fp8(normal(key, idx, 2, 0) * std, fmt)

    return _parallel_fill(np.empty(n, np.uint8), n, fn)


def normal_fp32(n: int, std: float = 0.02, cfg: int = 12, tensor: int = 0, start: int = 0) -> np.ndarray:
    """n fp32 ~ N(0, std), as uint32 bit patterns."""
    key = stream_key(cfg, tensor)

    def fn(lo, hi):
        idx = np.arange(start + lo, start + hi, dtype=np.uint64)
        return (normal(key, idx, 2, 0) * std).astype(np.float32).view(np.uint32)

    return _parallel_fill(np.empty(n, np.uint32), n, fn)


# --------------------------------------------------------------------------
# chunks whose coded stream grows faster than their exponent bytes are read
# (a coder runs a chunk from its last value down, so what sits at the top of
# a chunk is coded first)

GROWTH_RANDOM_TOPS = (0.46, 0.48, 0.50, 0.52, 0.55, 0.60)
GROWTH_RARE_COUNTS = (64, 80, 94, 110, 128)


def growth_exponents(tail: int = 4097) -> np.ndarray:
    """8-bit exponent fields, chunk by chunk (65536 values each).

    Chunk k < 6: exponent 127 below, uniformly random exponents in the top
    fraction GROWTH_RANDOM_TOPS[k].  Chunk 6 + j: the 255 exponents other than
    127, GROWTH_RARE_COUNTS[j] times each in a shuffled order, at the top; 127
    below.  Then `tail` values of exponent 126 or 127 (a partial chunk)."""
    chunks = []
    for k, p in enumerate(GROWTH_RANDOM_TOPS):
        key = stream_key(13, k)
        top = int(round(p * 65536))
        e = np.full(65536, 127, np.uint8)
        e[65536 - top:] = (raw64(key, np.arange(top, dtype=np.uint64), 1, 0) & np.uint64(0xFF)).astype(np.uint8)
        chunks.append(e)
    others = np.array([s for s in range(256) if s != 127], np.uint8)
    for j, c in enumerate(GROWTH_RARE_COUNTS):
        key = stream_key(13, 100 + j)
        top = np.repeat(others, c)
        order = np.argsort(raw64(key, np.arange(top.size, dtype=np.uint64), 1, 0), kind="stable")
        e = np.full(65536, 127, np.uint8)
        e[65536 - top.size:] = top[order]
        chunks.append(e)
    key = stream_key(13, 200)
    chunks.append((126 + (raw64(key, np.arange(tail, dtype=np.uint64), 1, 0) & np.uint64(1))).astype(np.uint8))
    return np.concatenate(chunks)


def growth_bf16(tail: int = 4097) -> np.ndarray:
    """bf16 bit patterns with growth_exponents() and random sign and fraction."""
    e = growth_exponents(tail).astype(np.uint16)
    r = raw64(stream_key(13, 300), np.arange(e.size, dtype=np.uint64), 1, 0)
    return ((e << np.uint16(7)) | (r & np.uint64(0x807F)).astype(np.uint16)).astype(np.uint16)


def growth_fp32(tail: int = 4097) -> np.ndarray:
    """fp32 bit patterns with growth_exponents() and random sign and fraction."""
    e = growth_exponents(tail).astype(np.uint32)
    r = raw64(stream_key(13, 301), np.arange(e.size, dtype=np.uint64), 1, 0)
    return ((e << np.uint32(23)) | (r & np.uint64(0x807FFFFF)).astype(np.uint32)).astype(np.uint32)
