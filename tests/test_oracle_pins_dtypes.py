"""Pins for the oracle's fp16 and fp8 element layouts (readings R21, R22).

UCCL-Zip Fig. 12 reports its codec on bfloat16, float16, float32,
float8_e4m3fn and float8_e5m2.  The split of each format into exponent field
and sign|fraction bits is pinned here against the formats' own value
definitions as decoded by libraries (numpy's float16, torch's float8 types),
not against a restatement of the oracle's bit arithmetic.
"""
import numpy as np
import pytest

import oracle


def _unpack(plane, n, w):
    """The n w-bit fields of a plane packed least significant bit first
    (numpy's own bit unpacking, independent of the oracle's loops)."""
    bits = np.unpackbits(plane, bitorder="little")[: n * w].reshape(n, w).astype(np.int64)
    return (bits << np.arange(w)).sum(axis=1)


def _fields(e, rem, mbits):
    r = rem.astype(np.int64)
    return e.astype(np.int64), (r >> mbits) & 1, r & ((1 << mbits) - 1)


def test_fp16_all_patterns_roundtrip_and_ieee_value():
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    e, r = oracle.split(x.view(np.float16))
    assert r.size == 11 * x.size // 8
    assert np.array_equal(oracle.merge(oracle.FP16, e, r), x)
    ex, sign, m = _fields(e, _unpack(r, x.size, 11), 10)
    v = x.view(np.float16).astype(np.float64)
    assert np.array_equal(sign.astype(bool), np.signbit(v))
    fin = np.isfinite(v)
    assert np.all(ex[~fin] == 31)
    a = np.abs(v[fin])
    normal = ex[fin] > 0
    expect = np.where(normal, (1.0 + m[fin] / 1024.0) * np.ldexp(1.0, ex[fin] - 15), m[fin] * 2.0 ** -24)
    assert np.array_equal(a, expect)
    assert np.all(m[np.isnan(v)] != 0) and np.all(m[np.isinf(v)] == 0)


@pytest.mark.parametrize("code,name,ebits,mbits,bias", [(oracle.FP8_E4M3, "float8_e4m3fn", 4, 3, 7),
                                                        (oracle.FP8_E5M2, "float8_e5m2", 5, 2, 15)])
def test_fp8_all_patterns_match_torch_decoding(code, name, ebits, mbits, bias):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, name):
        pytest.skip(f"torch has no {name}")
    x = np.arange(256, dtype=np.uint8)
    e, r = oracle.split(x, code)
    assert r.size == 256 * (1 + mbits) // 8
    assert np.array_equal(oracle.merge(code, e, r), x)
    nib = _unpack(r, 256, 1 + mbits)
    ex, sign, m = _fields(e, nib, mbits)
    assert np.all(ex < (1 << ebits)) and np.all(nib < (1 << (1 + mbits)))
    v = torch.from_numpy(x.copy()).view(getattr(torch, name)).float().double().numpy()
    assert np.array_equal(sign.astype(bool), np.signbit(v))
    fin = np.isfinite(v)
    a = np.abs(v[fin])
    normal = ex[fin] > 0
    scale = 1 << mbits
    expect = np.where(normal, (1.0 + m[fin] / scale) * np.ldexp(1.0, ex[fin] - bias),
                      m[fin] / scale * 2.0 ** (1 - bias))
    assert np.array_equal(a, expect)


def test_fp8_packing_worked_examples():
    """e4m3fn 1.0 (0x38), -1.5 (0xBC), NaN (0x7F): remainders 0, 1<<3|4, 7;
    element 0 in the low nibble of byte 0, element 2 alone in byte 1.
    e5m2 1.0 (0x3C), -inf (0xFC), smallest subnormal (0x01): 3-bit
    remainders 000, 100, 001 at bits 0-2, 3-5, 6-8: bytes 0x60, 0x00."""
    x = np.array([0x38, 0xBC, 0x7F], np.uint8)
    e, r = oracle.split(x, oracle.FP8_E4M3)
    assert list(e) == [7, 7, 15]
    assert list(r) == [0xC0, 0x07]
    y = np.array([0x3C, 0xFC, 0x01], np.uint8)
    e, r = oracle.split(y, oracle.FP8_E5M2)
    assert list(e) == [15, 31, 0]
    assert list(r) == [0x60, 0x00]


def test_fp16_packing_worked_example():
    """fp16 -2.5 (0xC100) and 1.0 (0x3C00): 11-bit remainders 0x500 and 0;
    fields at bits 0-10 and 11-21, so bytes 0x00, 0x05, 0x00."""
    x = np.array([0xC100, 0x3C00], np.uint16).view(np.float16)
    e, r = oracle.split(x)
    assert list(e) == [16, 15]
    assert list(r) == [0x00, 0x05, 0x00]


@pytest.mark.parametrize("code,n", [(oracle.FP16, 65536 * 2 + 5), (oracle.FP8_E4M3, 65536 + 7),
                                    (oracle.FP8_E5M2, 3 * 65536 + 1)])
def test_constant_exponent_container_size_closed_form(code, n):
    """Every chunk of a single exponent value codes to the 160-byte stream
    head plus one frequency (R8), so the container size follows from the
    layout alone: header and chunk table, the remainder plane, then one
    16-byte-padded 162-byte stream per chunk (or the RAW exponent bytes of a
    chunk too short for that to pay)."""
    rng = np.random.default_rng(3)
    if code == oracle.FP16:
        bits = (np.uint16(14 << 10) | rng.integers(0, 1 << 10, n).astype(np.uint16)
                | (rng.integers(0, 2, n).astype(np.uint16) << 15))
        plane = -(-11 * n // 8)
    else:
        mb = 3 if code == oracle.FP8_E4M3 else 2
        bits = ((np.uint8(6) << mb) | rng.integers(0, 1 << mb, n).astype(np.uint8)
                | (rng.integers(0, 2, n).astype(np.uint8) << 7)).astype(np.uint8)
        plane = -(-(1 + mb) * n // 8)
    C = -(-n // 65536)
    r16 = lambda v: -(-v // 16) * 16
    sizes = [min(65536, n - 65536 * c) for c in range(C)]
    # a chunk of 162 values or fewer is stored RAW (coding does not shrink it, R9)
    streams = sum(r16(162) if n_c > 162 else r16(n_c) for n_c in sizes)
    comp = oracle.compress(bits, code)
    assert comp.size == r16(r16(64 + 12 * C) + plane) + streams
    assert np.array_equal(oracle.decompress(comp, code, n), bits)


@pytest.mark.parametrize("code", [oracle.FP16, oracle.FP8_E4M3, oracle.FP8_E5M2])
@pytest.mark.parametrize("n", [1, 2, 3, 31, 33, 65535, 65537])
def test_random_roundtrip(code, n):
    rng = np.random.default_rng(n)
    bits = rng.integers(0, 1 << (16 if code == oracle.FP16 else 8), n).astype(np.uint16 if code == oracle.FP16 else np.uint8)
    comp = oracle.compress(bits, code)
    assert np.array_equal(oracle.decompress(comp, code, n), bits)
    assert comp.size <= oracle.container_bound(code, n)
