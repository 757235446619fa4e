"""Pins for the oracle's parametric (Gaussian-model) tables (reading R25;
ZipCCL abstract: exponent coding from the Gaussian shape of the values,
without statistics gathered online; survey next row 2).

The counts are checked against values worked by hand from a printed table of
the normal distribution (tests/golden/parametric_cases.txt), against scipy's
normal distribution for every format and a range of sigma, and against the
model's exact scale invariance (doubling sigma moves every binade up one
exponent).  The containers decode back losslessly whatever the data.
"""
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "parametric_cases.txt")
EBITS = {oracle.BF16: 8, oracle.FP32: 8, oracle.FP16: 5, oracle.FP8_E4M3: 4, oracle.FP8_E5M2: 5}


def _golden():
    cases = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (t.strip() for t in line.split("="))
        cases[key] = {int(a): int(b) for a, b in (p.split(":") for p in val.split())}
    return cases


@pytest.mark.parametrize("key,sigma", [("bf16.sigma1", 1.0), ("bf16.sigma2", 2.0)])
def test_counts_worked_by_hand(key, sigma):
    counts, total = oracle.parametric_counts(oracle.BF16, sigma)
    for e, c in _golden()[key].items():
        assert counts[e] == c, (e, counts[e], c)
    assert total == int(counts.sum())


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP32, oracle.FP16, oracle.FP8_E4M3, oracle.FP8_E5M2])
@pytest.mark.parametrize("sigma", [1e-3, 0.02, 0.7, 1.0, 37.5])
def test_counts_follow_the_normal_distribution(dtype, sigma):
    stats = pytest.importorskip("scipy.stats")
    eb = EBITS[dtype]
    bias = (1 << (eb - 1)) - 1
    counts, total = oracle.parametric_counts(dtype, sigma)
    for e in range(256):
        if e >= (1 << eb):
            assert counts[e] == 0
            continue
        hi = 2.0 ** (e - bias + 1) / sigma
        lo = 0.0 if e == 0 else 2.0 ** (e - bias) / sigma
        p = 2.0 * (stats.norm.sf(lo) - stats.norm.sf(hi))  # mass of the binade on both sides of zero
        want = max(1.0, np.floor(65536.0 * p + 0.5))
        assert abs(int(counts[e]) - want) <= 1, (e, counts[e], want)
        assert counts[e] >= 1
    assert total == int(counts.sum())
    assert abs(total - 65536) <= (1 << eb) + 8  # the mass, plus the raised counts


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16, oracle.FP8_E4M3])
def test_doubling_sigma_moves_every_binade_up_one_exponent(dtype):
    eb = EBITS[dtype]
    a, _ = oracle.parametric_counts(dtype, 0.3)
    b, _ = oracle.parametric_counts(dtype, 0.6)
    assert np.array_equal(b[2:1 << eb], a[1:(1 << eb) - 1])  # e >= 1: the same two erfc arguments, exactly


@pytest.mark.parametrize("sigma", [0.0, -1.0, float("inf"), float("nan")])
def test_sigma_must_be_finite_and_positive(sigma):
    counts, total = oracle.parametric_counts(oracle.BF16, sigma)
    assert total == 0 and not counts.any()
    with pytest.raises(oracle.OracleError):
        oracle.compress(synth.normal_bf16(1000, 0.02, 31, 0), mode=oracle.MODE_PARAMETRIC, sigma=sigma)


def test_every_chunk_uses_the_one_model_table():
    """Each coded chunk's stream lists every symbol of the format's range with
    the frequencies R5 makes of the model counts; the 500-value tail is
    stored RAW (its stream head alone, 160 + 512 bytes, exceeds it)."""
    bits = synth.normal_bf16(3 * 65536 + 500, 0.02, 31, 1)
    comp = oracle.compress(bits, mode=oracle.MODE_PARAMETRIC, sigma=0.02)
    counts, total = oracle.parametric_counts(oracle.BF16, 0.02)
    freq = oracle.normalise(counts, total)
    C = 4
    exp_off = int(comp[32:40].view(np.uint64)[0])
    lens = comp[64 + 8 * C:64 + 12 * C].view(np.uint32)
    assert lens[3] == 500 | 0x80000000
    for c in range(3):
        off = int(comp[64 + 8 * c:72 + 8 * c].view(np.uint64)[0])
        assert not lens[c] & 0x80000000
        s = comp[exp_off + off:]
        bitmap = np.unpackbits(s[128:160], bitorder="little")
        assert np.array_equal(np.nonzero(bitmap)[0], np.arange(256))
        f = s[160:160 + 512].view(np.uint16)
        assert np.array_equal(f, freq.astype(np.uint16))


@pytest.mark.parametrize("fmt", ["bf16", "fp32", "fp16", "e4m3"])
def test_round_trip_whatever_the_data(fmt):
    """Lossless for data the model fits, data it does not (heavy tails,
    random bits: those chunks go RAW) and a ragged tail."""
    rng = np.random.default_rng(5)
    if fmt == "bf16":
        bits, d = synth.c4(n=3 * 65536 + 77), oracle.BF16
        bits[65536:131072] = rng.integers(0, 1 << 16, 65536, dtype=np.uint16)
    elif fmt == "fp32":
        bits, d = synth.c3(n=2 * 65536 + 5, specials=64), oracle.FP32
    elif fmt == "fp16":
        bits, d = synth.normal_fp16(2 * 65536 + 9, 0.02).view(np.uint16), oracle.FP16
    else:
        bits, d = synth.normal_fp8(2 * 65536 + 3, "e4m3"), oracle.FP8_E4M3
    comp = oracle.compress(bits, d, mode=oracle.MODE_PARAMETRIC, sigma=0.05)
    assert np.array_equal(oracle.decompress(comp, d, bits.size), bits)


def test_size_near_the_full_histogram_when_the_model_fits():
    """N(0, 0.02) data with sigma = 0.02: within 2 % of the per-chunk exact
    tables (the model table lists all 256 symbols: +512 bytes a chunk)."""
    bits = synth.normal_bf16(8 * 65536, 0.02, 31, 2)
    exact = oracle.compress(bits).size
    model = oracle.compress(bits, mode=oracle.MODE_PARAMETRIC, sigma=0.02).size
    assert exact < model < 1.02 * exact
    wrong = oracle.compress(bits, mode=oracle.MODE_PARAMETRIC, sigma=2.0).size  # a hundredfold sigma
    assert wrong > model
