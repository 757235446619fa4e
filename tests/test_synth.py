"""Pins for the seeded input generators (no GPU): the counter-based generator
is SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), every value depends only on its stream and index
(so any partition or thread count gives the same tensor), and the bf16
rounding is IEEE round-to-nearest-even."""
import numpy as np
import pytest
import torch

import synth


def test_splitmix64_published_sequence():
    # the first three outputs of SplitMix64 from seed 0, as printed by the
    # generator's reference implementation
    with np.errstate(over="ignore"):
        z = np.array([synth.GAMMA * np.uint64(k) for k in (1, 2, 3)], dtype=np.uint64)
    assert [int(v) for v in synth.mix64(z)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_values_depend_only_on_stream_and_index(monkeypatch):
    n = synth.BLOCK + 12345  # spans two generation blocks
    whole = synth.normal_bf16(n, 0.02, 3, 1)
    parts = np.concatenate([synth.normal_bf16(1000, 0.02, 3, 1),
                            synth.normal_bf16(n - 1000, 0.02, 3, 1, start=1000)])
    assert np.array_equal(whole, parts)
    monkeypatch.setattr(synth, "_THREADS", 1)
    assert np.array_equal(whole, synth.normal_bf16(n, 0.02, 3, 1))
    assert not np.array_equal(whole, synth.normal_bf16(n, 0.02, 3, 2))  # another stream


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(1 << 16) * 10.0 ** rng.integers(-30, 30, 1 << 16)).astype(np.float32)
    # exact ties (low 16 bits 0x8000) of finite values, both parities of the
    # kept part: random sign, exponent 1..253, top 7 fraction bits
    sign = rng.integers(0, 2, 4096, dtype=np.uint32) << np.uint32(31)
    expo = rng.integers(1, 254, 4096, dtype=np.uint32) << np.uint32(23)
    frac = rng.integers(0, 1 << 7, 4096, dtype=np.uint32) << np.uint32(16)
    ties = sign | expo | frac | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), want)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_rounding_picks_the_nearest_finite_code(fmt):
    vals, codes = synth._fp8_positive_codes(fmt)
    # midpoints between neighbours go down, anything past them goes up
    mid = (vals[:-1] + vals[1:]) / 2
    assert np.array_equal(synth.round_to_fp8(mid, fmt), codes[:-1])
    assert np.array_equal(synth.round_to_fp8(np.nextafter(mid, np.inf), fmt), codes[1:])
    assert np.array_equal(synth.round_to_fp8(-vals, fmt), codes | np.uint8(0x80))
    assert synth.round_to_fp8(np.array([1e9]), fmt)[0] == codes[-1]  # saturates
