"""Pins for the oracle's sampled-table mode (reading R24; UCCL-Zip Fig. 5:
every block samples and builds its own table; survey next row 2).

The counts follow from the sampling rule by hand (positions 0, 16, 32, ...
of the chunk; a seen symbol counts 16 x its sample count, every unseen
symbol of the format's exponent range counts 1), and the table of a
constant chunk follows from those counts and R5 by hand.
"""
import numpy as np
import pytest

import oracle
import synth


def test_counts_of_a_constant_chunk():
    counts, total = oracle.sampled_counts(np.full(65536, 127, np.uint8), 8)
    assert counts[127] == 16 * 4096
    assert np.all(np.delete(counts, 127) == 1)
    assert total == 65536 + 255
    counts, total = oracle.sampled_counts(np.full(65536, 7, np.uint8), 5)  # fp16 / e5m2 exponent range
    assert counts[7] == 65536 and total == 65536 + 31
    assert np.all(counts[32:] == 0) and np.all(np.delete(counts[:32], 7) == 1)


def test_counts_read_only_every_sixteenth_position():
    e = np.full(65536, 120, np.uint8)
    e[::16] = 100
    counts, total = oracle.sampled_counts(e, 8)
    assert counts[100] == 65536 and counts[120] == 1 and total == 65536 + 255
    part = e[:1000]  # a partial chunk: positions 0, 16, ..., 992 (63 of them)
    counts, total = oracle.sampled_counts(part, 8)
    assert counts[100] == 16 * 63 and total == 16 * 63 + 255


def _stream_freqs(comp, c=0):
    C = int(comp[20:24].view(np.uint32)[0])
    exp_off = int(comp[32:40].view(np.uint64)[0])
    off = int(comp[64 + 8 * c:72 + 8 * c].view(np.uint64)[0])
    s = comp[exp_off + off:]
    bitmap = np.unpackbits(s[128:160], bitorder="little")
    K = int(bitmap.sum())
    return np.flatnonzero(bitmap), s[160:160 + 2 * K].view(np.uint16)


def test_constant_chunk_table_by_hand():
    """R5 on counts {127: 65536, others: 1}, total 65791: f[127] =
    floor(65536 * 4096 / 65791) = 4080, the 255 others are boosted to 1, the
    sum 4335 exceeds 4096 by 239, taken one by one from the largest, so
    f[127] = 3841 and K = 256 frequencies are stored."""
    x = np.full(65536, 0x3F80, np.uint16)  # bf16 1.0: exponent byte 127
    comp = oracle.compress(x, mode=oracle.MODE_SAMPLED)
    syms, f = _stream_freqs(comp)
    assert syms.size == 256 and f.size == 256
    assert f[127] == 3841 and np.all(np.delete(f, 127) == 1)
    assert np.array_equal(oracle.decompress(comp, oracle.BF16, x.size), x)


@pytest.mark.parametrize("code", [oracle.BF16, oracle.FP32, oracle.FP16, oracle.FP8_E4M3, oracle.FP8_E5M2])
def test_sampled_round_trip_and_cost(code):
    n = 2 * 65536 + 999
    if code == oracle.BF16:
        x = synth.c4(n=n)
    elif code == oracle.FP32:
        x = synth.normal_fp32(n)
    elif code == oracle.FP16:
        x = synth.normal_fp16(n)
    else:
        x = synth.normal_fp8(n, "e4m3" if code == oracle.FP8_E4M3 else "e5m2")
    full = oracle.compress(x, code)
    samp = oracle.compress(x, code, mode=oracle.MODE_SAMPLED)
    assert np.array_equal(oracle.decompress(samp, code, n), x.view(oracle.BITS_DTYPE[code]))
    # the full histogram is the better table; the sampled one stays close
    assert full.size <= samp.size <= 1.05 * full.size
