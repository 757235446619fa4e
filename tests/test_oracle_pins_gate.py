"""Pins for the oracle's whole-message modes (reading R23; NCCLZ Sec. IV-C,
Alg. 1: a message whose coding would not pay travels RAW).

A whole-message RAW container has a closed form (every chunk's exponent
bytes at offset 65536 c, RAW flag set, the size bound), and the gate's
decision depends only on the first 64 KiB of input, which the mixed
messages below expose from both sides.
"""
import numpy as np
import pytest

import oracle
import synth


def _u32(b, off):
    return int(b[off:off + 4].view(np.uint32)[0])


def _u64(b, off):
    return int(b[off:off + 8].view(np.uint64)[0])


@pytest.mark.parametrize("n", [1, 65536, 3 * 65536 + 17])
def test_raw_mode_closed_form(n):
    x = synth.c1(n=n)
    comp = oracle.compress(x, mode=oracle.MODE_RAW)
    assert comp.size == oracle.container_bound(oracle.BF16, n)
    C = -(-n // 65536)
    exp_off = _u64(comp, 32)
    exps, rem = oracle.split(x)
    for c in range(C):
        n_c = min(65536, n - 65536 * c)
        assert _u64(comp, 64 + 8 * c) == 65536 * c
        assert _u32(comp, 64 + 8 * C + 4 * c) == (n_c | 0x80000000)
        assert np.array_equal(comp[exp_off + 65536 * c: exp_off + 65536 * c + n_c], exps[65536 * c: 65536 * c + n_c])
    assert np.array_equal(oracle.decompress(comp, oracle.BF16, n), x)


def test_gate_codes_normal_data_and_sends_random_bits_raw():
    x = synth.c1(n=5 * 65536)
    assert not oracle.gate_says_raw(x)
    assert np.array_equal(oracle.compress(x, mode=oracle.MODE_GATE), oracle.compress(x))
    y = np.random.default_rng(4).integers(0, 1 << 16, 5 * 65536).astype(np.uint16)
    assert oracle.gate_says_raw(y)
    assert np.array_equal(oracle.compress(y, mode=oracle.MODE_GATE), oracle.compress(y, mode=oracle.MODE_RAW))


def test_gate_sees_only_the_first_64_kib():
    """bf16: the sample is the first 32768 values.  Random bits there and
    normal values after: RAW, although most chunks would code.  Normal
    values there and random bits after: coded per chunk (the later chunks
    go RAW one by one)."""
    rng = np.random.default_rng(5)
    rnd = rng.integers(0, 1 << 16, 32768).astype(np.uint16)
    nrm = synth.c1(n=4 * 65536)
    a = np.concatenate([rnd, nrm])
    assert oracle.gate_says_raw(a)
    assert oracle.compress(a, mode=oracle.MODE_GATE).size == oracle.container_bound(oracle.BF16, a.size)
    b = np.concatenate([nrm[:32768], rng.integers(0, 1 << 16, 4 * 65536).astype(np.uint16)])
    assert not oracle.gate_says_raw(b)
    assert np.array_equal(oracle.compress(b, mode=oracle.MODE_GATE), oracle.compress(b))
    # a sample of 32768 values: random bits in the first 32768 values only
    c = np.concatenate([rng.integers(0, 1 << 16, 32768).astype(np.uint16), nrm[:32768], nrm])
    assert oracle.gate_says_raw(c)


@pytest.mark.parametrize("code,sample", [(oracle.FP32, 16384), (oracle.FP16, 32768), (oracle.FP8_E4M3, 65536)])
def test_gate_sample_is_64_kib_of_input(code, sample):
    assert int(oracle.lib().orc_gate_sample_elems(code, 10 ** 9)) == sample
    assert int(oracle.lib().orc_gate_sample_elems(code, 1000)) == 1000
