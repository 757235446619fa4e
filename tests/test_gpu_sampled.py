"""Sampled tables on the GPU (UZIP_FLAG_SAMPLED_TABLES) against the
oracle's MODE_SAMPLED (reading R24; UCCL-Zip Fig. 5): containers equal byte
for byte, round trips bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _data(code, n, tensor=0):
    if code == gu.BF16:
        return synth.c4(n=n)
    if code == gu.FP32:
        return synth.normal_fp32(n, 0.02, 15, tensor)
    if code == gu.FP16:
        return synth.normal_fp16(n, 0.02, 15, tensor)
    return synth.normal_fp8(n, "e4m3" if code == gu.FP8_E4M3 else "e5m2", 0.02, 15, tensor)


def _check(bits, code):
    import lossless_float_tensor_gb300 as uz

    want = oracle.compress(bits, code, mode=oracle.MODE_SAMPLED)
    got, status = gu.gpu_compress(bits, flags=uz.UZIP_FLAG_SAMPLED_TABLES, dtype=code)
    assert status == 0
    assert got.size == want.size, (got.size, want.size)
    assert np.array_equal(got, want)
    back, st = gu.gpu_decompress(want, code, bits.size)
    assert st == 0 and np.array_equal(back, bits.view(gu.BITS[code]))
    return want


@pytest.mark.parametrize("code", [gu.BF16, gu.FP32, gu.FP16, gu.FP8_E4M3, gu.FP8_E5M2])
@pytest.mark.parametrize("n", [1, 17, 1000, 65536, 3 * 65536 + 333])
def test_sampled_parity(code, n):
    _check(_data(code, n, tensor=n % 5), code)


def test_sampled_chunk_kinds():
    """Constant chunk (one seen symbol, 255 unseen at 1), random bits (RAW),
    a chunk whose every 16th value differs from the rest, ragged tail."""
    rng = np.random.default_rng(9)
    inter = np.full(65536, 0x3C00, np.uint16)
    inter[::16] = 0x4200
    bits = np.concatenate([np.full(65536, 0x3F80, np.uint16), rng.integers(0, 1 << 16, 65536).astype(np.uint16),
                           inter, synth.c1(n=12345)])
    _check(bits, gu.BF16)


def test_sampled_full_c4_slice():
    bits = synth.c4(n=1 << 24)
    want = _check(bits, gu.BF16)
    assert want.size <= 1.03 * oracle.compress(bits).size
