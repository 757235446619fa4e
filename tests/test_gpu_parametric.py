"""Parametric (Gaussian-model) tables on the GPU (uzip_compress_parametric)
against the oracle's MODE_PARAMETRIC (reading R25; ZipCCL abstract):
containers equal byte for byte, round trips bit-exact, for data the model
fits and for data it does not."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _gpu_parametric(bits, code, sigma):
    import torch

    import lossless_float_tensor_gb300 as uz

    n = bits.size
    x = gu.to_device(bits) if n else None
    cap = uz.uzip_max_compressed_size(code, n)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.full((), -1, dtype=torch.int64, device="cuda")
    status = torch.full((), -1, dtype=torch.int32, device="cuda")
    rc = uz.uzip_compress_parametric(x.data_ptr() if n else None, code, n, out.data_ptr(), cap, size.data_ptr(),
                                     status.data_ptr(), sigma, torch.cuda.current_stream().cuda_stream)
    assert rc == uz.UZIP_OK, uz.uzip_status_string(rc)
    torch.cuda.synchronize()
    return out[: int(size.item())].cpu().numpy(), int(status.item())


def _check(bits, code, sigma):
    want = oracle.compress(bits, code, mode=oracle.MODE_PARAMETRIC, sigma=sigma)
    got, status = _gpu_parametric(bits, code, sigma)
    assert status == 0
    assert got.size == want.size, (got.size, want.size)
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"{bad.size} bytes differ, first at {bad[0]} of {want.size}")
    back, st = gu.gpu_decompress(want, code, bits.size)
    assert st == 0 and np.array_equal(back, bits.view(gu.BITS[code]))
    return want


def _normal(code, n, sigma, tensor=0):
    if code == gu.BF16:
        return synth.normal_bf16(n, sigma, 17, tensor)
    if code == gu.FP32:
        return synth.normal_fp32(n, sigma, 17, tensor)
    if code == gu.FP16:
        return synth.normal_fp16(n, sigma, 17, tensor)
    return synth.normal_fp8(n, "e4m3" if code == gu.FP8_E4M3 else "e5m2", sigma, 17, tensor)


@pytest.mark.parametrize("code", [gu.BF16, gu.FP32, gu.FP16, gu.FP8_E4M3, gu.FP8_E5M2])
@pytest.mark.parametrize("n", [0, 1, 17, 65536, 3 * 65536 + 333])
def test_parametric_parity(code, n):
    sigma = 0.02 if code != gu.FP8_E4M3 else 0.5
    _check(_normal(code, n, sigma, tensor=n % 5), code, sigma)


@pytest.mark.parametrize("sigma", [1e-6, 3e-4, 0.7, 300.0])
def test_parametric_far_from_the_data(sigma):
    """N(0, 0.02) data under a model a long way off: still lossless, still
    the oracle's container (chunks the model cannot shrink go RAW)."""
    _check(synth.normal_bf16(2 * 65536 + 5, 0.02, 17, 7), gu.BF16, sigma)


def test_parametric_heavy_tails_and_random_bits():
    """c4's activations (0.5 t(4), outlier channels) with one chunk of random
    bits, under sigma = 0.7, and fp32 gradients with special values."""
    rng = np.random.default_rng(3)
    a = synth.c4(n=5 * 65536 + 99)
    a[2 * 65536:3 * 65536] = rng.integers(0, 1 << 16, 65536, dtype=np.uint16)
    comp = _check(a, gu.BF16, 0.7)
    lens = comp[64 + 8 * 6:64 + 12 * 6].view(np.uint32)
    assert lens[2] == 65536 | 0x80000000 and not lens[0] & 0x80000000
    _check(synth.c3(n=3 * 65536 + 11, specials=64), gu.FP32, 1e-3)


def test_parametric_c4_full():
    """The 1 GiB benchmark tensor under its model (0.5 t(4) has standard
    deviation 0.5 sqrt 2)."""
    _check(synth.c4(), gu.BF16, 0.5 * 2 ** 0.5)
