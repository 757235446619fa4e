"""Whole-message choice on the GPU (uzip_compress_gated) against the
oracle's MODE_GATE / MODE_RAW (reading R23; NCCLZ Sec. IV-C, Alg. 1):
containers equal byte for byte, round trips bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

ALL = [gu.BF16, gu.FP32, gu.FP16, gu.FP8_E4M3, gu.FP8_E5M2]


def _normal(code, n, tensor=0):
    if code == gu.BF16:
        return synth.normal_bf16(n, 0.02, 14, tensor)
    if code == gu.FP32:
        return synth.normal_fp32(n, 0.02, 14, tensor)
    if code == gu.FP16:
        return synth.normal_fp16(n, 0.02, 14, tensor)
    return synth.normal_fp8(n, "e4m3" if code == gu.FP8_E4M3 else "e5m2", 0.02, 14, tensor)


def _random(code, n, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 1 << (8 * gu.ELEM_BYTES[code]), n, dtype=np.uint64).astype(gu.BITS[code])
    return b.view(np.float16) if code == gu.FP16 else b


def _gated(bits, code, raw_below=0):
    import torch

    import lossless_float_tensor_gb300 as uz

    n = bits.size
    x = gu.to_device(bits) if n else None
    cap = uz.uzip_max_compressed_size(code, n)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.full((), -1, dtype=torch.int64, device="cuda")
    status = torch.full((), -1, dtype=torch.int32, device="cuda")
    st = uz.uzip_compress_gated(x.data_ptr() if n else None, code, n, out.data_ptr(), cap, size.data_ptr(),
                                status.data_ptr(), raw_below, torch.cuda.current_stream().cuda_stream)
    assert st == uz.UZIP_OK, uz.uzip_status_string(st)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out[: int(size.item())].cpu().numpy()


def _check(bits, code, mode, raw_below=0):
    want = oracle.compress(bits, code, mode=mode)
    got = _gated(bits, code, raw_below)
    assert got.size == want.size, (got.size, want.size)
    assert np.array_equal(got, want)
    back, st = gu.gpu_decompress(want, code, bits.size)
    assert st == 0 and np.array_equal(back, bits.view(gu.BITS[code]))
    return want


@pytest.mark.parametrize("code", ALL)
def test_gate_codes_normal_data(code):
    x = _normal(code, 5 * 65536 + 123)
    assert not oracle.gate_says_raw(x, code)
    want = _check(x, code, oracle.MODE_GATE)
    assert np.array_equal(want, oracle.compress(x, code))


@pytest.mark.parametrize("code", ALL)
def test_gate_on_random_bits(code):
    """8-bit exponents of random bits do not code below a byte each, so bf16
    and fp32 go RAW; the 4- and 5-bit exponents of fp16 and fp8 still code
    below the byte a RAW chunk spends on each, so those stay coded."""
    y = _random(code, 4 * 65536 + 77, 1)
    raw = oracle.gate_says_raw(y, code)
    assert raw == (code in (gu.BF16, gu.FP32))
    want = _check(y, code, oracle.MODE_GATE)
    assert (want.size == oracle.container_bound(code, y.size)) == raw


@pytest.mark.parametrize("code", ALL)
def test_size_threshold_forces_raw(code):
    x = _normal(code, 2 * 65536 + 5, tensor=2)
    _check(x, code, oracle.MODE_RAW, raw_below=x.size * gu.ELEM_BYTES[code] + 1)
    _check(x, code, oracle.MODE_GATE, raw_below=x.size * gu.ELEM_BYTES[code])  # not below: the sample decides


def test_gate_reads_only_the_sample():
    rng = np.random.default_rng(2)
    a = np.concatenate([rng.integers(0, 1 << 16, 32768).astype(np.uint16), synth.c1(n=3 * 65536)])
    want = _check(a, gu.BF16, oracle.MODE_GATE)
    assert want.size == oracle.container_bound(gu.BF16, a.size)


@pytest.mark.parametrize("n", [0, 1, 33, 32768, 65537])
def test_gate_edge_sizes(n):
    x = synth.c1(n=n) if n else np.zeros(0, np.uint16)
    _check(x, gu.BF16, oracle.MODE_GATE)
    _check(x, gu.BF16, oracle.MODE_RAW, raw_below=1 << 62)
