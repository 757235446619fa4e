"""The allocation-free compression entry point.

Some callers only ever see the user's input and output buffers and are not
allowed to allocate device memory themselves (a per-message transport or
plugin hook working inside the application's memory plan, where cudaMalloc
could stall the device).  uzip_compress_noalloc serves them by keeping the
compressor's small work area in the library's own device array.  This file
checks, through the C ABI, that two calls in a row write exactly the
containers the oracle writes (the codec is lossless, so the tolerance is
zero: byte for byte), that the output buffer may be exactly as large as the
largest container the header documents and that nothing past the container
is touched, that the shared work area is cleared between calls, and that a
tensor beyond the array's limit is refused before any GPU work.  It is named
so that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A
FIELD_BITS = {gu.BF16: 8, gu.FP32: 24, gu.FP16: 11, gu.FP8_E4M3: 4, gu.FP8_E5M2: 3}


def documented_minimum(dtype, n):
    """The largest container, as include/uzip.h states it for the
    allocation-free entry point: round16(round16(64 + 12 C) + P)
    + (C - 1) * 65536 + round16(n - (C - 1) * 65536), or 64 for n = 0."""
    r16 = lambda v: (v + 15) // 16 * 16
    if n == 0:
        return 64
    C = -(-n // 65536)
    P = -(-n * FIELD_BITS[dtype] // 8)
    return r16(r16(64 + 12 * C) + P) + (C - 1) * 65536 + r16(n - (C - 1) * 65536)


def _inputs():
    rng = np.random.default_rng(41)
    # bf16 activations with a ragged last chunk, and one all-random-bits chunk
    # in the middle so the RAW writer runs
    a = synth.c4(n=37 * 65536 + 1234)
    a[5 * 65536:6 * 65536] = rng.integers(0, 1 << 16, 65536, dtype=np.uint16)
    b = synth.c3(n=5 * 65536 + 77, specials=64)  # fp32 gradients with specials
    return [a, b]


def test_noalloc_at_documented_minimum_matches_oracle_twice():
    import torch

    import lossless_float_tensor_gb300 as uz

    inputs = _inputs()
    want = [oracle.compress(b) for b in inputs]
    stream = torch.cuda.current_stream().cuda_stream
    dev = [gu.to_device(b) for b in inputs]
    outs, sizes, stats, caps = [], [], [], []
    for b, x in zip(inputs, dev):  # two calls in a row on one stream, no sync between them
        d = gu.dtype_of(b)
        cap = documented_minimum(d, b.size)
        assert cap == oracle.container_bound(d, b.size)
        out = torch.full((cap,), SENTINEL, dtype=torch.uint8, device="cuda")
        size = torch.full((), -1, dtype=torch.int64, device="cuda")
        st = torch.full((), -1, dtype=torch.int32, device="cuda")
        rc = uz.uzip_compress_noalloc(x.data_ptr(), d, b.size, out.data_ptr(), cap, size.data_ptr(), st.data_ptr(), stream)
        assert rc == uz.UZIP_OK, uz.uzip_status_string(rc)
        outs.append(out), sizes.append(size), stats.append(st), caps.append(cap)
    torch.cuda.synchronize()
    for w, out, size, st, cap in zip(want, outs, sizes, stats, caps):
        assert int(st.item()) == 0
        total = int(size.item())
        assert total == w.size
        host = out.cpu().numpy()
        assert np.array_equal(host[:total], w)
        assert np.all(host[total:cap] == SENTINEL), "bytes past the container were written"
    # the RAW chunk really is stored RAW
    C = -(-inputs[0].size // 65536)
    lens = want[0][64 + 8 * C:64 + 12 * C].view(np.uint32)
    assert lens[5] & 0x80000000


def test_noalloc_refuses_oversized_tensor_and_small_buffer():
    import torch

    import lossless_float_tensor_gb300 as uz

    fake = 1 << 40  # never dereferenced: both checks come first
    assert uz.uzip_compress_noalloc(fake, 0, uz.UZIP_NOALLOC_MAX_ELEMS + 1, fake, 1 << 62, None, None, 0) \
        == uz.UZIP_ERR_TOO_LARGE
    n = 65536 * 2
    x = gu.to_device(synth.c1(n=n))
    cap = documented_minimum(gu.BF16, n) - 16
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    assert uz.uzip_compress_noalloc(x.data_ptr(), 0, n, out.data_ptr(), cap, None, None,
                                    torch.cuda.current_stream().cuda_stream) == uz.UZIP_ERR_CAPACITY
