"""The allocation-free compression entry point.

Some callers only ever see the user's input and output buffers and are not
allowed to allocate device memory themselves (a per-message transport or
plugin hook working inside the application's memory plan, where cudaMalloc
could stall the device).  uzip_compress_noalloc serves them by keeping the
compressor's small work area in the library's own device array.  This file
checks, through the C ABI, that two calls in a row write exactly the
containers uzip_compress writes (the codec is lossless, so the tolerance is
zero: byte for byte), that the shared work area is cleared between calls, and
that a tensor beyond the array's limit is refused before any GPU work.  It is
named so that pytest collects it last.
"""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _regular(bits):
    got, status = gu.gpu_compress(bits)
    assert status == 0
    return got


def test_noalloc_matches_regular_entry_point_twice():
    import torch

    import lossless_float_tensor_gb300 as uz

    inputs = [synth.c4(n=37 * 65536 + 1234), synth.c3(n=5 * 65536 + 77, specials=64)]
    want = [_regular(b) for b in inputs]
    stream = torch.cuda.current_stream().cuda_stream
    dev = [gu.to_device(b) for b in inputs]
    outs, sizes, stats = [], [], []
    for b, x in zip(inputs, dev):  # two calls in a row on one stream, no sync between them
        d = gu.dtype_of(b)
        C = -(-b.size // 65536)
        cap = uz.uzip_max_compressed_size(d, b.size) - 16 - 8 * C
        out = torch.full((cap,), 0x5A, dtype=torch.uint8, device="cuda")
        size = torch.full((), -1, dtype=torch.int64, device="cuda")
        st = torch.full((), -1, dtype=torch.int32, device="cuda")
        rc = uz.uzip_compress_noalloc(x.data_ptr(), d, b.size, out.data_ptr(), cap, size.data_ptr(), st.data_ptr(), stream)
        assert rc == uz.UZIP_OK, uz.uzip_status_string(rc)
        outs.append(out), sizes.append(size), stats.append(st)
    torch.cuda.synchronize()
    for w, out, size, st in zip(want, outs, sizes, stats):
        assert int(st.item()) == 0
        assert int(size.item()) == w.size
        assert np.array_equal(out[: w.size].cpu().numpy(), w)


def test_noalloc_refuses_oversized_tensor_and_small_buffer():
    import torch

    import lossless_float_tensor_gb300 as uz

    fake = 1 << 40  # never dereferenced: both checks come first
    assert uz.uzip_compress_noalloc(fake, 0, uz.UZIP_NOALLOC_MAX_ELEMS + 1, fake, 1 << 62, None, None, 0) \
        == uz.UZIP_ERR_TOO_LARGE
    x = gu.to_device(synth.c1(n=65536 * 2))
    out = torch.empty(1000, dtype=torch.uint8, device="cuda")
    assert uz.uzip_compress_noalloc(x.data_ptr(), 0, 65536 * 2, out.data_ptr(), out.numel(), None, None,
                                    torch.cuda.current_stream().cuda_stream) == uz.UZIP_ERR_CAPACITY
