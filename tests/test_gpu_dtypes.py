"""GPU path against the oracle for fp16 and the two fp8 formats (the dtype
sweep of UCCL-Zip Fig. 12): containers equal byte for byte, round trips
bit-exact.  All calls go through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

NEW = [gu.FP16, gu.FP8_E4M3, gu.FP8_E5M2]
NAMES = {gu.FP16: "fp16", gu.FP8_E4M3: "e4m3", gu.FP8_E5M2: "e5m2"}


def _normal(code, n, std=0.02, tensor=0):
    if code == gu.FP16:
        return synth.normal_fp16(n, std, tensor=tensor)
    return synth.normal_fp8(n, NAMES[code], std, tensor=tensor)


def _random_bits(code, n, seed):
    rng = np.random.default_rng(seed)
    if code == gu.FP16:
        return rng.integers(0, 1 << 16, n).astype(np.uint16).view(np.float16)
    return rng.integers(0, 256, n).astype(np.uint8)


def _parity(bits, code):
    want = oracle.compress(bits, code)
    got, status = gu.gpu_compress(bits, dtype=code)
    assert status == 0
    assert got.size == want.size, (got.size, want.size)
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"{bad.size} bytes differ, first at {bad[0]} of {want.size}")
    back, st = gu.gpu_decompress(want, code, bits.size)
    assert st == 0
    assert np.array_equal(back, bits.view(gu.BITS[code]))
    return want


@pytest.mark.parametrize("n", [1, 2, 3, 31, 33, 161, 1000, 4097, 65535, 65536, 65537, 131073])
@pytest.mark.parametrize("code", NEW)
def test_edge_sizes(code, n):
    _parity(_normal(code, n, tensor=n % 7), code)


@pytest.mark.parametrize("code", NEW)
def test_all_patterns_and_chunk_kinds(code):
    """Every bit pattern (NaN, infinities, subnormals, both zeros), then a
    constant chunk, a random-bits chunk and a normal chunk with a ragged tail."""
    if code == gu.FP16:
        pats = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
        const = np.full(65536, 0x3C00, np.uint16).view(np.float16)
    else:
        pats = np.tile(np.arange(256, dtype=np.uint8), 256)
        const = np.full(65536, 0x38, np.uint8)
    bits = np.concatenate([pats, const, _random_bits(code, 65536, 5), _normal(code, 70001, tensor=3)])
    comp = _parity(bits, code)
    C = -(-bits.size // 65536)
    lens = comp[64 + 8 * C:64 + 12 * C].view(np.uint32)
    assert lens[1] == 162  # constant exponent: stream head plus one frequency


@pytest.mark.parametrize("code", NEW)
def test_large_normal(code):
    comp = _parity(_normal(code, 1 << 24, tensor=9), code)
    assert comp.size < (1 << 24) * gu.ELEM_BYTES[code]


@pytest.mark.parametrize("code", NEW)
def test_torch_round_trip(code):
    import torch

    import lossless_float_tensor_gb300 as uz

    table = uz._torch_dtypes()
    if code not in table:
        pytest.skip("torch lacks this dtype")
    bits = _normal(code, 300001, tensor=4)
    x = torch.from_numpy(bits.view(gu.BITS[code]).view(np.uint8 if code != gu.FP16 else np.int16).copy()).cuda()
    x = x.view(table[code])
    buf, size = uz.compress(x)
    comp = uz.compressed_bytes(buf, size)
    assert np.array_equal(comp.cpu().numpy(), oracle.compress(bits, code))
    y = uz.decompress(comp, table[code], x.numel())
    assert torch.equal(y.view(torch.uint8), x.view(torch.uint8))


@pytest.mark.parametrize("code", NEW)
def test_corruptions_rejected_like_oracle(code):
    from tests.test_oracle_pins import _corruptions

    x = _normal(code, 3 * 65536 + 777, tensor=6)
    comp = oracle.compress(x, code)
    for name, (b, size) in _corruptions(comp, x.size, code).items():
        want, _ = oracle.decompress_status(b[:size], code, x.size)
        _, st = gu.gpu_decompress(b[:size], code, x.size)
        assert want == oracle.ERR_CORRUPT, name
        assert st == want, name


@pytest.mark.parametrize("code", NEW)
def test_noalloc_matches_regular(code):
    import torch

    import lossless_float_tensor_gb300 as uz

    x = _normal(code, 9 * 65536 + 4321, tensor=8)
    want = oracle.compress(x, code)
    d = gu.to_device(x)
    C = -(-x.size // 65536)
    cap = uz.uzip_max_compressed_size(code, x.size) - 16 - 8 * C
    out = torch.full((cap,), 0x5A, dtype=torch.uint8, device="cuda")
    size = torch.full((), -1, dtype=torch.int64, device="cuda")
    rc = uz.uzip_compress_noalloc(d.data_ptr(), code, x.size, out.data_ptr(), cap, size.data_ptr(), None,
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == uz.UZIP_OK
    torch.cuda.synchronize()
    assert int(size.item()) == want.size
    assert np.array_equal(out[: want.size].cpu().numpy(), want)


@pytest.mark.parametrize("code", NEW)
def test_pipeline_send_sized(code):
    import torch

    import lossless_float_tensor_gb300 as uz

    msgs = [_normal(code, (1 << 20) + 321, tensor=10), _normal(code, 3 * 65536, tensor=11)]
    d_msgs = [gu.to_device(m) for m in msgs]
    cap = uz.uzip_max_compressed_size(code, max(m.size for m in msgs))
    banks = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hb = [torch.zeros(cap, dtype=torch.uint8).pin_memory() for _ in range(2)]
    sizes = torch.zeros(len(msgs), dtype=torch.int64).pin_memory()
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    st = uz.uzip_pipeline_send(code, [t.data_ptr() for t in d_msgs], [m.size for m in msgs], [b.data_ptr() for b in banks],
                               cap, [h.data_ptr() for h in hb], cap, sizes.data_ptr(), uz.UZIP_PIPE_SIZED,
                               s0.cuda_stream, s1.cuda_stream)
    assert st == 0, uz.uzip_status_string(st)
    torch.cuda.synchronize()
    for k, m in enumerate(msgs):  # under the default threshold: whole-message RAW
        mode = oracle.MODE_RAW if m.nbytes < uz.UZIP_PIPE_RAW_BELOW_DEFAULT else oracle.MODE_CHUNK
        want = oracle.compress(m, code, mode=mode)
        assert int(sizes[k]) == want.size
        assert np.array_equal(hb[k % 2].numpy()[: want.size], want)


def _msgs_of(code):
    CH = 65536
    if code == gu.BF16:
        msgs = [synth.normal_bf16(n, 0.02, 8, 30 + t) for t, n in enumerate((5 * CH + 77, 2 * CH, CH + 1))]
        rnd = np.random.default_rng(31).integers(0, 1 << 16, 2 * CH + 9, dtype=np.uint16)
    elif code == gu.FP32:
        msgs = [synth.normal_fp32(n, 0.02, tensor=30 + t) for t, n in enumerate((5 * CH + 77, 2 * CH, CH + 1))]
        rnd = np.random.default_rng(31).integers(0, 1 << 32, 2 * CH + 9, dtype=np.uint64).astype(np.uint32)
    else:
        msgs = [_normal(code, n, tensor=30 + t) for t, n in enumerate((5 * CH + 77, 2 * CH, CH + 1))]
        rnd = _random_bits(code, 2 * CH + 9, 31)
    return msgs + [rnd]  # the last one's chunks are stored RAW


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("code", [gu.BF16, gu.FP32] + NEW)
def test_pipeline_coded_messages_every_format_and_mode(code, mode):
    """Coded containers (no whole-message RAW) of every element format through
    every pipeline mode, including the streamed one, whose early copies of
    finished remainder and stream runs follow each format's plane layout;
    every container equals the oracle's."""
    import torch

    import lossless_float_tensor_gb300 as uz

    msgs = _msgs_of(code)
    d_msgs = [gu.to_device(m) for m in msgs]
    largest = max(m.size for m in msgs)
    cap = uz.uzip_max_compressed_size(code, largest)
    banks = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hcap = cap + 16 * (-(-largest // 65536))  # the streamed mode's progress words
    hb = [torch.zeros(hcap, dtype=torch.uint8).pin_memory() for _ in msgs]
    sizes = torch.zeros(len(msgs), dtype=torch.int64).pin_memory()
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    st = uz.uzip_pipeline_send_ex(code, [t.data_ptr() for t in d_msgs], [m.size for m in msgs],
                                  [b.data_ptr() for b in banks], cap, [h.data_ptr() for h in hb], hcap,
                                  sizes.data_ptr(), mode, 0, s0.cuda_stream, s1.cuda_stream)
    assert st == 0, uz.uzip_status_string(st)
    torch.cuda.synchronize()
    for k, m in enumerate(msgs):
        want = oracle.compress(m, code)
        assert int(sizes[k]) == want.size, k
        assert np.array_equal(hb[k].numpy()[: want.size], want), k
