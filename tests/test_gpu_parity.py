"""GPU path against the oracle: containers equal byte for byte, round trips
bit-exact, corrupt containers rejected exactly where the oracle rejects them.
All calls go through the C ABI (lossless_float_tensor_gb300 ctypes layer)."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _parity(bits):
    want = oracle.compress(bits)
    got, status = gu.gpu_compress(bits)
    assert status == 0
    assert got.size == want.size, (got.size, want.size)
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"{bad.size} bytes differ, first at {bad[0]} of {want.size}")
    back, st = gu.gpu_decompress(want, gu.dtype_of(bits), bits.size)
    assert st == 0
    assert np.array_equal(back, bits)
    return want


@pytest.mark.parametrize("n", [0, 1, 31, 32, 33, 161, 1000, 4096, 65535, 65536, 65537, 100003, 131073])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_edge_sizes(n, dtype):
    if dtype == "bf16":
        bits = synth.normal_bf16(n, 0.02, 11, n % 89)
    else:
        bits = synth.c3(n=n, specials=min(16, n)) if n else np.zeros(0, np.uint32)
    _parity(bits)


@pytest.mark.parametrize("chunks", [1217, 2433])
def test_chunk_counts_past_a_full_grid(chunks):
    """Chunk counts one past a whole number of compressor rounds (8 warps per
    SM on 152 SMs) and a ragged tail: the trimmed grids still cover every
    chunk once, and the container is the oracle's."""
    _parity(synth.normal_bf16(chunks * 65536 - 77, 0.02, 14, chunks))


def test_decoder_two_rounds_with_ragged_tail():
    """More chunks than the decoder's resident warps (28 per SM on 152 SMs):
    the trimmed grid decodes every chunk of a compressed tensor exactly."""
    n = 4257 * 65536 + 5
    bits = synth.normal_bf16(n, 0.02, 15, 0)
    comp, status = gu.gpu_compress(bits)
    assert status == 0
    back, st = gu.gpu_decompress(comp, gu.dtype_of(bits), n)
    assert st == 0 and np.array_equal(back, bits)


def test_c1_full():
    comp = _parity(synth.c1())
    assert abs(comp.size / (2 << 20) - 0.661) < 0.01


def test_constant_and_random_chunks():
    """A constant chunk codes to 162 bytes; a random-bits chunk is stored RAW;
    a chunk of 6-bit exponent entropy overflows shared staging and takes the
    in-place path; ragged tails and single-symbol tails."""
    rng = np.random.default_rng(21)
    parts = [
        np.full(65536, 0x3C00, np.uint16),                                   # constant
        rng.integers(0, 1 << 16, 65536).astype(np.uint16),                   # random bits -> RAW
        ((rng.integers(60, 124, 65536) << 7) | rng.integers(0, 128, 65536)).astype(np.uint16),  # H = 6 bits
        ((rng.integers(110, 126, 65536) << 7) | rng.integers(0, 1 << 8, 65536)).astype(np.uint16),  # ~4 bits
        np.full(777, 0xBF80, np.uint16),                                     # short constant tail
    ]
    bits = np.concatenate(parts)
    comp = _parity(bits)
    C = 5
    lens = comp[64 + 8 * C:64 + 12 * C].view(np.uint32)
    assert lens[0] == 162
    assert lens[1] == (65536 | 0x80000000)
    assert not (lens[2] & 0x80000000) and (lens[2] & 0x7FFFFFFF) > 28 * 1024


def test_chunks_whose_tail_outgrows_the_slot():
    """Chunks coded from a slot's exponent bytes fall back to coding from the
    input when the words written from the chunk's end would outrun the bytes
    consumed: a constant chunk whose last 3072 values have random exponents
    (about 12 bits each), the same with the noise in the middle (the fast path
    holds), and a chunk of random bits ending in a constant run."""
    rng = np.random.default_rng(33)
    noisy_tail = np.full(65536, 0x3F80, np.uint16)
    noisy_tail[-3072:] = (rng.integers(0, 256, 3072) << 7).astype(np.uint16)
    noisy_mid = np.full(65536, 0x3F80, np.uint16)
    noisy_mid[30000:33072] = (rng.integers(0, 256, 3072) << 7).astype(np.uint16)
    random_then_const = rng.integers(0, 1 << 16, 65536).astype(np.uint16)
    random_then_const[-5000:] = 0x4000
    bits = np.concatenate([noisy_tail, noisy_mid, random_then_const, noisy_tail])
    comp = _parity(bits)
    lens = comp[64 + 8 * 4:64 + 12 * 4].view(np.uint32)
    assert not (lens[0] & 0x80000000) and lens[0] == lens[3]
    assert not (lens[1] & 0x80000000)


@pytest.mark.parametrize("fmt", ["bf16", "fp32"])
def test_streams_growing_faster_than_their_exponents_are_read(fmt):
    """Chunks whose top part (coded first) costs more than 8 bits a value:
    random exponents over a constant run (six fractions), and the 255 rarer
    exponents 64 to 128 times each over a constant run.  The words written
    from the slot's end reach the 1 KiB block of exponent bytes just read
    (all of them) or would pass blocks still to be read (80, 94 and 110 per
    exponent, which then code from the input); every chunk stays coded.
    Formats with 4- or 5-bit exponent fields cannot get there: 31 rare
    symbols add at most ~0.5 KiB of words over their bytes, against the
    4 KiB the slot keeps above the exponent bytes."""
    bits = synth.growth_bf16() if fmt == "bf16" else synth.growth_fp32()
    comp = _parity(bits)
    c = -(-bits.size // 65536)
    lens = comp[64 + 8 * c:64 + 12 * c].view(np.uint32)
    assert not np.any(lens & 0x80000000)
    assert np.all(lens[:11] > 20000)


def test_all_bf16_patterns_and_fp32_specials():
    x = np.arange(65536 * 3, dtype=np.uint32).astype(np.uint16)
    _parity(x)
    y = synth.c3(n=300000, specials=4096)
    _parity(y)


def test_uniform_closed_form_ratio():
    comp = _parity(synth.uniform_pm1_bf16(1 << 22))
    assert 0.625 <= comp.size / (2 << 22) <= 0.632


@pytest.mark.parametrize("t", range(7))
def test_c2_layer_tensors(t):
    _parity(synth.c2_tensor(t))


def test_c3_full():
    comp = _parity(synth.c3())
    assert abs(comp.size / (4 * synth.C3_N) - 0.837) < 0.01


def test_c4_full():
    bits = synth.c4()
    comp = _parity(bits)
    C = bits.size // 65536
    lens = comp[64 + 8 * C:64 + 12 * C].view(np.uint32)
    assert lens[synth.C4_RANDOM_CHUNK] & 0x80000000  # the random-bits chunk is RAW
    assert abs(comp.size / (2 * bits.size) - 0.675) < 0.01


def test_c5_message_ends():
    """First 64 Mi values of message 0 and the tail of the last message (which
    ends in a 4096-element partial chunk)."""
    _parity(synth.c5_message(0, n=1 << 26))
    sizes = synth.c5_message_sizes()
    k = len(sizes) - 1
    start = sizes[k] - (3 * 65536 + 4096)
    tail = synth.normal_bf16(3 * 65536 + 4096, 0.02, 5, 0, start=k * synth.C5_MESSAGE + start)
    _parity(tail)


def test_deterministic():
    bits = synth.c4(n=1 << 22)
    a, _ = gu.gpu_compress(bits)
    b, _ = gu.gpu_compress(bits)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# receiver validation: same verdict as the oracle on host-made corruptions

def test_corruptions_rejected_like_oracle():
    from tests.test_oracle_pins import _corruptions

    x = synth.normal_bf16(3 * 65536 + 777, 0.02, 8, 1)
    comp = oracle.compress(x)
    for name, (b, size) in _corruptions(comp, x.size, oracle.BF16).items():
        want, _ = oracle.decompress_status(b[:size], oracle.BF16, x.size)
        _, st = gu.gpu_decompress(b[:size], gu.BF16, x.size)
        assert want == oracle.ERR_CORRUPT
        assert st == want, name


def test_wrong_dtype_or_length_rejected():
    x = synth.normal_bf16(70000, 0.02, 8, 2)
    comp = oracle.compress(x)
    assert gu.gpu_decompress(comp, gu.FP32, x.size)[1] == oracle.ERR_CORRUPT
    assert gu.gpu_decompress(comp, gu.BF16, x.size - 1)[1] == oracle.ERR_CORRUPT
    assert gu.gpu_decompress(comp[:40], gu.BF16, x.size)[1] == oracle.ERR_CORRUPT


# ---------------------------------------------------------------------------
# bounded waits: a chunk that never publishes makes its successors time out

def test_lookback_timeout_reports_status():
    import lossless_float_tensor_gb300 as uz

    bits = synth.normal_bf16(4 * 65536, 0.02, 12, 0)
    got, status = gu.gpu_compress(bits, flags=uz.UZIP_TESTFLAG_SKIP_CHUNK0)
    assert status == uz.UZIP_ERR_TIMEOUT
    assert got.size == 0
    # the context is still healthy
    _parity(bits)


def test_query_size():
    import torch

    import lossless_float_tensor_gb300 as uz

    bits = synth.c1(n=300000)
    x = gu.to_device(bits)
    buf, size = uz.compress(x)
    st, total, dt, n = uz.uzip_query_size(buf.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0 and total == int(size.item()) and dt == 0 and n == bits.size
    assert total == oracle.compress(bits).size


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_pipeline_send(mode):
    import torch

    import lossless_float_tensor_gb300 as uz

    msgs = [synth.c5_message(0, n=(1 << 20) + 12345), synth.normal_bf16(1 << 21, 0.02, 13, 1),
            synth.normal_bf16(3 * 65536, 0.02, 13, 2)]
    d_msgs = [gu.to_device(m) for m in msgs]
    largest = max(m.size for m in msgs)
    cap = uz.uzip_max_compressed_size(0, largest)
    banks = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hcap = cap + 16 * (-(-largest // 65536))  # room for the streamed mode's progress words
    hb = [torch.zeros(hcap, dtype=torch.uint8).pin_memory() for _ in range(2)]
    sizes = torch.zeros(len(msgs), dtype=torch.int64).pin_memory()
    s0 = torch.cuda.Stream()
    s1 = torch.cuda.Stream()
    torch.cuda.synchronize()
    st = uz.uzip_pipeline_send(0, [t.data_ptr() for t in d_msgs], [m.size for m in msgs],
                               [b.data_ptr() for b in banks], cap, [h.data_ptr() for h in hb], hcap,
                               sizes.data_ptr(), mode, s0.cuda_stream, s1.cuda_stream)
    assert st == 0, uz.uzip_status_string(st)
    torch.cuda.synchronize()
    # messages under the default threshold travel as whole-message RAW
    # containers (NCCLZ Sec. IV-C)
    want = [oracle.compress(m, mode=oracle.MODE_RAW if 2 * m.size < uz.UZIP_PIPE_RAW_BELOW_DEFAULT else oracle.MODE_CHUNK)
            for m in msgs]
    assert [int(v) for v in sizes] == [w.size for w in want]
    # banks now hold messages 2 (bank 0) and 1 (bank 1)
    for k, b in ((2, 0), (1, 1)):
        assert np.array_equal(hb[b].numpy()[: want[k].size], want[k])


@pytest.mark.parametrize("mode", [0, 3, 4])
def test_pipeline_send_ex_keeps_every_container(mode):
    """uzip_pipeline_send_ex with one host bank per message: every container
    stays on the host and equals the oracle's, coded (threshold 0) or, under
    the threshold, whole-message RAW; each decodes back bit for bit."""
    import torch

    import lossless_float_tensor_gb300 as uz

    msgs = [synth.normal_bf16((1 << 20) + 7 * k, 0.02, 19, k) for k in range(4)]
    d_msgs = [gu.to_device(m) for m in msgs]
    largest = max(m.size for m in msgs)
    cap = uz.uzip_max_compressed_size(0, largest)
    banks = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hcap = cap + 16 * (-(-largest // 65536))
    for raw_below, omode in ((0, oracle.MODE_CHUNK), (1 << 30, oracle.MODE_RAW)):
        hb = [torch.zeros(hcap, dtype=torch.uint8).pin_memory() for _ in msgs]
        sizes = torch.zeros(len(msgs), dtype=torch.int64).pin_memory()
        s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        st = uz.uzip_pipeline_send_ex(0, [t.data_ptr() for t in d_msgs], [m.size for m in msgs],
                                      [b.data_ptr() for b in banks], cap, [h.data_ptr() for h in hb], hcap,
                                      sizes.data_ptr(), mode, raw_below, s0.cuda_stream, s1.cuda_stream)
        assert st == 0, uz.uzip_status_string(st)
        torch.cuda.synchronize()
        for k, m in enumerate(msgs):
            want = oracle.compress(m, mode=omode)
            assert int(sizes[k]) == want.size
            got = hb[k].numpy()[: want.size]
            assert np.array_equal(got, want)
            back, status = gu.gpu_decompress(got, gu.BF16, m.size)
            assert status == 0 and np.array_equal(back, m)


def _send_all(msgs, mode, raw_below):
    """uzip_pipeline_send_ex with one host bank per message; returns the
    containers as numpy arrays."""
    import torch

    import lossless_float_tensor_gb300 as uz

    d_msgs = [gu.to_device(m) for m in msgs]
    largest = max(m.size for m in msgs)
    cap = uz.uzip_max_compressed_size(0, largest)
    banks = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hcap = cap + 16 * (-(-largest // 65536))
    hb = [torch.zeros(hcap, dtype=torch.uint8).pin_memory() for _ in msgs]
    sizes = torch.zeros(len(msgs), dtype=torch.int64).pin_memory()
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    st = uz.uzip_pipeline_send_ex(0, [t.data_ptr() for t in d_msgs], [m.size for m in msgs],
                                  [b.data_ptr() for b in banks], cap, [h.data_ptr() for h in hb], hcap,
                                  sizes.data_ptr(), mode, raw_below, s0.cuda_stream, s1.cuda_stream)
    assert st == 0, uz.uzip_status_string(st)
    torch.cuda.synchronize()
    return [hb[k].numpy()[: int(sizes[k])].copy() for k in range(len(msgs))]


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_pipeline_many_raw_messages_wrap_the_bank_slots(mode):
    """40 messages under the RAW threshold, 16 to 65,537 values: each device
    bank is cut into 8 slots, so message k reuses the slot of message k - 16
    (after its copy); every container equals the oracle's whole-message RAW
    container (NCCLZ Sec. IV-C)."""
    msgs = [synth.normal_bf16(16 + ((k * 7919) % 65522), 0.02, 23, k) for k in range(40)]
    got = _send_all(msgs, mode, 1 << 30)
    for k, m in enumerate(msgs):
        want = oracle.compress(m, mode=oracle.MODE_RAW)
        assert got[k].size == want.size and np.array_equal(got[k], want), f"message {k}"


@pytest.mark.parametrize("mode", [0, 3, 4])
def test_pipeline_mixed_raw_and_coded_messages(mode):
    """Messages on both sides of an explicit 1 MiB threshold, interleaved:
    the small ones travel RAW, the large ones coded, through two banks."""
    msgs = [synth.normal_bf16(((1 << 18) if k % 2 else (1 << 19)) + 31 * k, 0.02, 29, k) for k in range(7)]
    got = _send_all(msgs, mode, 1 << 20)
    for k, m in enumerate(msgs):
        want = oracle.compress(m, mode=oracle.MODE_RAW if 2 * m.size < (1 << 20) else oracle.MODE_CHUNK)
        assert got[k].size == want.size and np.array_equal(got[k], want), f"message {k}"
