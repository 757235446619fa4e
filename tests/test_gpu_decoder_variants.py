"""Both decoders on the same containers: the byte-table decoder (two shared
loads per step) and the packed-table decoder that grids of at most 608
chunks take (one u32 per slot: f - 1, the symbol and slot - cum).  Each
output is compared with the oracle's bit for bit, including the corners of
the packed entry: a constant chunk (one symbol, f = 4096), two symbols, and a
coded chunk with all 256 exponent values present."""
import numpy as np
import pytest

import oracle
import synth
from tests import _fuzz
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CH = 65536


def _cases():
    rng = np.random.default_rng(41)
    out = []
    for case in range(5):
        out.append(_fuzz.fuzz_input(case))
    const = np.full(2 * CH + 300, 0x3C00, np.uint16)  # one exponent everywhere: f = 4096
    const[::7] ^= 0x8000  # signs and fractions vary, the exponent does not
    const[3::5] ^= 0x0055
    out.append((const, gu.BF16))
    two = synth.normal_bf16(CH, 0.02, 8, 9)
    two = (two & 0x807F) | np.where(rng.random(CH) < 0.3, 0x3F00, 0x3E80).astype(np.uint16)
    out.append((two, gu.BF16))
    allsym = synth.normal_bf16(3 * CH, 0.02, 8, 10)
    allsym[: 256 * 40] = (allsym[: 256 * 40] & 0x807F) | (np.repeat(np.arange(256, dtype=np.uint16), 40) << 7)
    out.append((allsym, gu.BF16))
    return out


def _set(variant):
    import lossless_float_tensor_gb300 as uz

    uz.library().uzip_debug_set_decode_variant(variant)


@pytest.mark.parametrize("variant", [0, 1, -1])
def test_both_decoders_match_the_oracle(variant):
    _set(variant)
    try:
        for bits, dtype in _cases():
            comp = oracle.compress(bits, dtype)
            want = oracle.decompress(comp, dtype, bits.size)
            got, st = gu.gpu_decompress(comp, dtype, bits.size)
            assert st == 0, (variant, dtype, bits.size)
            assert np.array_equal(got, want), (variant, dtype, bits.size)
            assert np.array_equal(want, bits.view(want.dtype))
    finally:
        _set(-1)


def test_all_symbols_chunk_is_coded():
    bits, dtype = _cases()[-1]
    comp = oracle.compress(bits, dtype)
    C = -(-bits.size // CH)
    lw = np.frombuffer(comp[64 + 8 * C:64 + 12 * C].tobytes(), np.uint32)
    assert not lw[0] >> 31  # chunk 0, with all 256 exponents, is coded, not RAW
    exp_off = int(np.frombuffer(comp[32:40].tobytes(), np.uint64)[0])
    off = int(np.frombuffer(comp[64:72].tobytes(), np.uint64)[0])
    assert (comp[exp_off + off + 128:exp_off + off + 160] == 0xFF).all()  # every symbol present


@pytest.mark.parametrize("variant", [0, 1])
def test_packed_decoder_on_a_grid_past_one_round(variant):
    """700 chunks: past the automatic switch (608), decoded by each variant
    forced."""
    bits = synth.normal_bf16(700 * CH - 1234, 0.02, 8, 11)
    comp = oracle.compress(bits)
    _set(variant)
    try:
        got, st = gu.gpu_decompress(comp, gu.BF16, bits.size)
    finally:
        _set(-1)
    assert st == 0 and np.array_equal(got, bits)
