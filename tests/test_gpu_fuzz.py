"""Both GPU decoders against the oracle's on seeded random corruptions:
the same verdict (OK or CORRUPT) on every damaged container, and the same
output values whenever the damage cannot be detected."""
import numpy as np
import pytest

import oracle
from tests import _fuzz
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

COUNT = 150


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("case", range(5))
def test_random_corruptions_match_the_oracle(case, variant):
    """variant: the byte-table decoder (0) or the packed-table one (1)."""
    import lossless_float_tensor_gb300 as uz

    bits, dtype = _fuzz.fuzz_input(case)
    n = bits.size
    comp = oracle.compress(bits, dtype)
    accepted = 0
    uz.library().uzip_debug_set_decode_variant(variant)
    try:
        for kind, b, d in _fuzz.corruptions(comp, dtype, n, COUNT, seed=100 + case):
            want, wout = oracle.decompress_status(b, dtype, n)
            got, st = gu.gpu_decompress(b, dtype, n)
            assert st == want, (kind, d)
            if want == oracle.OK:
                accepted += 1
                assert np.array_equal(got, wout), (kind, d)
    finally:
        uz.library().uzip_debug_set_decode_variant(-1)
    assert 0 < accepted < COUNT
