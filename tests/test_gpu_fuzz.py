"""The GPU decoder against the oracle's on seeded random corruptions:
the same verdict (OK or CORRUPT) on every damaged container, and the same
output values whenever the damage cannot be detected."""
import numpy as np
import pytest

import oracle
from tests import _fuzz
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

COUNT = 150


@pytest.mark.parametrize("case", range(5))
def test_random_corruptions_match_the_oracle(case):
    bits, dtype = _fuzz.fuzz_input(case)
    n = bits.size
    comp = oracle.compress(bits, dtype)
    accepted = 0
    for kind, b, d in _fuzz.corruptions(comp, dtype, n, COUNT, seed=100 + case):
        want, wout = oracle.decompress_status(b, dtype, n)
        got, st = gu.gpu_decompress(b, dtype, n)
        assert st == want, (kind, d)
        if want == oracle.OK:
            accepted += 1
            assert np.array_equal(got, wout), (kind, d)
    assert 0 < accepted < COUNT
