"""The oracle's decoder on seeded random corruptions of its own containers.

It must never fail other than by reporting CORRUPT, and on the damage that
no check can see it must do exactly what the layout implies: a flipped
bit of the remainder plane or of a RAW chunk changes one bit of one output
value, a flipped bit of padding or of the reserved header bytes changes
nothing, and a flipped bit of a validated header field is rejected.
"""
import numpy as np
import pytest

import oracle
from tests import _fuzz

COUNT = 150


@pytest.mark.parametrize("case", range(5))
def test_random_corruptions(case):
    bits, dtype = _fuzz.fuzz_input(case)
    n = bits.size
    comp = oracle.compress(bits, dtype)
    seen = set()
    for kind, b, d in _fuzz.corruptions(comp, dtype, n, COUNT, seed=100 + case):
        st, out = oracle.decompress_status(b, dtype, n)
        assert st in (oracle.OK, oracle.ERR_CORRUPT), kind
        seen.add(kind)
        if kind == "header":
            assert st == oracle.ERR_CORRUPT, d
        elif kind in ("reserved", "gap", "stream_pad"):
            assert st == oracle.OK and np.array_equal(out, bits), (kind, d)
        elif kind in ("plane", "raw"):
            assert st == oracle.OK, (kind, d)
            diff = np.nonzero(out != bits)[0]
            e = _fuzz.expected_flip(comp, dtype, n, d[0], d[1], kind)
            if e is None:
                assert diff.size == 0, (kind, d)
            else:
                assert diff.tolist() == [e[0]], (kind, d)
                assert int(out[e[0]]) ^ int(bits[e[0]]) == 1 << e[1], (kind, d)
    # the draw reaches every region the container has
    assert {"header", "table", "plane", "coded", "byte", "truncate"} <= seen
    if case == 0:
        assert "raw" in seen


def test_layout_regions_tile_the_container():
    bits, dtype = _fuzz.fuzz_input(0)
    comp = oracle.compress(bits, dtype)
    reg = _fuzz.layout(comp, dtype, bits.size)
    spans = sorted(r for rs in reg.values() for r in rs)
    assert spans[0][0] == 0
    for (lo0, hi0), (lo1, hi1) in zip(spans, spans[1:]):
        assert hi0 == lo1
    assert spans[-1][1] == comp.size
