"""Pins for the oracle: checks against things other than the oracle itself.

Each test ties one step of the oracle to the pages, to a hand-worked value
(tests/golden), to a closed form or to brute force, so that a plausible slip
(a dropped term, a wrong sign, index or shift) fails at least one of them.
"""
import math
from fractions import Fraction
from itertools import product

import numpy as np
import pytest

import oracle
import synth
from tests import _golden

M = 4096


# ---------------------------------------------------------------------------
# R1: plane split / merge, against IEEE float semantics (numpy's own decoding)

def _bf16_as_f32(bits16):
    return (bits16.astype(np.uint32) << np.uint32(16)).view(np.float32)


def test_bf16_all_patterns_roundtrip():
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    e, r = oracle.split(x)
    assert np.array_equal(oracle.merge(oracle.BF16, e, r), x)


def test_bf16_fields_match_ieee_value():
    """Exponent byte, sign and fraction of every bf16 pattern, read back from
    the float value: |v| = (1 + m/128) * 2^(e-127) for normals, m * 2^-133
    for subnormals (UCCL-Zip Fig. 2: split into exponent field vs sign and
    fraction)."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    e, r = oracle.split(x)
    v = _bf16_as_f32(x).astype(np.float64)
    sign = (r >> 7).astype(bool)
    frac = (r & 0x7F).astype(np.float64)
    assert np.array_equal(sign, np.signbit(v))
    finite = np.isfinite(v)
    assert np.all(e[~finite] == 255)
    a = np.abs(v[finite])
    ef, ff = e[finite].astype(np.int64), frac[finite]
    normal = a >= 2.0 ** -126
    mant, ex = np.frexp(a[normal])  # a = mant * 2^ex, mant in [0.5, 1)
    assert np.array_equal(ef[normal], ex + 126)
    assert np.array_equal(ff[normal], (a[normal] / np.ldexp(1.0, ef[normal] - 127) - 1.0) * 128.0)
    assert np.all(ef[~normal] == 0)
    assert np.array_equal(ff[~normal], a[~normal] / 2.0 ** -133)
    nan = np.isnan(v)
    assert np.all((r[nan] & 0x7F) != 0)  # a NaN keeps a nonzero payload


def test_fp32_fields_and_roundtrip():
    rng = np.random.default_rng(1)
    mants = [0, 1, 0x3FFFFF, 0x400000, 0x7FFFFF] + list(rng.integers(1, 1 << 23, 3))
    pats = [(s << 31) | (ex << 23) | m for s in (0, 1) for ex in range(256) for m in mants]
    x = np.array(pats, np.uint32)
    e, r = oracle.split(x)
    assert np.array_equal(oracle.merge(oracle.FP32, e, r), x)
    rem = r.reshape(-1, 3).astype(np.uint32)
    rem24 = rem[:, 0] | (rem[:, 1] << 8) | (rem[:, 2] << 16)
    v = x.view(np.float32).astype(np.float64)
    assert np.array_equal((rem24 >> 23).astype(bool), np.signbit(v))
    fin = np.isfinite(v)
    a = np.abs(v[fin])
    normal = a >= 2.0 ** -126
    _, ex = np.frexp(a[normal])
    assert np.array_equal(e[fin][normal].astype(np.int64), ex + 126)
    m = (rem24[fin][normal] & 0x7FFFFF).astype(np.float64)
    assert np.array_equal(m, (a[normal] / np.ldexp(1.0, e[fin][normal].astype(np.int64) - 127) - 1.0) * 2.0 ** 23)
    assert np.all(e[~fin] == 255)
    nan = np.isnan(v)
    assert np.array_equal(rem24[nan] & 0x7FFFFF, x[nan] & 0x7FFFFF)  # NaN payloads kept bit for bit


# ---------------------------------------------------------------------------
# R5: normalisation

def _counts_from(text, n):
    toks = text.split()
    first = [t for t in toks if t.startswith("first201others:")]
    vals, rest = _golden.sym_map(" ".join(t for t in toks if t not in first))
    c = np.zeros(256, np.uint32)
    if rest is not None:
        c[:] = rest
    if first:
        others = [s for s in range(256) if s not in vals][:201]
        c[others] = int(first[0].split(":")[1])
    for s, v in vals.items():
        c[s] = v
    assert c.sum() == n
    return c


@pytest.mark.parametrize("case", ["a", "b", "c", "d"])
def test_normalise_hand_worked(case):
    g = _golden.load("normalise_cases.txt")
    n = int(g[f"{case}.n"])
    counts = _counts_from(g[f"{case}.counts"], n)
    want = _counts_from(g[f"{case}.freq"], M) if case != "c" else None
    f = oracle.normalise(counts, n)
    if want is None:
        vals, rest = _golden.sym_map(g["c.freq"])
        want = np.full(256, rest, np.uint16)
        for s, v in vals.items():
            want[s] = v
    assert np.array_equal(f, want)
    cum = np.concatenate([[0], np.cumsum(f)[:-1]])
    if case == "b":
        assert list(cum[:3]) == [0, 2458, 3277]


def test_normalise_identity_when_n_equals_m():
    """A histogram over exactly 4096 symbols is already normalised."""
    rng = np.random.default_rng(2)
    for _ in range(200):
        k = rng.integers(1, 40)
        syms = rng.choice(256, k, replace=False)
        c = np.zeros(256, np.uint32)
        np.add.at(c, rng.choice(syms, M), 1)
        assert np.array_equal(oracle.normalise(c, M), c.astype(np.uint16))


def test_normalise_exact_division():
    """N = 65536 with every count a multiple of 16: f = c / 16 exactly."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        parts = rng.multinomial(M, rng.dirichlet(np.ones(rng.integers(1, 30))))
        c = np.zeros(256, np.uint32)
        c[rng.choice(256, parts.size, replace=False)] = parts * 16
        assert np.array_equal(oracle.normalise(c, 65536), (c // 16).astype(np.uint16))


def _check_apportionment(c, n, f):
    c = c.astype(np.int64)
    f = f.astype(np.int64)
    present = c > 0
    assert f.sum() == M
    assert np.array_equal(f > 0, present)
    q_floor = c * M // n
    rem = c * M % n
    boosted = present & (q_floor == 0)
    base = np.where(boosted, 1, q_floor)
    s0 = base.sum()
    if s0 <= M:
        # quota property: every non-boosted symbol gets floor or floor+1
        up = f - base
        assert np.all((up == 0) | (up == 1))
        assert np.all(up[boosted] == 0)
        got = np.flatnonzero(present & ~boosted & (up == 1))
        not_got = np.flatnonzero(present & ~boosted & (up == 0))
        for s in got:  # every winner precedes every loser in (remainder desc, symbol asc)
            for t in not_got:
                assert rem[s] > rem[t] or (rem[s] == rem[t] and s < t)
    else:
        # only decrements, each taken from the current maximum (ties: smallest s)
        assert np.all(f <= base)
        cut = np.flatnonzero(f < base)
        if cut.size:
            lo = f[cut].min()
            assert f.max() <= lo + 1
            # the last cut of a symbol left at lo was taken while it was the
            # maximum, so every symbol still at lo + 1 has a larger index
            for s in cut[f[cut] == lo]:
                assert np.all(np.flatnonzero(f == lo + 1) > s)


def _exact_rule(counts, n):
    """R5 restated with exact fractions and a sort, for tiny cases."""
    q = {s: Fraction(int(c) * M, n) for s, c in enumerate(counts) if c}
    f = {s: max(1, math.floor(v)) for s, v in q.items()}
    boosted = {s for s, v in q.items() if math.floor(v) == 0}
    tot = sum(f.values())
    if tot < M:
        order = sorted((s for s in q if s not in boosted), key=lambda s: (-(q[s] - math.floor(q[s])), s))
        for s in order[: M - tot]:
            f[s] += 1
    while sum(f.values()) > M:
        s = min(f, key=lambda s: (-f[s], s))
        f[s] -= 1
    out = np.zeros(256, np.int64)
    for s, v in f.items():
        out[s] = v
    return out


def test_normalise_brute_force_small():
    """All count vectors over 3 symbols (ids 0, 5, 200) with N <= 12."""
    ids = [0, 5, 200]
    for n in range(1, 13):
        for a, b in product(range(n + 1), repeat=2):
            cc = n - a - b
            if cc < 0:
                continue
            c = np.zeros(256, np.uint32)
            c[ids[0]], c[ids[1]], c[ids[2]] = a, b, cc
            f = oracle.normalise(c, n)
            _check_apportionment(c, n, f)
            assert np.array_equal(f.astype(np.int64), _exact_rule(c, n))


def test_normalise_random_invariants():
    rng = np.random.default_rng(4)
    for trial in range(300):
        n = int(rng.integers(1, 65537))
        k = int(rng.integers(1, 257))
        probs = rng.dirichlet(np.full(k, rng.choice([0.05, 0.5, 5.0])))
        c = np.zeros(256, np.uint32)
        c[rng.choice(256, k, replace=False)] = rng.multinomial(n, probs)
        f = oracle.normalise(c, n)
        _check_apportionment(c, n, f)
        if trial < 40:
            assert np.array_equal(f.astype(np.int64), _exact_rule(c, n))


# ---------------------------------------------------------------------------
# R6/R7: rANS steps worked by hand, and round trips

def _freq_from(text):
    vals, _ = _golden.sym_map(text)
    f = np.zeros(256, np.uint16)
    for s, v in vals.items():
        f[s] = v
    return f


def _states_from(text):
    toks = text.split()
    rest = None
    vals = []
    for t in toks:
        if t.startswith("rest:"):
            rest = int(t[5:])
        else:
            vals.append(int(t))
    return np.array(vals + [rest] * (32 - len(vals)), np.uint32)


@pytest.mark.parametrize("case", ["w1", "w2"])
def test_rans_hand_worked(case):
    g = _golden.load("rans_cases.txt")
    syms = _golden.int_list(g[f"{case}.syms"])
    f = _freq_from(g[f"{case}.freq"])
    states, words = oracle.rans_encode(syms, f)
    assert np.array_equal(states, _states_from(g[f"{case}.states"]))
    assert list(words) == _golden.int_list(g[f"{case}.words"])
    assert list(oracle.rans_decode(states, words, f, len(syms))) == syms


def test_rans_hand_worked_with_renormalisation():
    g = _golden.load("rans_cases.txt")
    f = _freq_from(g["w3.freq"])
    syms = np.ones(65, np.uint8)
    syms[0] = syms[32] = 0
    states, words = oracle.rans_encode(syms, f)
    assert np.array_equal(states, _states_from(g["w3.states"]))
    assert list(words) == _golden.int_list(g["w3.words"])
    assert np.array_equal(oracle.rans_decode(states, words, f, 65), syms)


def test_rans_word_order_is_decoder_order():
    """Two lanes renormalise in the same step and one in an earlier step: the
    stream must list step 0's words first, lanes ascending (R7)."""
    f = np.zeros(256, np.uint16)
    f[0], f[1] = 1, 4095
    # lanes 0 and 1 each get A, A, B on steps 0, 1, 2; lane 2 gets A at step 1
    # and 2 only (B at step 0) so it renormalises at step 1.
    syms = np.ones(96, np.uint8)
    for lane in (0, 1):
        syms[lane] = syms[32 + lane] = 0
    syms[32 + 2] = syms[64 + 2] = 0
    states, words = oracle.rans_encode(syms, f)
    # lane 0/1: B then A then A from 65536 -> one word 0x1000 at step 0 (see W3)
    # lane 2: A (step 2) from 65536: 65536*4096 = 268435456; A (step 1):
    #   268435456 >= 2^20 -> emit 0x0000, x = 4096 -> 16777216; B (step 0):
    #   16777216 = 4097*4095 + 1 -> 4097*4096 + 1 + 1 = 16781314
    assert list(words) == [0x1000, 0x1000, 0x0000]
    assert states[0] == states[1] == 16781312 and states[2] == 16781314
    assert np.array_equal(oracle.rans_decode(states, words, f, 96), syms)


def test_chunk_roundtrip_brute_force_tiny():
    """Every sequence of length 1..4 over a 3-symbol alphabet, coded form forced."""
    for n in range(1, 5):
        for seq in product([7, 130, 255], repeat=n):
            stream, raw = oracle.encode_chunk(np.array(seq, np.uint8), force_coded=True)
            assert not raw
            assert list(oracle.decode_chunk(stream, False, n)) == list(seq)


def _ideal_bits(exps, f):
    c = np.bincount(exps, minlength=256)
    nz = c > 0
    return float(np.sum(c[nz] * np.log2(M / f[nz].astype(np.float64))))


@pytest.mark.parametrize("src", ["c1", "c4", "uniform"])
def test_coded_size_tracks_information_content(src):
    """rANS is near-optimal: the words plus the information left in the final
    states equal sum c_s*log2(M/f_s) to within a small fraction."""
    if src == "c1":
        x = synth.c1(n=1 << 18)
    elif src == "c4":
        x = synth.c4(n=1 << 18)
    else:
        x = synth.uniform_pm1_bf16(1 << 18)
    e, _ = oracle.split(x)
    for c in range(4):
        ch = e[c * 65536:(c + 1) * 65536]
        f = oracle.normalise(oracle.histogram(ch))
        states, words = oracle.rans_encode(ch, f)
        used = 16.0 * words.size + float(np.sum(np.log2(states.astype(np.float64)) - 16.0))
        ideal = _ideal_bits(ch, f)
        assert abs(used - ideal) <= 1e-3 * ideal + 64, (used, ideal)


def test_coded_size_within_one_percent_of_entropy():
    """Format check from the spec: coded bytes <= 1.01 * H * N / 8 plus table
    and state overhead, H the Shannon entropy of the chunk histogram."""
    for x in (synth.c1(n=1 << 18), synth.c4(n=1 << 18), synth.c2_tensor(0, rows=64)):
        e, _ = oracle.split(x)
        for c in range(e.size // 65536):
            ch = e[c * 65536:(c + 1) * 65536]
            stream, raw = oracle.encode_chunk(ch)
            assert not raw
            p = np.bincount(ch, minlength=256) / ch.size
            h = -np.sum(p[p > 0] * np.log2(p[p > 0]))
            k = int(np.count_nonzero(p))
            assert len(stream) <= 1.01 * h * ch.size / 8 + 160 + 2 * k + 2


# ---------------------------------------------------------------------------
# R8/R9: chunk streams and the RAW fallback

def test_random_bytes_chunk_is_raw():
    rng = np.random.default_rng(5)
    ch = rng.integers(0, 256, 65536).astype(np.uint8)
    stream, raw = oracle.encode_chunk(ch)
    assert raw and len(stream) == 65536 and np.array_equal(stream, ch)


def test_constant_chunk_is_162_bytes():
    ch = np.full(65536, 121, np.uint8)
    stream, raw = oracle.encode_chunk(ch)
    assert not raw and len(stream) == 162
    st = stream[:128].view(np.uint32)
    assert np.all(st == 65536)
    bitmap = stream[128:160]
    assert bitmap[121 >> 3] == 1 << (121 & 7) and bitmap.sum() == bitmap[121 >> 3]
    assert stream[160:162].view(np.uint16)[0] == 4096


def test_short_chunks_stay_raw():
    for n in (1, 31, 33, 159):
        stream, raw = oracle.encode_chunk(np.full(n, 120, np.uint8))
        assert raw and len(stream) == n


# ---------------------------------------------------------------------------
# R3/R10/R11: container layout and whole-tensor round trips

def _u64(b, o):
    return int(np.frombuffer(b[o:o + 8].tobytes(), np.uint64)[0])


def _u32(b, o):
    return int(np.frombuffer(b[o:o + 4].tobytes(), np.uint32)[0])


def _layout_checks(comp, dtype, n):
    rb = 1 if dtype == oracle.BF16 else 3
    C = -(-n // 65536)
    assert comp[:4].tobytes() == b"UZP1"
    assert int(comp[4]) | int(comp[5]) << 8 == 1
    assert comp[6] == dtype and comp[7] == 0
    assert _u64(comp, 8) == n and _u32(comp, 16) == 65536 and _u32(comp, 20) == C
    rem_off = -(-(64 + 12 * C) // 16) * 16
    exp_off = -(-(rem_off + n * rb) // 16) * 16
    assert _u64(comp, 24) == rem_off and _u64(comp, 32) == exp_off
    assert _u64(comp, 40) == comp.size
    assert np.all(comp[48:64] == 0)
    assert np.all(comp[64 + 12 * C:rem_off] == 0)
    assert np.all(comp[rem_off + n * rb:exp_off] == 0)
    off = 0
    for c in range(C):
        o = _u64(comp, 64 + 8 * c)
        lw = _u32(comp, 64 + 8 * C + 4 * c)
        ln = lw & 0x7FFFFFFF
        assert o == off and o % 16 == 0
        n_c = min(65536, n - 65536 * c)
        if lw >> 31:
            assert ln == n_c
        else:
            assert ln < n_c
        pad = -(-ln // 16) * 16
        assert np.all(comp[exp_off + o + ln:exp_off + o + pad] == 0)
        off += pad
    assert exp_off + off == comp.size


@pytest.mark.parametrize("n", [0, 1, 31, 32, 33, 1000, 65535, 65536, 65537, 100003, 131073])
@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP32])
def test_container_roundtrip_and_layout(n, dtype):
    if dtype == oracle.BF16:
        x = synth.normal_bf16(n, 0.02, 7, n % 97)
    else:
        x = synth.c3(n=n, specials=min(8, n)) if n else np.zeros(0, np.uint32)
    comp = oracle.compress(x)
    _layout_checks(comp, dtype, n)
    assert np.array_equal(oracle.decompress(comp, dtype, n), x)


def test_empty_tensor_is_header_only():
    comp = oracle.compress(np.zeros(0, np.uint16))
    assert comp.size == 64


def test_special_values_roundtrip():
    x = synth.c3(n=200000, specials=4096)
    v = x.view(np.float32)
    assert np.isnan(v).sum() > 0 and np.isinf(v).sum() > 0
    assert (x == 0x80000000).sum() > 0 and ((x & 0x7F800000) == 0).sum() > 0
    comp = oracle.compress(x)
    assert np.array_equal(oracle.decompress(comp, oracle.FP32, x.size), x)
    b = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC1, 0xFF81, 0x0001, 0x807F] * 5000, np.uint16)
    assert np.array_equal(oracle.decompress(oracle.compress(b), oracle.BF16, b.size), b)


def test_uniform_ratio_closed_form():
    """UCCL-Zip Fig. 8 text: a 64% ratio on bf16 uniform in [-1, 1].  For
    |x| ~ U[0,1) the exponent is geometric, P(127-1-k) = 2^-(k+1), entropy
    2 bits, so (8 + 2) / 16 = 0.625 before tables and states."""
    x = synth.uniform_pm1_bf16(1 << 22)
    ratio = oracle.compress(x).size / (2 * x.size)
    overhead = (160 + 2 * 20) / 65536 / 2
    assert 0.625 <= ratio <= 0.625 + overhead + 0.003
    assert abs(ratio - 0.64) < 0.02


def test_normal_ratio_closed_form():
    """N(0, s): P(exponent byte e) = 2[Phi(2^(e-126)/s) - Phi(2^(e-127)/s)];
    the container ratio is (8 + H)/16 plus table overhead."""
    s = 0.02

    def phi(z):
        return 0.5 * (1.0 + math.erf(z / math.sqrt(2.0)))

    p = [2 * (phi(2.0 ** (e - 126) / s) - phi(2.0 ** (e - 127) / s)) for e in range(1, 255)]
    h = -sum(q * math.log2(q) for q in p if q > 0)
    want = (8 + h) / 16
    x = synth.c1()
    got = oracle.compress(x).size / (2 * x.size)
    assert abs(got - want) < 0.004, (got, want, h)


# ---------------------------------------------------------------------------
# R12: receiver validation (host-made corruptions)

def _bf16_case():
    x = synth.normal_bf16(3 * 65536 + 777, 0.02, 8, 1)
    return x, oracle.compress(x)


def _corruptions(comp, n, dtype):
    C = -(-n // 65536)
    cases = {}

    def mod(name, fn):
        b = comp.copy()
        fn(b)
        cases[name] = (b, b.size)

    mod("magic", lambda b: b.__setitem__(0, ord("X")))
    mod("version", lambda b: b.__setitem__(4, 2))
    mod("flags", lambda b: b.__setitem__(7, 1))
    mod("n", lambda b: b.__setitem__(8, b[8] ^ 1))
    mod("chunk_elems", lambda b: b.__setitem__(18, 2))
    mod("num_chunks", lambda b: b.__setitem__(20, b[20] + 1))
    mod("rem_offset", lambda b: b.__setitem__(24, b[24] + 16))
    mod("exp_offset", lambda b: b.__setitem__(32, b[32] + 16))
    mod("total_big", lambda b: b[40:48].view(np.uint64).__setitem__(0, b.size + 16))
    mod("offset_misaligned", lambda b: b[64:72].view(np.uint64).__setitem__(0, 8))
    mod("offset_far", lambda b: b[72:80].view(np.uint64).__setitem__(0, 1 << 40))
    mod("length_far", lambda b: b[64 + 8 * C:68 + 8 * C].view(np.uint32).__setitem__(0, 0x7FFFFFF0))
    exp_off = _u64(comp, 32)
    mod("state", lambda b: b.__setitem__(exp_off + 5, b[exp_off + 5] ^ 0x10))
    mod("state_low", lambda b: b[exp_off:exp_off + 4].view(np.uint32).__setitem__(0, 5))
    mod("freq_sum", lambda b: b.__setitem__(exp_off + 160, b[exp_off + 160] ^ 1))
    ln0 = _u32(comp, 64 + 8 * C) & 0x7FFFFFFF
    mod("word", lambda b: b.__setitem__(exp_off + ln0 - 2, b[exp_off + ln0 - 2] ^ 0x5A))
    mod("len_minus_2", lambda b: b[64 + 8 * C:68 + 8 * C].view(np.uint32).__setitem__(0, ln0 - 2))
    mod("len_plus_2", lambda b: b[64 + 8 * C:68 + 8 * C].view(np.uint32).__setitem__(0, ln0 + 2))
    mod("raw_flag", lambda b: b[64 + 8 * C:68 + 8 * C].view(np.uint32).__setitem__(0, ln0 | 0x80000000))
    cases["truncated"] = (comp[:-16].copy(), comp.size - 16)
    cases["short_header"] = (comp[:40].copy(), 40)
    return cases


def test_decoder_rejects_corruptions():
    x, comp = _bf16_case()
    for name, (b, size) in _corruptions(comp, x.size, oracle.BF16).items():
        st, _ = oracle.decompress_status(b[:size], oracle.BF16, x.size)
        assert st == oracle.ERR_CORRUPT, name


def test_decoder_checks_arguments_against_header():
    x, comp = _bf16_case()
    assert oracle.decompress_status(comp, oracle.FP32, x.size)[0] == oracle.ERR_CORRUPT
    assert oracle.decompress_status(comp, oracle.BF16, x.size + 1)[0] == oracle.ERR_CORRUPT
    assert oracle.decompress_status(comp, 7, x.size)[0] == oracle.ERR_UNSUPPORTED_DTYPE
