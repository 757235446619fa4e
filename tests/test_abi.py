"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
symbol its headers declare, and its host-only arithmetic is right."""
import os
import random
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(uzip_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def uz():
    import __graft_entry__

    __graft_entry__.build_library()
    import lossless_float_tensor_gb300 as uz

    return uz


def test_exports_every_declared_symbol(uz):
    names = _declared_functions()
    assert {"uzip_max_compressed_size", "uzip_compress", "uzip_decompress", "uzip_query_size"} <= names
    lib = uz.library()
    for name in sorted(names):
        assert hasattr(lib, name), name


def test_max_compressed_size_is_container_bound_plus_work_area(uz):
    for dtype in range(5):  # bf16, fp32, fp16, fp8 e4m3fn, fp8 e5m2
        for n in [0, 1, 15, 16, 17, 65535, 65536, 65537, 3 * 65536 + 5, 5 * 65536, 700 * 65536 - 3, 1 << 29]:
            c = -(-n // 65536)
            bound = oracle.container_bound(dtype, n)
            off = uz.library().uzip_debug_scratch_offset(dtype, n)
            assert off == -(-bound // 16) * 16
            # counters and descriptors, 4 KiB of alignment slack, and two
            # 68 KiB slots for each of the 8 encoders of one block per 4
            # chunks, at most 160 blocks
            work = 16 + 8 * c + 4096 + min(-(-c // 4), 160) * 8 * 2 * 69632
            assert uz.uzip_max_compressed_size(dtype, n) == off + work
    assert uz.uzip_max_compressed_size(7, 10) == 0
    assert uz.uzip_max_compressed_size(0, (1 << 40) + 1) == 0


def test_division_magic_exact_for_every_frequency(uz):
    """x // f == (x*m + add) >> shift for x in [16f, f*2^20): the worst cases
    x = k f - 1 and x = k f at the top of the range, the bottom, and random x."""
    import ctypes

    lib = uz.library()
    m, add, sh = ctypes.c_uint32(), ctypes.c_uint32(), ctypes.c_uint32()
    rng = random.Random(7)
    for f in range(1, 4097):
        assert lib.uzip_debug_div_magic(f, ctypes.byref(m), ctypes.byref(add), ctypes.byref(sh)) == 1
        M, A, S = m.value, add.value, sh.value
        assert A in (0, M) and 32 <= S <= 44
        top = f << 20
        xs = {16 * f, 16 * f + 1, top - 1, top - f, top - f - 1, top - 2 * f, top - 2 * f + 1}
        xs |= {rng.randrange(16 * f, top) for _ in range(24)}
        for x in xs:
            assert (x * M + A) >> S == x // f, (f, x)
        # closed-form exactness over the whole range
        two_p = 1 << S
        if A == 0:
            assert (top - 1) * (M * f - two_p) < two_p
        else:
            assert (((1 << 20) - 1) * f + 1) * (two_p - M * f) <= two_p
    assert lib.uzip_debug_div_magic(0, None, None, None) == 0
    assert lib.uzip_debug_div_magic(4097, None, None, None) == 0


def test_33_bit_division_magic_exact_for_every_frequency(uz):
    """The warp-specialised encoder divides by f as
    (x * (2^32 + m_lo)) >> (32 + sh) for x in [0, f * 2^20): checked at the
    worst points (x = k f - 1 at the top and bottom of the range), random x,
    and against the closed-form error bound x e < 2^(32 + sh)."""
    import ctypes

    lib = uz.library()
    m, sh = ctypes.c_uint32(), ctypes.c_uint32()
    rng = random.Random(11)
    for f in range(1, 4097):
        assert lib.uzip_debug_div_magic33(f, ctypes.byref(m), ctypes.byref(sh)) == 1
        M, S = (1 << 32) + m.value, sh.value
        assert (1 << S) >= f and S <= 12 and (1 << 32) <= M < (1 << 33)
        top = f << 20
        xs = {0, 1, f - 1, f, top - 1, top - f, top - f - 1, top - 2 * f, top - 2 * f + 1, (1 << 16)}
        xs |= {rng.randrange(0, top) for _ in range(24)}
        for x in xs:
            assert (x * M) >> (32 + S) == x // f, (f, x)
            assert x * M < 1 << 64
        assert (top - 1) * (M * f - (1 << (32 + S))) < 1 << (32 + S)
    assert lib.uzip_debug_div_magic33(0, None, None) == 0
    assert lib.uzip_debug_div_magic33(4097, None, None) == 0


def test_status_strings(uz):
    assert uz.uzip_status_string(0) == "ok"
    assert uz.uzip_status_string(4) == "corrupt container"
    assert uz.uzip_status_string(99) == "unknown status"


def test_host_argument_checks(uz):
    """Rejected on the host before any CUDA call."""
    fake = 1 << 40  # aligned, never dereferenced
    assert uz.uzip_compress(fake, 5, 10, fake, 1 << 20, None, 0) == uz.UZIP_ERR_UNSUPPORTED_DTYPE
    assert uz.uzip_compress(None, 0, 10, fake, 1 << 20, None, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_compress(fake + 8, 0, 10, fake, 1 << 20, None, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_compress(fake, 0, 10, None, 1 << 20, None, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_compress(fake, 0, 10, fake, 100, None, 0) == uz.UZIP_ERR_CAPACITY
    assert uz.uzip_compress(fake, 0, (1 << 40) + 1, fake, 1 << 20, None, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_compress_ex(fake, 0, 10, fake, 1 << 20, None, None, 8, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_decompress(fake, 32, fake, 0, 10, None, 0) == uz.UZIP_ERR_CORRUPT
    assert uz.uzip_decompress(None, 1 << 20, fake, 0, 10, None, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_decompress(fake, 1 << 20, fake, 5, 10, None, 0) == uz.UZIP_ERR_UNSUPPORTED_DTYPE
    assert uz.uzip_query_size(None, 0)[0] == uz.UZIP_ERR_INVALID_ARG


def test_package_refuses_to_import_without_the_library(monkeypatch):
    """No CPU fallback: with the shared library absent, importing the binding
    fails loudly instead of degrading."""
    import importlib.util

    path = os.path.join(ROOT, "lossless_float_tensor_gb300", "__init__.py")
    real_exists = os.path.exists
    monkeypatch.setattr(os.path, "exists", lambda p: False if str(p).endswith("libuzip.so") else real_exists(p))
    spec = importlib.util.spec_from_file_location("_uzip_without_library", path)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="not built"):
        spec.loader.exec_module(mod)


def test_binding_constants_match_the_header(uz):
    """The Python binding repeats the header's #define and enum values."""
    text = open(os.path.join(ROOT, "include", "uzip.h")).read()
    defines = {m.group(1): m.group(2) for m in re.finditer(r"#define\s+(UZIP_[A-Z0-9_]+)\s+(.+)", text)}
    for name, expr in defines.items():
        if not hasattr(uz, name):
            continue
        expr = re.sub(r"(\d+)[uUlL]*", r"\1", expr.split("/*")[0]).strip()
        assert re.fullmatch(r"[\d\s()<]+", expr), expr
        value = eval(expr, {"__builtins__": {}})
        assert getattr(uz, name) == value, name
    assert uz.UZIP_PIPE_RAW_BELOW_DEFAULT == 32 << 20
    for name, value in re.findall(r"\b(UZIP_[A-Z0-9_]+)\s*=\s*(\d+)", text):
        if hasattr(uz, name):
            assert getattr(uz, name) == int(value), name


@pytest.mark.parametrize("dtype", [0, 1, 2, 3, 4])
def test_parametric_model_counts_equal_the_oracle(uz, dtype):
    """The library's host code and the oracle compute the Gaussian-model
    counts independently from one definition; they agree to the bit."""
    import ctypes

    import numpy as np

    for sigma in [1e-6, 3e-4, 0.02, 0.1234, 0.7, 1.0, 5.5, 300.0, 2.0 ** 40]:
        got = (ctypes.c_uint32 * 256)()
        assert uz.library().uzip_debug_model_counts(dtype, sigma, got) == 1
        want, _ = oracle.parametric_counts(dtype, sigma)
        assert np.array_equal(np.frombuffer(got, np.uint32), want), sigma
    for bad in [0.0, -0.5, float("inf"), float("nan")]:
        assert uz.library().uzip_debug_model_counts(dtype, bad, (ctypes.c_uint32 * 256)()) == 0


def test_parametric_refuses_bad_sigma_before_any_work(uz):
    fake = 1 << 40  # aligned, never dereferenced
    for bad in [0.0, -1.0, float("inf"), float("nan")]:
        assert uz.uzip_compress_parametric(fake, 0, 10, fake, 1 << 30, None, None, bad, 0) == uz.UZIP_ERR_INVALID_ARG
    assert uz.uzip_compress_parametric(fake, 5, 10, fake, 1 << 30, None, None, 1.0, 0) == uz.UZIP_ERR_UNSUPPORTED_DTYPE
