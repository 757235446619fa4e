"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer.

The oracle's C code is compiled with -fsanitize=address,undefined (any
report aborts) into tests/oracle_san_driver.c, which round-trips every
element format at the edge sizes and in every table and whole-message mode,
and decodes seeded random corruptions of containers; every buffer it hands
the oracle has exactly the size the call may touch.
"""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle
import synth
from tests import _fuzz

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
EDGE = [0, 1, 31, 33, 65535, 65537, 100003]


def _build(tmp):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    exe = os.path.join(tmp, "orc_san")
    cmd = ["gcc", "-O1", "-g", "-std=c99", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
           "-fno-omit-frame-pointer", "-o", exe, os.path.join(ROOT, "oracle", "uzip_oracle.c"),
           os.path.join(HERE, "oracle_san_driver.c"), "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if "sanitize" in r.stderr or "asan" in r.stderr.lower():
            pytest.skip("the compiler has no sanitizer runtime")
        raise AssertionError(r.stderr)
    return exe


def _case(path, kind, dtype, mode, n, payload, sigma=0.0):
    with open(path, "wb") as fh:
        fh.write(bytes([ord(kind), dtype, mode, 0, 0, 0, 0, 0]) + struct.pack("<Qd", n, sigma))
        fh.write(np.ascontiguousarray(payload).view(np.uint8).tobytes())


def _values(dtype, n, t):
    if dtype == 0:
        return synth.normal_bf16(n, 0.02, 14, t)
    if dtype == 1:
        return synth.normal_fp32(n, 0.02, tensor=t)
    if dtype == 2:
        return synth.normal_fp16(n, 0.02, tensor=t).view(np.uint16)
    return synth.normal_fp8(n, "e4m3" if dtype == 3 else "e5m2", 0.02, tensor=t)


def test_oracle_is_clean_under_sanitizers(tmp_path):
    exe = _build(str(tmp_path))
    files = []

    def add(kind, dtype, mode, n, payload, sigma=0.0):
        p = str(tmp_path / f"case{len(files):04d}.bin")
        _case(p, kind, dtype, mode, n, payload, sigma)
        files.append(p)

    rng = np.random.default_rng(7)
    for dtype in range(5):
        for i, n in enumerate(EDGE):
            add("C", dtype, 0, n, _values(dtype, n, i))
        n = 2 * 65536 + 77
        v = _values(dtype, n, 20)
        for mode in (1, 2, 3):
            add("C", dtype, mode, n, v)
        add("C", dtype, 4, n, v, 0.02)
        # random bit patterns: chunks stored RAW
        rnd = rng.integers(0, 256, n * v.itemsize, dtype=np.uint8).view(v.dtype)
        add("C", dtype, 0, n, rnd)
    # streams that outgrow eight bits a value for a while
    add("C", 0, 0, synth.growth_bf16().size, synth.growth_bf16())
    add("C", 1, 0, synth.growth_fp32().size, synth.growth_fp32())
    # damaged containers of every format
    for case in range(5):
        bits, dtype = _fuzz.fuzz_input(case)
        comp = oracle.compress(bits, dtype)
        for _, b, _ in _fuzz.corruptions(comp, dtype, bits.size, 40, seed=300 + case):
            add("D", dtype, 0, bits.size, b)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    r = subprocess.run([exe] + files, capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert f"{len(files)} cases, 0 failed" in r.stdout
