"""Python access to the uzip oracle (plain single-threaded C).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The library itself
never calls it: the GPU path has no CPU fallback.

The oracle follows the pages step by step (UCCL-Zip Fig. 2 and Fig. 5
captions for the exponent-plane split and the local tables; NCCLZ Sec. IV-B,
IV-C and Alg. 1/2 for the self-describing frame and the RAW fallback), with
the format readings R1..R20 where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, "uzip_oracle.c")]

BF16, FP32, FP16, FP8_E4M3, FP8_E5M2 = 0, 1, 2, 3, 4
ELEM_BYTES = {BF16: 2, FP32: 4, FP16: 2, FP8_E4M3: 1, FP8_E5M2: 1}
BITS_DTYPE = {BF16: np.uint16, FP32: np.uint32, FP16: np.uint16, FP8_E4M3: np.uint8, FP8_E5M2: np.uint8}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_DTYPE, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 2, 3, 4
CHUNK = 65536
M = 4096


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (plain gcc, -O2, no -march)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stale = force or not os.path.exists(LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(LIB_PATH) for s in SOURCES + [os.path.join(HERE, "uzip_oracle.h")]
    )
    if stale:
        tmp = LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-shared", "-fPIC", "-o", tmp] + SOURCES
                              + ["-lm"])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        vp = ctypes.c_void_p
        L.orc_split.argtypes = [ctypes.c_int, vp, ctypes.c_uint64, vp, vp]
        L.orc_merge.argtypes = [ctypes.c_int, vp, vp, ctypes.c_uint64, vp]
        L.orc_histogram.argtypes = [vp, ctypes.c_uint32, vp]
        L.orc_histogram.restype = None
        L.orc_normalise.argtypes = [vp, ctypes.c_uint32, vp]
        L.orc_rans_encode.argtypes = [vp, ctypes.c_uint32, vp, vp, vp, u32p]
        L.orc_rans_decode.argtypes = [vp, vp, ctypes.c_uint32, vp, ctypes.c_uint32, vp]
        L.orc_encode_chunk.argtypes = [vp, ctypes.c_uint32, ctypes.c_int, vp, u32p, ctypes.POINTER(ctypes.c_int)]
        L.orc_decode_chunk.argtypes = [vp, ctypes.c_uint32, ctypes.c_int, ctypes.c_uint32, vp]
        L.orc_container_bound.argtypes = [ctypes.c_int, ctypes.c_uint64]
        L.orc_container_bound.restype = ctypes.c_uint64
        L.orc_remainder_plane_bytes.argtypes = [ctypes.c_int, ctypes.c_uint64]
        L.orc_remainder_plane_bytes.restype = ctypes.c_uint64
        L.orc_compress_mode.argtypes = [ctypes.c_int, vp, ctypes.c_uint64, vp, ctypes.c_uint64, u64p, ctypes.c_int]
        L.orc_compress_mode.restype = ctypes.c_int
        L.orc_gate_sample_elems.argtypes = [ctypes.c_int, ctypes.c_uint64]
        L.orc_gate_sample_elems.restype = ctypes.c_uint64
        L.orc_gate_says_raw.argtypes = [vp, ctypes.c_uint32]
        L.orc_gate_says_raw.restype = ctypes.c_int
        L.orc_sampled_counts.argtypes = [vp, ctypes.c_uint32, ctypes.c_int, vp]
        L.orc_sampled_counts.restype = ctypes.c_uint32
        L.orc_parametric_counts.argtypes = [ctypes.c_int, ctypes.c_double, vp]
        L.orc_parametric_counts.restype = ctypes.c_uint32
        L.orc_compress_parametric.argtypes = [ctypes.c_int, vp, ctypes.c_uint64, vp, ctypes.c_uint64, u64p,
                                              ctypes.c_double]
        L.orc_compress_parametric.restype = ctypes.c_int
        L.orc_compress.argtypes = [ctypes.c_int, vp, ctypes.c_uint64, vp, ctypes.c_uint64, u64p]
        L.orc_decompress.argtypes = [vp, ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64, vp]
        for name in ("orc_split", "orc_merge", "orc_normalise", "orc_rans_encode", "orc_rans_decode",
                     "orc_encode_chunk", "orc_decode_chunk", "orc_compress", "orc_decompress"):
            getattr(L, name).restype = ctypes.c_int
        del u8p, u16p, u64p
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: oracle status {status}")
        self.status = status


def _check(st: int, what: str):
    if st != OK:
        raise OracleError(st, what)


def dtype_code(a: np.ndarray) -> int:
    """Container dtype implied by a numpy array: bf16 travels as uint16 bit
    patterns, fp16 as float16, fp32 as uint32 or float32.  The fp8 formats
    have no numpy type: pass dtype= explicitly with uint8 bit patterns."""
    if a.dtype in (np.uint16, np.int16):
        return BF16
    if a.dtype == np.float16:
        return FP16
    if a.dtype in (np.uint32, np.float32, np.int32):
        return FP32
    raise TypeError(f"no container dtype for numpy {a.dtype}")


def _bits(a: np.ndarray, dtype: int | None):
    d = dtype_code(a) if dtype is None else dtype
    a = np.ascontiguousarray(a).reshape(-1)
    if a.dtype.itemsize != ELEM_BYTES[d]:
        raise TypeError(f"{a.dtype} elements do not match dtype {d}")
    return d, a.view(BITS_DTYPE[d])


def remainder_plane_bytes(dtype: int, n: int) -> int:
    return int(lib().orc_remainder_plane_bytes(dtype, n))


def split(bits: np.ndarray, dtype: int | None = None):
    d, bits = _bits(bits, dtype)
    n = bits.size
    exps = np.empty(n, np.uint8)
    rem = np.empty(max(1, remainder_plane_bytes(d, n)), np.uint8)
    _check(lib().orc_split(d, _ptr(bits if n else np.zeros(1, bits.dtype)), n, _ptr(exps if n else np.zeros(1, np.uint8)),
                           _ptr(rem)), "split")
    return exps, rem[: remainder_plane_bytes(d, n)]


def merge(dtype: int, exps: np.ndarray, rem: np.ndarray) -> np.ndarray:
    n = exps.size
    out = np.empty(n, BITS_DTYPE[dtype])
    _check(lib().orc_merge(dtype, _ptr(np.ascontiguousarray(exps)), _ptr(np.ascontiguousarray(rem)), n, _ptr(out)), "merge")
    return out


def histogram(exps: np.ndarray) -> np.ndarray:
    exps = np.ascontiguousarray(exps, np.uint8)
    counts = np.zeros(256, np.uint32)
    lib().orc_histogram(_ptr(exps), exps.size, _ptr(counts))
    return counts


def normalise(counts, n_c: int | None = None) -> np.ndarray:
    counts = np.ascontiguousarray(np.asarray(counts, np.uint32))
    assert counts.size == 256
    if n_c is None:
        n_c = int(counts.sum())
    freq = np.zeros(256, np.uint16)
    _check(lib().orc_normalise(_ptr(counts), n_c, _ptr(freq)), "normalise")
    return freq


def rans_encode(syms, freq):
    syms = np.ascontiguousarray(np.asarray(syms, np.uint8))
    freq = np.ascontiguousarray(np.asarray(freq, np.uint16))
    states = np.zeros(32, np.uint32)
    words = np.zeros(max(1, syms.size), np.uint16)
    nw = ctypes.c_uint32(0)
    _check(lib().orc_rans_encode(_ptr(syms), syms.size, _ptr(freq), _ptr(states), _ptr(words), ctypes.byref(nw)), "rans_encode")
    return states, words[: nw.value].copy()


def rans_decode(states, words, freq, n_c: int):
    states = np.ascontiguousarray(np.asarray(states, np.uint32))
    words = np.ascontiguousarray(np.asarray(words, np.uint16))
    freq = np.ascontiguousarray(np.asarray(freq, np.uint16))
    syms = np.zeros(max(1, n_c), np.uint8)
    st = lib().orc_rans_decode(_ptr(states), _ptr(words if words.size else np.zeros(1, np.uint16)), words.size,
                               _ptr(freq), n_c, _ptr(syms))
    _check(st, "rans_decode")
    return syms[:n_c]


def encode_chunk(exps, force_coded: bool = False):
    exps = np.ascontiguousarray(np.asarray(exps, np.uint8))
    out = np.zeros(max(exps.size, 672 + 2 * exps.size), np.uint8)
    ln = ctypes.c_uint32(0)
    raw = ctypes.c_int(0)
    _check(lib().orc_encode_chunk(_ptr(exps), exps.size, int(force_coded), _ptr(out), ctypes.byref(ln), ctypes.byref(raw)),
           "encode_chunk")
    return out[: ln.value].copy(), bool(raw.value)


def decode_chunk(stream, raw: bool, n_c: int) -> np.ndarray:
    stream = np.ascontiguousarray(np.asarray(stream, np.uint8))
    exps = np.zeros(max(1, n_c), np.uint8)
    buf = stream if stream.size else np.zeros(1, np.uint8)
    _check(lib().orc_decode_chunk(_ptr(buf), stream.size, int(raw), n_c, _ptr(exps)), "decode_chunk")
    return exps[:n_c]


def container_bound(dtype: int, n: int) -> int:
    return int(lib().orc_container_bound(dtype, n))


MODE_CHUNK, MODE_RAW, MODE_GATE, MODE_SAMPLED, MODE_PARAMETRIC = 0, 1, 2, 3, 4


def compress(bits: np.ndarray, dtype: int | None = None, mode: int = MODE_CHUNK,
             sigma: float | None = None) -> np.ndarray:
    """Container bytes for an array of element bit patterns (see dtype_code;
    fp8 needs dtype=FP8_E4M3 or FP8_E5M2 with uint8 bits).  mode: per-chunk
    choice, whole-message RAW, RAW when the gate's sample says so, tables
    built from a sample of each chunk, or (MODE_PARAMETRIC, with sigma) the
    one Gaussian-model table of R25 for every chunk."""
    d, bits = _bits(bits, dtype)
    n = bits.size
    cap = container_bound(d, n)
    out = np.empty(max(cap, 1), np.uint8)
    total = ctypes.c_uint64(0)
    src = bits if n else np.zeros(1, bits.dtype)
    if mode == MODE_PARAMETRIC:
        st = lib().orc_compress_parametric(d, _ptr(src), n, _ptr(out), cap, ctypes.byref(total), float(sigma))
    else:
        st = lib().orc_compress_mode(d, _ptr(src), n, _ptr(out), cap, ctypes.byref(total), mode)
    _check(st, "compress")
    return out[: total.value].copy()


def parametric_counts(dtype: int, sigma: float):
    """R25 model counts for values ~ N(0, sigma^2) and their total (0 for a
    sigma that is not finite and positive)."""
    counts = np.zeros(256, np.uint32)
    total = lib().orc_parametric_counts(dtype, float(sigma), _ptr(counts))
    return counts, int(total)


def gate_says_raw(bits: np.ndarray, dtype: int | None = None) -> bool:
    """The gate's decision for a message: its sample's exponent bytes would be
    stored RAW if coded as one chunk."""
    d, bits = _bits(bits, dtype)
    ns = int(lib().orc_gate_sample_elems(d, bits.size))
    exps, _ = split(bits[:ns], d)
    r = lib().orc_gate_says_raw(_ptr(exps if ns else np.zeros(1, np.uint8)), ns)
    if r < 0:
        raise OracleError(ERR_INVALID_ARG, "gate")
    return bool(r)


def decompress_status(comp: np.ndarray, dtype: int, n: int):
    comp = np.ascontiguousarray(np.asarray(comp, np.uint8))
    out = np.empty(max(1, n), BITS_DTYPE.get(dtype, np.uint32))  # unknown dtype: the oracle refuses it
    buf = comp if comp.size else np.zeros(1, np.uint8)
    st = lib().orc_decompress(_ptr(buf), comp.size, dtype, n, _ptr(out))
    return st, out[:n]


def decompress(comp: np.ndarray, dtype: int, n: int) -> np.ndarray:
    st, out = decompress_status(comp, dtype, n)
    _check(st, "decompress")
    return out


def sampled_counts(exps: np.ndarray, ebits: int):
    """R24 counts of one chunk's exponent bytes and their total."""
    exps = np.ascontiguousarray(np.asarray(exps, np.uint8))
    counts = np.zeros(256, np.uint32)
    total = lib().orc_sampled_counts(_ptr(exps), exps.size, ebits, _ptr(counts))
    return counts, int(total)
