"""Python binding of libuzip: lossless compression of bf16, fp16, fp32 and fp8
GPU tensors.

Thin ctypes layer over the C ABI in include/uzip.h.  The functions named like
the C entry points (uzip_compress, ...) only marshal arguments: every step of
compression and decompression runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams in the convenience wrappers compress() /
decompress().  There is no CPU fallback: if the library is missing, importing
this package fails.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libuzip.so")

UZIP_BF16, UZIP_FP32, UZIP_FP16, UZIP_FP8_E4M3, UZIP_FP8_E5M2 = 0, 1, 2, 3, 4
UZIP_OK = 0
UZIP_ERR_INVALID_ARG = 1
UZIP_ERR_UNSUPPORTED_DTYPE = 2
UZIP_ERR_CAPACITY = 3
UZIP_ERR_CORRUPT = 4
UZIP_ERR_TIMEOUT = 5
UZIP_ERR_CUDA = 6
UZIP_ERR_TOO_LARGE = 7
UZIP_NOALLOC_MAX_ELEMS = 1 << 30
UZIP_TESTFLAG_SKIP_CHUNK0 = 1
UZIP_FLAG_SAMPLED_TABLES = 2
UZIP_PIPE_EXACT, UZIP_PIPE_BOUND, UZIP_PIPE_SERIAL, UZIP_PIPE_SIZED, UZIP_PIPE_STREAMED = 0, 1, 2, 3, 4
UZIP_PIPE_RAW_BELOW_DEFAULT = 32 << 20
UZIP_MAX_ELEMS = 1 << 40
CHUNK_ELEMS = 65536
HEADER_BYTES = 64

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB_PATH)
_u64, _u32, _i32, _vp, _int = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int

_lib.uzip_max_compressed_size.argtypes = [_int, _u64]
_lib.uzip_max_compressed_size.restype = _u64
_lib.uzip_compress.argtypes = [_vp, _int, _u64, _vp, _u64, _vp, _vp]
_lib.uzip_compress.restype = _int
_lib.uzip_compress_ex.argtypes = [_vp, _int, _u64, _vp, _u64, _vp, _vp, _u32, _vp]
_lib.uzip_compress_ex.restype = _int
_lib.uzip_compress_noalloc.argtypes = [_vp, _int, _u64, _vp, _u64, _vp, _vp, _vp]
_lib.uzip_compress_noalloc.restype = _int
_lib.uzip_compress_parametric.argtypes = [_vp, _int, _u64, _vp, _u64, _vp, _vp, ctypes.c_double, _vp]
_lib.uzip_compress_parametric.restype = _int
_lib.uzip_compress_gated.argtypes = [_vp, _int, _u64, _vp, _u64, _vp, _vp, _u64, _vp]
_lib.uzip_compress_gated.restype = _int
_lib.uzip_decompress.argtypes = [_vp, _u64, _vp, _int, _u64, _vp, _vp]
_lib.uzip_decompress.restype = _int
_lib.uzip_query_size.argtypes = [_vp, ctypes.POINTER(_u64), ctypes.POINTER(_int), ctypes.POINTER(_u64), _vp]
_lib.uzip_query_size.restype = _int
_lib.uzip_status_string.argtypes = [_int]
_lib.uzip_status_string.restype = ctypes.c_char_p
_lib.uzip_pipeline_send.argtypes = [_int, ctypes.POINTER(_vp), ctypes.POINTER(_u64), _u32, ctypes.POINTER(_vp), _u64,
                                    ctypes.POINTER(_vp), _u64, _vp, _int, _vp, _vp]
_lib.uzip_pipeline_send.restype = _int
_lib.uzip_pipeline_send_ex.argtypes = [_int, ctypes.POINTER(_vp), ctypes.POINTER(_u64), _u32, ctypes.POINTER(_vp), _u64,
                                       ctypes.POINTER(_vp), _u32, _u64, _vp, _int, _u64, _vp, _vp]
_lib.uzip_pipeline_send_ex.restype = _int
_lib.uzip_debug_div_magic.argtypes = [_u32, ctypes.POINTER(_u32), ctypes.POINTER(_u32), ctypes.POINTER(_u32)]
_lib.uzip_debug_div_magic.restype = _int
_lib.uzip_debug_model_counts.argtypes = [_int, ctypes.c_double, ctypes.POINTER(_u32)]
_lib.uzip_debug_model_counts.restype = _int
_lib.uzip_debug_scratch_offset.argtypes = [_int, _u64]
_lib.uzip_debug_scratch_offset.restype = _u64


def library():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


# ---- C entry points (same names, same arguments; integers for pointers) ----

def uzip_max_compressed_size(dtype: int, n: int) -> int:
    return int(_lib.uzip_max_compressed_size(dtype, n))


def uzip_compress(d_in: int, dtype: int, n: int, d_out: int, out_capacity: int, d_out_size: int | None,
                  stream: int) -> int:
    return int(_lib.uzip_compress(d_in, dtype, n, d_out, out_capacity, d_out_size, stream))


def uzip_compress_ex(d_in: int, dtype: int, n: int, d_out: int, out_capacity: int, d_out_size: int | None,
                     d_status: int | None, flags: int, stream: int) -> int:
    return int(_lib.uzip_compress_ex(d_in, dtype, n, d_out, out_capacity, d_out_size, d_status, flags, stream))


def uzip_compress_gated(d_in: int, dtype: int, n: int, d_out: int, out_capacity: int, d_out_size: int | None,
                        d_status: int | None, raw_below_bytes: int, stream: int) -> int:
    return int(_lib.uzip_compress_gated(d_in, dtype, n, d_out, out_capacity, d_out_size, d_status, raw_below_bytes,
                                        stream))


def uzip_compress_parametric(d_in: int, dtype: int, n: int, d_out: int, out_capacity: int, d_out_size: int | None,
                             d_status: int | None, sigma: float, stream: int) -> int:
    """Compression with one Gaussian-model table for every chunk (values ~
    N(0, sigma^2)); see include/uzip.h."""
    return int(_lib.uzip_compress_parametric(d_in, dtype, n, d_out, out_capacity, d_out_size, d_status, float(sigma),
                                             stream))


def uzip_compress_noalloc(d_in: int, dtype: int, n: int, d_out: int, out_capacity: int, d_out_size: int | None,
                          d_status: int | None, stream: int) -> int:
    """Compression that allocates nothing: the work area is the library's own
    device array (tensors up to UZIP_NOALLOC_MAX_ELEMS values; calls sharing a
    GPU must not overlap)."""
    return int(_lib.uzip_compress_noalloc(d_in, dtype, n, d_out, out_capacity, d_out_size, d_status, stream))


def uzip_decompress(d_comp: int, comp_capacity: int, d_out: int, dtype: int, n: int, d_status: int | None,
                    stream: int) -> int:
    return int(_lib.uzip_decompress(d_comp, comp_capacity, d_out, dtype, n, d_status, stream))


def uzip_query_size(d_comp: int, stream: int):
    """Returns (status, total_bytes, dtype, n)."""
    t, d, n = _u64(0), _int(0), _u64(0)
    st = int(_lib.uzip_query_size(d_comp, ctypes.byref(t), ctypes.byref(d), ctypes.byref(n), stream))
    return st, int(t.value), int(d.value), int(n.value)


def uzip_status_string(st: int) -> str:
    return _lib.uzip_status_string(st).decode()


def uzip_pipeline_send(dtype: int, d_msgs, msg_elems, d_bank, bank_capacity: int, h_bank, h_capacity: int,
                       h_sizes: int, mode: int, s_compress: int, s_copy: int) -> int:
    k = len(d_msgs)
    msgs = (_vp * k)(*d_msgs)
    elems = (_u64 * k)(*msg_elems)
    db = (_vp * 2)(*d_bank)
    hb = (_vp * 2)(*h_bank)
    return int(_lib.uzip_pipeline_send(dtype, msgs, elems, k, db, bank_capacity, hb, h_capacity, h_sizes, mode,
                                       s_compress, s_copy))


def uzip_pipeline_send_ex(dtype: int, d_msgs, msg_elems, d_bank, bank_capacity: int, h_bank, h_capacity: int,
                          h_sizes: int, mode: int, raw_below_bytes: int, s_compress: int, s_copy: int) -> int:
    k = len(d_msgs)
    msgs = (_vp * k)(*d_msgs)
    elems = (_u64 * k)(*msg_elems)
    db = (_vp * 2)(*d_bank)
    nh = len(h_bank)
    hb = (_vp * nh)(*h_bank)
    return int(_lib.uzip_pipeline_send_ex(dtype, msgs, elems, k, db, bank_capacity, hb, nh, h_capacity, h_sizes, mode,
                                          raw_below_bytes, s_compress, s_copy))


# ---- torch convenience layer (allocation and streams only) ----------------

class UzipError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {uzip_status_string(status)} ({status})")
        self.status = status


def _check(st: int, what: str):
    if st != UZIP_OK:
        raise UzipError(st, what)


def _torch_dtypes():
    """uzip dtype code <-> torch dtype (the fp8 types where torch has them)."""
    import torch

    m = {UZIP_BF16: torch.bfloat16, UZIP_FP32: torch.float32, UZIP_FP16: torch.float16}
    if hasattr(torch, "float8_e4m3fn"):
        m[UZIP_FP8_E4M3] = torch.float8_e4m3fn
    if hasattr(torch, "float8_e5m2"):
        m[UZIP_FP8_E5M2] = torch.float8_e5m2
    return m


def dtype_code(t) -> int:
    for code, tdt in _torch_dtypes().items():
        if t.dtype == tdt:
            return code
    raise UzipError(UZIP_ERR_UNSUPPORTED_DTYPE, f"dtype {t.dtype}")


def _stream(stream):
    import torch

    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def compress(t, stream=None, out=None, out_size=None):
    """Compress a contiguous CUDA bf16, fp16, fp32 or fp8 tensor.

    Returns (buffer, size): buffer is a uint8 CUDA tensor of
    uzip_max_compressed_size bytes whose first `size` bytes (a 0-dim int64
    CUDA tensor, filled on the device) are the container.
    """
    import torch

    if not t.is_cuda or not t.is_contiguous():
        raise UzipError(UZIP_ERR_INVALID_ARG, "compress needs a contiguous CUDA tensor")
    d = dtype_code(t)
    n = t.numel()
    cap = uzip_max_compressed_size(d, n)
    if out is None:
        out = torch.empty(cap, dtype=torch.uint8, device=t.device)
    if out_size is None:
        out_size = torch.empty((), dtype=torch.int64, device=t.device)
    _check(uzip_compress(t.data_ptr() if n else None, d, n, out.data_ptr(), out.numel(), out_size.data_ptr(),
                         _stream(stream)), "uzip_compress")
    return out, out_size


def compressed_bytes(buf, size) -> "torch.Tensor":
    """The container as a uint8 CUDA tensor (synchronises to read the size)."""
    return buf[: int(size.item())]


def decompress(comp, dtype, n: int, stream=None, out=None, status=None, check: bool = True):
    """Decompress a container held in a uint8 CUDA tensor into a new tensor.

    With check=True the device status is read back (one sync) and a corrupt
    container raises UzipError.
    """
    import torch

    table = _torch_dtypes()
    d = next((c for c, t in table.items() if dtype == c or dtype == t), -1)
    if d < 0:
        raise UzipError(UZIP_ERR_UNSUPPORTED_DTYPE, f"dtype {dtype}")
    tdt = table[d]
    if out is None:
        out = torch.empty(n, dtype=tdt, device=comp.device)
    if status is None:
        status = torch.empty((), dtype=torch.int32, device=comp.device)
    _check(uzip_decompress(comp.data_ptr(), comp.numel(), out.data_ptr() if n else None, d, n, status.data_ptr(),
                           _stream(stream)), "uzip_decompress")
    if check:
        st = int(status.item())
        if st != UZIP_OK:
            raise UzipError(st, "uzip_decompress (device)")
    return out
