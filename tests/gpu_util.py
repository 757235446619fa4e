"""Helpers for GPU tests: move bit patterns to the device and call the C ABI."""
import numpy as np

BF16, FP32, FP16, FP8_E4M3, FP8_E5M2 = 0, 1, 2, 3, 4
ELEM_BYTES = {BF16: 2, FP32: 4, FP16: 2, FP8_E4M3: 1, FP8_E5M2: 1}
BITS = {BF16: np.uint16, FP32: np.uint32, FP16: np.uint16, FP8_E4M3: np.uint8, FP8_E5M2: np.uint8}


def dtype_of(bits):
    """bf16 as uint16 bit patterns, fp16 as float16, fp32 as uint32/float32;
    fp8 arrays (uint8) need the dtype given explicitly."""
    if bits.dtype == np.uint16:
        return BF16
    if bits.dtype == np.float16:
        return FP16
    if bits.dtype in (np.uint32, np.float32):
        return FP32
    raise TypeError(f"pass the dtype for numpy {bits.dtype}")


def to_device(bits):
    import torch

    if bits.dtype == np.uint16:
        return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    if bits.dtype == np.float16:
        return torch.from_numpy(bits.copy()).cuda()
    if bits.dtype == np.uint8:
        return torch.from_numpy(bits.copy()).cuda()
    return torch.from_numpy(bits.view(np.int32).copy()).cuda().view(torch.float32)


def to_bits(t):
    import torch

    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def gpu_compress(bits, flags=0, dtype=None):
    """Compress through the C ABI.  Returns (container bytes, device status)."""
    import torch

    import lossless_float_tensor_gb300 as uz

    d = dtype_of(bits) if dtype is None else dtype
    n = bits.size
    x = to_device(bits) if n else None
    cap = uz.uzip_max_compressed_size(d, n)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.full((), -1, dtype=torch.int64, device="cuda")
    status = torch.full((), -1, dtype=torch.int32, device="cuda")
    st = uz.uzip_compress_ex(x.data_ptr() if n else None, d, n, out.data_ptr(), cap, size.data_ptr(), status.data_ptr(),
                             flags, torch.cuda.current_stream().cuda_stream)
    assert st == uz.UZIP_OK, uz.uzip_status_string(st)
    torch.cuda.synchronize()
    total = int(size.item())
    return out[:total].cpu().numpy(), int(status.item())


def gpu_decompress(comp, dtype, n, capacity=None):
    """Decompress host container bytes on the GPU.  Returns (bits, status)."""
    import torch

    import lossless_float_tensor_gb300 as uz

    c = torch.from_numpy(np.ascontiguousarray(comp)).cuda() if comp.size else torch.zeros(16, dtype=torch.uint8, device="cuda")
    cap = comp.size if capacity is None else capacity
    es = ELEM_BYTES[dtype]
    out = torch.full((max(n, 1) * es,), 0xA5, dtype=torch.uint8, device="cuda")
    status = torch.full((), -1, dtype=torch.int32, device="cuda")
    st = uz.uzip_decompress(c.data_ptr(), cap, out.data_ptr(), dtype, n, status.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    if st != uz.UZIP_OK:
        return None, st
    torch.cuda.synchronize()
    raw = out.cpu().numpy()[: n * es]
    return raw.view(BITS[dtype]), int(status.item())
