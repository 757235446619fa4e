"""Calls that run on the GPU at the same time.

Every call keeps its working state in the buffers it is given, so calls on
different streams (or from different host threads) that share no buffer may
overlap on the device.  These tests issue several compressions, then several
decompressions, at once and check each container against the oracle byte for
byte and each round trip bit for bit.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

CH = 65536
# (dtype, elements): mixed formats, whole and ragged chunk counts, one
# tensor under a chunk, so that small and large grids overlap
CASES = [
    (gu.BF16, 3 * CH + 17),
    (gu.BF16, 40 * CH),
    (gu.FP32, 1000),
    (gu.FP16, 12 * CH + 4095),
    (gu.BF16, 64 * CH),
    (gu.FP8_E4M3, 7 * CH + 1),
    (gu.FP8_E5M2, 25 * CH),
]


def _bits(dtype, n, t):
    if dtype == gu.BF16:
        return synth.normal_bf16(n, 0.02 * (1 + t), 13, t)
    if dtype == gu.FP32:
        return synth.normal_fp32(n, 0.02, tensor=t)
    if dtype == gu.FP16:
        return synth.normal_fp16(n, 0.02, tensor=t)
    return synth.normal_fp8(n, "e4m3" if dtype == gu.FP8_E4M3 else "e5m2", 0.02, tensor=t)


def _device(bits):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8).copy()).cuda()


class _Job:
    def __init__(self, dtype, bits):
        import torch

        import lossless_float_tensor_gb300 as uz

        self.dtype, self.bits, self.n = dtype, bits, bits.size
        self.x = _device(bits)
        self.cap = uz.uzip_max_compressed_size(dtype, self.n)
        self.comp = torch.empty(self.cap, dtype=torch.uint8, device="cuda")
        self.size = torch.full((), -1, dtype=torch.int64, device="cuda")
        self.out = torch.empty_like(self.x)
        self.status = torch.full((), -1, dtype=torch.int32, device="cuda")
        self.stream = torch.cuda.Stream()

    def compress(self):
        import lossless_float_tensor_gb300 as uz

        return uz.uzip_compress(self.x.data_ptr(), self.dtype, self.n, self.comp.data_ptr(), self.cap,
                                self.size.data_ptr(), self.stream.cuda_stream)

    def decompress(self):
        import lossless_float_tensor_gb300 as uz

        return uz.uzip_decompress(self.comp.data_ptr(), self.cap, self.out.data_ptr(), self.dtype, self.n,
                                  self.status.data_ptr(), self.stream.cuda_stream)

    def check(self):
        import torch

        total = int(self.size.item())
        want = oracle.compress(self.bits, self.dtype)
        got = self.comp[:total].cpu().numpy()
        assert got.size == want.size and np.array_equal(got, want), (self.dtype, self.n)
        assert int(self.status.item()) == 0
        assert torch.equal(self.out, self.x), (self.dtype, self.n)


def _all_at_once(jobs, method):
    """Every job's call issued behind one start event, so the launches can
    overlap on the device."""
    import torch

    start = torch.cuda.Event()
    start.record(torch.cuda.current_stream())
    for j in jobs:
        j.stream.wait_event(start)
        assert getattr(j, method)() == 0
    torch.cuda.synchronize()


def test_seven_calls_on_seven_streams_match_the_oracle():
    jobs = [_Job(d, _bits(d, n, t)) for t, (d, n) in enumerate(CASES)]
    for _ in range(2):  # the second round reuses every buffer
        _all_at_once(jobs, "compress")
        _all_at_once(jobs, "decompress")
        for j in jobs:
            j.check()


def test_calls_from_four_host_threads_match_the_oracle():
    import torch

    jobs = [_Job(d, _bits(d, n, 20 + t)) for t, (d, n) in enumerate(CASES)]
    torch.cuda.synchronize()

    def worker(mine):
        for _ in range(3):
            for j in mine:
                assert j.compress() == 0
                assert j.decompress() == 0
            for j in mine:
                j.stream.synchronize()
        return True

    groups = [jobs[i::4] for i in range(4)]
    with ThreadPoolExecutor(4) as pool:
        assert all(pool.map(worker, groups))
    torch.cuda.synchronize()
    for j in jobs:
        j.check()


def test_same_tensor_into_separate_buffers_at_once():
    """One input, read by four compressions at once (the input is never
    written), each into its own output."""
    bits = synth.normal_bf16(33 * CH + 5, 0.02, 13, 99)
    jobs = [_Job(gu.BF16, bits) for _ in range(4)]
    x = jobs[0].x
    for j in jobs[1:]:
        j.x = x
    _all_at_once(jobs, "compress")
    _all_at_once(jobs, "decompress")
    want = oracle.compress(bits, gu.BF16)
    for j in jobs:
        total = int(j.size.item())
        got = j.comp[:total].cpu().numpy()
        assert np.array_equal(got, want)
        assert int(j.status.item()) == 0
    import torch

    assert all(torch.equal(j.out, x) for j in jobs)


def test_round_trips_through_host_buffers_overlapped_on_three_streams():
    """Steps of input up, compress, container down at its exact size,
    container up, decompress, output down, run as a two-slot pipeline on
    upload, kernel and download streams (the schedule of the benchmark's
    end-to-end figure), with a different tensor every step so that a buffer
    reused too early would show: every container equals the oracle's and
    every output the input."""
    import torch

    import lossless_float_tensor_gb300 as uz

    steps, S, n = 6, 2, 5 * CH + 123
    inputs = [synth.normal_bf16(n, 0.01 * (1 + k), 13, 40 + k) for k in range(steps)]
    want = [oracle.compress(b) for b in inputs]
    cap = uz.uzip_max_compressed_size(gu.BF16, n)
    h_in = [torch.from_numpy(b.view(np.int16)).pin_memory() for b in inputs]
    h_comp = [torch.empty(cap, dtype=torch.uint8).pin_memory() for _ in range(S)]
    h_out = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(steps)]
    h_size = torch.zeros(S, dtype=torch.int64).pin_memory()
    got = [None] * steps
    d_in = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(S)]
    d_comp = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(S)]
    d_size = [torch.zeros((), dtype=torch.int64, device="cuda") for _ in range(S)]
    d_comp2 = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(S)]
    d_out = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(S)]
    d_status = [torch.full((), -1, dtype=torch.int32, device="cuda") for _ in range(S)]
    up, ks, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = [{k: torch.cuda.Event() for k in ("comp", "cdn", "cup", "dec", "odn", "in")} for _ in range(S)]
    tb = [0] * S
    statuses = []
    for k in range(steps + 1):
        if k < steps:  # input k up, compress k
            b, e = k % S, ev[k % S]
            if k >= S:
                up.wait_event(e["comp"])
            with torch.cuda.stream(up):
                d_in[b].copy_(h_in[k], non_blocking=True)
            e["in"].record(up)
            ks.wait_event(e["in"])
            if k >= S:
                ks.wait_event(e["cdn"])
            with torch.cuda.stream(ks):
                assert uz.uzip_compress(d_in[b].data_ptr(), gu.BF16, n, d_comp[b].data_ptr(), cap,
                                        d_size[b].data_ptr(), ks.cuda_stream) == 0
                h_size[b].copy_(d_size[b], non_blocking=True)
            e["comp"].record(ks)
        if k >= 1:  # container k - 1 up, decompress it
            j = k - 1
            b, e = j % S, ev[j % S]
            up.wait_event(e["cdn"])
            if j >= S:
                up.wait_event(e["dec"])
            with torch.cuda.stream(up):
                d_comp2[b][:tb[b]].copy_(h_comp[b][:tb[b]], non_blocking=True)
            e["cup"].record(up)
            ks.wait_event(e["cup"])
            if j >= S:
                ks.wait_event(e["odn"])
            with torch.cuda.stream(ks):
                assert uz.uzip_decompress(d_comp2[b].data_ptr(), tb[b], d_out[b].data_ptr(), gu.BF16, n,
                                          d_status[b].data_ptr(), ks.cuda_stream) == 0
            e["dec"].record(ks)
        if k < steps:  # the host reads size k; container k down
            b, e = k % S, ev[k % S]
            e["comp"].synchronize()
            tb[b] = int(h_size[b])
            down.wait_event(e["comp"])
            if k >= S:
                down.wait_event(e["cup"])
            with torch.cuda.stream(down):
                h_comp[b][:tb[b]].copy_(d_comp[b][:tb[b]], non_blocking=True)
            e["cdn"].record(down)
            e["cdn"].synchronize()  # keep a copy of container k for the oracle check
            got[k] = h_comp[b][:tb[b]].numpy().copy()
        if k >= 1:  # output k - 1 down
            j = k - 1
            b, e = j % S, ev[j % S]
            down.wait_event(e["dec"])
            with torch.cuda.stream(down):
                h_out[j].copy_(d_out[b], non_blocking=True)
            e["odn"].record(down)
            e["odn"].synchronize()
            statuses.append(int(d_status[b].item()))
    torch.cuda.synchronize()
    assert statuses == [0] * steps
    for k in range(steps):
        assert got[k].size == want[k].size and np.array_equal(got[k], want[k]), k
        assert np.array_equal(h_out[k].numpy().view(np.uint16), inputs[k]), k
