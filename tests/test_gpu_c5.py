"""The whole Llama-3-8B-shaped parameter set (8,030,261,248 bf16 values,
16.06 GB) through the split-send pipeline: 15 messages of 1 GiB, the last
ending in a 4,096-element chunk.  Every container is compared byte for byte
with the oracle's (the oracle runs single-threaded, one message per host
thread: "oracle x N threads") and decoded back on the GPU bit for bit.

The pipeline runs messages in groups of three with one host bank per message
(uzip_pipeline_send_ex), so two messages are always in flight and every
container stays on the host for the check.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

GROUP = 3


def _oracle_equal(bits, container):
    want = oracle.compress(bits)
    return want.size == container.size and bool(np.array_equal(want, container))


def test_c5_every_message_through_the_pipeline_matches_the_oracle():
    import torch

    import lossless_float_tensor_gb300 as uz

    sizes = synth.c5_message_sizes()
    assert len(sizes) == 15 and sum(sizes) == synth.C5_TOTAL
    assert sizes[-1] % 65536 == 4096
    largest = max(sizes)
    cap = uz.uzip_max_compressed_size(uz.UZIP_BF16, largest)
    banks = [torch.empty(cap, dtype=torch.uint8, device="cuda") for _ in range(2)]
    hcap = cap + 16 * (-(-largest // 65536))
    hb = [torch.empty(hcap, dtype=torch.uint8).pin_memory() for _ in range(GROUP)]
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    checks = []
    ratios = []
    with ThreadPoolExecutor(max(1, min(len(sizes), (os.cpu_count() or 2) - 1))) as pool:
        for g0 in range(0, len(sizes), GROUP):
            ks = list(range(g0, min(len(sizes), g0 + GROUP)))
            msgs = [synth.c5_message(k) for k in ks]
            d_msgs = [torch.from_numpy(m.view(np.int16)).cuda() for m in msgs]
            h_sizes = torch.zeros(len(ks), dtype=torch.int64).pin_memory()
            torch.cuda.synchronize()
            st = uz.uzip_pipeline_send_ex(uz.UZIP_BF16, [d.data_ptr() for d in d_msgs], [m.size for m in msgs],
                                          [b.data_ptr() for b in banks], cap, [h.data_ptr() for h in hb[:len(ks)]],
                                          hcap, h_sizes.data_ptr(), uz.UZIP_PIPE_SIZED, uz.UZIP_PIPE_RAW_BELOW_DEFAULT,
                                          s0.cuda_stream, s1.cuda_stream)
            assert st == 0, uz.uzip_status_string(st)
            torch.cuda.synchronize()
            for i, k in enumerate(ks):
                total = int(h_sizes[i])
                assert total > 0
                container = hb[i][:total].numpy().copy()
                ratios.append(total / (2 * msgs[i].size))
                # round trip on the GPU from the host copy
                d_c = torch.from_numpy(container).cuda()
                out = torch.empty_like(d_msgs[i])
                status = torch.full((), -1, dtype=torch.int32, device="cuda")
                rc = uz.uzip_decompress(d_c.data_ptr(), total, out.data_ptr(), uz.UZIP_BF16, msgs[i].size,
                                        status.data_ptr(), torch.cuda.current_stream().cuda_stream)
                assert rc == 0
                torch.cuda.synchronize()
                assert int(status.item()) == 0, f"message {k}"
                assert torch.equal(out, d_msgs[i]), f"message {k} does not round-trip"
                checks.append((k, pool.submit(_oracle_equal, msgs[i], container)))
                del d_c, out
            del d_msgs
        bad = [k for k, f in checks if not f.result()]
    assert not bad, f"containers differ from the oracle's for messages {bad}"
    assert len(checks) == 15
    assert all(0.65 < r < 0.67 for r in ratios), ratios
