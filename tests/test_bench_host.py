"""Host-side helpers of the benchmark (no GPU): the DRAM traffic figure is
taken from the committed ncu summary only while the kernel sources are the
ones it was captured on, and the replica throughput counts every rank."""
import json
import os

import pytest

import bench


def _committed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as fh:
        return json.load(fh)


def test_kernel_hash_is_stable_hex():
    for k in (None, "compress", "decompress"):
        h = bench.kernel_hash(k)
        assert h == bench.kernel_hash(k)
        assert len(h) == 16 and int(h, 16) >= 0
    assert bench.kernel_hash("compress") != bench.kernel_hash("decompress")


@pytest.mark.parametrize("kernel", ["compress", "decompress"])
def test_traffic_only_for_the_captured_sources(kernel, monkeypatch):
    entry = _committed()[kernel]
    monkeypatch.setattr(bench, "kernel_hash", lambda k=None: entry["source_hash"])
    got = bench.profiled_traffic(kernel)
    assert got == entry["dram_bytes_per_launch_full"]
    # scaled from the capture by the chunk counts of the two launches
    small = entry["dram_bytes_read_small"] + entry["dram_bytes_write_small"]
    chunks = lambda n: -(-n // 65536)  # noqa: E731
    assert got == pytest.approx(small * chunks(entry["elements_full"]) / chunks(entry["elements_small"]))
    monkeypatch.setattr(bench, "kernel_hash", lambda k=None: "0" * 16)
    assert bench.profiled_traffic(kernel) is None


def test_unknown_kernel_has_no_traffic():
    assert bench.profiled_traffic("no_such_kernel") is None


def test_replica_throughput_sums_ranks():
    one = bench.replica_throughput_gbs(1 << 30, 10, 5.0, 1)
    assert one == pytest.approx((1 << 30) * 10 / 5e-3 / 1e9)
    assert bench.replica_throughput_gbs(1 << 30, 10, 5.0, 4) == pytest.approx(4 * one)


def test_round_trip_counts_the_input_once():
    # a round trip of B input bytes at compress rate a and decompress rate b
    # (bytes/s) takes B/a + B/b seconds: its rate is the harmonic combination
    b, a, d = 1 << 30, 0.165e9, 0.197e9
    got = bench.round_trip_gbs(b, b / a, b / d)
    assert got == pytest.approx(1 / (1 / 0.165 + 1 / 0.197))
    # the GPU line's value uses the same measure: input bytes per round trip
    assert bench.replica_throughput_gbs(b, 1, (b / a + b / d) * 1e3, 1) == pytest.approx(got)
