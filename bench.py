"""Benchmark: compress + decompress of a 1 GiB bf16 activation tensor on GB300.

One step = the whole hot path over one tensor: plane split, histogram,
normalisation, rANS encode, look-back placement (one fused compress kernel)
and the table decoder with plane merge (one decompress kernel).  The
workload is [8, 8192, 8192] bf16 ~ 0.5 * Student-t(4) with 1% outlier
channels x50 and one random-bits chunk (the 1 GiB bf16 configuration).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  --impl reference times the oracle (single-threaded C)
on a bounded sample of the same workload on the host cores.  Under torchrun
every rank runs an independent replica (the codec has no exchange step);
value = elements of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compress & decompress GB/s (input bytes), ratio, % of HBM roofline, 1 GB300"
WORKLOAD = ("c4: bf16 activations [8, 8192, 8192] ~ 0.5*Student-t(4), 82 outlier channels x50, "
            "chunk 4096 random bits; 536,870,912 values (1 GiB)")
KERNEL_SOURCES = ["lossless_float_tensor_gb300/csrc/compress_kernels.cuh", "lossless_float_tensor_gb300/csrc/compress.cu",
                  "lossless_float_tensor_gb300/csrc/decompress.cu", "lossless_float_tensor_gb300/csrc/uzip_internal.cuh"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch_full")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [v for v in sm if mx and v >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(dev_index: int) -> str:
    import torch

    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's figure (every rank gets it).  Works on any backend:
    the tensor lives on `device` (a CUDA device for NCCL, the CPU for gloo)."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput_gbs(bytes_per_rank: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job input GB/s: every rank compresses and decompresses its own
    replica of the workload, so the job moves world * bytes per step, in the
    slowest rank's time."""
    return world * bytes_per_rank * steps / (max_ms / 1e3) / 1e9


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz
    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    bits = synth.c4(n=args.elements)
    n = bits.size
    x = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    cap = uz.uzip_max_compressed_size(uz.UZIP_BF16, n)
    comp = torch.empty(cap, dtype=torch.uint8, device=dev)
    size = torch.zeros((), dtype=torch.int64, device=dev)
    out = torch.empty_like(x)
    status = torch.zeros((), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        st = uz.uzip_compress(x.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), sp)
        if ev is not None:
            ev[1].record(stream)
        st2 = uz.uzip_decompress(comp.data_ptr(), cap, out.data_ptr(), uz.UZIP_BF16, n, status.data_ptr(), sp)
        if ev is not None:
            ev[2].record(stream)
        if st or st2:
            raise RuntimeError(f"uzip status {st} {st2}")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    total = int(size.item())
    if int(status.item()) != 0 or not torch.equal(out.view(torch.int16), x.view(torch.int16)):
        raise RuntimeError("round trip failed during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_id_for(local_rank)) as clk:
        t0 = time.perf_counter()
        for k in range(args.steps):
            step(events[k])
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    tc = [e[0].elapsed_time(e[1]) for e in events]
    td = [e[1].elapsed_time(e[2]) for e in events]
    step_ms = [e[0].elapsed_time(e[2]) for e in events]
    dev_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = dev_ms / args.steps
    in_bytes = 2 * n
    value = replica_throughput_gbs(in_bytes, args.steps, dev_ms, world)

    # end to end through the public API with host buffers
    e2e = None
    if rank == 0 and not args.no_e2e:
        e2e = run_e2e(args, x, bits, comp, cap, size, out, status, stream, dev, total)

    if rank != 0:
        return None
    peak, peak_kind = measured_peak_hbm()
    mc, md = statistics.mean(tc), statistics.mean(td)
    comp_bytes = in_bytes + total      # read input, write container
    dec_bytes = total + in_bytes       # read container, write output
    roof_c = {"bound": "hbm", "achieved": comp_bytes / (mc / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
              "frac": comp_bytes / (mc / 1e3) / 1e9 / peak, "traffic": profiled_traffic("compress"),
              "kernel": "compress_kernel<bf16>", "algorithmic_bytes_per_launch": comp_bytes, "ms_per_launch": mc,
              "peak_source": f"{peak_kind} hbm_gbs"}
    roof_d = {"bound": "hbm", "achieved": dec_bytes / (md / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
              "frac": dec_bytes / (md / 1e3) / 1e9 / peak, "traffic": profiled_traffic("decompress"),
              "kernel": "decompress_kernel<bf16>", "algorithmic_bytes_per_launch": dec_bytes, "ms_per_launch": md,
              "peak_source": f"{peak_kind} hbm_gbs"}
    dominant = roof_c if mc >= md else roof_d
    cpu = None if args.no_cpu_baseline else cpu_baseline(bits)
    pipe = None if args.no_pipeline else run_pipeline(args, dev)
    sweep = None if args.no_dtypes else run_dtype_sweep(args, dev, peak)
    gate = None if args.no_gate else run_gate(args, dev, x, n, peak)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": WORKLOAD if args.elements is None else f"first {n} values of " + WORKLOAD,
                   "elements": n, "input_bytes": in_bytes, "parallelism": f"replicas x{world}",
                   "l2": "inputs (1 GiB) larger than L2; no flush"},
        "compress_gbs": in_bytes / (mc / 1e3) / 1e9, "decompress_gbs": in_bytes / (md / 1e3) / 1e9,
        "ratio": total / in_bytes, "compressed_bytes": total,
        "roofline": dominant, "roofline_compress": roof_c, "roofline_decompress": roof_d,
        "clocks": clk.summary(), "e2e": e2e, "gpu_launches": 2 * args.steps,
        "wall_s_timed_region": wall, "cpu_baseline": cpu, "pipeline": pipe, "dtype_sweep": sweep, "gate": gate,
        "kernel_source_hash": kernel_hash(),
    }
    return line


def run_e2e(args, x, bits, comp, cap, size, out, status, stream, dev, total):
    """H2D of the input from pinned memory, compress, D2H of the container,
    H2D of the container, decompress, D2H of the output, every step."""
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz

    n = bits.size
    h_in = torch.from_numpy(bits.view(np.int16)).pin_memory()
    h_comp = torch.empty(cap, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(n, dtype=torch.int16).pin_memory()
    h_size = torch.zeros((), dtype=torch.int64).pin_memory()
    d_in = torch.empty(n, dtype=torch.int16, device=dev)
    d_comp2 = torch.empty(cap, dtype=torch.uint8, device=dev)
    sp = stream.cuda_stream
    steps = max(1, min(args.steps, 5))

    def one():
        with torch.cuda.stream(stream):
            d_in.copy_(h_in, non_blocking=True)
            st = uz.uzip_compress(d_in.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), sp)
            h_size.copy_(size, non_blocking=True)
        stream.synchronize()
        tb = int(h_size.item())
        with torch.cuda.stream(stream):
            h_comp[:tb].copy_(comp[:tb], non_blocking=True)
            d_comp2[:tb].copy_(h_comp[:tb], non_blocking=True)
            st2 = uz.uzip_decompress(d_comp2.data_ptr(), tb, out.data_ptr(), uz.UZIP_BF16, n, status.data_ptr(), sp)
            h_out.copy_(out.view(torch.int16), non_blocking=True)
        stream.synchronize()
        if st or st2:
            raise RuntimeError("e2e status")
        return tb

    one()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    tb = 0
    for _ in range(steps):
        tb = one()
    dt = (time.perf_counter() - t0) / steps
    ok = bool(np.array_equal(h_out.numpy().view(np.uint16), bits))
    return {"value": 2 * n / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 2 * n + tb,
            "d2h_bytes_per_step": tb + 2 * n + 8, "steps": steps, "bit_exact": ok}


def run_pipeline(args, dev):
    """Split-send pipeline (two streams, two ping-pong banks) on c5-shaped
    messages: the first 1 GiB message of the Llama-3-8B-shaped parameter set
    (bf16 ~ N(0, 0.02)) is sent `reps` times, and prefixes of it give the
    64 KiB .. 1 GiB size sweep.  Reported: input GB/s of the pipelined modes
    (exact-size copy kernel into mapped pinned memory; exact-size
    cudaMemcpyAsync issued once the host has read the size; streamed copies of
    finished remainder and stream runs while the message compresses;
    bound-size cudaMemcpyAsync), of compress-then-copy on one stream (no
    overlap), and of a plain device-to-host copy of the uncompressed bytes.
    Also the latency of one 1 GiB message: from the call to the last byte on
    the host, sized versus streamed."""
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz
    import synth

    msg = synth.c5_message(0)
    n_max = msg.size
    x = torch.from_numpy(msg.view(np.int16)).to(dev)
    cap = uz.uzip_max_compressed_size(uz.UZIP_BF16, n_max)
    banks = [torch.empty(cap, dtype=torch.uint8, device=dev) for _ in range(2)]
    hcap = cap + 16 * (-(-n_max // 65536))  # the streamed mode keeps progress words past the container
    hb = [torch.empty(hcap, dtype=torch.uint8).pin_memory() for _ in range(2)]
    h_raw = torch.empty(2 * n_max, dtype=torch.uint8).pin_memory()
    s0, s1 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    modes = {"exact": uz.UZIP_PIPE_EXACT, "sized": uz.UZIP_PIPE_SIZED, "streamed": uz.UZIP_PIPE_STREAMED,
             "bound": uz.UZIP_PIPE_BOUND, "serial": uz.UZIP_PIPE_SERIAL}
    sizes = [1 << 15, 1 << 17, 1 << 19, 1 << 21, 1 << 23, 1 << 25, 1 << 27, n_max]  # values (64 KiB .. 1 GiB)
    sweep = []
    for n in sizes:
        reps = int(max(4, min(64, (4 << 30) // (2 * n))))
        if n == n_max:
            reps = args.pipeline_messages
        hs = torch.zeros(reps, dtype=torch.int64).pin_memory()
        row = {"message_bytes": 2 * n, "messages": reps}
        for name, mode in modes.items():
            for it in range(2):  # first pass warms up
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                st = uz.uzip_pipeline_send(uz.UZIP_BF16, [x.data_ptr()] * reps, [n] * reps,
                                           [b.data_ptr() for b in banks], cap, [h.data_ptr() for h in hb], hcap,
                                           hs.data_ptr(), mode, s0.cuda_stream, s1.cuda_stream)
                torch.cuda.synchronize(dev)
                dt = time.perf_counter() - t0
                if st != 0:
                    raise RuntimeError(f"pipeline status {st}")
            row[name + "_gbs"] = reps * 2 * n / dt / 1e9
        row["ratio"] = int(hs[0]) / (2 * n)
        # plain copy of the raw bytes over the same link
        raw = x.view(torch.uint8)[: 2 * n]
        for it in range(2):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            with torch.cuda.stream(s1):
                for _ in range(reps):
                    h_raw[: 2 * n].copy_(raw, non_blocking=True)
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
        row["raw_d2h_gbs"] = reps * 2 * n / dt / 1e9
        sweep.append(row)
    # one 1 GiB message, from the call to its last byte on the host
    hs1 = torch.zeros(1, dtype=torch.int64).pin_memory()
    latency = {}
    for name in ("sized", "streamed"):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            st = uz.uzip_pipeline_send(uz.UZIP_BF16, [x.data_ptr()], [n_max], [b.data_ptr() for b in banks], cap,
                                       [h.data_ptr() for h in hb], hcap, hs1.data_ptr(), modes[name], s0.cuda_stream,
                                       s1.cuda_stream)
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
            if st != 0:
                raise RuntimeError(f"pipeline status {st}")
        latency[name + "_ms"] = best * 1e3
    full = sweep[-1]
    return {"one_message_latency": latency,
            "workload": "c5: first 1 GiB message of the Llama-3-8B-shaped bf16 parameter set ~ N(0, 0.02), "
                        f"sent {full['messages']} times; size sweep on its prefixes",
            "unit": "GB/s (input bytes, host wall clock incl. sync)", "sweep": sweep,
            "exact_gbs": full["exact_gbs"], "sized_gbs": full["sized_gbs"], "streamed_gbs": full["streamed_gbs"],
            "bound_gbs": full["bound_gbs"],
            "serial_gbs": full["serial_gbs"],
            "raw_d2h_gbs": full["raw_d2h_gbs"]}


def run_gate(args, dev, x, n, peak):
    """Whole-message choice (uzip_compress_gated): on the c4 tensor the 64 KiB
    sample codes, so the gated call costs the gate kernel on top of the usual
    compression; on 1 GiB of random bf16 bits the sample goes RAW and the
    whole message is split and stored RAW without statistics or coding.  Also
    c4 with tables from a sample of each chunk (UZIP_FLAG_SAMPLED_TABLES).
    CUDA events, mean of 5 launches after 3 warm-ups."""
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz

    cap = uz.uzip_max_compressed_size(uz.UZIP_BF16, n)
    comp = torch.empty(cap, dtype=torch.uint8, device=dev)
    size = torch.zeros((), dtype=torch.int64, device=dev)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
            for e0, e1 in ev:
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)

    def run(t, raw_below=None):
        if raw_below is None:
            st = uz.uzip_compress(t.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), sp)
        else:
            st = uz.uzip_compress_gated(t.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), None,
                                        raw_below, sp)
        if st:
            raise RuntimeError(f"uzip status {st}")

    rows = {}
    rows["c4_plain_ms"] = timed(lambda: run(x))
    rows["c4_gated_ms"] = timed(lambda: run(x, 0))
    rows["c4_gated_bytes"] = int(size.item())
    rows["c4_forced_raw_ms"] = timed(lambda: run(x, 1 << 62))
    rnd = torch.from_numpy(np.random.default_rng(17).integers(0, 1 << 16, n, dtype=np.uint16).view(np.int16)).to(dev)
    rows["random_plain_ms"] = timed(lambda: run(rnd))
    rows["random_gated_ms"] = timed(lambda: run(rnd, 0))
    rows["random_gated_bytes"] = int(size.item())
    rows["raw_frac_of_hbm"] = (4 * n) / (rows["random_gated_ms"] / 1e3) / 1e9 / peak

    def run_sampled():
        st = uz.uzip_compress_ex(x.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), None,
                                 uz.UZIP_FLAG_SAMPLED_TABLES, sp)
        if st:
            raise RuntimeError(f"uzip status {st}")

    rows["c4_sampled_tables_ms"] = timed(run_sampled)
    rows["c4_sampled_tables_bytes"] = int(size.item())
    del rnd
    return {"workload": "c4 (1 GiB bf16) and 1 GiB of random bf16 bits (numpy seed 17)", "unit": "ms per launch",
            **rows}


def run_dtype_sweep(args, dev, peak):
    """The five element formats of UCCL-Zip Fig. 12 on one 256 MiB tensor
    each, ~ N(0, 0.02) rounded to the format: compress and decompress GB/s of
    input (CUDA events, mean of 5 launches after 3 warm-ups), the ratio, the
    fraction of the HBM roofline, and whether the container equals the
    oracle's byte for byte and the round trip is bit-exact."""
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz
    import oracle
    import synth

    nbytes = 256 << 20
    gens = [("bf16", uz.UZIP_BF16, 2, lambda n: synth.normal_bf16(n, 0.02, 13, 0)),
            ("fp16", uz.UZIP_FP16, 2, lambda n: synth.normal_fp16(n, 0.02, 13, 1)),
            ("fp32", uz.UZIP_FP32, 4, lambda n: synth.normal_fp32(n, 0.02, 13, 2)),
            ("fp8_e4m3fn", uz.UZIP_FP8_E4M3, 1, lambda n: synth.normal_fp8(n, "e4m3", 0.02, 13, 3)),
            ("fp8_e5m2", uz.UZIP_FP8_E5M2, 1, lambda n: synth.normal_fp8(n, "e5m2", 0.02, 13, 4))]
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    rows = []
    for name, code, es, gen in gens:
        n = nbytes // es
        bits = gen(n)
        x = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8)).to(dev)
        cap = uz.uzip_max_compressed_size(code, n)
        comp = torch.empty(cap, dtype=torch.uint8, device=dev)
        size = torch.zeros((), dtype=torch.int64, device=dev)
        out = torch.empty_like(x)
        status = torch.zeros((), dtype=torch.int32, device=dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(5)]
        with torch.cuda.stream(stream):
            for k in range(3 + 5):
                e = ev[k - 3] if k >= 3 else None
                if e:
                    e[0].record(stream)
                st = uz.uzip_compress(x.data_ptr(), code, n, comp.data_ptr(), cap, size.data_ptr(), sp)
                if e:
                    e[1].record(stream)
                st2 = uz.uzip_decompress(comp.data_ptr(), cap, out.data_ptr(), code, n, status.data_ptr(), sp)
                if e:
                    e[2].record(stream)
                if st or st2:
                    raise RuntimeError(f"{name}: uzip status {st} {st2}")
        torch.cuda.synchronize(dev)
        total = int(size.item())
        exact = int(status.item()) == 0 and torch.equal(out, x)
        want = oracle.compress(bits, code)
        same = want.size == total and np.array_equal(comp[:total].cpu().numpy(), want)
        mc = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        md = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        moved = nbytes + total
        rows.append({"dtype": name, "elements": n, "input_bytes": nbytes, "ratio": total / nbytes,
                     "compress_gbs": nbytes / (mc / 1e3) / 1e9, "decompress_gbs": nbytes / (md / 1e3) / 1e9,
                     "compress_frac": moved / (mc / 1e3) / 1e9 / peak, "decompress_frac": moved / (md / 1e3) / 1e9 / peak,
                     "round_trip_exact": bool(exact), "oracle_bytes_equal": bool(same)})
        del x, comp, out
    return {"workload": "one 256 MiB tensor per format ~ N(0, 0.02) (UCCL-Zip Fig. 12 format sweep)", "rows": rows}


def cpu_baseline(bits):
    """The oracle (single-threaded C) on a bounded sample of the tensor (the
    first 2048 chunks), compress + decompress."""
    import oracle

    sample = bits[: 2048 * 65536]
    t0 = time.perf_counter()
    c = oracle.compress(sample)
    t1 = time.perf_counter()
    oracle.decompress(c, oracle.BF16, sample.size)
    t2 = time.perf_counter()
    return {"value": 2 * sample.size / (t2 - t0) / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {sample.size} values of the workload ({sample.size // 65536} chunks), "
                      f"compress {t1 - t0:.2f} s + decompress {t2 - t1:.2f} s",
            "compress_gbs": 2 * sample.size / (t1 - t0) / 1e9, "decompress_gbs": 2 * sample.size / (t2 - t1) / 1e9}


def run_reference(args):
    """Reference arm: the oracle on the host cores, each step one bounded sample
    (the first 256 chunks, 16,777,216 values) of the same workload."""
    import oracle
    import synth

    bits = synth.c4(n=256 * 65536)
    n = bits.size
    times = []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        c = oracle.compress(bits)
        oracle.decompress(c, oracle.BF16, n)
        if k >= args.warmup:
            times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    value = 2 * n / per / 1e9
    cpu = {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"first 256 chunks ({n} values) of the workload per step"}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "elements": n, "parallelism": "host, 1 thread"},
            "ratio": c.size / (2 * n), "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pipeline", action="store_true")
    ap.add_argument("--no-dtypes", action="store_true", help="skip the fp16/fp32/fp8 format sweep")
    ap.add_argument("--no-gate", action="store_true", help="skip the whole-message RAW / gate measurement")
    ap.add_argument("--pipeline-messages", type=int, default=8,
                    help="1 GiB messages sent through the split-send pipeline")
    ap.add_argument("--elements", type=int, default=None,
                    help="use only the first N values of the workload (profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import __graft_entry__

    __graft_entry__.build_library()
    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
