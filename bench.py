"""Benchmark: compress + decompress of a 1 GiB bf16 activation tensor on GB300.

One step = the whole hot path over one tensor: plane split, histogram,
normalisation, rANS encode, look-back placement (one fused compress kernel)
and the table decoder with plane merge (one decompress kernel).  The
workload is [8, 8192, 8192] bf16 ~ 0.5 * Student-t(4) with 1% outlier
channels x50 and one random-bits chunk (the 1 GiB bf16 configuration).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  value = input bytes of all ranks per round trip (one
compress plus one decompress) / the slowest rank's time; e2e is the same
measure through the public API from and to pinned host buffers, consecutive
steps overlapped on upload, kernel and download streams.  The line also
carries the per-config table, the split-send pipeline over the whole c5
parameter set, the format sweep and the whole-message choice.  --impl
reference times the oracle (single-threaded C) on a bounded sample of the
same workload on the host cores.  Under torchrun every rank runs an
independent replica (the codec has no exchange step).
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
_CSRC = "lossless_float_tensor_gb300/csrc/"
# Sources each kernel is compiled from; a committed DRAM-traffic figure is
# only used while the hash of its kernel's sources is unchanged.
KERNEL_SOURCES = {
    "compress": [_CSRC + f for f in ("compress_kernels.cuh", "compress_ws.cuh", "compress.cu", "compress_fmt_bf16.cu",
                                     "uzip_internal.cuh")],
    "decompress": [_CSRC + f for f in ("decompress.cu", "uzip_internal.cuh")],
}


def kernel_hash(kernel: str | None = None) -> str:
    """16 hex digits of sha256 over one kernel's sources (all sources when
    kernel is None)."""
    files = KERNEL_SOURCES[kernel] if kernel else sorted({f for v in KERNEL_SOURCES.values() for f in v})
    h = hashlib.sha256()
    for p in files:
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
    if not e or kernel not in KERNEL_SOURCES or e.get("source_hash") != kernel_hash(kernel):
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


def round_trip_gbs(input_bytes: int, compress_s: float, decompress_s: float) -> float:
    """Input GB/s of one compress plus one decompress of input_bytes: the
    same measure as the line's value, so the CPU baseline compares with it."""
    return input_bytes / (compress_s + decompress_s) / 1e9


def host_description():
    """Host cores and CPU model (x86: 'model name'; Arm: implementer/part)."""
    model, impl, part = None, None, None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k == "model name" and model is None:
                    model = v
                elif k == "CPU implementer" and impl is None:
                    impl = v
                elif k == "CPU part" and part is None:
                    part = v
    except OSError:
        pass
    if model is None and impl is not None:
        model = f"Arm CPU implementer {impl}, part {part}"
    return {"host_cores": os.cpu_count(), "cpu_model": model or "unknown"}


def config_inputs(name):
    """(dtype code, list of bit arrays) of one workload of the per-config table."""
    import synth

    if name == "c1":
        return 0, [synth.c1()]
    if name == "c2":
        return 0, [synth.c2_tensor(t) for t in range(7)]
    if name == "c3":
        return 1, [synth.c3()]
    if name == "c4":
        return 0, [synth.c4()]
    if name == "c5m0":
        return 0, [synth.c5_message(0)]
    raise ValueError(name)


def oracle_job(name):
    """One single-threaded oracle run (compress, then decompress) over a whole
    workload of the per-config table, in a process of its own; returns the
    timings and a hash of each container (compared with the GPU's)."""
    import hashlib

    import numpy as np

    import oracle

    dtype, arrays = config_inputs(name)
    t_c = t_d = 0.0
    hashes, total, nbytes = [], 0, 0
    for bits in arrays:
        t0 = time.perf_counter()
        c = oracle.compress(bits, dtype)
        t1 = time.perf_counter()
        back = oracle.decompress(c, dtype, bits.size)
        t2 = time.perf_counter()
        assert np.array_equal(back.view(bits.dtype), bits)
        t_c += t1 - t0
        t_d += t2 - t1
        hashes.append(hashlib.sha256(c.tobytes()).hexdigest())
        total += c.size
        nbytes += bits.nbytes
    return {"config": name, "input_bytes": nbytes, "compressed_bytes": total, "compress_s": t_c, "decompress_s": t_d,
            "compress_gbs": nbytes / t_c / 1e9, "decompress_gbs": nbytes / t_d / 1e9, "sha256": hashes}


def start_oracle_jobs(names):
    """Oracle runs in spawned processes (1 thread each), started before the
    GPU work so they overlap it."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    pool = ctx.Pool(processes=max(1, min(len(names), (os.cpu_count() or 2) - 1)))
    return pool, {n: pool.apply_async(oracle_job, (n,)) for n in names}


CONFIG_LABELS = {
    "c1": "1,048,576 bf16 ~ N(0, 0.02); L2-resident (2 MiB), no flush",
    "c2": "Llama-3-8B-shaped layer, 7 bf16 weight tensors (218,103,808 values), one call each, summed; L2 flushed",
    "c3": "268,435,456 fp32 gradients with specials (1 GiB)",
    "c4": "[8, 8192, 8192] bf16 activations, 0.5*t(4), outliers x50, one random chunk (1 GiB)",
    "c5m0": "c5 message 0: first 1 GiB of the Llama-3-8B-shaped parameter set, bf16 ~ N(0, 0.02)",
    "c2_streams": "c2's 7 calls issued at once on 7 streams (one call per tensor, buffers of their own); L2 flushed",
}


def measure_concurrent(name, dtype, arrays, dev, peak, oracle_config):
    """The tensors of a workload compressed (then decompressed) by one call
    each, all calls issued at once on a stream per tensor: CUDA events from
    a start event every stream waits on to the last stream's end, mean of 5
    rounds after 3 warm-ups, L2 flushed before each timed round; plus the
    container hashes (the same bytes as one call at a time) and a bit-exact
    round-trip check."""
    import hashlib

    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz

    main = torch.cuda.Stream(dev)
    streams = [torch.cuda.Stream(dev) for _ in arrays]
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    xs = [torch.from_numpy(np.ascontiguousarray(b).view(np.uint8)).to(dev) for b in arrays]
    ns = [b.size for b in arrays]
    caps = [uz.uzip_max_compressed_size(dtype, n) for n in ns]
    comps = [torch.empty(c, dtype=torch.uint8, device=dev) for c in caps]
    sizes = [torch.zeros((), dtype=torch.int64, device=dev) for _ in arrays]
    outs = [torch.empty_like(x) for x in xs]
    stats = [torch.zeros((), dtype=torch.int32, device=dev) for _ in arrays]
    torch.cuda.synchronize(dev)

    def round_(launch):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        done = [torch.cuda.Event() for _ in streams]
        with torch.cuda.stream(main):
            scrub.fill_(7)
        t0.record(main)
        for i, st in enumerate(streams):
            st.wait_event(t0)
            with torch.cuda.stream(st):
                if launch(i, st.cuda_stream):
                    raise RuntimeError(f"{name}: uzip status")
            done[i].record(st)
        for d in done:
            main.wait_event(d)
        t1.record(main)
        return t0, t1

    def comp(i, sp):
        return uz.uzip_compress(xs[i].data_ptr(), dtype, ns[i], comps[i].data_ptr(), caps[i], sizes[i].data_ptr(), sp)

    def dec(i, sp):
        return uz.uzip_decompress(comps[i].data_ptr(), caps[i], outs[i].data_ptr(), dtype, ns[i], stats[i].data_ptr(),
                                  sp)

    tc, td = [], []
    for k in range(8):
        ec = round_(comp)
        ed = round_(dec)
        if k >= 3:
            tc.append(ec)
            td.append(ed)
    torch.cuda.synchronize(dev)
    mc = statistics.mean(a.elapsed_time(b) for a, b in tc) / 1e3
    md = statistics.mean(a.elapsed_time(b) for a, b in td) / 1e3
    tots = [int(s_.item()) for s_ in sizes]
    exact = all(int(s_.item()) == 0 for s_ in stats) and all(torch.equal(o, x) for o, x in zip(outs, xs))
    hashes = [hashlib.sha256(c[:t].cpu().numpy().tobytes()).hexdigest() for c, t in zip(comps, tots)]
    nbytes, total = sum(b.nbytes for b in arrays), sum(tots)
    moved = nbytes + total
    return {"config": name, "workload": CONFIG_LABELS[name], "input_bytes": nbytes, "compressed_bytes": total,
            "ratio": total / nbytes, "compress_ms": mc * 1e3, "decompress_ms": md * 1e3,
            "compress_gbs": nbytes / mc / 1e9, "decompress_gbs": nbytes / md / 1e9,
            "compress_frac": moved / mc / 1e9 / peak, "decompress_frac": moved / md / 1e9 / peak,
            "round_trip_exact": bool(exact), "sha256": hashes, "oracle_config": oracle_config}


def measure_config(name, dtype, arrays, dev, peak, flush_l2):
    """GPU compress / decompress of every tensor of a workload: CUDA events,
    mean of 5 launches after 3 warm-ups (L2 flushed before each timed launch
    when the inputs are smaller than L2), summed over the tensors; plus the
    container hashes and a bit-exact round-trip check."""
    import hashlib

    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz

    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None
    tc = td = 0.0
    nbytes = total = 0
    hashes, exact = [], True
    for bits in arrays:
        x = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8)).to(dev)
        n = bits.size
        cap = uz.uzip_max_compressed_size(dtype, n)
        comp = torch.empty(cap, dtype=torch.uint8, device=dev)
        size = torch.zeros((), dtype=torch.int64, device=dev)
        out = torch.empty_like(x)
        status = torch.zeros((), dtype=torch.int32, device=dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(5)]
        with torch.cuda.stream(stream):
            for k in range(8):
                e = ev[k - 3] if k >= 3 else None
                if e and scrub is not None:
                    scrub.fill_(k)
                if e:
                    e[0].record(stream)
                st = uz.uzip_compress(x.data_ptr(), dtype, n, comp.data_ptr(), cap, size.data_ptr(), sp)
                if e:
                    e[1].record(stream)
                    if scrub is not None:
                        scrub.fill_(k + 1)
                    e[2].record(stream)
                st2 = uz.uzip_decompress(comp.data_ptr(), cap, out.data_ptr(), dtype, n, status.data_ptr(), sp)
                if e:
                    e[3].record(stream)
                if st or st2:
                    raise RuntimeError(f"{name}: uzip status {st} {st2}")
        torch.cuda.synchronize(dev)
        tot = int(size.item())
        exact = exact and int(status.item()) == 0 and torch.equal(out, x)
        hashes.append(hashlib.sha256(comp[:tot].cpu().numpy().tobytes()).hexdigest())
        tc += statistics.mean(e[0].elapsed_time(e[1]) for e in ev) / 1e3
        td += statistics.mean(e[2].elapsed_time(e[3]) for e in ev) / 1e3
        nbytes += bits.nbytes
        total += tot
        del x, comp, out
    moved = nbytes + total
    return {"config": name, "workload": CONFIG_LABELS[name], "input_bytes": nbytes, "compressed_bytes": total,
            "ratio": total / nbytes, "compress_ms": tc * 1e3, "decompress_ms": td * 1e3,
            "compress_gbs": nbytes / tc / 1e9, "decompress_gbs": nbytes / td / 1e9,
            "compress_frac": moved / tc / 1e9 / peak, "decompress_frac": moved / td / 1e9 / peak,
            "round_trip_exact": bool(exact), "sha256": hashes}


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz
    import synth

    # the oracle's single-threaded runs over whole workloads, in spawned
    # processes overlapping the GPU work (rank 0, default sizes only)
    oracle_pool, oracle_runs = None, {}
    if rank == 0 and not args.no_cpu_baseline and args.elements is None:
        names = ["c4"] if args.no_configs else ["c4", "c1", "c2", "c3", "c5m0"]
        oracle_pool, oracle_runs = start_oracle_jobs(names)
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
              "kernel": "compress_ws_kernel<bf16>", "algorithmic_bytes_per_launch": comp_bytes, "ms_per_launch": mc,
              "peak_source": f"{peak_kind} hbm_gbs"}
    roof_d = {"bound": "hbm", "achieved": dec_bytes / (md / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
              "frac": dec_bytes / (md / 1e3) / 1e9 / peak, "traffic": profiled_traffic("decompress"),
              "kernel": "decompress_kernel<bf16>", "algorithmic_bytes_per_launch": dec_bytes, "ms_per_launch": md,
              "peak_source": f"{peak_kind} hbm_gbs"}
    dominant = roof_c if mc >= md else roof_d
    c5_msgs = None
    pipe = None
    if not args.no_pipeline and args.elements is None:
        pipe, c5_msgs = run_pipeline(args, dev)
    configs = None
    if not args.no_configs and args.elements is None:
        configs = run_configs(args, dev, peak, x, bits, c5_msgs)
    del c5_msgs
    torch.cuda.empty_cache()
    sweep = None if args.no_dtypes else run_dtype_sweep(args, dev, peak)
    gate = None if args.no_gate else run_gate(args, dev, x, n, peak)
    cpu = None
    if oracle_pool is not None:
        results = {k: r.get() for k, r in oracle_runs.items()}
        oracle_pool.close()
        oracle_pool.join()
        c4r = results["c4"]
        cpu = {"value": round_trip_gbs(c4r["input_bytes"], c4r["compress_s"], c4r["decompress_s"]), "unit": "GB/s",
               "cores": 1, "kind": "oracle",
               "sample": "the whole workload (536,870,912 values), compress "
                         f"{c4r['compress_s']:.1f} s + decompress {c4r['decompress_s']:.1f} s, one thread",
               "compress_gbs": c4r["compress_gbs"], "decompress_gbs": c4r["decompress_gbs"], **host_description()}
        if configs is not None:
            for row in configs["rows"]:
                r = results.get(row.get("oracle_config", row["config"]))
                if r is not None:
                    row["oracle_compress_gbs"] = r["compress_gbs"]
                    row["oracle_decompress_gbs"] = r["decompress_gbs"]
                    row["oracle_bytes_equal"] = r["sha256"] == row["sha256"]
            configs["oracle"] = {"cores": 1, "kind": "oracle, single-threaded C, one process per config",
                                 **host_description()}
        # the headline tensor's container against the oracle's
        c4_gpu = hashlib.sha256(comp[:total].cpu().numpy().tobytes()).hexdigest()
        cpu["oracle_bytes_equal"] = c4r["sha256"] == [c4_gpu]
    if configs is not None:
        for row in configs["rows"]:
            row["sha256"] = [h[:16] for h in row["sha256"]]
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
        "wall_s_timed_region": wall, "cpu_baseline": cpu, "configs": configs, "pipeline": pipe,
        "dtype_sweep": sweep, "gate": gate, "kernel_source_hash": kernel_hash(),
        "kernel_source_hashes": {k: kernel_hash(k) for k in KERNEL_SOURCES},
    }
    return line


def run_configs(args, dev, peak, x4, bits4, c5_msgs):
    """The per-config table: GPU compress / decompress GB/s, ratio and
    fraction of the HBM roofline for c1 (L2-resident), c2 (seven tensors, one
    call each), c3 (fp32), c4 and the first c5 message, with a hash of every
    container (compared with the oracle's when its runs are done)."""
    import numpy as np

    rows = []
    for name in ["c1", "c2", "c3"]:
        dtype, arrays = config_inputs(name)
        rows.append(measure_config(name, dtype, arrays, dev, peak, flush_l2=name == "c2"))
        if name == "c2":
            rows.append(measure_concurrent("c2_streams", dtype, arrays, dev, peak, "c2"))
        del arrays
    rows.append(measure_config("c4", 0, [bits4], dev, peak, flush_l2=False))
    if c5_msgs is not None:
        m0 = c5_msgs[0].cpu().numpy().view(np.uint16)
        rows.append(measure_config("c5m0", 0, [m0], dev, peak, flush_l2=False))
    return {"unit": "GB/s of input bytes; fractions of the measured HBM copy bandwidth", "rows": rows}


def run_e2e(args, x, bits, comp, cap, size, out, status, stream, dev, total):
    """End to end through the public API with host buffers.  Every step: H2D
    of the input from pinned memory, compress, D2H of the container (its
    exact size read on the host), H2D of the container, decompress, D2H of
    the output.  Steps run back to back as a two-slot software pipeline on
    three streams (uploads, kernels, downloads): the host link carries both
    directions at once, so step k's container and output travel down while
    step k + 1's input and step k's container travel up.  A buffer a step
    writes is written again two steps later, after an event says its last
    reader is done.  The same chain run one step at a time on one stream is
    reported beside it ("serial_gbs")."""
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz

    n = bits.size
    S = 2
    h_in = torch.from_numpy(bits.view(np.int16)).pin_memory()
    h_comp = [torch.empty(cap, dtype=torch.uint8).pin_memory() for _ in range(S)]
    h_out = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(S)]
    h_size = torch.zeros(S, dtype=torch.int64).pin_memory()
    d_in = [torch.empty(n, dtype=torch.int16, device=dev) for _ in range(S)]
    d_comp = [comp, torch.empty(cap, dtype=torch.uint8, device=dev)]
    d_size = [size, torch.zeros((), dtype=torch.int64, device=dev)]
    d_comp2 = [torch.empty(cap, dtype=torch.uint8, device=dev) for _ in range(S)]
    d_out = [out.view(torch.int16), torch.empty(n, dtype=torch.int16, device=dev)]
    d_status = [status, torch.zeros((), dtype=torch.int32, device=dev)]
    up, ks, down = torch.cuda.Stream(dev), stream, torch.cuda.Stream(dev)
    ev = [{k: torch.cuda.Event() for k in ("in", "comp", "cdn", "cup", "dec", "odn")} for _ in range(S)]
    tb = [0] * S

    def encode(k):  # input up, compress
        b, e = k % S, ev[k % S]
        if k >= S:
            up.wait_event(e["comp"])  # compression k - 2 has read d_in[b]
        with torch.cuda.stream(up):
            d_in[b].copy_(h_in, non_blocking=True)
        e["in"].record(up)
        ks.wait_event(e["in"])
        if k >= S:
            ks.wait_event(e["cdn"])  # container k - 2 has left d_comp[b]
        with torch.cuda.stream(ks):
            st = uz.uzip_compress(d_in[b].data_ptr(), uz.UZIP_BF16, n, d_comp[b].data_ptr(), cap,
                                  d_size[b].data_ptr(), ks.cuda_stream)
            h_size[b].copy_(d_size[b], non_blocking=True)
        e["comp"].record(ks)
        if st:
            raise RuntimeError(f"e2e compress status {st}")

    def container_down(k):  # the host reads the size, then the container goes down
        b, e = k % S, ev[k % S]
        e["comp"].synchronize()
        tb[b] = int(h_size[b])
        if tb[b] <= 0:
            raise RuntimeError("e2e compress failed")
        down.wait_event(e["comp"])
        if k >= S:
            down.wait_event(e["cup"])  # container k - 2 has left h_comp[b]
        with torch.cuda.stream(down):
            h_comp[b][:tb[b]].copy_(d_comp[b][:tb[b]], non_blocking=True)
        e["cdn"].record(down)

    def decode(k):  # container up, decompress
        b, e = k % S, ev[k % S]
        up.wait_event(e["cdn"])
        if k >= S:
            up.wait_event(e["dec"])  # decompression k - 2 has read d_comp2[b]
        with torch.cuda.stream(up):
            d_comp2[b][:tb[b]].copy_(h_comp[b][:tb[b]], non_blocking=True)
        e["cup"].record(up)
        ks.wait_event(e["cup"])
        if k >= S:
            ks.wait_event(e["odn"])  # output k - 2 has left d_out[b]
        with torch.cuda.stream(ks):
            st = uz.uzip_decompress(d_comp2[b].data_ptr(), tb[b], d_out[b].data_ptr(), uz.UZIP_BF16, n,
                                    d_status[b].data_ptr(), ks.cuda_stream)
        e["dec"].record(ks)
        if st:
            raise RuntimeError(f"e2e decompress status {st}")

    def output_down(k):
        b, e = k % S, ev[k % S]
        down.wait_event(e["dec"])
        with torch.cuda.stream(down):
            h_out[b].copy_(d_out[b], non_blocking=True)
        e["odn"].record(down)

    def pipelined(steps):
        # per period the uplink carries input k and container k - 1, the
        # downlink container k and output k - 1, in that order
        for k in range(steps + 1):
            if k < steps:
                encode(k)
            if k >= 1:
                decode(k - 1)
            if k < steps:
                container_down(k)
            if k >= 1:
                output_down(k - 1)
        torch.cuda.synchronize(dev)

    def serial():
        b = 0
        with torch.cuda.stream(ks):
            d_in[b].copy_(h_in, non_blocking=True)
            st = uz.uzip_compress(d_in[b].data_ptr(), uz.UZIP_BF16, n, d_comp[b].data_ptr(), cap,
                                  d_size[b].data_ptr(), ks.cuda_stream)
            h_size[b].copy_(d_size[b], non_blocking=True)
        ks.synchronize()
        t = int(h_size[b])
        with torch.cuda.stream(ks):
            h_comp[b][:t].copy_(d_comp[b][:t], non_blocking=True)
            d_comp2[b][:t].copy_(h_comp[b][:t], non_blocking=True)
            st2 = uz.uzip_decompress(d_comp2[b].data_ptr(), t, d_out[b].data_ptr(), uz.UZIP_BF16, n,
                                     d_status[b].data_ptr(), ks.cuda_stream)
            h_out[b].copy_(d_out[b], non_blocking=True)
        ks.synchronize()
        if st or st2:
            raise RuntimeError("e2e status")
        return t

    steps = max(2, min(args.steps, 10))
    pipelined(2)  # warm-up
    for h in h_out:
        h.zero_()
    t0 = time.perf_counter()
    pipelined(steps)
    dt = (time.perf_counter() - t0) / steps
    ok = all(bool(np.array_equal(h.numpy().view(np.uint16), bits)) for h in h_out)
    ok = ok and all(int(s_.item()) == 0 for s_ in d_status) and tb[0] == tb[1]
    serial()
    t0 = time.perf_counter()
    ts = 0
    for _ in range(3):
        ts = serial()
    dts = (time.perf_counter() - t0) / 3
    ok = ok and ts == tb[0] and bool(np.array_equal(h_out[0].numpy().view(np.uint16), bits))
    return {"value": 2 * n / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 2 * n + tb[0],
            "d2h_bytes_per_step": tb[0] + 2 * n + 8, "steps": steps, "bit_exact": ok,
            "schedule": "two-slot pipeline over steps: uploads, kernels and downloads on three streams",
            "serial_gbs": 2 * n / dts / 1e9}


def run_pipeline(args, dev):
    """Split-send pipeline (two streams, two device banks, two pinned host
    banks) over the whole c5 workload: the 15 messages of the 8,030,261,248
    bf16 Llama-3-8B-shaped parameter set (16.06 GB) go through each mode in
    one call, against a plain device-to-host copy of the same bytes; then a
    message-size sweep (64 KiB .. 1 GiB, prefixes of message 0) with the
    default threshold under which a message travels as a whole-message RAW
    container.  Modes: exact-size copy kernel into mapped pinned memory;
    exact-size cudaMemcpyAsync once the host has read the size; streamed copies
    of finished remainder and stream runs while the message compresses;
    bound-size cudaMemcpyAsync; compress-then-copy on one stream (no overlap).
    Host wall clock including the final synchronisation.  Returns the figures
    and the device copies of the messages."""
    import numpy as np
    import torch

    import lossless_float_tensor_gb300 as uz
    import synth

    sizes = synth.c5_message_sizes()
    t_gen = time.perf_counter()
    msgs = [torch.from_numpy(synth.c5_message(k).view(np.int16)).to(dev) for k in range(len(sizes))]
    t_gen = time.perf_counter() - t_gen
    n_max = max(sizes)
    cap = uz.uzip_max_compressed_size(uz.UZIP_BF16, n_max)
    banks = [torch.empty(cap, dtype=torch.uint8, device=dev) for _ in range(2)]
    hcap = cap + 16 * (-(-n_max // 65536))  # the streamed mode keeps progress words past the container
    hb = [torch.empty(hcap, dtype=torch.uint8).pin_memory() for _ in range(2)]
    s0, s1 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    modes = {"exact": uz.UZIP_PIPE_EXACT, "sized": uz.UZIP_PIPE_SIZED, "streamed": uz.UZIP_PIPE_STREAMED,
             "bound": uz.UZIP_PIPE_BOUND, "serial": uz.UZIP_PIPE_SERIAL}

    def send(ptrs, elems, mode, h_sizes, raw_below):
        for it in range(2):  # the first pass warms up
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            st = uz.uzip_pipeline_send_ex(uz.UZIP_BF16, ptrs, elems, [b.data_ptr() for b in banks], cap,
                                          [h.data_ptr() for h in hb], hcap, h_sizes.data_ptr(), mode, raw_below,
                                          s0.cuda_stream, s1.cuda_stream)
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
            if st != 0:
                raise RuntimeError(f"pipeline status {st}")
        return dt

    def raw_copy(views):
        for it in range(2):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            with torch.cuda.stream(s1):
                for k, v in enumerate(views):
                    hb[k & 1][: v.numel()].copy_(v, non_blocking=True)
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
        return dt

    total_bytes = 2 * sum(sizes)
    hs = torch.zeros(len(sizes), dtype=torch.int64).pin_memory()
    stream_row = {"messages": len(sizes), "input_bytes": total_bytes}
    for name, mode in modes.items():
        dt = send([m.data_ptr() for m in msgs], sizes, mode, hs, uz.UZIP_PIPE_RAW_BELOW_DEFAULT)
        stream_row[name + "_gbs"] = total_bytes / dt / 1e9
    stream_row["compressed_bytes"] = int(hs.sum())
    stream_row["ratio"] = int(hs.sum()) / total_bytes
    stream_row["raw_d2h_gbs"] = total_bytes / raw_copy([m.view(torch.uint8) for m in msgs]) / 1e9
    # message-size sweep on prefixes of message 0
    x = msgs[0]
    sweep = []
    for n in [1 << 15, 1 << 17, 1 << 19, 1 << 21, 1 << 23, 1 << 24, 1 << 25, 1 << 27, n_max]:
        reps = int(max(4, min(64, (4 << 30) // (2 * n))))
        hsw = torch.zeros(reps, dtype=torch.int64).pin_memory()
        row = {"message_bytes": 2 * n, "messages": reps,
               "raw_container": 2 * n < uz.UZIP_PIPE_RAW_BELOW_DEFAULT}
        for name in ("sized", "exact"):
            row[name + "_gbs"] = reps * 2 * n / send([x.data_ptr()] * reps, [n] * reps, modes[name], hsw,
                                                     uz.UZIP_PIPE_RAW_BELOW_DEFAULT) / 1e9
        row["sized_coded_gbs"] = reps * 2 * n / send([x.data_ptr()] * reps, [n] * reps, modes["sized"], hsw, 0) / 1e9
        row["raw_d2h_gbs"] = reps * 2 * n / raw_copy([x.view(torch.uint8)[: 2 * n]] * reps) / 1e9
        sweep.append(row)
    # one 1 GiB message, from the call to its last byte on the host
    latency = {}
    for name in ("sized", "streamed"):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            st = uz.uzip_pipeline_send(uz.UZIP_BF16, [x.data_ptr()], [n_max], [b.data_ptr() for b in banks], cap,
                                       [h.data_ptr() for h in hb], hcap, hs.data_ptr(), modes[name], s0.cuda_stream,
                                       s1.cuda_stream)
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
            if st != 0:
                raise RuntimeError(f"pipeline status {st}")
        latency[name + "_ms"] = best * 1e3
    del banks
    return {"workload": "c5: all 15 messages (8,030,261,248 bf16 values, 16.06 GB) of the Llama-3-8B-shaped "
                        "parameter set ~ N(0, 0.02), one call per mode; size sweep on prefixes of message 0",
            "unit": "GB/s (input bytes, host wall clock incl. sync)", "generation_s": t_gen,
            "raw_below_bytes_default": uz.UZIP_PIPE_RAW_BELOW_DEFAULT, "stream": stream_row, "sweep": sweep,
            "one_message_latency": latency}, msgs


def run_gate(args, dev, x, n, peak):
    """Whole-message choice (uzip_compress_gated): on the c4 tensor the 64 KiB
    sample codes, so the gated call costs the gate kernel on top of the usual
    compression; on 1 GiB of random bf16 bits the sample goes RAW and the
    whole message is split and stored RAW without statistics or coding.  Also
    the other table modes: tables from a sample of each chunk
    (UZIP_FLAG_SAMPLED_TABLES) and one Gaussian-model table for every chunk
    (uzip_compress_parametric), on c4 and on c5 message 0.  CUDA events, mean
    of 5 launches after 3 warm-ups."""
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

    def run_sampled(t):
        st = uz.uzip_compress_ex(t.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), None,
                                 uz.UZIP_FLAG_SAMPLED_TABLES, sp)
        if st:
            raise RuntimeError(f"uzip status {st}")

    rows["c4_sampled_tables_ms"] = timed(lambda: run_sampled(x))
    rows["c4_sampled_tables_bytes"] = int(size.item())
    del rnd

    def run_model(t, sigma):
        st = uz.uzip_compress_parametric(t.data_ptr(), uz.UZIP_BF16, n, comp.data_ptr(), cap, size.data_ptr(), None,
                                         sigma, sp)
        if st:
            raise RuntimeError(f"uzip status {st}")

    # Gaussian-model tables: c4 under its standard deviation (0.5 t(4):
    # 0.5 sqrt 2), and c5 message 0 (N(0, 0.02), which the model fits) in all
    # three table modes
    rows["c4_parametric_ms"] = timed(lambda: run_model(x, 0.5 * 2 ** 0.5))
    rows["c4_parametric_bytes"] = int(size.item())
    import synth

    m0 = synth.c5_message(0)
    if m0.size == n:
        g = torch.from_numpy(m0.view(np.int16)).to(dev)
        del m0
        rows["c5m0_full_ms"] = timed(lambda: run(g))
        rows["c5m0_full_bytes"] = int(size.item())
        rows["c5m0_sampled_tables_ms"] = timed(lambda: run_sampled(g))
        rows["c5m0_sampled_tables_bytes"] = int(size.item())
        rows["c5m0_parametric_ms"] = timed(lambda: run_model(g, 0.02))
        rows["c5m0_parametric_bytes"] = int(size.item())
        del g
    return {"workload": "c4 (1 GiB bf16), 1 GiB of random bf16 bits (numpy seed 17), c5 message 0 (1 GiB bf16)",
            "unit": "ms per launch", **rows}


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
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config table (c1, c2, c3, c5)")
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
