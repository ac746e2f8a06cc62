#!/usr/bin/env python
"""Benchmark of the GB300 ZipCCL BF16 exponent-coding hot path.

Workload (one step = every stage of the path once): the gradient bucket of
67,108,864 BF16 values from N(0, 1e-3^2) in 8 per-destination chunks is
compressed (scale select + encode with look-back offsets) and decompressed,
and 8 peer chunks of 8,388,608 values each (independently seeded, received
compressed) are decompressed and summed in fp32 into one BF16 shard.

Metric: GB/s of uncompressed BF16 through the step (2 bytes per value
compressed + 2 per value decompressed + 2 per peer value reduced) per second
of device time; the per-stage rates, the compression ratio and the dominant
kernel's fraction of the measured HBM bandwidth ride along.  Inputs are
resident in HBM when timing starts; L2 is flushed before every timed step
(a buffer twice its size written, then another read).
``e2e`` times the same step through the public API with pinned host buffers
and the host<->device copies inside the timed region.

``configs`` (same JSON line) times each workload on its own, compress and
decompress with L2 flushed before every call: PR1 (1,048,576 values from
N(0, 0.02^2), plus the round trip of all 65,536 BF16 patterns), the gradient
bucket, MoE dispatch (134,217,728 values in 64 expert chunks), the FSDP
all-gather stack (872,415,232 values in 224 row chunks) and the stress mix
(268,435,456 values in 256 chunks, every 16th incompressible).  Each entry
gives GB/s of uncompressed BF16, the algorithmic HBM fraction, bits per
value, the gap to the entropy bound and the oracle's rate on a stated prefix.

``--impl reference`` times the plain single-threaded CPU oracle on a bounded
sample of the same workload instead.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under
torchrun, each rank runs its own bucket (weak scaling, no collective: the
chunks are independent), and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compress/decompress GB/s (uncompressed bf16) and % of HBM roofline; compression ratio"
UNIT = "GB/s"
N_BUCKET = 67_108_864
RANKS = 8
PEER_N = 8_388_608
K_PEERS = 8
L2_FLUSH_BYTES = 2 * 129 * 1024 * 1024
KERNELS_PER_STEP = 6  # select, encode, decode-prep, decode, reduce-prep, reduce
# Every workload is also timed on its own (compress and decompress), after the headline step.
CONFIG_NAMES = ["pr1", "gradient", "moe", "fsdp", "stress"]
# Stage whose kernel the `roofline` object describes: the encode kernel of the compress call, the
# largest HBM mover of the step and the stage the 60% bandwidth bar is set on, timed on its own by
# events the library records around its launch.  Fixed, so that the named kernel does not change
# between runs with noise; every stage's whole-call fraction is in `stages`.
ROOFLINE_STAGE = "compress"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--configs", default=",".join(CONFIG_NAMES),
                   help="comma-separated workloads timed after the headline step ('none' for none)")
    return p.parse_args()


def workload_config(n_gpus: int) -> dict:
    return {
        "workload": "gradient bucket: 67,108,864 bf16 from N(0, 1e-3^2) in 8 per-destination chunks "
                    "(compress + decompress) + decompress_reduce of 8 peer chunks x 8,388,608 (fp32 sum, rank order)",
        "n_elems": N_BUCKET, "chunks": RANKS, "reduce_peers": K_PEERS, "reduce_elems": PEER_N,
        "parallelism": f"replicas x{n_gpus} (independent buckets, no collective)",
        "l2": L2_NOTE,
    }


class L2Flush:
    """Untimed, before each timed call: write a buffer twice the L2's size, then read
    another of the same size.  The L2 then holds none of the call's data, and the
    written lines are already back in HBM, so the timed call does not pay for
    writing back the flush's own dirty lines."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)

    def __call__(self, i: int = 0) -> None:
        self.w.fill_(i & 0xFF)
        self.torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


L2_NOTE = "flushed before every timed call: 258 MiB written, then 258 MiB read (no dirty lines left)"


def peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "src": "fallback"}


def sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lossless_bf16_tensor_zipccl_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on these sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("sources_sha") == sources_sha():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples go to BENCH_CLOCKS_DIR if set, else to a temporary directory
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # nvidia-smi takes a moment to start: the timed region begins once it samples
        self.wait_samples(1, 5.0)
        return self

    def lines(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for line in f if line.count(",") >= 8)
        except OSError:
            return 0

    def wait_samples(self, n: int, limit_s: float, work=None) -> None:
        """Until the record holds n samples (or limit_s passes), calling work() meanwhile."""
        if self.proc is None:
            return
        t0 = time.time()
        while self.lines() < n and time.time() - t0 < limit_s:
            if work is not None:
                work()
            else:
                time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ reference arm / CPU baseline
def oracle_sample(seed_offset: int = 0):
    """A bounded sample of the workload for the CPU oracle: one 8,388,608-value
    chunk of the bucket (compress + decompress) and the reduce of 8 peers over
    1,048,576 values each."""
    import oracle
    import workloads
    oracle.lib()
    x = workloads.gaussian_bf16(N_BUCKET // RANKS, 1e-3, 100 + seed_offset, 0)
    peers = [workloads.gaussian_bf16(1 << 20, 1e-3, 100 + seed_offset, 1000 + p) for p in range(K_PEERS)]
    peer_chunks = [oracle.compress(p)[0] for p in peers]
    return x, peer_chunks


def oracle_step(x, peer_chunks) -> float:
    import oracle
    t0 = time.perf_counter()
    s, offs = oracle.compress(x)
    oracle.decompress(s, offs, x.size)
    oracle.decompress_reduce(peer_chunks, 1 << 20)
    return time.perf_counter() - t0


def oracle_sample_bytes() -> int:
    return 2 * (N_BUCKET // RANKS) * 2 + 2 * K_PEERS * (1 << 20)


SAMPLE_DESC = ("oracle compress + decompress of one 8,388,608-value chunk of the bucket and decompress_reduce "
               "of 8 peers x 1,048,576 values; same distribution, GB/s of uncompressed bf16")


def host_info() -> dict:
    """The host's logical CPU count and CPU model (lscpu's model name, else /proc/cpuinfo)."""
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"host_cpus": os.cpu_count(), "cpu_model": model or "unknown", "machine": platform.machine()}


def cpu_baseline(repeats: int = 3) -> dict:
    x, pc = oracle_sample()
    ts = [oracle_step(x, pc) for _ in range(repeats)]
    t = statistics.median(ts)
    return {"value": oracle_sample_bytes() / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": SAMPLE_DESC + f"; median of {repeats}", **host_info()}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    x, pc = oracle_sample()
    for _ in range(args.warmup):
        oracle_step(x, pc)
    ts = [oracle_step(x, pc) for _ in range(args.steps)]
    total = sum(ts)
    value = oracle_sample_bytes() * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16/u8 (integer coding), f32 reduce",
        "data": "synthetic (seeded numpy PCG64)", "config": workload_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": SAMPLE_DESC,
                         **host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (the job's time) on every rank; identity at world 1."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Each rank compresses its own bucket (weak scaling)."""
    return 100 + 10007 * rank


# ------------------------------------------------------------------ our arm
def run_ours(args, rank: int, world: int):
    import torch

    import lossless_bf16_tensor_zipccl_gb300 as zc
    import workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    zc.load()
    seed = rank_seed(rank)
    wl = workloads.gradient(seed=seed)
    peers = workloads.gradient_peers(seed=seed)
    chunk_elems = wl.chunk_elems
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    # received peer chunks: each peer's chunk compressed on its own (prepared outside timing)
    peer_chunks = []
    for p in peers:
        c = zc.compress(torch.from_numpy(p.view(np.int16)).to(dev))
        peer_chunks.append(c.data[: c.nbytes()].clone())
    peer_bytes = [int(t.numel()) for t in peer_chunks]

    cap = zc.zipccl_max_compressed_bytes(chunk_elems)
    out = torch.empty(cap, dtype=torch.uint8, device=dev)
    offs = torch.empty(len(chunk_elems) + 1, dtype=torch.int64, device=dev)
    ws_c = torch.empty(zc.zipccl_compress_workspace_bytes(chunk_elems), dtype=torch.uint8, device=dev)
    ws_d = torch.empty(zc.zipccl_decompress_workspace_bytes(N_BUCKET, RANKS), dtype=torch.uint8, device=dev)
    ws_r = torch.empty(zc.zipccl_reduce_workspace_bytes(K_PEERS), dtype=torch.uint8, device=dev)
    dec = torch.empty(N_BUCKET, dtype=torch.int16, device=dev)
    red = torch.empty(PEER_N, dtype=torch.int16, device=dev)
    flush = L2Flush(torch, dev)

    def check(st, what):
        if st != zc.OK:
            raise zc.ZipcclError(st, what)

    def do_compress():
        check(zc.zipccl_compress(x.data_ptr(), N_BUCKET, chunk_elems, None, out.data_ptr(), cap, offs.data_ptr(),
                                 ws_c.data_ptr(), ws_c.numel(), sp), "compress")

    def do_decompress():
        check(zc.zipccl_decompress(out.data_ptr(), offs.data_ptr(), RANKS, dec.data_ptr(), N_BUCKET,
                                   ws_d.data_ptr(), ws_d.numel(), sp), "decompress")

    def do_reduce():
        check(zc.zipccl_decompress_reduce([t.data_ptr() for t in peer_chunks], peer_bytes, K_PEERS, PEER_N,
                                          red.data_ptr(), ws_r.data_ptr(), ws_r.numel(), sp), "reduce")

    stages = [("compress", do_compress), ("decompress", do_decompress), ("decompress_reduce", do_reduce)]
    for _ in range(args.warmup):
        for _, f in stages:
            f()
    torch.cuda.synchronize(dev)
    for ws in (ws_c, ws_d, ws_r):
        st = zc.zipccl_get_device_status(ws.data_ptr(), sp)
        if st != zc.OK:
            raise zc.ZipcclError(st, "device status after warm-up")
    if not torch.equal(dec, x):
        raise RuntimeError("round trip mismatch in the benchmark")
    comp_bytes = int(offs[-1].item())

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        # the sampler's start leaves the GPU idle for a moment: the warm-up
        # steps run again here, so that the timed steps follow them directly
        for _ in range(args.warmup):
            flush(0)
            for _, f in stages:
                f()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        n0 = clk.lines()
        for i in range(args.steps):
            flush(i)                       # untimed: L2 flush
            ev[i][0].record(stream)
            for j, (_, f) in enumerate(stages):
                f()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)

        def more_steps():  # untimed, the same work: the clock record brackets the timed region under load
            for _ in range(50):
                flush(0)
                for _, f in stages:
                    f()
            torch.cuda.synchronize(dev)

        clk.wait_samples(n0 + 2, 3.0, more_steps)
    if world > 1:
        torch.distributed.barrier()
    stage_ms = {name: [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)]
                for j, (name, _) in enumerate(stages)}

    # The encode kernel's own launch duration, in a loop of its own so that
    # the step above carries no instrumentation (recording the events adds a
    # few microseconds to the call outside the interval they bracket): the
    # library records them on the call's stream right before and after the
    # encode launch.
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in kev:
        a.record(stream)  # the event handles exist once recorded
        b.record(stream)
    for i in range(args.steps):
        flush(i)
        check(zc.zipccl_profile_encode_events(kev[i][0].cuda_event, kev[i][1].cuda_event), "profile events")
        do_compress()
    check(zc.zipccl_profile_encode_events(0, 0), "profile events off")
    torch.cuda.synchronize(dev)
    kernel_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in kev), world, dev) / args.steps
    step_ms = [sum(stage_ms[n][i] for n, _ in stages) for i in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)

    unc = {"compress": 2 * N_BUCKET, "decompress": 2 * N_BUCKET, "decompress_reduce": 2 * K_PEERS * PEER_N}
    algo = {"compress": 2 * N_BUCKET + comp_bytes, "decompress": comp_bytes + 2 * N_BUCKET,
            "decompress_reduce": sum(peer_bytes) + 2 * PEER_N}
    step_bytes = sum(unc.values())
    value = world * step_bytes * args.steps / (total_ms * 1e-3) / 1e9
    pk = peaks()
    stage_info = {}
    for name, _ in stages:
        ms = sum(stage_ms[name]) / args.steps
        stage_info[name] = {"ms": ms, "gbs_uncompressed": unc[name] / (ms * 1e-3) / 1e9,
                            "hbm_gbs_algorithmic": algo[name] / (ms * 1e-3) / 1e9,
                            "hbm_frac_of_measured": algo[name] / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    dom = ROOFLINE_STAGE
    kernel_of = {"compress": "zc_encode_kernel", "decompress": "zc_decode_kernel", "decompress_reduce": "zc_reduce_kernel"}
    ach = algo[dom] / (kernel_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, zc, torch, dev, wl, peer_chunks, peer_bytes, comp_bytes)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u16/u8 (integer coding), f32 reduce", "data": "synthetic (seeded numpy PCG64)",
        "config": workload_config(world),
        "compression_ratio": comp_bytes / (2 * N_BUCKET), "bits_per_value": 8 * comp_bytes / N_BUCKET,
        "stages": stage_info,
        "roofline": {"bound": "hbm", "kernel": kernel_of[dom], "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / pk["hbm_gbs"], "traffic": traffic_for(kernel_of[dom]),
                     "peak_src": pk["src"], "kernel_ms": kernel_ms,
                     "timing": "CUDA events the library records on the call's stream right before and after the "
                               "encode kernel launch (select kernel excluded; the cooperative launch's start-up "
                               "gap of ~3 us included), mean of a separate loop of compress calls, L2 flushed "
                               "before each; the whole call's fraction is stages.compress"},
        "clocks": clk.summary(),
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        line["send_pipeline"] = measure_send_overlap(args, zc, torch, dev, wl)
    names = [c for c in args.configs.split(",") if c and c != "none"]
    if rank == 0 and names:
        line["configs"] = measure_configs(args, zc, torch, dev, pk, names, cpu=world == 1 and not args.no_cpu_baseline,
                                         gradient_wl=wl)
    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        print(json.dumps(line), flush=True)


def gaussian_exponent_entropy(sigma: float) -> float:
    """Entropy (bits) of the biased BF16 exponent of X ~ N(0, sigma^2): binade e >= 1 holds
    2^(e-127) <= |X| < 2^(e-126), e = 0 holds |X| < 2^-126.  The bound the coded size is set
    against (8 raw sign/mantissa bits + this per value)."""
    import math
    s = sigma * math.sqrt(2.0)

    def mass(lo, hi):  # P(lo <= |X| < hi), from the side of the distribution with more precision
        a, b = lo / s, hi / s
        return math.erfc(a) - math.erfc(b) if a > 0.5 else math.erf(b) - math.erf(a)

    ps = [mass(0.0, 2.0 ** -126)] + [mass(2.0 ** (e - 127), 2.0 ** (e - 126)) for e in range(1, 255)]
    return -sum(p * math.log2(p) for p in ps if p > 0)


def empirical_bound_bits(x: np.ndarray, chunk_elems) -> float:
    """Sum over chunks of n_c * (8 + empirical entropy of the chunk's exponents), per value."""
    total, pos = 0.0, 0
    for m in chunk_elems:
        if m:
            cnt = np.bincount(((x[pos:pos + m] >> 7) & 0xFF).astype(np.uint8), minlength=256).astype(np.float64)
            p = cnt[cnt > 0] / m
            total += m * (8.0 - float((p * np.log2(p)).sum()))
        pos += m
    return total / max(1, pos)


CONFIG_SIGMA = {"pr1": 0.02, "gradient": 1e-3, "fsdp": 0.02}  # Gaussian workloads with one sigma
CPU_PREFIX_VALUES = 8 << 20


def config_workload(name: str, gradient_wl):
    import workloads
    if name == "gradient" and gradient_wl is not None:
        return gradient_wl
    return workloads.WORKLOADS[name]()


def chunk_prefix(wl, min_values: int, must_hold=None):
    """Leading whole chunks of a workload holding at least min_values values (and chunk must_hold)."""
    tot, k = 0, 0
    for k, m in enumerate(wl.chunk_elems, 1):
        tot += m
        if tot >= min_values and (must_hold is None or k > must_hold):
            break
    return wl.x[:tot], wl.chunk_elems[:k]


def cpu_config_baseline(name: str, wl, repeats: int = 3) -> dict:
    """The oracle's compress + decompress on a stated prefix of the workload."""
    import oracle
    oracle.lib()
    x, ce = chunk_prefix(wl, CPU_PREFIX_VALUES, must_hold=15 if name == "stress" else None)
    ts = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        s, offs = oracle.compress(x, ce)
        oracle.decompress(s, offs, x.size)
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts)
    return {"value": 4 * x.size / t / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"oracle compress + decompress of the first {len(ce)} chunks ({x.size:,} values); "
                      f"GB/s of uncompressed bf16 in and out; median of {repeats}"}


def measure_configs(args, zc, torch, dev, pk, names, cpu: bool, gradient_wl=None) -> dict:
    """Each workload compressed and decompressed on its own: median CUDA-event time of each call over
    the timed steps, L2 flushed before every call; GB/s of uncompressed BF16 (2 bytes a value),
    algorithmic HBM bytes (2 a value + the stream) over the measured copy bandwidth, bits per value,
    and the gap to the entropy bound."""
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    flush = L2Flush(torch, dev)
    res = {}
    for name in names:
        wl = config_workload(name, gradient_wl)
        n, ce = wl.n, wl.chunk_elems
        x = torch.from_numpy(wl.x.view(np.int16)).to(dev)
        cap = zc.zipccl_max_compressed_bytes(ce)
        out = torch.empty(cap, dtype=torch.uint8, device=dev)
        offs = torch.empty(len(ce) + 1, dtype=torch.int64, device=dev)
        ws_c = torch.empty(zc.zipccl_compress_workspace_bytes(ce), dtype=torch.uint8, device=dev)
        ws_d = torch.empty(zc.zipccl_decompress_workspace_bytes(n, len(ce)), dtype=torch.uint8, device=dev)
        dec = torch.empty(max(1, n), dtype=torch.int16, device=dev)

        def comp():
            st = zc.zipccl_compress(x.data_ptr(), n, ce, None, out.data_ptr(), cap, offs.data_ptr(),
                                    ws_c.data_ptr(), ws_c.numel(), sp)
            if st != zc.OK:
                raise zc.ZipcclError(st, f"{name} compress")

        def decomp():
            st = zc.zipccl_decompress(out.data_ptr(), offs.data_ptr(), len(ce), dec.data_ptr(), n,
                                      ws_d.data_ptr(), ws_d.numel(), sp)
            if st != zc.OK:
                raise zc.ZipcclError(st, f"{name} decompress")

        for _ in range(max(3, args.warmup)):
            comp()
            decomp()
        torch.cuda.synchronize(dev)
        for ws in (ws_c, ws_d):
            st = zc.zipccl_get_device_status(ws.data_ptr(), sp)
            if st != zc.OK:
                raise zc.ZipcclError(st, f"{name} device status")
        if not torch.equal(dec[:n], x):
            raise RuntimeError(f"{name}: round trip mismatch")
        comp_bytes = int(offs[-1].item())
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush(i)
            ev[i][0].record(stream)
            comp()
            ev[i][1].record(stream)
            flush(i + 1)
            ev[i][2].record(stream)
            decomp()
            ev[i][3].record(stream)
        torch.cuda.synchronize(dev)
        tc = statistics.median(ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps))
        td = statistics.median(ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps))
        algo = 2 * n + comp_bytes
        bits = 8.0 * comp_bytes / max(1, n)
        emp = empirical_bound_bits(wl.x, ce)
        e = {
            "workload": wl.note, "n_elems": n, "chunks": len(ce),
            "compress_us": 1e3 * tc, "decompress_us": 1e3 * td,
            "compress_gbs": 2 * n / (tc * 1e-3) / 1e9, "decompress_gbs": 2 * n / (td * 1e-3) / 1e9,
            "compress_hbm_frac_of_measured": algo / (tc * 1e-3) / 1e9 / pk["hbm_gbs"],
            "decompress_hbm_frac_of_measured": algo / (td * 1e-3) / 1e9 / pk["hbm_gbs"],
            "compressed_bytes": comp_bytes, "bits_per_value": bits, "compression_ratio": comp_bytes / max(1, 2 * n),
            "empirical_bound_bits": emp, "gap_to_empirical_bound": bits / emp - 1.0,
            "round_trip": "bit-exact",
            "l2": L2_NOTE + ("; the input is smaller than L2" if 2 * n < (129 << 20) else ""),
        }
        if name in CONFIG_SIGMA:
            hb = 8.0 + gaussian_exponent_entropy(CONFIG_SIGMA[name])
            e["closed_form_bound_bits"] = hb
            e["gap_to_closed_form_bound"] = bits / hb - 1.0
        if name == "stress":
            o = offs.cpu().numpy().view(np.uint64)
            raw = [c for c in range(len(ce)) if c % 16 == 15]
            e["incompressible_chunk_expansion_max"] = max(float(o[c + 1] - o[c]) / (2 * ce[c]) for c in raw)
            e["worst_case_bound_ratio"] = cap / (2 * n)
        if name == "pr1":
            e["all_patterns_round_trip"] = all_patterns_round_trip(zc, torch, dev)
        if cpu:
            e["cpu_baseline"] = {**cpu_config_baseline(name, wl), **host_info()}
        res[name] = e
        del x, out, offs, ws_c, ws_d, dec
        torch.cuda.empty_cache()
    return res


def measure_send_overlap(args, zc, torch, dev, wl) -> dict:
    """Compress-and-send on the gradient bucket: the fused call (every tile stored to the
    output and to a send buffer from shared memory, each chunk posted as soon as its tiles
    are stored) against the compress call followed by a device-to-device copy of the whole
    stream into the send buffer.  Median CUDA-event times over the timed steps, L2 flushed
    before each; plus, from one more call, when each chunk was posted after the kernel began."""
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ce = wl.chunk_elems
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev)
    cap = zc.zipccl_max_compressed_bytes(ce)
    out = torch.empty(cap, dtype=torch.uint8, device=dev)
    send = torch.empty(cap, dtype=torch.uint8, device=dev)
    offs = torch.empty(len(ce) + 1, dtype=torch.int64, device=dev)
    ws = torch.empty(zc.zipccl_compress_workspace_bytes(ce), dtype=torch.uint8, device=dev)
    flush = L2Flush(torch, dev)

    def comp():
        st = zc.zipccl_compress(x.data_ptr(), x.numel(), ce, None, out.data_ptr(), cap, offs.data_ptr(),
                                ws.data_ptr(), ws.numel(), sp)
        if st != zc.OK:
            raise zc.ZipcclError(st, "compress")

    ready = torch.zeros(len(ce) + 1, dtype=torch.int64, device=dev)

    def comp_send():
        st = zc.zipccl_compress_send(x.data_ptr(), x.numel(), ce, None, out.data_ptr(), cap, offs.data_ptr(),
                                     send.data_ptr(), cap, ready.data_ptr(), ws.data_ptr(), ws.numel(), sp)
        if st != zc.OK:
            raise zc.ZipcclError(st, "compress_send")

    comp()
    torch.cuda.synchronize(dev)
    total = int(offs[-1].item())

    def copy():
        send[:total].copy_(out[:total])

    variants = {"compress_then_copy": lambda: (comp(), copy()), "compress_send": comp_send, "copy_alone": copy}
    for _ in range(max(3, args.warmup)):
        for f in variants.values():
            f()
    torch.cuda.synchronize(dev)
    if zc.zipccl_get_device_status(ws.data_ptr(), sp) != zc.OK:
        raise RuntimeError("compress_send: device status")
    send.zero_()
    flush(0)
    comp_send()
    torch.cuda.synchronize(dev)
    if not torch.equal(send[:total], out[:total]):
        raise RuntimeError("compress_send: the send buffer differs from the stream")
    r = ready.cpu().numpy()
    posted_us = [round((int(v) - int(r[-1])) / 1e3, 2) for v in r[:-1]]
    times = {k: [] for k in variants}
    for i in range(args.steps):
        for k, f in variants.items():
            flush(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            times[k].append((e0, e1))
    torch.cuda.synchronize(dev)
    med = {k: statistics.median(a.elapsed_time(b) for a, b in v) * 1e3 for k, v in times.items()}
    return {"workload": "gradient bucket, 8 chunks", "stream_bytes": total,
            "compress_then_copy_us": med["compress_then_copy"], "compress_send_us": med["compress_send"],
            "copy_alone_us": med["copy_alone"],
            "saved_us": med["compress_then_copy"] - med["compress_send"],
            "copy_hidden_fraction": (med["compress_then_copy"] - med["compress_send"]) / med["copy_alone"],
            "chunk_posted_us_after_kernel_start": posted_us,
            "l2": L2_NOTE}


def all_patterns_round_trip(zc, torch, dev) -> str:
    import workloads
    w = workloads.all_patterns()
    x = torch.from_numpy(w.x.view(np.int16)).to(dev)
    y = zc.decompress(zc.compress(x))
    torch.cuda.synchronize(dev)
    if not torch.equal(y.view(torch.int16), x):
        raise RuntimeError("all 65,536 BF16 patterns: round trip mismatch")
    return "bit-exact (all 65,536 patterns)"


def measure_e2e(args, zc, torch, dev, wl, peer_chunks, peer_bytes, comp_bytes):
    """Same step through the torch-level public API, inputs copied in from
    pinned host memory and results read back every step.  Steps are pipelined
    as a user would run them: host-to-device copies, the three calls and the
    device-to-host copies go on three streams, with two buffer sets, so the
    copies of one step overlap the compute of the next."""
    nbuf = 2
    h_x = torch.from_numpy(wl.x.view(np.int16)).pin_memory()
    h_peers = [t.cpu().pin_memory() for t in peer_chunks]
    cap = zc.zipccl_max_compressed_bytes(wl.chunk_elems)
    sets = []
    for _ in range(nbuf):
        sets.append({
            "d_x": torch.empty(N_BUCKET, dtype=torch.int16, device=dev),
            "d_peers": [torch.empty_like(t, device=dev) for t in h_peers],
            "d_out": torch.empty(cap, dtype=torch.uint8, device=dev),
            "d_offs": torch.empty(RANKS + 1, dtype=torch.int64, device=dev),
            "d_dec": torch.empty(N_BUCKET, dtype=torch.bfloat16, device=dev),
            "d_red": torch.empty(PEER_N, dtype=torch.bfloat16, device=dev),
            "ws_c": torch.empty(zc.zipccl_compress_workspace_bytes(wl.chunk_elems), dtype=torch.uint8, device=dev),
            "ws_d": torch.empty(zc.zipccl_decompress_workspace_bytes(N_BUCKET, RANKS), dtype=torch.uint8, device=dev),
            "ws_r": torch.empty(zc.zipccl_reduce_workspace_bytes(K_PEERS), dtype=torch.uint8, device=dev),
            "h_stream": torch.empty(comp_bytes, dtype=torch.uint8).pin_memory(),
            "h_offs": torch.empty(RANKS + 1, dtype=torch.int64).pin_memory(),
            "h_dec": torch.empty(N_BUCKET, dtype=torch.int16).pin_memory(),
            "h_red": torch.empty(PEER_N, dtype=torch.int16).pin_memory(),
            "in_ready": torch.cuda.Event(), "done": torch.cuda.Event(), "out_read": torch.cuda.Event(),
        })
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    for b in sets:  # nothing pending yet
        b["done"].record(s_run)
        b["out_read"].record(s_out)

    def step(i):
        b = sets[i % nbuf]
        with torch.cuda.stream(s_in):
            s_in.wait_event(b["done"])  # the previous step on this set has read its inputs
            b["d_x"].copy_(h_x, non_blocking=True)
            for d, h in zip(b["d_peers"], h_peers):
                d.copy_(h, non_blocking=True)
            b["in_ready"].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(b["in_ready"])
            s_run.wait_event(b["out_read"])  # its outputs have been copied out
            c = zc.compress(b["d_x"], wl.chunk_elems, out=b["d_out"], offsets=b["d_offs"], ws=b["ws_c"],
                            stream=s_run)
            zc.decompress(c, out=b["d_dec"], ws=b["ws_d"], stream=s_run)
            zc.decompress_reduce(b["d_peers"], PEER_N, out=b["d_red"], ws=b["ws_r"], stream=s_run)
            b["done"].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["done"])
            b["h_offs"].copy_(b["d_offs"], non_blocking=True)
            b["h_stream"].copy_(b["d_out"][:comp_bytes], non_blocking=True)
            b["h_dec"].copy_(b["d_dec"].view(torch.int16), non_blocking=True)
            b["h_red"].copy_(b["d_red"].view(torch.int16), non_blocking=True)
            b["out_read"].record(s_out)

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_in.wait_stream(s_out)  # the timed region starts with every earlier step finished
    for i in range(args.steps):
        step(i)
    s_out.wait_stream(s_run)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    last = sets[(args.steps - 1) % nbuf]
    if int(last["h_offs"][-1]) != comp_bytes or not torch.equal(last["h_dec"], h_x):
        raise RuntimeError("e2e round trip mismatch")
    h2d = 2 * N_BUCKET + sum(peer_bytes)
    d2h = comp_bytes + 8 * (RANKS + 1) + 2 * N_BUCKET + 2 * PEER_N
    step_bytes = 2 * N_BUCKET + 2 * N_BUCKET + 2 * K_PEERS * PEER_N
    return {"value": step_bytes / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "two buffer sets; H2D, compute and D2H on three streams"}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
