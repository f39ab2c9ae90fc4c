#!/usr/bin/env python3
"""Benchmark: split-K GEMM + reduce, BF16 M=256 N=1024 K=2048, 2 splits.

One "step" is one pack of 8 complete operations (partial pass + accumulation),
the pages' pack=8 mode ("Aligned shared rows for pipelined NAX on CUDA",
section "Measurement protocol": device events over a captured complete-
operation graph, weights prepared and resident, preparation outside timing).
Each operation of a step works on its own seeded instance (A, B, out,
workspace), drawn from a pool of 40 instances whose inputs (200 MB) exceed the
129 MB L2, so every operation reads its operands from HBM.

Printed (one JSON line, rank 0): value = microseconds per operation (lower is
better), the roofline of the dominant kernel measured live with CUDA events,
the end-to-end figure through the C ABI with host buffers (gemm_bt_host_batch:
activations in and results out every step, pipelined), the clocks
seen during the timed region, and the CPU oracle's time for the same work.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--mode fused|two_pass] [--pack 8] [--pool 40]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M, N, K, SPLITS, KPS = 256, 1024, 2048, 2, 1024
DTYPE = "bf16"
WORKLOAD = "BF16 split-K GEMM M=256 N=1024 K=2048 splits=2 (k_per_split=1024) + reduce"
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal
METRIC = BASE_METRIC = "split-K GEMM+reduce µs/op & TFLOP/s, % of roofline (BF16 M256/N1024/K2048)"
FLOPS_PER_OP = 2 * M * N * K
BYTES_2PASS = M * K * 2 + N * K * 2 + 2 * SPLITS * M * N * 4 + M * N * 4   # A+B, P write+read, out
BYTES_FUSED = M * K * 2 + N * K * 2 + M * N * 4                             # A+B, out
BYTES_GEMM = M * K * 2 + N * K * 2 + SPLITS * M * N * 4                     # A+B, P write
BYTES_REDUCE = SPLITS * M * N * 4 + M * N * 4                               # P read, out write


def code_of(text: str) -> str:
    """C/C++/CUDA source without its comments and blank lines (string and
    character literals kept as they are), so that a comment-only edit leaves
    the traffic record valid."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                       # a literal, escapes included
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_traffic(ops_per_launch=1):
    """DRAM bytes per launch of the tensor-core kernel from the committed ncu
    record, or None when the kernel's code changed since it was taken (the
    record's sources without comments, each up to the record's end-of-device-
    code marker where it has one) or the record's launches computed another
    number of operations."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "tc_splitk_traffic.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                rec[k.strip()] = v.strip()
    h = hashlib.sha256()
    cut = rec.get("device_code_ends_at", "")
    constants_only = set(rec.get("constants_only", "").split())
    for src in rec.get("sources", "").split():
        with open(os.path.join(ROOT, src)) as f:
            text = code_of(f.read())
        if cut and cut in text:   # the device code only: the host planner below may change
            text = text[:text.index(cut)]
        if src in constants_only:  # a host header: only the constants the kernel is built from
            text = "\n".join(line for line in text.splitlines() if line.startswith("constexpr"))
        h.update(text.encode())
    if h.hexdigest() != rec.get("code_sha256") or int(rec.get("ops_per_launch", 1)) != ops_per_launch:
        return None
    return int(rec["dram_bytes_per_launch"])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


# Nominal dense tensor rates of a GB300 (PFLOP/s): BF16/F16 2.25, TF32 1.1.  F32
# operands run as three TF32 products each, so their tensor term is the BF16
# measured peak x 1.1 / 2.25 / 3 per useful FLOP.
TF32_OVER_BF16 = 1.1 / 2.25


def op_roofline(M_, N_, K_, S_, dt, hbm_gbs, bf16_tflops):
    """Roofline times (us) of one operation: the slower of its FLOPs at the
    tensor peak for its element type and its bytes at the HBM bandwidth, for
    the two-pass bytes (A, B, partials written and read, output) and for the
    fused kernel's minimal bytes (A, B, output)."""
    e = 4 if dt == "f32" else 2
    flops = 2 * M_ * N_ * K_
    peak = bf16_tflops * (TF32_OVER_BF16 / 3 if dt == "f32" else 1.0)
    t_flop = flops / (peak * 1e12) * 1e6
    b2 = M_ * K_ * e + N_ * K_ * e + 2 * S_ * M_ * N_ * 4 + M_ * N_ * 4
    bmin = M_ * K_ * e + N_ * K_ * e + M_ * N_ * 4
    t2, tmin = b2 / (hbm_gbs * 1e9) * 1e6, bmin / (hbm_gbs * 1e9) * 1e6
    return {"flops": flops, "bytes_2pass": b2, "bytes_min": bmin, "tensor_peak_tflops": round(peak, 1),
            "t_flop_us": round(t_flop, 4), "t_roof_us_2pass": round(max(t_flop, t2), 4),
            "t_roof_us_min": round(max(t_flop, tmin), 4),
            "bound_2pass": "tensor" if t_flop > t2 else "hbm", "bound_min": "tensor" if t_flop > tmin else "hbm"}


# The pages' workloads beside the headline: the M96 and M256/N512 shapes, the
# single tile, and the dtype x split sweep over the skinny and short-K shapes
# with the short-final-split case ("Wider consecutive-weight NAX GEMM",
# section "Performance method"; "Aligned shared rows for pipelined NAX on
# CUDA", section "Measurement protocol").
CONFIGS = [("bf16", 32, 64, 128, 2, 64), ("bf16", 96, 512, 2048, 4, 512), ("bf16", 256, 512, 2048, 4, 512)]
for _dt in ("bf16", "f16", "f32"):
    for _S in (1, 2, 4, 8, 16):
        CONFIGS.append((_dt, 32, 512, 2048, _S, 2048 // _S))
        CONFIGS.append((_dt, 96, 512, 512, _S, 512 // _S))
    CONFIGS.append((_dt, 64, 128, 160, 3, 64))


def measure_configs(sk, torch, stream, dev, hbm, tflops, pool_bytes=160 << 20, max_inst=128):
    """Per workload: fused and two-kernel us per operation (graphs of 8 calls,
    CUDA events), TFLOP/s and the roofline fractions.  Each workload cycles a
    pool of seeded instances of at least `pool_bytes` of A + B where
    `max_inst` instances reach that (else the pool is L2-resident, and the
    entry says so).  The fused and two-kernel outputs of one instance must be
    equal bit for bit."""
    import numpy as np

    import splitk_inputs as gen

    res = []
    for dt, M_, N_, K_, S_, kps_ in CONFIGS:
        e = 4 if dt == "f32" else 2
        ab = (M_ * K_ + N_ * K_) * e
        n = max(8, min(max_inst, -(-pool_bytes // ab)))
        n -= n % 8
        nb = sk.gemm_bt_workspace_bytes(M_, N_, K_, S_, kps_)
        pool = []
        for i in range(n):
            ops = gen.uniform(M_, N_, K_, dt, seed=i)
            if dt == "f32":
                A_ = torch.from_numpy(np.ascontiguousarray(ops.A, np.float32)).to(dev)
                B_ = torch.from_numpy(np.ascontiguousarray(ops.B, np.float32)).to(dev)
            else:
                tdt = torch.bfloat16 if dt == "bf16" else torch.float16
                A_ = torch.from_numpy(ops.A.view(np.int16)).to(dev).view(tdt)
                B_ = torch.from_numpy(ops.B.view(np.int16)).to(dev).view(tdt)
            pool.append((A_, B_, torch.empty((M_, N_), dtype=torch.float32, device=dev),
                         torch.empty((nb // 4,), dtype=torch.float32, device=dev)))
        groups = [pool[g * 8:(g + 1) * 8] for g in range(n // 8)]
        entry = {"workload": f"{dt.upper()} M{M_} N{N_} K{K_} splits={S_} (k_per_split={kps_})",
                 "instances": n, "pool_mb": round(n * ab / 1e6, 1),
                 "l2": "cold (pool larger than L2)" if n * ab > 129e6 else "warm (pool fits in L2)"}
        plan = sk.splitk_describe_launch(M_, N_, K_, S_, kps_, dt, fused=1)
        entry["fused_in_kernel"] = plan["fused_in_kernel"]
        for fused, key in ((1, "fused_us"), (0, "two_pass_us")):
            graphs = [capture(torch, stream, lambda grp=grp, f=fused: [
                sk.gemm_bt(a, b, o, w, nb, M_, N_, K_, S_, kps_, dt, fused=f, stream=stream) for a, b, o, w in grp])
                for grp in groups]
            time_graphs(torch, stream, graphs, max(3, len(graphs)))
            reps = max(len(graphs), 40)
            entry[key] = round(min(time_graphs(torch, stream, graphs, reps) for _ in range(3)) * 1e3 / (reps * 8), 4)
        a, b, o, w = pool[0]
        sk.gemm_bt(a, b, o, w, nb, M_, N_, K_, S_, kps_, dt, fused=0, stream=stream)
        torch.cuda.synchronize()
        ref = o.clone()
        sk.gemm_bt(a, b, o, w, nb, M_, N_, K_, S_, kps_, dt, fused=1, stream=stream)
        torch.cuda.synchronize()
        entry["fused_bitwise_two_pass"] = bool(torch.equal(ref.view(torch.int32), o.view(torch.int32)))
        r = op_roofline(M_, N_, K_, S_, dt, hbm, tflops)
        entry["tflops_fused"] = round(r["flops"] / (entry["fused_us"] * 1e-6) / 1e12, 2)
        entry["frac_min_bytes_fused"] = round(r["t_roof_us_min"] / entry["fused_us"], 4)
        entry["frac_2pass_fused"] = round(r["t_roof_us_2pass"] / entry["fused_us"], 4)
        entry["frac_2pass_two_pass"] = round(r["t_roof_us_2pass"] / entry["two_pass_us"], 4)
        entry["roofline"] = r
        res.append(entry)
        del pool, groups
    if sk.splitk_get_device_status(stream) != 0:
        raise RuntimeError("a kernel's bounded wait ran out during the per-workload runs")
    return res


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock and throttle reasons through NVML during a region."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.period = period_s
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
                self.max_mhz = mx.value
            self.nv, self.h, self.ok = nv, h, True
        except OSError:
            pass

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


# ----------------------------------------------------------------- CPU oracle

class OracleSample:
    """The oracle's evaluation (every partial slab, plus the unsplit output and
    its bounds) of `rows` output rows of the workload.  The work is linear in
    the rows, so its time scales to one whole operation by M/rows."""

    def __init__(self, rows: int = 32, threads=None):
        import oracle
        import splitk_inputs as gen

        self.oracle = oracle
        ops = gen.uniform(M, N, K, DTYPE, seed=0)
        self.A = ops.A[:rows].copy()
        self.B = ops.B
        self.rows = rows
        self.threads = threads or max(1, len(os.sched_getaffinity(0)))
        self.cores = min(self.threads, rows)

    def once(self) -> float:
        """Seconds for one sample."""
        t0 = time.perf_counter()
        self.oracle.partials(self.A, self.B, DTYPE, K, SPLITS, KPS, threads=self.threads)
        self.oracle.output(self.A, self.B, DTYPE, threads=self.threads)
        return time.perf_counter() - t0

    def us_per_op(self, seconds: float) -> float:
        return seconds * (M / self.rows) * 1e6

    def describe(self, reps: int) -> str:
        return (f"{self.rows} of {M} output rows (all {N} columns, all of K), {reps} repetition(s) of "
                f"the oracle's partials + unsplit output, scaled by {M}/{self.rows}")


def oracle_rows_timing(seconds: float, rows: int = 32, threads=None):
    smp = OracleSample(rows, threads)
    smp.once()   # warm-up
    reps, total = 0, 0.0
    while total < seconds or reps == 0:
        total += smp.once()
        reps += 1
    return smp.us_per_op(total / reps), smp.cores, smp.describe(reps)


def nvml_index(torch, dev) -> int:
    """NVML index of the CUDA device (matched by PCI bus id when possible)."""
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        nv.nvmlInit_v2()
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0:
            idx = ctypes.c_uint()
            if nv.nvmlDeviceGetIndex(h, ctypes.byref(idx)) == 0:
                return idx.value
    except (OSError, AttributeError):
        pass
    return 0


# ----------------------------------------------------------------- GPU arm

def make_pool(torch, n_inst, dev):
    import numpy as np

    import splitk_inputs as gen

    pool = []
    for i in range(n_inst):
        ops = gen.uniform(M, N, K, DTYPE, seed=i)
        A = torch.from_numpy(ops.A.view(np.int16)).to(dev).view(torch.bfloat16)
        B = torch.from_numpy(ops.B.view(np.int16)).to(dev).view(torch.bfloat16)
        pool.append({"A_host": torch.from_numpy(ops.A.view(np.int16)).view(torch.bfloat16),
                     "A_bits": ops.A, "B_bits": ops.B,
                     "A": A, "B": B,
                     "out": torch.empty((M, N), dtype=torch.float32, device=dev),
                     "ws": torch.empty((SPLITS * M * N,), dtype=torch.float32, device=dev)})
    return pool


TOL_BF16_FINAL = 2e-2   # the pages' final tolerance for BF16, times sum |a*b|


def f64_check(insts, rows_per=8, seed=0):
    """Sampled rows of each instance's output against an F64 product of its
    BF16 operands (decoded from the same bits), as max |out - ref| / sum|ab|;
    rows whose sum|ab| is 0 (the zero first row of A) must be exactly 0.
    Returns (worst scaled error, outputs checked)."""
    import numpy as np

    def f64(bits):
        return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    rng = np.random.default_rng(seed)
    worst, count = 0.0, 0
    for inst in insts:
        rows = sorted({0, 1, M // 2, M - 1, *rng.integers(0, M, rows_per - 4).tolist()})
        a = f64(inst["A_bits"].reshape(M, K)[rows])
        b = f64(inst["B_bits"].reshape(N, K))
        ref, bound = a @ b.T, np.abs(a) @ np.abs(b).T
        got = inst["out"][rows].cpu().numpy().astype(np.float64)
        err = np.abs(got - ref)
        zero = bound == 0
        if not np.all(np.isfinite(err)) or np.any(err[zero] != 0):
            return float("inf"), count + got.size
        worst = max(worst, float(np.max(err[~zero] / bound[~zero])))
        count += got.size
    return worst, count


def job_time(ms_local, steps, pack, world, dist=None, device="cpu"):
    """The job's timed region is the slowest rank's (max over ranks); the
    value is microseconds per operation over every rank's operations (each
    rank runs `steps` steps of `pack` independent operations: weak scaling).
    Returns (ms, us_per_op)."""
    ms = float(ms_local)
    if dist is not None and world > 1:
        import torch

        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, ms * 1e3 / (steps * pack * world)


def capture(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_graphs(torch, stream, graphs, steps):
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for k in range(steps):
            graphs[k % len(graphs)].replay()
        stop.record(stream)
    stop.synchronize()
    return start.elapsed_time(stop)   # ms


def measure_e2e(sk, torch, stream, groups, pack, fused, steps):
    """µs/op through gemm_bt_host_batch: per step one group's `pack`
    activations come from pinned host memory and its results go back to
    pinned host memory, all inside the timed region.  Steps alternate two
    staging buffers and two caller streams (each call joins its stream), so
    that a step's kernels need not wait for the previous step's copy out;
    the CUDA events bracket both streams.  Also times the same batches on one
    stream with one copy each way (no overlap of copies and kernels) and the
    host's enqueue time per call."""
    import time

    dev = groups[0][0]["A"].device
    hosts = []
    for grp in groups:
        a = torch.cat([inst["A_host"].reshape(-1) for inst in grp]).pin_memory()
        o = torch.empty((pack * M * N,), dtype=torch.float32).pin_memory()
        hosts.append((a, o, sk.pointer_array([inst["B"] for inst in grp])))
    sb = sk.gemm_bt_host_staging_bytes(pack, M, N, K, SPLITS, KPS, DTYPE)
    # two staging buffers, alternated: a step's activations come in while
    # the previous step computes
    stagings = [torch.empty((sb // 4,), dtype=torch.float32, device=dev) for _ in range(2)]
    for st in stagings:
        sk.gemm_bt_workspace_init(st, sb, stream=stream)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, min(steps, 200))
    second = torch.cuda.Stream(device=dev)

    def run(opc, nstreams):
        streams = [stream, second][:nstreams]
        host_s = 0.0
        for k in range(3):
            a, o, b = hosts[k % len(hosts)]
            sk.gemm_bt_host_batch(a, b, o, pack, stagings[k % 2], sb, M, N, K, SPLITS, KPS, DTYPE,
                                  fused=fused, ops_per_copy=opc, stream=streams[k % nstreams])
        torch.cuda.synchronize()
        start.record(stream)
        second.wait_event(start)
        for k in range(n):
            a, o, b = hosts[k % len(hosts)]
            t0 = time.perf_counter()
            sk.gemm_bt_host_batch(a, b, o, pack, stagings[k % 2], sb, M, N, K, SPLITS, KPS, DTYPE,
                                  fused=fused, ops_per_copy=opc, stream=streams[k % nstreams])
            host_s += time.perf_counter() - t0
        stream.wait_stream(second)
        stop.record(stream)
        stop.synchronize()
        return start.elapsed_time(stop) * 1e3 / (n * pack), host_s * 1e6 / n

    us, host_us = run(0, 2)
    # the step just timed ended on group (n-1) % len(groups): its host results
    # must equal the resident-operand outputs of the same operations
    last = (n - 1) % len(groups)
    for i, inst in enumerate(groups[last]):
        got = hosts[last][1][i * M * N:(i + 1) * M * N].view(M, N)
        if not torch.equal(got, inst["out"].cpu()):
            raise RuntimeError("host-buffer results differ from the resident-operand outputs")
    one_stream_us, _ = run(0, 1)
    serial_us, _ = run(pack, 1)
    if sk.splitk_get_device_status(stream) != 0:
        raise RuntimeError("a kernel's bounded wait ran out during the end-to-end run")
    return {"value": round(us, 4), "unit": "µs/op", "h2d_bytes_per_step": pack * M * K * 2,
            "d2h_bytes_per_step": pack * M * N * 4,
            "how": f"gemm_bt_host_batch per step: {pack} activations copied in from pinned host memory and "
                   "results copied out to pinned host memory on two copy streams, pipelined against the "
                   "kernels (the operations of a copy group in one launch), two staging buffers and two "
                   "caller streams alternated so that a step's copy in and its kernels overlap the previous "
                   f"step's copy out; weights resident; CUDA events around both streams over {n} steps",
            "one_stream_us": round(one_stream_us, 4),
            "unpipelined": "one stream, one copy each way for the whole step (no overlap of copies and kernels)",
            "unpipelined_us": round(serial_us, 4), "host_enqueue_us_per_step": round(host_us, 2)}


def run_ours(args, rank, world, dev, torch, dist):
    import split_bf16_gemm_gb300 as sk

    sk.build()
    sk.lib()
    pack = args.pack
    n_inst = max(args.pool, pack)
    n_inst -= n_inst % pack
    pool = make_pool(torch, n_inst, dev)
    nbytes = sk.gemm_bt_workspace_bytes(M, N, K, SPLITS, KPS)
    for inst in pool:
        inst["ws"] = torch.empty((nbytes // 4,), dtype=torch.float32, device=dev)
        sk.gemm_bt_workspace_init(inst["ws"], nbytes)
    fused = 1 if args.mode == "fused" else 0
    plan = sk.splitk_describe_launch(M, N, K, SPLITS, KPS, DTYPE, fused=fused)
    stream = torch.cuda.Stream(device=dev)
    groups = [pool[g * pack:(g + 1) * pack] for g in range(n_inst // pack)]

    def op(inst):
        sk.gemm_bt(inst["A"], inst["B"], inst["out"], inst["ws"], nbytes, M, N, K, SPLITS, KPS,
                   DTYPE, fused=fused, stream=stream)

    def gemm_only(inst):
        sk.gemm_splitk_bt(inst["A"], inst["B"], inst["ws"], M, N, K, SPLITS, KPS, DTYPE, stream=stream)

    def reduce_only(inst):
        sk.splitk_reduce(inst["ws"], inst["out"], SPLITS, M, N, stream=stream)

    torch.cuda.synchronize()
    # each call's tensor-core launch as captured: a call that starts a launch
    # reports group 1, one that joins the launch before it a larger group
    joined = []

    def op_recorded(inst):
        op(inst)
        joined.append(sk.splitk_last_launch()["group"])

    graphs = [capture(torch, stream, lambda grp=grp: [op_recorded(i) for i in grp]) for grp in groups]
    # the operations the last captured launch computes: a step's calls join
    # one launch where they can (group), so a launch is a whole step
    ops_per_launch = joined[-1]
    # kernels one step launches: the tensor-core launches the step's calls
    # started, plus a reduce per call where the splits are summed apart
    tc_per_step = sum(1 for g in joined[-pack:] if g == 1)
    launches_per_step = tc_per_step + (pack if plan["kernels_per_call"] == 2 else 0)

    # sanity before timing: the fused and two-kernel paths agree bitwise
    inst = pool[0]
    sk.gemm_bt(inst["A"], inst["B"], inst["out"], inst["ws"], nbytes, M, N, K, SPLITS, KPS, DTYPE,
               fused=0, stream=stream)
    torch.cuda.synchronize()
    ref = inst["out"].clone()
    sk.gemm_bt(inst["A"], inst["B"], inst["out"], inst["ws"], nbytes, M, N, K, SPLITS, KPS, DTYPE,
               fused=1, stream=stream)
    torch.cuda.synchronize()
    if not torch.equal(ref, inst["out"]):
        raise RuntimeError("fused and two-kernel outputs differ")

    time_graphs(torch, stream, graphs, max(args.warmup, 3, len(graphs)))
    torch.cuda.synchronize()
    # F64 checks of sampled outputs right before and right after the timed
    # region: two instances of every group of the pool
    checked = [grp[j] for grp in groups for j in (0, len(grp) - 1)]
    before = f64_check(checked)
    if not before[0] <= TOL_BF16_FINAL:
        raise RuntimeError(f"outputs before timing fail the F64 check: {before[0]:.3e}")
    for inst in checked:   # poisoned, so that the check after timing sees the timed region's results
        inst["out"].fill_(float("nan"))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(nvml_index(torch, dev)) as clocks:
        ms = time_graphs(torch, stream, graphs, args.steps)
    torch.cuda.synchronize()
    ms, us_per_op = job_time(ms, args.steps, pack, world, dist, dev)
    if sk.splitk_get_device_status(stream) != 0:
        raise RuntimeError("a kernel's bounded wait ran out during the timed region")
    ran = {id(i) for grp in groups[:min(args.steps, len(groups))] for i in grp}
    after = f64_check([i for i in checked if id(i) in ran], seed=1)
    if not after[0] <= TOL_BF16_FINAL:
        raise RuntimeError(f"outputs after timing fail the F64 check: {after[0]:.3e}")
    ms_per_step = ms / args.steps

    if args.profile:
        return {"metric": METRIC, "value": round(us_per_op, 4), "unit": "µs/op", "profile_run": True,
                "mode": args.mode, "plan": plan}

    # dominant kernel(s), timed alone over the same pool
    # the pages' sampling protocol beside the contract's single timed region:
    # 9 rounds of 40 replays of the same graphs, the median round; and pack=1
    # (one operation per replay, over the same pool)
    round_us = []
    with ClockSampler(nvml_index(torch, dev), period_s=0.0005) as round_clocks:
        for _ in range(9):
            round_us.append(time_graphs(torch, stream, graphs, 40) * 1e3 / (40 * pack))
    single = [capture(torch, stream, lambda i=i: op(i)) for i in pool]
    time_graphs(torch, stream, single, 10)
    pack1_us = time_graphs(torch, stream, single, 400) * 1e3 / 400
    gemm_graphs = [capture(torch, stream, lambda grp=grp: [gemm_only(i) for i in grp]) for grp in groups]
    red_graphs = [capture(torch, stream, lambda grp=grp: [reduce_only(i) for i in grp]) for grp in groups]
    reps = max(args.steps, 50)
    time_graphs(torch, stream, gemm_graphs, 5)
    gemm_us = time_graphs(torch, stream, gemm_graphs, reps) * 1e3 / (reps * pack)
    time_graphs(torch, stream, red_graphs, 5)
    red_us = time_graphs(torch, stream, red_graphs, reps) * 1e3 / (reps * pack)
    two_pass_graphs = [capture(torch, stream, lambda grp=grp: [(gemm_only(i), reduce_only(i)) for i in grp])
                       for grp in groups]
    time_graphs(torch, stream, two_pass_graphs, 5)
    two_pass_us = time_graphs(torch, stream, two_pass_graphs, reps) * 1e3 / (reps * pack)
    if fused:
        dom_name = f"tc_splitk_kernel (fused: partials + split sum; {ops_per_launch} operations per launch)"
        dom_us, dom_bytes = us_per_op * world * ops_per_launch, BYTES_FUSED * ops_per_launch
    else:
        dom_name, dom_us, dom_bytes = "tc_splitk_kernel (partial pass)", gemm_us, BYTES_GEMM

    # end to end through the C ABI with HOST buffers: every step copies its
    # operations' activations in from pinned host memory and their results
    # out to pinned host memory (gemm_bt_host_batch), weights resident
    e2e = measure_e2e(sk, torch, stream, groups, pack, fused, args.steps)

    # the same operations reading the weight in its [K,N] layout (gemm_kn):
    # W = B^T, made on the device with the preparation kernel (B^T of an
    # [N,K] matrix), so every operation has its own resident W
    for inst in pool:
        inst["W"] = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
        sk.splitk_prepare_bt(inst["B"], inst["W"], N, K, DTYPE, stream=stream)
    torch.cuda.synchronize()

    def op_kn(inst, f):
        sk.gemm_kn(inst["A"], inst["W"], inst["out"], inst["ws"], nbytes, M, N, K, SPLITS, KPS, DTYPE,
                   fused=f, stream=stream)

    kn_us = {}
    for f, name in ((1, "fused_op"), (0, "two_pass_op")):
        kg = [capture(torch, stream, lambda grp=grp, f=f: [op_kn(i, f) for i in grp]) for grp in groups]
        time_graphs(torch, stream, kg, 5)
        kn_us[name] = round(time_graphs(torch, stream, kg, reps) * 1e3 / (reps * pack), 4)
    ref = pool[0]["out"].clone()
    op(pool[0])
    torch.cuda.synchronize()
    if not torch.equal(ref, pool[0]["out"]):
        raise RuntimeError("the [K,N] and [N,K] weight layouts give different outputs")
    for inst in pool:
        del inst["W"]

    # the same operations eagerly (no graph): one gemm_bt call each, or a
    # step's calls as one gemm_bt_batch call (grouped launches)
    ptrs = [tuple(sk.pointer_array([i[k] for i in grp]) for k in ("A", "B", "out")) for grp in groups]
    eager_us = {}
    for name in ("calls", "batch"):
        def eager_step(g):
            if name == "batch":
                sk.gemm_bt_batch(*ptrs[g], pack, pool[0]["ws"], nbytes, M, N, K, SPLITS, KPS, DTYPE, fused=fused,
                                 stream=stream)
            else:
                for inst in groups[g]:
                    op(inst)
        for g in range(len(groups)):
            eager_step(g)
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for r in range(reps):
                eager_step(r % len(groups))
            stop.record(stream)
        stop.synchronize()
        eager_us[name] = round(start.elapsed_time(stop) * 1e3 / (reps * pack), 4)

    # weight preparation (B = W^T), a one-shot cost outside the operation
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prep_n = 24
    Ws = [torch.empty((K, N), dtype=torch.bfloat16, device=dev).normal_() for _ in range(prep_n)]
    Bs = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for _ in range(prep_n)]
    for i in range(prep_n):
        sk.splitk_prepare_bt(Ws[i], Bs[i], K, N, DTYPE, stream=stream)
    torch.cuda.synchronize()
    # replayed from a CUDA graph (as the operation is), so that the host's
    # launch rate does not set the figure
    prep_graph = capture(torch, stream, lambda: [sk.splitk_prepare_bt(Ws[i], Bs[i], K, N, DTYPE, stream=stream)
                                                 for i in range(prep_n)])
    prep_graph.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for r in range(4):
            prep_graph.replay()
        stop.record(stream)
    stop.synchronize()
    prep_us = start.elapsed_time(stop) * 1e3 / (4 * prep_n)
    if not torch.equal(Bs[0], Ws[0].t().contiguous()):
        raise RuntimeError("weight preparation result differs from the transpose")
    del Ws, Bs

    hbm, tflops, peak_kind = load_peaks()
    # the same fused graphs with every launch waiting for the one before (the
    # overlap of independent launches inside a capture turned off)
    sk.splitk_set_overlap(False)
    strict_graphs = [capture(torch, stream, lambda grp=grp: [op(i) for i in grp]) for grp in groups]
    sk.splitk_set_overlap(True)
    time_graphs(torch, stream, strict_graphs, 5)
    strict_us = time_graphs(torch, stream, strict_graphs, reps) * 1e3 / (reps * pack)
    configs = measure_configs(sk, torch, stream, dev, hbm, tflops) if args.configs else None
    roof = op_roofline(M, N, K, SPLITS, DTYPE, hbm, tflops)
    achieved = dom_bytes / (dom_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(us_per_op, 4), "unit": "µs/op", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded uniform[-1,1], zero first A row, x4 last A row)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "splits": SPLITS,
                   "k_per_split": KPS, "mode": args.mode, "ops_per_step": pack,
                   "instances": n_inst,
                   "l2": f"inputs larger than L2: {n_inst} distinct instances, "
                         f"{n_inst * (M * K + N * K) * 2 / 1e6:.0f} MB of A+B, cycled",
                   "timing": "CUDA graph per step, CUDA events on the launching stream",
                   "launches_per_step": launches_per_step,
                   "plan": plan},
        "tflops": round(FLOPS_PER_OP / (us_per_op * 1e-6) / 1e12 / 1, 2),
        "op_roofline": {
            "what": "the slower of the FLOPs at the measured dense BF16 peak and the bytes at the measured "
                    "HBM bandwidth, for the two-pass bytes and for the fused kernel's minimal bytes",
            "t_flop_us": roof["t_flop_us"], "bound": roof["bound_2pass"],
            "t_roof_us_2pass_bytes": roof["t_roof_us_2pass"],
            "frac_2pass_bytes": round(roof["t_roof_us_2pass"] / us_per_op, 4),
            "t_roof_us_min_bytes": roof["t_roof_us_min"],
            "frac_min_bytes": round(roof["t_roof_us_min"] / us_per_op, 4),
            "peak": f"{peak_kind} {hbm} GB/s",
            # against the nominal HBM3e bandwidth as well
            "nominal_gbs": NOMINAL_HBM_GBS,
            "frac_2pass_bytes_nominal": round(BYTES_2PASS / (NOMINAL_HBM_GBS * 1e9) * 1e6 / us_per_op, 4),
            "frac_min_bytes_nominal": round(BYTES_FUSED / (NOMINAL_HBM_GBS * 1e9) * 1e6 / us_per_op, 4)},
        "roofline": {"bound": roof["bound_min"] if fused else roof["bound_2pass"], "kernel": dom_name,
                     "t_flop_us": roof["t_flop_us"], "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": kernel_traffic(ops_per_launch) if fused else None, "bytes_per_launch": dom_bytes,
                     "ops_per_launch": ops_per_launch if fused else 1,
                     "launch_us": round(dom_us, 4), "peak_kind": peak_kind},
        "sampling": {"median_of_9_rounds_x_40_replays_us": round(statistics.median(round_us), 4),
                     "rounds_min_max_us": [round(min(round_us), 4), round(max(round_us), 4)],
                     "pack1_us": round(pack1_us, 4),
                     "pack1": "one operation per graph replay, the pool's instances in turn (each replay "
                              "pays a graph launch; no dependent-launch overlap across replays)",
                     "clocks": round_clocks.summary()},
        "kernels_us": {"partial_pass": round(gemm_us, 4), "reduce": round(red_us, 4),
                       "two_pass_op": round(two_pass_us, 4),
                       "fused_op" if fused else "two_pass_op_graph": round(us_per_op * world, 4),
                       "fused_op_every_launch_waits": round(strict_us, 4)},
        "overlap": "inside each captured graph, a call whose operands no running launch writes loads "
                   "before the previous launch ends and waits only before its first store, or (nothing "
                   "in flight touching its outputs either) stores at once and has one block wait before "
                   "the grid finishes; kernels_us.fused_op_every_launch_waits is the same graphs with "
                   "that turned off",
        "e2e": e2e,
        "eager": {"what": "the same operations outside a graph: one gemm_bt per operation (every launch waits "
                           "for the one before), or each step's 8 as one gemm_bt_batch call", "us": eager_us},
        "kn_layout": {"what": "the same operations with the weight in its [K,N] layout (gemm_kn, MN-major B)",
                      "us": kn_us},
        "prepare": {"what": "weight preparation B[N,K] = W[K,N]^T (one-shot, outside the operation); "
                            "24 distinct weights per CUDA graph, replayed 4 times",
                    "us": round(prep_us, 3), "bytes": 2 * K * N * 2,
                    "achieved_gbs": round(2 * K * N * 2 / (prep_us * 1e-6) / 1e9, 1),
                    "frac_of_hbm": round(2 * K * N * 2 / (prep_us * 1e-6) / 1e9 / hbm, 4)},
        "checks": {"reference": "F64 product of the BF16 operands (numpy, from the same bits), sampled rows of "
                                "two instances per group, max |out - ref| / sum|a*b|",
                   "tolerance": TOL_BF16_FINAL,
                   "before_timing": {"outputs": before[1], "max_scaled_err": float(f"{before[0]:.3e}")},
                   "after_timing": {"outputs": after[1], "max_scaled_err": float(f"{after[0]:.3e}")}},
        "configs": configs,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(),
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["fused", "two_pass"], default="fused")
    ap.add_argument("--pack", type=int, default=8)
    ap.add_argument("--pool", type=int, default=40)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the per-workload measurements of the pages' other shapes")
    ap.add_argument("--profile", action="store_true",
                    help="short run for ncu: the timed graphs only, no secondary timings, no CPU leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # The reference arm is the oracle, timed on the host cores; rank 0 only.
        if rank != 0:
            return
        smp = OracleSample()
        for _ in range(args.warmup):
            smp.once()
        us_list = [smp.us_per_op(smp.once()) for _ in range(args.steps)]
        cores, sample = smp.cores, smp.describe(1)
        us = statistics.mean(us_list)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(us, 2), "unit": "µs/op",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us * 32 / M / 1e3, 4), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "splits": SPLITS,
                       "k_per_split": KPS},
            "cpu_baseline": {"value": round(us, 2), "unit": "µs/op", "cores": cores,
                             "kind": "oracle", "sample": "per step: " + sample},
            "e2e": {"value": round(us, 2), "unit": "µs/op", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    import torch

    dist = None
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
        dist = tdist
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    line = run_ours(args, rank, world, dev, torch, dist)
    if rank == 0 and world == 1 and not args.profile:
        us, cores, sample = oracle_rows_timing(args.cpu_seconds)
        # the same oracle on one core
        us1, _, sample1 = oracle_rows_timing(args.cpu_seconds / 3, threads=1)
        line["cpu_baseline"] = {"value": round(us, 2), "unit": "µs/op", "cores": cores,
                                "kind": "oracle", "sample": sample,
                                "single_thread": {"value": round(us1, 2), "unit": "µs/op", "cores": 1,
                                                  "sample": sample1}}
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
