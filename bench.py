#!/usr/bin/env python
"""Throughput bench of the MLX-affine quantized row product (GB/s of HBM).

A step is one pass of the hot path over its workload; the default workload is
the one-row 4096 x 4096 width sweep (every bits in {2,3,4,5,6,8} x group in
{32,64,128}: 18 products a step).  Inputs are resident in HBM when the timed
region starts; every product reads a different copy of its weights in turn so
that a buffer is reused only after several L2 sizes of other traffic.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded column sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

GATHER_EXPERTS, GATHER_N, GATHER_K = 8, 2048, 2048
METRIC = "achieved HBM GB/s (and % of GB300 peak) of quantized GEMV per bits/group/rows"
L2_BYTES = 129 * 2 ** 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def workload_cases(name: str):
    """[(label, N, K, bits, group, seed, rows)] of a workload."""
    if name == "sweep":
        return [("%d/%d" % (b, g), 4096, 4096, b, g, s, 1) for (b, g, s) in synth.width_sweep_cases()]
    if name == "lmhead":
        return [("lmhead %d/%d r%d" % (b, g, r), synth.LMHEAD_N, synth.LMHEAD_K, b, g, s, r)
                for (b, g, s) in synth.LMHEAD_CASES for r in (1,)]
    if name == "lmhead16":
        return [("lmhead %d/%d r16" % (b, g), synth.LMHEAD_N, synth.LMHEAD_K, b, g, s, 16)
                for (b, g, s) in synth.LMHEAD_CASES]
    if name == "stack":   # the members (the GPU arm runs them as one fused stack per row count)
        return [("stack member %d/%d r%d" % (m.bits, m.group, r), m.n_cols, synth.STACK_K, m.bits, m.group, m.seed, r)
                for r in synth.STACK_ROWS for m in synth.STACK_MEMBERS]
    if name == "gather":   # the expert matrices (the GPU arm runs one gather call per step)
        return [("gather expert %d" % e, GATHER_N, GATHER_K, 4, 64, 150 + e, 2) for e in range(GATHER_EXPERTS)]
    if name == "options":
        return [("decode 12288x2048 r%d %s" % (r, o), 12288, 2048, 6, 32, 19, r)
                for r in (1, 16) for o in ("fp32", "bf16+relu2")]
    if name == "decode":
        return [("decode %dx%d r%d" % (N, K, r), N, K, 6, 32, s, r)
                for (N, K, s) in synth.DECODE_SHAPES for r in synth.DECODE_ROWS]
    if name == "prompt":   # tf_qmm_prompt: 64-row windows on the tensor cores
        return ([("prompt lmhead %d/%d r64" % (b, g), synth.LMHEAD_N, synth.LMHEAD_K, b, g, s, 64)
                 for (b, g, s) in synth.LMHEAD_CASES]
                + [("prompt %dx%d r64" % (N, K), N, K, 6, 32, s, 64) for (N, K, s) in synth.DECODE_SHAPES])
    raise SystemExit("unknown workload " + name)


WORKLOAD_TEXT = {
    "sweep": "width sweep: N=K=4096, 1 bf16 row, bits {2,3,4,5,6,8} x group {32,64,128} (18 GEMVs a step)",
    "lmhead": "LM head: N=248320, K=2048, 1 row, 6-bit g32 and 4-bit g64 (2 GEMVs a step)",
    "lmhead16": "LM head: N=248320, K=2048, 16 rows, 6-bit g32 and 4-bit g64 (2 GEMVs a step)",
    "stack": "fused mixed-width stack, K=2048: members 4/g64 4096, 5/g128 2048, 5/g128 48, 6/g64 48 "
             "widened to a 5-bit g64 run of 6192 columns and a 6-bit g64 run of 48, one tf_qmm_stack "
             "into a 6240-column strided output; rows 1 and 16 (2 stacks a step)",
    "gather": "expert gather: 16 slots over 8 experts of 2048 x 2048, 4-bit g64, two slots an expert "
              "(one tf_qmm_gather a step)",
    "options": "decode 12288 x 2048 6-bit g32, rows 1 and 16: fp32 output and bf16 output with the "
               "squared-ReLU epilogue (tf_qmm_ex)",
    "decode": "decode windows: 6-bit g32, 12288x2048 and 2048x12288, rows {1,2,3,8,16} (10 GEMVs a step)",
    "prompt": "prompt windows (tf_qmm_prompt, 64 rows): the LM head 6-bit g32 and 4-bit g64, and 6-bit g32 "
              "12288x2048 and 2048x12288 (4 products a step)",
}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            import tempfile
            self.path = os.path.join(tempfile.gettempdir(), "tfqmm_clocks_%d.csv" % os.getpid())
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


_CPU_INPUTS = {}


def cpu_sample(cases, cols_per_case: int, nthreads: int):
    """Time the oracle on `cols_per_case` columns of every case; (GB/s, seconds, desc)."""
    import oracle
    total_bytes, t_total = 0, 0.0
    for (label, N, K, bits, group, seed, rows) in cases:
        key = (N, K, bits, group, seed, rows)
        if key not in _CPU_INPUTS:            # generated once, outside the timing
            _CPU_INPUTS[key] = (synth.make_matrix(min(N, 4096), K, bits, group, seed, 0.001, 0.03),
                                synth.make_x(rows, K, seed))
        m, x = _CPU_INPUTS[key]
        cols = np.arange(min(cols_per_case, m.N), dtype=np.int64)
        t0 = time.perf_counter()
        oracle.qmm(x, m.W, m.scales, m.biases, m.N, K, bits, group, cols=cols, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        total_bytes += len(cols) * (K * bits // 8 + (K // group) * 4 + rows * 4) + rows * K * 2
    return total_bytes / t_total / 1e9, t_total, total_bytes


def max_over_ranks(v: float, dev) -> float:
    """The slowest rank's time (each rank times its own replica); v unchanged on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: int, world: int, ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time (weak scaling)."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def run_reference(args, cases):
    import oracle
    oracle.build()
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    cols = 64                                 # output columns of each product per step
    for _ in range(args.warmup):
        cpu_sample(cases, cols, cores)
    gbs_list, secs, nbytes = [], 0.0, 0
    for _ in range(args.steps):
        g, t, b = cpu_sample(cases, cols, cores)
        gbs_list.append(g)
        secs += t
        nbytes += b
    value = nbytes / secs / 1e9
    sample = "fp64 oracle, the first %d output columns of each of the %d products per step" % (cols, len(cases))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_TEXT[args.workload], "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def stack_items(cases, dev, tf):
    """One fused stack per row count: members 0-2 widened on the device to a
    5-bit g64 run of 6192 columns, member 3 a 6-bit g64 run of 48 columns,
    written through the member column map into one 6240-column output."""
    import torch
    K = synth.STACK_K
    mats = synth.stack_member_matrices()

    def to_dev(a, dt):
        return torch.from_numpy(a.view(dt)).to(dev)

    parts = []
    for m in mats[:3]:
        Wo = torch.zeros((m.N, K * 5 // 32), dtype=torch.int32, device=dev)
        so = torch.zeros((m.N, K // 64), dtype=torch.int16, device=dev)
        bo = torch.zeros_like(so)
        tf.tf_widen(to_dev(m.W, np.int32), to_dev(m.scales, np.int16), to_dev(m.biases, np.int16),
                    m.N, K, m.bits, m.group, Wo, so, bo, 5, 64)
        parts.append((Wo, so, bo))
    W5 = torch.cat([q[0] for q in parts]).contiguous()
    s5 = torch.cat([q[1] for q in parts]).contiguous()
    b5 = torch.cat([q[2] for q in parts]).contiguous()
    m6 = mats[3]
    runs = ((W5, s5, b5, 6192, 5, 64),
            (to_dev(m6.W, np.int32), to_dev(m6.scales, np.int16), to_dev(m6.biases, np.int16), 48, 6, 64))
    members = [(0, 0, 4096, 0), (0, 4096, 2048, 4096), (0, 6144, 48, 6144), (1, 0, 48, 6192)]
    stride = 6240
    items, per_step = [], 0
    for rows in synth.STACK_ROWS:
        nb = (synth.algorithmic_bytes(6192, K, 5, 64, rows) + synth.algorithmic_bytes(48, K, 6, 64, rows)
              - rows * K * 2)                          # x is read once
        x_h = synth.make_x(rows, K, 60 + rows)

        def grow(it, copies):
            it["reps"] += [tuple((W.clone(), sc.clone(), bc.clone(), N, b, g) for (W, sc, bc, N, b, g) in it["reps"][0])
                           for _ in range(copies - 1)]

        offs = [0, 4096, 6144, 6192]                   # member columns in the output
        items.append(dict(label="stack r%d" % rows, N=stride, K=K, rows=rows, stack=True, members=members,
                          reps=[runs], x=torch.from_numpy(x_h.view(np.int16)).to(dev),
                          y=torch.empty((rows, stride), dtype=torch.float32, device=dev),
                          x_pin=torch.from_numpy(x_h.view(np.int16)).pin_memory(),
                          y_pin=torch.empty((rows, stride), dtype=torch.float32).pin_memory(), bytes=nb,
                          check=[(m, x_h, o) for m, o in zip(mats, offs)]))
        items[-1]["grow"] = lambda copies, it=items[-1]: grow(it, copies)
        per_step += nb
    torch.cuda.synchronize()
    return items, per_step


def _dev_matrix(m, dev):
    import torch
    return (torch.from_numpy(m.W.view(np.int32)).to(dev), torch.from_numpy(m.scales.view(np.int16)).to(dev),
            torch.from_numpy(m.biases.view(np.int16)).to(dev))


def _io_item(label, rows, K, N, nbytes, dev, out_dtype, call, grow):
    import torch
    x_h = synth.make_x(rows, K, 150)
    it = dict(label=label, N=N, K=K, rows=rows, bytes=nbytes, reps=[None],
              x=torch.from_numpy(x_h.view(np.int16)).to(dev), x_pin=torch.from_numpy(x_h.view(np.int16)).pin_memory(),
              y=torch.empty((rows, N), dtype=out_dtype, device=dev),
              y_pin=torch.empty((rows, N), dtype=out_dtype).pin_memory())
    it["call"] = lambda c, st: call(it, c, st)
    it["grow"] = lambda copies: grow(it, copies)
    return it


def gather_items(cases, dev, tf):
    """One tf_qmm_gather a step: 16 slots (x rows 0..15) over 8 expert matrices, two slots an expert."""
    import torch
    mats = [synth.make_matrix(N, K, b, g, s, 0.001, 0.03) for (_, N, K, b, g, s, _) in cases]
    base = [_dev_matrix(m, dev) for m in mats]
    n_slots = 2 * len(mats)
    se = [i % len(mats) for i in range(n_slots)]
    sr = list(range(n_slots))
    K = GATHER_K
    nb = sum(synth.algorithmic_bytes(m.N, K, m.bits, m.group, 2) - 2 * K * 2 for m in mats) + n_slots * K * 2

    def call(it, c, st):
        ex = [(W, s_, b_, GATHER_N, 4, 64) for (W, s_, b_) in it["reps"][c % len(it["reps"])]]
        tf.tf_qmm_gather(it["x"], n_slots, K, ex, se, sr, it["y"], GATHER_N, 0, st)

    def grow(it, copies):
        it["reps"] = [base] + [[tuple(t.clone() for t in e) for e in base] for _ in range(copies - 1)]

    it = _io_item("gather 16 slots / 8 experts", n_slots, K, GATHER_N, nb, dev, torch.float32, call, grow)
    it["launches"] = len(mats)
    return [it], nb


def options_items(cases, dev, tf):
    """tf_qmm_ex on the 12288 x 2048 decode shape: fp32 output, and bf16 output with relu2."""
    import torch
    m = synth.make_matrix(12288, 2048, 6, 32, 19, 0.001, 0.03)
    base = _dev_matrix(m, dev)
    items, per_step = [], 0
    for (label, N, K, bits, group, seed, rows) in cases:
        flags = 0 if label.endswith("fp32") else tf.TF_OUT_BF16 | tf.TF_EPI_RELU2
        out_bytes = 4 if flags == 0 else 2
        nb = synth.algorithmic_bytes(N, K, bits, group, rows) - rows * N * 4 + rows * N * out_bytes

        def call(it, c, st, flags=flags):
            W, s_, b_ = it["reps"][c % len(it["reps"])]
            tf.tf_qmm_ex(it["x"], it["rows"], K, W, s_, b_, N, bits, group, it["y"], N, flags, st)

        def grow(it, copies):
            it["reps"] = [base] + [tuple(t.clone() for t in base) for _ in range(copies - 1)]

        items.append(_io_item(label, rows, K, N, nb, dev, torch.float32 if flags == 0 else torch.int16, call, grow))
        per_step += nb
    return items, per_step


def kernel_source_sha() -> str:
    """SHA-256 (16 hex digits) of the library's CUDA sources and headers: a
    committed traffic figure counts only for the source it was captured on."""
    import glob
    import hashlib
    h = hashlib.sha256()
    pat = [os.path.join(ROOT, "mlx_affine_bit_gb300", "csrc", e) for e in ("*.cu", "*.cuh", "*.h")]
    for f in sorted(sum((glob.glob(x) for x in pat), [])):
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """(bytes per step, note) from profiles/traffic_<workload>.txt, or (None, why)."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.txt" % workload)
    if not os.path.exists(path):
        return None, "no ncu capture of this workload is committed"
    vals = {}
    for line in open(path):
        f = line.split()
        if len(f) == 2 and not line.startswith("#"):
            vals[f[0]] = f[1]
    if vals.get("kernel_source_sha") != kernel_source_sha():
        return None, "the committed ncu capture predates the current kernel source"
    return int(vals["dram_bytes_per_step"]), "ncu dram__bytes_read.sum + dram__bytes_write.sum, " + \
        vals.get("captured", "date not recorded")


def _host_matrix(N, K, bits, group, seed):
    return synth.make_matrix(N, K, bits, group, seed, 0.001, 0.03 if N < 100000 else 0.02)


def product_items(cases, dev, min_bytes):
    """Device inputs of one tf_qmm per case; each case rotates over enough weight
    copies that a buffer is reused only after `min_bytes` of other traffic."""
    import torch
    items = []
    for (label, N, K, bits, group, seed, rows) in cases:
        m = _host_matrix(N, K, bits, group, seed)
        W = torch.from_numpy(m.W.view(np.int32)).to(dev)
        s = torch.from_numpy(m.scales.view(np.int16)).to(dev)
        b = torch.from_numpy(m.biases.view(np.int16)).to(dev)
        nb = synth.algorithmic_bytes(N, K, bits, group, rows)
        pc = max(1, -(-min_bytes // nb))
        reps = [(W, s, b)] + [(W.clone(), s.clone(), b.clone()) for _ in range(pc - 1)]
        x_h = synth.make_x(rows, K, seed)
        items.append(dict(label=label, N=N, K=K, bits=bits, group=group, rows=rows, reps=reps,
                          x=torch.from_numpy(x_h.view(np.int16)).to(dev),
                          y=torch.empty((rows, N), dtype=torch.float32, device=dev),
                          x_pin=torch.from_numpy(x_h.view(np.int16)).pin_memory(),
                          y_pin=torch.empty((rows, N), dtype=torch.float32).pin_memory(), bytes=nb,
                          check=[(m, x_h, 0)]))
    return items


def launch_item(tf, it, c, st):
    """Launch copy c of an item on stream st (one product, stack, gather or options call)."""
    if "call" in it:
        it["call"](c, st)
        return
    if it.get("stack"):
        tf.tf_qmm_stack(it["x"], it["rows"], it["K"], it["reps"][c % len(it["reps"])], it["members"],
                        it["y"], it["N"], st)
        return
    W, s, b = it["reps"][c % len(it["reps"])]
    tf.tf_qmm(it["x"], it["rows"], it["K"], W, s, b, it["N"], it["bits"], it["group"], it["y"], it["N"], st)


def item_launches(it) -> int:
    """Kernel launches of one call of the item."""
    return it.get("launches", len(it["reps"][0]) if it.get("stack") else 1)


def time_item(tf, it, stream, warmup, replays=7, min_calls=8):
    """Per-call device time (us): a CUDA graph of calls cycling over every weight
    copy (>= 4 L2 sizes of weights, and at least `min_calls` calls so that the
    graph's own start is spread thin), replayed `replays` times, each replay
    timed with CUDA events on the replay stream; the median over replays of
    time / calls."""
    import torch
    n = max(len(it["reps"]), min_calls)
    with torch.cuda.stream(stream):
        for w in range(max(1, warmup)):
            launch_item(tf, it, w, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in range(n):
            launch_item(tf, it, c, stream)
    torch.cuda.synchronize()
    per = []
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(replays):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            per.append((e0, e1))
    torch.cuda.synchronize()
    del g
    return statistics.median(e0.elapsed_time(e1) * 1e3 / n for e0, e1 in per)


def case_row(label, nbytes, us, peak):
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"case": label, "bytes": nbytes, "median_us": round(us, 3), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "frac_of_8tbs": round(gbs / 8000.0, 4)}


# Target configurations timed in every default run beside the headline sweep.
EXTRA_WORKLOADS = ("lmhead", "lmhead16", "decode", "stack", "prompt")


def prompt_items(cases, dev, tf, min_bytes):
    """tf_qmm_prompt calls: the product items, each call one x prepass, one launch
    per 64-row window and, when the chunks are split over work items, one fold."""
    import torch
    items = product_items(cases, dev, min_bytes)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    for it in items:
        def call(c, st, it=it):
            W, s, b = it["reps"][c % len(it["reps"])]
            tf.tf_qmm_prompt(it["x"], it["rows"], it["K"], W, s, b, it["N"], it["bits"], it["group"], it["y"],
                             it["N"], 0, st)
        it["call"] = call
        windows = -(-it["rows"] // 64)
        ntiles, nchunks = -(-it["N"] // 128), it["K"] // 2048
        split = ntiles < nsm and nchunks > 1
        it["launches"] = 1 + windows * (2 if split else 1)
    return items


def build_items(workload, cases, dev, tf, min_bytes):
    if workload == "prompt":
        items = prompt_items(cases, dev, tf, min_bytes)
        return items, sum(it["bytes"] for it in items)
    if workload == "gather":
        items, per_step = gather_items(cases, dev, tf)
    elif workload == "options":
        items, per_step = options_items(cases, dev, tf)
    elif workload == "stack":
        items, per_step = stack_items(cases, dev, tf)
    else:
        items = product_items(cases, dev, min_bytes)
        return items, sum(it["bytes"] for it in items)
    copies = max(1, -(-min_bytes // per_step))
    for it in items:
        it["grow"](copies)
    return items, per_step


def oracle_checks(items, cols_per_case, nthreads):
    """CPU-baseline leg: the fp64 oracle on a column sample of each case's last GPU
    output.  Per case: worst |y - y64| / bound and the 1%-off control (max over
    the sampled outputs of |y - y64(scales * 1.01)| / bound)."""
    import oracle
    out = {}
    for it in items:
        y_gpu = it["y_host"]
        worst, ctrl = 0.0, float("inf")
        for (m, x_h, col0) in it.get("check", []):
            rng = np.random.default_rng(m.seed)
            cols = np.unique(np.concatenate([[0, m.N - 1], rng.choice(m.N, min(cols_per_case, m.N), replace=False)]))
            y64, absum = oracle.qmm(x_h, m.W, m.scales, m.biases, m.N, m.K, m.bits, m.group, cols=cols,
                                    nthreads=nthreads)
            B = oracle.bound(absum, m.K)
            yg = y_gpu[:x_h.shape[0], col0 + cols].astype(np.float64)
            xf = synth.bf16_bits_to_f32(x_h).astype(np.float64)
            sx = xf.reshape(x_h.shape[0], m.K // m.group, m.group).sum(axis=2)
            bias_part = sx @ synth.bf16_bits_to_f32(m.biases[cols]).astype(np.float64).T
            worst = max(worst, float(np.max(np.abs(yg - y64) / B)))
            ctrl = min(ctrl, float(np.max(np.abs(yg - (y64 + 0.01 * (y64 - bias_part))) / B)))
        if it.get("check"):
            out[it["label"]] = (worst, ctrl)
    return out


def run_gpu(args, cases):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    import mlx_affine_bit_gb300 as tf

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    tf.lib()
    modes = {"plain": 0, "pdl": tf.TF_LAUNCH_PDL, "early": tf.TF_LAUNCH_EARLY_WEIGHTS,
             "indep": tf.TF_LAUNCH_EARLY_WEIGHTS | tf.TF_LAUNCH_EARLY_X}
    tf.tf_set_launch_mode(modes[args.launch])
    stream = torch.cuda.current_stream()
    cap = torch.cuda.Stream(device=dev)
    min_bytes = 4 * L2_BYTES

    # Device-resident inputs; enough weight copies that a buffer is reused only
    # after >= 4 L2 sizes of other traffic.
    items, per_step = build_items(args.workload, cases, dev, tf, min_bytes)
    copies = max(1, -(-min_bytes // per_step))
    torch.cuda.synchronize()

    # The timed region replays CUDA graphs, so host launch overhead does not
    # enter the device timing: a graph of `copies` consecutive steps (every
    # call once per step, each step on the next weight copy) and one of the
    # remaining steps % copies steps, so that exactly --steps steps are timed.
    with torch.cuda.stream(cap):
        for w in range(args.warmup):
            for it in items:
                launch_item(tf, it, w, cap)
    torch.cuda.synchronize()

    def step_graph(nsteps, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for c in range(first, first + nsteps):
                for it in items:
                    launch_item(tf, it, c, cap)
        return g

    full = step_graph(min(copies, args.steps), 0)
    n_full, rem = divmod(args.steps, min(copies, args.steps))
    rest = step_graph(rem, 0) if rem else None
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        full.replay()
        if rest is not None:
            rest.replay()
    torch.cuda.synchronize()

    clk = ClockSampler(local)
    clk.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        t0.record(cap)
        for _ in range(n_full):
            full.replay()
        if rest is not None:
            rest.replay()
        t1.record(cap)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = clk.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    tf.tf_device_status()
    del full, rest

    # Per-call device times of the headline's calls (each its own graph).
    peak, peak_kind = _peaks()
    case_us = [time_item(tf, it, cap, 2) for it in items]
    case_rows = [case_row(it["label"], it["bytes"], us, peak) for it, us in zip(items, case_us)]
    # The same calls when every product waits for the one before it before it
    # reads x (early weights only): the order a chain of dependent layers needs.
    dependent = None
    prompt_wl = args.workload == "prompt"      # tf_qmm_prompt: plain launches, no launch modes
    if args.launch == "indep" and not prompt_wl:
        tf.tf_set_launch_mode(modes["early"])
        dep_us = [time_item(tf, it, cap, 2) for it in items]
        tf.tf_set_launch_mode(modes[args.launch])
        dep_gbs = per_step / (sum(dep_us) * 1e-6) / 1e9
        dependent = {"launch": "programmatic dependent launch, weights streamed before the dependency wait, x "
                               "read after it (each product waits for the previous one)",
                     "achieved": dep_gbs, "frac": dep_gbs / peak, "unit": "GB/s",
                     "per_case_us": [round(u, 3) for u in dep_us]}
    for it in items:
        it["y_host"] = it["y"].float().cpu().numpy() if it["y"].dtype == torch.float32 else None

    # ---- end to end: pinned host x in, host y out, through the C ABI ----
    # A step's activations arrive in one host-to-device copy and its results
    # leave in one device-to-host copy (every call's x and y are views of one
    # device buffer each, 256-byte aligned).
    def joint(key, pin_key):
        offs, total = [], 0
        for it in items:
            offs.append(total)
            total += -(-it[key].numel() * it[key].element_size() // 256) * 256
        dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
        pin_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        views = []
        for it, o in zip(items, offs):
            t = it[key]
            nb = t.numel() * t.element_size()
            views.append(dev_buf[o:o + nb].view(t.dtype).view(t.shape))
            pin_buf[o:o + nb].copy_(it[pin_key].reshape(-1).view(torch.uint8))
        return dev_buf, pin_buf, views

    x_dev, x_pin, x_views = joint("x", "x_pin")
    y_dev, y_pin, y_views = joint("y", "y_pin")
    saved = [(it["x"], it["y"]) for it in items]
    for it, xv, yv in zip(items, x_views, y_views):
        it["x"], it["y"] = xv, yv
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 200))
    e0.record(stream)
    for k in range(e2e_steps):
        x_dev.copy_(x_pin, non_blocking=True)
        for it in items:
            launch_item(tf, it, k, stream)
        y_pin.copy_(y_dev, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    for it, (xo, yo) in zip(items, saved):
        it["x"], it["y"] = xo, yo
    h2d, d2h = x_pin.numel(), y_pin.numel()
    del x_dev, x_pin, y_dev, y_pin, x_views, y_views

    # ---- the other target configurations: each timed in its own graph ----
    checked = list(items)
    if args.workload == "sweep" and not args.no_extra:
        for wl in EXTRA_WORKLOADS:
            ex_items, _ = build_items(wl, workload_cases(wl), dev, tf, min_bytes)
            for it in ex_items:
                us = time_item(tf, it, cap, 2)
                case_rows.append(case_row(it["label"], it["bytes"], us, peak))
                it["y_host"] = it["y"].cpu().numpy()
                for k in ("reps", "x", "y", "x_pin", "y_pin"):
                    it.pop(k, None)
                checked.append(it)
            del ex_items
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
    tf.tf_device_status()

    value = job_throughput(per_step * args.steps, world, ms)
    kern_ms = sum(case_us) * 1e-3                            # a step's summed per-call times
    achieved = per_step / (kern_ms * 1e-3) / 1e9
    traffic, traffic_note = committed_traffic(args.workload)
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cores = os.cpu_count() or 1
            gbs, secs, nb = cpu_sample(cases, 1, cores)      # probe
            cols = max(1, min(4096, int(12.0 / max(secs, 1e-3))))
            # About 10 s of oracle work: the column sample, repeated when even the
            # whole workload takes less.
            secs, nb, reps = 0.0, 0, 0
            while secs < 10.0 and reps < 200:
                _, t, b = cpu_sample(cases, cols, cores)
                secs, nb, reps = secs + t, nb + b, reps + 1
            cpu = {"value": nb / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                   "sample": "fp64 oracle on the first %d output columns of each product, %d pass%s (%.1f s)"
                             % (cols, reps, "" if reps == 1 else "es", secs)}
            # The same oracle checks each timed case's GPU output: every column up to
            # 16384 columns, a sample of 16384 columns beyond.
            checks = oracle_checks(checked, 16384, cores)
            for row in case_rows:
                if row["case"] in checks:
                    w, c = checks[row["case"]]
                    row["oracle_worst_err_over_bound"] = round(w, 4)
                    row["control_1pct_over_bound"] = round(c, 3)
            cpu["checks"] = "each case's last GPU output against the fp64 oracle on every column (a sample of " \
                            "16384 columns of the LM heads): worst err/bound, and the max ratio of the " \
                            "1%-off-scales control (must exceed 1)"
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "parallelism": "replicas" if world > 1 else "1 GPU",
                       "launch": "plain launches (x prepass, one kernel per 64-row window, a fold when chunks are "
                                 "split); launch modes do not apply" if prompt_wl else
                                 {"plain": "plain launches", "pdl": "programmatic dependent launch",
                                  "early": "programmatic dependent launch; weights streamed before the "
                                           "dependency wait (weights are never written in the step)",
                                  "indep": "programmatic dependent launch; the step's products are independent "
                                           "(no call writes any weights or x of the step), so each streams its "
                                           "weights and reads x before its dependency wait and waits only before "
                                           "writing y (TF_LAUNCH_EARLY_WEIGHTS | TF_LAUNCH_EARLY_X)"}[args.launch],
                       "l2": "weights rotate over %d copies (%.0f MB a step, >= 4x L2 between reuses)"
                             % (copies, per_step / 1e6)},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "frac_of_8tbs_nominal": achieved / 8000.0,
                         "traffic": traffic, "traffic_note": traffic_note,
                         "traffic_unit": "bytes per step (all %s launches of one step)"
                                         % ("prompt" if prompt_wl else "qmm"),
                         "kernel": ("tfq::prompt::prompt_kernel" if prompt_wl else "tfq::qmm_kernel")
                                   + " (all products of the step, bytes / summed per-call time)"},
            "dependent_x": dependent,
            "cpu_baseline": cpu,
            "e2e": {"value": job_throughput(per_step * e2e_steps, world, e2e_ms), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": sum(item_launches(it) for it in items) * args.steps,
            "timing": "exactly %d steps: a CUDA graph of %d steps replayed %d times%s; per-case time: the median "
                      "over 7 replays of a graph of calls cycling over the weight copies (>= 4 L2 sizes of "
                      "weights, >= 8 calls)"
                      % (args.steps, min(copies, args.steps), n_full,
                         " plus one of %d steps" % rem if rem else ""),
            "kernel_source_sha": kernel_source_sha(),
            "clocks": clocks,
            "cases": case_rows,
        }))
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sweep", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the headline workload (no LM head / decode / stack cases)")
    ap.add_argument("--launch", default="indep", choices=["plain", "pdl", "early", "indep"])
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    cases = workload_cases(args.workload)
    if args.impl == "reference":
        run_reference(args, cases)
    else:
        run_gpu(args, cases)


if __name__ == "__main__":
    main()
