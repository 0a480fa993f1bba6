"""Benchmark: on-device sampling of a [256, 129,280] bf16 mixed-parameter batch.

One step = one arc_sample_batch call over one batch (every row: penalties,
mode dispatch, top-k / top-p / min-p, inverse-CDF draw).  Prints one JSON line.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

value: rows/s with the logits already resident in HBM; K launches are
replayed back to back from CUDA graphs, cycling over input copies whose total
is larger than L2, and timed with CUDA events on the launch stream; the
per-step time is the median over --repeats such regions (min and max beside).
configs: the same measurement for each of the five synthetic workloads (the
small fp32 batch, the single-row decode loop greedy and with the defaults,
the mixed batch, the penalised batch, the tied fp32 batch), plus the cost of
the design the library replaces: one D2H copy of the bench batch's logits.
e2e: the same metric through the C ABI from pinned host buffers, with the
host->device copy of the logits and parameters and the device->host read of
the tokens inside every step.
cpu_baseline: the fp64 oracle on every host core (and on one thread).
--impl reference: the fp64 oracle on the host cores (a bounded sample of rows
per step), the only CPU use of oracle/ besides the cpu_baseline leg.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sampled rows/s and achieved HBM GB/s (% of GB300 roofline) at B=256, V=129,280"
NBUF = 6  # input copies cycled per step: 6 x 66 MB > L2
PROFILE = os.path.join(ROOT, "profiles", "scan_finish_mixed_quarters_B256.md")
KERNELS_PER_STEP = 2  # scan_kernel + finish_kernel
CSRC = os.path.join(ROOT, "device_logits_sampling_gb300", "csrc")


def kernel_hash() -> str:
    """Hash of the kernel sources' code: comments and layout do not count, so a
    profile stays matched to the build it measured until the code changes."""
    h = hashlib.sha256()
    for f in sorted(x for x in os.listdir(CSRC) if x.endswith((".cu", ".cuh"))):
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def profiled_traffic():
    """dram bytes of one step (both kernels) from the committed ncu summary, if it
    matches the current kernel sources."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    mh = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not mh or not mt or mh.group(1) != kernel_hash():
        return None
    return int(mt.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rows_of_shard(B: int, world: int, rank: int) -> range:
    """Weak scaling: every rank samples its own full batch; shard r owns global rows [r*B, (r+1)*B)."""
    return range(rank * B, (rank + 1) * B)


def _oracle_rows(task):
    """Worker of the host-core oracle pool: sample rows (logits, params, row index)."""
    import oracle

    z, prm, rows = task
    for zi, pi, r in zip(z, prm, rows):
        oracle.sample_row(zi, pi, int(r))
    return len(rows)


def host_info() -> dict:
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


def oracle_rate(z, params, rows, workers: int, passes: int = 1) -> float:
    """Rows per second of the fp64 oracle over `rows` of a batch (repeated `passes`
    times), on `workers` host processes (spawn start: no state shared with CUDA);
    pool start-up is outside the timed region."""
    import multiprocessing as mp

    rows = list(rows)
    if workers <= 1:
        t0 = time.perf_counter()
        for _ in range(passes):
            _oracle_rows((z[rows], params[rows], rows))
        return passes * len(rows) / (time.perf_counter() - t0)
    per = max(1, len(rows) // (workers * 2))
    tasks = [(z[rows[i:i + per]], params[rows[i:i + per]], rows[i:i + per]) for i in range(0, len(rows), per)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_rows, tasks[:workers])  # warm the workers (imports)
        t0 = time.perf_counter()
        n = 0
        for _ in range(passes):
            n += sum(pool.map(_oracle_rows, tasks))
        dt = time.perf_counter() - t0
    return n / dt


def cpu_baseline() -> dict:
    """The oracle as it stands on this host: every host core over the whole
    mixed batch (4 passes), and one thread over its first 48 rows."""
    from device_logits_sampling_gb300 import workloads

    w = workloads.mixed_batch()
    z = w.logits_f32()
    info = host_info()
    cores = info["nproc"] or 1
    all_cores = oracle_rate(z, w.params, range(w.B), cores, passes=4)
    one = oracle_rate(z, w.params, range(48), 1)
    return {"value": all_cores, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"4 passes over the 256 rows of the B=256 mixed batch (row%4 mix kept), fp64 numpy, "
                      f"{cores} processes",
            "single_thread_value": one, "single_thread_sample": "first 48 rows of the same batch, one thread",
            "cpu_model": info["cpu_model"], "nproc": info["nproc"]}


def bench_reference(args) -> None:
    """--impl reference: the fp64 oracle on the host cores, K timed steps of a bounded row sample."""
    import multiprocessing as mp

    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    from device_logits_sampling_gb300 import workloads

    w = workloads.mixed_batch()
    z = w.logits_f32()
    info = host_info()
    cores = info["nproc"] or 1
    # size the per-step sample so K + W steps take about a minute on every core
    t0 = time.perf_counter()
    for r in range(4):
        oracle.sample_row(z[r], w.params[r], r)
    per_row = (time.perf_counter() - t0) / 4
    rows = int(max(4, min(w.B, cores * 60.0 / max(1, args.steps + args.warmup) / per_row)))
    rows -= rows % 4
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        per = max(1, rows // cores)

        def step(i):
            base = (i * rows) % w.B
            idx = [(base + j) % w.B for j in range(rows)]
            tasks = [(z[idx[a:a + per]], w.params[idx[a:a + per]], idx[a:a + per]) for a in range(0, rows, per)]
            pool.map(_oracle_rows, tasks)

        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(i)
        dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "V": w.V, "logits_dtype": "bf16",
                   "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows per step of the B=256 mixed batch, fp64 numpy, {cores} processes",
                         "cpu_model": info["cpu_model"]},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


def graph_steps(sampler, stream, bufs, call, n):
    """A CUDA graph of n steps, step i sampling input copy i % len(bufs)."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                call(bufs[i % len(bufs)])
    return g


def time_steps(stream, graphs, repeats):
    """Per-step microseconds of `repeats` timed regions, each replaying `graphs`
    once back to back, with CUDA events on the launch stream."""
    import torch

    steps = sum(n for _, n in graphs)
    out = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g, _ in graphs:
                g.replay()
            e1.record(stream)
        stream.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / steps)
    return out


def bench_config(sampler, workloads, name, peak, steps, repeats):
    """One named workload: graph-replayed steps over rotating input copies
    (more than L2 in total), per-step time median and min over `repeats`
    regions; the share of filtered rows that took the direct selection."""
    import numpy as np
    import torch

    kw = {k: v for k, v in name[1].items() if k != "f16"}
    w = getattr(workloads, name[0])(**kw)
    if name[1].get("f16"):
        w = workloads.as_f16(w)
    B, V = w.B, w.V
    nbuf = max(2, min(NBUF, int(3 * 129e6 // (B * V * w.elem_bytes)) + 1))
    bufs = [sampler.logits_tensor(w) for _ in range(nbuf)]
    prm = sampler.params_tensor(w.params)
    hoff, hids = sampler.history_tensors(w)
    mhl = int(np.diff(w.hist_offsets).max()) if hoff is not None else 0
    out = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = sampler.workspace_tensor(B, V, w.dtype, hoff is not None, max_hist_len=mhl)
    dbg = sampler.debug_tensor(B)
    st = torch.cuda.Stream()
    autoinc = name[0] == "single_row_peaked"  # the decode loop: the step advances on device
    with torch.cuda.stream(st):
        sampler.sample_batch(bufs[0], prm, out, hoff, hids, workspace=ws, max_hist_len=mhl, debug=dbg, stream=st)
    st.synchronize()
    d = sampler.debug_records(dbg)

    def call(x):
        sampler.sample_batch(x, prm, out, hoff, hids, workspace=ws, max_hist_len=mhl, autoinc=autoinc, stream=st)

    g = graph_steps(sampler, st, bufs, call, steps)
    g.replay()
    st.synchronize()
    ts = time_steps(st, [(g, steps)], repeats)
    med, mn = statistics.median(ts), min(ts)
    alg = B * V * w.elem_bytes + B * 48 + B * 4 + (4 * int(w.hist_ids.size) + 4 * (B + 1) if hoff is not None else 0)
    filt = d["mode"] == 2
    rec = {"B": B, "V": V, "logits_dtype": {workloads.DTYPE_F32: "f32", workloads.DTYPE_BF16: "bf16",
                                            workloads.DTYPE_F16: "f16"}[w.dtype],
           "us_per_step_median": med, "us_per_step_min": mn, "rows_per_s": B / (med * 1e-6),
           "achieved_gbs": alg / (med * 1e-6) / 1e9, "frac_of_measured_peak": alg / (med * 1e-6) / 1e9 / peak,
           "alg_bytes": alg, "steps": steps, "repeats": repeats, "input_copies": nbuf,
           "filtered_rows": int(filt.sum()), "direct_selection_rows": int(((d["passes"] == 1) & filt).sum())}
    if autoinc:
        rec["note"] = "decode loop: the step counter advances on device (ARC_OPT_STEP_AUTOINC)"
    del bufs, ws
    torch.cuda.empty_cache()
    return w.name, rec


CONFIGS = [  # the five synthetic workloads, in the order of the configuration list
    ("small_fp32", {}),
    ("single_row_peaked", {"greedy": True}),
    ("single_row_peaked", {}),
    ("mixed_batch", {}),
    ("penalized_batch", {}),
    ("adversarial_ties", {}),
    ("mixed_batch", {"f16": True}),  # the mixed batch's values as fp16 logits
]


def bench_only_config(args) -> None:
    """--only-config NAME: one synthetic workload's record (for profiling one
    configuration's kernels), K steps, one timed region."""
    import torch

    from device_logits_sampling_gb300 import sampler, workloads

    torch.cuda.set_device(0)
    sampler.load()
    peak = measured_peaks().get("hbm_gbs") or 6800.0
    kw = {"greedy": True} if args.only_config == "single_row_peaked_greedy" else {}
    name = "single_row_peaked" if args.only_config.startswith("single_row_peaked") else args.only_config
    if name.endswith("_f16"):  # e.g. mixed_batch_f16: the workload's values as fp16 logits
        name, kw = name[: -len("_f16")], {**kw, "f16": True}
    key, rec = bench_config(sampler, workloads, (name, kw), peak, max(1, args.steps), max(1, args.repeats))
    print(json.dumps({"workload": key, **rec}))


def bench_gpu(args) -> None:
    import numpy as np
    import torch

    from device_logits_sampling_gb300 import sampler, workloads

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sampler.load()

    w = workloads.mixed_batch()
    B, V = w.B, w.V
    # weak scaling: rank r samples rows [r*B, (r+1)*B) of a larger job; the
    # seeds follow the global row so every rank draws different tokens
    params_np = w.params.copy()
    params_np["seed"] = np.array(list(rows_of_shard(B, ws, rank)), dtype=np.uint64)
    params = sampler.params_tensor(params_np)
    bufs = [sampler.logits_tensor(w) for _ in range(NBUF)]
    out = torch.zeros(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    geom = sampler.plan(B, V, w.dtype)
    wspace = sampler.workspace_tensor(B, V, w.dtype)
    stream = torch.cuda.Stream()

    # first call on the device sets kernel attributes (outside any capture)
    with torch.cuda.stream(stream):
        sampler.sample_batch(bufs[0], params, out, err_word=err, workspace=wspace, stream=stream)
    stream.synchronize()
    assert int(err.item()) == 0, hex(int(err.item()))

    def call(x):
        sampler.sample_batch(x, params, out, err_word=err, workspace=wspace, stream=stream)

    chunk = min(args.steps, 480)
    graphs = [(graph_steps(sampler, stream, bufs, call, chunk), chunk)] * (args.steps // chunk)
    if args.steps % chunk:
        graphs.append((graph_steps(sampler, stream, bufs, call, args.steps % chunk), args.steps % chunk))

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # warm-up: W untimed steps
    gw = graph_steps(sampler, stream, bufs, call, args.warmup)
    gw.replay()
    stream.synchronize()

    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = ClockSampler(int(vis[local]) if local < len(vis) and vis[local].isdigit() else local)
    repeats = max(1, args.repeats)
    barrier()
    clocks.start()
    time.sleep(0.05)
    ts = time_steps(stream, graphs, repeats)
    barrier()
    clk = clocks.stop()
    assert int(err.item()) == 0, hex(int(err.item()))
    us = statistics.median(ts)
    if ws > 1:
        t = torch.tensor([us], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        us = float(t.item())
    ms_per_step = us * 1e-3
    value = ws * B / (us * 1e-6)

    # ---- end to end through the C ABI from pinned host buffers
    host_logits = bufs[0].cpu().pin_memory()
    host_params = params.cpu().pin_memory()
    host_out = torch.zeros(B, dtype=torch.int32).pin_memory()
    dev_logits = torch.empty_like(bufs[0])
    dev_params = torch.empty_like(params)
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_step():
        with torch.cuda.stream(stream):
            dev_logits.copy_(host_logits, non_blocking=True)
            dev_params.copy_(host_params, non_blocking=True)
            sampler.sample_batch(dev_logits, dev_params, out, err_word=err, workspace=wspace, stream=stream)
            host_out.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    barrier()
    e2e_s = time.perf_counter() - t0
    if ws > 1:
        t = torch.tensor([e2e_s], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_value = ws * B * e2e_steps / e2e_s

    if rank == 0:
        es = 2
        alg_bytes = B * V * es + B * 48 + B * 4
        achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
        peaks = measured_peaks()
        peak = peaks.get("hbm_gbs")
        peak_src = "measured" if peak else "fallback"
        peak = peak or 6800.0
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {
                "workload": w.name, "B": B, "V": V, "logits_dtype": "bf16",
                "params": "row%4: greedy | T=1 defaults | top_k=50 T=0.7 | top_p=0.9 min_p=0.05 T=0.8",
                "l2": f"inputs larger than L2: {NBUF} rotating copies of the batch "
                      f"({NBUF * B * V * es / 1e6:.0f} MB)",
                "ctas_per_row": geom.ctas_per_row, "launch": "CUDA graph, one launch per step",
                "parallelism": f"rows sharded, {ws} independent rank(s)",
            },
            "timing": {"repeats": repeats, "steps_per_repeat": args.steps,
                       "us_per_step_median": statistics.median(ts), "us_per_step_min": min(ts),
                       "us_per_step_max": max(ts)},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(),
                         "peak_source": peak_src, "alg_bytes_per_launch": alg_bytes,
                         "scope": "one step: scan_kernel (reads every logit once) + finish_kernel, "
                                  "timed together with CUDA events on the launch stream",
                         "frac_of_nominal_8tbs": achieved / 8000.0},
            "e2e": {"value": e2e_value, "unit": "rows/s",
                    "h2d_bytes_per_step": int(host_logits.numel() * host_logits.element_size()
                                              + host_params.numel()),
                    "d2h_bytes_per_step": int(B * 4)},
            "gpu_launches": KERNELS_PER_STEP * args.steps * repeats,
            "clocks": clk,
        }
        if ws == 1 and not args.no_configs:
            # the design the library replaces: the whole logits tensor to pinned host memory per step
            host = torch.empty(bufs[0].shape, dtype=bufs[0].dtype).pin_memory()
            d2h = []
            for i in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    host.copy_(bufs[i % NBUF], non_blocking=True)
                    e1.record(stream)
                stream.synchronize()
                d2h.append(e0.elapsed_time(e1))
            nbytes = B * V * es
            line["d2h_context"] = {"bytes": nbytes, "ms_median": statistics.median(d2h), "ms_min": min(d2h),
                                   "gbs": nbytes / (statistics.median(d2h) * 1e-3) / 1e9,
                                   "what": "one D2H copy of the B=256 bf16 logits into pinned host memory"}
            del bufs, wspace
            torch.cuda.empty_cache()
            cfg = {}
            for nm in CONFIGS:
                steps = 1000 if nm[0] == "single_row_peaked" else (40 if nm[0] in ("penalized_batch", "adversarial_ties")
                                                                   else 400)
                key, rec = bench_config(sampler, workloads, nm, peak, steps, 5)
                cfg[key] = rec
            line["configs"] = cfg
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def bench_small_batches(args) -> None:
    """--small-batches: per-step latency of small batches of the mixed rows
    (V = 129,280 bf16) on the one-launch cluster path and on the two-kernel
    path (forced by an explicit slice count), and the path the library picks,
    so that the choice per B can be checked against both."""
    import torch

    from device_logits_sampling_gb300 import sampler, workloads

    torch.cuda.set_device(0)
    sampler.load()
    n = max(1, args.steps)
    rows = []
    for B in (1, 2, 4, 8, 16, 19, 20, 32, 64):
        w = workloads.mixed_batch(B=B)
        nbuf = max(2, min(NBUF, int(3 * 129e6 // (B * w.V * w.elem_bytes)) + 1))
        bufs = [sampler.logits_tensor(w) for _ in range(nbuf)]
        prm = sampler.params_tensor(w.params)
        out = torch.zeros(B, dtype=torch.int32, device="cuda")
        st = torch.cuda.Stream()
        rec = {"B": B, "chosen_launches": sampler.plan(B, w.V, w.dtype).launches}
        for label, cpr in (("auto_us", 0), ("two_kernel_us", 16)):
            ws = sampler.workspace_tensor(B, w.V, w.dtype, ctas_per_row=cpr)

            def call(x, ws=ws, cpr=cpr):
                sampler.sample_batch(x, prm, out, workspace=ws, ctas_per_row=cpr, stream=st)

            with torch.cuda.stream(st):
                call(bufs[0])
            st.synchronize()
            g = graph_steps(sampler, st, bufs, call, n)
            g.replay()
            st.synchronize()
            rec[label] = statistics.median(time_steps(st, [(g, n)], max(1, args.repeats)))
        rows.append(rec)
        del bufs
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "small-batch step latency, mixed rows, V=129,280 bf16: the library's choice "
                                "(one cluster launch for B <= 8) against two kernels with 16 slices per row",
                      "unit": "us", "higher_is_better": False, "steps": n, "rows": rows}))


def bench_decode_loop(args) -> None:
    """--decode-loop: the decode step after sampling (arc_decode_commit into a
    pinned host ring).  Times, with CUDA events over graph replays on the
    mixed B=256 batch, one step of sampling alone, one step of sampling
    followed by the commit kernel, the commit kernel alone, and sampling with
    the commit folded into its finish (arc_sample_batch_commit); the host
    drains every record of the timed replays afterwards and checks their
    count and owners."""
    import numpy as np
    import torch

    from device_logits_sampling_gb300 import decode, sampler, workloads

    w = workloads.mixed_batch()
    B, V = w.B, w.V
    bufs = [sampler.logits_tensor(w) for _ in range(NBUF)]
    prm = sampler.params_tensor(w.params)
    out = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = sampler.workspace_tensor(B, V, w.dtype)
    ids = torch.zeros(B, dtype=torch.int32, device="cuda")
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    owners = torch.arange(B, dtype=torch.int32, device="cuda")
    head = torch.zeros(2, dtype=torch.int64, device="cuda")  # [1]: the folded commit's arrival count
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = max(1, args.steps)
    ring = decode.Ring(B * (n * 4 + args.warmup * 4 + 8))
    s = torch.cuda.Stream()

    def timed(fn):
        with torch.cuda.stream(s):
            sampler.sample_batch(bufs[0], prm, out, workspace=ws, stream=s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(NBUF):
                    fn(i)
            for _ in range(max(1, args.warmup // NBUF)):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(1, n // NBUF)
            e0.record(s)
            for _ in range(reps):
                g.replay()
            e1.record(s)
            s.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * NBUF)

    def sample(i):
        sampler.sample_batch(bufs[i], prm, out, workspace=ws, autoinc=True, stream=s)

    def commit():
        decode.decode_commit(out, ids, pos, 1 << 30, V, ring, head[:1], owners=owners, fault_word=fault, stream=s)

    def both(i):
        sample(i)
        commit()

    def folded(i):
        decode.sample_and_commit(bufs[i], prm, out, ids, pos, 1 << 30, ring, head, owners=owners, fault_word=fault,
                                 workspace=ws, autoinc=True, stream=s)

    t_sample = timed(sample)
    t_both = timed(both)
    t_commit = timed(lambda i: commit())
    t_folded = timed(folded)
    published = int(head[0].item())
    assert int(head[1].item()) == 0
    recs = ring.drain(published, max_spins=1 << 20)
    assert len(recs) == published and int(fault.item()) == 0
    assert np.array_equal(recs["owner"], np.tile(np.arange(B), published // B))
    print(json.dumps({
        "metric": "decode step after sampling: sample + commit into a pinned host ring", "unit": "us",
        "B": B, "V": V, "sample_us": t_sample, "sample_and_commit_us": t_both, "commit_alone_us": t_commit,
        "commit_added_us": t_both - t_sample, "sample_with_folded_commit_us": t_folded,
        "folded_commit_added_us": t_folded - t_sample, "records_drained": published, "higher_is_better": False,
    }))
    ring.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' figures")
    ap.add_argument("--repeats", type=int, default=5, help="timed regions of K steps (median and min reported)")
    ap.add_argument("--only-config", default=None,
                    help="time one synthetic workload only (small_fp32, single_row_peaked[_greedy], mixed_batch, "
                         "penalized_batch, adversarial_ties; a _f16 suffix: as fp16 logits) and print its record")
    ap.add_argument("--decode-loop", action="store_true", help="time the decode-loop commit (separate JSON line)")
    ap.add_argument("--small-batches", action="store_true",
                    help="small-batch latency: cluster path against two kernels (separate JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only_config:
        bench_only_config(args)
    elif args.small_batches:
        bench_small_batches(args)
    elif args.decode_loop:
        bench_decode_loop(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
