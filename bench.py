"""Benchmark: on-device sampling of a [256, 129,280] bf16 mixed-parameter batch.

One step = one arc_sample_batch call over one batch (every row: penalties,
mode dispatch, top-k / top-p / min-p, inverse-CDF draw).  Prints one JSON line.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

value: rows/s with the logits already resident in HBM; K launches are
replayed back to back from CUDA graphs, cycling over input copies whose total
is larger than L2, and timed with CUDA events on the launch stream.
e2e: the same metric through the C ABI from pinned host buffers, with the
host->device copy of the logits and parameters and the device->host read of
the tokens inside every step.
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
KERNEL_SOURCES = ["arc_sample.cu", "stream_kernel.cuh", "row_select.cuh", "arc_device.cuh"]


def kernel_hash() -> str:
    """Hash of the kernel sources' code: comments and layout do not count, so a
    profile stays matched to the build it measured until the code changes."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "device_logits_sampling_gb300", "csrc", f), encoding="utf-8") as fh:
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


def cpu_baseline(seconds: float = 12.0) -> dict:
    """The oracle as it stands on this host, over the first rows of the batch (row mix kept)."""
    import oracle
    from device_logits_sampling_gb300 import workloads

    w = workloads.mixed_batch()
    z = w.logits_f32()
    t0 = time.perf_counter()
    n = 0
    while n < w.B and (n < 16 or time.perf_counter() - t0 < seconds):
        oracle.sample_row(z[n], w.params[n], n)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"first {n} rows of the B=256 mixed batch (row%4 mix kept), fp64 numpy, one thread"}


def bench_reference(args) -> None:
    """--impl reference: the fp64 oracle on the host cores, K timed steps of a bounded row sample."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    from device_logits_sampling_gb300 import workloads

    w = workloads.mixed_batch()
    z = w.logits_f32()
    # size the per-step sample so K + W steps take about a minute
    t0 = time.perf_counter()
    for r in range(4):
        oracle.sample_row(z[r], w.params[r], r)
    per_row = (time.perf_counter() - t0) / 4
    rows = int(max(1, min(w.B, 60.0 / max(1, args.steps + args.warmup) / per_row)))
    rows = max(4, rows - rows % 4) if rows >= 4 else rows

    def step(i):
        base = (i * rows) % w.B
        for j in range(rows):
            r = (base + j) % w.B
            oracle.sample_row(z[r], w.params[r], r)

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
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} rows per step of the B=256 mixed batch, fp64 numpy, one thread"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


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

    chunk = min(args.steps, 480)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    sampler.sample_batch(bufs[i % NBUF], params, out, err_word=err, workspace=wspace,
                                         stream=stream)
        return g

    g_main = capture(chunk)
    rem = args.steps % chunk
    g_rem = capture(rem) if rem else None
    reps = args.steps // chunk

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # warm-up: W untimed steps
    with torch.cuda.stream(stream):
        gw = capture(args.warmup) if args.warmup else None
        if gw is not None:
            gw.replay()
    stream.synchronize()

    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = ClockSampler(int(vis[local]) if local < len(vis) and vis[local].isdigit() else local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    clocks.start()
    time.sleep(0.05)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    assert int(err.item()) == 0, hex(int(err.item()))
    if ws > 1:
        t = torch.tensor([ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / args.steps
    value = ws * B * args.steps / (ms / 1e3)

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
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clk,
        }
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def bench_decode_loop(args) -> None:
    """--decode-loop: the decode step after sampling (arc_decode_commit into a
    pinned host ring).  Times, with CUDA events over graph replays on the
    mixed B=256 batch, one step of sampling alone, one step of sampling
    followed by the commit, and the commit alone; the host drains every
    record of the timed replays afterwards and checks their count and owners."""
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
    head = torch.zeros(1, dtype=torch.int64, device="cuda")
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = max(1, args.steps)
    ring = decode.Ring(B * (n * 3 + args.warmup * 3 + 8))
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
        decode.decode_commit(out, ids, pos, 1 << 30, V, ring, head, owners=owners, fault_word=fault, stream=s)

    def both(i):
        sample(i)
        commit()

    t_sample = timed(sample)
    t_both = timed(both)
    t_commit = timed(lambda i: commit())
    published = int(head.item())
    recs = ring.drain(published, max_spins=1 << 20)
    assert len(recs) == published and int(fault.item()) == 0
    assert np.array_equal(recs["owner"], np.tile(np.arange(B), published // B))
    print(json.dumps({
        "metric": "decode step after sampling: sample + commit into a pinned host ring", "unit": "us",
        "B": B, "V": V, "sample_us": t_sample, "sample_and_commit_us": t_both, "commit_alone_us": t_commit,
        "commit_added_us": t_both - t_sample, "records_drained": published, "higher_is_better": False,
    }))
    ring.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-loop", action="store_true", help="time the decode-loop commit (separate JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.decode_loop:
        bench_decode_loop(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
