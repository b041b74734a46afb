#!/usr/bin/env python
"""Benchmark of the GB300 sparse-attention prefill indexer.

One step = one idx_score_topk call (sampled thresholds, the tcgen05 scoring
pass with candidate emission, the slab top-k and the exact rescan) on the fused
prefill workload: 4096 query rows, 65536 keys, 64 heads, D = 128, topk 2048,
fp8 e4m3 q/k, causal visible ranges.  Inputs are synthetic and seeded.

Prints ONE JSON line (rank 0).  Timing: W untimed warm-up steps, then K steps
timed on the device with CUDA events on the launching stream; the L2 is flushed
between steps, outside the timed events (a 256 MiB write, then a 256 MiB read
that writes the dirty lines back), and a short device-side spin keeps the
stream busy while the host issues the next call, so that the events time the
device work.  --impl reference
times the CPU oracle instead (rank 0, a bounded sample of the same workload).

Multi-GPU (torchrun): every rank runs its own copy of the workload (the rows of
different prefills are independent), no collective on the data path; value is
the sum over ranks of the work divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("scored row·key pairs/s (fused score+top-k) and top-k rows/s; % of roofline")
WORKLOAD = "fused_prefill"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extra", action="store_true", help="skip the secondary measurements")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--clocks-file", default=None)
    p.add_argument("--rows", type=int, default=0,
                   help="profiling: use only the last N query rows of the workload")
    p.add_argument("--workload", default=WORKLOAD,
                   choices=["fused_prefill", "long_context", "mixed_batch", "tiny"],
                   help="fused workload of the main line (default: the one the metric is "
                        "quoted on)")
    p.add_argument("--route-sweep", action="store_true",
                   help="time the fused and the two-pass path over short key lengths (the "
                        "routing gate's crossover) and print one JSON line per case")
    p.add_argument("--only", choices=["all", "fused", "topk", "split"], default="all",
                   help="profiling: run only the fused step, the standalone top-k or the "
                        "row split")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# The sources each recorded kernel is built from (a recorded ncu figure stays
# valid while these are unchanged).
KERNEL_SOURCES = {
    "score_kernel": ["common.cuh", "plan.cuh", "radix.cuh", "score.cuh", "score_impl.cuh",
                     "score_launch.cuh", "score_fp8.cu", "score_bf16.cu"],
    "topk_rows_kernel": ["common.cuh", "plan.cuh", "radix.cuh", "threshold.cuh", "topk.cu",
                         "topk.cuh"],
}


def kernel_source_hash(kernel: str = "score_kernel") -> str:
    """Hash of the CUDA sources of `kernel` (its name up to the first '<'): a
    recorded ncu traffic figure is only valid for the sources it was taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_tiles_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[kernel.split("<")[0]]):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
    except ValueError:
        return None
    for e in rec.get("entries", []):
        if e.get("kernel") == kernel and e.get("workload") == workload and \
                e.get("source_hash") == kernel_source_hash(kernel):
            return e.get("bytes_per_launch")
    return None


def smi_gpu_id(device) -> str:
    """The id under which nvidia-smi knows a torch CUDA device.  nvidia-smi
    numbers GPUs physically and ignores CUDA_VISIBLE_DEVICES, so the CUDA
    ordinal can name another GPU of the machine; the device's UUID cannot."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
    except (AttributeError, RuntimeError):
        u = ""
    if u:
        return u if u.startswith("GPU-") else f"GPU-{u}"
    idx = device.index if hasattr(device, "index") else int(device)
    return str(idx or 0)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region.
    gpu_id is what nvidia-smi's --id takes: a UUID ("GPU-...") or an index."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id, path: str | None):
        self.path = path or os.path.join("/tmp", f"idx_clocks_{os.getpid()}.csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def wait_first(self, timeout: float = 3.0):
        """Wait (at most `timeout` seconds) until the sampler has written its
        first sample, so that it is already sampling when the timed region
        starts."""
        if self.proc is None:
            return
        t0 = time.time()
        while time.time() - t0 < timeout:
            try:
                if os.path.getsize(self.path) > 0:
                    return
            except OSError:
                return
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = list(csv.reader(io.StringIO(open(self.path).read())))
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def cpu_baseline_sample(inp, target_s: float = 10.0, seed: int = 7):
    """The oracle as it stands on the host cores, over a seeded row sample
    sized to about `target_s` seconds of wall time."""
    import oracle
    import synth
    threads = oracle.default_threads()
    n_all = (inp.ke - inp.ks).clamp_min(0).long()
    probe = synth.sample_rows(inp.ks, inp.ke, min(threads, inp.rows), seed)
    t0 = time.perf_counter()
    oracle.score_topk(inp, rows=probe, nthreads=threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    per_row = dt / len(probe)
    count = int(max(len(probe), min(inp.rows, target_s / per_row)))
    rows = synth.sample_rows(inp.ks, inp.ke, count, seed + 1)
    t0 = time.perf_counter()
    oracle.score_topk(inp, rows=rows, nthreads=threads)
    wall = time.perf_counter() - t0
    pairs = int(n_all[rows].sum())
    # the oracle's selection alone on the standalone top-k workload (given scores)
    si = synth.workload("standalone_topk")
    trows = synth.sample_rows(si.ks, si.ke, 4 * threads, seed + 2)
    t0 = time.perf_counter()
    oracle.topk_from_scores(si.scores, si.ks, si.ke, si.topk, rows=trows, nthreads=threads)
    twall = time.perf_counter() - t0
    return {"value": pairs / wall, "unit": "pairs/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} seeded rows of the workload ({pairs} pairs), fp64 scores "
                      f"+ full-sort top-k, {wall:.1f} s wall",
            "core_us_per_row": wall / len(rows) * threads * 1e6,
            "standalone_topk_rows_per_s": len(trows) / twall,
            "standalone_topk_sample": f"{len(trows)} seeded rows of standalone_topk (131072 "
                                      f"scores each), full sort, {twall:.2f} s wall"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle timed on host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    import synth
    inp = synth.workload(args.workload)
    threads = oracle.default_threads()
    n_all = (inp.ke - inp.ks).clamp_min(0).long()
    per_step_rows = max(threads, 16)
    for i in range(args.warmup):
        oracle.score_topk(inp, rows=synth.sample_rows(inp.ks, inp.ke, per_step_rows, 100 + i),
                          nthreads=threads)
    times, pairs = [], 0
    for i in range(args.steps):
        rows = synth.sample_rows(inp.ks, inp.ke, per_step_rows, 1000 + i)
        t0 = time.perf_counter()
        oracle.score_topk(inp, rows=rows, nthreads=threads)
        times.append(time.perf_counter() - t0)
        pairs += int(n_all[rows].sum())
    total = sum(times)
    value = pairs / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "pairs/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(inp, args.workload),
            "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"{per_step_rows} seeded rows per step of the workload"},
            "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def slowest_ms(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank runs its own replica, the job is done
    when the last one is."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput (weak scaling): all ranks' units over the slowest time."""
    return world * units_per_rank / (ms * 1e-3)


def config_block(inp, name):
    dt = "bf16" if inp.q.dtype == torch_bf16() else "fp8 e4m3"
    return {"workload": f"{name}: rows={inp.rows} keys={inp.keys} H={inp.H} D={inp.D} "
                        f"topk={inp.topk} {dt} q/k, {inp.meta.get('ranges', 'given')} ranges",
            "rows": inp.rows, "keys": inp.keys, "heads": inp.H, "dim": inp.D, "topk": inp.topk,
            "pairs_per_step": inp.pairs(),
            "l2": "flushed between timed steps (256 MiB write + 256 MiB read, outside "
                  "the events: inputs cold, L2 clean)"}


def torch_bf16():
    import torch
    return torch.bfloat16


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch

    import synth
    import sparse_attention_indexer_tiles_gb300 as idx
    from sparse_attention_indexer_tiles_gb300 import build as _build
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk = peaks()

    if args.route_sweep:
        route_sweep(idx, dev)
        return

    if args.only == "topk":
        print(json.dumps(standalone_topk(idx, dev, L2Flush(dev), pk, args)))
        return
    if args.only == "split":
        print(json.dumps(split_topk(idx, dev, L2Flush(dev), pk, args)))
        return

    # ---------------------------------------------------------------- inputs
    inp = synth.workload(args.workload)
    if args.rows:
        inp = last_rows(inp, args.rows)
    g = {n: getattr(inp, n).to(dev) for n in ("q", "k", "k_scale", "w", "ks", "ke")}
    pairs = inp.pairs()
    out = torch.empty(inp.rows, inp.topk, dtype=torch.int32, device=dev)
    need = idx.idx_score_topk_workspace(inp.rows, inp.keys, 0, inp.H, inp.D, inp.topk,
                                        inp.q.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stats = idx.Stats(dev)

    def step(ev=None, o=None):
        opts = o or idx.Options()
        if ev is not None:
            opts.stage_events = ev.ptr
        idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk,
                           out=out, ws=ws, options=opts)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    # one checked call: the counters of the path (rescans) on this workload
    stats.reset()
    step(o=idx.make_options(None, stats))
    torch.cuda.synchronize()
    path_stats = stats.read()

    # ------------------------------------------------------------- timed loop
    evs = [idx.StageEvents(5) for _ in range(args.steps)]
    sampler = ClockSampler(smi_gpu_id(dev), args.clocks_file)
    sampler.wait_first()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = idx.idx_launch_count()
    for i in range(args.steps):
        flush.zero_()
        hold_gpu()
        step(evs[i])
    torch.cuda.synchronize()
    launches = idx.idx_launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [e.elapsed(0, 4) for e in evs]
    emit_ms = [e.elapsed(1, 2) for e in evs]
    stage_ms = {
        "sample_and_threshold": statistics.mean(e.elapsed(0, 1) for e in evs),
        "score_and_emit": statistics.mean(emit_ms),
        "slab_topk": statistics.mean(e.elapsed(2, 3) for e in evs),
        "rescan": statistics.mean(e.elapsed(3, 4) for e in evs),
    }
    ms = slowest_ms(statistics.mean(step_ms), world, dev)
    value = job_throughput(pairs, world, ms)

    # --------------------------------------------------------------- roofline
    flops = 2.0 * inp.H * inp.D * pairs
    emit_s = statistics.mean(emit_ms) * 1e-3
    # fp8 dense = 2 x bf16 dense (nominal ratio); bf16 inputs run at the bf16 peak
    bf16_in = inp.q.dtype == torch.bfloat16
    fp8_peak = pk["bf16_tflops"] * (1.0 if bf16_in else 2.0)
    achieved = flops / emit_s / 1e12
    kname = f"score_kernel<{'bf16' if bf16_in else 'fp8'},H{inp.H},D{inp.D}> emit"
    traffic = recorded_traffic(kname, args.workload)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": traffic,
                "kernel": kname + " pass",
                "algorithmic": f"2*H*D flop per visible pair = {flops:.4g} flop per launch",
                "peak_note": f"{pk['source']} bf16 {pk['bf16_tflops']} TFLOP/s"
                             f"{'' if bf16_in else ' x 2 for fp8'}"}
    whole_frac = flops / (ms * 1e-3) / 1e12 / fp8_peak

    # ------------------------------------------------------------ end to end
    # The public call on host memory: idx_score_topk_host takes page-locked host
    # inputs and returns the indices in host memory, its copies (inputs in,
    # indices out) overlapping the compute of other row chunks.
    host = {n: getattr(inp, n).contiguous().pin_memory() for n in ("q", "k", "k_scale", "w",
                                                                    "ks", "ke")}
    out_h = torch.empty(inp.rows, inp.topk, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    hws = torch.empty(idx.idx_score_topk_host_workspace(inp.rows, inp.keys, 0, inp.H, inp.D,
                                                        inp.topk, inp.q.dtype),
                      dtype=torch.uint8, device=dev)

    def host_step():
        idx.idx_score_topk_host(host["q"], host["k"], host["k_scale"], host["w"], host["ks"],
                                host["ke"], inp.topk, out=out_h, ws=hws, stream=stream)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms = []
    for i in range(e2e_steps + 2):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        host_step()
        b.record(stream)
        b.synchronize()
        if i >= 2:
            e2e_ms.append(a.elapsed_time(b))
    e2e_same = bool(torch.equal(out_h, out.cpu()))
    e2e_val = pairs / (statistics.mean(e2e_ms) * 1e-3) * world
    del hws

    line = {"metric": METRIC, "value": value, "unit": "pairs/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if bf16_in else "e4m3", "data": "synthetic",
            "config": config_block(inp, args.workload),
            "roofline": roofline, "whole_step_tensor_frac": whole_frac,
            "stage_ms": stage_ms, "path_stats": path_stats,
            "e2e": {"value": e2e_val, "unit": "pairs/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": statistics.mean(e2e_ms),
                    "call": "idx_score_topk_host (page-locked host inputs and output)",
                    "identical_to_device_call": e2e_same},
            "gpu_launches": launches, "clocks": clocks}

    # ------------------------------------------------------ secondary numbers
    if not args.no_extra and rank == 0:
        line["extra"] = secondary(idx, dev, g, inp, out, ws, flush, pk, args, ms)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(inp)
    if "extra" in line:
        # the headline figures of the other workloads, last on the line
        line.update(summary(line))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def summary(line):
    """One short entry per measured workload, for the end of the JSON line:
    the standalone top-k (rows/s, fraction of the HBM copy peak), each fused
    workload's whole call against the fp8 tensor peak, and the fused over
    two-pass speed-ups."""
    ex = line["extra"]
    st = ex["standalone_topk"]
    out = {"standalone_topk": {"rows_per_s": st["rows_per_s"], "ms": st["ms"],
                               "hbm_frac": st["roofline"]["frac"],
                               "workload": st["workload"].split(",")[0]},
           "fused_prefill": {"pairs_per_s": line["value"], "ms": line["ms_per_step"],
                             "whole_call_tensor_frac": line["whole_step_tensor_frac"],
                             "emit_tensor_frac": line["roofline"]["frac"],
                             "fused_over_two_pass": ex["two_pass"]["fused_over_two_pass"]}}
    for name in ("long_context", "mixed_batch", "decode"):
        w = ex.get(name)
        if not w:
            continue
        out[name] = {"pairs_per_s": w["pairs_per_s"], "ms": w["ms"],
                     "whole_call_tensor_frac": w["whole_call_tensor_frac"],
                     "emit_tensor_frac": w["emit_roofline"]["frac"],
                     "fused_over_two_pass": w.get("two_pass", {}).get("fused_over_two_pass"),
                     "fallback_rows": w["path_stats"]["fallback_rows"]}
    sp = ex["split_topk"]
    out["split_topk"] = {"rows_per_s": sp["rows_per_s"], "ms": sp["ms"],
                         "hbm_frac": sp["roofline"]["frac"]}
    mx = ex.get("mxfp4")
    if mx:
        out["mxfp4"] = {"pairs_per_s": mx["pairs_per_s"], "ms": mx["ms"],
                        "whole_call_tensor_frac": mx["whole_call_tensor_frac"],
                        "emit_tensor_frac": mx["emit_roofline"]["frac"]}
    return {"summary": out}


def last_rows(inp, n):
    """The last n query rows of a workload (same keys): a smaller case of the
    same kernel for profiling."""
    import synth
    return synth.IndexerInputs(q=inp.q[-n:].contiguous(), k=inp.k, k_scale=inp.k_scale,
                               w=inp.w[-n:].contiguous(), ks=inp.ks[-n:].contiguous(),
                               ke=inp.ke[-n:].contiguous(), topk=inp.topk, meta=inp.meta)


class L2Flush:
    """Before each timed call: write a 256 MiB buffer, so the 129 MB L2 keeps
    no line of the previous call, then read another 256 MiB, so the write's
    dirty lines go back to HBM now and not inside the next timed region."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(32 << 20, dtype=torch.int64, device=dev)
        self.acc = torch.empty((), dtype=torch.int64, device=dev)

    def zero_(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


def hold_gpu():
    """Keep the stream busy (~50 us spin) while the host issues the next
    call, so that the events around a short launch time the device work and
    not the binding's host overhead (the end-to-end figures include that)."""
    import torch
    torch.cuda._sleep(100_000)


def timed(fn, flush, reps):
    import torch
    ts = []
    for _ in range(reps):
        flush.zero_()
        hold_gpu()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def two_pass(idx, dev, g, inp, out, flush, reps=5):
    """The two-pass baseline on a workload: materialise the fp32 logits
    [rows, longest visible range], then their exact top-k; timed separately,
    L2 flushed before each, and checked against the fused path's indices."""
    import torch
    n_max = int((inp.ke - inp.ks).max())
    S = torch.empty(inp.rows, n_max, dtype=torch.float32, device=dev)
    out2 = torch.empty_like(out)
    rel = idx.Options(relative_rows=1)
    need = idx.idx_topk_workspace(inp.rows, n_max, inp.topk, rel)
    tws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def mat():
        idx.idx_score_materialise(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], out=S)

    def tk():
        idx.idx_topk_from_scores(S, g["ks"], g["ke"], inp.topk, out=out2, ws=tws, options=rel)

    for _ in range(2):
        mat()
        tk()
    t_mat = timed(mat, flush, reps)
    t_tk = timed(tk, flush, reps)
    identical = bool(torch.equal(out, out2))
    del S, out2, tws
    torch.cuda.empty_cache()
    flops = 2.0 * inp.H * inp.D * inp.pairs()
    return {"materialise_ms": t_mat, "topk_ms": t_tk, "total_ms": t_mat + t_tk,
            "identical_indices": identical,
            "logits_bytes": 4 * inp.rows * n_max,
            "materialise_tflops": flops / (t_mat * 1e-3) / 1e12}


def secondary(idx, dev, g, inp, out, ws, flush, pk, args, fused_ms):
    """Standalone top-k rows/s (HBM roofline), the row split, the other fused
    workloads (with their two-pass baselines), a decode-shaped call, the tiny
    workload and the page-table transform."""
    import torch
    import synth
    res = {}
    tp = two_pass(idx, dev, g, inp, out, flush)
    tp["fused_over_two_pass"] = tp["total_ms"] / fused_ms
    res["two_pass"] = tp
    res["split_topk"] = split_topk(idx, dev, flush, pk, args)
    res["long_context"] = other_fused(idx, dev, flush, pk, args, "long_context", with_two_pass=True)
    torch.cuda.empty_cache()
    res["mixed_batch"] = other_fused(idx, dev, flush, pk, args, "mixed_batch", with_two_pass=True)
    torch.cuda.empty_cache()
    dec = synth.indexer_inputs(16, 1 << 20, 32, 128, 2048, "fp8", seed=6, ranges="full")
    res["decode"] = other_fused(idx, dev, flush, pk, args, "decode", inp=dec, with_two_pass=True)
    torch.cuda.empty_cache()
    res["tiny"] = other_fused(idx, dev, flush, pk, args, "tiny")
    res["mxfp4"] = mxfp4_fused(idx, dev, flush, pk, args)
    torch.cuda.empty_cache()
    res["page_table_transform"] = page_transform(idx, dev, flush, pk, out, inp)
    res["standalone_topk"] = standalone_topk(idx, dev, flush, pk, args)
    return res


def page_transform(idx, dev, flush, pk, out, inp):
    """idx_page_table_transform on the fused step's output (rows x topk), one
    request of keys / 64 pages: HBM roofline on 8 B per entry."""
    import torch
    import synth
    table, row_map = synth.paged_layout(1, (inp.keys + 63) // 64, inp.rows, seed=77)
    table, row_map = table.to(dev), row_map.to(dev)
    work = torch.empty_like(out)
    ts = []
    for it in range(13):
        work.copy_(out)
        flush.zero_()
        hold_gpu()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        idx.idx_page_table_transform(work, table, 64, row_map=row_map)
        b.record()
        b.synchronize()
        if it >= 3:
            ts.append(a.elapsed_time(b))
    ms = statistics.mean(ts)
    nbytes = 8 * out.numel()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"fused_prefill output: rows={out.shape[0]} topk={out.shape[1]}, page 64",
            "ms": ms, "entries_per_s": out.numel() / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "algorithmic": f"4 B read + 4 B written per entry = {nbytes} B"}}


def route_sweep(idx, dev):
    """Fused vs two-pass (materialise + top-k) over key lengths around the
    routing gate: 4096 causal rows of e4m3 q/k, H 64 / 32, topk 2048 / 512."""
    import torch
    import synth
    flush = L2Flush(dev)
    for H, topk in ((64, 2048), (32, 2048), (64, 512)):
        for keys in (4096, 6144, 8192, 12288, 16384, 24576, 32768, 65536):
            rows = 4096
            inp = synth.indexer_inputs(rows, keys, H, 128, topk, "fp8", seed=90)
            g = {n: getattr(inp, n).to(dev) for n in ("q", "k", "k_scale", "w", "ks", "ke")}
            out = torch.empty(rows, topk, dtype=torch.int32, device=dev)
            out2 = torch.empty_like(out)
            need = idx.idx_score_topk_workspace(rows, keys, 0, H, 128, topk, inp.q.dtype)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            S = torch.empty(rows, int((inp.ke - inp.ks).max()), dtype=torch.float32, device=dev)
            rel = idx.Options(relative_rows=1)

            def fused():
                idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], topk,
                                   out=out, ws=ws)

            def two_pass():
                idx.idx_score_materialise(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"],
                                          out=S)
                idx.idx_topk_from_scores(S, g["ks"], g["ke"], topk, out=out2, options=rel)

            for _ in range(2):
                fused()
                two_pass()
            tf, tt = timed(fused, flush, 6), timed(two_pass, flush, 6)
            print(json.dumps({"H": H, "topk": topk, "rows": rows, "keys": keys,
                              "fused_ms": tf, "two_pass_ms": tt, "two_pass_over_fused": tt / tf,
                              "identical": bool(torch.equal(out, out2)),
                              "gate_fused": idx.idx_route_fused(rows, keys, topk)}), flush=True)
            del S, g, inp
            torch.cuda.empty_cache()


def other_fused(idx, dev, flush, pk, args, name, inp=None, with_two_pass=False):
    """idx_score_topk on another fused workload: whole-call pairs/s and the
    emit pass against the fp8 tensor peak, with the path counters (and the
    two-pass baseline on the same inputs when asked)."""
    import torch
    import synth
    inp = inp if inp is not None else synth.workload(name)
    g = {n: getattr(inp, n).to(dev) for n in ("q", "k", "k_scale", "w", "ks", "ke")}
    out = torch.empty(inp.rows, inp.topk, dtype=torch.int32, device=dev)
    need = idx.idx_score_topk_workspace(inp.rows, inp.keys, 0, inp.H, inp.D, inp.topk,
                                        inp.q.dtype)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    stats = idx.Stats(dev)

    def call(ev=None, o=None):
        opts = o or idx.Options()
        if ev is not None:
            opts.stage_events = ev.ptr
        idx.idx_score_topk(g["q"], g["k"], g["k_scale"], g["w"], g["ks"], g["ke"], inp.topk,
                           out=out, ws=ws, options=opts)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    stats.reset()
    call(o=idx.make_options(None, stats))
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 5))
    evs = [idx.StageEvents(5) for _ in range(reps)]
    for e in evs:
        flush.zero_()
        hold_gpu()
        call(e)
    torch.cuda.synchronize()
    ms = statistics.mean(e.elapsed(0, 4) for e in evs)
    emit_ms = statistics.mean(e.elapsed(1, 2) for e in evs)
    pairs = inp.pairs()
    flops = 2.0 * inp.H * inp.D * pairs
    # fp8 dense = 2 x bf16 dense (nominal ratio); bf16 inputs run at the bf16 peak
    peak = pk["bf16_tflops"] * (1.0 if inp.q.dtype == torch.bfloat16 else 2.0)
    emit_tf = flops / (emit_ms * 1e-3) / 1e12
    res = {"workload": f"{name}: rows={inp.rows} keys={inp.keys} H={inp.H} D={inp.D} "
                       f"topk={inp.topk}",
           "pairs_per_s": pairs / (ms * 1e-3), "rows_per_s": inp.rows / (ms * 1e-3), "ms": ms,
            "stage_ms": {"sample_and_threshold": statistics.mean(e.elapsed(0, 1) for e in evs),
                         "score_and_emit": emit_ms,
                         "slab_topk": statistics.mean(e.elapsed(2, 3) for e in evs),
                         "rescan": statistics.mean(e.elapsed(3, 4) for e in evs)},
            "emit_roofline": {"bound": "tensor", "achieved": emit_tf, "peak": peak,
                              "unit": "TFLOP/s", "frac": emit_tf / peak},
            "whole_call_tensor_frac": flops / (ms * 1e-3) / 1e12 / peak,
            "path_stats": stats.read()}
    if with_two_pass:
        tp = two_pass(idx, dev, g, inp, out, flush, reps=3)
        tp["fused_over_two_pass"] = tp["total_ms"] / ms
        res["two_pass"] = tp
    return res


def mxfp4_fused(idx, dev, flush, pk, args):
    """idx_score_topk_mxfp4 on the fused-prefill shape with MXFP4 q/k (e2m1 +
    e8m0 block scales): the whole call (the exact expansion to e4m3 included)
    and its emit pass, whose MMAs run on e4m3 operands, against the fp8 peak."""
    import torch
    import synth
    inp = synth.indexer_inputs(4096, 65536, 64, 128, 2048, "mxfp4", seed=2)
    g = {n: getattr(inp, n).to(dev) for n in ("q", "q_sf", "k", "k_sf", "k_scale", "w", "ks",
                                              "ke")}
    out = torch.empty(inp.rows, inp.topk, dtype=torch.int32, device=dev)
    need = int(idx.load().idx_score_topk_mxfp4_workspace(inp.rows, inp.keys, 0, inp.H, inp.D,
                                                         inp.topk, None))
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def call(ev=None):
        o = idx.Options()
        if ev is not None:
            o.stage_events = ev.ptr
        idx.idx_score_topk_mxfp4(g["q"], g["q_sf"], g["k"], g["k_sf"], g["k_scale"], g["w"],
                                 g["ks"], g["ke"], inp.topk, out=out, ws=ws, options=o)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 5))
    evs = [idx.StageEvents(5) for _ in range(reps)]
    ts = []
    for e in evs:
        flush.zero_()
        hold_gpu()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        call(e)
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.mean(ts)
    emit_ms = statistics.mean(e.elapsed(1, 2) for e in evs)
    pairs = inp.pairs()
    flops = 2.0 * inp.H * inp.D * pairs
    fp8_peak = pk["bf16_tflops"] * 2.0
    emit_tf = flops / (emit_ms * 1e-3) / 1e12
    return {"workload": f"mxfp4: rows={inp.rows} keys={inp.keys} H={inp.H} D={inp.D} "
                        f"topk={inp.topk}, e2m1 + e8m0 q/k, causal ranges",
            "ms": ms, "pairs_per_s": pairs / (ms * 1e-3),
            "expand_ms": ms - statistics.mean(e.elapsed(0, 4) for e in evs),
            "emit_roofline": {"bound": "tensor", "achieved": emit_tf, "peak": fp8_peak,
                              "unit": "TFLOP/s", "frac": emit_tf / fp8_peak,
                              "note": "MMAs on the exactly expanded e4m3 operands: fp8 peak "
                                      "(measured bf16 x 2); the nominal fp4 dense rate is "
                                      "twice that"},
            "whole_call_tensor_frac": flops / (ms * 1e-3) / 1e12 / fp8_peak}


def split_topk(idx, dev, flush, pk, args):
    """idx_topk_from_scores on 8 rows x 1M keys: low batch, long rows, the row split
    path (g blocks per row)."""
    import torch
    import synth
    si = synth.workload("split_topk")
    sc = si.scores.to(dev)
    ks, ke = si.ks.to(dev), si.ke.to(dev)
    o = torch.empty(si.rows, si.topk, dtype=torch.int32, device=dev)
    need = idx.idx_topk_workspace(si.rows, si.stride, si.topk)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def st():
        idx.idx_topk_from_scores(sc, ks, ke, si.topk, out=o, ws=ws)

    for _ in range(args.warmup):
        st()
    t = timed(st, flush, max(5, args.steps))
    bytes_alg = 4 * int((si.ke - si.ks).sum()) + 4 * si.rows * si.topk
    gbs = bytes_alg / (t * 1e-3) / 1e9
    return {"workload": "split_topk: rows=8 keys=1048576 topk=2048 (row split)",
            "rows_per_s": si.rows / (t * 1e-3), "ms": t,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"]}}


def standalone_topk(idx, dev, flush, pk, args):
    """idx_topk_from_scores on 1024 rows x 131072 fp32 scores, topk 2048."""
    import torch
    import synth
    si = synth.workload("standalone_topk")
    sc = si.scores.to(dev)
    ks, ke = si.ks.to(dev), si.ke.to(dev)
    o3 = torch.empty(si.rows, si.topk, dtype=torch.int32, device=dev)
    need = idx.idx_topk_workspace(si.rows, si.stride, si.topk)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    def st():
        idx.idx_topk_from_scores(sc, ks, ke, si.topk, out=o3, ws=ws)

    for _ in range(args.warmup):
        st()
    t_st = timed(st, flush, max(5, args.steps))
    vis = int((si.ke - si.ks).sum())
    bytes_alg = 4 * vis + 4 * si.rows * si.topk
    gbs = bytes_alg / (t_st * 1e-3) / 1e9
    return {
        "workload": "standalone_topk: rows=1024 keys=131072 topk=2048, fp32 N(0,0.05) on the "
                    "bf16 grid, 5% rows shorter than topk",
        "rows_per_s": si.rows / (t_st * 1e-3), "ms": t_st,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / pk["hbm_gbs"], "traffic": recorded_traffic(
                         "topk_rows_kernel", "standalone_topk"),
                     "algorithmic": f"4 B per visible score + 4 B per output = {bytes_alg} B"}}

if __name__ == "__main__":
    main()
