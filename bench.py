"""Benchmark of the CVR scoring path on GB300: candidates scored per second, request latency, roofline.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config prod] [--impl reference]

A step is one cvr_score call over one full batch of the workload (all stages of the forward pass:
embedding bags, sequence encoders, tokeniser, Query Decoding, Token Mixer, PLE with the heads), inputs
resident in HBM, L2 flushed (256 MB write) before every step and each step timed alone with CUDA
events on the scorer's stream. ``e2e`` repeats the measurement through cvr_score_host with pinned
host buffers, which the kernels read (inputs) and write (output) in place over the C2C link inside the
timed region. ``roofline`` is the
dominant kernel's algorithmic FLOPs per launch over its event-timed duration. ``cpu_baseline`` times
the CPU oracle on a bounded sample of the same workload. ``--impl reference`` times that oracle
alone (the method has no other runnable reference implementation).

Under torchrun every rank scores its own replica of the batch (requests are independent: weak
scaling, no collective on the data path); rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
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

METRIC = "candidates scored/sec and p50 request latency on 1 GB300; % of roofline"
UNIT = "candidates/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------------------------------------
# algorithmic work (user side once per request, K/V and mean-pool once per request)
def algorithmic_work(wl, nnz: int, seq_events=None):
    """FLOPs per step and bytes; ``seq_events`` = the real sequence events of the batch per request (variable
    lengths), default every slot."""
    D, H = 128, 256
    R, B, NL = wl.n_req, wl.n_cand, wl.n_layers
    SL = wl.sum_len if seq_events is None else seq_events
    swiglu_row = 2 * D * 2 * H + 2 * H * D                       # 196,608 FLOP per row
    flops = {
        "seq_mlp": R * SL * swiglu_row,
        "request_side": R * 2 * 256 * 1664 + NL * R * 3 * 2 * D * D,
        "tokenizer": B * 2 * 256 * 1664,
        "query": NL * B * 2 * 1664 * 384,
        "attention": NL * B * 4 * D * SL,                        # q.k and p.v: 2 * 2 * 128 per position
        "token_mixer": NL * B * 16 * swiglu_row,
        # PLE experts and gates, then per task the heads 256->128 and 128->1 (one kernel)
        "ple_heads": B * 2 * 2048 * (768 + 6) + B * 2 * 2 * (256 * 128 + 128),
    }
    bf16_weights = (1664 * 512 + 3 * (512 * 128 + 128 * 256) + NL * (3 * 128 * 1792 + 512 * 128 + 128 * 256)
                    + 774 * 2048 + 2 * 128 * 256) * 2
    gathered = nnz * 128 + R * SL * 4 * 128                      # fp32 rows of 32
    ids = nnz * 8 + R * SL * 4 * 8 + (R * 8 + B * 8 + 1) * 8 + B * 4
    total_bytes = gathered + ids + bf16_weights + B * 8
    sparse_bytes = gathered + ids + (R * 256 + B * 256 + R * SL * 128) * 2   # + bf16 outputs written
    return flops, total_bytes, sparse_bytes


def source_digest(rel_path: str) -> str:
    import hashlib
    p = os.path.join(ROOT, rel_path)
    if not os.path.exists(p):
        return ""
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ---------------------------------------------------------------------------------------------
# multi-rank host logic (one process per GPU; every rank scores its own batch, no data-path collective)
def workload_for_rank(cfg_name: str, rank: int, **over):
    """Rank 0 scores the configuration's own batch; rank r > 0 an independent batch of the same shape
    (the configuration's seed + 7919 r)."""
    import synth
    if rank == 0:
        return synth.make_workload(cfg_name, **over)
    return synth.make_workload(cfg_name, seed=synth.default_seed(cfg_name) + 7919 * rank, **over)


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    import torch
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, batch: int, steps: int, total_ms: float) -> float:
    """Candidates per second of the whole job: every rank's batches over the slowest rank's time."""
    return world * batch * steps / (total_ms / 1e3)


def measured_traffic(config: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when there is none for this kernel
    and workload or the kernel's source has changed since the counters were taken."""
    tr = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tr):
        return None
    with open(tr) as f:
        ent = json.load(f).get(f"{config}:{kernel}")
    if ent and source_digest(ent["source"]) == ent["source_sha256_16"]:
        return ent["bytes_per_launch"]
    return None


# ---------------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 20 ms) around the timed region.

    A timed region of a few ms holds one sample at best, so the same steps go on (``soak``) for about a
    second right after it, under the same sampler: the clock record covers the timed region and that window
    of identical work, and says how many samples fell inside each."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t_timed_end = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu=timestamp,{self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        self.t0 = time.time()
        return self

    def mark_timed_end(self):
        """End of the timed region (what follows until exit is the soak window)."""
        self.t_timed_end = time.time()

    def __exit__(self, *exc):
        self.t1 = time.time()
        if self.t_timed_end is None:
            self.t_timed_end = self.t1
        time.sleep(0.1)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        """Median SM clock and the throttle reasons seen among the samples taken inside the timed region and
        the soak window after it (all samples if none falls inside them)."""
        from datetime import datetime
        if not self.proc or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows, inside, timed = [], [], 0
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                row = (float(parts[2]), float(parts[3]), parts[6:10])
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append(row)
            if self.t0 <= ts <= self.t1:
                inside.append(row)
                timed += ts <= self.t_timed_end
        os.unlink(self.path)
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in use for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in use), "sm_max_mhz": max(r[1] for r in use),
                "sm_mhz_min": min(r[0] for r in use), "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": timed, "samples_in_soak": len(inside) - timed,
                "timed_region_s": round(self.t_timed_end - self.t0, 4),
                "soak_s": round(self.t1 - self.t_timed_end, 3),
                "window": "timed region, then the same steps repeated for the soak window"}


# ---------------------------------------------------------------------------------------------
def oracle_baseline(cfg_name: str, budget_s: float = 10.0):
    """The CPU oracle, as it stands, on a bounded sample of the workload: the benchmark's own batch,
    scored again until about budget_s seconds of CPU work have been spent."""
    import oracle
    import synth
    threads = oracle.threads_used(0)
    wl = synth.make_workload(cfg_name)
    w = synth.make_weights(wl.n_layers, wl.seed)
    reps, t = 0, 0.0
    while t < budget_s and reps < 100:
        t0 = time.perf_counter()
        oracle.score(wl, w)
        t += time.perf_counter() - t0
        reps += 1
    return {"value": reps * wl.n_cand / t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the {cfg_name} batch ({wl.n_req} requests x {wl.n_cand // wl.n_req} candidates) scored "
                      f"{reps} times by the fp64 loop-nest oracle (OpenMP over candidates), {t:.1f} s wall"}


def run_reference(args):
    import oracle
    import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = oracle.threads_used(0)
    # per-step sample sized so that warmup + steps take ~2 minutes
    wl = synth.make_workload(args.config, n_req=1, n_cand=8)
    w = synth.make_weights(wl.n_layers, wl.seed)
    t0 = time.perf_counter()
    oracle.score(wl, w)
    per = (time.perf_counter() - t0) / 8
    total_steps = max(1, args.steps + args.warmup)
    n = int(max(8, min(512, 120.0 / total_steps / max(per, 1e-6))))
    wl = synth.make_workload(args.config, n_req=1, n_cand=n)
    w = synth.make_weights(wl.n_layers, wl.seed)
    for _ in range(args.warmup):
        oracle.score(wl, w)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.score(wl, w)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * args.steps / tot
    p50 = statistics.median(times) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.config} shapes, 1 request x {n} candidates per step (CPU oracle)"},
            "p50_ms": p50,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"1 request x {n} candidates of the {args.config} workload per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------------------------
def gather_roofline(dev: str, stream, flush, peak_bw: float, n_steps: int = 50):
    """The embedding gathers on a workload where they move enough bytes to be bandwidth-bound: deep, 32
    requests x 2048 candidates (a1-a3: 1.2 M bag ids and 115 k sequence events, ~340 MB of algorithmic bytes).
    The sparse kernel's time comes from the events the scorer records after each kernel (profiling on), L2
    flushed before every step."""
    import torch

    import cvr_ranking_model_gb300 as cvr
    import synth
    from synth.harness import DeviceWorkload, make_scorer
    wl = synth.make_workload("deep", n_cand=2048)
    w = synth.make_weights(wl.n_layers, synth.default_seed("deep"))
    with torch.cuda.stream(stream):
        dw = DeviceWorkload(wl, device=dev)
    torch.cuda.synchronize(dev)
    sc = make_scorer(dw, w, stream=stream.cuda_stream)
    sc.set_option(cvr.OPT_PROFILE, 1)
    r, b, o, s, out = dw.ptrs()
    ms = []
    with torch.cuda.stream(stream):
        for i in range(3 + n_steps):
            flush.zero_()
            sc.score(wl.n_req, wl.n_cand, r, b, o, s, out)
            if i >= 3:
                ms.append(sum(t for name, t in sc.stage_list() if name == "sparse"))
    sc.close()
    nnz = int(wl.bag_offsets[-1])
    _, _, sparse_bytes = algorithmic_work(wl, nnz)
    t = statistics.median(ms)
    gbs = sparse_bytes / (t / 1e3) / 1e9
    return {"kernel": "sparse", "workload": f"deep: R={wl.n_req} x C=2048, L={'/'.join(map(str, wl.seq_len))}, "
                                           f"{nnz} bag ids, tables 100000/1000000 rows",
            "bound": "hbm", "achieved": gbs, "peak": peak_bw, "unit": "GB/s", "frac": gbs / peak_bw,
            "bytes_per_launch": sparse_bytes, "launch_ms": t, "traffic": measured_traffic("deep2048", "sparse"),
            "timing": f"median of {n_steps} launches, events after each kernel, L2 flushed before each step"}


def run_timeline(args):
    """Per-CTA timeline of one synchronous call (L2 flushed, the GPU idle before it) from the diagnostic build with
    per-CTA timestamps (cvr_timeline): for every kernel, when its CTAs started, when their wait for the previous
    kernel's data returned and when they finished, in microseconds from the first CTA of the call. Median of 5 calls
    per figure. Prints a table, not a benchmark line."""
    os.environ["CVR_TIMELINE"] = "1"
    import torch

    import cvr_ranking_model_gb300._build as cvr_build
    cvr_build.LIB = cvr_build.LIB_TIMELINE
    cvr_build.build(timeline=True)
    import cvr_ranking_model_gb300 as cvr
    import synth
    from synth.harness import DeviceWorkload, make_scorer
    wl = synth.make_workload(args.config, n_cand=args.n_cand)
    w = synth.make_weights(wl.n_layers, synth.default_seed(args.config))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dw = DeviceWorkload(wl)
    torch.cuda.synchronize()
    sc = make_scorer(dw, w, stream=stream.cuda_stream)
    r, b, o, s, out = dw.ptrs()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    reps = []
    with torch.cuda.stream(stream):
        for rep in range(5 + args.warmup):
            flush.zero_()
            torch.cuda.synchronize()
            sc.timeline(clear=True)
            sc.score(wl.n_req, wl.n_cand, r, b, o, s, out)
            if rep >= args.warmup:
                reps.append(sc.timeline(clear=False).astype(np.int64))
    rows = {}
    for t in reps:
        t0 = t[:, :, 0][t[:, :, 0] > 0].min()
        for k, name in enumerate(cvr.binding.TIMELINE_KERNELS):
            e = t[k]
            m = e[:, 0] > 0
            if not m.any():
                continue
            st, en = (e[m, 0] - t0) / 1e3, (e[m, 2] - t0) / 1e3
            wd = (e[m, 1][e[m, 1] > 0] - t0) / 1e3
            rows.setdefault(name, []).append((int(m.sum()), st.min(), np.median(st), st.max(),
                                               np.median(wd) if len(wd) else float("nan"), np.median(en), en.max()))
    print(f"timeline of one {args.config} call (us from the first CTA; median of {len(reps)} calls)")
    print(f"{'kernel':13s} {'CTAs':>5s} {'start min':>9s} {'start med':>9s} {'start max':>9s} {'wait med':>9s} "
          f"{'end med':>9s} {'end max':>9s}")
    for name, lst in sorted(rows.items(), key=lambda kv: np.median([x[1] for x in kv[1]])):
        v = np.median(np.array(lst), axis=0)
        print(f"{name:13s} {int(v[0]):5d} " + " ".join(f"{x:9.2f}" for x in v[1:]))
    sc.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="prod", choices=["tiny", "prod", "longseq", "embheavy", "deep"])
    ap.add_argument("--n-cand", type=int, default=None, help="candidates per request (deep sweep)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-gather", action="store_true", help="skip the embedding-gather roofline on deep C=2048")
    ap.add_argument("--timeline", action="store_true",
                    help="print the per-CTA timeline of one call (diagnostic build with per-CTA timestamps), no bench line")
    ap.add_argument("--minimal", action="store_true",
                    help="warm-up and timed steps only (for profiler captures): no clock soak, latency loops, "
                         "per-kernel region, end-to-end leg, gather roofline or CPU baseline")
    ap.add_argument("--ple-int8", action="store_true",
                    help="time the PLE on 8-bit weights (CVR_OPT_PLE_INT8) in the headline region as well")
    ap.add_argument("--attention-tc", action="store_true",
                    help="time the cross-attention on its tcgen05 kernel (CVR_OPT_ATTENTION_TC) in the headline region")
    ap.add_argument("--varlen", action="store_true",
                    help="variable-length sequences: every request's length per group uniform in [1, L_g]")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.minimal:
        args.no_cpu_baseline = args.no_e2e = args.no_gather = True
    if args.impl == "reference":
        run_reference(args)
        return
    if args.timeline:
        run_timeline(args)
        return

    import torch
    import torch.distributed as dist

    import cvr_ranking_model_gb300 as cvr
    import synth
    from synth.harness import DeviceWorkload, make_scorer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    stream = torch.cuda.Stream(device=dev)

    wl = workload_for_rank(args.config, rank, n_cand=args.n_cand)
    w = synth.make_weights(wl.n_layers, synth.default_seed(args.config))  # one model, every replica
    with torch.cuda.stream(stream):
        dw = DeviceWorkload(wl, device=dev)
    torch.cuda.synchronize(dev)
    sc = make_scorer(dw, w, stream=stream.cuda_stream)
    sc.set_option(cvr.OPT_CUDA_GRAPH, 1)
    sc.set_option(cvr.OPT_PLE_INT8, int(args.ple_int8))
    sc.set_option(cvr.OPT_ATTENTION_TC, int(args.attention_tc))
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    r, b, o, s, out = dw.ptrs()
    B = wl.n_cand
    lens = d_lens = None
    if args.varlen:
        lens = synth.make_seq_lens(wl, min_len=1)
        d_lens = torch.from_numpy(lens).to(dev)

    def step():
        if args.varlen:
            sc.score_varlen(wl.n_req, B, r, b, o, s, d_lens.data_ptr(), out)
        else:
            sc.score(wl.n_req, B, r, b, o, s, out)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step()
    torch.cuda.synchronize(dev)

    def timed_region(profile: bool, n_steps: int):
        """K steps, L2 flushed before each, each step bracketed by CUDA events on the scorer's stream.

        Without profiling the steps are enqueued back to back through cvr_score_async (the host runs ahead;
        one cvr_sync at the end checks every step's device-side status), so each event pair times the GPU
        work of one batch alone. With profiling (an event after every kernel inside the graph, read back
        after each call) the steps are synchronous calls."""
        sc.set_option(cvr.OPT_PROFILE, int(profile))
        with torch.cuda.stream(stream):   # recapture the graph for this mode before timing
            for _ in range(3):
                flush.zero_()
                step()
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        stages, n_launch = {}, 0
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            for i in range(n_steps):
                flush.zero_()
                starts[i].record(stream)
                if profile:
                    step()
                    for name, ms in sc.stage_list():
                        stages.setdefault(name, []).append(ms)
                elif args.varlen:
                    sc.score_varlen_async(wl.n_req, B, r, b, o, s, d_lens.data_ptr(), out)
                else:
                    sc.score_async(wl.n_req, B, r, b, o, s, out)
                ends[i].record(stream)
                n_launch += sc.last_launch_count()
            if not profile:
                sc.sync()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        return [starts[i].elapsed_time(ends[i]) for i in range(n_steps)], stages, n_launch

    # timed region: the scoring calls alone (no per-kernel events inside the graph); then the same steps for
    # about a second more under the clock sampler (the soak window), which is not timed
    with ClockSampler(local) as clocks:
        step_ms, _, launches = timed_region(profile=False, n_steps=args.steps)
        clocks.mark_timed_end()
        t_soak = time.time()
        with torch.cuda.stream(stream):
            while not args.minimal and time.time() - t_soak < 1.0:
                for _ in range(50):
                    flush.zero_()
                    if args.varlen:
                        sc.score_varlen_async(wl.n_req, B, r, b, o, s, d_lens.data_ptr(), out)
                    else:
                        sc.score_async(wl.n_req, B, r, b, o, s, out)
                sc.sync()
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dev)
    # second timed region, same steps, with an event recorded after every kernel: per-kernel durations
    n_prof = min(args.steps, 1000)
    prof_ms, stage_sum = [float("nan")], {}
    if not args.minimal:
        prof_ms, stage_sum, _ = timed_region(profile=True, n_steps=n_prof)
    # request latency as the caller sees it: host wall clock around the synchronous call (argument checks, graph
    # launch, the wait and the error-word read), the GPU idle and L2 flushed before each call; 500 calls after
    # 50 warm-up calls, for the batch and for a single request of the same shape (R = 1, same C)
    def call_latency(n_req, n_cand, ptrs, n_calls=500, n_warm=50):
        rr, bb, oo, ss, oo_out = ptrs
        sc.set_option(cvr.OPT_PROFILE, 0)
        ms = []
        with torch.cuda.stream(stream):
            for i in range(n_warm + n_calls):
                flush.zero_()
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                sc.score(n_req, n_cand, rr, bb, oo, ss, oo_out)
                if i >= n_warm:
                    ms.append((time.perf_counter() - t0) * 1e3)
        return ms

    call_ms = call_latency(wl.n_req, B, (r, b, o, s, out)) if not (args.varlen or args.minimal) else []
    r1 = None
    if not (args.varlen or args.minimal):
        wl1 = synth.make_workload(args.config, n_req=1, n_cand=args.n_cand)
        with torch.cuda.stream(stream):
            dw1 = DeviceWorkload(wl1, device=dev, tables=dw.tables)
        torch.cuda.synchronize(dev)
        r1_ms = call_latency(1, wl1.n_cand, dw1.ptrs())
        r1 = {"n_req": 1, "n_cand": wl1.n_cand, "p50_ms": statistics.median(r1_ms),
              "p99_ms": float(np.percentile(r1_ms, 99)),
              "what": "synchronous cvr_score call, host wall clock, 500 calls after 50 warm-up, L2 flushed"}
    value = job_throughput(world, B, args.steps, total_ms)

    # per-kernel times (events recorded between the kernels, on the scorer's stream, every timed step)
    per_kernel = {}
    for name, lst in stage_sum.items():
        # a name repeats once per layer; stage_list already returns every launch -> group per step
        per_kernel[name] = sum(lst) / n_prof
    nnz = int(wl.bag_offsets[-1])
    seq_events = None if lens is None else float(lens.sum()) / wl.n_req
    flops, total_bytes, sparse_bytes = algorithmic_work(wl, nnz, seq_events)
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks["bf16_tflops"])
    peak_bw = float(peaks["hbm_gbs"])
    gemm_like = {k: v for k, v in per_kernel.items() if k in flops and k != "attention"}
    dom = max(gemm_like, key=lambda k: gemm_like[k]) if gemm_like else None
    launches_per_kernel = {"query": wl.n_layers, "attention": wl.n_layers, "token_mixer": wl.n_layers}
    roofline = None
    if dom:
        n_l = launches_per_kernel.get(dom, 1)
        avg_launch_ms = per_kernel[dom] / n_l
        ach = flops[dom] / n_l / (avg_launch_ms / 1e3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": ach / peak_tf, "traffic": None,
                    "peak_source": f"{peak_src} bf16 dense burst (cuBLAS)",
                    "flop_per_launch": flops[dom] / n_l, "launch_ms": avg_launch_ms}
        roofline["traffic"] = measured_traffic(args.config, dom)
    sparse = None
    if "sparse" in per_kernel:
        gbs = sparse_bytes / (per_kernel["sparse"] / 1e3) / 1e9
        sparse = {"kernel": "sparse", "bound": "hbm", "achieved": gbs, "peak": peak_bw, "unit": "GB/s",
                  "frac": gbs / peak_bw, "bytes_per_launch": sparse_bytes,
                  "traffic": measured_traffic(args.config, "sparse")}
    p50 = statistics.median(step_ms)
    p99 = float(np.percentile(step_ms, 99))
    total_flop = sum(flops.values())
    t_roof_us = max(total_flop / (peak_tf * 1e12), total_bytes / (peak_bw * 1e9)) * 1e6
    path = {"t_roof_us": t_roof_us, "p50_us": p50 * 1e3, "frac": t_roof_us / (p50 * 1e3),
            "gflop_per_batch": total_flop / 1e9, "mbytes_per_batch": total_bytes / 1e6,
            "bound": "tensor" if total_flop / (peak_tf * 1e12) > total_bytes / (peak_bw * 1e9) else "hbm"}

    # ---- end to end through the host-buffer entry point (pinned buffers crossing the link inside the timed region)
    e2e = None
    if not args.no_e2e and not args.varlen:  # the host-buffer entry point has fixed lengths
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory().numpy()
        h_req, h_ids, h_off, h_seq = pin(wl.req_ids), pin(wl.bag_ids), pin(wl.bag_offsets), pin(wl.seq_ids)
        h_out = torch.empty((B, 2), dtype=torch.float32).pin_memory().numpy()
        sc.set_option(cvr.OPT_PROFILE, 0)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                sc.score_host(wl.n_req, B, h_req, h_ids, h_off, h_seq, h_out)
            e_ms = []
            for i in range(args.steps):
                flush.zero_()
                ev0 = torch.cuda.Event(enable_timing=True)
                ev1 = torch.cuda.Event(enable_timing=True)
                ev0.record(stream)
                sc.score_host(wl.n_req, B, h_req, h_ids, h_off, h_seq, h_out)
                ev1.record(stream)
                ev1.synchronize()
                e_ms.append(ev0.elapsed_time(ev1))
        h2d = h_req.nbytes + h_ids.nbytes + h_off.nbytes + h_seq.nbytes
        e_tot = sum(e_ms)
        e_tot = max_over_ranks(e_tot, dev)
        e2e = {"value": job_throughput(world, B, args.steps, e_tot), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(h_out.nbytes), "p50_ms": statistics.median(e_ms),
               "api": "cvr_score_host (pinned host buffers, read and written in place by the kernels)"}

    # the same steps with the PLE on 8-bit weights (the option the accuracy gate admits): batch time and the
    # PLE + heads kernel's own time
    int8 = None
    if not (args.minimal or args.varlen or args.ple_int8):
        sc.set_option(cvr.OPT_PLE_INT8, 1)
        i8_ms, _, _ = timed_region(profile=False, n_steps=min(args.steps, 1000))
        _, i8_stages, _ = timed_region(profile=True, n_steps=200)
        sc.set_option(cvr.OPT_PLE_INT8, 0)
        i8_tot = max_over_ranks(sum(i8_ms), dev)
        int8 = {"value": job_throughput(world, B, len(i8_ms), i8_tot), "unit": UNIT,
                "p50_ms": statistics.median(i8_ms),
                "ple_heads_ms": sum(i8_stages.get("ple_heads", [float("nan")])) / 200,
                "what": "CVR_OPT_PLE_INT8: PLE expert and gate weights int8 with a scale per row, bf16 activations"}

    gather = None
    if rank == 0 and not args.no_gather and not args.varlen:
        gather = gather_roofline(dev, stream, flush, peak_bw)

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = oracle_baseline(args.config)
        Lstr = "/".join(str(x) for x in wl.seq_len)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (PLE weights int8)" if args.ple_int8 else "bf16", "data": "synthetic",
            **({"attention": "tcgen05 kernel (CVR_OPT_ATTENTION_TC)"} if args.attention_tc else {}),
            "config": {"workload": f"{args.config}: R={wl.n_req} requests x C={B // wl.n_req} candidates, "
                                   f"L={Lstr}, {wl.n_layers} interaction layer(s), tables {wl.user_rows}/"
                                   f"{wl.item_rows}/{wl.seq_rows} rows x 32 fp32, bags 1-8, Zipf({wl.zipf_s})",
                       "global_batch": B * world, "parallelism": f"replicas x{world}",
                       "l2": "flushed (256 MB write) before every timed step",
                       **({"seq_lens": f"variable: uniform in [1, L_g] per request and group, "
                                       f"{float(lens.sum()) / wl.n_req:.1f} of {wl.sum_len} events per request"}
                          if args.varlen else {})},
            "latency": ({"p50_ms": statistics.median(call_ms), "p99_ms": float(np.percentile(call_ms, 99)),
                         "what": "request latency: synchronous cvr_score call on the batch, host wall clock "
                                 "(checks, graph launch, wait, error-word read), 500 calls after 50 warm-up, "
                                 "L2 flushed and the GPU idle before each"} if call_ms else None),
            "r1_latency_ms": r1["p50_ms"] if r1 else None, "single_request": r1,
            "p50_ms": p50, "p99_ms": p99, "device_time": "p50_ms / p99_ms: GPU time of one batch (CUDA events "
                                                          "around back-to-back calls)",
            "profiled_p50_ms": statistics.median(prof_ms),
            "roofline": roofline, "sparse_roofline": sparse, "gather_roofline": gather, "path_roofline": path,
            "stage_ms": {k: round(v, 5) for k, v in per_kernel.items()},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks.summary(), "ple_int8": int8,
            "gpu_launches": launches,
        }
        print(json.dumps(line))
    sc.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
