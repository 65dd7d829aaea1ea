"""Benchmark of the fused causal-conv1d + KDA verify decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--variant auto|one_item|pipelined]

One step = one kda_conv_verify call over the whole workload (default: the
large-batch verify, N=256 sequences, T=4 tokens, H=HV=32, K=V=128, bf16
activations, fp32 state, softplus gate).  `value` is verify head-steps/s
(N*T*HV per call) timed with CUDA events on the launching stream with the
inputs resident in HBM; `e2e` is the same metric through the same public call
with the inputs copied in from pinned host memory and every output copied
back inside the timed region.  `roofline` compares the algorithmic bytes of
one launch divided by its measured duration with the measured HBM copy
bandwidth.  `cpu_baseline` times the CPU oracle on a bounded sample of the
same workload on the host cores.

Under torchrun every rank runs its own copy of the workload on its own GPU
(weak scaling, no collective on the data path); the time is the maximum over
ranks.  `--impl reference` times the CPU oracle as the reference arm.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify head-steps/s (N·T·HV) and achieved HBM GB/s vs GB300 peak, 1 GPU"
UNIT = "head-steps/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large_bf16_n256_t4_h32")
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--plan", default="",
                    help="explicit launch plan variant:columns[:grid[:prefetch[:qk_roll]]], e.g. item:32, "
                         "pipe:64 or item:64:0:0:cluster (overrides --variant)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time the stream-launched kernel only: no graph, e2e or CPU legs, and no "
                         "device buffers beyond the one workload (for profiler captures)")
    ap.add_argument("--scaling", default="weak", choices=["weak", "strong"],
                    help="weak: every rank runs the whole workload; strong: the ranks split "
                         "its sequences")
    ap.add_argument("--N", type=int, default=0,
                    help="override the number of sequences (small profiling cases)")
    ap.add_argument("--op", default="verify", choices=["verify", "commit", "decode"],
                    help="commit: time kda_commit (accept a random count per sequence); "
                         "decode: time kda_conv_decode (no snapshots, state in place)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every point of the T x N x heads x gate sweep with every plan of --sweep-plans")
    ap.add_argument("--sweep-out", default="")
    ap.add_argument("--sweep-filter", default="",
                    help="regular expression: only sweep points whose name matches")
    ap.add_argument("--sweep-report", default="",
                    help="read a --sweep-out file and print its markdown summary (no GPU)")
    ap.add_argument("--sweep-plans", default="auto,item:32,item:64,item:128,smem:128,pipe:64,pipe:128",
                    help="plans timed at every sweep point")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload(name):
    """A named workload, a sweep point, or 'custom:N,T,H,HV,K,V[,act[,gate]]'
    (decode distributions, seed 0)."""
    from linear_attention_speculative_gb300 import workloads as wk
    if name in wk.WORKLOADS:
        return wk.WORKLOADS[name]
    if name.startswith("custom:"):
        f = name[len("custom:"):].split(",")
        nums = [int(x) for x in f[:6]]
        act = f[6] if len(f) > 6 else "bf16"
        gate = f[7] if len(f) > 7 else "softplus"
        return wk.custom(*nums, act=act, gate=gate)
    for w in wk.sweep():
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}")


class L2Flush:
    """Evict the previous launch's lines from L2 before a timed launch: write a
    buffer twice the size of L2, then read another one as large.  The read
    leaves L2 holding clean lines, so the timed launch does not pay for writing
    back the flush's own dirty lines (a plain write-only flush left ~129 MB of
    them, ~2 us on a 23 us call)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self, i):
        import torch
        self.w.fill_(float(i))
        torch.sum(self.r, dim=(0,), out=self.sink[0])


L2_FLUSH_NOTE = "L2 flushed before every timed launch (258 MB written, then 258 MB read)"


# back-to-back figures only where this many sets suffice (calls of >= L2 / 4)
MAX_ROTATION_SETS = 16


def rotation_sets(nbytes):
    """Independent input/output sets to rotate over when calls of `nbytes` run
    back to back: enough that together they hold over three times L2, so that
    the other sets' traffic evicts a set between two of its uses."""
    return -(-3 * L2_BYTES // max(1, nbytes)) + 1


def time_back_to_back(call, R, B, stream, flush):
    """Mean milliseconds per call of B calls queued back to back on `stream`,
    call(i % R) for i < B, between one pair of events after an L2 flush (no
    flush between the calls): each call's launch may overlap the previous
    call's end, as consecutive calls of a serving loop do."""
    import torch
    for r in range(R):
        call(r)
    torch.cuda.synchronize()
    flush(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(B):
        call(i % R)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / B


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# kernel that each plan variant launches (ONE_ITEM, PIPELINED, ONE_ITEM_SMEM, SPLIT)
KERNEL_OF_VARIANT = {1: "kda_tile_kernel", 2: "kda_pipe_kernel", 3: "kda_tile_kernel_sms",
                     4: "kda_split"}
VARIANT_NAME = {1: "one_item", 2: "pipelined", 3: "one_item_smem", 4: "split"}

# device sources each profiled kernel is built from (host-only files such as
# the dispatcher in kda_api.cu do not change the kernels' code)
COMMIT_SOURCES = ("kda_commit.cu", "kda_device.cuh")
VERIFY_SOURCES = ("kda_kernel.cuh", "kda_device.cuh", "kda_launch.cuh", "kda_inst_tile_bf16.cu",
                  "kda_inst_tile_f32.cu", "kda_inst_tile_cl_bf16.cu", "kda_inst_tile_cl_f32.cu",
                  "kda_inst_tile_dec_bf16.cu", "kda_inst_tile_dec_f32.cu",
                  "kda_inst_pipe_bf16.cu", "kda_inst_pipe_f32.cu",
                  "kda_inst_split_bf16.cu", "kda_inst_split_f32.cu", "kda_roll.cu")


def kernel_src_hash(kernel="verify"):
    """Hash of the CUDA sources of `kernel` ("verify" or "commit") with comments
    and whitespace removed, so that a comment-only edit, or a change to another
    kernel's file, keeps the committed ncu summaries valid."""
    d = os.path.join(ROOT, "linear_attention_speculative_gb300", "csrc")
    names = sorted(os.listdir(d))
    names = [f for f in names if f in (COMMIT_SOURCES if kernel == "commit" else VERIFY_SOURCES)]
    h = hashlib.sha256()
    for f in names:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        code = " ".join(code.split())
        h.update(f.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def ncu_traffic(wl_name, kernel_tag):
    """DRAM bytes per launch (total, read, write) from the committed ncu summary
    of this kernel (profiles/ncu_<kernel_tag>_<workload>.md), or Nones when
    absent or taken on other kernel sources."""
    none = (None, None, None)
    path = os.path.join(ROOT, "profiles", f"ncu_{kernel_tag}_{wl_name}.md")
    if not os.path.exists(path):
        return none
    text = open(path).read()
    h = re.search(r"kernel_src_sha256:\s*([0-9a-f]+)", text)
    if not h or h.group(1) != kernel_src_hash():
        return none
    get = lambda key: (lambda m: float(m.group(1)) if m else None)(
        re.search(key + r":\s*([0-9.eE+]+)", text))
    return get("dram_bytes_per_launch"), get("dram_bytes_read_per_launch"), get("dram_bytes_write_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.t_on = None
        self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [s for t, s in self.samples
                if self.t_on is not None and self.t_on - 0.1 <= t <= (self.t_off or t) + 0.1]
        if not rows:
            rows = [s for _, s in self.samples]
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(wl, inputs_cpu, cpu_seconds=12.0):
    """Time the CPU oracle as it stands on a bounded sample of the workload:
    whole passes over its sequences (one sequence per thread at a time, all
    host cores), repeated until about `cpu_seconds` of CPU time were spent."""
    import oracle
    cores = os.cpu_count() or 1
    s = wl.shape
    # bf16/fp32 -> fp64 conversion of the inputs happens outside the timed region
    sub = {k: (oracle._f64(v) if v is not None else None) for k, v in inputs_cpu.items()}
    passes, dt = 0, 0.0
    while passes == 0 or (dt * cores < cpu_seconds and passes < 64):
        t0 = time.perf_counter()
        oracle.verify(sub, wl.gate, threads=cores)
        dt += time.perf_counter() - t0
        passes += 1
    hs = passes * s.head_steps
    # the same oracle on one core: the first min(N, 4) sequences, one pass
    n1 = min(s.N, 4)
    t0 = time.perf_counter()
    oracle.verify(sub, wl.gate, seqs=list(range(n1)), threads=1)
    dt1 = time.perf_counter() - t0
    bytes_per_head_step = s.algorithmic_bytes(wl.gate) / s.head_steps
    return {"value": hs / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "gb_per_s": hs / dt * bytes_per_head_step / 1e9,
            "single_core_value": n1 * s.T * s.HV / dt1,
            "sample": f"{passes} full pass(es) over the {s.N} sequences of {wl.name} ({hs} head-steps), "
                      f"fp64 C oracle, {cores} threads, {dt:.2f} s wall (~{dt * cores:.0f} s CPU); "
                      f"single_core_value: {n1} sequences on one thread"}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from linear_attention_speculative_gb300 import workloads as wk
    inputs = wk.make_inputs(wl)
    cores = os.cpu_count() or 1
    s = wl.shape
    seqs = list(range(min(s.N, cores)))
    sub = {k: (v[seqs] if v is not None and k in ("mixed_qkv", "conv_state", "a", "b", "S0") else v)
           for k, v in inputs.items()}
    oracle.build()
    sub = {k: (oracle._f64(v) if v is not None else None) for k, v in sub.items()}
    for _ in range(args.warmup):
        oracle.verify(sub, wl.gate, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify(sub, wl.gate, threads=cores)
    dt = time.perf_counter() - t0
    hs = len(seqs) * s.T * s.HV
    value = hs * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "N": s.N, "T": s.T, "H": s.H, "HV": s.HV, "K": s.K,
                   "V": s.V, "act": s.act, "gate": wl.gate,
                   "sample_per_step": f"{len(seqs)} sequences ({hs} head-steps)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{len(seqs)} of {s.N} sequences per step, {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, wl):
    import dataclasses

    import torch
    from linear_attention_speculative_gb300 import kda
    from linear_attention_speculative_gb300 import workloads as wk
    from linear_attention_speculative_gb300.replicas import max_over_ranks, shard

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inputs_cpu = wk.make_inputs(wl)
    global_head_steps = wl.shape.head_steps * (world if args.scaling == "weak" else 1)
    if args.scaling == "strong" and world > 1:
        # this rank's contiguous slice of the global batch: no data exchange
        lo, hi = shard(wl.shape.N, rank, world)
        inputs_cpu = {k: (v[lo:hi].contiguous() if v is not None and k in
                          ("mixed_qkv", "conv_state", "a", "b", "S0") else v)
                      for k, v in inputs_cpu.items()}
        wl = dataclasses.replace(wl, shape=dataclasses.replace(wl.shape, N=hi - lo))
    s = wl.shape
    inp = {k: (v.to(dev) if v is not None else None) for k, v in inputs_cpu.items()}
    shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"])
    ws = kda.alloc_workspace(shape, dev)
    out = {k: v.to(dev) for k, v in wk.empty_outputs(wl).items()}
    stream = torch.cuda.current_stream(dev)
    alg_bytes = s.algorithmic_bytes(wl.gate)
    flush_l2 = alg_bytes < 2 * L2_BYTES
    flush_buf = L2Flush(dev) if flush_l2 else None

    def step(x=inp, validate=False):
        # the binding checks every tensor against the shape on the first call;
        # the timed calls skip the host-side checks, which on a call of a few
        # microseconds could otherwise leave the GPU idle inside the events
        kda.conv_verify(x["mixed_qkv"], x["conv_w"], x["conv_state"], x["A_log"], x["dt_bias"],
                        x["a"], x["b"], x["S0"], wl.gate, out["o"], out["inter_ssm"],
                        out["conv_snapshots"], ws, stream=stream, variant=args.variant,
                        shape=shape, plan=args.plan or None, validate=validate)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    step(validate=True)  # the first warm-up step
    for _ in range(max(3, args.warmup) - 1):
        step()
    barrier()

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    K = args.steps
    barrier()
    clocks.mark_on()
    if flush_l2:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            flush_buf(i)  # evict the previous step's lines from L2
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
        kernel_ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        barrier()
        kernel_ms = e0.elapsed_time(e1)
    clocks.mark_off()
    kernel_ms = max_over_ranks(kernel_ms, dev)
    ms_per_step = kernel_ms / K
    value = global_head_steps * K / (kernel_ms / 1e3)

    graph_line = None
    if not args.kernel_only:
        # the same step captured once in a CUDA graph and replayed (no host launch
        # work per step); reported beside the stream-launched figure
        G = min(K, 50)
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gstream):
            step_g = lambda: kda.conv_verify(
                inp["mixed_qkv"], inp["conv_w"], inp["conv_state"], inp["A_log"], inp["dt_bias"],
                inp["a"], inp["b"], inp["S0"], wl.gate, out["o"], out["inter_ssm"],
                out["conv_snapshots"], ws, stream=gstream, variant=args.variant, shape=shape,
                plan=args.plan or None, validate=False)
            step_g()  # outside capture: per-device attribute set-up
        gstream.synchronize()
        with torch.cuda.graph(graph, stream=gstream):
            step_g()
        barrier()
        g_ms = 0.0
        with torch.cuda.stream(gstream):
            if flush_l2:
                for i in range(G):
                    flush_buf(i)
                    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a_ev.record(gstream)
                    graph.replay()
                    b_ev.record(gstream)
                    b_ev.synchronize()
                    g_ms += a_ev.elapsed_time(b_ev)
            else:
                a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_ev.record(gstream)
                for _ in range(G):
                    graph.replay()
                b_ev.record(gstream)
                b_ev.synchronize()
                g_ms = a_ev.elapsed_time(b_ev)
        barrier()
        g_ms = max_over_ranks(g_ms, dev)
        graph_line = {"ms_per_step": g_ms / G, "value": global_head_steps * G / (g_ms / 1e3), "steps": G}
        del graph

    b2b_line = None
    if flush_l2 and not args.kernel_only and rotation_sets(alg_bytes) <= MAX_ROTATION_SETS:
        # A call that fits in L2 is timed above one launch at a time, each between
        # its own events after a flush, so every step also carries the launch's
        # few microseconds between the events.  Here the same call runs back to
        # back, as consecutive layers' calls do, over R independent input, output
        # and workspace sets that together hold over three times L2: between two
        # uses of one set the other sets' traffic has evicted it.  One event pair
        # around all the calls, no flush between them.
        R = rotation_sets(alg_bytes)
        sets = [(inp, out, ws)]
        for _ in range(R - 1):
            sets.append(({k: (v.clone() if v is not None else None) for k, v in inp.items()},
                         {k: torch.empty_like(v) for k, v in out.items()},
                         kda.alloc_workspace(shape, dev)))

        def call(x, y, w):
            kda.conv_verify(x["mixed_qkv"], x["conv_w"], x["conv_state"], x["A_log"], x["dt_bias"],
                            x["a"], x["b"], x["S0"], wl.gate, y["o"], y["inter_ssm"],
                            y["conv_snapshots"], w, stream=stream, variant=args.variant,
                            shape=shape, plan=args.plan or None, validate=False)

        B = max(K, 4 * R)
        barrier()
        b_ms = max_over_ranks(B * time_back_to_back(lambda r: call(*sets[r]), R, B, stream, flush_buf), dev)
        b2b_line = {"ms_per_step": b_ms / B, "value": global_head_steps * B / (b_ms / 1e3),
                    "steps": B, "sets": R,
                    "frac": alg_bytes / (b_ms / B / 1e3) / 1e9 / measured_hbm_peak()[0],
                    "note": (f"back-to-back calls over {R} independent input/output sets "
                             f"({R * alg_bytes / 1e6:.0f} MB moved per round, over 3x L2), one event "
                             "pair, no flush between calls")}
        del sets

    e2e_line = None
    if not args.kernel_only:
        # end to end: pinned host inputs in, every output back, through the same
        # call.  Two streams with their own device buffers alternate steps, so one
        # step's device->host copy overlaps the next step's host->device copy and
        # kernel (the copy engines of the two directions run concurrently).
        E = max(2, min(args.e2e_steps, K))
        host_in = {k: (v.pin_memory() if v is not None else None) for k, v in inputs_cpu.items()}
        h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
        lanes = []
        for r in range(2):
            dev_in = inp if r == 0 else {k: (torch.empty_like(v) if v is not None else None)
                                         for k, v in inp.items()}
            dev_out = out if r == 0 else {k: torch.empty_like(v) for k, v in out.items()}
            host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
            host_out["conv_state"] = torch.empty(inp["conv_state"].shape,
                                                 dtype=inp["conv_state"].dtype).pin_memory()
            lanes.append(dict(stream=stream if r == 0 else torch.cuda.Stream(dev), inp=dev_in,
                              out=dev_out, host_out=host_out, ws=ws if r == 0 else
                              kda.alloc_workspace(shape, dev)))
        d2h = sum(v.numel() * v.element_size() for v in lanes[0]["host_out"].values())

        # the inputs a serving step receives anew (the new tokens' projections and
        # gate inputs) and the output it returns; the other tensors are state
        STEP_IN, STEP_OUT = ("mixed_qkv", "a", "b"), ("o",)

        def e2e_step(lane, resident=False):
            st, x, y, ho = lane["stream"], lane["inp"], lane["out"], lane["host_out"]
            with torch.cuda.stream(st):
                for k, v in host_in.items():
                    if v is not None and (not resident or k in STEP_IN):
                        x[k].copy_(v, non_blocking=True)
                kda.conv_verify(x["mixed_qkv"], x["conv_w"], x["conv_state"], x["A_log"],
                                x["dt_bias"], x["a"], x["b"], x["S0"], wl.gate, y["o"],
                                y["inter_ssm"], y["conv_snapshots"], lane["ws"], stream=st,
                                variant=args.variant, shape=shape, plan=args.plan or None)
                for k in (STEP_OUT if resident else ("o", "inter_ssm", "conv_snapshots")):
                    ho[k].copy_(y[k], non_blocking=True)
                if not resident:
                    ho["conv_state"].copy_(x["conv_state"], non_blocking=True)

        def e2e_time(steps, resident=False):
            barrier()
            f0 = torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            lanes[1]["stream"].wait_event(f0)
            for i in range(steps):
                e2e_step(lanes[i % 2], resident)
            ends = []
            for lane in lanes:
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(lane["stream"])
                ends.append(ev)
            barrier()
            return max_over_ranks(max(f0.elapsed_time(ev) for ev in ends), dev)

        for r in range(2):
            e2e_step(lanes[r])  # also fills both lanes' state buffers
        e2e_ms = e2e_time(E)
        e2e_value = global_head_steps * E / (e2e_ms / 1e3)
        e2e_line = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": E,
                    "note": "pinned host buffers; two streams alternate steps so copies overlap"}
        # the same call with the state resident on the device, as a serving loop
        # keeps it: per step the new inputs in and o out
        ER = max(2, min(K, 50))
        for r in range(2):
            e2e_step(lanes[r], resident=True)
        er_ms = e2e_time(ER, resident=True)
        e2e_line["state_resident"] = {
            "value": global_head_steps * ER / (er_ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": sum(host_in[k].numel() * host_in[k].element_size() for k in STEP_IN),
            "d2h_bytes_per_step": sum(lanes[0]["host_out"][k].numel() * lanes[0]["host_out"][k].element_size()
                                      for k in STEP_OUT),
            "steps": ER,
            "note": ("S0, conv_state, the weights and the snapshots stay on the device; per step "
                     "mixed_qkv, a and b in from pinned host memory and o back")}

    if rank == 0:
        clocks.stop()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peak, peak_src = measured_hbm_peak()
    achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
    plan = kda.make_plan(shape, torch.cuda.get_device_properties(dev).multi_processor_count,
                         args.variant)
    if args.plan:
        plan = kda.resolve_plan(shape, torch.cuda.get_device_properties(dev).multi_processor_count,
                                args.plan)
    traffic = ncu_traffic(wl.name, KERNEL_OF_VARIANT[plan.variant])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": args.scaling, "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "N": s.N, "T": s.T, "H": s.H, "HV": s.HV, "K": s.K,
                   "V": s.V, "W": s.W, "act": s.act, "state": "f32", "gate": wl.gate,
                   "variant": VARIANT_NAME[plan.variant],
                   "v_tile": plan.bv, "plan": args.plan or f"auto ({plan_label(plan)})",
                   "qk_roll": ("single reader" if (s.HV // s.H) * (s.V // plan.bv) == 1 else
                               "prep kernel" if plan.variant == kda.VARIANT_SPLIT else
                               {v: k for k, v in kda.QK_ROLL_NAMES.items()}[plan.qk_roll]),
                   "l2": (L2_FLUSH_NOTE if flush_l2 else
                          f"inputs larger than L2: {alg_bytes / 1e9:.2f} GB moved per step"),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": traffic[0], "traffic_read": traffic[1], "traffic_write": traffic[2],
                     "traffic_source": ("one-pass ncu capture of the same launch, steady state "
                                        f"(profiles/ncu_{KERNEL_OF_VARIANT[plan.variant]}_{wl.name}.md)"
                                        if traffic[0] is not None else "no current capture"),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_source": f"{peak_src} (hbm_gbs, STREAM-style copy)",
                     "kernel": KERNEL_OF_VARIANT[plan.variant]},
        "e2e": e2e_line,
        "gpu_launches": K * max(1, plan.launches),
        "graph": graph_line,
        "back_to_back": b2b_line,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline and not args.kernel_only:
        line["cpu_baseline"] = cpu_baseline(wl, inputs_cpu)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def plan_label(plan) -> str:
    from linear_attention_speculative_gb300 import kda
    return kda.plan_label(plan)


def run_sweep(args):
    """Time each sweep point with every plan of --sweep-plans ("auto" = the
    dispatcher's pick) -- the verify call, or with --op decode the plain
    decode.  Inputs are drawn on the device (timing only); L2 is flushed
    before every timed launch.  Median of --steps launches."""
    import torch
    from linear_attention_speculative_gb300 import kda
    from linear_attention_speculative_gb300 import workloads as wk

    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    K = max(3, args.steps)
    decode = args.op == "decode"
    plans = [p for p in args.sweep_plans.split(",") if p]
    rows = []
    sink = open(args.sweep_out, "w") if args.sweep_out else None
    for wl in wk.sweep():
        if args.sweep_filter and not re.search(args.sweep_filter, wl.name):
            continue
        s = wl.shape
        inp = wk.make_inputs_on_device(wl, dev)
        out = {k: v for k, v in wk.empty_outputs(wl, device=dev).items()}
        shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"])
        ws = kda.alloc_workspace(shape, dev)
        auto_plan = kda.make_plan(shape, sms, "auto", decode=decode)
        auto = plan_label(auto_plan)
        # who rolls the q/k conv_state when several items read it
        shared = (s.HV // s.H) * (s.V // auto_plan.bv) > 1 and auto_plan.variant != kda.VARIANT_SPLIT
        roll_names = {v: k for k, v in kda.QK_ROLL_NAMES.items()}
        alg = decode_bytes(s, wl.gate) if decode else s.algorithmic_bytes(wl.gate)
        row = {"workload": wl.name, "op": args.op if decode else "verify", "N": s.N, "T": s.T,
               "H": s.H, "HV": s.HV, "gate": wl.gate, "alg_bytes": alg,
               "head_steps": s.head_steps, "auto": auto,
               "auto_roll": roll_names[auto_plan.qk_roll] if shared else "", "us": {}}
        launched = {}
        for spec in plans:
            plan = None if spec == "auto" else spec
            if plan is not None:
                try:  # a plan the library does not build for this point is left out
                    rp = kda.resolve_plan(shape, sms, plan, decode=decode)
                except kda.KdaError:
                    continue
                # explicit plans that resolve to the same launch (e.g. "item:64" and
                # "item:64:0:0:cluster" where the dispatcher rolls by the cluster)
                # are timed once: the minimum over repeats of one launch would
                # bias "best" low
                key = (rp.variant, rp.bv, rp.grid, rp.prefetch, rp.qk_roll)
                if key in launched:
                    row["us"][spec] = row["us"][launched[key]]
                    row.setdefault("same_launch", {})[spec] = launched[key]
                    continue
                launched[key] = spec

            def step(validate=False):
                if decode:
                    kda.conv_decode(inp["mixed_qkv"], inp["conv_w"], inp["conv_state"],
                                    inp["A_log"], inp["dt_bias"], inp["a"], inp["b"], inp["S0"],
                                    wl.gate, out["o"], ws, stream=stream, shape=shape, plan=plan,
                                    validate=validate)
                else:
                    kda.conv_verify(inp["mixed_qkv"], inp["conv_w"], inp["conv_state"],
                                    inp["A_log"], inp["dt_bias"], inp["a"], inp["b"], inp["S0"],
                                    wl.gate, out["o"], out["inter_ssm"], out["conv_snapshots"], ws,
                                    stream=stream, shape=shape, plan=plan, validate=validate)
            step(validate=True)  # three warm-up launches, the first one checked
            for _ in range(2):
                step()
            times = []
            for i in range(K):
                flush(i)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step()
                e1.record(stream)
                times.append((e0, e1))
            torch.cuda.synchronize(dev)
            row["us"][spec] = 1e3 * sorted(a.elapsed_time(b) for a, b in times)[len(times) // 2]
        explicit = {k: v for k, v in row["us"].items() if k != "auto"}
        best = min(explicit, key=explicit.get) if explicit else "auto"
        row["best"] = best
        row["best_gbs"] = alg / (row["us"][best] / 1e6) / 1e9
        if "auto" in row["us"]:
            row["auto_over_best"] = row["us"]["auto"] / row["us"][best]
        rows.append(row)
        if sink:
            sink.write(json.dumps(row) + "\n")
            sink.flush()
        cols = "  ".join(f"{k} {v:8.1f}" for k, v in row["us"].items())
        print(f"{wl.name:38s} {cols}  auto={auto} best={best} "
              f"x{row.get('auto_over_best', 1.0):.3f} {row['best_gbs']:6.0f} GB/s", flush=True)
        del inp, out, ws
        torch.cuda.empty_cache()
    if rows and "auto_over_best" in rows[0]:
        worst = max(rows, key=lambda r: r["auto_over_best"])
        print(json.dumps({"sweep_points": len(rows),
                          "worst_auto_over_best": worst["auto_over_best"],
                          "worst_point": worst["workload"]}))


def sweep_report(path, peak_gbs, peak_src):
    """Markdown summary of a --sweep-out file: per point the dispatcher's plan
    and time, the fastest explicit plan, their ratio, the bandwidth fraction,
    and which kernel wins where."""
    rows = [json.loads(line) for line in open(path) if line.strip()]
    plans = []
    for r in rows:
        plans += [k for k in r["us"] if k != "auto" and k not in plans]
    out = []
    op = rows[0].get("op", "verify") if rows else "verify"
    out.append("Operation: " + ("the plain decode (kda_conv_decode: state updated in place, no snapshots)"
                                if op == "decode" else "the verify call (kda_conv_verify)") + ".")
    out.append("")
    out.append(f"Peak: {peak_gbs:.1f} GB/s ({peak_src}, MEASURED_PEAKS.json hbm_gbs).  Times are the median of "
               "per-launch CUDA events with L2 flushed before each launch (258 MB written, then 258 MB read); "
               "GB/s = algorithmic bytes (from the point's shape and gate) / time.  An explicit plan that resolves to the same launch as an "
               "earlier column (e.g. a q/k roll the dispatcher would pick anyway) is timed once and shares "
               "that column's time.")
    out.append("")
    out.append("| T | N | H | HV | gate | auto plan | auto us | best plan | best us | auto/best | "
               "best GB/s | of peak | " + " | ".join(f"{p} us" for p in plans) + " |")
    out.append("|" + "---|" * (12 + len(plans)))
    for r in rows:
        best = r["best"]
        b_us = r["us"][best]
        gbs = row_bytes(r) / (b_us / 1e6) / 1e9
        auto = r["auto"] + (f" ({r['auto_roll']})" if r.get("auto_roll") else "")
        out.append(f"| {r['T']} | {r['N']} | {r['H']} | {r['HV']} | {r['gate']} | {auto} | "
                   f"{r['us']['auto']:.1f} | {best} | {b_us:.1f} | {r['us']['auto'] / b_us:.3f} | "
                   f"{gbs:.0f} | {gbs / peak_gbs:.3f} | "
                   + " | ".join(f"{r['us'][p]:.1f}" if p in r["us"] else "—" for p in plans) + " |")
    ratios = [r["us"]["auto"] / r["us"][r["best"]] for r in rows]
    out.append("")
    out.append(f"Points: {len(rows)}.  auto / best: mean {sum(ratios) / len(ratios):.4f}, "
               f"max {max(ratios):.4f}.")
    # the dispatcher's plan timed as an explicit plan (the same launches as
    # `best`'s column, so no second measurement's timer steps in the ratio)
    own = [r["us"][r["auto"]] / r["us"][r["best"]] for r in rows if r["auto"] in r["us"]]
    if own:
        out.append(f"The dispatcher's plan's own column / best: mean {sum(own) / len(own):.4f}, "
                   f"max {max(own):.4f} ({len(own)} points; the auto column is a second measurement of the "
                   "same plan, so its ratio also carries the event timer's steps).")
    for lo, hi in ((1, 1), (8, 32), (128, 512)):
        sub = [x for x, r in zip(ratios, rows) if lo <= r["N"] <= hi]
        if sub:
            out.append(f"- N in [{lo}, {hi}]: auto / best mean {sum(sub) / len(sub):.4f}, max {max(sub):.4f} "
                       f"({len(sub)} points)")
    # which kernel is fastest, by T and units (N * HV)
    out.append("")
    out.append("Fastest explicit plan by T (rows) and N * HV (columns), as kernel:v-tile columns (the "
               "dispatch crossovers); item = one item per CTA (state in registers), smem = one item per CTA "
               "(state in shared memory), pipe = pipelined, split = prep kernel + recurrence kernel:")
    units = sorted({r["N"] * r["HV"] for r in rows})
    Ts = sorted({r["T"] for r in rows})
    out.append("")
    out.append("| T \\ N*HV | " + " | ".join(str(u) for u in units) + " |")
    out.append("|" + "---|" * (1 + len(units)))
    for T in Ts:
        cells = []
        for u in units:
            kinds = sorted({":".join(r["best"].split(":")[:2]) for r in rows
                            if r["T"] == T and r["N"] * r["HV"] == u})
            cells.append("/".join(kinds) if kinds else "")
        out.append(f"| {T} | " + " | ".join(cells) + " |")
    for pick, what in ((lambda p: p.startswith("pipe:"), "Pipelined kernel"),
                       (lambda p: p.startswith("split:"), "Split variant (prep kernel + recurrence kernel)"),
                       (lambda p: p.endswith(":cluster"), "Cluster q/k roll (one-item kernel, a q/k group's "
                        "items as one thread-block cluster)")):
        mine = [p for p in plans if pick(p)]
        if not mine:
            continue
        out.append("")
        out.append(f"{what} against the dispatcher's plan (its best plan's time / auto time; "
                   "below 1 = faster than the dispatcher's pick):")
        out.append("")
        out.append("| T \\ N*HV | " + " | ".join(str(u) for u in units) + " |")
        out.append("|" + "---|" * (1 + len(units)))
        for T in Ts:
            cells = []
            for u in units:
                rs = [r for r in rows if r["T"] == T and r["N"] * r["HV"] == u
                      and any(p in r["us"] for p in mine)]
                if not rs:
                    cells.append("")
                    continue
                q = [min(r["us"][p] for p in mine if p in r["us"]) / r["us"]["auto"] for r in rs]
                cells.append(f"{min(q):.2f}-{max(q):.2f}" if len(q) > 1 else f"{q[0]:.2f}")
            out.append(f"| {T} | " + " | ".join(cells) + " |")
    return "\n".join(out)


def row_bytes(r) -> int:
    """Algorithmic bytes of a sweep row's call, from its shape and gate with the
    current byte count (rows store the count they were timed with)."""
    from linear_attention_speculative_gb300 import workloads as wk
    s = wk.custom(r["N"], r["T"], r["H"], r["HV"], r.get("K", 128), r.get("V", 128), gate=r["gate"]).shape
    return decode_bytes(s, r["gate"]) if r.get("op") == "decode" else s.algorithmic_bytes(r["gate"])


def commit_bytes(s) -> int:
    """Algorithmic bytes of one commit: per sequence the accepted state and
    conv-window snapshots read and the state and conv_state written, plus the
    accepted counts."""
    return 2 * s.N * (4 * s.HV * s.K * s.V + 3 * s.dim * s.act_bytes) + 4 * s.N


def run_commit(args, wl):
    """HBM bandwidth of kda_commit after one verify of the workload."""
    import torch
    from linear_attention_speculative_gb300 import kda
    from linear_attention_speculative_gb300 import workloads as wk
    dev = torch.device("cuda", 0)
    s = wl.shape
    inp = wk.make_inputs_on_device(wl, dev)
    out = kda.run(dict(inp, conv_state=inp["conv_state"].clone()), wl.gate)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed)
    acc = torch.randint(1, s.T + 1, (s.N,), generator=g, device=dev, dtype=torch.int32)
    S = torch.empty_like(inp["S0"])
    cs = torch.empty_like(inp["conv_state"])
    stream = torch.cuda.current_stream(dev)

    def step(validate=False):
        kda.commit(acc, out["inter_ssm"], out["conv_snapshots"], S, cs, stream=stream,
                   validate=validate)
    step(validate=True)  # the first warm-up step
    for _ in range(max(3, args.warmup) - 1):
        step()
    flush = L2Flush(dev)
    ev = []
    for i in range(args.steps):
        flush(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize(dev)
    us = 1e3 * sorted(a.elapsed_time(b) for a, b in ev)[len(ev) // 2]
    nbytes = commit_bytes(s)
    peak, src = measured_hbm_peak()
    # back to back over independent copies of everything the call touches
    R = rotation_sets(nbytes)
    b2b = None
    if R <= MAX_ROTATION_SETS:
        sets = [(out["inter_ssm"], out["conv_snapshots"], S, cs)] + [
            (out["inter_ssm"].clone(), out["conv_snapshots"].clone(), torch.empty_like(S), torch.empty_like(cs))
            for _ in range(R - 1)]
        b_us = 1e3 * time_back_to_back(
            lambda r: kda.commit(acc, *sets[r], stream=stream, validate=False), R, max(args.steps, 4 * R),
            stream, flush)
        del sets
        b2b = {"us": b_us, "frac": nbytes / (b_us / 1e6) / 1e9 / peak, "sets": R,
               "timing": "mean of back-to-back calls between one event pair"}
    print(json.dumps({"op": "commit", "workload": wl.name, "us": us, "bytes": nbytes,
                      "GB/s": nbytes / (us / 1e6) / 1e9, "frac": nbytes / (us / 1e6) / 1e9 / peak,
                      "peak_source": src, "timing": "median of per-launch CUDA events, L2 flushed",
                      "back_to_back": b2b}))


def decode_bytes(s, gate="softplus") -> int:
    """Algorithmic bytes of one plain decode call: the state read and written in
    place, the raw inputs, conv_state read and written, o, the weights (A_log
    and dt_bias only under the softplus gate)."""
    return (8 * s.N * s.HV * s.K * s.V + s.act_bytes * (
        s.N * s.T * s.dim + 2 * s.N * s.dim * 3 + s.N * s.T * s.HV * s.K + s.N * s.T * s.HV
        + s.N * s.T * s.HV * s.V + 4 * s.dim) + (4 * s.HV * (1 + s.K) if gate == "softplus" else 0))


def run_decode(args, wl):
    """Head-steps/s and HBM bandwidth of the plain decode (state in place)."""
    import torch
    from linear_attention_speculative_gb300 import kda
    from linear_attention_speculative_gb300 import workloads as wk
    dev = torch.device("cuda", 0)
    s = wl.shape
    inp = wk.make_inputs_on_device(wl, dev)
    shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"])
    ws = kda.alloc_workspace(shape, dev)
    o = torch.empty((s.N, s.T, s.HV, s.V), dtype=s.torch_act, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(validate=False):
        kda.conv_decode(inp["mixed_qkv"], inp["conv_w"], inp["conv_state"], inp["A_log"],
                        inp["dt_bias"], inp["a"], inp["b"], inp["S0"], wl.gate, o, ws,
                        stream=stream, shape=shape, plan=args.plan or None, validate=validate)
    nbytes = decode_bytes(s, wl.gate)
    flush = nbytes < 2 * L2_BYTES
    fbuf = L2Flush(dev) if flush else None
    step(validate=True)  # the first warm-up step
    for _ in range(max(3, args.warmup) - 1):
        step()
    ev = []
    for i in range(args.steps):
        if flush:
            fbuf(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize(dev)
    us = 1e3 * sorted(a.elapsed_time(b) for a, b in ev)[len(ev) // 2]
    peak, src = measured_hbm_peak()
    gbs = nbytes / (us / 1e6) / 1e9
    # back to back over independent copies of everything the call touches
    R = rotation_sets(nbytes)
    b2b = None
    if R <= MAX_ROTATION_SETS:
        sets = [(inp, o, ws)] + [({k: (v.clone() if v is not None else None) for k, v in inp.items()},
                                  torch.empty_like(o), kda.alloc_workspace(shape, dev)) for _ in range(R - 1)]

        def call(r):
            x, y, w = sets[r]
            kda.conv_decode(x["mixed_qkv"], x["conv_w"], x["conv_state"], x["A_log"], x["dt_bias"], x["a"],
                            x["b"], x["S0"], wl.gate, y, w, stream=stream, shape=shape, plan=args.plan or None,
                            validate=False)
        b_us = 1e3 * time_back_to_back(call, R, max(args.steps, 4 * R), stream, fbuf or L2Flush(dev))
        del sets
        b2b = {"us": b_us, "frac": nbytes / (b_us / 1e6) / 1e9 / peak, "sets": R,
               "head_steps_per_s": s.head_steps / (b_us / 1e6),
               "timing": "mean of back-to-back calls between one event pair"}
    print(json.dumps({"op": "decode", "workload": wl.name, "us": us, "bytes": nbytes,
                      "head_steps_per_s": s.head_steps / (us / 1e6), "GB/s": gbs,
                      "frac": gbs / peak, "peak_source": src,
                      "timing": "median of per-launch CUDA events" + (", L2 flushed" if flush else ""),
                      "back_to_back": b2b}))


def main():
    args = parse()
    if args.sweep_report:
        peak, src = measured_hbm_peak()
        print(sweep_report(args.sweep_report, peak, src))
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.op == "commit":
        run_commit(args, workload(args.workload))
        return
    if args.op == "decode":
        run_decode(args, workload(args.workload))
        return
    wl = workload(args.workload)
    if args.N:
        import dataclasses
        sh = dataclasses.replace(wl.shape, N=args.N)
        wl = dataclasses.replace(wl, shape=sh, name=f"{wl.name}_as_N{args.N}")
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
