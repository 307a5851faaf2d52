"""Benchmark of the PRISM mixer forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one whole mixer forward pass (anchor + refinement kernel, then the
chunkwise scan kernel) over one batch of the workload, inputs resident in HBM.
Prints one JSON line on rank 0.  Under torchrun each rank runs its own replica
of the workload (the (b, h) sequences are independent, so the path shards with
no collective): weak scaling.

``--impl reference`` times the fp64 CPU oracle (the only other implementation
of the method) on the host cores, on a bounded sample of the same workload.

``--backward`` times the backward pass instead (prism_backward: all gradients given
d_out and d_final_state), with the gradient oracle as its CPU baseline.

``--decode`` times the single-token step (prism_decode_step) for every sequence of the
workload from a resident state, with the oracle's one-token forward as its CPU baseline.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_recurrent_sequence_causal_gb300 import inputs as I  # noqa: E402

METRIC = "PRISM mixer fwd tokens/s on 1 GB300; % of roofline (BF16 TC vs 8 TB/s HBM)"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "longctx_bf16"


# ---------------------------------------------------------------- roofline model
def algorithmic(wl, L):
    """Algorithmic bytes and flops per launch of each kernel.

    Per token-head (d = d_k = d_v, e = bytes per input element, C = chunk):
      prepare: reads q, k, v, gates: 3 d e + 8; writes the chunk's factored map:
               W, Kt, Qt_hi, Qt_lo (fp16) + U, O_intra (fp32) = 16 d, plus
               N (d x d fp32 per chunk) = 4 d^2 / C when L > 0.
               flops = 2 w d + L (4 d^2 + 2 d) + C d (10 + 8 L) + C^2 / 3 + 2 L d^2
      scan:    reads that map, writes out (fp32): 16 d + 4 d^2 / C [L > 0] + 4 d
               flops = 6 d^2
    plus the weights once per call (prepare) and the final state (d^2 fp32) once
    per sequence (scan).  The flop total over both kernels equals the chunk-form
    count C d (10 + 8L) + d^2 (6 + 2L) + C^2 / 3 plus the anchor/refinement count.
    """
    d, e, C, w = wl.dk, (4 if wl.dtype == "f32" else 2), wl.chunk, wl.w
    th = wl.B * wl.T * wl.H
    mid = 16 * d + (4 * d * d / C if L > 0 else 0) + 4.0 / C
    k1_bytes = th * (3 * d * e + 8 + mid) + wl.H * (L * (2 * d * d + d) + w * d) * 4
    k1_flops = th * (2 * w * d + L * (4 * d * d + 2 * d) + C * d * (10 + 8 * L) + C * C / 3.0
                     + 2 * L * d * d)
    k2_bytes = th * (mid + 4 * d) + wl.B * wl.H * d * d * 4
    k2_flops = th * (6.0 * d * d)
    return {"prepare": (k1_bytes, k1_flops), "scan": (k2_bytes, k2_flops)}


def method_counts(wl, L):
    """The method's own work per launch, with no intermediate of this build counted.

    Per token-head (d = d_k = d_v, e = bytes per I/O element, C = chunk, w = taps):
      F_scan   = C d (10 + 8 L) + d^2 (6 + 2 L) + C^2 / 3   (the chunk form of the recurrence)
      F_anchor = 2 w d + L (4 d^2 + 2 d)                     (anchor and refinement)
      bytes    = (2 d_k + 2 d_v) e + 8                       (q, k, v read, out written, gates)
    plus the final state (d^2 fp32) once per sequence and the weights once per call.
    Attribution: the scan kernel carries the state chain, 6 d^2 flops per token-head
    (W S0^T, Qt S0^T, Kt^T E), and writes out and the final state; the prepare kernel does
    the rest and reads q, k, v and the gates.  (out is fp32 here, 4 d bytes, where the
    count above takes the I/O width.)"""
    d, e, C, w = wl.dk, (4 if wl.dtype == "f32" else 2), wl.chunk, wl.w
    th = wl.B * wl.T * wl.H
    f_scan = C * d * (10 + 8 * L) + d * d * (6 + 2 * L) + C * C / 3.0
    f_anchor = 2 * w * d + L * (4 * d * d + 2 * d)
    weights = wl.H * (L * (2 * d * d + d) + w * d) * 4
    state = wl.B * wl.H * d * d * 4
    prep = (th * (3 * d * e + 8) + weights, th * (f_anchor + f_scan - 6.0 * d * d))
    scan = (th * d * e + state, th * 6.0 * d * d)
    path = (th * ((2 * d + 2 * d) * e + 8) + weights + state, th * (f_anchor + f_scan))
    return {"prepare": prep, "scan": scan, "path": path}


NOMINAL_HBM_GBS, NOMINAL_BF16_TFLOPS = 8000.0, 2250.0   # the metric's stated roofline figures


def roofline_of(by, fl, ms, hbm, tc):
    """Bound, achieved and fraction for `by` bytes and `fl` flops done in `ms`."""
    if by / (hbm * 1e9) >= fl / (tc * 1e12):
        r = {"bound": "hbm", "achieved": by / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s"}
        nominal = NOMINAL_HBM_GBS
    else:
        r = {"bound": "tensor", "achieved": fl / (ms / 1e3) / 1e12, "peak": tc, "unit": "TFLOP/s"}
        nominal = NOMINAL_BF16_TFLOPS
    r["frac"] = r["achieved"] / r["peak"]
    r["frac_nominal"] = r["achieved"] / nominal
    return r


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Sources of each forward kernel (the backward and decode kernels do not change them).
_COMMON = ("tc_common.cuh", "prism_common.cuh", "kernels_tc.cuh", "inst_tc_16.cu", "inst_tc_32.cu",
           "inst_tc_64.cu", "inst_tc_128.cu")
KERNEL_SOURCES = {"prepare": ("prep_tc.cuh",) + _COMMON, "scan": ("scan_tc.cuh",) + _COMMON}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_recurrent_sequence_causal_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        path = os.path.join(csrc, f)
        if os.path.exists(path):
            with open(path, "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t[kernel][workload]
        if ent.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.samples = []
        self.proc = None
        self.sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.sel = vis.split(",")[device_index] if vis else str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        s = self.samples
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in s if num(p[0]) is not None]
        mx = [num(p[1]) for p in s if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in s for i in range(4) if p[4 + i].lower().startswith("active")})
        power = [num(p[2]) for p in s if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(s), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(inp, wl, L, target_s, threads):
    """Time the oracle on a bounded sample of the workload's host inputs:
    sequence 0, all heads, a prefix whose length is calibrated to about
    ``target_s`` seconds."""
    import oracle

    def run(T):
        sub = {k: (v[:1, :T].contiguous() if k in ("q", "k", "v", "log_alpha", "beta") else
                   (v[:1] if k == "seq_lens" and v is not None else v)) for k, v in inp.items()}
        t0 = time.perf_counter()
        oracle.forward(sub, L=L, threads=threads)
        return time.perf_counter() - t0

    probe_T = min(wl.T, 256)
    dt = run(probe_T)
    T = max(probe_T, min(wl.T, int(probe_T * target_s / max(dt, 1e-6)) // 64 * 64))
    dt = run(T) if T != probe_T else dt
    return T, dt


def reference_arm(args, wl, L):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    per_step = max(0.5, 150.0 / (args.steps + args.warmup))
    import oracle
    inp = I.generate(wl, L=L)
    T, _ = oracle_sample(inp, wl, L, per_step, threads)      # calibration + first warm-up
    sub = {k: (v[:1, :T].contiguous() if k in ("q", "k", "v", "log_alpha", "beta") else
               (v[:1] if k == "seq_lens" and v is not None else v)) for k, v in inp.items()}
    for _ in range(max(0, args.warmup - 1)):
        oracle.forward(sub, L=L, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(sub, L=L, threads=threads)
    el = time.perf_counter() - t0
    tok = T * args.steps
    value = tok / el
    sample = f"sequence 0, all {wl.H} heads, first {T} of {wl.T} tokens per step (fp64 oracle)"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "d_k": wl.dk,
                       "d_v": wl.dv, "L": L, "conv_width": wl.w, "chunk": wl.chunk},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


L2_BYTES = 129e6


class L2Flush:
    """A write of four times the L2 size (about 80 us on the device) before each timed step
    of a workload whose inputs fit in L2: no input is left in L2 from the step before, and
    the device stays ahead of the host, so a step timed by events around it starts as soon
    as its flush ends and the flush itself is outside the events."""

    def __init__(self, dev):
        self.buf = torch.empty(int(4 * L2_BYTES) // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.zero_()


E2E_LOOPS = 5                     # timed loops of the end-to-end leg (median reported)
L2_FLUSHED = "L2 flushed before each step (a 516 MB write outside the timed events)"


# ---------------------------------------------------------------- ranks
def replica_seed(wl, rank):
    """Each rank times its own replica of the workload (independent sequences): the
    inputs differ by rank through the seed."""
    return wl.seed + rank


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (the whole job ends when it does); ``ms`` unchanged on one
    process."""
    if dist is None:
        return ms
    t = torch.tensor([float(ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s: the units all ranks processed over the slowest rank's time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


# ---------------------------------------------------------------- our arm
def our_arm(args, wl, L):
    from linear_recurrent_sequence_causal_gb300 import build, prism
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if build.stale():
        raise RuntimeError("libprism.so is missing or stale: run __graft_entry__.build() first")
    prism.load()
    dev = torch.device("cuda", local)
    host = I.generate(wl, L=L, seed=replica_seed(wl, rank))
    d = prism.inputs_to_device(host, dev)
    B, T, H, D = wl.B, wl.T, wl.H, wl.dk
    dt = wl.torch_dtype
    out = torch.empty((B, T, H, D), dtype=torch.float32, device=dev)
    fs = torch.empty((B, H, D, D), dtype=torch.float32, device=dev)
    flags = prism.PRISM_FLAG_NO_SEQ_SPLIT if args.no_seq_split else 0
    dims = prism.make_dims(B, T, H, D, D, wl.w, L, wl.chunk, dt, flags=flags)
    nseg = prism.scan_segments(dims)
    ws = prism.alloc_workspace(dims, dev)
    stream = torch.cuda.current_stream(dev)
    sl = d.get("seq_lens")

    def step(ev=None, current=False):
        st = None if current else stream       # current: whatever stream is current (a capture's)
        if ev is not None:
            ev[0].record(stream)
        prism.prism_prepare(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"],
                            d["Wk"], d["Wp"], d["wbeta"], L, wl.chunk, ws, seq_lens=sl,
                            stream=st, flags=flags)
        if ev is not None:
            ev[1].record(stream)
        prism.prism_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], L, wl.chunk, wl.w, ws,
                         out=out, final_state=fs, seq_lens=sl, stream=st, flags=flags)
        if ev is not None:
            ev[2].record(stream)

    # kernels per step: weight conversion (L > 0, bf16 path) + prepare + scan (three launches
    # when the sequence is split: affine maps, entering states when P > 2, final pass)
    scan_launches = 1 if nseg <= 1 else (3 if nseg > 2 else 2)
    launches_per_step = ((1 if (L > 0 and wl.dtype == "bf16") else 0) + (1 if (L > 0 or wl.dtype == "bf16") else 0)
                         + scan_launches)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # inputs that fit in L2 would stay there from one step to the next: such workloads are
    # timed step by step with L2 flushed in between
    small = 3 * B * T * H * D * (2 if wl.dtype == "bf16" else 4) <= L2_BYTES
    flush = L2Flush(dev) if small else None

    def split_steps():
        """K steps with events between the launches (L2 flushed before each when small)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            if flush:
                flush()
            step(evs[i])
        torch.cuda.synchronize(dev)
        return evs

    # each kernel's time
    evs = split_steps()
    k1_ms = [e[0].elapsed_time(e[1]) for e in evs]
    k2_ms = [e[1].elapsed_time(e[2]) for e in evs]
    # the timed region: inputs larger than L2, the K steps captured in one CUDA graph and
    # replayed once, so that the host's launch rate cannot pace them; else the K flushed
    # steps, each between its own events
    graph = None if small else capture_graph(lambda: [step(current=True) for _ in range(args.steps)], dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if small:
        elapsed_ms = sum(e[0].elapsed_time(e[2]) for e in split_steps())
    else:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        elapsed_ms = t_start.elapsed_time(t_end)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    ms_per_step = elapsed_ms / args.steps
    tokens = B * T * world
    value = job_throughput(B * T, world, ms_per_step)

    # ---- end to end through the public API: host (pinned) inputs, copies timed
    pinned = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    h_out = torch.empty((B, T, H, D), dtype=torch.float32).pin_memory()
    h_fs = torch.empty((B, H, D, D), dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)
    d2h = h_out.numel() * h_out.element_size() + h_fs.numel() * 4

    # the public host-to-host entry: copies in, kernels and copies out overlapped piece by
    # piece (groups of sequences, or token segments resumed from the previous state)
    pipe = prism.HostPipeline({k: tuple(v.shape) for k, v in host.items() if v is not None}, dt, L,
                              wl.chunk, device=dev)

    def e2e_step():
        pipe.run(pinned, h_out, h_fs, stream=stream)

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()

    def e2e_loop():
        if small:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(e2e_steps)]
            for a, b in pairs:
                flush()
                a.record(stream)
                e2e_step()
                b.record(stream)
            torch.cuda.synchronize(dev)
            return sum(a.elapsed_time(b) for a, b in pairs) / e2e_steps
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / e2e_steps

    # The host link is shared with the machine's other GPUs, and a single loop occasionally
    # runs 30-80 % slower: the median of E2E_LOOPS loops is reported, each loop beside it.
    e2e_samples = [e2e_loop() for _ in range(E2E_LOOPS)]
    e2e_ms = max_over_ranks(statistics.median(e2e_samples), dist, dev)
    e2e_value = job_throughput(B * T, world, e2e_ms)

    # ---- roofline of the dominant kernel, against the method's own work
    hbm, tc, peak_kind = load_peaks()
    alg = algorithmic(wl, L)
    meth = method_counts(wl, L)
    k1_avg = statistics.mean(k1_ms)
    k2_avg = statistics.mean(k2_ms)
    dom = "scan" if k2_avg >= k1_avg else "prepare"
    dom_ms = k2_avg if dom == "scan" else k1_avg
    by, fl = meth[dom]
    roof = roofline_of(by, fl, dom_ms, hbm, tc)
    roof["kernel"] = dom
    roof["counts"] = "method work (chunk-form flops; q, k, v, gates / out bytes), no intermediates"
    roof["peak_source"] = f"{peak_kind} ({'MEASURED_PEAKS.json' if peak_kind == 'measured' else 'recipe fallback'})"
    roof["kernel_ms"] = dom_ms
    roof["algorithmic_bytes"] = by
    roof["algorithmic_flops"] = fl
    # the same kernel against the bytes and flops it moves as built (its chunk maps included)
    ab, af = alg[dom]
    built = roofline_of(ab, af, dom_ms, hbm, tc)
    roof["as_built"] = {"bound": built["bound"], "achieved": built["achieved"], "unit": built["unit"],
                        "frac": built["frac"], "algorithmic_bytes": ab, "algorithmic_flops": af}
    traffic = committed_traffic(dom, wl.name)
    roof["traffic"] = traffic
    roof["traffic_over_method_bytes"] = traffic / by if traffic else None
    kernels = {"prepare_ms": k1_avg, "scan_ms": k2_avg,
               "share_scan": k2_avg / max(k1_avg + k2_avg, 1e-9), "scan_segments": nseg}
    for name, (kb, kf) in alg.items():
        kms = k1_avg if name == "prepare" else k2_avg
        kernels[f"{name}_GBps_as_built"] = kb / (kms / 1e3) / 1e9
        kernels[f"{name}_TFLOPs_as_built"] = kf / (kms / 1e3) / 1e12
        mb, mf = meth[name]
        kernels[f"{name}_frac_method"] = roofline_of(mb, mf, kms, hbm, tc)["frac"]
    # whole path: the fused-path roofline of the method (inputs, outputs, total flops), and
    # the two kernels as built (chunk maps written and read)
    pb, pf = meth["path"]
    kernels["path_roofline_ms"] = 1e3 * max(pb / (hbm * 1e9), pf / (tc * 1e12))
    kernels["path_frac"] = kernels["path_roofline_ms"] / ms_per_step
    tb = sum(v[0] for v in alg.values()) / (hbm * 1e9)
    tf = sum(v[1] for v in alg.values()) / (tc * 1e12)
    kernels["path_roofline_ms_as_built"] = 1e3 * max(tb, tf)
    kernels["path_frac_as_built"] = kernels["path_roofline_ms_as_built"] / ms_per_step

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "d_k": wl.dk,
                       "d_v": wl.dv, "L": L, "conv_width": wl.w, "chunk": wl.chunk,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "scan": (f"sequence split into {nseg} segments" if nseg > 1
                                else "one serial chain per sequence"),
                       "l2": L2_FLUSHED if small else "inputs larger than L2 (no flush)"},
            "roofline": roof, "kernels": kernels, "clocks": clk,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "loops_ms_per_step": e2e_samples, "steps_per_loop": e2e_steps},
            "gpu_launches": args.steps * launches_per_step}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        Ts, dts = oracle_sample(host, wl, L, args.cpu_seconds, threads)
        cb = Ts / dts
        line["cpu_baseline"] = {"value": cb, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"sequence 0, all {wl.H} heads, first {Ts} tokens; "
                                          f"{dts:.1f} s of fp64 oracle work on {threads} threads"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------- backward arm
BWD_METRIC = "PRISM mixer bwd tokens/s on 1 GB300 (all gradients, fp32 CUDA-core kernels)"
# FP32 FMA rate of the CUDA cores: 152 SMs x 128 lanes x 2 flop x 2.07 GHz (unit counts and
# the maximum SM clock); the backward kernels are fp32 arithmetic, not tensor-core work.
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def bwd_algorithmic(wl, L):
    """Flops and unavoidable bytes of one backward pass (per token-head, d = d_k = d_v):
    flops d^2 (28 + 20 L): the state sweep forward, its block recompute and the reverse
    step (2 d^2 (14 + 4 L)), the refinement projections and their transposes (8 L d^2),
    the weight-gradient outer products (4 L d^2); bytes: q, k, v, gates and d_out read,
    dq, dk, dv, dlog_alpha, dbeta written (fp32): 3 d e + 4 d + 8 + 12 d + 8."""
    d, e = wl.dk, (4 if wl.dtype == "f32" else 2)
    th = wl.B * wl.T * wl.H
    flops = th * d * d * (28.0 + 20.0 * L)
    by = th * (3 * d * e + 16 * d + 16) + wl.H * (2 * L * d * d + L * d + wl.w * d) * 4 * 2
    return by, flops


def grad_oracle_sample(host, wl, L, target_s):
    """Time the gradient oracle on a bounded sample: sequence 0, one head, a prefix
    calibrated to about ``target_s`` seconds."""
    from oracle import grad as G

    def run(T):
        sub = {}
        for k, v in host.items():
            if k in ("q", "k", "v", "log_alpha", "beta"):
                sub[k] = v[:1, :T, :1].contiguous()
            elif k in ("conv_w", "Wk", "Wp", "wbeta"):
                sub[k] = v[:1].contiguous()
            else:
                sub[k] = None
        d_out = torch.ones((1, T, 1, wl.dv), dtype=torch.float64)
        t0 = time.perf_counter()
        G.backward(sub, d_out, None, L=L)
        return time.perf_counter() - t0

    probe = min(wl.T, 32)
    dt = run(probe)
    T = max(probe, min(wl.T, int(probe * target_s / max(dt, 1e-6))))
    dt = run(T) if T != probe else dt
    return T, dt


def backward_launches(B, T, H, D, L):
    """Kernels one prism_backward call launches: refinement forward, state (+ the row-slice
    reduction when a (b, h) is split over CTAs), refinement backward, dW_k / dW_p (L > 0;
    + the token-split reduction), dw_beta / dconv (+ its reduction), the anchor's dv.  The
    splits follow the library's own choices (bwd_pick_rs / _nsw / _nss)."""
    ntok = B * T
    rs_split = B * H < 152
    nsw = min(32, max(1, ntok // 2048)) if L > 0 else 1
    nss = min(64, max(1, ntok // 512))
    return (5 + (1 if rs_split else 0) + (1 if L > 0 else 0) + (1 if nsw > 1 else 0)
            + (1 if nss > 1 else 0))


def backward_arm(args, wl, L):
    from linear_recurrent_sequence_causal_gb300 import build, prism
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if build.stale():
        raise RuntimeError("libprism.so is missing or stale: run __graft_entry__.build() first")
    prism.load()
    dev = torch.device("cuda", local)
    host = I.generate(wl, L=L, seed=wl.seed)
    d = prism.inputs_to_device(host, dev)
    B, T, H, D = wl.B, wl.T, wl.H, wl.dk
    g = torch.Generator().manual_seed(wl.seed + 1)
    h_dout = torch.randn((B, T, H, D), generator=g, dtype=torch.float32)
    h_dfs = torch.randn((B, H, D, D), generator=g, dtype=torch.float32)
    d_out, d_fs = h_dout.to(dev), h_dfs.to(dev)
    dims = prism.make_dims(B, T, H, D, D, wl.w, L, wl.chunk, wl.torch_dtype)
    ws = torch.empty(prism.load().prism_backward_workspace_bytes(ctypes_byref(dims)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    grads = prism.prism_backward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"],
                                 d["Wp"], d["wbeta"], L, d_out, d_final_state=d_fs,
                                 seq_lens=d.get("seq_lens"), workspace=ws, stream=stream)

    def step():
        prism.prism_backward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["conv_w"], d["Wk"],
                             d["Wp"], d["wbeta"], L, d_out, d_final_state=d_fs,
                             seq_lens=d.get("seq_lens"), workspace=ws, grads=grads, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    small = 3 * B * T * H * D * (2 if wl.dtype == "bf16" else 4) <= L2_BYTES
    flush = L2Flush(dev) if small else None

    def timed(fn, n):
        """Mean device time of n steps: back to back, or each between its own events after
        an L2 flush when the inputs fit in L2."""
        if not small:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / n
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in pairs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in pairs) / n

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = timed(step, args.steps)
    clk = clocks.stop()
    tokens = B * T
    value = tokens / (ms / 1e3)

    # end to end: inputs and d_out from pinned host memory, every gradient back to the host
    pinned = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    p_dout, p_dfs = h_dout.pin_memory(), h_dfs.pin_memory()
    host_g = {k: (torch.empty(v.shape, dtype=v.dtype).pin_memory() if v is not None else None)
              for k, v in grads.items()}
    h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None) \
        + p_dout.numel() * 4 + p_dfs.numel() * 4
    d2h = sum(v.numel() * 4 for v in host_g.values() if v is not None)

    def e2e_step():
        for k, v in pinned.items():
            if v is not None:
                d[k].copy_(v, non_blocking=True)
        d_out.copy_(p_dout, non_blocking=True)
        d_fs.copy_(p_dfs, non_blocking=True)
        step()
        for k, v in host_g.items():
            if v is not None:
                v.copy_(grads[k], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 5))
    e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = timed(e2e_step, e2e_steps)

    hbm, _, peak_kind = load_peaks()
    by, fl = bwd_algorithmic(wl, L)
    roof = {"bound": "alu", "achieved": fl / (ms / 1e3) / 1e12, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
            "traffic": None, "kernel": "prism_backward (five kernels, timed as one call)",
            "peak_source": "fp32 FMA lanes x maximum SM clock (derived; not in MEASURED_PEAKS.json)",
            "algorithmic_flops": fl, "algorithmic_bytes": by,
            "hbm_view": {"achieved_GBps": by / (ms / 1e3) / 1e9, "peak_GBps": hbm, "peak_kind": peak_kind}}
    roof["frac"] = roof["achieved"] / roof["peak"]
    line = {"metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "T": T, "H": H, "d_k": D, "d_v": D, "L": L,
                       "conv_width": wl.w, "pass": "backward",
                       "l2": L2_FLUSHED if small else "inputs larger than L2 (no flush)"},
            "roofline": roof, "clocks": clk,
            "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * backward_launches(B, T, H, D, L)}
    if not args.no_cpu_baseline:
        Ts, dts = grad_oracle_sample(host, wl, L, args.cpu_seconds)
        line["cpu_baseline"] = {"value": Ts / dts / H, "unit": UNIT, "cores": torch.get_num_threads(),
                                "kind": "oracle",
                                "sample": f"gradient oracle (torch fp64 autograd), sequence 0, head 0 of "
                                          f"{H}, first {Ts} tokens: {dts:.1f} s; scaled to tokens of all "
                                          f"{H} heads"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- graphs
def capture_graph(fn, dev):
    """A CUDA graph of the work ``fn`` issues on the current stream (warmed up before)."""
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.graph(graph, stream=side):
        fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    return graph


# ---------------------------------------------------------------- decode arm
DEC_METRIC = "PRISM mixer decode tokens/s on 1 GB300 (one token for every sequence, fp32 state)"


def dec_algorithmic(wl, L):
    """Bytes and flops of one decode step (every (b, h) advances one token), d = d_k = d_v,
    e = I/O bytes: per (b, h) the state read and written (8 d^2), q, k, v in (3 d e), the
    gates (8), out (4 d), the history read and rewritten (2 w d e); per head the L-step
    weights once (4 L (2 d^2 + d)) and the taps (4 w d).  Flops per (b, h): the
    projections 4 L d^2, S k and S q 4 d^2, the rank-(L+2) update 2 (L + 2) d^2."""
    d, e, w = wl.dk, (4 if wl.dtype == "f32" else 2), wl.w
    bh = wl.B * wl.H
    by = bh * (8 * d * d + 3 * d * e + 8 + 4 * d + 2 * w * d * e) + wl.H * 4 * (L * (2 * d * d + d) + w * d)
    fl = bh * (4 * L * d * d + 4 * d * d + 2 * (L + 2) * d * d)
    return by, fl


def decode_arm(args, wl, L):
    from linear_recurrent_sequence_causal_gb300 import build, prism
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if build.stale():
        raise RuntimeError("libprism.so is missing or stale: run __graft_entry__.build() first")
    prism.load()
    dev = torch.device("cuda", local)
    B, H, D, w = wl.B, wl.H, wl.dk, wl.w
    one = wl.with_(T=1, ragged=False)
    host = I.generate(one, L=L, seed=wl.seed)
    g = torch.Generator().manual_seed(wl.seed + 2)
    h_state = torch.randn((B, H, D, D), generator=g) * 0.1
    h_hist = torch.randn((B, H, w, D), generator=g).to(wl.torch_dtype)
    tok = {n: host[n][:, 0].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")}
    d_tok = {n: t.to(dev) for n, t in tok.items()}
    par = {n: host[n].to(dev) for n in ("conv_w", "Wk", "Wp", "wbeta")}
    state, hist = h_state.to(dev), h_hist.to(dev)
    out = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        prism.prism_decode_step(d_tok["q"], d_tok["k"], d_tok["v"], d_tok["log_alpha"], d_tok["beta"],
                                par["conv_w"], par["Wk"], par["Wp"], par["wbeta"], L, state, hist, out=out,
                                stream=stream)

    def step_on_current():                      # on the current stream (a graph capture's)
        prism.prism_decode_step(d_tok["q"], d_tok["k"], d_tok["v"], d_tok["log_alpha"], d_tok["beta"],
                                par["conv_w"], par["Wk"], par["Wp"], par["wbeta"], L, state, hist, out=out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    # The state of every sequence fits in L2 at these sizes, and a serving loop runs other
    # layers between two steps of this one: L2 is flushed before each step.  A decode step
    # is one short kernel, so it is timed inside CUDA graphs (as a serving loop issues it):
    # a graph of n_inner (flush, step) pairs and a graph of the n_inner flushes alone are
    # replayed in turn, and the step's device time is their difference over n_inner (the
    # median over the replays).  Events bracketing a single launch would add the launch's
    # own latency (several microseconds) to every step.
    flush = L2Flush(dev)
    n_inner = 20
    reps = max(1, max(args.steps, 100) // n_inner)
    steps = reps * n_inner

    def replay_ms(graph):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    def flushed_ms(fn):
        g_pair = capture_graph(lambda: [(flush(), fn()) for _ in range(n_inner)], dev)
        g_flush = capture_graph(lambda: [flush() for _ in range(n_inner)], dev)
        replay_ms(g_pair)
        replay_ms(g_flush)
        return statistics.median((replay_ms(g_pair) - replay_ms(g_flush)) / n_inner for _ in range(reps))

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = flushed_ms(step_on_current)
    clk = clocks.stop()
    value = B / (ms / 1e3)
    # for comparison, back-to-back steps with the state left in L2
    graph = capture_graph(lambda: [step_on_current() for _ in range(n_inner)], dev)
    replay_ms(graph)
    warm_ms = statistics.median(replay_ms(graph) / n_inner for _ in range(reps))

    # end to end: the token's q, k, v and gates from pinned host memory (packed in one
    # buffer, one copy), out back to the host
    names = ("q", "k", "v", "log_alpha", "beta")
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += (tok[n].numel() * tok[n].element_size() + 255) // 256 * 256
    h_pack = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for n in names:
        nb = tok[n].numel() * tok[n].element_size()
        h_pack[offs[n]:offs[n] + nb].copy_(tok[n].reshape(-1).view(torch.uint8))
    d_pack = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {n: d_pack[offs[n]:offs[n] + tok[n].numel() * tok[n].element_size()].view(tok[n].dtype)
             .view(tok[n].shape) for n in names}
    h_out = torch.empty((B, H, D), dtype=torch.float32).pin_memory()
    h2d = total
    d2h = h_out.numel() * 4

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        prism.prism_decode_step(views["q"], views["k"], views["v"], views["log_alpha"], views["beta"],
                                par["conv_w"], par["Wk"], par["Wp"], par["wbeta"], L, state, hist, out=out)
        h_out.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = flushed_ms(e2e_step)

    hbm, _, peak_kind = load_peaks()
    by, fl = dec_algorithmic(wl, L)
    roof = {"bound": "hbm", "achieved": by / (ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s", "traffic": None,
            "kernel": "decode_kernel", "peak_source": f"{peak_kind} (MEASURED_PEAKS.json)",
            "kernel_ms": ms, "algorithmic_bytes": by, "algorithmic_flops": fl}
    roof["frac"] = roof["achieved"] / roof["peak"]
    line = {"metric": DEC_METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "H": H, "d_k": D, "d_v": D, "L": L, "conv_width": w,
                       "pass": "decode (one token per sequence)",
                       "l2": "L2 flushed before each step (a 516 MB write); step time = (graph of "
                             "flush + step pairs - graph of the flushes) / steps",
                       "l2_resident_ms_per_step": warm_ms},
            "roofline": roof, "clocks": clk,
            "e2e": {"value": B / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": steps}
    if not args.no_cpu_baseline:
        import oracle
        inp1 = dict(host)
        inp1["seq_lens"] = None
        s0 = h_state.double().numpy()
        vh = h_hist.float().double().numpy()
        threads = os.cpu_count() or 1
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 5.0):
            oracle.forward(inp1, L=L, initial_state=s0, v_hist=vh, threads=threads)
            n += 1
        dt = (time.perf_counter() - t0) / n
        line["cpu_baseline"] = {"value": B / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"the fp64 oracle's forward on one token of all {B} x {H} "
                                          f"sequences from the same state, {n} runs"}
    print(json.dumps(line), flush=True)


def ctypes_byref(x):
    import ctypes
    return ctypes.byref(x)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--L", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true")
    ap.add_argument("--decode", action="store_true")
    ap.add_argument("--no-seq-split", action="store_true",
                    help="run the scan as one serial chain per sequence (PRISM_FLAG_NO_SEQ_SPLIT)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)     # at least 3 untimed warm-up steps, reported as run
    wl = I.get_workload(args.workload)
    L = wl.L if args.L is None else args.L
    if args.backward:
        backward_arm(args, wl, L)
    elif args.decode:
        decode_arm(args, wl, L)
    elif args.impl == "reference":
        reference_arm(args, wl, L)
    else:
        our_arm(args, wl, L)


if __name__ == "__main__":
    main()
