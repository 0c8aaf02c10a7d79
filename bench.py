"""Benchmark of the CSA2 decode step on GB300 (one JSON line on stdout).

Workload (default): decoder Full-mode decode, 32 sequences x 65,536 cached
tokens (m = 1), 8 indexer heads x 128 (FP8), 64 query heads, top-2048,
128-token window.  One step = append of the new token of every sequence
(FP4 latent + FP8 key) -> Full-mode indexer over the whole visible context ->
top-k -> sparse attention over the 2,048 selected entries + the window.
Metric: decode queries per second per layer (higher is better).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl csa2|reference]

`value`: device time of K steps with every input already in HBM; each step is
a CUDA-graph replay timed with CUDA events; L2 is flushed (a 512 MB write)
between steps, outside the timed events.  `e2e`: the same steps through the
public layer call with host (pinned) inputs copied in and the output copied
back inside the timed region, run back to back with the copies of one step
overlapping the kernels of its neighbours (`e2e.isolated`: each step timed
alone).  With N > 1 (torchrun) every rank runs its own
replica of the workload (weak scaling, no collective on the data path) and
the time is the max over ranks.  `--impl reference` times the float64 CPU
oracle on the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import csa2_inputs as ci  # noqa: E402

METRIC = "CSA2 decode queries/s/layer at 64K-1M ctx; HBM GB/s & FP8 util vs GB300 peak"
UNIT = "queries/s/layer"
L2_FLUSH_BYTES = 512 << 20
DTYPE = ("fp8 e4m3 indexer MMA (fp32 accumulate); f16 attention MMA operands (FP4 latents "
         "dequantised exactly to f16, bf16 q and window converted to f16, P in f16), fp32 "
         "accumulate and softmax")
# DRAM bytes (read + write) per visible entry of the decode indexer kernel,
# index_main_kernel, from ncu (dram__bytes_read.sum + dram__bytes_write.sum)
# on the 32 x 32,768 decode case; the capture's provenance is stated with the
# measurement notes.  None once the kernel has changed since that capture.
INDEX_DRAM_BYTES_PER_ENTRY = 135.8


def idx_bytes_per_entry(d_idx):
    """Algorithmic bytes of the indexer per scored entry: the FP8 key and its
    fp32 scale (the score write is not counted: it need not leave the chip)."""
    return d_idx + 4


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class _Nvml:
    """Read-only NVML queries through ctypes (the driver's libnvidia-ml), for
    the device torch calls `index` (found by UUID, else by PCI bus id)."""
    CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(index)
        rc = -1
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            u = str(uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            rc = self.lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h))
        if rc != 0 and hasattr(props, "pci_bus_id"):
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError(f"no NVML handle for device {index} (rc {rc})")
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    def sample(self):
        ct = self.ct
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(clk)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        if self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, ct.byref(rs)) != 0:
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(self.h, ct.byref(rs))
        names = [n for bit, n in self.REASONS.items() if rs.value & bit]
        return float(clk.value), pw.value / 1000.0, names


class Clocks:
    """SM clock, power and clock-event reasons sampled every millisecond during
    the timed region, in-process through NVML (read-only queries) on a
    background thread; if NVML cannot be used, an nvidia-smi child process
    queries the same device by UUID every 10 ms.  Errors are kept in the
    summary."""

    def __init__(self, index):
        self.index = index
        self.samples, self.errors = [], []
        self.max_mhz = None
        self._stop = None

    def __enter__(self):
        import threading
        try:
            nv = _Nvml(self.index)
            self.max_mhz = nv.max_mhz
            self._stop = threading.Event()

            def loop():
                while not self._stop.is_set():
                    try:
                        s_ = nv.sample()
                        if s_ is not None:
                            self.samples.append(s_)
                    except Exception as e:   # keep sampling; record the first error
                        if len(self.errors) < 3:
                            self.errors.append(f"nvml sample: {e}")
                    self._stop.wait(0.001)
            self._thr = threading.Thread(target=loop, daemon=True)
            self._thr.start()
            self.proc = None
        except Exception as e:
            self.errors.append(f"nvml: {e}")
            self._start_smi()
        return self

    def _start_smi(self):
        try:
            u = str(torch.cuda.get_device_properties(self.index).uuid)
            dev = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            dev = str(self.index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", dev,
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        except OSError as e:
            self.proc = None
            self.errors.append(f"nvidia-smi: {e}")

    def __exit__(self, *a):
        if self._stop is not None:
            self._stop.set()
            self._thr.join(timeout=5)
        if getattr(self, "proc", None) is not None:
            self.proc.terminate()
            try:
                out, err = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, err = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.max_mhz = float(f[1])
                    self.samples.append((float(f[0]), float(f[2]),
                                         [n for n, v in zip(names, f[3:7]) if v.lower() == "active"]))
                except (ValueError, IndexError):
                    continue
            if not self.samples and err:
                self.errors.append("nvidia-smi: " + err.strip()[:200])

    def summary(self):
        sm = [x[0] for x in self.samples]
        pw = [x[1] for x in self.samples]
        reasons = sorted({r for x in self.samples for r in x[2]})
        res = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(sm),
               "power_w_max": round(max(pw), 1) if pw else None,
               "source": "nvml" if self._stop is not None else "nvidia-smi"}
        if self.errors:
            res["errors"] = self.errors
        return res


def job_time(local_seconds, world, device):
    """The job's time: the slowest rank's time (every rank ran its own replica)."""
    if world <= 1:
        return local_seconds
    t = torch.tensor([local_seconds], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(queries_per_rank, world, seconds):
    """Whole-job throughput: the queries of every rank over the job's time."""
    return world * queries_per_rank / seconds


# ------------------------------------------------------------------ workload
def build_cache(csa, wl, dev, extra):
    """Fills every sequence's cache through the library's append (m = 1 here)."""
    caps = [(t + wl.new_tokens) // wl.m + extra for t in wl.ctx_tokens]
    cache = csa.Cache(caps, wl.d_idx, wl.m, dev)
    chunk = 65536
    for b, T in enumerate(wl.ctx_tokens):
        done = 0
        while done < T:
            n = min(chunk, T - done)
            C, Z = ci.latent_rows(wl, b, done, n, dev)
            key = ci.key_rows(wl, b, done // wl.m, n // wl.m, dev)
            csa.quantize_append(cache, C[None].contiguous(),
                                None if Z is None else Z[None].contiguous(), key[None].contiguous(),
                                seq=b)
            done += n
    torch.cuda.synchronize()
    return cache


def step_inputs(wl, step, B, dev):
    """Inputs of decode step `step`: the new token of every sequence, the
    indexer and attention queries of the layer."""
    T0 = wl.ctx_tokens[0]
    C = torch.stack([ci.latent_rows(wl, b, T0 + step, 1, dev)[0] for b in range(B)])
    key = torch.stack([ci.key_rows(wl, b, T0 + step, 1, dev) for b in range(B)])
    qi, w, qa = ci.query_inputs(wl, B, dev, layer=1000 + step)
    return dict(C=C.contiguous(), key=key.contiguous(), q_idx=qi.contiguous(), w=w.contiguous(),
                q=qa.contiguous())


def run_csa2(args, rank, world):
    import sparse_attention_decode_step_gb300 as csa
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = ci.config(2)
    if args.ctx:
        wl.ctx_tokens = [args.ctx] * wl.batch
        wl.name = f"decode_full_b{wl.batch}_ctx{args.ctx + 1}"
    if args.d_idx != 128:
        wl.d_idx = args.d_idx
        wl.name += f"_didx{args.d_idx}"
    B = wl.batch
    T0 = wl.ctx_tokens[0]
    n_steps = args.warmup + args.steps
    cache = build_cache(csa, wl, dev, extra=5 * n_steps + 16)   # value, phase, e2e (3 ways) steps
    wcap = 512
    win = ci.window_rows(wl, B, wcap, dev)          # ring buffers; every needed position filled

    # fixed staging buffers (the graph's inputs) and outputs
    stage = step_inputs(wl, 0, B, dev)
    inputs = [step_inputs(wl, s, B, dev) for s in range(n_steps)]
    q_pos = torch.full((B,), T0, dtype=torch.int32, device=dev)
    qs = csa.Queries(list(range(B)), [T0] * B, 1, dev)
    max_n = T0 + 2 * n_steps + 1
    ld = (max_n + 3) // 4 * 4
    scores = torch.empty(B, ld, device=dev)
    nv = torch.empty(B, dtype=torch.int32, device=dev)
    idx = torch.empty(B, wl.k, dtype=torch.int32, device=dev)
    cnt = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, wl.heads, 512, device=dev)
    lse = torch.empty(B, wl.heads, device=dev)
    counters = csa.new_counters(dev)
    iws = csa.workspace(csa.index_workspace_size(B, 1, wl.h_idx, wl.d_idx), dev)
    tws = csa.workspace(csa.topk_workspace_size(B, max_n), dev)
    aws = csa.workspace(csa.attn_workspace_size(B, wl.heads, wl.k, wl.n_win), dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    outer = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def ph_append():
        csa.quantize_append(cache, stage["C"], None, stage["key"], counters=counters)

    def ph_index():
        csa.index_full(cache, qs, stage["q_idx"], stage["w"], max_n, scores, n_valid=nv, ws=iws,
                       counters=counters)

    def ph_topk():
        csa.topk(scores, nv, wl.k, idx, cnt, max_n=max_n, ws=tws)

    def ph_attn():
        csa.sparse_attn(cache, qs, idx, cnt, stage["q"], win, wl.n_win, out, lse=lse,
                        ws=aws, counters=counters)

    # the step as a serving loop runs it: the append, then the layer call
    # (csa2_layer_step: indexer with the top-k's first histogram, top-k, attention)
    layer = csa.Layer(csa.FULL, cache, qs, k=wl.k, q=stage["q"], win=win, n_win=wl.n_win, out=out,
                      idx=idx, cnt=cnt, q_idx=stage["q_idx"], w=stage["w"], max_n=max_n, lse=lse,
                      counters=counters)
    step_fns = [ph_append, layer]
    # the same work as separate library calls, one graph each, for the phase split
    phase_fns = [ph_append, ph_index, ph_topk, ph_attn]
    appended = [0]

    def load_step(s):
        # step s appends the token at position T0 + (tokens appended so far)
        for k_ in stage:
            stage[k_].copy_(inputs[s % n_steps][k_])
        qs.q_pos.fill_(T0 + appended[0])
        appended[0] += 1

    # one CUDA graph for the whole step, and one per phase (for the phase split)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    l0 = csa.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for f in step_fns:
            f()
    launches_per_step = csa.launch_count() - l0
    pgraphs = []
    for f in phase_fns:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            f()
        pgraphs.append(g)

    times = []
    # clocks are sampled from the start of the warm-up to the end of the timed steps
    clocks = Clocks(torch.cuda.current_device()).__enter__()
    torch.cuda.synchronize()
    for s in range(n_steps):
        load_step(s)
        flush.fill_(s & 0xFF)                      # evict L2 between steps (not timed)
        if s == args.warmup:
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
        outer[0].record()
        graph.replay()
        outer[1].record()
        if s >= args.warmup:
            torch.cuda.synchronize()
            times.append(outer[0].elapsed_time(outer[1]) / 1e3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks.__exit__(None, None, None)
    total = job_time(sum(times), world, dev)
    ms = total / args.steps * 1e3

    # ---- phase split: the same steps with one graph per phase, events between them
    ph = np.zeros(4)
    n_ph = max(1, min(args.steps, 50))
    for s in range(n_ph):
        load_step(s)
        flush.fill_(s & 0xFF)
        torch.cuda.synchronize()
        ev[0].record()
        for i, g in enumerate(pgraphs):
            g.replay()
            ev[i + 1].record()
        torch.cuda.synchronize()
        ph += [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(4)]
    ph /= n_ph
    assert int(counters[csa.CNT_BAD_INPUT]) == 0 and int(counters[csa.CNT_TIMEOUT]) == 0, counters

    # ---- end to end: pinned host inputs in, output back, through the layer call
    e2e = None if args.quick else run_e2e(csa, args, wl, cache, win, dev, n_steps, B, T0, world)

    # ---- kernel durations for the rooflines: the library call alone between two
    # CUDA events on its stream, queued behind the L2 flush (so the GPU never
    # waits for the host to submit it), averaged over 20 calls
    def timed_call(fn, reps=20):
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for s in range(reps + 2):
            flush.fill_(s & 0xFF)
            ea.record()
            fn()
            eb.record()
            torch.cuda.synchronize()
            if s >= 2:
                ts.append(ea.elapsed_time(eb) / 1e3)
        return sum(ts) / len(ts)

    t_index = timed_call(ph_index)
    t_attn = timed_call(ph_attn)
    t_layer = timed_call(layer)
    # the append variant whose indexer keys are projected from the stored
    # entries (random-init bf16 W_IK), the same 32 new tokens
    g = torch.Generator(device=dev).manual_seed(7)
    w_ik = (torch.randn(512, wl.d_idx, generator=g, device=dev) / 16).to(torch.bfloat16)
    t_proj = timed_call(lambda: csa.quantize_append_project(cache, stage["C"], None, w_ik,
                                                            counters=counters))

    # ---- roofline of the dominant kernel (Full-mode indexer)
    hbm, bf16, src = peaks()
    entries = B * (int(qs.q_pos[0]) + 1)                 # visible entries of those calls
    idx_bytes = entries * idx_bytes_per_entry(wl.d_idx)
    achieved = idx_bytes / t_index / 1e9
    traffic = INDEX_DRAM_BYTES_PER_ENTRY if wl.d_idx == 128 else None
    roof = {"kernel": "index_main_kernel (+ index_prep_kernel; one csa2_index_full call)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_source": src,
            "traffic": None if traffic is None else round(traffic * entries),
            "algorithmic_bytes_per_launch": round(idx_bytes),
            "launch_us": round(t_index * 1e6, 2)}
    attn_bytes = B * (wl.k * 288 + wl.n_win * 1024 + wl.heads * 512 * 2 + wl.heads * 512 * 4 +
                      wl.k * 4)
    attn_flops = B * 4 * wl.heads * 512 * (wl.k + wl.n_win)
    res = {
        "metric": METRIC, "value": round(job_value(B * args.steps, world, total), 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic (seeded counter-hash generator; N(0,1) latents scaled to norm sqrt(512))",
        "config": {"workload": wl.name, "batch": B, "ctx_tokens": T0 + 1, "m": wl.m,
                   "indexer_heads": wl.h_idx, "d_idx": wl.d_idx, "heads": wl.heads, "k": wl.k,
                   "n_win": wl.n_win, "layers": 1, "l2": "flushed between steps (512 MB write)",
                   "graph": "one CUDA graph replay per step (csa2_quantize_append + "
                            "csa2_layer_step)", "parallelism": f"replicas x{world}"},
        "phases_us": {"append": round(ph[0] * 1e6, 2), "index_full": round(ph[1] * 1e6, 2),
                      "topk": round(ph[2] * 1e6, 2), "sparse_attn": round(ph[3] * 1e6, 2),
                      "note": "the step's work as separate library calls, one graph each; the "
                              "timed step is the append plus one csa2_layer_step call"},
        "layer_call_us": round(t_layer * 1e6, 2),
        "attn_roofline": {"kernel": "attn_tc_kernel (one csa2_sparse_attn call)", "bound": "hbm",
                          "achieved": round(attn_bytes / t_attn / 1e9, 1), "peak": hbm,
                          "unit": "GB/s", "frac": round(attn_bytes / t_attn / 1e9 / hbm, 4),
                          "peak_source": src, "traffic": None,
                          "algorithmic_bytes_per_launch": attn_bytes,
                          "launch_us": round(t_attn * 1e6, 2),
                          "hbm_frac": round(attn_bytes / t_attn / 1e9 / hbm, 4),
                          "bf16": {"achieved": round(attn_flops / t_attn / 1e12, 1),
                                   "peak": bf16, "unit": "TFLOP/s",
                                   "frac": round(attn_flops / t_attn / 1e12 / bf16, 4),
                                   "algorithmic_flops_per_launch": attn_flops},
                          "bf16_frac": round(attn_flops / t_attn / 1e12 / bf16, 4)},
        "roofline": roof, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "append_project": {"entries": B, "launch_us": round(t_proj * 1e6, 2),
                           "note": "append with keys projected from the stored entries (not "
                                   "part of the timed step)"},
    }
    if rank == 0 and not args.quick:
        res["cpu_baseline"] = cpu_baseline(wl, cache, win, inputs[args.warmup], T0 + args.warmup)
    return res


def run_e2e(csa, args, wl, cache, win, dev, n_steps, B, T0, world):
    """Pinned host inputs -> device -> append + layer call -> output back to the
    host.  A step's inputs travel packed in one buffer of a pinned ring (filled
    before the timed region, as a serving loop's staging ring would be) with one
    host-to-device copy; the output comes back with one copy.

    The headline figure runs the steps back to back as a serving loop would:
    step s's input copy and output copy run on their own streams, overlapping
    the kernels of the neighbouring steps (every step's copies are inside the
    timed region; the 270 MB key cache keeps the inputs larger than L2).  The
    `isolated` figures time each step alone, L2 flushed before it, eagerly and
    as a CUDA graph."""
    order = ["C", "key", "q_idx", "w", "q"]
    first = step_inputs(wl, 0, B, "cpu")
    offs, nbytes = {}, 0
    for k_ in order:
        offs[k_] = nbytes
        nbytes += (first[k_].numel() * first[k_].element_size() + 255) // 256 * 256
    ring = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(4)]
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def view(buf, k_):
        t = first[k_]
        n = t.numel() * t.element_size()
        return buf[offs[k_]:offs[k_] + n].view(t.dtype).view(t.shape)

    dstage = {k_: view(dbuf, k_) for k_ in order}
    qs = csa.Queries(list(range(B)), [T0] * B, 1, dev)
    idx = torch.empty(B, wl.k, dtype=torch.int32, device=dev)
    cnt = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, wl.heads, 512, device=dev)
    out_h = torch.empty(B, wl.heads, 512).pin_memory()
    max_n = T0 + 5 * n_steps + 2
    layer = csa.Layer(csa.FULL, cache, qs, k=wl.k, q=dstage["q"], win=win, n_win=wl.n_win,
                      out=out, idx=idx, cnt=cnt, q_idx=dstage["q_idx"], w=dstage["w"], max_n=max_n)
    base_len = cache.seq_len.clone()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for s in range(n_steps):
        slot = ring[s % len(ring)]
        inp = step_inputs(wl, s, B, "cpu")
        for k_ in order:
            view(slot, k_).copy_(inp[k_])            # host-side staging, not timed
        qs.q_pos.copy_(base_len + s)      # the new token's position (after earlier appends)
        flush.fill_(1)
        torch.cuda.synchronize()
        e0.record()
        dbuf.copy_(slot, non_blocking=True)
        csa.quantize_append(cache, dstage["C"], None, dstage["key"])
        layer()
        out_h.copy_(out, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        if s >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    total = job_time(sum(times), world, dev)
    res = {"value": round(job_value(B * args.steps, world, total), 1), "unit": UNIT,
           "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": out_h.numel() * 4,
           "ms_per_step": round(total / args.steps * 1e3, 4)}

    # The same calls and copies captured once per staging slot as a CUDA graph
    # (what a serving loop does to take the host's launch cost off the step),
    # replayed with the same per-step staging and timing.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = []
    for slot in ring:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            dbuf.copy_(slot, non_blocking=True)
            csa.quantize_append(cache, dstage["C"], None, dstage["key"])
            layer()
            out_h.copy_(out, non_blocking=True)
        graphs.append(g)
    torch.cuda.synchronize()
    base_len = cache.seq_len.clone()
    times = []
    for s in range(n_steps):
        slot = ring[s % len(ring)]
        inp = step_inputs(wl, n_steps + s, B, "cpu")
        for k_ in order:
            view(slot, k_).copy_(inp[k_])
        qs.q_pos.copy_(base_len + s)
        flush.fill_(1)
        torch.cuda.synchronize()
        e0.record()
        graphs[s % len(ring)].replay()
        e1.record()
        torch.cuda.synchronize()
        if s >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    total = job_time(sum(times), world, dev)
    res["graph"] = {"value": round(job_value(B * args.steps, world, total), 1),
                    "ms_per_step": round(total / args.steps * 1e3, 4)}

    # ---- pipelined: R slots of device inputs and outputs; H2D, compute and D2H
    # of consecutive steps on three streams, ordered by events
    R = len(ring)
    dbufs = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(R)]
    douts = [torch.empty(B, wl.heads, 512, device=dev) for _ in range(R)]
    outs_h = [torch.empty(B, wl.heads, 512).pin_memory() for _ in range(R)]
    layers = [csa.Layer(csa.FULL, cache, qs, k=wl.k, q=view(dbufs[r], "q"), win=win, n_win=wl.n_win,
                        out=douts[r], idx=idx, cnt=cnt, q_idx=view(dbufs[r], "q_idx"),
                        w=view(dbufs[r], "w"), max_n=max_n, ws=layer.ws) for r in range(R)]
    main = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(R)]
    ev_done = [torch.cuda.Event() for _ in range(R)]
    ev_out = [torch.cuda.Event() for _ in range(R)]
    base_len = cache.seq_len.clone()

    def run(s0, count):
        for s in range(s0, s0 + count):
            r = s % R
            if s >= R:
                h2d.wait_event(ev_done[r])           # step s - R has finished with dbufs[r]
            with torch.cuda.stream(h2d):
                dbufs[r].copy_(ring[r], non_blocking=True)
                ev_in[r].record(h2d)
            main.wait_event(ev_in[r])
            if s >= R:
                main.wait_event(ev_out[r])           # step s - R's output has left douts[r]
            qs.q_pos.copy_(base_len + s)
            csa.quantize_append(cache, view(dbufs[r], "C"), None, view(dbufs[r], "key"))
            layers[r]()
            ev_done[r].record(main)
            d2h.wait_event(ev_done[r])
            with torch.cuda.stream(d2h):
                outs_h[r].copy_(douts[r], non_blocking=True)
                ev_out[r].record(d2h)
        main.wait_stream(d2h)
        main.wait_stream(h2d)

    run(0, args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0.record()
    run(args.warmup, args.steps)
    e1.record()
    torch.cuda.synchronize()
    total = job_time(e0.elapsed_time(e1) / 1e3, world, dev)
    isolated = {"value": res["value"], "ms_per_step": res["ms_per_step"], "graph": res.pop("graph"),
                "l2": "flushed before each step"}
    res["value"] = round(job_value(B * args.steps, world, total), 1)
    res["ms_per_step"] = round(total / args.steps * 1e3, 4)
    res["l2"] = "not flushed: steps back to back, inputs (the key cache) larger than L2"
    res["isolated"] = isolated
    return res


def cpu_baseline(wl, cache, win, inp, t):
    """The float64 oracle on a bounded sample: one step's 32 queries, each over
    its full 65,536-entry context (host cores, OpenMP over queries), repeated
    until about 10 s of wall time have been spent."""
    import oracle as O
    B = wl.batch
    n = t + 1
    rows = []
    codes = cache.codes.cpu().numpy()
    scales = cache.scales.cpu().numpy()
    kidx = cache.kidx.cpu().numpy()
    ksc = cache.kscale.cpu().numpy()
    base = np.array(cache.base_host[:B], np.int64)
    O.set_threads(os.cpu_count() or 1)
    q_attn = inp["q"][:B].cpu().numpy().view(np.uint16)
    win_h = win[:B].cpu().numpy().view(np.uint16)
    q_idx, w = inp["q_idx"][:B].cpu().numpy(), inp["w"][:B].cpu().numpy()
    reps = 0
    t0 = time.perf_counter()
    while True:
        O.layer(O.FULL, codes=codes, scales=scales, kidx=kidx, kscale=ksc, seq_base=base, m=1,
                q_seq=list(range(B)), q_pos=[t] * B, k=wl.k, H=wl.heads, q_attn=q_attn,
                win=win_h, wcap=win.shape[1], n_win=wl.n_win, sm_scale=1.0, q_idx=q_idx, w=w)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0 or reps >= 200:
            break
    return {"value": round(B * reps / dt, 3), "unit": UNIT, "cores": O.max_threads(), "kind": "oracle",
            "sample": f"{reps} x {B} queries x {n} entries (one Full layer: scoring, top-{wl.k}, "
                      f"attention), {dt:.1f} s wall"}


# ---------------------------------------------------------------- other workloads
# Reindex decode at 1M, encoder prefill and the 20-layer decoder schedule: the
# same library calls, timed as CUDA-graph replays with L2 flushed between steps.
# They print their own JSON line (python bench.py --workload NAME); the default
# line above is the 64K Full-mode decode.

def timed_graphs(fns, steps, warmup, flush, before=None):
    """One graph for the whole step and one per phase; returns (seconds per
    step, seconds per phase)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=side):
        for f in fns:
            f()
    gs = []
    for f in fns:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            f()
        gs.append(g)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
    tot = []
    for s in range(warmup + steps):
        if before:
            before(s)
        flush.fill_(s & 0xFF)
        torch.cuda.synchronize()
        ev[0].record()
        g_all.replay()
        ev[1].record()
        torch.cuda.synchronize()
        if s >= warmup:
            tot.append(ev[0].elapsed_time(ev[1]) / 1e3)
    ph = np.zeros(len(fns))
    n_ph = max(1, min(steps, 20))
    for s in range(n_ph):
        if before:
            before(s)
        flush.fill_(s & 0xFF)
        torch.cuda.synchronize()
        ev[0].record()
        for i, g in enumerate(gs):
            g.replay()
            ev[i + 1].record()
        torch.cuda.synchronize()
        ph += [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(len(fns))]
    return sum(tot) / len(tot), ph / n_ph


def _line(name, wl, args, world, value, unit, ms, phases, roofline, clocks, extra):
    res = {"metric": METRIC, "value": round(value, 1), "unit": unit, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": DTYPE,
           "data": "synthetic (seeded counter-hash generator)",
           "config": {"workload": wl.name, "l2": "flushed between steps (512 MB write)",
                      "graph": "one CUDA graph replay per step", "parallelism": f"replicas x{world}"},
           "phases_us": {k: round(v * 1e6, 2) for k, v in phases.items()},
           "roofline": roofline, "clocks": clocks.summary()}
    res["config"].update(extra)
    return res


def run_reindex(csa, args, world, dev):
    """Reindex layer over the 2,048 x 8 candidate pool at 1M context, 8 sequences."""
    wl = ci.config(3)
    B, T = wl.batch, wl.ctx_tokens[0]
    cache = build_cache(csa, wl, dev, extra=8)
    n = T                                          # entries visible to a query at position T - 1
    qs = csa.Queries(list(range(B)), [T - 1] * B, 1, dev)
    wcap = 512
    win = ci.window_rows(wl, B, wcap, dev)
    pool_blk = torch.zeros(B, 2048, dtype=torch.int32, device=dev)
    pool_n = torch.zeros(B, dtype=torch.int32, device=dev)
    qi0, w0, qa0 = ci.query_inputs(wl, B, dev, layer=0)
    qi, w, qa = ci.query_inputs(wl, B, dev, layer=1)
    idx = torch.zeros(B, wl.k, dtype=torch.int32, device=dev)
    cnt = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.zeros(B, wl.heads, 512, device=dev)
    counters = csa.new_counters(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # the Full layer that builds the pool (timed once, for context)
    full = csa.Layer(csa.FULL, cache, qs, k=wl.k, q=qa0, win=win, n_win=wl.n_win, out=out,
                     idx=idx, cnt=cnt, q_idx=qi0, w=w0, max_n=n, build_pool=True,
                     pool_blk=pool_blk, pool_n=pool_n, counters=counters)
    full()
    torch.cuda.synchronize()
    flush.fill_(1)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    full()
    e1.record()
    torch.cuda.synchronize()
    full_us = e0.elapsed_time(e1) * 1e3
    npool = 2048 * 8
    scores = torch.empty(B, npool, device=dev)
    nv = torch.empty(B, dtype=torch.int32, device=dev)
    iws = csa.workspace(csa.index_workspace_size(B, 1, wl.h_idx, wl.d_idx), dev)
    tws = csa.workspace(csa.topk_workspace_size(B, npool), dev)
    aws = csa.workspace(csa.attn_workspace_size(B, wl.heads, wl.k, wl.n_win), dev)
    fns = [lambda: csa.index_reindex(cache, qs, qi, w, pool_blk, pool_n, scores, n_valid=nv,
                                     ws=iws, counters=counters),
           lambda: csa.topk(scores, nv, wl.k, idx, cnt, max_n=npool, pool_blk=pool_blk, ws=tws),
           lambda: csa.sparse_attn(cache, qs, idx, cnt, qa, win, wl.n_win, out, ws=aws,
                                   counters=counters)]
    clocks = Clocks(torch.cuda.current_device()).__enter__()
    sec, ph = timed_graphs(fns, args.steps, args.warmup, flush)
    clocks.__exit__(None, None, None)
    assert int(counters[csa.CNT_BAD_INPUT]) == 0 and int(counters[csa.CNT_TIMEOUT]) == 0, counters
    pn = int(pool_n.sum())
    hbm, _bf16, src = peaks()
    ib = pn * idx_bytes_per_entry(wl.d_idx) + B * 2048 * 4
    roof = {"kernel": "index_main_kernel (Reindex, 8-row TMA boxes)", "bound": "hbm",
            "achieved": round(ib / ph[0] / 1e9, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(ib / ph[0] / 1e9 / hbm, 4), "peak_source": src, "traffic": None,
            "algorithmic_bytes_per_launch": ib}
    return _line("reindex", wl, args, world, B / sec, UNIT, sec * 1e3,
                 {"index_reindex": ph[0], "topk_pool": ph[1], "sparse_attn": ph[2]}, roof, clocks,
                 {"batch": B, "ctx_tokens": T, "m": 1, "pool_positions": pn // B, "k": wl.k,
                  "heads": wl.heads, "full_layer_with_pool_us": round(full_us, 1)})


def run_prefill(csa, args, world, dev):
    """Encoder prefill chunk at m = 2: 4,096 causal queries after a 262,144-token
    prefix; one Full layer (scoring all visible entries, top-2048, attention)
    and five Reuse layers."""
    wl = ci.config(4)
    if args.ctx or args.queries:                          # smaller profiling case
        wl.ctx_tokens = [args.ctx or wl.ctx_tokens[0]]
        wl.q_per_seq = wl.new_tokens = args.queries or wl.q_per_seq
        assert wl.ctx_tokens[0] % wl.m == 0 and wl.q_per_seq % (wl.group * wl.m) == 0
        wl.name = f"prefill_m{wl.m}_prefix{wl.ctx_tokens[0]}_q{wl.q_per_seq}"
    P, nq, m = wl.ctx_tokens[0], wl.q_per_seq, wl.m
    cache = build_cache(csa, wl, dev, extra=nq // m + 8)
    C, Z = ci.latent_rows(wl, 0, P, nq, dev)
    key = ci.key_rows(wl, 0, P // m, nq // m, dev)
    csa.quantize_append(cache, C[None].contiguous(), Z[None].contiguous(), key[None].contiguous(), seq=0)
    q_pos = [P + i for i in range(nq)]
    qs = csa.Queries([0] * nq, q_pos, wl.group, dev)
    n_max = (P + nq) // m
    ld = (n_max + 3) // 4 * 4
    scores = torch.empty(nq, ld, device=dev)
    nv = torch.empty(nq, dtype=torch.int32, device=dev)
    idx = torch.zeros(nq, wl.k, dtype=torch.int32, device=dev)
    cnt = torch.zeros(nq, dtype=torch.int32, device=dev)
    wcap = 8192
    layers = []
    for layer in range(6):
        qi, w, qa = ci.query_inputs(wl, nq, dev, layer=layer)
        layers.append(dict(qi=qi, w=w, qa=qa, win=ci.window_rows(wl, 1, wcap, dev, layer=layer),
                           out=torch.empty(nq, wl.heads, 512, device=dev)))
    counters = csa.new_counters(dev)
    iws = csa.workspace(csa.index_workspace_size(nq, wl.group, wl.h_idx, wl.d_idx), dev)
    tws = csa.workspace(csa.topk_workspace_size(nq, n_max), dev)
    aws = csa.workspace(csa.attn_workspace_size(nq, wl.heads, wl.k, wl.n_win), dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    L0 = layers[0]
    fns = [lambda: csa.index_full(cache, qs, L0["qi"], L0["w"], n_max, scores, n_valid=nv, ws=iws,
                                  counters=counters),
           lambda: csa.topk(scores, nv, wl.k, idx, cnt, max_n=n_max, ws=tws),
           lambda: csa.sparse_attn(cache, qs, idx, cnt, L0["qa"], L0["win"], wl.n_win, L0["out"],
                                   ws=aws, counters=counters)]
    for Ly in layers[1:]:
        fns.append(lambda Ly=Ly: csa.sparse_attn(cache, qs, idx, cnt, Ly["qa"], Ly["win"], wl.n_win,
                                                 Ly["out"], ws=aws, counters=counters))
    clocks = Clocks(torch.cuda.current_device()).__enter__()
    sec, ph = timed_graphs(fns, args.steps, args.warmup, flush)
    clocks.__exit__(None, None, None)
    assert int(counters[csa.CNT_BAD_INPUT]) == 0 and int(counters[csa.CNT_TIMEOUT]) == 0, counters
    pairs = sum((t + 1) // m for t in q_pos)              # (query, visible entry) pairs
    flops = pairs * 2 * wl.h_idx * wl.d_idx
    _hbm, bf16, src = peaks()
    fp8 = 2.0 * bf16                                      # FP8 dense = 2 x bf16 (nominal ratio)
    roof = {"kernel": "index_main_kernel (prefill, N = 32 queries x 8 heads)", "bound": "tensor",
            "achieved": round(flops / ph[0] / 1e12, 1), "peak": round(fp8, 1), "unit": "TFLOP/s",
            "frac": round(flops / ph[0] / 1e12 / fp8, 4),
            "peak_source": f"{src} bf16 x 2 (nominal fp8/bf16 ratio)", "traffic": None,
            "algorithmic_flops_per_launch": flops}
    attn_flops = nq * 4 * wl.heads * 512 * (wl.k + wl.n_win)
    phases = {"index_full": ph[0], "topk": ph[1], "sparse_attn_full": ph[2],
              "sparse_attn_reuse_x5": float(sum(ph[3:]))}
    res = _line("prefill", wl, args, world, nq * 6 / sec, "queries*layers/s", sec * 1e3, phases,
                roof, clocks, {"queries": nq, "prefix_tokens": P, "m": m, "group": wl.group,
                               "k": wl.k, "heads": wl.heads, "layers": "1 Full + 5 Reuse"})
    res["attn_bf16_frac"] = round(attn_flops / ph[2] / 1e12 / bf16, 4)
    # the chunk's append with keys projected from the stored entries (random-init
    # bf16 W_IK): nq / m entries, re-appended at the same rows each time
    g = torch.Generator(device=dev).manual_seed(7)
    w_ik = (torch.randn(512, wl.d_idx, generator=g, device=dev) / 16).to(torch.bfloat16)
    len0 = cache.seq_len.clone() - nq // m
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for s_ in range(22):
        flush.fill_(s_ & 0xFF)
        cache.seq_len.copy_(len0)
        ea.record()
        csa.quantize_append_project(cache, C[None].contiguous(), Z[None].contiguous(), w_ik,
                                    counters=counters, seq=0)
        eb.record()
        torch.cuda.synchronize()
        if s_ >= 2:
            ts.append(ea.elapsed_time(eb) / 1e3)
    res["append_project"] = {"entries": nq // m, "launch_us": round(sum(ts) / len(ts) * 1e6, 2),
                             "note": "append with keys projected from the stored entries (not "
                                     "part of the timed step)"}
    return res


def run_encoder(csa, args, world, dev):
    """The encoder's 18 CSA2 layers over one chunk of 4,096 causal queries
    after a 262,144-token prefix: three blocks of 1 Full + 5 Reuse at m = 2,
    each block with its own cache (the chunk's tokens appended to all three)."""
    from sparse_attention_decode_step_gb300 import schedule as S
    base = ci.config(4)
    P, nq, m = base.ctx_tokens[0], base.q_per_seq, base.m
    if args.ctx or args.queries:                          # smaller profiling case
        P, nq = args.ctx or P, args.queries or nq
        assert P % m == 0 and nq % (base.group * m) == 0
    name = f"encoder_m{m}_prefix{P}_q{nq}"
    wls = [ci.Workload(f"{name}_block{b}", 1, [P], nq, m, rms_norm=True, seed=base.seed + 100 * b,
                       group=base.group, q_per_seq=nq) for b in range(3)]
    caches = []
    for wl in wls:
        cache = build_cache(csa, wl, dev, extra=nq // m + 8)
        C, Z = ci.latent_rows(wl, 0, P, nq, dev)
        key = ci.key_rows(wl, 0, P // m, nq // m, dev)
        csa.quantize_append(cache, C[None].contiguous(), Z[None].contiguous(), key[None].contiguous(),
                            seq=0)
        caches.append(cache)
    q_pos = [P + i for i in range(nq)]
    qs = csa.Queries([0] * nq, q_pos, base.group, dev)
    n_max = (P + nq) // m
    wcap = 8192
    plan = S.encoder_csa2_layers()
    per_layer = []
    for i, p in enumerate(plan):
        wl = wls[p.cache]
        qi, w, qa = ci.query_inputs(wl, nq, dev, layer=i)
        per_layer.append(dict(q_idx=qi, w=w, q=qa, win=ci.window_rows(wl, 1, wcap, dev, layer=i),
                              out=torch.empty(nq, wl.heads, 512, device=dev)))
    counters = csa.new_counters(dev)
    chunk = S.EncoderChunk(csa, caches, qs, per_layer, k=base.k, n_win=base.n_win, max_n=n_max,
                           counters=counters)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fns = list(chunk.layers)                              # one phase per layer
    clocks = Clocks(torch.cuda.current_device()).__enter__()
    sec, ph = timed_graphs(fns, args.steps, args.warmup, flush)
    clocks.__exit__(None, None, None)
    assert int(counters[csa.CNT_BAD_INPUT]) == 0 and int(counters[csa.CNT_TIMEOUT]) == 0, counters
    _hbm, bf16, src = peaks()
    reuse = [ph[i] for i, p in enumerate(plan) if p.mode == S.REUSE]
    attn_flops = nq * 4 * base.heads * 512 * (base.k + base.n_win)   # one layer's attention
    achieved = attn_flops * len(reuse) / sum(reuse) / 1e12
    roof = {"kernel": "attn_tc_kernel (the 15 Reuse layers: attention alone)", "bound": "tensor",
            "achieved": round(achieved, 1), "peak": round(bf16, 1), "unit": "TFLOP/s",
            "frac": round(achieved / bf16, 4), "peak_source": src, "traffic": None,
            "algorithmic_flops_per_launch": attn_flops}
    phases = {}
    for b in range(3):
        lay = [i for i, p in enumerate(plan) if p.cache == b]
        phases[f"block{b + 1}_full"] = ph[lay[0]]
        phases[f"block{b + 1}_reuse_x5"] = float(sum(ph[i] for i in lay[1:]))
    wl0 = wls[0]
    wl0.name = name
    return _line("encoder", wl0, args, world, nq * len(plan) / sec, "queries*layers/s", sec * 1e3,
                 phases, roof, clocks,
                 {"queries": nq, "prefix_tokens": P, "m": m, "group": base.group, "k": base.k,
                  "heads": base.heads, "layers": "3 x (1 Full + 5 Reuse), three caches"})


def run_schedule(csa, args, world, dev):
    """The 20-layer decoder (1 Full + 4 Reindex + 15 Reuse) over 64 sequences
    with log-uniform contexts in [4,096, 1,048,576], one query each."""
    from sparse_attention_decode_step_gb300 import schedule as S
    base = ci.config(5)
    lens = base.ctx_tokens
    wl = ci.Workload(base.name, base.batch, lens, 0, 1, rms_norm=True, seed=base.seed)
    cache = build_cache(csa, wl, dev, extra=8)
    B = wl.batch
    q_pos = [t - 1 for t in lens]
    qs = csa.Queries(list(range(B)), q_pos, 1, dev)
    wcap = 256
    per_layer = []
    for layer in range(20):
        qi, w, qa = ci.query_inputs(wl, B, dev, layer=layer)
        per_layer.append(dict(q_idx=qi, w=w, q=qa, win=ci.window_rows(wl, B, wcap, dev, layer=layer),
                              out=torch.empty(B, wl.heads, 512, device=dev)))
    counters = csa.new_counters(dev)
    step = S.DecoderStep(csa, cache, qs, per_layer, k=wl.k, n_win=wl.n_win,
                         max_n=max(lens), counters=counters)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fns = [step.layers[0]] + [lambda: [L() for L in step.layers[1:]]]
    clocks = Clocks(torch.cuda.current_device()).__enter__()
    sec, ph = timed_graphs(fns, args.steps, args.warmup, flush)
    clocks.__exit__(None, None, None)
    assert int(counters[csa.CNT_BAD_INPUT]) == 0 and int(counters[csa.CNT_TIMEOUT]) == 0, counters
    hbm, _bf16, src = peaks()
    ib = sum(lens) * idx_bytes_per_entry(wl.d_idx)
    roof = {"kernel": "index_main_kernel (layer-1 Full scoring)", "bound": "hbm",
            "achieved": None, "peak": hbm, "unit": "GB/s", "frac": None, "peak_source": src,
            "traffic": None, "algorithmic_bytes_full_layer": ib,
            "note": "the Full layer's phase also holds its pool build, top-k and attention"}
    return _line("schedule", wl, args, world, B * 20 / sec, "queries*layers/s", sec * 1e3,
                 {"layer1_full_with_pool": ph[0], "layers2_20": ph[1]}, roof, clocks,
                 {"batch": B, "ctx_tokens": "log-uniform [4096, 1048576]",
                  "mean_ctx": int(sum(lens) / B), "layers": "1 Full + 4 Reindex + 15 Reuse",
                  "k": wl.k, "heads": wl.heads})


def extra_workloads(args, world):
    """The other configurations at their full sizes, each as in its own
    --workload run but with fewer steps: Reindex decode over the candidate pool
    at 1M context, the 20-layer decoder over 64 log-uniform contexts, and the
    m = 2 prefill chunk (its FP8 scoring roofline).  Each entry keeps the
    workload's value, ms_per_step, phase split, roofline and clock record."""
    import sparse_attention_decode_step_gb300 as csa
    dev = torch.device("cuda", torch.cuda.current_device())
    sub = argparse.Namespace(**vars(args))
    sub.steps, sub.warmup, sub.ctx, sub.queries = min(args.steps, 10), 3, 0, 0
    out = {}
    for key, fn in (("reindex_b8_1m", run_reindex), ("schedule20_b64", run_schedule),
                    ("prefill_m2_q4096", run_prefill)):
        torch.cuda.empty_cache()
        r = fn(csa, sub, world, dev)
        keep = ["value", "unit", "ms_per_step", "steps", "warmup", "phases_us", "roofline",
                "clocks", "config", "attn_bf16_frac", "append_project"]
        out[key] = {k_: r[k_] for k_ in keep if k_ in r}
    torch.cuda.empty_cache()
    return out


def run_reference(args, rank, world):
    """The float64 oracle, timed on the host cores, on the same workload."""
    if rank != 0:
        return None
    import oracle as O
    wl = ci.config(2)
    B_s = max(1, min(wl.batch, os.cpu_count() or 1))   # one query per host core per step
    T0 = wl.ctx_tokens[0]
    n = T0 + 1
    # the sample's caches: oracle-encoded entries of B_s sequences
    caches = []
    for b in range(B_s):
        C, _ = ci.latent_rows(wl, b, 0, n, "cpu")
        key = ci.key_rows(wl, b, 0, n, "cpu")
        codes, scales, kidx, ksc, _x, _ = O.append(C.numpy()[None], None, key.numpy()[None], 1)
        caches.append((codes, scales, kidx, ksc))
    codes = np.concatenate([c[0] for c in caches])
    scales = np.concatenate([c[1] for c in caches])
    kidx = np.concatenate([c[2] for c in caches])
    ksc = np.concatenate([c[3] for c in caches])
    base = np.arange(B_s, dtype=np.int64) * n
    win = ci.window_rows(wl, B_s, 512, "cpu").numpy().view(np.uint16)
    O.set_threads(os.cpu_count() or 1)
    times = []
    for s in range(args.warmup + args.steps):
        qi, w, qa = ci.query_inputs(wl, wl.batch, "cpu", layer=1000 + s)
        t0 = time.perf_counter()
        O.layer(O.FULL, codes=codes, scales=scales, kidx=kidx, kscale=ksc, seq_base=base, m=1,
                q_seq=list(range(B_s)), q_pos=[T0] * B_s, k=wl.k, H=wl.heads,
                q_attn=qa[:B_s].numpy().view(np.uint16), win=win, wcap=512, n_win=wl.n_win,
                sm_scale=1.0, q_idx=qi[:B_s].numpy(), w=w[:B_s].numpy())
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    v = round(B_s * args.steps / total, 3)
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "batch": wl.batch, "ctx_tokens": n, "m": 1,
                       "k": wl.k, "heads": wl.heads, "sample_queries_per_step": B_s},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": O.max_threads(), "kind": "oracle",
                             "sample": f"{B_s} of {wl.batch} queries per step, full 65,536-entry "
                                       f"contexts, {args.steps} steps"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="csa2", choices=["csa2", "reference"])
    ap.add_argument("--ctx", type=int, default=0,
                    help="profiling case: cached tokens per sequence instead of 65,535 "
                         "(prefill, encoder: prefix tokens instead of 262,144)")
    ap.add_argument("--queries", type=int, default=0,
                    help="profiling case, prefill / encoder: queries instead of 4,096 (a multiple "
                         "of 64)")
    ap.add_argument("--quick", action="store_true",
                    help="profiling case: skip the e2e and CPU-baseline legs")
    ap.add_argument("--no-extra", action="store_true",
                    help="decode_full: skip the Reindex 1M, 20-layer schedule and prefill "
                         "workloads that the default run reports under `workloads`")
    ap.add_argument("--d-idx", type=int, default=128, choices=[64, 128],
                    help="indexer key width of the decode_full workload (64: the 890 B/token layout)")
    ap.add_argument("--workload", default="decode_full",
                    choices=["decode_full", "reindex", "prefill", "encoder", "schedule"],
                    help="decode_full (default): 32 x 64K Full-mode decode step; reindex: Reindex "
                         "layer at 1M; prefill: m = 2 encoder chunk, one Full + five Reuse layers; "
                         "encoder: the same chunk through the encoder's 18 CSA2 layers (three "
                         "caches); schedule: 20-layer decoder")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.workload == "decode_full":
        res = run_csa2(args, rank, world)
        if not args.quick and not args.no_extra:
            res["workloads"] = extra_workloads(args, world)
    else:
        import sparse_attention_decode_step_gb300 as csa
        dev = torch.device("cuda", torch.cuda.current_device())
        run = {"reindex": run_reindex, "prefill": run_prefill, "encoder": run_encoder,
               "schedule": run_schedule}
        res = run[args.workload](csa, args, world, dev)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
