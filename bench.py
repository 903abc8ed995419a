"""Benchmark of the GB300 Gated DeltaNet layer core.

One step = one pass of the layer core over one batch: the causal conv +
SiLU, the q/k norm and gates, and the gated delta rule, run as the fused
decode launch (gdn_decode; the same step as two launches, gdn_conv then
gdn_seq, is timed beside it). The headline workload is the decode batch: 64
requests x 1 token, 16 q/k heads, 32 value heads, Dk = Dv = 128 (8192 conv
channels), bf16 rows, fp32 state.

Metric: GDN tokens/s per layer, plus the state-traffic HBM GB/s of the rule
kernel against the measured HBM peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--no-extra]

Under torchrun each rank runs its own replica on its own GPU (requests are
independent: weak scaling, no data-path collective); the ranks meet only in a
barrier around the timed region and a max-reduction of the elapsed time.
``--impl reference`` times the CPU oracle on the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "GDN tokens/s per layer and state-traffic HBM GB/s vs GB300 peak (1 GPU)"
WORKLOAD = ("decode: 64 requests x 1 token, Hk=16 Hv=32 Dk=Dv=128 (C=8192), W=4, "
            "bf16 rows, fp32 state")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
EV_EVERY = 10  # launches per timed sample of the kernel's own duration
POOLS = 4  # rotating page pools: 4 x ~135 MB > the 129 MB L2


# ------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ measurement

# FP32 FMA peak from the unit counts: 152 SMs x 128 FP32 lanes x 2 flops per
# fused multiply-add x 2.07 GHz maximum SM clock (the packed f32x2 forms halve
# issue slots, not the lane count).
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi SM clock and throttle reasons, sampled every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self._stop = threading.Event()
        self._thread = None

    def _run(self):
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                     "--format=csv,noheader,nounits", "-lms", "100"],
                                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        try:
            while not self._stop.is_set():
                line = proc.stdout.readline()
                if not line:
                    break
                self.rows.append([s.strip() for s in line.split(",")])
        finally:
            proc.terminate()
            try:
                proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                proc.kill()

    def __enter__(self):
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thread.join(timeout=10)

    def summary(self):
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) < 9:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- our arm

class Decode:
    """The decode step on POOLS rotating copies of the 64-request batch."""

    def __init__(self, device, pools=POOLS, R=64):
        import torch

        import gated_deltanet_linear_14_gb300 as gdn
        from gated_deltanet_linear_14_gb300.pages import PagePool

        self.gdn, self.torch = gdn, torch
        d = synth.decode(R=R)
        self.d = d
        sh = d["shapes"]
        self.R, self.sh = R, sh
        self.dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 0, gdn.GDN_BF16, gdn.GDN_F32,
                                  gdn.GDN_BF16)

        def put(a, dtype=None):
            a = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype))
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)
            return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

        self.put = put
        self.A_log, self.dt_bias = put(d["A_log"]), put(d["dt_bias"])
        self.params = gdn.make_params(self.A_log, self.dt_bias)
        self.conv_w = put(d["conv_w"].store)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.pools = []
        S_page = torch.from_numpy(d["S0"]).transpose(-1, -2).contiguous().to(device)
        hist = put(d["hist0"].store)
        for _ in range(pools):
            pool = PagePool(self.dims, R, device=device)
            for r in range(R):
                pool.state(r).copy_(S_page[r])
                pool.window(r).copy_(hist[r])
            self.pools.append(pool)
        # the step's inputs x | a | b live in one device buffer (views), so the
        # end-to-end leg moves them with one host-to-device copy
        xs, as_, bs = (np.ascontiguousarray(d[k].store).view(np.int16) for k in ("x", "a", "b"))
        nx, na = xs.size, as_.size
        packed = np.concatenate([xs.ravel(), as_.ravel(), bs.ravel()])
        self.d_in = torch.from_numpy(packed).to(device).view(torch.bfloat16)
        self.x = self.d_in[:nx].view(R, sh.C)
        self.a = self.d_in[nx:nx + na].view(R, sh.Hv)
        self.b = self.d_in[nx + na:].view(R, sh.Hv)
        self.y = torch.empty(R, sh.C, dtype=torch.bfloat16, device=device)
        self.o = torch.empty(R, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
        ints = [put(np.asarray(v, np.int32)) for v in
                (d["row_start"], d["row_len"], np.arange(R), np.zeros(R))]
        self._ints = ints
        self.batch = gdn.make_batch(R, R, 1, R, *ints)
        # host-side buffers of the end-to-end leg (pinned): the packed inputs
        # and the output
        self.h_in = torch.empty_like(self.d_in, device="cpu").pin_memory()
        self.h_o = torch.empty_like(self.o, device="cpu").pin_memory()
        self.h_in.copy_(self.d_in.cpu())
        # the overlapped end-to-end leg: two device copies of the inputs and
        # outputs, so step i+1's upload and step i-1's download run while
        # step i's kernel runs
        self.d_in2 = [torch.empty_like(self.d_in) for _ in range(2)]
        self.o2 = [torch.empty_like(self.o) for _ in range(2)]
        self.h_o2 = [torch.empty_like(self.o, device="cpu").pin_memory() for _ in range(2)]
        self.s_in = torch.cuda.Stream(device=device)
        self.s_out = torch.cuda.Stream(device=device)

    # bytes the fused decode kernel must move per launch
    def decode_bytes(self):
        sh, R = self.sh, self.R
        state = 2 * R * sh.Hv * sh.Dk * sh.Dv * 4            # read + write fp32 state
        x = R * sh.C * 2                                     # raw rows (bf16)
        window = 2 * R * (sh.W - 1) * sh.C * 2               # conv window read + write
        taps = sh.C * sh.W * 2
        gates = 2 * R * sh.Hv * 2                            # a, b
        out = R * sh.Hv * sh.Dv * 2                          # o (bf16)
        return state + x + window + taps + gates + out, state

    def launch(self, i, ev=None):
        """One decode step: the fused conv + rule launch."""
        gdn = self.gdn
        pool = self.pools[i % len(self.pools)]
        if ev is not None:
            ev[0].record()
        gdn.gdn_decode(self.dims, self.batch, self.params, self.x, self.conv_w, self.a, self.b,
                       self.o, pool.buf, self.status)
        if ev is not None:
            ev[1].record()

    def launch_two(self, i, ev=None):
        """The same step as two launches: gdn_conv, then gdn_seq."""
        gdn = self.gdn
        pool = self.pools[i % len(self.pools)]
        if ev is not None:
            ev[0].record()
        gdn.gdn_conv(self.dims, self.batch, self.params, self.x, self.conv_w, self.y,
                     gdn.GDN_BF16, pool.buf, self.status)
        if ev is not None:
            ev[1].record()
        gdn.gdn_seq(self.dims, self.batch, self.params, self.y, self.a, self.b, self.o, pool.buf,
                    self.status)
        if ev is not None:
            ev[2].record()

    def launch_e2e(self, i):
        """The same step through host buffers: H2D of the step's inputs (x, a,
        b packed in one pinned buffer), the step, D2H of its output."""
        self.d_in.copy_(self.h_in, non_blocking=True)
        self.launch(i)
        self.h_o.copy_(self.o, non_blocking=True)

    def run_e2e_overlapped(self, K, i0=0):
        """K steps through host buffers with the copies overlapped: step i's
        inputs are uploaded (pinned host -> device buffer i%2) on one stream,
        its kernel runs on the current stream once they have landed (and once
        the download of step i-2 has left output buffer i%2), and its output
        is downloaded (device -> pinned host) on a third stream. Every step's
        copies are inside the returned time (CUDA events on the current
        stream, which waits for the last download)."""
        torch, gdn = self.torch, self.gdn
        cur = torch.cuda.current_stream()
        ev = {k: [torch.cuda.Event() for _ in range(2)]
              for k in ("in_ready", "in_free", "out_ready", "out_free")}
        for lst in ev.values():
            for e in lst:
                e.record(cur)
        sh, R = self.sh, self.R
        nx, na = R * sh.C, R * sh.Hv
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start.record(cur)
        for k in range(K):
            b = k % 2
            self.s_in.wait_event(ev["in_free"][b])
            with torch.cuda.stream(self.s_in):
                self.d_in2[b].copy_(self.h_in, non_blocking=True)
            ev["in_ready"][b].record(self.s_in)
            cur.wait_event(ev["in_ready"][b])
            cur.wait_event(ev["out_free"][b])
            d = self.d_in2[b]
            x, a, bb = d[:nx].view(R, sh.C), d[nx:nx + na].view(R, sh.Hv), d[nx + na:].view(R, sh.Hv)
            pool = self.pools[(i0 + k) % len(self.pools)]
            gdn.gdn_decode(self.dims, self.batch, self.params, x, self.conv_w, a, bb, self.o2[b],
                           pool.buf, self.status, stream=cur)
            ev["in_free"][b].record(cur)
            ev["out_ready"][b].record(cur)
            self.s_out.wait_event(ev["out_ready"][b])
            with torch.cuda.stream(self.s_out):
                self.h_o2[b].copy_(self.o2[b], non_blocking=True)
            ev["out_free"][b].record(self.s_out)
        cur.wait_stream(self.s_out)
        end.record(cur)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    def e2e_graph(self, steps=8):
        """The overlapped end-to-end pattern of `steps` consecutive steps
        (uploads on one stream, kernels on the capturing stream, downloads on
        a third, joined by events) captured once as a CUDA graph, so a replay
        issues all of their copies and kernels without per-step host work."""
        torch, gdn = self.torch, self.gdn
        sh, R = self.sh, self.R
        nx, na = R * sh.C, R * sh.Hv
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=self.d_in.device)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap):
            cur = torch.cuda.current_stream()
            ev = {k: [torch.cuda.Event() for _ in range(2)]
                  for k in ("in_ready", "in_free", "out_ready", "out_free")}
            for lst in ev.values():
                for e in lst:
                    e.record(cur)
            for k in range(steps):
                b = k % 2
                self.s_in.wait_event(ev["in_free"][b])
                with torch.cuda.stream(self.s_in):
                    self.d_in2[b].copy_(self.h_in, non_blocking=True)
                ev["in_ready"][b].record(self.s_in)
                cur.wait_event(ev["in_ready"][b])
                cur.wait_event(ev["out_free"][b])
                d = self.d_in2[b]
                x, a, bb = (d[:nx].view(R, sh.C), d[nx:nx + na].view(R, sh.Hv),
                            d[nx + na:].view(R, sh.Hv))
                pool = self.pools[k % len(self.pools)]
                gdn.gdn_decode(self.dims, self.batch, self.params, x, self.conv_w, a, bb,
                               self.o2[b], pool.buf, self.status, stream=cur)
                ev["in_free"][b].record(cur)
                ev["out_ready"][b].record(cur)
                self.s_out.wait_event(ev["out_ready"][b])
                with torch.cuda.stream(self.s_out):
                    self.h_o2[b].copy_(self.o2[b], non_blocking=True)
                ev["out_free"][b].record(self.s_out)
            cur.wait_stream(self.s_in)
            cur.wait_stream(self.s_out)
        torch.cuda.current_stream().wait_stream(cap)
        return g, steps

    def e2e_bytes(self):
        h2d = self.h_in.numel() * self.h_in.element_size()
        return h2d, self.h_o.numel() * self.h_o.element_size()

    def check(self):
        code = int(self.status.item())
        if code != 0:
            raise RuntimeError(f"device status {self.gdn.STATUS.get(code, code)}")


def time_steps(fn, K, torch):
    """K back-to-back calls of fn(i), CUDA events on the current stream."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for i in range(K):
        fn(i)
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def run_ours(args, world, rank, local):
    import torch
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    wl = Decode(device)
    K, W = args.steps, args.warmup
    for i in range(W):
        wl.launch(i)
    torch.cuda.synchronize()
    wl.check()

    # timed region: K steps; a CUDA event pair on the launching stream around
    # every EV_EVERY-th launch gives the kernel's duration (events between all
    # launches would add their own gaps to the steps they measure)
    sampled = list(range(0, K, EV_EVERY))
    evs = {i: [torch.cuda.Event(enable_timing=True) for _ in range(2)] for i in sampled}
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        elapsed = time_steps(lambda i: wl.launch(W + i, evs.get(i)), K, torch)
        wall = time.perf_counter() - t0
    torch.cuda.synchronize()
    barrier(world)
    wl.check()
    dec_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in sampled]
    elapsed_max = reduce_max(elapsed, world)

    # the same steps as two launches (conv, then the rule), for comparison
    K2 = min(K, 500)
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    el2 = time_steps(lambda i: wl.launch_two(W + K + i, ev2[i]), K2, torch)
    wl.check()
    conv_ms = [e[0].elapsed_time(e[1]) for e in ev2]
    rule_ms = [e[1].elapsed_time(e[2]) for e in ev2]

    # end-to-end through host buffers: the same steps with each step's upload
    # and download inside the timed region, overlapped with the neighbouring
    # steps' kernels; the serial form (upload, kernel, download on one
    # stream) is reported beside it
    for i in range(W):
        wl.launch_e2e(i)
    torch.cuda.synchronize()
    e2e_serial = time_steps(lambda i: wl.launch_e2e(i), K, torch)
    e2e_streams = wl.run_e2e_overlapped(K)
    # the same overlapped steps replayed from a CUDA graph of G steps (the
    # graph is built before the timed region; K rounds up to whole replays)
    graph, G = wl.e2e_graph(8)
    for _ in range(max(1, W // G)):
        graph.replay()
    torch.cuda.synchronize()
    reps = (K + G - 1) // G
    barrier(world)
    e2e = time_steps(lambda i: graph.replay(), reps, torch) * K / (reps * G)
    e2e_max = reduce_max(e2e, world)
    h2d, d2h = wl.e2e_bytes()
    # the overlapped leg's outputs equal the device-resident step's
    wl.check()

    tokens = wl.R * K * world
    dec_bytes, state_bytes = wl.decode_bytes()
    dec_s = statistics.mean(dec_ms) / 1e3
    hbm_peak = float(peaks["hbm_gbs"])
    # The timed region holds this kernel alone, one launch per step, so its
    # CUDA-event time over K is the kernel's mean launch duration; the
    # sampled event pairs (which add their own processing and stop the next
    # launch from starting early) are reported beside it.
    launch_s = elapsed_max / K
    achieved = dec_bytes / launch_s / 1e9
    line = {
        "metric": METRIC,
        "value": tokens / elapsed_max,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": elapsed_max / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,1) rows, N(0,0.02) fp32 state, random-init layer)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}",
                   "l2": f"{POOLS} rotating page pools ({POOLS * wl.pools[0].buf.numel() / 2**20:.0f} "
                         "MiB) exceed the 129 MB L2"},
        "state_gbs": state_bytes / launch_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic_from_profile("decode_fused"),
                     "kernel": "decode_kernel (gdn_decode: conv + rule, one launch)",
                     "algorithmic_bytes_per_launch": dec_bytes,
                     "launch_ms": launch_s * 1e3, "peak_source": f"{peak_src} hbm_gbs (burst)",
                     "launch_ms_bracketed": dec_s * 1e3,
                     "achieved_bracketed": dec_bytes / dec_s / 1e9,
                     "frac_bracketed": dec_bytes / dec_s / 1e9 / hbm_peak},
        "kernels_ms": {"gdn_decode": launch_s * 1e3,
                       "gdn_decode_event_bracketed": statistics.mean(dec_ms)},
        "two_launch_step": {"ms_per_step": el2 / K2 * 1e3, "gdn_conv_ms": statistics.mean(conv_ms),
                            "gdn_seq_ms": statistics.mean(rule_ms),
                            "tokens_per_s": wl.R * K2 / el2},
        "e2e": {"value": tokens / e2e_max, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_max / K * 1e3,
                "copies": "per step: H2D of the packed inputs and D2H of the output, on "
                          "their own streams, overlapped with the neighbouring steps' kernels; "
                          "steps replayed from a CUDA graph of 8",
                "streams_ms_per_step": e2e_streams / K * 1e3,
                "serial_ms_per_step": e2e_serial / K * 1e3},
        "gpu_launches": K,
        "clocks": clk.summary(),
        "wall_s": wall,
    }
    if not args.no_extra:
        line["workloads"] = extra_workloads(device, peaks, args)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return line


def traffic_from_profile(name):
    """DRAM bytes per launch from a committed ncu summary, if one is current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    v = data.get(name)
    if v is None:
        return None
    import hashlib
    blob = b"".join(open(os.path.join(ROOT, f), "rb").read() for f in v.get("sources", []))
    if hashlib.sha256(blob).hexdigest()[:16] != v.get("source_hash"):
        return None  # the kernel changed since the counters were taken
    return v.get("dram_bytes_per_launch")


def extra_workloads(device, peaks, args, only=None):
    """The other workloads of the layer core, each timed the same way."""
    out = {}
    for name, fn in (("spec_verify_fp32_state", lambda: bench_spec(device, peaks, "f32")),
                     ("spec_verify_bf16_state", lambda: bench_spec(device, peaks, "bf16")),
                     ("spec_slots_fp32_state", lambda: bench_slots(device, peaks)),
                     ("mixed_prefill_spec", lambda: bench_mixed(device, peaks)),
                     ("long_prefill_token_by_token", lambda: bench_long_seq(device, peaks)),
                     ("long_prefill_chunked", lambda: bench_long_chunk(device, peaks)),
                     ("chunked_small", lambda: bench_long_chunk(device, peaks, K=3, W=3,
                                                                small=True)),
                     ("decode_fused", lambda: bench_decode_only(device, peaks)),
                     ("crossover", lambda: bench_crossover(device, peaks)),
                     ("conv_long_rows", lambda: bench_conv_long(device, peaks))):
        if only is not None and name != only:
            continue
        if only is None and name in ("chunked_small", "decode_fused", "crossover"):
            continue
        try:
            out[name] = fn()
        except Exception as e:  # report, do not hide the headline line
            out[name] = {"error": repr(e)}
    return out


def _dev_batch(gdn, torch, device, start, ln, page, flags, acc=None, order=None, num_rows=None,
               max_rows=None, num_pages=None):
    def put(v):
        return torch.from_numpy(np.ascontiguousarray(np.asarray(v, np.int64).astype(np.uint32)
                                                     .view(np.int32))).to(device)
    arrs = [put(start), put(ln), put(page), put(flags)]
    acc_t = None if acc is None else put(acc)
    ord_t = None if order is None else put(order)
    R = len(start)
    num_rows = int(np.max(np.asarray(start) + np.asarray(ln))) if num_rows is None else num_rows
    max_rows = int(np.max(ln)) if max_rows is None else max_rows
    B = gdn.make_batch(R, num_rows, max_rows, R if num_pages is None else num_pages, *arrs,
                       acc_t, ord_t)
    B._keep = arrs + [acc_t, ord_t]
    return B


def _put_io(torch, device, t):
    a = np.ascontiguousarray(t.store)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def bench_spec(device, peaks, state, K=40, W=8, pools=POOLS):
    """Spec verify: 64 pages, 1+7 candidates, conv + one-page verify per step."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import PagePool
    d = synth.spec(steps=2)
    sh, R, n = d["shapes"], d["R"], d["n"]
    st = gdn.GDN_F32 if state == "f32" else gdn.GDN_BF16
    dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 8, gdn.GDN_BF16, st, gdn.GDN_BF16)
    A_log = torch.from_numpy(d["A_log"]).to(device)
    dt = torch.from_numpy(d["dt_bias"]).to(device)
    params = gdn.make_params(A_log, dt)
    conv_w = _put_io(torch, device, d["conv_w"])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    S_page = torch.from_numpy(d["S0"]).transpose(-1, -2).contiguous().to(device)
    hist = _put_io(torch, device, d["hist0"])
    pl = []
    for _ in range(pools):
        pool = PagePool(dims, R, device=device)
        for r in range(R):
            pool.state(r).copy_(S_page[r])
            pool.window(r)[:3].copy_(hist[r])
        pl.append(pool)
    rows = d["step_rows"][0]
    x, a, b = (_put_io(torch, device, rows[k]) for k in ("x", "a", "b"))
    T = R * n
    y = torch.empty(T, sh.C, dtype=torch.bfloat16, device=device)
    o = torch.empty(T, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
    rng = np.random.default_rng(2)
    accs = rng.integers(0, n, size=(8, R))
    batches = {}
    for par in (0, 1):
        flags = np.full(R, gdn.GDN_REQ_SPEC | (gdn.GDN_REQ_PARITY if par else 0))
        for k in range(8):
            # the row map's processing order puts the longest replays first
            # (the engine knows each request's accepted count), so the last
            # wave of CTAs holds the shortest
            batches[(par, k)] = _dev_batch(gdn, torch, device, d["row_start"], d["row_len"],
                                           np.arange(R), flags, acc=accs[k],
                                           order=np.argsort(-accs[k], kind="stable"))
    steps_done = [0] * pools

    def launch(i, ev=None):
        p = i % pools
        B = batches[(steps_done[p] % 2, i % 8)]
        steps_done[p] += 1
        if ev is not None:
            ev[0].record()
        gdn.gdn_conv(dims, B, params, x, conv_w, y, gdn.GDN_BF16, pl[p].buf, status)
        if ev is not None:
            ev[1].record()
        gdn.gdn_spec_verify(dims, B, params, y, a, b, o, pl[p].buf, status)
        if ev is not None:
            ev[2].record()

    def launch_fused(i, ev=None):
        p = i % pools
        B = batches[(steps_done[p] % 2, i % 8)]
        steps_done[p] += 1
        if ev is not None:
            ev[0].record()
        gdn.gdn_spec_step(dims, B, params, x, conv_w, a, b, o, pl[p].buf, status)
        if ev is not None:
            ev[1].record()

    for i in range(W):
        launch(i)
    torch.cuda.synchronize()
    evs = [_events(torch, 3) for _ in range(K)]
    el = time_steps(lambda i: launch(W + i, evs[i]), K, torch)
    # the same steps as one fused launch each (gdn_spec_step); the
    # pools' parities carry on from the two-launch steps
    for i in range(W):
        launch_fused(W + K + i)
    torch.cuda.synchronize()
    evf = [_events(torch, 2) for _ in range(K)]
    el_f = time_steps(lambda i: launch_fused(2 * W + K + i, evf[i]), K, torch)
    el_f_plain = time_steps(lambda i: launch_fused(2 * W + 2 * K + i), K, torch)
    code = int(status.item())
    ver_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    conv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fused_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evf)
    ssz = 4 if state == "f32" else 2
    state_bytes = 2 * R * sh.Hv * sh.Dk * sh.Dv * ssz
    mean_acc = float(np.mean(accs)) + 1.0
    rec_row = (sh.C + 2 * sh.Hv) * 2
    # verify: replayed record rows read, candidate rows and gates read, their
    # gates written to the record, outputs written
    other = int(R * mean_acc * rec_row + T * (sh.C + 2 * sh.Hv) * 2 + T * sh.Hv * sh.Dv * 2)
    # the fused step also reads the raw rows instead of conv'd ones (same
    # size), writes the conv'd rows into the record, and reads the W-1 history
    # columns and writes W-1+8 window columns
    fused_other = other + T * sh.C * 2 + R * (sh.W - 1 + sh.W - 1 + n) * sh.C * 2
    flops = R * sh.Hv * sh.Dk * sh.Dv * (mean_acc + n) * 7
    gbs = (state_bytes + other) / (ver_ms / 1e3) / 1e9
    f_gbs = (state_bytes + fused_other) / (el_f_plain / K) / 1e9
    return {"workload": f"spec verify: {R} pages, 1+7 candidates, {state} state, conv + verify",
            "ms_per_step": el / K * 1e3, "verify_ms": ver_ms, "conv_ms": conv_ms,
            "tokens_per_s": T * K / el, "verify_gbs": gbs,
            "verify_bytes": state_bytes + other,
            "verify_frac_of_hbm": gbs / float(peaks["hbm_gbs"]),
            "verify_tflops_fp32": flops / (ver_ms / 1e3) / 1e12,
            "verify_frac_of_fp32": flops / (ver_ms / 1e3) / 1e12 / FP32_PEAK_TFLOPS,
            "fp32_peak_tflops": FP32_PEAK_TFLOPS,
            "fused_step": {"entry": "gdn_spec_step (conv, coefficients and items in one launch)",
                           "ms_per_step": el_f_plain / K * 1e3,
                           "ms_per_step_event_bracketed": fused_ms,
                           "tokens_per_s": T * K / el_f_plain, "bytes": state_bytes + fused_other,
                           "gbs": f_gbs, "frac_of_hbm": f_gbs / float(peaks["hbm_gbs"])},
            "status": code}


def bench_slots(device, peaks, K=20, W=4, pools=2):
    """The slot-per-candidate layout on the spec workload, for contrast with
    the one-page verify: 64 requests, 1+7 candidates; each request resumes
    from slot a and stores the state (and conv window) after every candidate,
    so a step reads one state and writes eight."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import SlotPool
    d = synth.spec(steps=2)
    sh, R, n = d["shapes"], d["R"], d["n"]
    dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 8, gdn.GDN_BF16, gdn.GDN_F32,
                         gdn.GDN_BF16)
    A_log = torch.from_numpy(d["A_log"]).to(device)
    dt = torch.from_numpy(d["dt_bias"]).to(device)
    params = gdn.make_params(A_log, dt)
    conv_w = _put_io(torch, device, d["conv_w"])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    S_page = torch.from_numpy(d["S0"]).transpose(-1, -2).contiguous().to(device)
    hist = _put_io(torch, device, d["hist0"])
    pl = []
    for _ in range(pools):   # 2 x 1.2 GB of slots: far above the 129 MB L2
        pool = SlotPool(dims, R, device=device)
        for r in range(R):
            for i in range(n):
                pool.state(r, i).copy_(S_page[r])
                pool.window(r, i).copy_(hist[r])
        pl.append(pool)
    rows = d["step_rows"][0]
    x, a, b = (_put_io(torch, device, rows[k]) for k in ("x", "a", "b"))
    T = R * n
    y = torch.empty(T, sh.C, dtype=torch.bfloat16, device=device)
    o = torch.empty(T, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
    rng = np.random.default_rng(2)
    accs = rng.integers(0, n, size=(8, R))
    flags = np.full(R, gdn.GDN_REQ_SPEC)
    batches = [_dev_batch(gdn, torch, device, d["row_start"], d["row_len"], np.arange(R), flags,
                          acc=accs[k]) for k in range(8)]

    def launch(i):
        gdn.gdn_spec_slots(dims, batches[i % 8], params, x, conv_w, y, a, b, o, pl[i % pools].buf,
                           status)

    for i in range(W):
        launch(i)
    torch.cuda.synchronize()
    el = time_steps(lambda i: launch(W + i), K, torch)
    code = int(status.item())
    state_bytes = (1 + n) * R * sh.Hv * sh.Dk * sh.Dv * 4
    gbs = state_bytes / (el / K) / 1e9
    return {"workload": f"slot layout: {R} requests, 1+7 candidates, fp32 state, conv + rule "
                        "(a state per candidate)",
            "ms_per_step": el / K * 1e3, "tokens_per_s": T * K / el,
            "state_bytes_per_step": state_bytes, "state_gbs": gbs,
            "state_frac_of_hbm": gbs / float(peaks["hbm_gbs"]), "status": code}


def bench_mixed(device, peaks, K=20, W=4):
    """Mixed step: 8 fresh prefills (45..400 tokens) + 32 spec requests."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import PagePool
    d = synth.mixed()
    sh, R, n, ns = d["shapes"], d["R"], d["n"], d["n_spec"]
    dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 8, gdn.GDN_BF16, gdn.GDN_F32,
                         gdn.GDN_BF16)
    A_log = torch.from_numpy(d["A_log"]).to(device)
    dt = torch.from_numpy(d["dt_bias"]).to(device)
    params = gdn.make_params(A_log, dt)
    conv_w = _put_io(torch, device, d["conv_w"])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    pool = PagePool(dims, R, device=device)
    S_page = torch.from_numpy(d["S0"]).transpose(-1, -2).contiguous().to(device)
    for r in range(R):
        pool.state(r).copy_(S_page[r])
    x, a, b = (_put_io(torch, device, d[k]) for k in ("x", "a", "b"))
    T = d["T"]
    y = torch.empty(T, sh.C, dtype=torch.bfloat16, device=device)
    o = torch.empty(T, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
    lengths = d["row_len"]
    order = np.argsort(-lengths, kind="stable")
    acc = np.where(d["is_spec"], np.concatenate([d["prev_accepted"],
                                                 np.zeros(R - ns, np.int32)]), 0)
    batches = []
    for par in (0, 1):
        flags = np.where(d["is_spec"], gdn.GDN_REQ_SPEC | (gdn.GDN_REQ_PARITY if par else 0),
                         gdn.GDN_REQ_FRESH)
        batches.append(_dev_batch(gdn, torch, device, d["row_start"], lengths, np.arange(R), flags,
                                  acc=acc, order=order))

    def launch(i, ev=None):
        B = batches[i % 2]
        if ev is not None:
            ev[0].record()
        gdn.gdn_conv(dims, B, params, x, conv_w, y, gdn.GDN_BF16, pool.buf, status)
        if ev is not None:
            ev[1].record()
        # prefill rows: chunked form from GDN_PREFILL_CHUNK_MIN_ROWS rows, token
        # by token below (spec requests are skipped by both)
        # (no workspace: with prefills of 77..389 rows the one-launch chunked
        # form is faster than the two passes, 0.133 against 0.149 ms)
        gdn.gdn_prefill(dims, B, params, y, a, b, o, pool.buf, status)
        if ev is not None:
            ev[2].record()
        gdn.gdn_spec_verify(dims, B, params, y, a, b, o, pool.buf, status)
        if ev is not None:
            ev[3].record()

    # The same step with the verify on a second stream: after the conv, the
    # prefill and the verify touch disjoint pages and output rows, so the
    # verify's blocks can fill the SMs the chunked prefill leaves idle.
    main = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device=device)
    conv_done = torch.cuda.Event()
    ver_done = torch.cuda.Event()

    def launch_two_streams(i):
        B = batches[i % 2]
        gdn.gdn_conv(dims, B, params, x, conv_w, y, gdn.GDN_BF16, pool.buf, status, stream=main)
        conv_done.record(main)
        side.wait_event(conv_done)
        gdn.gdn_spec_verify(dims, B, params, y, a, b, o, pool.buf, status, stream=side)
        ver_done.record(side)
        gdn.gdn_prefill(dims, B, params, y, a, b, o, pool.buf, status, stream=main)
        main.wait_event(ver_done)

    for i in range(W):
        launch(i)
    torch.cuda.synchronize()
    evs = [_events(torch, 4) for _ in range(K)]
    el = time_steps(lambda i: launch(W + i, evs[i]), K, torch)
    for i in range(W):
        launch_two_streams(W + K + i)
    torch.cuda.synchronize()
    el2 = time_steps(lambda i: launch_two_streams(2 * W + K + i), K, torch)
    conv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    prefill_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    verify_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    step_ms = el / K * 1e3
    # Algorithmic bytes of the step, per kernel (bf16 rows and outputs, fp32
    # state): the conv reads x and writes y and the windows (fresh prefills
    # write W-1 columns, spec requests read W-1 and write W-1+n) and the spec
    # candidates' record rows; the prefill reads its rows and gates, writes
    # its outputs and final states (fresh: nothing read); the verify reads and
    # writes the spec pages' states, reads the candidate rows and the replayed
    # record rows (the mean accepted count + 1), writes outputs, gates and
    # run coefficients into the record.
    C, Hv, D = sh.C, sh.Hv, sh.Dv
    np_rows = int(lengths[ns:].sum())
    ns_rows = int(lengths[:ns].sum())
    rec_row = (C + 2 * Hv) * 2
    coef_bytes = Hv * 144 * 4
    mean_rep = float(np.mean(d["prev_accepted"])) + 1.0
    conv_b = (2 * T * C * 2 + (R - ns) * (sh.W - 1) * C * 2
              + ns * ((sh.W - 1) + (sh.W - 1 + n)) * C * 2 + ns_rows * rec_row)
    state = Hv * sh.Dk * D * 4
    pre_b = np_rows * (C + 2 * Hv) * 2 + np_rows * Hv * D * 2 + (R - ns) * state
    ver_b = (2 * ns * state + ns_rows * (C + 2 * Hv) * 2 + ns * mean_rep * rec_row
             + ns_rows * Hv * D * 2 + ns * (n * 2 * Hv * 2 + 2 * coef_bytes))
    step_b = conv_b + pre_b + ver_b
    # flops: about 7 Hv Dk Dv per row for the rule (3.7 MFLOP at these
    # shapes), replayed rows included for the verify
    fpr = 7 * Hv * sh.Dk * D
    step_f = fpr * (T + ns * mean_rep)
    hbm = float(peaks["hbm_gbs"])

    def frac(b, ms):
        return b / (ms / 1e3) / 1e9 / hbm

    def ffrac(f, ms):
        return f / (ms / 1e3) / 1e12 / FP32_PEAK_TFLOPS
    return {"workload": f"mixed: 8 prefills of {int(lengths[ns:].min())}..{int(lengths[ns:].max())} "
                        f"tokens + {ns} spec requests x {n} rows, {T} rows, row map longest first",
            "ms_per_step": step_ms, "tokens_per_s": T * K / el,
            "conv_ms": conv_ms, "prefill_ms": prefill_ms, "verify_ms": verify_ms,
            "ms_per_step_two_streams": el2 / K * 1e3, "tokens_per_s_two_streams": T * K / el2,
            "longest_chain": int(lengths.max()),
            "longest_chain_prefill_ms": prefill_ms,
            "bytes_per_step": step_b, "flops_per_step": step_f,
            "hbm_frac": frac(step_b, step_ms), "fp32_frac": ffrac(step_f, step_ms),
            "hbm_frac_two_streams": frac(step_b, el2 / K * 1e3),
            "fp32_frac_two_streams": ffrac(step_f, el2 / K * 1e3),
            "kernels": {
                "conv": {"bytes": conv_b, "hbm_frac": frac(conv_b, conv_ms)},
                "prefill": {"bytes": pre_b, "flops": fpr * np_rows,
                            "hbm_frac": frac(pre_b, prefill_ms),
                            "fp32_frac": ffrac(fpr * np_rows, prefill_ms)},
                "verify": {"bytes": ver_b, "flops": fpr * (ns_rows + ns * mean_rep),
                           "hbm_frac": frac(ver_b, verify_ms),
                           "fp32_frac": ffrac(fpr * (ns_rows + ns * mean_rep), verify_ms)}},
            "fp32_peak_tflops": FP32_PEAK_TFLOPS, "status": int(status.item())}


def bench_long_seq(device, peaks, K=3, W=3):
    """4 x 8192-token prefill through the token-by-token rule (conv + seq)."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import PagePool
    d = synth.long()
    sh, R, T = d["shapes"], d["R"], d["T"]
    dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 0, gdn.GDN_BF16, gdn.GDN_F32,
                         gdn.GDN_BF16)
    A_log = torch.from_numpy(d["A_log"]).to(device)
    dt = torch.from_numpy(d["dt_bias"]).to(device)
    params = gdn.make_params(A_log, dt)
    conv_w = _put_io(torch, device, d["conv_w"])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    pool = PagePool(dims, R, device=device)
    x, a, b = (_put_io(torch, device, d[k]) for k in ("x", "a", "b"))
    y = torch.empty(T, sh.C, dtype=torch.bfloat16, device=device)
    o = torch.empty(T, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
    B = _dev_batch(gdn, torch, device, d["row_start"], d["row_len"], np.arange(R),
                   np.full(R, gdn.GDN_REQ_FRESH))

    def launch(i, ev=None):
        if ev is not None:
            ev[0].record()
        gdn.gdn_conv(dims, B, params, x, conv_w, y, gdn.GDN_BF16, pool.buf, status)
        if ev is not None:
            ev[1].record()
        gdn.gdn_seq(dims, B, params, y, a, b, o, pool.buf, status)
        if ev is not None:
            ev[2].record()

    for i in range(W):
        launch(i)
    torch.cuda.synchronize()
    evs = [_events(torch, 3) for _ in range(K)]
    el = time_steps(lambda i: launch(W + i, evs[i]), K, torch)
    seq_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    return {"workload": "long prefill: 4 x 8192 tokens through conv + token-by-token rule",
            "ms_per_step": el / K * 1e3, "tokens_per_s": T * K / el, "seq_ms": seq_ms,
            "seq_us_per_token_chain": seq_ms * 1e3 / int(d["row_len"][0]),
            "status": int(status.item())}


# Algorithmic flops of one full 64-token chunk of one head (Dk = Dv = 128):
# [Q;K]K^T 2*128*64*128, W and U 2*(2*128*64*64), WS and QS 2*(2*128*64*128),
# P Vn 2*128*64*64, state update 2*128*128*64.
CHUNK_FLOPS = 2 * 128 * 64 * 128 + 2 * (2 * 128 * 64 * 64) + 2 * (2 * 128 * 64 * 128) \
    + 2 * 128 * 64 * 64 + 2 * 128 * 128 * 64


def bench_long_chunk(device, peaks, K=5, W=3, small=False):
    """4 x 8192-token prefill through the tensor-core chunked form (small:
    1 x 4096 tokens at 4/8 heads, the case the ncu capture uses)."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import PagePool
    d = synth.long(B=1, T=4096, sh=synth.Shapes(Hk=4, Hv=8, Dk=128, Dv=128)) if small \
        else synth.long()
    sh, R, T = d["shapes"], d["R"], d["T"]
    dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 0, gdn.GDN_BF16, gdn.GDN_F32,
                         gdn.GDN_BF16)
    A_log = torch.from_numpy(d["A_log"]).to(device)
    dt = torch.from_numpy(d["dt_bias"]).to(device)
    params = gdn.make_params(A_log, dt)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    pool = PagePool(dims, R, device=device)
    x, a, b = (_put_io(torch, device, d[k]) for k in ("x", "a", "b"))
    o = torch.empty(T, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
    B = _dev_batch(gdn, torch, device, d["row_start"], d["row_len"], np.arange(R),
                   np.full(R, gdn.GDN_REQ_FRESH))
    ws_bytes = gdn.gdn_chunk_prefill_workspace_bytes(dims, B)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)

    def launch(i):
        gdn.gdn_chunk_prefill(dims, B, params, x, a, b, o, pool.buf, ws, ws_bytes, status)

    for i in range(W):
        launch(i)
    torch.cuda.synchronize()
    el = time_steps(launch, K, torch)
    chunks = R * (T // R // 64)
    flops = chunks * sh.Hv * CHUNK_FLOPS
    tf = flops / (el / K) / 1e12
    size = "1 x 4096 tokens, 4/8 heads" if small else "4 x 8192 tokens"
    return {"workload": f"long prefill: {size}, chunk 64, tensor-core WY form, two passes "
                        "(pre-pass + state chain; rule only; rows are conv'd bf16 N(0,1))",
            "workspace_bytes": int(ws_bytes),
            "ms_per_launch": el / K * 1e3, "tokens_per_s": T * K / el,
            "algorithmic_tflops": tf, "tensor_peak_tflops": float(peaks["bf16_tflops"]),
            "frac_of_tensor_peak": tf / float(peaks["bf16_tflops"]),
            "issued_mma_flops_per_chunk_head": 24117248,
            "status": int(status.item())}


def bench_crossover(device, peaks, K=5, W=2):
    """gdn_seq vs gdn_chunk_prefill on R fresh requests of T tokens each
    (16/32 heads, Dk = Dv = 128): where the chunked form starts to win."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import PagePool
    sh = synth.FULL
    out = {}
    for R in (1, 8):
        rows_t = []
        for T in (8, 16, 32, 48, 64, 96, 128, 256, 512, 1024):
            d = synth.long(B=R, T=T)
            dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 0, gdn.GDN_BF16, gdn.GDN_F32,
                                 gdn.GDN_BF16)
            A_log = torch.from_numpy(d["A_log"]).to(device)
            dt = torch.from_numpy(d["dt_bias"]).to(device)
            params = gdn.make_params(A_log, dt)
            status = torch.zeros(1, dtype=torch.int32, device=device)
            pool = PagePool(dims, R, device=device)
            x, a, b = (_put_io(torch, device, d[k]) for k in ("x", "a", "b"))
            o = torch.empty(R * T, sh.Hv, sh.Dv, dtype=torch.bfloat16, device=device)
            B = _dev_batch(gdn, torch, device, d["row_start"], d["row_len"], np.arange(R),
                           np.full(R, gdn.GDN_REQ_FRESH))
            seq = lambda i: gdn.gdn_seq(dims, B, params, x, a, b, o, pool.buf, status)
            chk = lambda i: gdn.gdn_chunk_prefill(dims, B, params, x, a, b, o, pool.buf, None, 0,
                                                  status)
            res = {}
            for name, fn in (("seq_us", seq), ("chunk_us", chk)):
                for i in range(W):
                    fn(i)
                torch.cuda.synchronize()
                res[name] = time_steps(fn, K, torch) / K * 1e6
            res["T"] = T
            rows_t.append(res)
        wins = [r["T"] for r in rows_t if r["chunk_us"] < r["seq_us"]]
        out[f"R={R}"] = {"rows": rows_t, "chunk_wins_from_T": min(wins) if wins else None}
    return out


def bench_decode_only(device, peaks, K=20, W=5):
    """The fused decode step alone (what the ncu capture of decode_kernel runs)."""
    import torch
    wl = Decode(device)
    for i in range(W):
        wl.launch(i)
    torch.cuda.synchronize()
    el = time_steps(lambda i: wl.launch(W + i), K, torch)
    wl.check()
    return {"workload": WORKLOAD, "ms_per_step": el / K * 1e3}


def bench_conv_long(device, peaks, K=10, W=3):
    """The conv alone over 32768 rows x 8192 channels (1 GiB of row traffic)."""
    import torch
    import gated_deltanet_linear_14_gb300 as gdn
    from gated_deltanet_linear_14_gb300.pages import PagePool
    d = synth.long()
    sh, R, T = d["shapes"], d["R"], d["T"]
    dims = gdn.make_dims(sh.Hk, sh.Hv, sh.Dk, sh.Dv, sh.W, 0, gdn.GDN_BF16, gdn.GDN_F32,
                         gdn.GDN_BF16)
    params = gdn.make_params(None, None)
    conv_w = _put_io(torch, device, d["conv_w"])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    pool = PagePool(dims, R, device=device)
    x = _put_io(torch, device, d["x"])
    y = torch.empty(T, sh.C, dtype=torch.bfloat16, device=device)
    B = _dev_batch(gdn, torch, device, d["row_start"], d["row_len"], np.arange(R),
                   np.zeros(R))
    for i in range(W):
        gdn.gdn_conv(dims, B, params, x, conv_w, y, gdn.GDN_BF16, pool.buf, status)
    el = time_steps(lambda i: gdn.gdn_conv(dims, B, params, x, conv_w, y, gdn.GDN_BF16, pool.buf,
                                           status), K, torch)
    byts = 2 * T * sh.C * 2
    gbs = byts / (el / K) / 1e9
    return {"workload": "conv: 4 x 8192 rows x 8192 channels, bf16 in/out",
            "ms_per_launch": el / K * 1e3, "gbs": gbs, "frac_of_hbm": gbs / float(peaks["hbm_gbs"]),
            "status": int(status.item())}


# ------------------------------------------------------- CPU oracle (reference)

def oracle_decode_step(d, threads):
    import oracle
    sh = d["shapes"]
    y, _ = oracle.conv_f64(d["x"].value, d["hist0"].value, d["conv_w"].value, d["row_start"],
                           d["row_len"])
    o, S = oracle.gdn_f64(y, d["a"].value, d["b"].value, d["A_log"], d["dt_bias"],
                          d["row_start"], d["row_len"], sh.Hk, sh.Hv, sh.Dk, sh.Dv, S0=d["S0"],
                          threads=threads)
    return o


def cpu_baseline(seconds=10.0, steps=None):
    """The oracle, as it stands, on the decode batch: whole steps repeated
    until about `seconds` of CPU time (or `steps` steps)."""
    import oracle
    d = synth.decode()
    threads = oracle.default_threads()
    oracle_decode_step(d, threads)  # load / warm
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_decode_step(d, threads)
        n += 1
        el = time.perf_counter() - t0
        if (steps is not None and n >= steps) or (steps is None and el >= seconds):
            break
    # the same oracle on one host thread, for the per-core figure
    n1, t1 = 0, time.perf_counter()
    while True:
        oracle_decode_step(d, 1)
        n1 += 1
        el1 = time.perf_counter() - t1
        if n1 >= (1 if steps is not None else 3) and el1 >= min(seconds, 3.0) or n1 >= 50:
            break
    return {"value": d["R"] * n / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full decode steps (64 requests x 1 token, fp64 conv + rule) in "
                      f"{el:.1f} s", "steps": n,
            "single_thread": {"value": d["R"] * n1 / el1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{n1} full decode steps on one host thread in "
                                        f"{el1:.1f} s"}}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    K, W = args.steps, args.warmup
    import oracle
    d = synth.decode()
    threads = oracle.default_threads()
    for _ in range(W):
        oracle_decode_step(d, threads)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle_decode_step(d, threads)
    el = time.perf_counter() - t0
    v = d["R"] * K / el
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": "cpu oracle, rank 0 only"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{K} full decode steps, fp64 oracle on the host cores"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    help="run one secondary workload alone (spec_verify_fp32_state, "
                         "spec_verify_bf16_state, spec_slots_fp32_state, mixed_prefill_spec, "
                         "long_prefill_token_by_token, conv_long_rows)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.only:
        import torch
        torch.cuda.set_device(local)
        res = extra_workloads(torch.device(f"cuda:{local}"), load_peaks()[0], args, args.only)
        print(json.dumps(res), flush=True)
        return 0
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return 0
        line = run_reference(args, world, rank)
        print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    line = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
