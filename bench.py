#!/usr/bin/env python
"""Benchmark of the 2-bit rotated KV-cache hot path on one GPU (replicas on N GPUs).

A step = for every layer of the workload: quantize-append of the step's new tokens
(rotation, routing, eviction into INT2), then fused split-K decode attention of one new
query token per request (q rotation, INT2 + BF16 sink/recent attention, merge, output
rotation).  The host part of a step (page reservation, append and split-K plans) is
inside the timed region too.  Default workload: the Qwen3-8B-shaped layer stack
(B1, 32 query / 8 KV heads, 32768 context, 36 layers, 16 appended + 1 decoded token per
layer-step).  Inputs are seeded synthetic tensors (no datasets or weights).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the host cores
instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT2 decode-attn µs/layer/step & achieved HBM GB/s vs ~8 TB/s peak"


FILL_CHUNK = 16384  # context tokens appended per request and call while filling


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all",
                    help="one workload, or 'all': the headline workload (the 32B-shaped capacity run) and "
                         "every other workload under per_workload")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=2026)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling runs only)")
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16 comparison")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-serving", action="store_true", help="skip the throughput-mode serving comparison")
    ap.add_argument("--format", default="int2", choices=["int2", "int2_cm"],
                    help="INT2 page format: token-major (int2) or channel-major value pages (int2_cm)")
    ap.add_argument("--folded", action="store_true",
                    help="plan with OSCAR_PLAN_FOLDED_ROTATIONS (q arrives rotated, the output stays rotated)")
    ap.add_argument("--no-folded", action="store_true",
                    help="skip the 8B-shaped step's second run with OSCAR_PLAN_FOLDED_ROTATIONS")
    ap.add_argument("--no-cm", action="store_true",
                    help="skip the headline workload's second run in the channel-major format (tcgen05 decode)")
    ap.add_argument("--rotation", default="oscar", choices=["oscar", "hadamard"],
                    help="calibrated rotations: OSCAR's (default) or the Hadamard-only ablation")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------- distributed
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (the slowest replica sets the time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------- clocks
class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock-event reasons);
    nothing here changes a setting of the GPU."""

    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, cuda_index: int):
        import ctypes

        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        bus = self._pci_bus_id(cuda_index)
        if bus is None or self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.dev)) != 0:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.dev)) != 0:
                raise OSError("no NVML handle")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @staticmethod
    def _pci_bus_id(cuda_index: int):
        try:
            import torch

            p = torch.cuda.get_device_properties(cuda_index)
            return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except (AttributeError, RuntimeError, AssertionError):
            return None

    def sample(self):
        c = self.c
        mhz, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.dev, self.SM, c.byref(mhz))
        self.lib.nvmlDeviceGetMaxClockInfo(self.dev, self.SM, c.byref(mx))
        self.reasons_fn(self.dev, c.byref(rs))
        return mhz.value, mx.value, [n for b, n in self.REASONS.items() if rs.value & b]

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs: NVML every
    2 ms when the library loads, else nvidia-smi every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.nvml = None
        self.thread = None
        self.rows = []
        self.stop_evt = threading.Event()
        try:
            self.nvml = _Nvml(gpu_index)
            self.nvml.sample()
        except (OSError, AttributeError):
            self.nvml = None

    def _poll(self):
        while not self.stop_evt.is_set():
            self.rows.append(self.nvml.sample())
            time.sleep(0.002)

    def start(self):
        if self.nvml is not None:
            self.rows = [self.nvml.sample()]
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self.stop_evt.set()
            self.thread.join()
            self.rows.append(self.nvml.sample())
            self.nvml.close()
            sm = [r[0] for r in self.rows]
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in self.rows),
                    "reasons": sorted({n for r in self.rows for n in r[2]}), "samples": len(self.rows),
                    "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi"}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------- workload model
class Plan:
    """Request lengths and the per-step append schedule of a workload."""

    def __init__(self, w, seed, n_layers, total_steps):
        from int2_rotated_kv_rotate_gb300 import workloads as wl

        self.w = w
        self.n_layers = n_layers
        self.lengths = wl.context_lengths(w, seed)
        self.B = len(self.lengths)
        self.steps = []
        cur = list(self.lengths)
        for s in range(total_steps):
            n_new = [w.append_per_step if w.append_per_step else 1] * self.B
            for r in wl.chunk_appenders(w, s):
                n_new[r] = w.chunk_tokens
            self.steps.append((list(cur), n_new))
            cur = [c + n for c, n in zip(cur, n_new)]
        self.final = cur

    def max_len(self):
        return max(self.final)


def percentile(xs, f):
    """Linear-interpolated quantile f in [0, 1] of a non-empty list."""
    v = sorted(xs)
    k = f * (len(v) - 1)
    lo = int(math.floor(k))
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (k - lo)


def int2_bytes_per_layer(w, L_list, H_list, shared=None):
    """Algorithmic bytes of one layer's decode: INT2 codes + scale/zero of positions
    [S, H), BF16 sinks and ring tokens, fp32 R_K and R_V, q and out.  With `shared` (tokens
    each request maps from its group owner's prefix pages), the shared INT2 rows count once,
    with the owner: the unique bytes."""
    ng = w.head_dim // w.group
    per_int2 = 2 * (w.head_dim // 4 + ng * 4)
    total = 0
    shared = shared or [0] * len(L_list)
    for L, H, sh in zip(L_list, H_list, shared):
        n_int2 = max(0, H - max(w.n_sink, sh))
        n_bf16 = min(L, w.n_sink) + max(0, L - H)
        total += w.n_kv_heads * (n_int2 * per_int2 + n_bf16 * 2 * w.head_dim * 2)
    total += 2 * w.n_kv_heads * w.head_dim * w.head_dim * 4
    total += 2 * len(L_list) * w.n_q_heads * w.head_dim * 2
    return total


def append_bytes_per_layer(w, L0, H0, L1, H1):
    """Algorithmic bytes of one layer's quantize-append: new K/V rows in, their bf16 sink or
    ring rows out (or INT2 rows when they go straight to the history), evicted ring rows in
    and their INT2 rows out, and R_V (R_K is already counted by the decode)."""
    ng = w.head_dim // w.group
    per_int2 = 2 * (w.head_dim // 4 + ng * 4)
    row2 = 2 * w.head_dim * 2  # K and V bf16 rows
    total = w.n_kv_heads * w.head_dim * w.head_dim * 4
    for l0, h0, l1, h1 in zip(L0, H0, L1, H1):
        new = l1 - l0
        direct = max(0, min(l1, h1) - max(l0, w.n_sink))  # new tokens that go straight to INT2
        evicted = max(0, min(l0, h1) - h0)
        total += w.n_kv_heads * (new * row2 + (new - direct) * row2 + direct * per_int2 + evicted * (row2 + per_int2))
    return total


def source_digest() -> str:
    """sha256 over the kernel sources: a profile's counters apply while this is unchanged."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int2_rotated_kv_rotate_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h", ".cpp")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per layer-step of the step's kernel(s) from the committed ncu summary of
    this workload, if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"step_kernels_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ": " in line:
                k, v = line[2:].strip().split(": ", 1)
                fields[k.strip("`")] = v.strip().strip("`")
    if fields.get("source_sha256") != source_digest():
        return None
    try:
        return int(fields["dram_bytes_per_step_kernels"])
    except (KeyError, ValueError):
        return None


def bf16_bytes_per_layer(w, L_list):
    return sum(w.n_kv_heads * L * 2 * w.head_dim * 2 for L in L_list) + 2 * len(L_list) * w.n_q_heads * w.head_dim * 2


# ---------------------------------------------------------------------------- our arm
def run_ours(args, w, world, rank, local):
    import torch

    from int2_rotated_kv_rotate_gb300 import KVCache, OSCAR_FORMAT_BF16, calibrate, workloads as wl
    from int2_rotated_kv_rotate_gb300 import _native as N

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    n_layers = args.layers or w.n_layers
    seed = args.seed + 1000 * rank  # each replica holds its own requests
    total_steps = args.warmup + args.steps
    E2E_STEPS = 10
    plan = Plan(w, seed, n_layers, total_steps + 2 + E2E_STEPS)  # sizes the page pool for every step
    B = plan.B
    ppr = (plan.max_len() + 63) // 64 + 2
    # page pool: private pages of every request (shared prefixes counted once per group)
    pages = sum((L + 63) // 64 + 1 for L in plan.final) + 8
    fmt = N.OSCAR_FORMAT_INT2_CM if args.format == "int2_cm" else N.OSCAR_FORMAT_INT2
    cache = KVCache(fmt=fmt, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, group=w.group, n_sink=w.n_sink,
                    window=w.window, n_layers=n_layers, max_requests=B, max_pages=pages, max_pages_per_request=ppr,
                    device=dev)
    t_cal = time.time()
    for layer in range(n_layers):
        qc, kc, vc = wl.gen_calibration(w, seed, layer, device=dev)
        RK, RV, cK, cV = calibrate.calibrate_layer_gpu(qc, kc, vc, w.clip_percentile, rotation=args.rotation)
        cache.set_layer_params(layer, RK, RV, cK, cV)
    t_cal = time.time() - t_cal
    slots = [cache.alloc() for _ in range(B)]

    # ---- fill the context (prefix owners first, then sharers map the shared pages)
    t_fill = time.time()
    shared = fill_context(cache, w, seed, n_layers, slots, plan.lengths, dev)
    torch.cuda.synchronize()
    t_fill = time.time() - t_fill

    # ---- per-step inputs (device) and fixed buffers the captured step reads
    Hkv, Hq, d = w.n_kv_heads, w.n_q_heads, w.head_dim
    steps_in = []
    n_inputs = total_steps + 1 + (0 if args.no_e2e else E2E_STEPS)  # timed, roofline, end-to-end steps
    for s in range(n_inputs):
        cur, n_new = plan.steps[s]
        rows = sum(n_new)
        K = torch.empty((n_layers, rows, Hkv, d), dtype=torch.bfloat16, device=dev)
        V = torch.empty_like(K)
        for layer in range(n_layers):
            ks, vs = [], []
            for r in range(B):
                k, v = wl.gen_kv(w, seed, layer, r, cur[r], n_new[r], device=dev)
                ks.append(k)
                vs.append(v)
            K[layer] = torch.cat(ks)
            V[layer] = torch.cat(vs)
        Q = torch.stack([wl.gen_q(w, seed, layer, s, B, device=dev) for layer in range(n_layers)])
        steps_in.append((K, V, Q, n_new))
    rows0 = sum(plan.steps[0][1])
    kin = torch.empty((n_layers, rows0, Hkv, d), dtype=torch.bfloat16, device=dev)
    vin = torch.empty_like(kin)
    qin = torch.empty((n_layers, B, Hq, d), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(qin)
    stream = torch.cuda.current_stream()

    plan_flags = N.OSCAR_PLAN_FOLDED_ROTATIONS if args.folded else 0

    def host_plan(s):
        cache.reserve(slots, steps_in[s][3])
        cache.plan(slots, flags=plan_flags)

    # per-layer views, made once (the calls below are the step's whole host work per layer)
    kin_l, vin_l = [kin[layer] for layer in range(n_layers)], [vin[layer] for layer in range(n_layers)]
    qin_l, out_l = [qin[layer] for layer in range(n_layers)], [out[layer] for layer in range(n_layers)]

    def device_step(strm=None, s=None):
        # per layer, one call: quantize-append of the step's tokens, then decode attention;
        # s: read step s's resident inputs in place (else the fixed input buffers)
        n = 0  # kernels the library put on the stream (its own count, per call)
        ks, vs, qs = (kin_l, vin_l, qin_l) if s is None else steps_in[s][:3]
        for layer in range(n_layers):
            cache.append_decode(layer, ks[layer], vs[layer], qs[layer], out=out_l[layer], stream=strm)
            n += N.oscar_last_launch_count()
        return n

    def load_inputs(s):
        K, V, Q, _ = steps_in[s]
        kin.copy_(K)
        vin.copy_(V)
        qin.copy_(Q)

    for s in range(args.warmup):  # eager warm-up steps
        host_plan(s)
        load_inputs(s)
        device_step()
        cache.commit()
    torch.cuda.synchronize()
    st, flags = cache.status()
    assert st == 0, f"device status {flags:#x} after warm-up"

    # ---- capture each timed step's device work (append + decode of every layer) as a graph
    # that reads that step's inputs where they already are in HBM
    s0 = args.warmup
    host_plan(s0)
    graphs = {}
    for s in range(s0, s0 + args.steps):
        graphs[s] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[s]):
            launches_per_step = device_step(s=s)

    # ---- timed region: K steps (host plans + graph replay + commit)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e0.record()
    for i, s in enumerate(range(s0, s0 + args.steps)):
        if s > s0:
            host_plan(s)
        graphs[s].replay()
        cache.commit()
        marks[i].record()
    e1.record()
    torch.cuda.synchronize()
    step_ms = e0.elapsed_time(e1) / args.steps
    # per-step times (between consecutive step ends; the first from the region's start)
    per_step = [e0.elapsed_time(marks[0])] + [marks[i - 1].elapsed_time(marks[i]) for i in range(1, args.steps)]
    step_pct = [percentile(per_step, f) for f in (0.1, 0.5, 0.9)]
    barrier(world)
    step_ms = max_over_ranks(step_ms, world, dev)
    clk = clocks.stop()
    st, flags = cache.status()
    assert st == 0, f"device status {flags:#x}"

    # ---- the step's kernel alone (the roofline's duration): one reservation, the n_layers
    # fused append + decode launches captured and replayed back to back (replays rewrite
    # the same rows), CUDA events on the capturing stream
    n_new_k = steps_in[total_steps][3]
    L_pre = [cache.info(sl)[0] for sl in slots]
    H_pre = [cache.info(sl)[1] for sl in slots]
    cache.reserve(slots, n_new_k)
    cache.plan(slots, flags=plan_flags)
    fgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(fgraph):
        device_step()
    for _ in range(3):
        fgraph.replay()
    torch.cuda.synchronize()
    reps = max(5, args.steps)
    e0.record()
    for _ in range(reps):
        fgraph.replay()
    e1.record()
    torch.cuda.synchronize()
    fused_us = e0.elapsed_time(e1) * 1000.0 / (reps * n_layers)
    cache.commit()
    L_now, H_now = zip(*[cache.info(sl)[:2] for sl in slots])
    app_bytes = append_bytes_per_layer(w, L_pre, H_pre, L_now, H_now)
    fused_bytes = int2_bytes_per_layer(w, L_now, H_now, shared) + app_bytes  # unique (shared prefixes once)
    reader_bytes = int2_bytes_per_layer(w, L_now, H_now) + app_bytes  # every request's reads
    st, flags = cache.status()
    assert st == 0, f"device status {flags:#x} after the fused timing"

    # ---- decode-only timing (n_layers back-to-back decode calls, captured)
    dgraph = torch.cuda.CUDAGraph()
    cache.plan(slots, flags=plan_flags)
    with torch.cuda.graph(dgraph):
        for layer in range(n_layers):
            cache.decode(layer, qin[layer], out=out[layer])
    for _ in range(3):
        dgraph.replay()
    torch.cuda.synchronize()
    reps = max(5, args.steps)
    e0.record()
    for _ in range(reps):
        dgraph.replay()
    e1.record()
    torch.cuda.synchronize()
    decode_us = e0.elapsed_time(e1) * 1000.0 / (reps * n_layers)
    bytes_layer = int2_bytes_per_layer(w, L_now, H_now)
    int2_pages = w.n_kv_heads * sum((H + 63) // 64 if H > w.n_sink else 0 for H in H_now)  # over all items
    n_items, n_bf16_items, max_item_pages = cache.plan_info()

    # ---- end to end through the C ABI with host buffers (no graph: one call per layer).
    # Every step copies its inputs in from pinned host memory and its output out; the
    # copies run on a second stream, double-buffered, so step i + 1's inputs arrive while
    # step i computes (both inside the timed region)
    e2e = None
    if not args.no_e2e:
        # the end-to-end steps continue the sequence after the roofline's step (their own
        # appends, as the plan sized the page pool for)
        e2e_first = total_steps + 1
        hK = {s: steps_in[s][0].cpu().pin_memory() for s in range(e2e_first, n_inputs)}
        hV = {s: steps_in[s][1].cpu().pin_memory() for s in range(e2e_first, n_inputs)}
        hQ = {s: steps_in[s][2].cpu().pin_memory() for s in range(e2e_first, n_inputs)}
        hout = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        bufs = [(kin, vin, qin, out), tuple(torch.empty_like(t) for t in (kin, vin, qin, out))]
        views = [tuple([t[layer] for layer in range(n_layers)] for t in bset) for bset in bufs]
        # roll the cache back is not possible; e2e continues the sequence on fresh steps
        n_e2e = min(args.steps, E2E_STEPS)
        comp = torch.cuda.current_stream()
        cs = torch.cuda.Stream()
        stream_handle = comp.cuda_stream
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready, in_free, out_ready, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]

        def upload(i, b):
            s = e2e_first + i
            with torch.cuda.stream(cs):
                if used[b]:
                    cs.wait_event(in_free[b])
                bufs[b][0].copy_(hK[s], non_blocking=True)
                bufs[b][1].copy_(hV[s], non_blocking=True)
                bufs[b][2].copy_(hQ[s], non_blocking=True)
                in_ready[b].record(cs)

        torch.cuda.synchronize()
        e0.record(comp)
        cs.wait_event(e0)
        upload(0, 0)
        for i in range(n_e2e):
            b = i % 2
            if i + 1 < n_e2e:
                upload(i + 1, 1 - b)
            cache.reserve(slots, steps_in[e2e_first + i][3])
            cache.plan(slots, flags=plan_flags)
            comp.wait_event(in_ready[b])
            if used[b]:
                comp.wait_event(out_free[b])
            ks, vs, qs, os_ = views[b]
            for layer in range(n_layers):  # the public calls themselves, launched eagerly
                cache.append_decode(layer, ks[layer], vs[layer], qs[layer], out=os_[layer], stream=stream_handle)
            in_free[b].record(comp)
            out_ready[b].record(comp)
            with torch.cuda.stream(cs):
                cs.wait_event(out_ready[b])
                hout[b].copy_(bufs[b][3], non_blocking=True)
                out_free[b].record(cs)
            used[b] = True
            cache.commit()
        comp.wait_stream(cs)
        e1.record(comp)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        h2d = (kin.numel() + vin.numel() + qin.numel()) * 2
        d2h = out.numel() * 2
        e2e = {"value": round(e2e_ms * 1000.0 / n_layers, 3), "unit": "us/layer/step",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
        st, flags = cache.status()
        assert st == 0, f"device status {flags:#x} after e2e"

    # ---- BF16 comparison (decode over the same lengths, uncompressed pages)
    bf16 = None
    if not args.no_bf16:
        bf16 = bf16_comparison(w, seed, n_layers, [cache.info(sl)[0] for sl in slots], qin, dev, reps)
    cache.close()
    return dict(step_ms=step_ms, clocks=clk, decode_us=decode_us, bytes_layer=bytes_layer, n_layers=n_layers, B=B,
                fused_us=fused_us, fused_bytes=fused_bytes, reader_bytes=reader_bytes, step_pct=step_pct,
                launches=launches_per_step * args.steps, e2e=e2e, bf16=bf16, n_items=n_items,
                max_item_pages=max_item_pages, int2_pages=int2_pages,
                n_bf16_items=n_bf16_items, t_cal=t_cal, t_fill=t_fill, world=world, w=w)


def fill_context(cache, w, seed, n_layers, slots, lengths, dev):
    """The workload's context: prefix owners are filled first, then each sharer maps its group
    owner's prefix pages and appends the rest of its own context.  Returns the shared token
    count of every request."""
    from int2_rotated_kv_rotate_gb300 import workloads as wl

    B = len(lengths)
    shared = [0] * B
    owners = [r for r in range(B) if r % w.prefix_group == 0] if w.prefix_tokens else list(range(B))
    fill(cache, w, seed, n_layers, [slots[r] for r in owners], owners, [0] * len(owners),
         [lengths[r] for r in owners], dev)
    if w.prefix_tokens:
        sharers = [r for r in range(B) if r % w.prefix_group != 0]
        for r in sharers:
            src = r - r % w.prefix_group
            n_sh = min(wl.shared_prefix_tokens(w, lengths[r]), (cache.info(slots[src])[1] // 64) * 64)
            if n_sh > 0:
                cache.share_prefix(slots[r], slots[src], n_sh)
                shared[r] = n_sh
        fill(cache, w, seed, n_layers, [slots[r] for r in sharers], sharers, [shared[r] for r in sharers],
             [lengths[r] - shared[r] for r in sharers], dev)
    return shared


def fill(cache, w, seed, n_layers, slots, reqs, starts, counts, dev, chunk=FILL_CHUNK):
    """Append the context of `reqs` in pieces of at most `chunk` tokens per request."""
    import torch

    from int2_rotated_kv_rotate_gb300 import workloads as wl

    done = [0] * len(reqs)
    while any(d < c for d, c in zip(done, counts)):
        n_new = [min(chunk, c - d) for d, c in zip(done, counts)]
        act = [i for i, n in enumerate(n_new) if n > 0]
        cache.reserve([slots[i] for i in act], [n_new[i] for i in act])
        for layer in range(n_layers):
            ks, vs = [], []
            for i in act:
                k, v = wl.gen_kv(w, seed, layer, reqs[i], starts[i] + done[i], n_new[i], device=dev)
                ks.append(k)
                vs.append(v)
            cache.append(layer, torch.cat(ks).contiguous(), torch.cat(vs).contiguous())
        cache.commit()
        for i in act:
            done[i] += n_new[i]


def bf16_comparison(w, seed, n_layers, lengths, qin, dev, reps):
    import torch

    from int2_rotated_kv_rotate_gb300 import KVCache, OSCAR_FORMAT_BF16

    B = len(lengths)
    free = torch.cuda.mem_get_info(dev)[0]
    per_req = sum(w.n_kv_heads * ((L + 63) // 64) * 64 * 512 for L in lengths[:1]) * n_layers
    fit = max(1, min(B, int(0.85 * free // max(per_req, 1))))
    use = lengths[:fit]
    ppr = max((L + 63) // 64 for L in use) + 1
    bc = KVCache(fmt=OSCAR_FORMAT_BF16, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, n_layers=n_layers,
                 max_requests=fit, max_pages=sum((L + 63) // 64 + 1 for L in use) + 4, max_pages_per_request=ppr,
                 device=dev)
    slots = [bc.alloc() for _ in use]
    fill(bc, w, seed, n_layers, slots, list(range(fit)), [0] * fit, use, dev)
    bc.plan(slots)
    q = qin[:, :fit].contiguous()
    o = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for layer in range(n_layers):
            bc.decode(layer, q[layer], out=o[layer])
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / (reps * n_layers)
    st, flags = bc.status()
    assert st == 0, f"bf16 device status {flags:#x}"
    nbytes = bf16_bytes_per_layer(w, use)
    bc.close()
    return {"us_per_layer": round(us, 3), "requests": fit, "bytes_per_layer": nbytes,
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}


# ---------------------------------------------------------------------------- CPU oracle
def oracle_sample(w, seed, heads, context: int):
    """One (layer 0, request 0) oracle stream pair per entry of `heads` (a kv-head index;
    entries may repeat, each gets its own streams) at `context` tokens (built untimed), and
    a function that times one step of entry i: append of the step's tokens and decode of
    one query."""
    import numpy as np

    import oracle
    from int2_rotated_kv_rotate_gb300 import workloads as wl
    from oracle import calibration as ocal
    from oracle.model import as_bits

    qc, kc, vc = wl.gen_calibration(w, seed, 0)
    G = w.gqa
    K, V = wl.gen_kv(w, seed, 0, 0, 0, context)
    kb, vb = as_bits(K), as_bits(V)
    q = as_bits(wl.gen_q(w, seed, 0, 0, 1))[0]
    n_app = w.append_per_step or 1
    newK, newV = wl.gen_kv(w, seed, 0, 0, context, n_app)
    nkb, nvb = as_bits(newK), as_bits(newV)
    params = {}
    streams = []
    for h in heads:
        if h not in params:
            params[h] = ocal.calibrate_head(qc[:, h * G:(h + 1) * G].float().numpy(), kc[:, h].float().numpy(),
                                            vc[:, h].float().numpy(), w.clip_percentile)
        RK, RV, cK, cV = params[h]
        cap = context + 4096
        sk = oracle.Stream(w.head_dim, w.group, w.n_sink, w.window, cap, RK, cK)
        sv = oracle.Stream(w.head_dim, w.group, w.n_sink, w.window, cap, RV, cV)
        sk.append(np.ascontiguousarray(kb[:, h]))
        sv.append(np.ascontiguousarray(vb[:, h]))
        streams.append((h, sk, sv, RK, RV))

    def one_head_step(i):
        h, sk, sv, RK, RV = streams[i]
        t = time.perf_counter()
        if sk.length + n_app <= sk.capacity:
            sk.append(np.ascontiguousarray(nkb[:, h]))
            sv.append(np.ascontiguousarray(nvb[:, h]))
        oracle.decode(np.ascontiguousarray(q[h * G:(h + 1) * G]), sk, sv, RK, RV)
        return time.perf_counter() - t

    return one_head_step


def host_cpu():
    """(logical cores, CPU model) of the host."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.startswith("Model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform

    return os.cpu_count() or 1, (model or "unknown") + f" ({platform.machine()})"


def cpu_baseline(w, seed, budget_s=12.0):
    """The oracle, as it stands, on the host cores, scaled from a bounded sample of one
    layer-step of the workload: its decode of one (request, kv-head) is serial C, so the
    single-thread row runs one head at a time on one thread, and the all-cores row runs one
    head per host core at once (threads: the oracle's C calls release the interpreter lock).
    Both rows: layer 0 of request 0 at up to 32768 tokens of context, append of the
    step's tokens + decode of one query per head, scaled to the workload's batch, kv-heads
    and context."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.set_threads(1)
    nproc, model = host_cpu()
    context = min(w.context, 32768)
    heads = [i % w.n_kv_heads for i in range(min(nproc, w.n_kv_heads * w.batch))]
    step = oracle_sample(w, seed, heads, context)  # one stream pair per thread of the all-cores row
    scale = w.n_kv_heads * w.batch * (w.context / context)  # head-steps of one layer-step
    # one thread
    times = []
    t_end = time.time() + budget_s / 2
    while time.time() < t_end and len(times) < 30:
        times.append(step(len(times) % len(heads)))
    per_head = statistics.median(times)
    one = per_head * scale * 1e6
    # all cores: one head per thread, nproc heads at once (heads beyond the workload's
    # kv-heads reuse their streams: the same work)
    rounds = []
    t_end = time.time() + budget_s / 2
    with ThreadPoolExecutor(max_workers=len(heads)) as ex:
        while time.time() < t_end and len(rounds) < 10:
            t = time.perf_counter()
            list(ex.map(step, range(len(heads))))
            rounds.append(time.perf_counter() - t)
    per_round = statistics.median(rounds)
    allc = per_round * (scale / len(heads)) * 1e6
    return {"value": round(one, 1), "unit": "us/layer/step", "cores": 1, "kind": "oracle", "nproc": nproc,
            "cpu_model": model,
            "sample": f"layer 0 of request 0, context {context}: append {w.append_per_step or 1} token(s) + decode "
                      f"1 query per kv-head; one thread: median of {len(times)} head-steps, scaled x{scale:.0f} "
                      f"(kv-heads x batch x context ratio) to one layer-step",
            "all_cores": {"value": round(allc, 1), "unit": "us/layer/step", "cores": len(heads),
                          "sample": f"{len(heads)} head-steps at once on {len(heads)} threads, median of "
                                    f"{len(rounds)} rounds, scaled x{scale / len(heads):.1f}"}}


# ---------------------------------------------------------------------------- output
def config_of(w, n_layers, rotation="oscar"):
    return {"workload": w.name, "description": w.description, "layers": n_layers, "batch": w.batch,
            "rotation": rotation,
            "context": w.context, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
            "group": w.group, "page": w.page, "sink": w.n_sink, "window": w.window,
            "l2": "inputs larger than L2: every layer's cache is distinct and the step cycles through all layers"
                  if n_layers > 1 or w.batch > 1 else
                  "one layer of one request (about 1 MB) fits in L2: the step is launch-bound and reported in us only"}


def serving_comparison(seed: int, dev, budget_gib: float = 2.0):
    """Throughput mode: the serving loop (continuous batching, prefix-cache hits) over the
    INT2 cache and over the BF16 cache, each sized to the same HBM budget, serving the same
    requests to completion.  Shape: the 8B-shaped layer (32q/8kv, g128) with 8 layers."""
    import torch

    from int2_rotated_kv_rotate_gb300 import OSCAR_FORMAT_BF16, OSCAR_FORMAT_INT2, calibrate, serving
    from int2_rotated_kv_rotate_gb300 import workloads as wl

    w = wl.scaled(wl.WORKLOADS["qwen3_8b_layer"], name="serving_8b_8layers", n_layers=8)
    budget = int(budget_gib * (1 << 30))
    spec = dict(n=48, prompt=(4096, 12288), gen=(64, 192), groups=12, prefix=2048)
    tokens = serving.TokenSource(w, seed, pool_tokens=16384, device=dev)
    params = [[], [], [], []]
    for layer in range(w.n_layers):
        qc, kc, vc = wl.gen_calibration(w, seed, layer, device=dev)
        for i, a in enumerate(calibrate.calibrate_layer_gpu(qc, kc, vc, w.clip_percentile)):
            params[i].append(a)
    out = {"shape": w.description.split(",")[0] + ", 8 layers", "hbm_budget_bytes": budget,
           "requests": spec["n"], "prompt_tokens": list(spec["prompt"]), "generated_tokens": list(spec["gen"]),
           "prefix": f"{spec['groups']} groups of {spec['n'] // spec['groups']} requests share a "
                     f"{spec['prefix']}-token prefix (prefix holder + shared pages)"}
    for name, fmt in (("int2", OSCAR_FORMAT_INT2), ("bf16", OSCAR_FORMAT_BF16)):
        reqs = serving.make_requests(spec["n"], spec["prompt"], spec["gen"], spec["groups"], seed)
        loop = serving.ServingLoop(w, fmt, budget, tokens, layer_params=params if fmt == OSCAR_FORMAT_INT2 else None,
                                   max_requests=spec["n"] + spec["groups"] + 1, max_len=spec["prompt"][1] + spec["gen"][1] + 64,
                                   prefix_tokens=spec["prefix"], device=dev)
        st = loop.run(reqs)
        status, flags = loop.cache.status()
        assert status == 0, f"serving {name}: device flags {flags:#x}"
        loop.close()
        out[name] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in st.items() if k != "batch_sum"}
        del loop
        torch.cuda.empty_cache()
    out["throughput_ratio_int2_over_bf16"] = round(out["int2"]["tokens_per_s"] / out["bf16"]["tokens_per_s"], 3)
    out["decode_throughput_ratio_int2_over_bf16"] = round(
        out["int2"]["decode_tokens_per_s"] / out["bf16"]["decode_tokens_per_s"], 3)
    return out


HEADLINE = "qwen3_32b_capacity"
OTHERS = ["tiny", "qwen3_8b_layer", "long_batch", "ragged_prefix"]


def result_line(args, w, r, world):
    """The JSON object of one workload's measurement."""
    n_layers = r["n_layers"]
    us_layer_step = r["step_ms"] * 1000.0 / n_layers
    peak, peak_kind = measured_peaks()
    achieved = r["fused_bytes"] / (r["fused_us"] * 1e-6) / 1e9
    line = {
        "metric": METRIC,
        "value": round(us_layer_step, 3),
        "unit": "us/layer/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["step_ms"], 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int2 codes + bf16 scale/zero; fp16 mma, fp32 softmax",
        "data": "synthetic (seeded N(0,1) bf16 K/V/q with channel outliers and log-normal token norms)",
        "config": config_of(w, n_layers, args.rotation),
        "decode_us_per_layer": round(r["decode_us"], 3),
        "append_decode_tokens_per_s": round(r["B"] * world / (r["step_ms"] * 1e-3), 1),
        "roofline": {"bound": "hbm",
                     "kernel": ("split_kernel (fused quantize-append + decode), one launch per layer"
                                if args.format == "int2" else
                                "append_kernel, then split_kernel with INT2 items on tcgen05 (tensor memory)"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     # the committed ncu summaries cover the token-major format's kernels
                     "traffic": profiled_traffic(w.name) if args.format == "int2" else None, "peak_kind": peak_kind,
                     "algorithmic_bytes": r["fused_bytes"], "algorithmic_bytes_per_reader": r["reader_bytes"],
                     "launch_us": round(r["fused_us"], 3)},
        "step_us_per_layer_p10_p50_p90": [round(x * 1000.0 / n_layers, 3) for x in r["step_pct"]],
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "plan": {"items": r["n_items"], "bf16_items": r["n_bf16_items"], "max_item_pages": r["max_item_pages"],
                 "mean_int2_item_pages": round(r["int2_pages"] / max(1, r["n_items"] - r["n_bf16_items"]), 1)},
        "setup_s": {"calibration": round(r["t_cal"], 2), "fill": round(r["t_fill"], 2)},
    }
    if r["e2e"]:
        line["e2e"] = r["e2e"]
    if r["bf16"]:
        line["bf16_comparison"] = r["bf16"]
        # per request-layer: the BF16 cache may hold fewer requests of the batch (HBM capacity)
        line["speedup_vs_bf16_decode"] = round((r["bf16"]["us_per_layer"] / r["bf16"]["requests"]) /
                                               (r["decode_us"] / r["B"]), 3)
    return line


def release_gpu_memory():
    import gc

    import torch

    gc.collect()
    torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_info()
    from int2_rotated_kv_rotate_gb300 import workloads as wl

    names = [HEADLINE] + OTHERS if args.workload == "all" else [args.workload]
    if args.impl == "reference":
        return main_reference(args, world, rank, wl.WORKLOADS[names[0]])
    if args.layers and len(names) > 1:
        raise SystemExit("--layers applies to one workload (--workload NAME)")
    lines = {}
    for name in names:
        w = wl.WORKLOADS[name]
        r = run_ours(args, w, world, rank, local)
        lines[name] = result_line(args, w, r, world)
        if rank == 0 and world == 1 and not args.no_cpu_baseline and name == names[0]:
            lines[name]["cpu_baseline"] = cpu_baseline(w, args.seed)
        del r
        release_gpu_memory()
    cm_line = None
    if len(names) > 1 and not args.no_cm and args.format == "int2":
        # the headline workload again, channel-major value pages decoded on tcgen05: the
        # same metric, steps and inputs; reported beside the headline, not instead of it
        import copy

        a2 = copy.copy(args)
        a2.format, a2.no_bf16, a2.no_e2e = "int2_cm", True, True
        w = wl.WORKLOADS[names[0]]
        r = run_ours(a2, w, world, rank, local)
        full = result_line(a2, w, r, world)
        cm_line = {k: full[k] for k in ("value", "unit", "ms_per_step", "decode_us_per_layer", "roofline",
                                        "step_us_per_layer_p10_p50_p90", "gpu_launches", "clocks", "plan")}
        cm_line["format"] = "OSCAR_FORMAT_INT2_CM"
        del r
        release_gpu_memory()
    folded_line = None
    if len(names) > 1 and not args.no_folded and not args.folded and "qwen3_8b_layer" in names:
        # the latency-bound 8B-shaped step again with the rotations folded into the model's
        # projections (q~ in, o~ out): the q and output rotations leave the launch
        import copy

        a2 = copy.copy(args)
        a2.folded, a2.no_bf16 = True, True
        w = wl.WORKLOADS["qwen3_8b_layer"]
        r = run_ours(a2, w, world, rank, local)
        full = result_line(a2, w, r, world)
        folded_line = {k: full[k] for k in ("value", "unit", "ms_per_step", "decode_us_per_layer", "roofline",
                                            "step_us_per_layer_p10_p50_p90", "gpu_launches", "clocks")}
        if "e2e" in full:
            folded_line["e2e"] = full["e2e"]
        folded_line["plan_flags"] = "OSCAR_PLAN_FOLDED_ROTATIONS"
        del r
        release_gpu_memory()
    serving_line = None
    if len(names) > 1 and not args.no_serving:
        import torch

        serving_line = serving_comparison(args.seed + 1000 * rank, torch.device("cuda", local))
        release_gpu_memory()
    if rank != 0:
        return 0
    line = lines[names[0]]
    if cm_line:
        line["int2_cm_format"] = cm_line
    if serving_line:
        line["serving"] = serving_line
    if len(names) > 1:
        line["per_workload"] = {n: {k: v for k, v in lines[n].items() if k not in ("metric", "n_gpus", "steps", "warmup",
                                                                                  "higher_is_better", "scaling",
                                                                                  "vs_baseline", "data")}
                                for n in names[1:]}
        if folded_line and "qwen3_8b_layer" in line["per_workload"]:
            line["per_workload"]["qwen3_8b_layer"]["folded_rotations"] = folded_line
    print(json.dumps(line), flush=True)
    return 0


def main_reference(args, world, rank, w):
    """The CPU oracle on the host cores, same metric and workload: each step is a bounded
    sample (one kv-head of one request at up to 32768 tokens: append + decode), timed as
    it runs; the line's value scales the sample to one layer-step of the workload, and
    ms_per_step is the sample's own measured time, so ms_per_step x steps is time spent."""
    if rank != 0:
        return 0
    import oracle

    oracle.set_threads(1)  # the oracle's decode is serial; its rotation alone would use more
    nproc, model = host_cpu()
    context = min(w.context, 32768)
    step = oracle_sample(w, args.seed, [0], context)
    for s in range(args.warmup):
        step(0)
    times = [step(0) for s in range(args.steps)]
    scale = w.n_kv_heads * w.batch * (w.context / context)
    us = statistics.mean(times) * scale * 1e6
    sample = (f"one thread; per step one kv-head of request 0, layer 0, context {context}: append "
              f"{w.append_per_step or 1} token(s) + decode 1 query, measured {statistics.mean(times) * 1e3:.1f} ms; "
              f"value = that x{scale:.0f} (kv-heads x batch x context ratio) = one layer-step of the workload")
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/layer/step", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 3),
            "sample_scale": round(scale, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 quantizer",
            "data": "synthetic", "config": config_of(w, w.n_layers),
            "cpu_baseline": {"value": round(us, 1), "unit": "us/layer/step", "cores": 1, "kind": "oracle",
                             "nproc": nproc, "cpu_model": model, "sample": sample},
            "e2e": {"value": round(us, 1), "unit": "us/layer/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
