"""Benchmark of the W4A16 linear layer on GB300.

One step = one pass of the decode hot path over one batch: the four linear
layers of a Qwen3-4B-shaped model (qkv 6144x2560, o_proj 2560x4096, gate_up
19456x2560, down 2560x9728), symmetric uint4b8 weights, G = 128, bf16
activations, M = 1 token.  `value` is the algorithmic weight + metadata +
activation byte stream per step divided by the device time per step (GB/s),
with every input resident in HBM; weight sets rotate so that each step
streams from HBM (the sets together are larger than 3x the L2).

The second half of the metric, the M = 1920 prefill GEMM in TFLOP/s, is
measured in the same run on the Llama-3.1-8B-shaped asymmetric bf16 G = 64
layers and reported under "prefill".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --profile-case decode|prefill [--profile-m M] --steps K --warmup W   (ncu)
  python bench.py --crossover        (decode vs prefill kernel time, M = 1..16)

--impl reference times the CPU oracle (plain C, fp64) on the same workload
(a bounded sample of steps) on the host cores.  With N > 1 (torchrun) every
rank runs an independent replica (the layer has no data-path exchange);
timing is the max over ranks and value the sum of their work.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w4a16_group_quantised_gb300 import workloads as wl  # noqa: E402

METRIC = ("M=1 decode weight-stream GB/s (% HBM peak); "
          "M=1920 prefill TFLOP/s (% TC peak)")
DECODE_WORKLOAD = "qwen3-4b-decode-m1-sym-g128-bf16"
PREFILL_WORKLOAD = "llama-3.1-8b-prefill-m1920-asym-g64-bf16"
L2_BYTES_FALLBACK = 126 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0     # the nominal "~8 TB/s" of HBM3e, shown beside the measured peak


# ----------------------------------------------------------------- helpers
def decode_bytes(M, N, K, G, sym):
    """Algorithmic bytes of one decode GEMM: packed weights, scales, zero
    points (asymmetric), x and y."""
    b = N * K // 2 + N * (K // G) * 2 + M * K * 2 + M * N * 2
    if not sym:
        b += (N // 8) * (K // G) * 4
    return b


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "w4a16_group_quantised_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag, src_hash):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed ncu summary profiles/traffic.txt, whose lines read
    `<tag> <source hash> <bytes per launch>`; None unless the figure was taken
    on the current source of that kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 3 and parts[0] == kernel_tag and parts[1] == src_hash:
                    return int(float(parts[2]))
    except OSError:
        pass
    return None


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes) while
    the timed region runs.  Reads only; changes no setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index=0, period_s=0.0005):
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
                self.max_mhz = mx.value
            self.ok = True
        except Exception:
            self.ok = False

    def sample(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
            self.samples.append(clk.value)
        if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
            for bit, name in self.REASONS.items():
                if rs.value & bit:
                    self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            self.sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.sample()
            self._stop.clear()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()
            self.sample()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": len(self.samples)}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- our arm
def upload(w, p):
    q = torch.from_numpy(p.q).cuda()
    qweight = w.w4a16_pack(q)
    del q
    qzeros = None
    if p.z is not None:
        qzeros = w.w4a16_pack_zeros(torch.from_numpy(p.z).cuda())
    td = torch.float16 if p.dtype == 0 else torch.bfloat16
    scales = torch.from_numpy(p.scales.view(np.int16)).view(td).cuda()
    x = torch.from_numpy(p.x.view(np.int16)).view(td).cuda()
    return dict(qweight=qweight, scales=scales, qzeros=qzeros, x=x, M=p.M, N=p.N, K=p.K, G=p.G,
                sym=p.sym, dtype=p.dtype)


def layer_bytes(d):
    return decode_bytes(d["M"], d["N"], d["K"], d["G"], d["sym"])


def rotated_sets(base, n_sets):
    """n_sets weight sets of the same layers.  Set 0 is `base` (from the
    seeded generator); the others are copies with bytes permuted by a cheap
    device roll so that every set is distinct memory (the values are equally
    distributed)."""
    sets = [base]
    for s in range(1, n_sets):
        cur = []
        for d in base:
            e = dict(d)
            e["qweight"] = torch.roll(d["qweight"], shifts=s, dims=1).contiguous()
            e["scales"] = torch.roll(d["scales"], shifts=s, dims=0).contiguous()
            if d["qzeros"] is not None:
                e["qzeros"] = torch.roll(d["qzeros"], shifts=s, dims=0).contiguous()
            cur.append(e)
        sets.append(cur)
    return sets


def make_sets(w, make, n_sets, shapes_count):
    return rotated_sets([upload(w, make(i)) for i in range(shapes_count)], n_sets)


def run_step(w, layers, outs, only=None):
    for i, (d, o) in enumerate(zip(layers, outs)):
        if only is None or i == only:
            if d.get("epi") is not None or d.get("bias") is not None:
                w.w4a16_gemm_fused(d["x"], d["qweight"], d["scales"], d["qzeros"], d["G"], bias=d.get("bias"),
                                   epilogue=d.get("epi") or 0, out=o, path=d.get("path", 0))
            else:
                w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], d["G"], out=o,
                             path=d.get("path", 0))


class LayerStream:
    """The layers of one workload, in rotating weight sets larger than 3x the
    L2 together (every launch streams its weights from HBM), launched from
    CUDA graphs on a side stream.  A graph of `chunk` steps ends on the set it
    started from (chunk is a multiple of the set count), so replays rotate.
    Every graph is replayed once right after capture, so no timed replay is a
    graph's first."""

    def __init__(self, w, base, l2_bytes, launches_target=64):
        self.w = w
        self.step_bytes = sum(layer_bytes(d) for d in base)
        self.layer_bytes = [layer_bytes(d) for d in base]
        self.n_sets = max(2, int(np.ceil(3 * l2_bytes / self.step_bytes)) + 1)
        self.sets = rotated_sets(base, self.n_sets)
        td = torch.float16 if base[0]["dtype"] == 0 else torch.bfloat16
        self.outs = [torch.empty((d["M"], d["N"] // 2 if d.get("epi") == 1 else d["N"]), dtype=td, device="cuda")
                     for d in base]
        self.stream = torch.cuda.Stream()
        self.chunk = self.n_sets * max(1, launches_target // self.n_sets)
        self.graphs = {}
        with torch.cuda.stream(self.stream):
            for s in range(self.n_sets):   # first calls outside capture (per-device set-up)
                run_step(w, self.sets[s], self.outs)
        torch.cuda.synchronize()

    def graph(self, n, only=None):
        key = (n, only)
        if key not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g, stream=self.stream):
                    for i in range(n):
                        run_step(self.w, self.sets[i % self.n_sets], self.outs, only)
                g.replay()
            torch.cuda.synchronize()
            self.graphs[key] = g
        return self.graphs[key]

    def prepare(self, *counts):
        for n in counts:
            if n % self.chunk:
                self.graph(n % self.chunk)
        self.graph(self.chunk)

    def replay_steps(self, n, only=None):
        """Exactly n steps: n // chunk replays of the chunk graph, then one
        replay of the graph of the remaining steps."""
        with torch.cuda.stream(self.stream):   # replay() launches on the current stream
            for _ in range(n // self.chunk):
                self.graph(self.chunk, only).replay()
            if n % self.chunk:
                self.graph(n % self.chunk, only).replay()

    def timed(self, n, ws=1, only=None):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        start.record(self.stream)
        self.replay_steps(n, only)
        end.record(self.stream)
        torch.cuda.synchronize()
        barrier(ws)
        return start.elapsed_time(end) / 1000.0

    def median_step_s(self, reps=20, only=None):
        """Median over `reps` replays of the chunk graph, per step."""
        self.graph(self.chunk, only)
        return statistics.median(self.timed(self.chunk, 1, only) for _ in range(reps)) / self.chunk

    def per_layer(self, reps=20):
        """Each layer alone (single-launch timing per shape): median seconds
        per launch and GB/s."""
        out = []
        for i, b in enumerate(self.layer_bytes):
            t = self.median_step_s(reps, only=i)
            out.append((t, b / t / 1e9))
        return out


def stream_summary(st, hbm, layer_names, reps=20):
    """Whole-step median (the layer stream) and per-shape figures of one
    LayerStream."""
    t_step = st.median_step_s(reps)
    per = st.per_layer(reps)
    gbs = st.step_bytes / t_step / 1e9
    return {"step_us": round(t_step * 1e6, 3), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
            "frac_nominal_8000": round(gbs / NOMINAL_HBM_GBS, 4), "step_bytes": st.step_bytes,
            "per_shape": {name: {"us": round(t * 1e6, 3), "GB/s": round(g, 1), "frac": round(g / hbm, 4),
                                 "bytes": b}
                          for name, (t, g), b in zip(layer_names, per, st.layer_bytes)}}


def bench_decode_e2e(w, st, steps):
    """End to end through the public API: every step copies the step's
    activations (the four layers' x, one pinned host buffer) to the device in
    one transfer, runs the four layers with w4a16_gemm on views of it, copies
    the four outputs back to one pinned host buffer in one transfer, and
    synchronises.  The step is captured once per weight set in a CUDA graph
    (transfers and kernels), as a serving loop would, and each step replays
    one."""
    layers = st.sets[0]
    dt_ = layers[0]["x"].dtype
    xk = [d["M"] * d["K"] for d in layers]
    yn = [d["M"] * d["N"] for d in layers]
    x_host = torch.cat([d["x"].reshape(-1) for d in layers]).cpu().pin_memory()
    y_host = torch.empty(sum(yn), dtype=dt_).pin_memory()
    x_dev = torch.empty(sum(xk), dtype=dt_, device="cuda")
    y_dev = torch.empty(sum(yn), dtype=dt_, device="cuda")
    xo = np.concatenate([[0], np.cumsum(xk)])
    yo = np.concatenate([[0], np.cumsum(yn)])
    xv = [x_dev[xo[i]:xo[i + 1]].view(d["M"], d["K"]) for i, d in enumerate(layers)]
    yv = [y_dev[yo[i]:yo[i + 1]].view(d["M"], d["N"]) for i, d in enumerate(layers)]
    h2d = x_host.numel() * x_host.element_size()
    d2h = y_host.numel() * y_host.element_size()
    n = max(3, min(steps, 2000))
    stream = st.stream

    def enqueue(layers_i):
        x_dev.copy_(x_host, non_blocking=True)
        for d, a, b in zip(layers_i, xv, yv):
            w.w4a16_gemm(a, d["qweight"], d["scales"], d["qzeros"], d["G"], out=b, stream=stream)
        y_host.copy_(y_dev, non_blocking=True)

    with torch.cuda.stream(stream):
        enqueue(layers)
        stream.synchronize()
        graphs = []
        for sset in st.sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                enqueue(sset)
            graphs.append(g)
        for g in graphs:
            g.replay()
        graphs[0].replay()
        stream.synchronize()
        for i, d in enumerate(layers):   # the replayed step's host result is the device call's
            ref = w.w4a16_gemm(d["x"], d["qweight"], d["scales"], d["qzeros"], d["G"]).reshape(-1).cpu()
            assert torch.equal(y_host[yo[i]:yo[i + 1]], ref), "e2e step differs from the device call"
        t0 = time.perf_counter()
        for i in range(n):
            graphs[i % len(graphs)].replay()
            stream.synchronize()
        dt = (time.perf_counter() - t0) / n
    return dict(dt=dt, h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h, steps=n)


def bench_fused_epilogue(w, l2, hbm):
    """The Qwen3-4B gate_up layer at M = 1 alone, plain, with a bias, and with
    the fused SiLU-and-multiply (same weights, rotating sets past L2):
    median microseconds per launch and weight-stream GB/s of each."""
    name, N, K = wl.QWEN3_4B_SHAPES[2]
    d0 = upload(w, wl.qwen3_4b_decode(2, 1))
    bias = torch.randn((N,), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
    out = {}
    for tag, extra in (("plain", {}), ("bias", {"bias": bias}), ("silu_mul", {"epi": 1}),
                       ("bias_silu_mul", {"bias": bias, "epi": 1})):
        st = LayerStream(w, [dict(d0, **extra)], l2, launches_target=32)
        t = st.median_step_s(15)
        out[tag] = {"us": round(t * 1e6, 3), "GB/s": round(st.step_bytes / t / 1e9, 1)}
        del st
        torch.cuda.empty_cache()
    return {"workload": f"qwen3-4b {name} {N}x{K} M=1 bf16 sym G128", **out}


def bench_prefill(w, steps, reps=5):
    """M = 1920 prefill on the four Llama-3.1-8B-shaped layers (one weight set:
    the contraction is compute-bound, ~0.1-0.4 ms per launch).  Per shape:
    median over `reps` regions of `steps` back-to-back launches; the step: the
    four layers in order, same median."""
    shapes = wl.LLAMA31_8B_SHAPES
    layers = [upload(w, wl.llama31_8b_prefill(i, 1920)) for i in range(len(shapes))]
    outs = [torch.empty((1920, N), dtype=torch.bfloat16, device="cuda") for (_, N, K) in shapes]
    flops = [2 * 1920 * N * K for (_, N, K) in shapes]
    stream = torch.cuda.Stream()

    def region(only):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            run_step(w, layers, outs, only)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1000.0 / steps

    with torch.cuda.stream(stream):
        for _ in range(3):
            run_step(w, layers, outs)
        torch.cuda.synchronize()
        per_s = [statistics.median(region(i) for _ in range(reps)) for i in range(len(shapes))]
        dt = statistics.median(region(None) for _ in range(reps))
    del layers, outs
    return dict(tflops=sum(flops) / dt / 1e12, ms_per_step=dt * 1e3, flops_per_step=sum(flops),
                per_shape_ms=[t * 1e3 for t in per_s],
                per_shape_tflops=[f / t / 1e12 for f, t in zip(flops, per_s)])


def bench_prefill_cache(w, M, steps, reps=5):
    """The Llama-3.1-8B-shaped layers at M through the dequantised prefill
    cache (w4a16_gemm_dense on W = RN((q - z) s) built once by
    w4a16_dequantize, not timed): per-shape and whole-step medians."""
    shapes = wl.LLAMA31_8B_SHAPES
    layers = [upload(w, wl.llama31_8b_prefill(i, M)) for i in range(len(shapes))]
    caches = [w.w4a16_dequantize(d["qweight"], d["scales"], d["qzeros"], d["G"]) for d in layers]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for (_, N, K) in shapes]
    flops = [2 * M * N * K for (_, N, K) in shapes]
    stream = torch.cuda.Stream()

    def region(only):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            for i, (d, c, o) in enumerate(zip(layers, caches, outs)):
                if only is None or i == only:
                    w.w4a16_gemm_dense(d["x"], c, out=o)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1000.0 / steps

    with torch.cuda.stream(stream):
        for _ in range(3):
            region(None)
        per_s = [statistics.median(region(i) for _ in range(reps)) for i in range(len(shapes))]
        dt = statistics.median(region(None) for _ in range(reps))
    del layers, caches, outs
    torch.cuda.empty_cache()
    return dict(tflops=sum(flops) / dt / 1e12, ms_per_step=dt * 1e3,
                per_shape_tflops={n: round(f / t / 1e12, 1) for (n, _, _), f, t in zip(shapes, flops, per_s)},
                per_shape_us={n: round(t * 1e6, 2) for (n, _, _), t in zip(shapes, per_s)})


def bench_moe(w, hbm, T=1, topk=8, E=128, steps_per_graph=48, reps=20):
    """MoE decode on Qwen3-30B-A3B-like experts (128 experts, top-8, bf16,
    symmetric, G = 128): per step one grouped GEMM over the experts' gate_up
    (1536 x 2048) and one over their down (2048 x 768), each step with its own
    seeded routing (a different id buffer per step in the graph), so the
    experts' weights (about 300 MB in all) stream from HBM.  Algorithmic
    bytes per step: the packed weights and scales of the distinct experts the
    step routes to (averaged over the steps' routings), x and y."""
    shapes = [("experts gate_up", 1536, 2048), ("experts down", 2048, 768)]
    G = 128
    stacks = []
    for si, (name, N, K) in enumerate(shapes):
        q = torch.randint(0, 16, (E * N, K), dtype=torch.uint8,
                          generator=torch.Generator(device="cuda").manual_seed(si), device="cuda")
        qw = w.w4a16_pack(q).view(E, N, K // 8)
        del q
        sc = (torch.rand((E, N, K // G), generator=torch.Generator().manual_seed(10 + si)) * 0.018 + 0.002)
        stacks.append(dict(N=N, K=K, qweight=qw, scales=sc.to(torch.bfloat16).cuda()))
    rng = np.random.default_rng(7)
    ids_h = [np.stack([rng.choice(E, topk, replace=False) for _ in range(T)]).astype(np.int32)
             for _ in range(steps_per_graph)]
    ids = [torch.from_numpy(a).cuda() for a in ids_h]
    distinct = float(np.mean([len(np.unique(a)) for a in ids_h]))   # experts each step must stream
    rw = torch.full((T, topk), 1.0 / topk, dtype=torch.float32, device="cuda")
    x0 = torch.randn((T, shapes[0][2]), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).cuda()
    x1 = torch.randn((T * topk, shapes[1][2]), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).cuda()
    outs = [torch.empty((T, topk, N), dtype=torch.bfloat16, device="cuda") for (_, N, _) in shapes]

    def step(i):
        a, b = stacks
        w.w4a16_moe_gemm(x0, a["qweight"], a["scales"], None, G, ids[i], out=outs[0])
        # down: each (token, slot) row is its own token routed to its expert once
        w.w4a16_moe_gemm(x1, b["qweight"], b["scales"], None, G, ids[i].view(T * topk, 1), route_weights=rw.view(-1, 1),
                         out=outs[1].view(T * topk, 1, -1))

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step(0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps_per_graph):
                step(i)
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3 / steps_per_graph)
    dt = statistics.median(ts)
    per_expert = sum(N * K // 2 + N * (K // G) * 2 for (_, N, K) in shapes)
    step_bytes = int(distinct * per_expert) + T * shapes[0][2] * 2 + \
        T * topk * (shapes[0][1] + shapes[1][2] + shapes[1][1]) * 2
    del stacks, ids, outs
    torch.cuda.empty_cache()
    return {"workload": f"moe-decode T={T} top{topk} of {E} experts, gate_up 1536x2048 + down 2048x768, bf16 sym G128",
            "distinct_experts_per_step": round(distinct, 2), "step_us": round(dt * 1e6, 3), "GB/s": round(step_bytes / dt / 1e9, 1),
            "frac": round(step_bytes / dt / 1e9 / hbm, 4), "step_bytes": step_bytes}


def profile_case(w, which, steps, warmup, m=None):
    """A short run for ncu captures: `warmup` then `steps` eager passes over
    the four layers of one workload (one set of inputs, launched in layer
    order); `m` overrides the workload's batch size (prefill: any M, e.g.
    128 for the K split over a cluster).  Prints a timing line of its own,
    not a bench line."""
    if which == "decode":
        layers = [upload(w, wl.qwen3_4b_decode(i, m or 1)) for i in range(len(wl.QWEN3_4B_SHAPES))]
    else:
        layers = [upload(w, wl.llama31_8b_prefill(i, m or 1920)) for i in range(len(wl.LLAMA31_8B_SHAPES))]
    td = torch.float16 if layers[0]["dtype"] == 0 else torch.bfloat16
    outs = [torch.empty((d["M"], d["N"]), dtype=td, device="cuda") for d in layers]
    for _ in range(warmup):
        run_step(w, layers, outs)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        run_step(w, layers, outs)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": which, "M": layers[0]["M"], "steps": steps, "warmup": warmup,
                      "host_ms_per_step": (time.perf_counter() - t0) / steps * 1e3,
                      "device_status": w.w4a16_last_device_error()}))


def crossover(w, reps=15):
    """Decode vs prefill kernel time for M = 1..16 on the dispatcher sweep
    shapes, every group size, both quantisation forms and both dtypes; L2 is
    flushed before every launch.  Prints one JSON line per cell and a summary
    of the largest M at which the decode kernel is still the faster one."""
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    summary = {}
    for si, (N, K) in enumerate(wl.SWEEP_SHAPES):
        for G in (32, 64, 128):
            for sym in (True, False):
                for dtype in (0, 1):
                    td = torch.float16 if dtype == 0 else torch.bfloat16
                    p = wl.make_problem(16, N, K, G, sym, dtype, seed=7000 + si * 100 + G + 2 * sym + dtype)
                    d = upload(w, p)
                    best_m = 0
                    for M in range(1, 17):
                        x = d["x"][:M].contiguous()
                        out = torch.empty((M, N), dtype=td, device="cuda")
                        times = {}
                        for path in ((1, 2) if M <= 8 else (2,)):
                            ts = []
                            for r in range(reps + 2):
                                flush.zero_()
                                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                                e0.record()
                                w.w4a16_gemm(x, d["qweight"], d["scales"], d["qzeros"], G, out=out, path=path)
                                e1.record()
                                torch.cuda.synchronize()
                                if r >= 2:
                                    ts.append(e0.elapsed_time(e1) * 1e3)
                            times[path] = float(np.median(ts))
                        if 1 in times and times[1] <= times[2]:
                            best_m = M
                        print(json.dumps({"crossover_cell": {"N": N, "K": K, "G": G, "sym": sym,
                                                             "dtype": wl.DTYPE_NAME[dtype], "M": M,
                                                             "decode_us": times.get(1), "prefill_us": times[2]}}))
                    summary[f"{N}x{K} G{G} {'sym' if sym else 'asym'} {wl.DTYPE_NAME[dtype]}"] = best_m
                    del d
                    torch.cuda.empty_cache()
    print(json.dumps({"crossover_largest_decode_m": summary}))


def crossover_graph(w, hbm):
    """Decode vs prefill kernel in the regime the product runs in: each
    kernel forced, one layer per step, CUDA graphs with programmatic
    dependent launch, weight sets rotating past L2.  One JSON line per cell
    and M, then the largest M at which the decode kernel is the faster."""
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size or L2_BYTES_FALLBACK
    summary = {}
    for si, (N, K) in enumerate(wl.SWEEP_SHAPES):
        for (G, sym, dtype) in ((128, True, 1), (32, False, 0)):
            best_m = 0
            for M in (1, 2, 4, 6, 8, 12, 16):
                times = {}
                for path in ((1, 2) if M <= 8 else (2,)):
                    d = upload(w, wl.make_problem(M, N, K, G, sym, dtype, seed=8000 + si * 10 + M))
                    d["path"] = path
                    st = LayerStream(w, [d], l2, launches_target=32)
                    times[path] = st.median_step_s(9) * 1e6
                    del st, d
                    torch.cuda.empty_cache()
                if 1 in times and times[1] <= times[2]:
                    best_m = M
                print(json.dumps({"crossover_graph_cell": {"N": N, "K": K, "G": G, "sym": sym,
                                                           "dtype": wl.DTYPE_NAME[dtype], "M": M,
                                                           "decode_us": None if 1 not in times else round(times[1], 2),
                                                           "prefill_us": round(times[2], 2)}}), flush=True)
            summary[f"{N}x{K} G{G} {'sym' if sym else 'asym'} {wl.DTYPE_NAME[dtype]}"] = best_m
    print(json.dumps({"crossover_graph_largest_decode_m": summary}))


def decode_timeline(w, reps=3):
    """Where one M = 1 decode step goes: the benchmark's graphed step of the
    four Qwen3-4B-shaped layers (rotating weight sets, early launch) on the
    trace build of the library (libw4a16_trace.so: the decode kernel with its
    timeline stamps compiled in) with the hook on.  After each of `reps`
    graph replays, per layer: the min / median / max over CTAs of entry,
    release (grid dependency wait returned), first weight stage ready and
    exit, the median loop time and the tail (last minus median exit), in
    microseconds from the step's first CTA entry.  One JSON line per replay."""
    shapes = wl.QWEN3_4B_SHAPES
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size or L2_BYTES_FALLBACK
    base = [upload(w, wl.qwen3_4b_decode(i, 1)) for i in range(len(shapes))]
    st = LayerStream(w, base, l2, launches_target=32)
    buf = w.w4a16_debug_decode_trace([(N, K) for (_, N, K) in shapes])
    try:
        for rep in range(reps):
            st.replay_steps(st.chunk)
            torch.cuda.synchronize()
            tr = buf.cpu().numpy()
            used = tr[:, :, 0] > 0
            t0 = tr[:, :, 0][used].min()
            q = lambda v: [round(float(v.min()), 2), round(float(np.median(v)), 2), round(float(v.max()), 2)]
            out, prev_exit = {}, None
            for li, (name, N, K) in enumerate(shapes):
                a = (tr[li][used[li]].astype(np.int64) - t0) / 1000.0
                d = {"ctas": int(a.shape[0]), "entry": q(a[:, 0]), "released": q(a[:, 1]),
                     "first_stage": q(a[:, 3]), "exit": q(a[:, 6]),
                     "loop_us_median": round(float(np.median(a[:, 4] - a[:, 3])), 2),
                     "tail_us": round(float(a[:, 6].max() - np.median(a[:, 6])), 2)}
                if prev_exit is not None:
                    d["release_after_previous_last_exit_us"] = round(float(a[:, 1].min() - prev_exit), 2)
                prev_exit = float(a[:, 6].max())
                out[name] = d
            print(json.dumps({"decode_timeline": out, "replay": rep}), flush=True)
    finally:
        w.w4a16_debug_decode_trace(None)
        del buf, st, base
        torch.cuda.empty_cache()


def cpu_baseline(sample_steps=None, budget_s=15.0):
    """The oracle (as it stands) on the host cores, on whole decode steps."""
    import oracle
    oracle.build()
    shapes = wl.QWEN3_4B_SHAPES
    probs = [wl.qwen3_4b_decode(i, 1) for i in range(len(shapes))]
    packed = [oracle.pack(p.q) for p in probs]
    step_bytes = sum(decode_bytes(1, N, K, 128, True) for (_, N, K) in shapes)
    t0 = time.perf_counter()
    n = 0
    while True:
        for p, qw in zip(probs, packed):
            oracle.gemm(p.x, p.M, p.K, qw, p.scales, None, p.G, p.N, p.dtype)
        n += 1
        el = time.perf_counter() - t0
        if (sample_steps is not None and n >= sample_steps) or (sample_steps is None and el >= budget_s):
            break
    dt = (time.perf_counter() - t0) / n
    return dict(value=step_bytes / dt / 1e9, unit="GB/s", cores=oracle.num_threads(), kind="oracle",
                sample=f"{n} whole decode steps (4 Qwen3-4B-shaped layers, M=1) in fp64 C",
                s_per_step=dt, nproc=os.cpu_count())


def cpu_baseline_single_thread(budget_s):
    """The same oracle timing in a child process with one OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-only",
                        "--cpu-budget", str(budget_s)], env=env, capture_output=True, text=True,
                       timeout=budget_s * 20 + 300)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def reference_arm(steps, warmup, budget_s=150.0):
    """The oracle (as it stands) on the host cores, over `warmup` untimed and
    `steps` timed steps of the decode workload.  A whole step (the four
    layers, every weight row) takes ~0.2 s on the host, so when steps +
    warmup of them would not fit in `budget_s` each step is a bounded sample:
    the same contiguous fraction of every layer's weight rows (a multiple of
    8, at least 8), moving through the rows from step to step.  The metric is
    bytes streamed per second, so it is the same quantity either way."""
    import oracle
    oracle.build()
    shapes = wl.QWEN3_4B_SHAPES
    probs = [wl.qwen3_4b_decode(i, 1) for i in range(len(shapes))]
    packed = [oracle.pack(p.q) for p in probs]
    t0 = time.perf_counter()
    for p, qw in zip(probs, packed):
        oracle.gemm(p.x, p.M, p.K, qw, p.scales, None, p.G, p.N, p.dtype)
    t_full = time.perf_counter() - t0
    total = max(1, steps + warmup)
    frac = min(1.0, budget_s / (total * t_full))
    nrows = [min(p.N, max(8, int(p.N * frac) // 8 * 8)) for p in probs]

    def one_step(i):
        nbytes = 0
        for p, qw, nr in zip(probs, packed, nrows):
            n0 = (i * nr) % (p.N - nr + 1) // 8 * 8
            oracle.gemm(p.x, p.M, p.K, qw[n0:n0 + nr], p.scales[n0:n0 + nr], None, p.G, nr, p.dtype)
            nbytes += decode_bytes(p.M, nr, p.K, p.G, True)
        return nbytes

    for i in range(warmup):
        one_step(i)
    nbytes = 0
    t0 = time.perf_counter()
    for i in range(steps):
        nbytes += one_step(warmup + i)
    dt = max(time.perf_counter() - t0, 1e-9)
    sample = (f"each step: rows {nrows} of the four Qwen3-4B-shaped layers "
              f"(N = {[p.N for p in probs]}), M=1, in fp64 C" if frac < 1.0 else
              "each step: the whole decode step (4 Qwen3-4B-shaped layers, M=1) in fp64 C")
    return dict(value=nbytes / dt / 1e9, unit="GB/s", cores=oracle.num_threads(), kind="oracle",
                sample=sample, s_per_step=dt / max(steps, 1))


def decode_config(ws):
    """The `config` of the headline line; both arms print this same dict."""
    return {"workload": DECODE_WORKLOAD, "M": 1,
            "layers": "qkv 6144x2560, o_proj 2560x4096, gate_up 19456x2560, down 2560x9728",
            "G": 128, "quant": "uint4b8 (symmetric)", "act": "bf16",
            "l2": "rotating weight sets larger than 3x L2",
            "parallelism": "replicas" if ws > 1 else "single-gpu"}


def extra_decode(w, make, shapes, M, l2, hbm):
    base = [upload(w, make(i, M)) for i in range(len(shapes))]
    st = LayerStream(w, base, l2)
    out = stream_summary(st, hbm, [n for (n, _, _) in shapes])
    del st, base
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the extra workloads (Llama decode, M sweep, M=128 prefill)")
    ap.add_argument("--no-median", action="store_true",
                    help="skip the per-shape and whole-step median replays of the decode layers")
    ap.add_argument("--profile-case", choices=["decode", "prefill"],
                    help="run only the short eager case that ncu captures")
    ap.add_argument("--profile-m", type=int, default=None,
                    help="batch size of the --profile-case workload (default: its own)")
    ap.add_argument("--crossover", action="store_true",
                    help="time both kernels at M = 1..16 (the dispatcher's threshold sweep)")
    ap.add_argument("--crossover-graph", action="store_true",
                    help="the same comparison in CUDA graphs with early launch and rotating weights")
    ap.add_argument("--decode-timeline", action="store_true",
                    help="per-CTA timeline of one graphed M=1 decode step (builds and loads the trace build)")
    ap.add_argument("--cpu-baseline-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_baseline_only:
        print(json.dumps(cpu_baseline(sample_steps=None, budget_s=args.cpu_budget)))
        return
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)
    ws, rank, local = dist_info()
    hbm, tc, tc_sus, peak_src = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        cb = reference_arm(max(args.steps, 1), max(args.warmup, 0))
        line = {"metric": METRIC, "value": round(cb["value"], 4), "unit": "GB/s", "n_gpus": args.gpus,
                "steps": max(args.steps, 1), "warmup": max(args.warmup, 0), "ms_per_step": cb["s_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference", "config": decode_config(ws),
                "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": round(cb["value"], 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    from w4a16_group_quantised_gb300 import build as libbuild
    if args.decode_timeline:                         # the profiling build, stamps compiled in
        os.environ["W4A16_LIBRARY"] = "trace"
        libbuild.build(variant="trace")
    else:
        libbuild.build()
    import w4a16_group_quantised_gb300 as w
    w.load_library()

    if args.profile_case:
        profile_case(w, args.profile_case, steps, warmup, args.profile_m)
        return
    if args.crossover:
        crossover(w)
        return
    if args.crossover_graph:
        crossover_graph(w, hbm)
        return
    if args.decode_timeline:
        decode_timeline(w)
        return

    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size or L2_BYTES_FALLBACK
    qshapes = wl.QWEN3_4B_SHAPES
    st = LayerStream(w, [upload(w, wl.qwen3_4b_decode(i, 1)) for i in range(len(qshapes))], l2)
    st.prepare(steps, warmup)
    st.replay_steps(warmup)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        dt = st.timed(steps, ws)
    # A short timed region yields few clock samples: keep sampling over
    # about 0.3 s more of the same replays (untimed) right after it.
    soak = None
    if dt < 0.3:
        per_chunk = max(dt / steps * st.chunk, 1e-6)
        n_soak = st.chunk * int(np.ceil(0.3 / per_chunk))
        with ClockSampler(torch.cuda.current_device()) as soak:
            st.replay_steps(n_soak)
            torch.cuda.synchronize()
    dt = max_over_ranks(dt, ws)
    ms_per_step = dt / steps * 1e3
    value = st.step_bytes * steps * ws / dt / 1e9
    launches = steps * len(qshapes)
    per_launch_s = dt / launches
    achieved = st.step_bytes / len(qshapes) / per_launch_s / 1e9
    qsum = None if args.no_median else stream_summary(st, hbm, [n for (n, _, _) in qshapes])

    e2e = None
    if not args.no_e2e:
        r = bench_decode_e2e(w, st, min(args.steps, 500))
        edt = max_over_ranks(r["dt"], ws)
        e2e = dict(value=st.step_bytes * ws / edt / 1e9, unit="GB/s",
                   h2d_bytes_per_step=r["h2d_bytes_per_step"],
                   d2h_bytes_per_step=r["d2h_bytes_per_step"], steps=r["steps"],
                   ms_per_step=edt * 1e3,
                   api="one pinned host->device copy of the step's activations, w4a16_gemm per layer, one "
                       "device->host copy of the outputs, captured as a CUDA graph; one replay and one stream "
                       "sync per step")
    del st
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra:
        lshapes = wl.LLAMA31_8B_SHAPES
        extra["decode_llama31_8b_m1"] = dict(
            workload="llama-3.1-8b-decode-m1-asym-g128-fp16",
            **extra_decode(w, wl.llama31_8b_decode, lshapes, 1, l2, hbm))
        sweep = {}
        for M in (2, 3, 4, 5):
            for tag, make, shp in (("qwen3-4b", wl.qwen3_4b_decode, qshapes),
                                   ("llama-3.1-8b", wl.llama31_8b_decode, lshapes)):
                r = extra_decode(w, make, shp, M, l2, hbm)
                sweep[f"{tag} M={M}"] = {"step_us": r["step_us"], "GB/s": r["GB/s"], "frac": r["frac"],
                                         "per_shape_GB/s": {k: v["GB/s"] for k, v in r["per_shape"].items()}}
        extra["decode_m_sweep"] = sweep
        r = extra_decode(w, wl.llama31_8b_prefill, lshapes, 128, l2, hbm)
        for name, N, K in lshapes:
            r["per_shape"][name]["TFLOP/s"] = round(2 * 128 * N * K / (r["per_shape"][name]["us"] * 1e-6) / 1e12, 1)
        r["TFLOP/s"] = round(sum(2 * 128 * N * K for (_, N, K) in lshapes) / (r["step_us"] * 1e-6) / 1e12, 1)
        extra["prefill_llama31_8b_m128"] = dict(workload="llama-3.1-8b-prefill-m128-asym-g64-bf16", **r)
        extra["moe_decode"] = bench_moe(w, hbm)
        extra["moe_decode_t4"] = bench_moe(w, hbm, T=4)
        extra["decode_fused_epilogue"] = bench_fused_epilogue(w, l2, hbm)
        for Mc in (1920, 128):
            rc = bench_prefill_cache(w, Mc, max(2, args.prefill_steps))
            extra[f"prefill_dense_cache_m{Mc}"] = dict(
                workload=f"llama-3.1-8b-prefill-m{Mc}-bf16, dequantised weight cache (w4a16_gemm_dense)",
                value=round(rc["tflops"], 2), unit="TFLOP/s", ms_per_step=round(rc["ms_per_step"], 4),
                per_shape_tflops=rc["per_shape_tflops"], per_shape_us=rc["per_shape_us"],
                frac_of_burst=round(rc["tflops"] / tc, 4))

    pre = bench_prefill(w, max(2, args.prefill_steps))
    dom = int(np.argmax(pre["per_shape_ms"]))

    dec_hash = source_hash("decode.cu", "skinny.cuh", "dequant.cuh", "ptx.cuh")
    pre_hash = source_hash("prefill.cu", "dequant.cuh", "ptx.cuh")
    status = w.w4a16_last_device_error()

    if rank != 0:
        return
    cb = None
    if not args.no_cpu_baseline:
        c = cpu_baseline(sample_steps=None, budget_s=12.0)
        cb = {k: c[k] for k in ("value", "unit", "cores", "kind", "sample", "nproc")}
        cb["single_thread"] = cpu_baseline_single_thread(8.0)
    clocks = clk.summary()
    if soak is not None:
        ss = soak.summary()
        clocks["timed_region_samples"] = clocks.pop("samples")
        clocks["soak_samples"] = ss["samples"]
        clocks["soak_sm_mhz"] = ss["sm_mhz"]
        clocks["soak_reasons"] = ss["reasons"]
        clocks["reasons"] = sorted(set(clocks["reasons"]) | set(ss["reasons"]))
        if ss["sm_mhz"] is not None:
            clocks["sm_mhz"] = statistics.median(clk.samples + soak.samples)
        clocks["note"] = ("timed region shorter than 0.3 s: sm_mhz is the median over it and ~0.3 s "
                          "of the same replays right after it")
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": decode_config(ws),
        "launch": "CUDA graphs of whole steps, programmatic dependent launch; every graph replayed once before timing",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                     "frac_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": profiled_traffic("decode_qwen3_4b_m1", dec_hash),
                     "kernel": "decode_kernel (split-K skinny GEMM; all four launches)",
                     "per_launch_us": round(per_launch_s * 1e6, 3),
                     "bytes_per_launch": st_bytes_mean(qshapes)},
        "decode_median": qsum,       # per-shape and whole-step medians (null with --no-median)
        "prefill": {"workload": PREFILL_WORKLOAD, "value": round(pre["tflops"], 2), "unit": "TFLOP/s",
                    "ms_per_step": round(pre["ms_per_step"], 4),
                    "per_shape_tflops": {n: round(v, 1) for (n, _, _), v in
                                         zip(wl.LLAMA31_8B_SHAPES, pre["per_shape_tflops"])},
                    "roofline": {"bound": "tensor", "achieved": round(pre["per_shape_tflops"][dom], 2),
                                 "peak": tc, "unit": "TFLOP/s",
                                 "frac": round(pre["per_shape_tflops"][dom] / tc, 4),
                                 "peak_source": peak_src + " burst (launches of ~0.4 ms timed in short regions)",
                                 "traffic": profiled_traffic("prefill_llama_gate_up_m1920", pre_hash),
                                 "kernel": f"prefill_kernel, {wl.LLAMA31_8B_SHAPES[dom][0]}"}},
        "clocks": clocks,
        "gpu_launches": launches,
        "device_status": status,
    }
    line.update(extra)
    if e2e is not None:
        line["e2e"] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in e2e.items()}
    if cb is not None:
        line["cpu_baseline"] = cb
    print(json.dumps(line))


def st_bytes_mean(shapes):
    return int(sum(decode_bytes(1, N, K, 128, True) for (_, N, K) in shapes) / len(shapes))


if __name__ == "__main__":
    main()
