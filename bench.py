#!/usr/bin/env python3
"""Benchmark of the output-centric ("warp decode") MoE decode layer on GB300.

One step = one MoE-layer decode call (moe_gate_up + moe_down through the C
ABI) over one batch of B synthetic tokens. Default workload: the
Qwen-3-30B-A3B-shaped layer (H=2048, I=768, E=128, top-8) at B=32 decode
tokens with independent uniform routing per token -- the pages' bandwidth
headline point ("Better MoE model inference with warp decode", Key claims
[§Hardware Efficiency]: 3.95 TB/s at B=32 on B200).

L2 hygiene: two different layers' MXFP8 weights (2 x 623 MB, far above the
129 MB L2) alternate step by step, and every step uses a different batch of
tokens, so no step finds its weights in L2 (a real decode step also reads a
different layer's weights each time).

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle
instead (on the host cores, bounded sample per step). Multi-GPU: one process
per GPU via torch.distributed.run; each rank runs an independent replica on
its own batches (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

N_LAYERS = 2        # distinct weight sets alternated per step
N_BATCHES = 8       # distinct token batches cycled per step
METRIC = "MoE-layer decode tokens/s and achieved HBM GB/s (% of GB300 peak) at B=1..64"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="q30_b32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak", type=float, default=SOAK_S,
                    help="seconds of untimed steps before the warm-up, so that the clock "
                         "samples cover the load of the timed region (0: none, e.g. under ncu)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="leave out the B=1..64 sweep and accuracy keys of the contract line")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work the oracle baseline sample aims at")
    ap.add_argument("--gate-up-forms", action="store_true",
                    help="with --sweep: also time moe_gate_up and moe_gate_up_grouped alone "
                         "(CUDA graph, same rotation) for every workload")
    ap.add_argument("--down-forms", action="store_true",
                    help="with --sweep: also time moe_down and moe_down_grouped alone "
                         "(CUDA graph, same rotation) for every workload")
    ap.add_argument("--kernels-once", metavar="WORKLOAD", default=None,
                    help="for ncu: build layer 0 of WORKLOAD, then launch every gate/up and "
                         "down kernel twice on its first batch (eager), and exit")
    ap.add_argument("--sweep", nargs="*", default=None,
                    help="instead of the single contract line, print one line per workload "
                         "(default: the batch sweep of the pages' metric), timing CUDA-graph "
                         "replays of the layer")
    return ap.parse_args()


# ------------------------------------------------------------- accounting --

def expert_bytes(s) -> int:
    """MXFP8 bytes of one expert: 3*H*I E4M3 codes + 3*H*I/32 E8M0 scales."""
    return 3 * s.H * s.I + 3 * s.H * s.I // 32


def gate_up_bytes(s, ids: np.ndarray) -> int:
    """Algorithmic bytes of one moe_gate_up launch: unique touched experts'
    gate+up codes and scales, x, ids, and the BF16 intermediate written."""
    B, k = ids.shape
    U = len(np.unique(ids))
    return U * (2 * s.H * s.I + 2 * s.H * s.I // 32) + B * s.H * 2 + B * k * 4 + B * k * s.I * 2


def down_bytes(s, ids: np.ndarray) -> int:
    """Algorithmic bytes of one moe_down launch: unique touched experts' down
    codes and scales, the intermediate read, ids, weights and y written."""
    B, k = ids.shape
    U = len(np.unique(ids))
    return U * (s.H * s.I + s.H * s.I // 32) + B * k * s.I * 2 + B * k * 8 + B * s.H * 4


def layer_bytes(s, ids) -> int:
    return gate_up_bytes(s, ids) + down_bytes(s, ids)


def measured_peaks():
    p = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {
    "moe_gate_up": ["wd_device.cuh", "wd_gate_up.cuh", "wd_gate_up.cu", "wd_gate_up_fixed.cu"],
    "moe_gate_up_grouped": ["wd_device.cuh", "wd_gate_up_grouped.h", "wd_gate_up_grouped.cu"],
    "moe_down": ["wd_device.cuh", "wd_down.cu"],
    "moe_down_grouped": ["wd_device.cuh", "wd_down_grouped.h", "wd_down_grouped.cu"],
}


def kernel_source_sha(kernel: str) -> str:
    """Hash of the source files that define a kernel and its launch."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(REPO, "output_centric_expert_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic_stale(kernel: str, workload: str) -> bool:
    """Whether the committed ncu summary for the kernel and workload was taken
    on an earlier source of the kernel (so its bytes are not reported)."""
    p = os.path.join(REPO, "profiles", "traffic.json")
    if not os.path.exists(p):
        return False
    with open(p) as f:
        ent = json.load(f).get(kernel, {}).get(workload)
    return bool(ent) and ent.get("kernel_sha") != kernel_source_sha(kernel)


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(REPO, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel, {}).get(workload)
    if not ent or ent.get("kernel_sha") != kernel_source_sha(kernel):
        return None
    return ent.get("dram_bytes_per_launch"), ent.get("algorithmic_bytes_same_launches")


# ------------------------------------------------------------ multi-rank --

def max_over_ranks(v: float, world: int, device) -> float:
    """The slowest rank's time: every rank's value, reduced with MAX."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank_per_step: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest
    rank's time (replicas: every rank runs its own batches, weak scaling)."""
    return tokens_per_rank_per_step * world * steps / (max_ms / 1e3)


def rank_seed(seed: int, rank: int) -> int:
    """Each replica draws its own token batches."""
    return seed + 1000 * rank


# ----------------------------------------------------------------- clocks --

SOAK_S = 0.3  # seconds of untimed steps before the warm-up, for the clock record

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 20 ms, timestamped; started
    before the warm-up (nvidia-smi takes a moment to start) and stopped after
    the timed region. Samples whose timestamp falls inside the timed region
    (host wall clock from the first launch to the closing synchronize) are the
    ones "under load"."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except FileNotFoundError:
            self.proc = None
        time.sleep(1.0)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _epoch(ts: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(ts.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self, t0: float, t1: float, timed=None, soak_s=None):
        """Samples taken from t0 to t1 (host wall clock). timed: the timed
        region inside that window, whose own sample count is reported."""
        sm, mx, reasons, power, in_timed = [], None, set(), [], 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                clk, mxv = float(f[1]), float(f[2])
            except ValueError:
                continue
            mx = mxv
            when = self._epoch(f[0])
            if when is None or not (t0 <= when <= t1):  # outside the timed region
                continue
            sm.append(clk)
            if timed is not None and timed[0] <= when <= timed[1]:
                in_timed += 1
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        extra = {}
        if timed is not None:
            extra = {"window": f"a {soak_s:g} s soak of the same step, the warm-up and the timed "
                               "region, back to back", "samples_in_timed_region": in_timed}
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0, **extra}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None, **extra}


# ---------------------------------------------------------- workload setup --

def build_device_layers(shape, n_layers, seed, device):
    from concurrent.futures import ThreadPoolExecutor

    from output_centric_expert_gb300 import ops, workload
    sh = ops.make_shape(shape.H, shape.I, shape.E, shape.top_k)
    layers = []
    for layer in range(n_layers):
        packed = ops.empty_packed_host(sh)

        def one(e):
            g, u, d = workload.expert_weights(shape, e, seed, layer)
            ops.moe_pack_weights(sh, g[None], u[None], d[None], out=packed, expert_offset=e)

        with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(one, range(shape.E)))
        layers.append(ops.DeviceWeights(sh, packed, device))
    return layers


def make_batches(wl, n, seed):
    from output_centric_expert_gb300 import workload
    return [workload.tokens(wl.shape, wl.B, seed=seed, batch=b, routing=wl.routing) for b in range(n)]


# -------------------------------------------------------------- CPU oracle --

def oracle_baseline(wl, seconds: float, seed: int = 0):
    """Time the oracle (single-threaded FP64 C) on whole batches of the
    workload until about `seconds` of CPU work. Returns tokens/s and sample."""
    import oracle
    from output_centric_expert_gb300 import workload
    batches = make_batches(wl, 4, seed)
    need = np.unique(np.concatenate([b[1].ravel() for b in batches]))
    ref = _oracle_layer(wl.shape, seed, 0, need)
    tokens = 0
    t0 = time.perf_counter()
    i = 0
    while True:
        x, ids, w = batches[i % len(batches)]
        oracle.moe_layer(ref, x, ids, w)
        tokens += wl.B
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds or i >= 64:
            break
    return tokens / el, f"{i} batches x {wl.B} tokens of {wl.name} (layer 0), {el:.1f} s"


def oracle_baseline_all_cores(wl, seconds: float, seed: int = 0):
    """The same oracle, unchanged, on every host core: each batch's tokens are
    handed to a thread pool one token per task (the C oracle runs with the GIL
    released). Returns tokens/s, the sample and the thread count."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    cores = os.cpu_count() or 1
    batches = make_batches(wl, 4, seed)
    need = np.unique(np.concatenate([b[1].ravel() for b in batches]))
    ref = _oracle_layer(wl.shape, seed, 0, need)
    # one call before any thread starts: the oracle fills its decode tables on
    # first use, and thread creation orders that before every worker's reads
    x, ids, w = batches[0]
    oracle.moe_layer(ref, x[:1], ids[:1], w[:1])
    tokens, i = 0, 0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        while True:
            x, ids, w = batches[i % len(batches)]
            list(ex.map(lambda t: oracle.moe_layer(ref, x[t:t + 1], ids[t:t + 1], w[t:t + 1]),
                        range(wl.B)))
            tokens += wl.B
            i += 1
            el = time.perf_counter() - t0
            if el >= seconds or i >= 256:
                break
    return tokens / el, f"{i} batches x {wl.B} tokens of {wl.name} (layer 0), {el:.1f} s", cores


def _oracle_layer(shape, seed, layer, experts):
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from output_centric_expert_gb300 import workload
    E, I, H = shape.E, shape.I, shape.H
    gc = np.zeros((E, I, H), np.uint8)
    gs = np.zeros((E, I, H // 32), np.uint8)
    uc, us = np.zeros_like(gc), np.zeros_like(gs)
    dc = np.zeros((E, H, I), np.uint8)
    ds = np.zeros((E, H, I // 32), np.uint8)

    def one(e):
        g, u, d = workload.expert_weights(shape, int(e), seed, layer)
        gc[e], gs[e] = oracle.quantize_mxfp8(g)
        uc[e], us[e] = oracle.quantize_mxfp8(u)
        dc[e], ds[e] = oracle.quantize_mxfp8(d)

    with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(one, experts))
    return oracle.QuantizedLayer(gc, gs, uc, us, dc, ds)


def run_reference(args, wl, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle
    per_step_tokens = max(1, min(wl.B, 2))  # bounded sample of each step's batch
    batches = make_batches(wl, N_BATCHES, 0)
    need = np.unique(np.concatenate([b[1][:per_step_tokens].ravel() for b in batches]))
    ref = _oracle_layer(wl.shape, 0, 0, need)
    for s in range(args.warmup):
        x, ids, w = batches[s % N_BATCHES]
        oracle.moe_layer(ref, x[:per_step_tokens], ids[:per_step_tokens], w[:per_step_tokens])
    t0 = time.perf_counter()
    for s in range(args.steps):
        x, ids, w = batches[s % N_BATCHES]
        oracle.moe_layer(ref, x[:per_step_tokens], ids[:per_step_tokens], w[:per_step_tokens])
    el = time.perf_counter() - t0
    value = per_step_tokens * args.steps / el
    sample = f"{per_step_tokens} of the {wl.B} tokens of each step's batch"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "H": wl.shape.H, "I": wl.shape.I, "E": wl.shape.E,
                   "top_k": wl.shape.top_k, "B": wl.B, "routing": wl.routing},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ GPU arm --

def run_ours(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from output_centric_expert_gb300 import ops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    s = wl.shape
    seed = 0
    layers = build_device_layers(s, N_LAYERS, seed, dev)
    batches = make_batches(wl, N_BATCHES, rank_seed(seed, rank))
    dx = [torch.from_numpy(b[0].view(np.int16)).to(dev) for b in batches]
    dids = [torch.from_numpy(b[1]).to(dev) for b in batches]
    dw = [torch.from_numpy(b[2]).to(dev) for b in batches]
    h = torch.empty((wl.B, s.top_k, s.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.B, s.H), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def eager_step(i, st=None):
        b = i % N_BATCHES
        ops.moe_layer(layers[i % N_LAYERS], dx[b], dids[b], dw[b], h, y, err, st)

    # The steps run as CUDA graphs of moe_layer calls through the C ABI,
    # captured once, so that the host's launch work stays out of the GPU's way
    # as in a graph-driven decode loop: one graph per (layer, batch) for the
    # soak, the warm-up and the per-step times, and graphs of many steps for
    # the timed region.
    rot = math.lcm(N_LAYERS, N_BATCHES)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(rot):  # first calls outside capture
            eager_step(i)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    graphs = []
    for i in range(rot):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            eager_step(i)
        graphs.append(g)

    def step(i):
        graphs[i % rot].replay()

    # the timed region: K steps as replays of a graph of `chunk` consecutive
    # steps (a multiple of the rotation) and one graph of the remainder
    chunk = min(args.steps - args.steps % rot, 64 * rot) if args.steps >= rot else 0
    def multi_step_graph(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                eager_step(i)
        return g
    g_chunk = multi_step_graph(chunk) if chunk else None
    n_chunks = args.steps // chunk if chunk else 0
    rem = args.steps - n_chunks * chunk
    g_rem = multi_step_graph(rem) if rem else None

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local_rank)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        # A soak of the same step right before the warm-up and the timed region:
        # K steps take a few ms, shorter than the sampler's period, so the
        # clock record covers the soak and the timed region together.
        soak0 = time.time()
        i = 0
        while time.time() - soak0 < args.soak:
            for _ in range(64):
                step(i)
                i += 1
            torch.cuda.synchronize(dev)
        for i in range(max(3, args.warmup)):
            step(i)
        barrier()
        # ---- main timed region: K whole-layer steps ----------------------
        barrier()
        wall0 = time.time()
        ev0.record(stream)
        for _ in range(n_chunks):
            g_chunk.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
        barrier()
        wall1 = time.time()
    el_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    # per-step times: the same K steps again, one graph replay each with an
    # event between them (a replay per step adds its own launch gap)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    step_ev[0].record(stream)
    for i in range(args.steps):
        step(i)
        step_ev[i + 1].record(stream)
    barrier()
    step_ms = sorted(step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps))
    ms_per_step = el_ms / args.steps
    value = job_tokens_per_s(wl.B, world, args.steps, el_ms)
    if int(err.item()) != 0:
        raise RuntimeError("device error flag set: an expert id was out of range")

    # ---- per-kernel durations (same steps, an event between the kernels) --
    # the gate/up kernel the layer itself runs at this shape and batch
    gu_form = ops.layer_gate_up_kernel(layers[0].shape, wl.B, layers[0])
    gu_kernel = "moe_gate_up_grouped" if gu_form == "grouped" else "moe_gate_up"
    gate_up_fn = getattr(ops, gu_kernel)
    # and the down kernel it runs
    dn_kernel = ("moe_down_grouped" if ops.layer_down_kernel(layers[0].shape, wl.B, layers[0])
                 == "grouped" else "moe_down")
    down_fn = getattr(ops, dn_kernel)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        b = i % N_BATCHES
        L = layers[i % N_LAYERS]
        evs[i][0].record(stream)
        gate_up_fn(L, dx[b], dids[b], h, err, stream)
        evs[i][1].record(stream)
        down_fn(L, h, dids[b], dw[b], y, err, stream)
        evs[i][2].record(stream)
    barrier()
    gu_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    gu_bytes = [gate_up_bytes(s, batches[i % N_BATCHES][1]) for i in range(args.steps)]
    dn_bytes = [down_bytes(s, batches[i % N_BATCHES][1]) for i in range(args.steps)]
    lay_bytes = [a + b for a, b in zip(gu_bytes, dn_bytes)]
    peak, peak_kind = measured_peaks()
    gu_gbs = sum(gu_bytes) / (sum(gu_ms) / 1e3) / 1e9
    dn_gbs = sum(dn_bytes) / (sum(dn_ms) / 1e3) / 1e9
    layer_gbs = sum(lay_bytes) / args.steps / (ms_per_step / 1e3) / 1e9

    # ---- end to end from pinned host buffers (copies inside the region) ----
    # Every step copies its x, ids and routing weights in from pinned host
    # memory and its y back out, through moe_layer_host. value: one stream,
    # so each step's copies and kernels run in series. pipelined: two streams
    # take alternate steps with their own buffers, so one step's copies (and
    # kernels) overlap the other's, as a serving loop with two requests in
    # flight would run.
    px = [torch.from_numpy(b[0].view(np.int16)).pin_memory() for b in batches]
    pids = [torch.from_numpy(b[1]).pin_memory() for b in batches]
    pw = [torch.from_numpy(b[2]).pin_memory() for b in batches]
    e2e_streams = [stream, torch.cuda.Stream(device=dev)]
    e2e_bufs = [{"py": torch.empty((wl.B, s.H), dtype=torch.float32).pin_memory(),
                 "sx": torch.empty_like(dx[0]), "sids": torch.empty_like(dids[0]),
                 "sw": torch.empty_like(dw[0]), "h": torch.empty_like(h), "y": torch.empty_like(y)}
                for _ in e2e_streams]

    def e2e_step(i, nstreams):
        b, k = i % N_BATCHES, i % nstreams
        q = e2e_bufs[k]
        ops.moe_layer_host(layers[i % N_LAYERS], px[b], pids[b], pw[b], q["sx"], q["sids"], q["sw"],
                           q["h"], q["y"], q["py"], err, e2e_streams[k])

    def e2e_run(nstreams):
        for i in range(4):
            e2e_step(i, nstreams)
        barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(e2e_streams[0])
        for k in range(1, nstreams):
            e2e_streams[k].wait_event(t0)
        for i in range(args.steps):
            e2e_step(i, nstreams)
        for k in range(1, nstreams):
            done = torch.cuda.Event()
            done.record(e2e_streams[k])
            e2e_streams[0].wait_event(done)
        t1.record(e2e_streams[0])
        barrier()
        return t0, t1

    p0, p1 = e2e_run(2)
    e2e_pipe_ms = max_over_ranks(p0.elapsed_time(p1), world, dev)
    e0, e1 = e2e_run(1)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = job_tokens_per_s(wl.B, world, args.steps, e2e_ms)
    h2d = px[0].numel() * 2 + pids[0].numel() * 4 + pw[0].numel() * 4
    d2h = e2e_bufs[0]["py"].numel() * 4

    if rank != 0:
        return
    cpu = cpu_all = None
    if not args.no_cpu_baseline:
        v, sample = oracle_baseline(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}
        v, sample, cores = oracle_baseline_all_cores(wl, args.cpu_seconds)
        cpu_all = {"value": v, "unit": "tokens/s", "cores": cores,
                   "kind": "oracle, one token per thread", "sample": sample}
    sweep = acc = None
    if not args.no_sweep:
        sweep, acc = metric_sweep(layers, dev, peak)
    traffic, traffic_alg = ncu_traffic(gu_kernel, wl.name) or (None, None)
    gu_launch_bytes = sum(gu_bytes) / args.steps
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "H": s.H, "I": s.I, "E": s.E, "top_k": s.top_k,
                   "B": wl.B, "routing": wl.routing, "parallelism": f"replicas x{world}",
                   "formats": "MXFP8 (E4M3 + E8M0/32) weights, BF16 x and h, FP32 accumulators and y",
                   "l2": f"inputs larger than L2: {N_LAYERS} layers' weights "
                         f"({N_LAYERS * layers[0].nbytes / 1e9:.2f} GB) alternate per step, "
                         f"{N_BATCHES} token batches cycle",
                   "launch": "the K timed steps replay CUDA graphs of consecutive moe_layer "
                             "calls (C ABI), captured once",
                   "layer_gbs": layer_gbs, "layer_frac_of_peak": layer_gbs / peak,
                   # the pages' one absolute figure for this layer and batch, measured on
                   # B200 (context, not a target): 3.95 TB/s effective bandwidth at B=32
                   "pages_b200_gbs_b32": 3950.0 if (wl.shape.H, wl.shape.I, wl.B) == (2048, 768, 32) else None,
                   "layer_bytes_per_step": sum(lay_bytes) / args.steps,
                   "gate_up_us": sum(gu_ms) / args.steps * 1e3,
                   "down_us": sum(dn_ms) / args.steps * 1e3,
                   "down_gbs": dn_gbs, "down_frac_of_peak": dn_gbs / peak,
                   "down_kernel": dn_kernel},
        "roofline": {"bound": "hbm", "kernel": gu_kernel, "achieved": gu_gbs, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": gu_gbs / peak,
                     "algorithmic_bytes_per_launch": gu_launch_bytes,
                     "traffic": traffic,
                     "traffic_note": (
                         f"mean of the ncu-captured launches, whose own algorithmic bytes average "
                         f"{traffic_alg} (ratio {traffic / traffic_alg:.4f}); profiles/traffic.json"
                         if traffic is not None else
                         "the capture in profiles/traffic.json was taken on an earlier source of "
                         "this kernel, so it is not reported"
                         if ncu_traffic_stale(gu_kernel, wl.name) else None)},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "api": "moe_layer_host, one stream",
                "pipelined": {"value": job_tokens_per_s(wl.B, world, args.steps, e2e_pipe_ms),
                              "unit": "tokens/s",
                              "how": "moe_layer_host on 2 streams taking alternate steps; one "
                                     "step's copies and kernels overlap the other's"}},
        "step_ms": {"median": statistics.median(step_ms), "p90": step_ms[int(0.9 * (len(step_ms) - 1))],
                    "min": step_ms[0], "max": step_ms[-1], "how": "CUDA events between the same K steps replayed one graph per step after the timed region"},
        "sweep": sweep,
        "accuracy": acc,
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(soak0, wall1, timed=(wall0, wall1), soak_s=args.soak),
    }
    print(json.dumps(out), flush=True)


def graph_layer_us(layers, dx, dids, dw, h, y, reps: int) -> float:
    """moe_layer captured in one CUDA graph over a rotation of the layers and
    token batches (step i: layer i % len(layers), batch i % len(dx)), replayed
    `reps` times; CUDA-event microseconds per step. Launch overhead of the host
    is outside the measurement, as in a graph-driven decode loop."""
    import torch

    from output_centric_expert_gb300 import ops
    dev = dx[0].device
    rot = 2 * len(dx)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for i in range(rot):  # warm-up outside capture
            ops.moe_layer(layers[i % len(layers)], dx[i % len(dx)], dids[i % len(dx)],
                          dw[i % len(dx)], h, y)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(rot):
            ops.moe_layer(layers[i % len(layers)], dx[i % len(dx)], dids[i % len(dx)],
                          dw[i % len(dx)], h, y)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / (reps * rot)


# The pages' metric covers B=1..64 ("Better MoE model inference with warp
# decode", [§Hardware Efficiency]: accuracy "across all batch sizes"); the
# default run times every point of the batch sweep and the larger layer, and
# checks each against the oracle.
METRIC_SWEEP = ([("q30", B, r) for r in ("uniform", "skewed") for B in (1, 2, 4, 8, 16, 32, 64)]
                + [("q235", B, "uniform") for B in (1, 16, 64)])
ACCURACY_TOKENS = {"q30": 4, "q235": 2}  # oracle tokens per point (first, last, evenly between)


def metric_sweep(q30_layers, dev, peak, reps: int = 6):
    """Every point of METRIC_SWEEP: the layer's time (graph_layer_us over 8
    token batches and the layers given: the bench's two Qwen-3-30B-A3B-shaped
    layers, one Qwen-3-235B-A22B-shaped layer of 2.5 GB, both far above L2), and
    the achieved max |y - y_oracle| and minimum per-token cosine on sampled
    tokens of the point's first batch. The oracle runs on the host cores, one
    token per thread. Returns (sweep, accuracy) dicts for the JSON line."""
    from concurrent.futures import ThreadPoolExecutor

    import torch

    import oracle
    from output_centric_expert_gb300 import ops, workload
    t_start = time.time()
    points, checks = [], []
    oracle_jobs = []
    for name in ("q30", "q235"):
        s = workload.SHAPES[name]
        if name == "q30":
            layers = q30_layers
        else:
            torch.cuda.empty_cache()
            layers = build_device_layers(s, 1, 0, dev)
        todo = [(B, r) for (n, B, r) in METRIC_SWEEP if n == name]
        all_batches = {}
        need = set()
        for B, r in todo:
            wl = workload.Workload(f"{name}_{r}_b{B}", s, B, r)
            bs = make_batches(wl, N_BATCHES, 0)
            all_batches[(B, r)] = (wl, bs)
            smp = sorted(set(np.linspace(0, B - 1, min(B, ACCURACY_TOKENS[name])).round().astype(int)))
            need |= set(bs[0][1][smp].ravel().tolist())
        ref = _oracle_layer(s, 0, 0, sorted(need))
        for B, r in todo:
            wl, bs = all_batches[(B, r)]
            dx = [torch.from_numpy(b[0].view(np.int16)).to(dev) for b in bs]
            dids = [torch.from_numpy(b[1]).to(dev) for b in bs]
            dw = [torch.from_numpy(b[2]).to(dev) for b in bs]
            h = torch.empty((B, s.top_k, s.I), dtype=torch.int16, device=dev)
            y = torch.empty((B, s.H), dtype=torch.float32, device=dev)
            us = graph_layer_us(layers, dx, dids, dw, h, y, reps)
            lay_bytes = float(np.mean([layer_bytes(s, b[1]) for b in bs]))
            points.append({"workload": wl.name, "B": B, "routing": r, "us": round(us, 2),
                           "tokens_per_s": round(B / us * 1e6),
                           "gbs": round(lay_bytes / us / 1e3, 1),
                           "frac_of_peak": round(lay_bytes / us / 1e3 / peak, 4),
                           "unique_experts": float(np.mean([len(np.unique(b[1])) for b in bs])),
                           "gate_up_kernel": ops.layer_gate_up_kernel(layers[0].shape, B, layers[0]),
                           "down_kernel": ops.layer_down_kernel(layers[0].shape, B, layers[0])})
            # accuracy: the first batch once more, eagerly, against the oracle
            ops.moe_layer(layers[0], dx[0], dids[0], dw[0], h, y)
            torch.cuda.synchronize(dev)
            yg = y.cpu().numpy().astype(np.float64)
            x, ids, w = bs[0]
            smp = sorted(set(np.linspace(0, B - 1, min(B, ACCURACY_TOKENS[name])).round().astype(int)))
            for t in smp:
                oracle_jobs.append((wl.name, t, yg[t], ref, x[t:t + 1], ids[t:t + 1], w[t:t + 1]))
        del layers
    # one call before any thread starts: the oracle fills its decode tables on
    # first use, and thread creation orders that before every worker's reads
    _, _, _, ref0, x0, ids0, w0 = oracle_jobs[0]
    oracle.moe_layer(ref0, x0, ids0, w0)

    def one(job):
        name, t, yt, ref, x, ids, w = job
        yo, _ = oracle.moe_layer(ref, x, ids, w)
        yo = yo[0]
        d = float(np.max(np.abs(yt - yo)))
        cos = float(np.dot(yt, yo) / (np.linalg.norm(yt) * np.linalg.norm(yo)))
        return name, d, cos
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        res = list(ex.map(one, oracle_jobs))
    per = {}
    for name, d, cos in res:
        a = per.setdefault(name, {"workload": name, "tokens": 0, "max_abs": 0.0, "min_cos": 1.0})
        a["tokens"] += 1
        a["max_abs"] = max(a["max_abs"], d)
        a["min_cos"] = min(a["min_cos"], cos)
    checks = list(per.values())
    sweep = {"timing": f"CUDA graph of 16 steps over 8 token batches and the layers (Q30: 2 layers, "
                       f"Q235: 1 layer of 2.5 GB), replayed {reps} times; cold L2",
             "peak_gbs": peak, "points": points}
    acc = {"vs": "FP64 CPU oracle on the same packed weights",
           "points": checks, "max_abs": max(c["max_abs"] for c in checks),
           "min_cos": min(c["min_cos"] for c in checks),
           "bar": {"max_abs": 4e-3, "min_cos": 0.99999},
           "pages_b200_context": {"max_abs": 0.001953, "min_cos": 0.999996},
           "seconds": round(time.time() - t_start, 1)}
    return sweep, acc


SWEEP_DEFAULT = ([f"q30_{r}_b{b}" for r in ("uniform", "skewed") for b in (1, 2, 4, 8, 16, 32, 64)]
                 + ["q235_b1", "q235_b16", "q235_b64", "tiny_b1"])
SWEEP_VARIANTS = ["dsv3_b1", "dsv3_b16", "dsv3_b64", "mixtral_b1", "mixtral_b16", "mixtral_b64"]


def run_sweep(names, steps: int, gate_up_forms: bool = False, down_forms: bool = False):
    """Per workload: the layer (moe_layer, both kernels) captured in a CUDA graph
    over a rotation of 2 layers x 8 token batches, replayed; CUDA-event time per
    step. Launch overhead of the host is outside the measurement, as in a
    graph-driven decode loop."""
    import torch

    from output_centric_expert_gb300 import ops, workload
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, _ = measured_peaks()
    built = {}
    for name in names:
        wl = workload.WORKLOADS[name]
        s = wl.shape
        key = (s.H, s.I, s.E, s.top_k)
        if key not in built:
            built.clear()
            torch.cuda.empty_cache()
            built[key] = build_device_layers(s, N_LAYERS, 0, dev)
        layers = built[key]
        batches = make_batches(wl, N_BATCHES, 0)
        dx = [torch.from_numpy(b[0].view(np.int16)).to(dev) for b in batches]
        dids = [torch.from_numpy(b[1]).to(dev) for b in batches]
        dw = [torch.from_numpy(b[2]).to(dev) for b in batches]
        h = torch.empty((wl.B, s.top_k, s.I), dtype=torch.int16, device=dev)
        y = torch.empty((wl.B, s.H), dtype=torch.float32, device=dev)
        rot = 2 * N_BATCHES  # steps per graph replay
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for i in range(rot):  # warm-up outside capture
                ops.moe_layer(layers[i % N_LAYERS], dx[i % N_BATCHES], dids[i % N_BATCHES],
                              dw[i % N_BATCHES], h, y)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(rot):
                ops.moe_layer(layers[i % N_LAYERS], dx[i % N_BATCHES], dids[i % N_BATCHES],
                              dw[i % N_BATCHES], h, y)
        reps = max(3, steps // rot)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / (reps * rot)
        # warm L2: the same layer and batch every step (the weights stay in L2
        # when they fit in it, 129 MB)
        gw = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gw):
            for i in range(rot):
                ops.moe_layer(layers[0], dx[0], dids[0], dw[0], h, y)
        for _ in range(2):
            gw.replay()
        torch.cuda.synchronize(dev)
        e0.record()
        for _ in range(reps):
            gw.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        warm_us = e0.elapsed_time(e1) * 1e3 / (reps * rot)
        lay_bytes = float(np.mean([layer_bytes(s, b[1]) for b in batches]))
        uniq = float(np.mean([len(np.unique(b[1])) for b in batches]))
        forms = {}
        if gate_up_forms:
            # each gate/up kernel alone over the same rotation; GB/s of its own bytes
            gu_b = float(np.mean([gate_up_bytes(s, b[1]) for b in batches]))
            for form, fn in (("per_token", ops.moe_gate_up), ("grouped", ops.moe_gate_up_grouped)):
                if form == "grouped" and not (s.H % 256 == 0 and s.I % 64 == 0):
                    continue
                gf = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gf):
                    for i in range(rot):
                        fn(layers[i % N_LAYERS], dx[i % N_BATCHES], dids[i % N_BATCHES], h)
                for _ in range(2):
                    gf.replay()
                torch.cuda.synchronize(dev)
                e0.record()
                for _ in range(reps):
                    gf.replay()
                e1.record()
                torch.cuda.synchronize(dev)
                f_us = e0.elapsed_time(e1) * 1e3 / (reps * rot)
                forms[form] = {"us": round(f_us, 2), "gbs": round(gu_b / f_us / 1e3, 1)}
        down = {}
        if down_forms:
            # each down kernel alone over the same rotation, fed each batch's
            # intermediate; GB/s of its own bytes
            hs = []
            for b in range(N_BATCHES):
                hb = torch.empty_like(h)
                ops.moe_gate_up(layers[0], dx[b], dids[b], hb)
                hs.append(hb)
            dn_b = float(np.mean([down_bytes(s, b[1]) for b in batches]))
            for form, fn in (("per_token", ops.moe_down), ("grouped", ops.moe_down_grouped)):
                try:  # the grouped kernel refuses some shapes and batches
                    fn(layers[0], hs[0], dids[0], dw[0], y)
                except ops.WarpDecodeError:
                    continue
                torch.cuda.synchronize(dev)
                gf = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gf):
                    for i in range(rot):
                        fn(layers[i % N_LAYERS], hs[i % N_BATCHES], dids[i % N_BATCHES],
                           dw[i % N_BATCHES], y)
                for _ in range(2):
                    gf.replay()
                torch.cuda.synchronize(dev)
                e0.record()
                for _ in range(reps):
                    gf.replay()
                e1.record()
                torch.cuda.synchronize(dev)
                f_us = e0.elapsed_time(e1) * 1e3 / (reps * rot)
                down[form] = {"us": round(f_us, 2), "gbs": round(dn_b / f_us / 1e3, 1),
                              "frac_of_measured_peak": round(dn_b / f_us / 1e3 / peak, 4)}
        print(json.dumps({"workload": name, "H": s.H, "I": s.I, "E": s.E, "top_k": s.top_k,
                          "B": wl.B, "routing": wl.routing,
                          "gate_up_kernel": ops.layer_gate_up_kernel(layers[0].shape, wl.B, layers[0]),
                          "down_kernel": ops.layer_down_kernel(layers[0].shape, wl.B, layers[0]),
                          "us_per_layer": round(us, 2),
                          "tokens_per_s": round(wl.B / us * 1e6), "unique_experts": uniq,
                          "layer_bytes": lay_bytes, "layer_gbs": round(lay_bytes / us / 1e3, 1),
                          "frac_of_measured_peak": round(lay_bytes / us / 1e3 / peak, 4),
                          "timing": "CUDA graph of 16 steps (2 layers x 8 batches), replayed",
                          "warm_l2_us_per_layer": round(warm_us, 2),
                          "warm_l2_bytes_per_layer": layer_bytes(s, batches[0][1]),
                          **({"gate_up_alone": forms} if gate_up_forms else {}),
                          **({"down_alone": down} if down_forms else {})}),
              flush=True)


def run_kernels_once(name: str):
    """Each kernel of the layer, launched twice on the first token batch of a
    workload (layer 0 of the bench's weights): moe_gate_up, moe_gate_up_grouped,
    moe_down, moe_down_grouped (the grouped ones where they take the shape and
    batch). A target for ncu captures of one kernel (-k regex:<name> -s 1 -c 1)."""
    import torch

    from output_centric_expert_gb300 import ops, workload
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = workload.WORKLOADS[name]
    s = wl.shape
    L = build_device_layers(s, 1, 0, dev)[0]
    x, ids, w = make_batches(wl, 1, 0)[0]
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    idd = torch.from_numpy(ids).to(dev)
    wd = torch.from_numpy(w).to(dev)
    h = torch.empty((wl.B, s.top_k, s.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.B, s.H), dtype=torch.float32, device=dev)
    ran = []
    for kname, fn, args in (("moe_gate_up", ops.moe_gate_up, (L, xd, idd, h)),
                            ("moe_gate_up_grouped", ops.moe_gate_up_grouped, (L, xd, idd, h)),
                            ("moe_down", ops.moe_down, (L, h, idd, wd, y)),
                            ("moe_down_grouped", ops.moe_down_grouped, (L, h, idd, wd, y))):
        try:
            for _ in range(2):
                fn(*args)
            ran.append(kname)
        except ops.WarpDecodeError:
            pass
    torch.cuda.synchronize(dev)
    print(json.dumps({"kernels_once": name, "launched_twice": ran}), flush=True)


def main():
    args = parse()
    if args.kernels_once is not None:
        run_kernels_once(args.kernels_once)
        return
    if args.sweep is not None:
        run_sweep(args.sweep or SWEEP_DEFAULT, args.steps, args.gate_up_forms, args.down_forms)
        return
    from output_centric_expert_gb300 import workload
    wl = workload.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            raise SystemExit("--gpus N > 1 needs torch.distributed.run with N processes")
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
