#!/usr/bin/env python3
"""Benchmark of the MSA fused producer on GB300; prints one JSON line.

Default workload: the prefill batch, 8 sequences x 8,192 tokens (65,536 tokens),
64 Q / 8 K-V / 8 index-Q / 1 index-K heads of dim 128, fp8 E4M3 HND caches with a
shuffled page table.  One step = one producer launch over the whole batch (all
steps of the path: placement, RMSNorm, RoPE, compact Q/index-Q, three cache
scatters).  The rows read per step (1.49 GB) are far larger than L2, so no flush
is needed between steps.

Also reported: the 60-layer decode step at batch 256 (tiny shapes, one launch per
layer, all 60 captured in one CUDA graph; microseconds per layer and per step),
the decode indexer, the projection GEMM with the producer in its epilogue
(hidden 6,144 -> 11,392 outputs on the tcgen05 tensor cores, against the measured
cuBLAS bf16 peak and against cuBLAS GEMM + producer),
an end-to-end figure through the same C-ABI call with pinned host buffers and the
host<->device copies inside the timed region, the roofline of the producer kernel
against the measured HBM copy bandwidth, and the CPU oracle timed on a bounded
sample of the same workload on this machine's host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (under torchrun) every rank runs its own replica of the workload
(tokens are independent; there is no exchange step), and value = tokens of all
ranks / the slowest rank's time.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "producer tokens/s & HBM GB/s (% of peak); us/layer at decode batch 256"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCE = os.path.join(ROOT, "paged_kv_cache_msa_gb300", "csrc", "msa_producer.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash() -> str:
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(workload: str):
    """dram bytes per launch from a committed ncu capture of this exact kernel
    source (None when the kernel has changed since)."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_sha") == kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline / reference arm)
# ---------------------------------------------------------------------------

class OracleRunner:
    """The CPU oracle over a workload, with its host pools prepared once so that
    only the oracle's own work is timed."""

    def __init__(self, w):
        import oracle
        from paged_kv_cache_msa_gb300 import workloads as wl
        oracle.build()
        self.oracle = oracle
        self.w = w
        self.pools = wl.host_pools(w)
        self.ca = wl.oracle_cache_args(w, self.pools)
        self.q, self.iq = wl.empty_outputs(w)
        self.next = 0

    def run(self, n: int) -> int:
        """Runs the next n tokens (wrapping around); returns the tokens done."""
        w = self.w
        if self.next >= w.num_tokens:
            self.next = 0
        n = min(n, w.num_tokens - self.next)
        self.oracle.forward(w.shape, w.qkv, w.row_stride, w.positions, w.slot_mapping,
                            w.page_table, w.weights, self.q, self.iq, self.ca["k"], self.ca["v"],
                            self.ca["idx_k"], w.scales, num_tokens=n, token_offset=self.next)
        self.next += n
        return n

    def timed(self, budget_s: float, chunk: int = 256):
        """Consecutive chunks until the budget is spent; returns (tokens, seconds)."""
        done, t0 = 0, time.perf_counter()
        while True:
            done += self.run(chunk)
            if time.perf_counter() - t0 >= budget_s or done >= self.w.num_tokens:
                break
        return done, time.perf_counter() - t0


def make_workload(name: str, prefill_seqs: int = 8):
    from paged_kv_cache_msa_gb300 import workloads as wl
    if name == "prefill":
        return wl.config4_prefill(num_seqs=prefill_seqs)
    if name == "decode64":
        return wl.config2_decode64()
    if name == "mixed":
        return wl.config5_mixed()
    if name == "tiny":
        return wl.config1_tiny_decode()
    raise ValueError(name)


WORKLOAD_DESC = {
    "prefill": "prefill 8x8192 = 65,536 tokens; Q64/KV8/idxQ8/idxK1 heads, head_dim 128, "
               "rotary 128 NeoX; fp8 E4M3 K/V/idx-K HND caches, page 64, shuffled table",
    "decode64": "decode batch 64; big shapes; padded HND fp8 pages; 10% padded slots",
    "mixed": "mixed 4x2048 prefill + 192 decode; rotary 64/128; strided rows; pool > 2^31 elements",
    "tiny": "tiny decode batch 4",
}


def host_cpu() -> dict:
    """The host the oracle runs on: its core count (the oracle itself uses one) and
    CPU model, as lscpu or /proc/cpuinfo report them."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() in ("Model name", "Vendor ID") and v.strip() and model is None:
                model = v.strip()
            if k.strip() == "Model name" and v.strip():
                model = v.strip()
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return {"host_cores": os.cpu_count(), "cpu_model": model, "threads_used": 1}


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    w = make_workload(args.workload, args.prefill_seqs)
    runner = OracleRunner(w)
    cores = 1
    sample = 64
    for _ in range(args.warmup):
        runner.run(sample)
    t0 = time.perf_counter()
    tok = 0
    for _ in range(args.steps):
        tok += runner.run(sample)
    el = time.perf_counter() - t0
    value = tok / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "tokens_per_step": sample,
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} consecutive tokens of the workload per step "
                                   f"(cycling through it), single-threaded C oracle",
                         **host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def decode_step_timing(replays: int, big: bool, pdl: bool):
    """60 decode layers at batch 256 captured as 60 launches in one CUDA graph."""
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import workloads as wl
    from paged_kv_cache_msa_gb300.device import DeviceWorkload
    layers = [DeviceWorkload(wl.config3_decode_step(l, big=big)) for l in range(60)]
    flags = B.MSA_LAUNCH_PERSISTENT | (B.MSA_LAUNCH_PDL if pdl else 0)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for dw in layers:
            dw.run(flags, stream=s)
    with torch.cuda.stream(s):
        for _ in range(20):
            g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(replays):
            g.replay()
        e1.record(s)
        e1.synchronize()
    us_step = 1e3 * e0.elapsed_time(e1) / replays
    tokens = layers[0].w.num_tokens
    nodes = graph_kernel_nodes(lambda: [dw.run(flags, stream=s) for dw in layers], s)
    del g, layers
    torch.cuda.empty_cache()
    return {"us_per_step": us_step, "us_per_layer": us_step / 60, "layers": 60,
            "tokens_per_layer": tokens, "launches_per_step": 60, "kernel_nodes_in_graph": nodes,
            "shapes": "big" if big else "tiny", "pdl": pdl, "replays": replays}


def empty_graph_floor(nodes: int = 60, replays: int = 1000):
    """The launch floor of a CUDA graph of ``nodes`` kernel nodes that do next to
    nothing (a 4-byte fill each): microseconds per replay and per node."""
    import torch
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(nodes):
            t.fill_(1)
    with torch.cuda.stream(s):
        for _ in range(20):
            g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(replays):
            g.replay()
        e1.record(s)
        e1.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / replays
    return {"nodes": nodes, "us_per_graph": us, "us_per_node": us / nodes,
            "what": "a graph of 4-byte fill kernels, the cost of a launch inside a graph"}


def graph_kernel_nodes(fn, stream):
    """Kernel nodes of a CUDA graph captured from fn() on `stream`: the number of
    kernels fn launches (counted through the driver's graph API), or None."""
    import ctypes
    import torch
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
        with torch.cuda.graph(g, stream=stream):
            fn()
        h = ctypes.c_void_p(g.raw_cuda_graph())
        cu = ctypes.CDLL("libcuda.so.1")
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(h, None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * max(1, n.value))()
        if cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) != 0:
            return None
        kernels, t = 0, ctypes.c_int(-1)
        for i in range(n.value):
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0 and t.value == 0:
                kernels += 1   # CU_GRAPH_NODE_TYPE_KERNEL
        del g
        return kernels
    except Exception as e:   # context only
        log(f"[bench] kernel count unavailable: {type(e).__name__}: {e}"[:160])
        return None


def legacy_write_path_timing(replays: int = 200, layers: int = 60):
    """The write path the fused producer replaces, as the pages describe it: per
    cache a division kernel (page), a remainder kernel (in-page offset), an index
    cast and an index_put scatter into the paged HND cache -- 12 launches per layer
    for K, V and index-K -- in PyTorch eager ops on the GPU, ``layers`` layers of the
    decode step (batch 256, tiny shapes, each layer its own caches, physical slots)
    captured in one CUDA graph.  The values are taken as already encoded (fp8 K/V,
    bf16 index-K); the fused producer's 60 launches do the norm, RoPE, compact Q /
    index-Q and encoding as well."""
    import torch
    from paged_kv_cache_msa_gb300 import workloads as wl
    dev = torch.device("cuda")
    g_rng = torch.Generator(device=dev)
    g_rng.manual_seed(11)
    stack = []
    for l in range(layers):
        w = wl.config3_decode_step(l)
        s_, T = w.shape, w.num_tokens
        D, P = s_["head_dim"], s_["page_size"]
        pt = w.page_table.reshape(-1).astype(np.int64)
        # the physical slots the producer's table lookup gives (legacy callers pass these)
        blk = w.slot_mapping // P
        phys = np.where(w.slot_mapping >= 0, pt[np.clip(blk, 0, pt.size - 1)] * P + w.slot_mapping % P, -1)
        assert (phys >= 0).all(), "the decode-step workload has no padded slots"
        caches = []
        for key in ("k", "v", "idx_k"):
            c = w.caches[key]
            es = c.elem_size()
            dt = torch.uint8 if es == 1 else torch.int16
            pool = torch.zeros(c.num_pages * c.num_heads * P * D, dtype=dt, device=dev)
            view = pool.view(c.num_pages, c.num_heads, P, D).permute(0, 2, 1, 3)   # [pages, P, H, D]
            vals = torch.randint(0, 120, (T, c.num_heads, D), generator=g_rng, device=dev).to(dt)
            caches.append((view, vals))
        stack.append((torch.from_numpy(phys.astype(np.int32)).to(dev), P, caches))

    def layer(slot32, P, caches):
        for view, vals in caches:
            page = torch.div(slot32, P, rounding_mode="floor")      # division
            off = torch.remainder(slot32, P)                         # remainder
            page64 = page.long()                                     # index cast
            view.index_put_((page64, off), vals)                     # scatter
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for item in stack:
            layer(*item)
        s.synchronize()
        kernels = graph_kernel_nodes(lambda: layer(*stack[0]), s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for item in stack:
                layer(*item)
        for _ in range(10):
            g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(replays):
            g.replay()
        e1.record(s)
        e1.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / replays
    del g, stack
    torch.cuda.empty_cache()
    return {"workload": f"decode step, {layers} layers x 256 tokens, tiny shapes: the legacy write "
                        f"path (per cache: division, remainder, index cast, index_put) in eager "
                        f"PyTorch ops, one CUDA graph",
            "us_per_step": us, "us_per_layer": us / layers,
            "launches_per_layer_measured": kernels, "launches_per_step_designed": 12 * layers}


def graph_launch_us(dw, flags, launches: int, replays: int) -> float:
    """Mean time of one producer launch inside a CUDA graph of `launches`
    back-to-back launches (host submission cost excluded)."""
    import torch
    s = torch.cuda.Stream(device=dw.qkv.device)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(launches):
            dw.run(flags, stream=s)
    with torch.cuda.stream(s):
        g.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(replays):
            g.replay()
        e1.record(s)
        e1.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / (launches * replays)
    del g
    return us


def indexer_timing(replays: int = 200, calls: int = 20):
    """The indexer of the decode-batch-64 layer (64 queries, contexts U{1..9216},
    8 index heads of dim 128, fp8 index-K): one call = score kernel + top-k kernel;
    `calls` back-to-back calls captured in a graph, with programmatic dependent
    launch of the score kernel (and, for comparison, without)."""
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import workloads as wl
    from paged_kv_cache_msa_gb300.device import DeviceIndexer
    w = wl.indexer_decode64()
    dv = DeviceIndexer(w)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()

    def graph_us(flags, fused=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(calls):
                dv.run(stream=s, launch_flags=flags, fused=fused)
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(replays):
                g.replay()
            e1.record(s)
            e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / (replays * calls)

    us_plain = graph_us(0)
    us = graph_us(B.MSA_LAUNCH_PDL)
    us_fused = graph_us(B.MSA_LAUNCH_PDL, fused=True)
    alg = w.algorithmic_bytes()
    peak, _ = peaks()
    return {"workload": "decode batch 64, contexts U{1..9216}, 8 index heads x 128, fp8 index-K, "
                        "top-16 of 128-token blocks",
            "us_per_call": us, "us_per_call_without_pdl": us_plain, "launches_per_call": 2,
            "single_launch": {"entry": "msa_indexer_forward_fused", "us_per_call": us_fused,
                              "launches_per_call": 1,
                              "gbs": alg / (us_fused * 1e-6) / 1e9,
                              "frac_of_peak": alg / (us_fused * 1e-6) / 1e9 / peaks()[0]},
            "algorithmic_bytes": alg,
            "gbs": alg / (us * 1e-6) / 1e9, "frac_of_peak": alg / (us * 1e-6) / 1e9 / peak,
            "index_k_tokens_scanned": int(w.kv_len.sum())}


def decode_layer_timing(layers: int = 60, replays: int = 50):
    """The decode layer's MSA hot path at batch 64 (big shapes): the producer, then
    the indexer on what it wrote (compact index-Q, the index-K cache; contexts
    U{1..9216}), both with programmatic dependent launch, `layers` layers in one
    CUDA graph.  Each layer has its own index-K history pool (random codes, on the
    device); K/V pools are shared by the layers (the producer writes 64 rows)."""
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import workloads as wl
    from paged_kv_cache_msa_gb300.device import DecodeLayer, DeviceWorkload
    w = wl.config2_decode64()
    first = DeviceWorkload(w)
    g_cpu = torch.Generator(device="cuda")
    g_cpu.manual_seed(7)
    stack = []
    for l in range(layers):
        pools = dict(first.pools)
        pools["idx_k"] = torch.randint(0, 255, first.pools["idx_k"].shape, dtype=torch.uint8,
                                       device=first.device, generator=g_cpu)
        stack.append(DecodeLayer(DeviceWorkload(w, pools_on_device=pools), max_blocks_per_seq=144))
    s = torch.cuda.Stream()
    out = {}
    for name, flags, fused in (("pdl", B.MSA_LAUNCH_PDL, False), ("no_pdl", 0, False),
                               ("pdl_single_launch_indexer", B.MSA_LAUNCH_PDL, True)):
        with torch.cuda.stream(s):
            for layer in stack:
                layer.run(s, flags, fused=fused)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for layer in stack:
                    layer.run(s, flags, fused=fused)
            for _ in range(3):
                g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(replays):
                g.replay()
            e1.record(s)
            e1.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / replays
        out[name] = {"us_per_step": us, "us_per_layer": us / layers,
                     "launches_per_layer": 2 if fused else 3}
    return {"workload": f"decode batch 64, big shapes, contexts U{{1..9216}}: producer + indexer "
                        f"(top-16 of 128-token blocks) per layer, {layers} layers in one CUDA graph",
            "launches_per_layer": 3, **out}


def indexer_prefill_timing(reps: int = 5, num_seqs: int = 8):
    """The indexer of the prefill batch (8 x 8192 causal queries, 8 index heads of
    dim 128, fp8 index-K, top-16 of 128-token blocks): the query-run kernel (tiles
    of 16 queries on the tcgen05 tensor cores) and, for comparison, the per-query
    kernel; each call = score kernel + top-k kernel, CUDA events on the stream."""
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import workloads as wl
    from paged_kv_cache_msa_gb300.device import DeviceIndexer
    w = wl.indexer_prefill(num_seqs=num_seqs)
    dv = DeviceIndexer(w)
    s = torch.cuda.Stream()

    def timed(flags):
        with torch.cuda.stream(s):
            for _ in range(2):
                dv.run(stream=s, launch_flags=flags)
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(reps):
                dv.run(stream=s, launch_flags=flags)
            e1.record(s)
            e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps

    us_runs = timed(B.MSA_LAUNCH_QUERY_RUNS)
    us_plain = timed(0)
    T, H, D = w.idx_q.shape
    dots = 2.0 * float(w.kv_len.astype(np.int64).sum()) * H * D   # visible (query, key, head) dots
    # The query-run kernel multiplies each E4M3 key by the query's two E4M3 halves (hi
    # and lo): twice the visible dot products, at the E4M3 rate, which is twice the
    # bf16 rate (nominal 4.5 / 2.25 PFLOP/s), so the fraction equals that of the
    # visible dots against the bf16 peak.
    flops = 2.0 * dots
    burst, _, kind = tensor_peaks()
    peak = 2.0 * burst
    tf = flops / (us_runs * 1e-6) / 1e12
    return {"workload": f"prefill {num_seqs} x 8192 causal queries, 8 index heads x 128, fp8 index-K, "
                        "top-16 of 128-token blocks",
            "us_per_call": us_runs, "us_per_call_per_query_kernel": us_plain,
            "queries_per_s": T / (us_runs * 1e-6), "launches_per_call": 2,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "flops_per_call": flops,
                         "visible_dot_flops_per_call": dots,
                         "note": "E4M3 MMA flops of the hi and lo query halves on visible "
                                 "query-key-head dots only; the tiles also multiply padded "
                                 "and invisible entries",
                         "peak_kind": f"{kind} cuBLAS bf16 burst x 2 (nominal E4M3 / bf16 ratio)"}}


def tensor_peaks():
    """(burst, sustained) dense bf16 TFLOP/s measured on this machine (cuBLAS), with
    the kind; the fallback figures when the measurement file is absent."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def projection_timing(launches: int = 10, warmup: int = 3, num_seqs: int = 8,
                      operand_dtype: int = 0):
    """The projection GEMM with the producer in its epilogue on the prefill batch
    (8 x 8192 tokens, hidden 6,144 -> 11,392 outputs, big shapes, fp8 caches), with
    bf16 operands (0) or E4M3 operands with per-token / per-output scales (1),
    against the unfused pair it replaces: the cuBLAS GEMM of the same operand type
    (torch.matmul, or torch._scaled_mm for E4M3) writing the bf16 rows, then
    msa_producer_forward on them."""
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import workloads as wl
    from paged_kv_cache_msa_gb300.device import DeviceProjection, DeviceWorkload
    fp8 = operand_dtype == wl.DTYPE_E4M3
    pw = wl.projection_prefill(num_seqs=num_seqs, operand_dtype=operand_dtype)
    dp = DeviceProjection(pw)
    s = torch.cuda.Stream()

    def timed(fn):
        with torch.cuda.stream(s):
            for _ in range(warmup):
                fn()
            s.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(launches)]
            for a, b in ev:
                a.record(s)
                fn()
                b.record(s)
            s.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / launches

    ms = timed(lambda: dp.run(stream=s))
    status = int(dp.status.item())
    K = pw.hidden_size
    rows = torch.empty((pw.num_tokens, pw.width), dtype=torch.bfloat16, device=dp.device)
    comparator = None
    try:
        if fp8:
            X = dp.hidden.view(torch.float8_e4m3fn)[:, :K]
            Wt = dp.weight.view(torch.float8_e4m3fn)[:, :K]
            one = torch.ones((), dtype=torch.float32, device=dp.device)
            gemm = lambda: torch._scaled_mm(X, Wt.t(), scale_a=one, scale_b=one,
                                            out_dtype=torch.bfloat16, out=rows)
            comparator = "cuBLAS E4M3 GEMM (torch._scaled_mm, per-tensor scales) + producer"
        else:
            X = dp.hidden.view(torch.bfloat16)[:, :K]
            Wt = dp.weight.view(torch.bfloat16)[:, :K]
            gemm = lambda: torch.matmul(X, Wt.t(), out=rows)
            comparator = "cuBLAS bf16 GEMM (torch.matmul) + producer"
        ms_gemm = timed(gemm)
    except Exception as e:   # a torch build without the comparator GEMM
        ms_gemm, comparator = None, f"unavailable: {type(e).__name__}: {e}"[:160]
    dw = DeviceWorkload(pw.producer, pools_on_device=dp.pools)
    args = list(dw.args(B.MSA_LAUNCH_PERSISTENT))
    args[2], args[3] = int(rows.data_ptr()), pw.width
    ms_prod = timed(lambda: B.msa_producer_forward(*args, stream=s.cuda_stream))
    fl = pw.flops()
    tf = fl / (ms * 1e-3) / 1e12
    burst, sustained, kind = tensor_peaks()
    ratio = 2.0 if fp8 else 1.0   # nominal dense E4M3 : bf16 tensor rate (4.5 : 2.25 PFLOP/s)
    out = {"workload": f"prefill {num_seqs}x8192 tokens, hidden {K} -> {pw.width} outputs "
                       f"(64/8/8/1 heads x 128), fp8 caches; {'E4M3' if fp8 else 'bf16'} operands"
                       f"{' with per-token / per-output scales' if fp8 else ''}, fp32 accumulate",
           "ms_per_launch": ms, "tokens_per_s": pw.num_tokens / (ms * 1e-3),
           "launches_per_step": 1, "status": status,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": burst * ratio, "unit": "TFLOP/s",
                        "frac": tf / (burst * ratio), "frac_of_sustained": tf / (sustained * ratio),
                        "peak_kind": (f"{kind} cuBLAS bf16 (burst; sustained {sustained})"
                                      + (" x 2, the nominal E4M3 : bf16 ratio" if fp8 else "")),
                        "flops_per_launch": fl, "traffic": None},
           "unfused": {"comparator": comparator, "gemm_ms": ms_gemm, "producer_ms": ms_prod}}
    if ms_gemm is not None:
        out["unfused"].update(total_ms=ms_gemm + ms_prod,
                              gemm_tflops=fl / (ms_gemm * 1e-3) / 1e12)
        out["speedup_vs_unfused"] = (ms_gemm + ms_prod) / ms
    return out


def projection_decode_timing(batch: int = 64, calls: int = 20, replays: int = 20):
    """The projection with the producer in its epilogue on a decode batch (``batch``
    sequences x 1 token, hidden 6,144 -> 11,392 outputs, big shapes, fp8 caches),
    bf16 and E4M3 operands, each against its unfused pair (cuBLAS GEMM of the same
    operand type, then msa_producer_forward).  Every leg is a CUDA graph of
    ``calls`` launches replayed ``replays`` times; the figure is per launch (for
    the unfused pair, per GEMM + producer)."""
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import workloads as wl
    from paged_kv_cache_msa_gb300.device import DeviceProjection, DeviceWorkload
    s = torch.cuda.Stream()

    def graph_us(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            fn()
            s.synchronize()
            with torch.cuda.graph(g, stream=s):
                for _ in range(calls):
                    fn()
            for _ in range(3):
                g.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(replays):
                g.replay()
            e1.record(s)
            s.synchronize()
        return 1e3 * e0.elapsed_time(e1) / (calls * replays)

    out = {}
    for name, dt in (("bf16", wl.DTYPE_BF16), ("e4m3", wl.DTYPE_E4M3)):
        pw = wl.projection_decode(batch=batch, operand_dtype=dt)
        dp = DeviceProjection(pw)
        fused = graph_us(lambda: B.msa_projection_forward(*dp.args(), stream=s.cuda_stream))
        status = int(dp.status.item())
        K = pw.hidden_size
        rows = torch.empty((pw.num_tokens, pw.width), dtype=torch.bfloat16, device=dp.device)
        try:
            if dt == wl.DTYPE_E4M3:
                X = dp.hidden.view(torch.float8_e4m3fn)[:, :K]
                Wt = dp.weight.view(torch.float8_e4m3fn)[:, :K]
                one = torch.ones((), dtype=torch.float32, device=dp.device)
                gemm = graph_us(lambda: torch._scaled_mm(X, Wt.t(), scale_a=one, scale_b=one,
                                                         out_dtype=torch.bfloat16, out=rows))
            else:
                X = dp.hidden.view(torch.bfloat16)[:, :K]
                Wt = dp.weight.view(torch.bfloat16)[:, :K]
                gemm = graph_us(lambda: torch.matmul(X, Wt.t(), out=rows))
        except Exception as e:   # a torch build without the comparator GEMM
            gemm = None
            log(f"[bench] decode comparator unavailable: {type(e).__name__}: {e}"[:160])
        dw = DeviceWorkload(pw.producer, pools_on_device=dp.pools)
        args = list(dw.args(B.MSA_LAUNCH_PERSISTENT))
        args[2], args[3] = int(rows.data_ptr()), pw.width
        prod = graph_us(lambda: B.msa_producer_forward(*args, stream=s.cuda_stream))
        wbytes = pw.width * K * (1 if dt == wl.DTYPE_E4M3 else 2)
        out[name] = {"workload": f"decode {batch} tokens, hidden {K} -> {pw.width} outputs, "
                                 f"{name} operands, fp8 caches",
                     "us_per_launch": fused, "status": status,
                     "weight_read_gbs": wbytes / (fused * 1e-6) / 1e9,
                     "unfused": {"gemm_us": gemm, "producer_us": prod,
                                 "total_us": None if gemm is None else gemm + prod},
                     "speedup_vs_unfused": None if gemm is None else (gemm + prod) / fused}
        del dp, dw
    return out


def run_ours(args):
    import torch
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300 import build as build_mod
    from paged_kv_cache_msa_gb300.device import DeviceWorkload

    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        build_mod.build()
    barrier(world)
    B.load()

    t_gen = time.perf_counter()
    w = make_workload(args.workload, args.prefill_seqs)
    log(f"[bench] workload {w.name}: {w.num_tokens} tokens, generated in "
        f"{time.perf_counter() - t_gen:.1f}s")
    dw = DeviceWorkload(w, device=dev)
    flags = B.MSA_LAUNCH_PERSISTENT
    grid, block, _ = B.msa_producer_launch_shape(dw.cfg, w.num_tokens, flags)
    stream = torch.cuda.Stream(device=dev)
    alg_bytes = w.algorithmic_bytes()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            dw.run(flags, stream=stream)
        stream.synchronize()

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
        clocks.start()
        time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            dw.run(flags, stream=stream)
            ends[i].record(stream)
        t_end.record(stream)
        t_end.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop()
    elapsed_ms = t_begin.elapsed_time(t_end)
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_avg_ms = sum(kernel_ms) / len(kernel_ms)
    elapsed_ms = max_over_ranks(elapsed_ms, world)

    tokens_total = w.num_tokens * args.steps * world
    value = tokens_total / (elapsed_ms / 1e3)
    peak, peak_kind = peaks()
    achieved = alg_bytes / (kernel_avg_ms / 1e3) / 1e9
    traffic = ncu_traffic(args.workload)

    big = alg_bytes > 256e6
    us_graph = graph_launch_us(dw, flags, launches=20 if big else 100, replays=5 if big else 20)

    # end to end: pinned host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(dw, w, flags, steps=min(args.steps, 20), warmup=2, world=world)

    decode = None
    if not args.no_decode_step:
        decode = {"tiny": decode_step_timing(1000, big=False, pdl=True),
                  "tiny_no_pdl": decode_step_timing(1000, big=False, pdl=False),
                  "big": decode_step_timing(200, big=True, pdl=True),
                  "empty_graph_floor": empty_graph_floor(60),
                  "legacy_write_path": legacy_write_path_timing()}

    indexer = None
    if not args.no_decode_step:
        indexer = indexer_timing()
        indexer["prefill"] = indexer_prefill_timing()
        decode["layer_with_indexer"] = decode_layer_timing()

    projection = None
    if not args.no_projection:
        projection = {"bf16": projection_timing(num_seqs=args.projection_seqs, operand_dtype=0),
                      "e4m3": projection_timing(num_seqs=args.projection_seqs, operand_dtype=1),
                      "decode_64": projection_decode_timing()}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n, dt = OracleRunner(w).timed(budget_s=args.cpu_budget)
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n} of {w.num_tokens} tokens of the same workload "
                         f"({dt:.1f}s, single-threaded C oracle on the host)",
               **host_cpu()}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload] if args.prefill_seqs == 8 or args.workload != "prefill"
                   else f"prefill {args.prefill_seqs}x8192 (reduced)", "tokens_per_step": w.num_tokens,
                   "global_batch": w.num_tokens * world, "launch": f"persistent grid {grid}x{block}",
                   "l2": "inputs larger than L2 (1.49 GB of rows per step), no flush",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps,
        "clocks": clk,
        # the large per-leg records first; the headline figures at the end of the line
        "projection": projection,
        "indexer": indexer,
        "decode_step_detail": decode,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "us_per_launch": kernel_avg_ms * 1e3,
        "us_per_launch_in_graph": us_graph,
        "hbm_gbs": achieved, "hbm_frac_of_peak": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "kernel_avg_us": kernel_avg_ms * 1e3},
        "decode_step": decode_summary(decode),
    }
    print(json.dumps(line), flush=True)
    return 0


def decode_summary(decode):
    """The decode-step figures in a few numbers (the full records are in
    decode_step_detail)."""
    if not decode:
        return None
    t = decode["tiny"]
    out = {"workload": "60 layers x 256 tokens, tiny shapes, one CUDA graph, PDL",
           "us_per_layer": t["us_per_layer"], "us_per_step": t["us_per_step"],
           "launches_per_step": t["launches_per_step"],
           "us_per_layer_no_pdl": decode["tiny_no_pdl"]["us_per_layer"],
           "us_per_layer_big_shapes": decode["big"]["us_per_layer"]}
    f = decode.get("empty_graph_floor")
    if f:
        out["empty_graph_us_per_node"] = f["us_per_node"]
    lw = decode.get("legacy_write_path")
    if lw:
        out["legacy_write_path_us_per_step"] = lw["us_per_step"]
        out["legacy_write_path_launches_per_layer"] = lw["launches_per_layer_measured"]
    li = decode.get("layer_with_indexer")
    if li:
        out["layer_with_indexer_us_per_layer"] = li["pdl"]["us_per_layer"]
        if "pdl_single_launch_indexer" in li:
            out["layer_with_single_launch_indexer_us_per_layer"] = \
                li["pdl_single_launch_indexer"]["us_per_layer"]
    return out


def run_e2e(dw, w, flags, steps, warmup, world, chunk_tokens=8192):
    """End to end from pinned host memory through the package's HostPipeline: per step
    the rows, positions and slots go from host to device and the compact Q / index-Q
    come back, either inside the kernel over the CPU-GPU link (zero copy, the
    headline) or by chunked copies overlapped with the kernel.  Timed with the host
    clock around whole steps."""
    import torch
    from paged_kv_cache_msa_gb300.pipeline import HostPipeline
    h_qkv = torch.from_numpy(w.qkv.view(np.int16)).pin_memory()
    h_pos = torch.from_numpy(w.positions).pin_memory()
    h_slot = torch.from_numpy(w.slot_mapping).pin_memory()
    h_q = torch.empty(dw.q_out.shape, dtype=torch.int16).pin_memory()
    h_iq = torch.empty(dw.idx_q_out.shape, dtype=torch.int16).pin_memory()
    pipe = HostPipeline(dw.cfg, w.row_stride, min(chunk_tokens, w.num_tokens), dw.qkv.device,
                        (dw.weights.get("q"), dw.weights.get("k"), dw.weights.get("idx_q"),
                         dw.weights.get("idx_k")),
                        (dw.caches["k"], dw.caches["v"], dw.caches["idx_k"]), dw.scales,
                        dw.page_table, flags)
    h2d = h_qkv.numel() * 2 + h_pos.numel() * 4 + h_slot.numel() * 8
    d2h = h_q.numel() * 2 + h_iq.numel() * 2
    def timed(fn):
        for _ in range(warmup):
            fn(h_qkv, h_pos, h_slot, h_q, h_iq)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(steps):
            fn(h_qkv, h_pos, h_slot, h_q, h_iq)
        torch.cuda.synchronize()
        return max_over_ranks(1e3 * (time.perf_counter() - t0), world)

    ms_zero = timed(pipe.run_zero_copy)
    ms_copy = timed(pipe.run)
    link = pinned_copy_bandwidth(h_qkv, h_q, dw.qkv.device)
    return {"value": w.num_tokens * steps * world / (ms_zero / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms_zero / steps,
            "api": "paged_kv_cache_msa_gb300.pipeline.HostPipeline.run_zero_copy: the kernel reads "
                   "rows from and writes compact outputs to pinned host memory over NVLink-C2C",
            "copy_pipeline": {"value": w.num_tokens * steps * world / (ms_copy / 1e3),
                              "ms_per_step": ms_copy / steps,
                              "chunk_tokens": min(chunk_tokens, w.num_tokens),
                              "api": "HostPipeline.run: chunked cudaMemcpyAsync in, kernel, out"},
            "link": link,
            "frac_of_copy_link": ((h2d + d2h) / (ms_zero / steps * 1e-3) / 1e9) / link["gbs_both_ways_serial"]}


def pinned_copy_bandwidth(h_in, h_out, device, reps: int = 5):
    """Plain cudaMemcpyAsync of the step's input bytes host -> device and output
    bytes device -> host (pinned host memory, one copy each, CUDA events): the
    CPU-GPU link's throughput for exactly the end-to-end step's traffic."""
    import torch
    d_in = torch.empty(h_in.shape, dtype=h_in.dtype, device=device)
    d_out = torch.empty(h_out.shape, dtype=h_out.dtype, device=device)
    s = torch.cuda.Stream(device=device)

    def timed(fn):
        with torch.cuda.stream(s):
            fn()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(reps):
                fn()
            e1.record(s)
            e1.synchronize()
        return e0.elapsed_time(e1) / reps
    ms_h2d = timed(lambda: d_in.copy_(h_in, non_blocking=True))
    ms_d2h = timed(lambda: h_out.copy_(d_out, non_blocking=True))
    b_in = h_in.numel() * h_in.element_size()
    b_out = h_out.numel() * h_out.element_size()
    del d_in, d_out
    return {"h2d_gbs": b_in / (ms_h2d * 1e-3) / 1e9, "d2h_gbs": b_out / (ms_d2h * 1e-3) / 1e9,
            "h2d_bytes": b_in, "d2h_bytes": b_out,
            "gbs_both_ways_serial": (b_in + b_out) / ((ms_h2d + ms_d2h) * 1e-3) / 1e9,
            "what": "one pinned cudaMemcpyAsync each way of the rows in and compact Q out"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["prefill", "decode64", "mixed", "tiny"], default="prefill")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode-step", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--indexer-only", action="store_true",
                    help="time only the decode-batch-64 indexer and print its JSON")
    ap.add_argument("--indexer-prefill-only", action="store_true",
                    help="time only the prefill (query-run) indexer and print its JSON")
    ap.add_argument("--no-projection", action="store_true",
                    help="skip the projection GEMM + producer leg")
    ap.add_argument("--projection-only", action="store_true",
                    help="time only the projection GEMM + producer and print its JSON")
    ap.add_argument("--projection-seqs", type=int, default=8,
                    help="sequences of 8,192 tokens in the projection leg (8 = the full batch)")
    ap.add_argument("--prefill-seqs", type=int, default=8,
                    help="sequences of 8,192 tokens in the prefill workload (8 = the full batch)")
    args = ap.parse_args()
    if args.warmup < 3:
        log("[bench] warmup raised to 3 (timing rule)")
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.projection_only:
        from paged_kv_cache_msa_gb300 import build as build_mod
        build_mod.build()
        out = {dt: projection_timing(launches=max(1, args.steps), warmup=args.warmup,
                                     num_seqs=args.projection_seqs, operand_dtype=i)
               for i, dt in enumerate(("bf16", "e4m3"))}
        out["decode_64"] = projection_decode_timing()
        print(json.dumps(out), flush=True)
        return 0
    if args.indexer_prefill_only:
        from paged_kv_cache_msa_gb300 import build as build_mod
        build_mod.build()
        print(json.dumps(indexer_prefill_timing(reps=max(1, args.steps), num_seqs=args.prefill_seqs)),
              flush=True)
        return 0
    if args.indexer_only:
        from paged_kv_cache_msa_gb300 import build as build_mod
        build_mod.build()
        out = indexer_timing(replays=max(1, args.steps), calls=20)
        out["prefill"] = indexer_prefill_timing(num_seqs=args.prefill_seqs)
        out["decode_layer"] = decode_layer_timing()
        print(json.dumps(out), flush=True)
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
