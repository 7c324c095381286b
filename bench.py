"""Benchmark: the quantized paged KV-cache hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. nvfp4_ds_mla write of 4,194,304 tokens (fills the 65536 x 64 x 352 cache)
  2. fp8_ds_mla gather-upconvert: 16 requests x 16384 rows (32768 x 64 x 656 cache)
  3. nvfp4_ds_mla gather-upconvert: 32 requests, 4k-32k rows each, from cache 1
  4. per-head NVFP4 reshape_and_cache: K, V bf16 [16384, 8, 128]
Inputs are resident in HBM before timing starts and exceed the 129 MB L2
(about 7.8 GB move per step), so no L2 flush is needed between steps.

value = algorithmic bytes of the step / device time of the step (GB/s);
tokens_per_s counts written tokens + gathered rows + per-head tokens.
--impl reference times the CPU oracle (the only reference that exists for
this path) on bounded samples of the same workloads, on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch one process per GPU with torch.distributed.run; each rank
runs an independent replica of the step (no data-path collective).
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "write & gather-upconvert HBM GB/s (fraction of GB300 peak) and tokens/s"
WORKLOAD = ("nvfp4_ds_mla write 4,194,304 tok (65536x64x352 fill) + fp8_ds_mla gather 16x16384 rows "
            "(32768x64x656) + nvfp4_ds_mla gather 32 req U[4k,32k] rows + per-head NVFP4 "
            "reshape_and_cache K,V [16384,8,128] (16384x2x16x8x72)")

# Algorithmic bytes per unit of work (inputs read once + outputs written once).
BYTES_WRITE_NVFP4 = 1024 + 128 + 8 + 352       # per valid token; 8 per padding token
BYTES_WRITE_FP8 = 1024 + 128 + 8 + 656
BYTES_GATHER_NVFP4 = 352 + 1152                # per output row
BYTES_GATHER_FP8 = 656 + 1152
ATTN_FLOPS_PER_SLOT_HEAD = 2 * 576 + 2 * 512    # q . k and the weighted sum of v, per valid slot and head


def per_head_bytes_per_token(H, D):
    return 2 * H * (2 * D + D // 2 + D // 16) + 8


KERNEL_ORDER = ["write_nvfp4_ds_mla", "gather_fp8_ds_mla", "gather_nvfp4_ds_mla",
                "reshape_and_cache_nvfp4"]


# --------------------------------------------------------------------------
# distributed helpers (one process per GPU, replicas)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 20 ms, timestamped."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: str):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "20"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if len(inside) < 3:          # very short timed region: widen to the loaded span around it
            inside = [p for (t, p) in self.samples if t0 - 0.5 <= t <= t1 + 0.5]
            window = "timed region +-0.5 s"
        if not inside:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        mx = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[4:8]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


def measured_peak_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def committed_traffic():
    """DRAM bytes per unit of work per kernel from the committed ncu summary
    (profiles/dram_traffic.txt), keyed by the source hash of the kernel file;
    a kernel whose source changed since the capture gets None."""
    out = {}
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return out
    for line in open(path):
        if line.startswith("#") or "=" not in line:
            continue
        kv = dict(item.split("=", 1) for item in line.split())
        if kernel_source_sha(kv.get("source", "")) == kv.get("source_sha"):
            out[kv["kernel"]] = float(kv["dram_bytes_per_unit"])
    return out


def kernel_source_sha(source: str):
    """12-hex-digit sha256 of a kernel file together with the headers it
    includes (kvq_device.cuh, kvq_launch.h, include/kvq.h), or None."""
    import hashlib
    csrc = os.path.join(ROOT, "fp8_quantized_paged_concat_gb300", "csrc")
    paths = [os.path.join(csrc, source), os.path.join(csrc, "kvq_device.cuh"),
             os.path.join(csrc, "kvq_launch.h"), os.path.join(ROOT, "include", "kvq.h")]
    if not source or not all(os.path.exists(q) for q in paths):
        return None
    h = hashlib.sha256()
    for q in paths:
        h.update(open(q, "rb").read())
    return h.hexdigest()[:12]


# --------------------------------------------------------------------------
# GPU path
# --------------------------------------------------------------------------

class GpuStep:
    """Device-resident inputs and outputs of one step, and its launches."""

    def __init__(self, device, size: str = "full"):
        import fp8_quantized_paged_concat_gb300 as kvq
        kvq.load_library()
        self.kvq = kvq
        self.device = device
        self.size = size
        if size == "full":
            self.g3 = wl.prefill_gather(device)
            self.g4 = wl.fp8_gather(device)
        else:    # profiling case: same kernels, a few hundred MB (still above the 129 MB L2)
            g = np.random.Generator(np.random.PCG64(3003))
            f3 = wl.make_fill("small fill 4096x64", 4096, 64, 3003, device, rng="device")
            self.g3 = wl.make_gather("small nvfp4 gather", f3, g.integers(4096, 16384, 8, endpoint=True),
                                     g.integers(1, 4095, 8, endpoint=True), 3003, device)
            f4 = wl.make_fill("small fp8 fill 4096x64", 4096, 64, 3004, device, entry_bytes=656, rng="device")
            self.g4 = wl.make_gather("small fp8 gather", f4, [16384] * 4,
                                     g.integers(1, 4095, 4, endpoint=True), 3004, device)
        self.ph = wl.per_head(device)
        f3, f4 = self.g3.fill, self.g4.fill
        self.cache3 = torch.zeros((f3.num_blocks, f3.block_size, 352), dtype=torch.uint8, device=device)
        self.cache4 = torch.zeros((f4.num_blocks, f4.block_size, 656), dtype=torch.uint8, device=device)
        kvq.kvq_write_fp8_ds_mla(f4.kv_c, f4.k_pe, self.cache4, f4.slot_mapping)      # setup fill
        self.ws3 = torch.empty((self.g3.num_out_tokens, 576), dtype=torch.bfloat16, device=device)
        self.ws4 = torch.empty((self.g4.num_out_tokens, 576), dtype=torch.bfloat16, device=device)
        T, H, D = self.ph.key.shape
        self.phc = torch.zeros((self.ph.num_pages, 2, self.ph.block_size, H, kvq.nvfp4_full_dim(D)),
                               dtype=torch.uint8, device=device)
        self.ks = torch.tensor([self.ph.k_scale], dtype=torch.float32, device=device)
        self.vs = torch.tensor([self.ph.v_scale], dtype=torch.float32, device=device)
        self.units = {
            "write_nvfp4_ds_mla": (f3.num_tokens, "tokens", BYTES_WRITE_NVFP4 * f3.num_tokens),
            "gather_fp8_ds_mla": (self.g4.num_out_tokens, "rows", BYTES_GATHER_FP8 * self.g4.num_out_tokens),
            "gather_nvfp4_ds_mla": (self.g3.num_out_tokens, "rows", BYTES_GATHER_NVFP4 * self.g3.num_out_tokens),
            "reshape_and_cache_nvfp4": (T, "tokens", per_head_bytes_per_token(H, D) * T),
        }
        torch.cuda.synchronize(device)

    def bytes_per_step(self):
        return sum(b for _, _, b in self.units.values())

    def tokens_per_step(self):
        return sum(n for n, _, _ in self.units.values())

    def launches(self):
        k, f3, g3, g4, ph = self.kvq, self.g3.fill, self.g3, self.g4, self.ph
        return [
            lambda: k.kvq_write_nvfp4_ds_mla(f3.kv_c, f3.k_pe, self.cache3, f3.slot_mapping),
            lambda: k.kvq_gather_upconvert_fp8_ds_mla(self.cache4, self.ws4, g4.block_table,
                                                      g4.workspace_starts, g4.seq_starts),
            lambda: k.kvq_gather_upconvert_nvfp4_ds_mla(self.cache3, self.ws3, g3.block_table,
                                                        g3.workspace_starts, g3.seq_starts),
            lambda: k.kvq_reshape_and_cache_nvfp4(ph.key, ph.value, self.phc, ph.slot_mapping,
                                                  self.ks, self.vs),
        ]


def time_device(step: GpuStep, K: int, W: int, world: int, clocks: ClockSampler | None):
    """W untimed steps, then K steps bracketed by barrier + synchronize, with
    an event between consecutive kernels (same stream)."""
    launches = step.launches()
    for _ in range(W):
        for fn in launches:
            fn()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    h0 = time.time()
    start.record()
    for k in range(K):
        for i, fn in enumerate(launches):
            evs[k][i].record()
            fn()
        evs[k][-1].record()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    h1 = time.time()
    total_ms = start.elapsed_time(end)
    per_kernel = {name: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K))
                  for i, name in enumerate(KERNEL_ORDER)}
    return total_ms, per_kernel, (h0, h1), K * len(launches)


def bind_to_gpu_numa_node(device):
    """Runs this process on the host CPUs local to the GPU (from sysfs), so
    that the pinned host buffers allocated next sit on the GPU's NUMA node.
    Returns (the previous CPU set or None, a note for the JSON line)."""
    try:
        p = torch.cuda.get_device_properties(device)
        bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        base = f"/sys/bus/pci/devices/{bdf}"
        with open(os.path.join(base, "local_cpulist")) as f:
            spec = f.read().strip()
        with open(os.path.join(base, "numa_node")) as f:
            node = f.read().strip()
    except (AttributeError, OSError, ValueError):
        return None, "process CPU set unchanged (the GPU's local CPUs are not known)"
    local = set()
    for part in spec.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            local.update(range(int(lo), int(hi) + 1))
        elif part:
            local.add(int(part))
    saved = os.sched_getaffinity(0)
    usable = local & saved
    if not usable:
        return None, f"process CPU set unchanged (none of the GPU's local CPUs {spec} is available)"
    os.sched_setaffinity(0, usable)
    return saved, f"pinned buffers allocated from the GPU's NUMA node {node} ({len(usable)} local CPUs)"


def time_e2e(step: GpuStep, K: int, chunks: int = 8):
    """The step through the public API with host buffers.  Every step copies
    each per-step input from pinned host memory to the device and every result
    (the written cache, both workspaces, the per-head cache) back, inside the
    timed region.  Three streams overlap the two copy directions with the
    kernels: the per-head write and the fp8 gather run, and their results flow
    back, while the 4.9 GB of write inputs stream in; the nvfp4 write runs on
    each of `chunks` token chunks as it lands (the same per-token work as one
    launch); the written cache and the nvfp4 workspace are read back last."""
    g3, g4, ph, kvq = step.g3, step.g4, step.ph, step.kvq
    f3 = g3.fill
    small_in = [g3.block_table, g3.workspace_starts, g3.seq_starts, g4.block_table, g4.workspace_starts,
                g4.seq_starts, ph.key, ph.value, ph.slot_mapping]
    big_in = [f3.kv_c, f3.k_pe, f3.slot_mapping]
    outs = [step.phc, step.ws4, step.cache3, step.ws3]
    h_small = [t.cpu().pin_memory() for t in small_in]
    h_big = [t.cpu().pin_memory() for t in big_in]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_small + h_big)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    T = f3.num_tokens
    bounds = [T * i // chunks for i in range(chunks + 1)]
    # a step's input copies wait until the previous step's kernels are done
    # with the input buffers; its kernels wait until the previous step's
    # results have been copied out (input copies of one step may overlap the
    # previous step's result copies: the two directions share no buffer)
    prev = {"run": None, "out": None}

    def one():
        ev_small = torch.cuda.Event()
        if prev["run"] is not None:
            s_in.wait_event(prev["run"])
            s_run.wait_event(prev["out"])
        with torch.cuda.stream(s_in):
            for d, h in zip(small_in, h_small):
                d.copy_(h, non_blocking=True)
            ev_small.record()
        ev_chunk = []
        for i in range(chunks):
            sl = slice(bounds[i], bounds[i + 1])
            with torch.cuda.stream(s_in):
                for d, h in zip(big_in, h_big):
                    d[sl].copy_(h[sl], non_blocking=True)
                e = torch.cuda.Event()
                e.record()
                ev_chunk.append(e)
        ev_ph, ev_g4, ev_w, ev_g3 = (torch.cuda.Event() for _ in range(4))
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_small)
            kvq.kvq_reshape_and_cache_nvfp4(ph.key, ph.value, step.phc, ph.slot_mapping, step.ks, step.vs)
            ev_ph.record()
            kvq.kvq_gather_upconvert_fp8_ds_mla(step.cache4, step.ws4, g4.block_table, g4.workspace_starts,
                                                g4.seq_starts)
            ev_g4.record()
            for i in range(chunks):
                s_run.wait_event(ev_chunk[i])
                sl = slice(bounds[i], bounds[i + 1])
                kvq.kvq_write_nvfp4_ds_mla(f3.kv_c[sl], f3.k_pe[sl], step.cache3, f3.slot_mapping[sl])
            ev_w.record()
            kvq.kvq_gather_upconvert_nvfp4_ds_mla(step.cache3, step.ws3, g3.block_table, g3.workspace_starts,
                                                  g3.seq_starts)
            ev_g3.record()
        with torch.cuda.stream(s_out):
            for ev, d, h in zip((ev_ph, ev_g4, ev_w, ev_g3), outs, h_out):
                s_out.wait_event(ev)
                h.copy_(d, non_blocking=True)
            ev_out = torch.cuda.Event()
            ev_out.record()
        prev["run"], prev["out"] = ev_g3, ev_out

    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(K):
        one()
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / K
    return ms, h2d, d2h


def graph_replay_us(launches, reps: int = 20) -> float:
    """Device time per launch of ``launches`` captured back to back in one
    CUDA graph (no host launch overhead), median over ``reps`` replays."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for fn in launches:
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for fn in launches:
            fn()
    graph.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / len(launches))
    return statistics.median(times) * 1e3


def time_extra(step: GpuStep):
    """Kernels measured outside the step.  Small launches are timed as CUDA
    graph replays over rotated input copies whose total exceeds L2 (no host
    launch overhead, no warm L2); the fp8_ds_mla fill is one large launch."""
    kvq, dev = step.kvq, step.device
    out = {}

    def record(name, us, units, nbytes, copies):
        out[name] = {"units": units, "us": round(us, 2), "gbs": round(nbytes / us / 1e3, 1),
                     "method": f"CUDA graph over {copies} input copies" if copies else "CUDA events"}

    # decode-step write: 8192 tokens, 12 copies (144 MB of inputs + caches)
    ds = [wl.make_write("decode", 8192, 4096, 64, 164, 1002 + 100 * i, dev, outlier_p=0.01) for i in range(12)]
    caches = [torch.zeros((4096, 64, 352), dtype=torch.uint8, device=dev) for _ in ds]
    us = graph_replay_us([lambda d=d, c=c: kvq.kvq_write_nvfp4_ds_mla(d.kv_c, d.k_pe, c, d.slot_mapping)
                          for d, c in zip(ds, caches)])
    valid = int((ds[0].slot_mapping >= 0).sum())
    record("write_nvfp4_ds_mla decode T=8192", us, 8192, BYTES_WRITE_NVFP4 * valid + 8 * (8192 - valid), 12)
    del ds, caches
    # per-head write and read-back: 16384 tokens x 8 heads x 128, 4 copies
    T, H, D = step.ph.key.shape
    phs = [wl.make_per_head("per-head", 16384, 8, 128, 16384, 16, 0, 1005 + 7 * i, dev) for i in range(4)]
    phcs = [torch.zeros((16384, 2, 16, 8, kvq.nvfp4_full_dim(128)), dtype=torch.uint8, device=dev) for _ in phs]
    us = graph_replay_us([lambda p=p, c=c: kvq.kvq_reshape_and_cache_nvfp4(p.key, p.value, c, p.slot_mapping,
                                                                           step.ks, step.vs) for p, c in zip(phs, phcs)])
    record("reshape_and_cache_nvfp4 T=16384 H=8 D=128", us, T, per_head_bytes_per_token(H, D) * T, 4)
    outs = [(torch.empty_like(p.key), torch.empty_like(p.value)) for p in phs]
    us = graph_replay_us([lambda p=p, c=c, o=o: kvq.kvq_dequant_nvfp4_per_head(c, p.slot_mapping, step.ks, step.vs,
                                                                               o[0], o[1])
                          for p, c, o in zip(phs, phcs, outs)])
    record("dequant_nvfp4_per_head T=16384 H=8 D=128", us, T, per_head_bytes_per_token(H, D) * T, 4)
    # the same in the HND layout [pages, 2, heads, block_size, full_dim]
    phcs = [c.view(16384, 2, 8, 16, -1) for c in phcs]
    us = graph_replay_us([lambda p=p, c=c: kvq.kvq_reshape_and_cache_nvfp4(p.key, p.value, c, p.slot_mapping,
                                                                           step.ks, step.vs, layout="HND")
                          for p, c in zip(phs, phcs)])
    record("reshape_and_cache_nvfp4 HND T=16384 H=8 D=128", us, T, per_head_bytes_per_token(H, D) * T, 4)
    us = graph_replay_us([lambda p=p, c=c, o=o: kvq.kvq_dequant_nvfp4_per_head(c, p.slot_mapping, step.ks, step.vs,
                                                                               o[0], o[1], layout="HND")
                          for p, c, o in zip(phs, phcs, outs)])
    record("dequant_nvfp4_per_head HND T=16384 H=8 D=128", us, T, per_head_bytes_per_token(H, D) * T, 4)
    del phs, phcs, outs
    # sparse-decode index conversion: 4096 decode tokens x 2048 positions over 64
    # requests of 4k-32k tokens (synthetic sizes), 10 % unused entries, 3 copies
    g = np.random.Generator(np.random.PCG64(4001))
    lens = g.integers(4096, 32768, 64, endpoint=True)
    table = torch.from_numpy(wl.make_gather_batch(65536, 64, lens, [0] * 64, 4001)[0]).to(dev)
    sets = []
    for _ in range(3):
        req = g.integers(0, 64, 4096).astype(np.int32)
        idx = (g.random((4096, 2048)) * lens[req][:, None]).astype(np.int32)
        idx[g.random((4096, 2048)) < 0.1] = -1
        sets.append((torch.from_numpy(req).to(dev), torch.from_numpy(idx).to(dev),
                     torch.empty((4096, 2048), dtype=torch.int32, device=dev)))
    us = graph_replay_us([lambda r=r, i=i, o=o: kvq.kvq_req_index_to_global_slot(r, i, table, 64, 65536, out=o)
                          for r, i, o in sets])
    record("req_index_to_global_slot 4096 x 2048", us, 4096 * 2048, 8 * 4096 * 2048 + 4 * 4096, 3)
    del sets
    # sparse MLA attention straight from the nvfp4_ds_mla cache (tensor
    # cores): 4096 decode tokens x 128 heads, top-2048 slots over the step's
    # 65536 x 64 cache (filled by the step's write), 10 % unused
    # (the same over the step's 32768 x 64 fp8_ds_mla cache)
    if step.size == "full":
        for fmt, fill, cache, entry, fn in (
                ("nvfp4_ds_mla", step.g3.fill, step.cache3, 352, kvq.kvq_sparse_mla_attention_nvfp4_ds_mla),
                ("fp8_ds_mla", step.g4.fill, step.cache4, 656, kvq.kvq_sparse_mla_attention_fp8_ds_mla)):
            aw = wl.sparse_attention(dev, fill=fill)
            ao = torch.empty((aw.num_tokens, 128, 512), dtype=torch.bfloat16, device=dev)
            al = torch.empty((aw.num_tokens, 128), dtype=torch.float32, device=dev)
            times = []
            for r in range(8):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn(aw.q, aw.indices, cache, aw.softmax_scale, out=ao, lse=al)
                b.record()
                torch.cuda.synchronize()
                if r >= 2:
                    times.append(a.elapsed_time(b))
            us = statistics.median(times) * 1e3
            n_valid = int((aw.indices >= 0).sum())
            flops = ATTN_FLOPS_PER_SLOT_HEAD * 128 * n_valid
            peak_tf, peak_src = measured_peak_tflops()
            nbytes = entry * n_valid + aw.q.numel() * 2 + ao.numel() * 2 + al.numel() * 4 + aw.indices.numel() * 4
            out[f"sparse_mla_attention_{fmt} T=4096 H=128 top-2048"] = {
                "units": aw.num_tokens, "us": round(us, 2), "tflops": round(flops / us / 1e6, 1),
                "bound": "tensor", "peak_tflops": peak_tf, "peak": f"{peak_src} bf16 burst",
                "frac": round(flops / us / 1e6 / peak_tf, 4), "gbs": round(nbytes / us / 1e3, 1),
                "valid_slots": n_valid, "method": "CUDA events"}
            if fmt == "nvfp4_ds_mla":
                # the same batch as decoded early in a sequence: only the first
                # 512 entries of each list are used (a 512-position context),
                # the rest -1; the tiles past the last used entry are skipped
                short = aw.indices.clone()
                short[:, 512:] = -1
                times = []
                for r in range(8):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    fn(aw.q, short, cache, aw.softmax_scale, out=ao, lse=al)
                    b.record()
                    torch.cuda.synchronize()
                    if r >= 2:
                        times.append(a.elapsed_time(b))
                us = statistics.median(times) * 1e3
                n_short = int((short >= 0).sum())
                flops_s = ATTN_FLOPS_PER_SLOT_HEAD * 128 * n_short
                out[f"sparse_mla_attention_{fmt} T=4096 H=128 top-2048, 512 used"] = {
                    "units": aw.num_tokens, "us": round(us, 2), "tflops": round(flops_s / us / 1e6, 1),
                    "bound": "tensor", "peak_tflops": peak_tf, "peak": f"{peak_src} bf16 burst",
                    "frac": round(flops_s / us / 1e6 / peak_tf, 4), "valid_slots": n_short, "method": "CUDA events"}
                del short
            del aw, ao, al
        # a small decode batch: 8 tokens x 128 heads x top-2048 over the same
        # nvfp4 cache, one CTA pair per token (16 CTAs on the GPU) against
        # the split over the keys (default_num_splits ranges, a combine
        # launch); CUDA-graph replays over 24 index sets (138 MB of entries,
        # more than L2)
        sets = [wl.make_attention(f"small decode {i}", 8, 128, 2048, 65536, 64, 600 + i, dev, p_unused=0.1,
                                  fill=step.g3.fill, rng="device") for i in range(24)]
        so = torch.empty((8, 128, 512), dtype=torch.bfloat16, device=dev)
        sl = torch.empty((8, 128), dtype=torch.float32, device=dev)
        splits = kvq.default_num_splits(8, 2048)
        ws = torch.empty(kvq.kvq_sparse_mla_attention_split_workspace_bytes(8, 128, splits), dtype=torch.uint8,
                         device=dev)
        n_valid = sum(int((s.indices >= 0).sum()) for s in sets) / len(sets)
        flops = ATTN_FLOPS_PER_SLOT_HEAD * 128 * n_valid
        peak_tf, peak_src = measured_peak_tflops()
        for name, fn in (
                ("sparse_mla_attention_nvfp4_ds_mla T=8 H=128 top-2048 (one range)",
                 lambda s: kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(s.q, s.indices, step.cache3, s.softmax_scale,
                                                                     out=so, lse=sl)),
                (f"sparse_mla_attention_split_nvfp4_ds_mla T=8 H=128 top-2048 ({splits} ranges)",
                 lambda s: kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla(s.q, s.indices, step.cache3,
                                                                           s.softmax_scale, num_splits=splits,
                                                                           workspace=ws, out=so, lse=sl))):
            us = graph_replay_us([lambda s=s, fn=fn: fn(s) for s in sets])
            out[name] = {"units": 8, "us": round(us, 2), "tflops": round(flops / us / 1e6, 1), "bound": "tensor",
                         "peak_tflops": peak_tf, "peak": f"{peak_src} bf16 burst",
                         "frac": round(flops / us / 1e6 / peak_tf, 4),
                         "method": "CUDA graph over 24 index sets"}
        del sets, so, sl, ws
        # dense prefill straight from the caches: each request of a gather
        # batch attends with 16 new tokens x 128 heads to its whole context
        # (seq_start + length positions) through the same block table
        for fmt, gather, cache, fn in (
                ("nvfp4_ds_mla", step.g3, step.cache3, kvq.kvq_prefill_mla_attention_nvfp4_ds_mla),
                ("fp8_ds_mla", step.g4, step.cache4, kvq.kvq_prefill_mla_attention_fp8_ds_mla)):
            pw = wl.prefill_attention(gather, dev)
            po = torch.empty((pw.num_tokens, 128, 512), dtype=torch.bfloat16, device=dev)
            pl = torch.empty((pw.num_tokens, 128), dtype=torch.float32, device=dev)
            times = []
            for r in range(8):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn(pw.q, pw.query_start, pw.context_lens, pw.block_table, cache, pw.softmax_scale,
                   pw.max_query_len, out=po, lse=pl)
                b.record()
                torch.cuda.synchronize()
                if r >= 2:
                    times.append(a.elapsed_time(b))
            us = statistics.median(times) * 1e3
            ctx = wl.host(pw.context_lens).astype(np.int64)
            ql = np.diff(wl.host(pw.query_start)).astype(np.int64)
            flops = ATTN_FLOPS_PER_SLOT_HEAD * 128 * int((ctx * ql).sum())
            peak_tf, peak_src = measured_peak_tflops()
            out[f"prefill_mla_attention_{fmt} B={len(ctx)} q=16 H=128 ctx {int(ctx.min())}-{int(ctx.max())}"] = {
                "units": pw.num_tokens, "us": round(us, 2), "tflops": round(flops / us / 1e6, 1),
                "bound": "tensor", "peak_tflops": peak_tf, "peak": f"{peak_src} bf16 burst",
                "frac": round(flops / us / 1e6 / peak_tf, 4), "context_positions": int(ctx.sum()),
                "method": "CUDA events"}
            # the pages' own flow for the same batch: gather every context
            # into a packed bf16 workspace, then attention over it
            ctx64 = wl.host(pw.context_lens).astype(np.int64)
            wstarts = np.zeros(len(ctx64), np.int32)
            wstarts[1:] = np.cumsum(ctx64)[:-1]
            wst = torch.from_numpy(wstarts).to(dev)
            zeros = torch.zeros(len(ctx64), dtype=torch.int32, device=dev)
            ws = torch.empty((int(ctx64.sum()), 576), dtype=torch.bfloat16, device=dev)
            gfn = kvq.kvq_gather_upconvert_nvfp4_ds_mla if fmt == "nvfp4_ds_mla" else kvq.kvq_gather_upconvert_fp8_ds_mla
            times_g, times_a = [], []
            for r in range(8):
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                e0.record()
                gfn(cache, ws, pw.block_table, wst, zeros, batch_size=len(ctx64))
                e1.record()
                kvq.kvq_prefill_mla_attention_workspace(pw.q, pw.query_start, pw.context_lens, wst, ws,
                                                        pw.softmax_scale, pw.max_query_len, out=po, lse=pl)
                e2.record()
                torch.cuda.synchronize()
                if r >= 2:
                    times_g.append(e0.elapsed_time(e1))
                    times_a.append(e1.elapsed_time(e2))
            ug, ua = statistics.median(times_g) * 1e3, statistics.median(times_a) * 1e3
            out[f"prefill over gathered workspace, {fmt} B={len(ctx)} q=16 H=128"] = {
                "units": pw.num_tokens, "us": round(ug + ua, 2), "gather_us": round(ug, 2),
                "attention_us": round(ua, 2), "tflops": round(flops / (ug + ua) / 1e6, 1),
                "attention_tflops": round(flops / ua / 1e6, 1), "bound": "tensor", "peak_tflops": peak_tf,
                "peak": f"{peak_src} bf16 burst", "frac": round(flops / (ug + ua) / 1e6 / peak_tf, 4),
                "attention_frac": round(flops / ua / 1e6 / peak_tf, 4), "method": "CUDA events"}
            del pw, po, pl, ws
        # one request with the longest context of the nvfp4 prefill batch, 16
        # query tokens x 128 heads: 32 CTAs, against the split over its
        # context (default_prefill_num_splits ranges, a combine launch)
        pw = wl.prefill_attention(step.g3, dev)
        b = int(np.argmax(wl.host(pw.context_lens)))
        qs = wl.host(pw.query_start)
        one = wl.PrefillWorkload("one request", None, pw.q[int(qs[b]):int(qs[b + 1])].contiguous(),
                                 torch.tensor([0, 16], dtype=torch.int32, device=dev), pw.context_lens[b:b + 1],
                                 pw.block_table[b:b + 1], pw.softmax_scale, 16)
        ctx1 = int(wl.host(one.context_lens)[0])
        po = torch.empty((16, 128, 512), dtype=torch.bfloat16, device=dev)
        pl = torch.empty((16, 128), dtype=torch.float32, device=dev)
        splits = kvq.default_prefill_num_splits(16, 128, 1, ctx1)
        ws = torch.empty(kvq.kvq_sparse_mla_attention_split_workspace_bytes(16, 128, splits), dtype=torch.uint8,
                         device=dev)
        flops = ATTN_FLOPS_PER_SLOT_HEAD * 128 * ctx1 * 16
        peak_tf, peak_src = measured_peak_tflops()
        for name, fn in (
                (f"prefill_mla_attention_nvfp4_ds_mla B=1 q=16 H=128 ctx {ctx1} (one range)",
                 lambda: kvq.kvq_prefill_mla_attention_nvfp4_ds_mla(one.q, one.query_start, one.context_lens,
                                                                    one.block_table, step.cache3, one.softmax_scale,
                                                                    16, out=po, lse=pl)),
                (f"prefill_mla_attention_split_nvfp4_ds_mla B=1 q=16 H=128 ctx {ctx1} ({splits} ranges)",
                 lambda: kvq.kvq_prefill_mla_attention_split_nvfp4_ds_mla(one.q, one.query_start, one.context_lens,
                                                                          one.block_table, step.cache3,
                                                                          one.softmax_scale, 16,
                                                                          max_context_len=ctx1, num_splits=splits,
                                                                          workspace=ws, out=po, lse=pl))):
            times = []
            for r in range(8):
                a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b2.record()
                torch.cuda.synchronize()
                if r >= 2:
                    times.append(a.elapsed_time(b2))
            us = statistics.median(times) * 1e3
            out[name] = {"units": 16, "us": round(us, 2), "tflops": round(flops / us / 1e6, 1), "bound": "tensor",
                         "peak_tflops": peak_tf, "peak": f"{peak_src} bf16 burst",
                         "frac": round(flops / us / 1e6 / peak_tf, 4),
                         "method": "CUDA events, repeated launches (its 12 MB of entries stay in L2)"}
        del pw, one, po, pl, ws
    # fp8_ds_mla cache fill: 2,097,152 tokens, one launch
    f4 = step.g4.fill
    times = []
    for r in range(13):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        kvq.kvq_write_fp8_ds_mla(f4.kv_c, f4.k_pe, step.cache4, f4.slot_mapping)
        b.record()
        torch.cuda.synchronize()
        if r >= 3:
            times.append(a.elapsed_time(b))
    record("write_fp8_ds_mla fill 2,097,152 tok", statistics.median(times) * 1e3, f4.num_tokens,
           BYTES_WRITE_FP8 * f4.num_tokens, 0)
    return out


# --------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# --------------------------------------------------------------------------

class CpuSample:
    """Bounded host samples of the four workloads, for the oracle."""

    def __init__(self, threads):
        import oracle
        self.oracle = oracle
        self.threads = threads
        g = np.random.Generator(np.random.PCG64(2003))
        # write: 262,144 tokens of the fill, into a 4096 x 64 cache
        w = wl.make_fill("cpu write sample", 4096, 64, 2003)
        self.w = (wl.bf16_bits(w.kv_c), wl.bf16_bits(w.k_pe), wl.host(w.slot_mapping))
        self.c_w = np.zeros((4096, 64, 352), np.uint8)
        # nvfp4 gather: 8 requests with the prefill length / start mix
        lens = g.integers(4096, 32768, size=8, endpoint=True)
        starts = g.integers(1, 4095, size=8, endpoint=True)
        nb = int(sum(-(-(s + n) // 64) for s, n in zip(starts, lens))) + 8
        f = wl.make_fill("cpu nvfp4 cache", nb, 64, 2004)
        self.c3 = np.zeros((nb, 64, 352), np.uint8)
        oracle.write_nvfp4_ds_mla(wl.bf16_bits(f.kv_c), wl.bf16_bits(f.k_pe), wl.host(f.slot_mapping),
                                  self.c3, threads=threads)
        self.b3 = wl.make_gather_batch(nb, 64, lens, starts, 2005)
        # fp8 gather: 8 requests x 16384 rows
        starts4 = g.integers(1, 4095, size=8, endpoint=True)
        nb4 = int(sum(-(-(s + 16384) // 64) for s in starts4)) + 8
        f4 = wl.make_fill("cpu fp8 cache", nb4, 64, 2006, entry_bytes=656)
        self.c4 = np.zeros((nb4, 64, 656), np.uint8)
        oracle.write_fp8_ds_mla(wl.bf16_bits(f4.kv_c), wl.bf16_bits(f4.k_pe), wl.host(f4.slot_mapping),
                                self.c4, threads=threads)
        self.b4 = wl.make_gather_batch(nb4, 64, [16384] * 8, starts4, 2007)
        # per-head: 8192 tokens of the [T, 8, 128] workload
        p = wl.make_per_head("cpu per-head sample", 8192, 8, 128, 16384, 16, 0, 2008)
        self.p = (wl.bf16_bits(p.key), wl.bf16_bits(p.value), wl.host(p.slot_mapping))
        self.pc = np.zeros((16384, 2, 16, 8, 72), np.uint8)
        self.units = {
            "write_nvfp4_ds_mla": (self.w[2].size, BYTES_WRITE_NVFP4 * self.w[2].size),
            "gather_fp8_ds_mla": (self.b4[3], BYTES_GATHER_FP8 * self.b4[3]),
            "gather_nvfp4_ds_mla": (self.b3[3], BYTES_GATHER_NVFP4 * self.b3[3]),
            "reshape_and_cache_nvfp4": (8192, per_head_bytes_per_token(8, 128) * 8192),
        }
        self.description = (f"oracle on {threads} host threads: write {self.w[2].size} tokens, "
                            f"fp8 gather {self.b4[3]} rows, nvfp4 gather {self.b3[3]} rows, "
                            f"per-head {8192} tokens per step")

    def bytes_per_step(self):
        return sum(b for _, b in self.units.values())

    def tokens_per_step(self):
        return sum(n for n, _ in self.units.values())

    def step(self):
        o, t = self.oracle, self.threads
        times = {}
        a = time.perf_counter()
        o.write_nvfp4_ds_mla(*self.w, self.c_w, threads=t)
        b = time.perf_counter()
        times["write_nvfp4_ds_mla"] = b - a
        tbl, ws, st, T = self.b4
        o.gather_fp8_ds_mla(self.c4, tbl, ws, st, T, threads=t)
        c = time.perf_counter()
        times["gather_fp8_ds_mla"] = c - b
        tbl, ws, st, T = self.b3
        o.gather_nvfp4_ds_mla(self.c3, tbl, ws, st, T, threads=t)
        d = time.perf_counter()
        times["gather_nvfp4_ds_mla"] = d - c
        o.reshape_and_cache_nvfp4(*self.p, self.pc, threads=t)
        times["reshape_and_cache_nvfp4"] = time.perf_counter() - d
        return times


def cpu_baseline(threads):
    """The oracle on all host cores over the bounded sample, repeated until
    about 10 s of wall time (at most 64 passes)."""
    s = CpuSample(threads)
    total, passes = 0.0, 0
    while passes < 64 and (passes == 0 or total < 10.0):
        total += sum(s.step().values())
        passes += 1
    return {"value": round(passes * s.bytes_per_step() / total / 1e9, 3), "unit": "GB/s",
            "cores": threads, "kind": "oracle", "sample": f"{passes} passes of: {s.description}",
            "tokens_per_s": round(passes * s.tokens_per_step() / total, 1), "seconds": round(total, 2)}


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0                          # rank 0 alone times the oracle
    import oracle
    threads = oracle.default_threads()
    s = CpuSample(threads)
    for _ in range(args.warmup):
        s.step()
    per = {k: 0.0 for k in KERNEL_ORDER}
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for k, v in s.step().items():
            per[k] += v
    sec = (time.perf_counter() - t0) / args.steps
    value = s.bytes_per_step() / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": s.description},
        "tokens_per_s": round(s.tokens_per_step() / sec, 1),
        "kernels": {k: {"units": s.units[k][0], "gbs": round(s.units[k][1] * args.steps / per[k] / 1e9, 3)}
                    for k in KERNEL_ORDER},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": s.description},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    step = GpuStep(device, args.size)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in visible.split(",") if v.strip()]
    clocks = ClockSampler(ids[local] if local < len(ids) else str(local))
    clocks.start()
    time.sleep(0.3)
    total_ms, per_kernel, (h0, h1), launches = time_device(step, args.steps, args.warmup, world, clocks)
    clocks.stop()
    clock_summary = clocks.summary(h0, h1)
    max_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = max_ms / args.steps
    bytes_step = step.bytes_per_step()
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peak_gbs()
    traffic = committed_traffic()

    kernels = {}
    for name in KERNEL_ORDER:
        units, unit_name, nbytes = step.units[name]
        ms = per_kernel[name]
        gbs = nbytes / ms / 1e6
        kernels[name] = {"units": units, "unit": unit_name, "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                         "frac": round(gbs / peak, 4), "units_per_s": round(units / ms * 1e3, 1)}
    dom = "write_nvfp4_ds_mla"
    d_units, _, d_bytes = step.units[dom]
    roofline = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kernels[dom]["frac"], "peak_source": peak_kind,
                "traffic": (round(traffic[dom] * d_units) if dom in traffic else None),
                "algorithmic_bytes": d_bytes}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD if args.size == "full" else "profiling case (--size small): " +
                   "nvfp4 fill 4096x64, nvfp4 gather 8 req U[4k,16k], fp8 gather 4x16384, per-head as full",
                   "bytes_per_step": bytes_step,
                   "l2": "no flush: every step moves ~7.8 GB, inputs exceed the 129 MB L2"},
        "frac_of_peak": round(value / world / peak, 4),
        "tokens_per_s": round(world * step.tokens_per_step() / (ms_per_step * 1e-3), 1),
        "kernels": kernels, "roofline": roofline, "gpu_launches": launches,
        "clocks": clock_summary,
    }
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 10))
        saved_cpus, numa_note = bind_to_gpu_numa_node(device)
        try:
            ms, h2d, d2h = time_e2e(step, e2e_steps)
        finally:
            if saved_cpus is not None:
                os.sched_setaffinity(0, saved_cpus)
        ms = max_over_ranks(ms, world, device)
        line["e2e"] = {"value": round(world * bytes_step / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
                       "steps": e2e_steps, "timing": "host clock around K steps, synchronize on both sides",
                       "overlap": "3 streams: copies in / kernels / copies out, write in 8 token chunks; "
                                  "a step's input copies may overlap the previous step's result copies",
                       "host_memory": numa_note}
    if not args.no_extra:
        line["kernels_extra"] = time_extra(step)
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        import oracle
        line["cpu_baseline"] = cpu_baseline(oracle.default_threads())
    barrier(world)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_prefill_only(query_len: int) -> int:
    """Profiler hook: the dense prefill alone on a small cache: 8 requests
    with contexts of 4k-16k positions over an 8192 x 64 cache, query_len new
    tokens x 128 heads each, 3 launches."""
    import fp8_quantized_paged_concat_gb300 as kvq
    kvq.load_library()
    dev = torch.device("cuda:0")
    fill = wl.make_fill("prefill profiling fill 8192x64", 8192, 64, 1007, dev, rng="device")
    cache = torch.zeros((8192, 64, 352), dtype=torch.uint8, device=dev)
    kvq.kvq_write_nvfp4_ds_mla(fill.kv_c, fill.k_pe, cache, fill.slot_mapping)
    g = np.random.Generator(np.random.PCG64(1007))
    w = wl.make_prefill("prefill profiling case", g.integers(4096, 16384, 8, endpoint=True), [query_len] * 8, 128,
                        8192, 64, 1007, dev, fill=fill, rng="device")
    for r in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        kvq.kvq_prefill_mla_attention_nvfp4_ds_mla(w.q, w.query_start, w.context_lens, w.block_table, cache,
                                                   w.softmax_scale, w.max_query_len)
        b.record()
        torch.cuda.synchronize()
        print(f"prefill_mla_attention q={query_len}: {a.elapsed_time(b) * 1e3:.1f} us", flush=True)
    return 0


def run_workspace_prefill_only(query_len: int) -> int:
    """Profiler hook: the case of run_prefill_only by the gather-then-attend
    flow (the contexts gathered into a packed bf16 workspace, then the
    prefill over it), 3 times."""
    import fp8_quantized_paged_concat_gb300 as kvq
    kvq.load_library()
    dev = torch.device("cuda:0")
    fill = wl.make_fill("prefill profiling fill 8192x64", 8192, 64, 1007, dev, rng="device")
    cache = torch.zeros((8192, 64, 352), dtype=torch.uint8, device=dev)
    kvq.kvq_write_nvfp4_ds_mla(fill.kv_c, fill.k_pe, cache, fill.slot_mapping)
    g = np.random.Generator(np.random.PCG64(1007))
    w = wl.make_prefill("prefill profiling case", g.integers(4096, 16384, 8, endpoint=True), [query_len] * 8, 128,
                        8192, 64, 1007, dev, fill=fill, rng="device")
    ctx = wl.host(w.context_lens).astype(np.int64)
    starts = np.zeros(len(ctx), np.int32)
    starts[1:] = np.cumsum(ctx)[:-1]
    wst = torch.from_numpy(starts).to(dev)
    ws = torch.empty((int(ctx.sum()), 576), dtype=torch.bfloat16, device=dev)
    zeros = torch.zeros(len(ctx), dtype=torch.int32, device=dev)
    for r in range(3):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record()
        kvq.kvq_gather_upconvert_nvfp4_ds_mla(cache, ws, w.block_table, wst, zeros, batch_size=len(ctx))
        b.record()
        kvq.kvq_prefill_mla_attention_workspace(w.q, w.query_start, w.context_lens, wst, ws, w.softmax_scale,
                                                w.max_query_len)
        c.record()
        torch.cuda.synchronize()
        print(f"gather {a.elapsed_time(b) * 1e3:.1f} us + prefill over the workspace q={query_len}: "
              f"{b.elapsed_time(c) * 1e3:.1f} us", flush=True)
    return 0


def run_attention_only(tokens: int, fmt: str = "nvfp4_ds_mla") -> int:
    """Profiler hook: the attention alone on a small cache (a few hundred MB)
    of either entry format."""
    import fp8_quantized_paged_concat_gb300 as kvq
    kvq.load_library()
    dev = torch.device("cuda:0")
    entry = 352 if fmt == "nvfp4_ds_mla" else 656
    fill = wl.make_fill("attention profiling fill 8192x64", 8192, 64, 1006, dev, entry_bytes=entry, rng="device")
    cache = torch.zeros((8192, 64, entry), dtype=torch.uint8, device=dev)
    if fmt == "nvfp4_ds_mla":
        kvq.kvq_write_nvfp4_ds_mla(fill.kv_c, fill.k_pe, cache, fill.slot_mapping)
        attend = kvq.kvq_sparse_mla_attention_nvfp4_ds_mla
    else:
        kvq.kvq_write_fp8_ds_mla(fill.kv_c, fill.k_pe, cache, fill.slot_mapping)
        attend = kvq.kvq_sparse_mla_attention_fp8_ds_mla
    w = wl.make_attention("attention profiling case", tokens, 128, 2048, 8192, 64, 1006, dev, p_unused=0.1,
                          fill=fill, rng="device")
    for r in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        attend(w.q, w.indices, cache, w.softmax_scale)
        b.record()
        torch.cuda.synchronize()
        print(f"sparse_mla_attention {fmt} T={tokens}: {a.elapsed_time(b) * 1e3:.1f} us", flush=True)
    return 0


KERNEL_ONLY = ["reshape_and_cache_nvfp4", "reshape_and_cache_nvfp4_hnd", "dequant_nvfp4_per_head",
               "dequant_nvfp4_per_head_hnd", "req_index_to_global_slot"]


def run_kernel_only(name: str) -> int:
    """Profiler hook: one kernel of the bench's extra measurements on its own
    workload (per-head: K, V [16384, 8, 128] into 16384 x 2 x 16 x 8 x 72;
    index conversion: 4096 x 2048 positions), 3 launches after one set-up
    launch, times printed; nothing else runs."""
    import fp8_quantized_paged_concat_gb300 as kvq
    kvq.load_library()
    dev = torch.device("cuda:0")
    if name.startswith(("reshape", "dequant")):
        layout = "HND" if name.endswith("_hnd") else "NHD"
        p = wl.make_per_head("per-head", 16384, 8, 128, 16384, 16, 0, 1005, dev)
        ks = torch.ones(1, dtype=torch.float32, device=dev)
        shape = (16384, 2, 16, 8, 72) if layout == "NHD" else (16384, 2, 8, 16, 72)
        cache = torch.zeros(shape, dtype=torch.uint8, device=dev)
        ko, vo = torch.empty_like(p.key), torch.empty_like(p.value)
        write = lambda: kvq.kvq_reshape_and_cache_nvfp4(p.key, p.value, cache, p.slot_mapping, ks, ks, layout=layout)
        fn = write if name.startswith("reshape") else \
            (lambda: kvq.kvq_dequant_nvfp4_per_head(cache, p.slot_mapping, ks, ks, ko, vo, layout=layout))
        write()
    else:
        g = np.random.Generator(np.random.PCG64(4001))
        lens = g.integers(4096, 32768, 64, endpoint=True)
        table = torch.from_numpy(wl.make_gather_batch(65536, 64, lens, [0] * 64, 4001)[0]).to(dev)
        req = g.integers(0, 64, 4096).astype(np.int32)
        idx = (g.random((4096, 2048)) * lens[req][:, None]).astype(np.int32)
        idx[g.random((4096, 2048)) < 0.1] = -1
        r, i = torch.from_numpy(req).to(dev), torch.from_numpy(idx).to(dev)
        o = torch.empty((4096, 2048), dtype=torch.int32, device=dev)
        fn = lambda: kvq.kvq_req_index_to_global_slot(r, i, table, 64, 65536, out=o)
    torch.cuda.synchronize()
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        print(f"{name}: {a.elapsed_time(b) * 1e3:.1f} us", flush=True)
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-extra", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--size", choices=["full", "small"], default="full",
                   help="small: the same kernels on ~0.4 GB inputs, for profiler captures")
    p.add_argument("--attention-only", type=int, default=0, metavar="T",
                   help="profiler hook: T decode tokens of the sparse MLA attention (128 heads, top-2048 "
                        "over an 8192 x 64 cache), 3 launches, times printed; nothing else runs")
    p.add_argument("--attention-fp8-only", type=int, default=0, metavar="T",
                   help="profiler hook: the same over a fp8_ds_mla cache of 8192 x 64 656-byte entries")
    p.add_argument("--workspace-prefill-only", type=int, default=0, metavar="Q",
                   help="profiler hook: the prefill case by gather + prefill over the workspace")
    p.add_argument("--prefill-only", type=int, default=0, metavar="Q",
                   help="profiler hook: the dense prefill alone, 8 requests with contexts of 4k-16k, Q new "
                        "tokens x 128 heads each, over an 8192 x 64 cache, 3 launches; nothing else runs")
    p.add_argument("--kernel-only", choices=KERNEL_ONLY, default=None,
                   help="profiler hook: one kernel of the extra measurements, 3 launches on its own "
                        "workload, times printed; nothing else runs")
    args = p.parse_args(argv)
    if args.attention_only > 0:
        return run_attention_only(args.attention_only)
    if args.attention_fp8_only > 0:
        return run_attention_only(args.attention_fp8_only, "fp8_ds_mla")
    if args.kernel_only:
        return run_kernel_only(args.kernel_only)
    if args.prefill_only > 0:
        return run_prefill_only(args.prefill_only)
    if args.workspace_prefill_only > 0:
        return run_workspace_prefill_only(args.workspace_prefill_only)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by torch.distributed.run: start one process per GPU through it
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", os.environ.get("MASTER_PORT", "29517"),
               os.path.abspath(__file__), *(sys.argv[1:] if argv is None else argv)]
        return subprocess.call(cmd)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
