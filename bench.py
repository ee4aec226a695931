"""Benchmark of the routed-MoE expert-slot cache on one GB300 (or N replicas).

Default workload (decode): 30 MoE layers, 128 experts/layer, top-8, hidden 2816,
expert FFN 704, Q4_0 experts (3,345,408 B each) in pinned host RAM, 32 slots per
layer, one token per step, Zipf(1.1) routing with 39% of a token's picks copied
from the previous token, fp32 activations N(0,1).  One step = one token through
all 30 layer calls (router, slot map, miss fill, FFN, combine).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (a bounded sample of the same workload).
N > 1 (torchrun): every rank runs its own replica on its own token stream
(independent sequences; no data-path collective), value = all ranks' tokens / max
time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import ctypes
import json
import mmap
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 GB300; achieved HBM GB/s vs roofline; cache hit rate"
UNIT = "tokens/s"
COLD_STEPS = 64        # decode steps reported as the cold start
DECODE_WARMUP = 1024   # decode steps before the timed region
PROFILE_STREAM = 777   # token stream that the warm-start profile is counted over (the timed one is 0)



_HOST_MAPS = []


def host_store(nbytes: int, node: int = -1, strict: bool = False):
    """The expert store in ordinary anonymous memory (transparent huge pages
    requested, 512 MB-aligned), as a torch uint8 tensor; the library pins and
    maps it with cudaHostRegister.  On this Grace host such memory reads over
    the host link faster and more steadily than a cudaHostAlloc buffer for the
    scattered expert blocks of the workload.  node >= 0: its pages are taken
    from that NUMA node (bound before the first touch; if the binding is
    refused, first touch decides, unless strict)."""
    import torch
    align = 512 << 20
    mm = mmap.mmap(-1, nbytes + align, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    if hasattr(mmap, "MADV_HUGEPAGE"):
        mm.madvise(mmap.MADV_HUGEPAGE)
    base = ctypes.addressof(ctypes.c_char.from_buffer(mm))
    off = (-base) % align
    if node >= 0 and not bind_to_node(base + off, nbytes, node) and strict:
        raise SystemExit(f"could not bind the host store to NUMA node {node}")
    arr = np.frombuffer(mm, dtype=np.uint8, count=nbytes, offset=off)
    _HOST_MAPS.append(mm)
    return torch.from_numpy(arr)


def shared_host_store(nbytes: int, node: int, fill, tag: str):
    """One host store per NUMA node, shared by the replicas (ranks) whose GPUs
    sit on that node, instead of one copy per rank (8 replicas of the decode
    model would otherwise hold 103 GB, of the large model 1 TB).  The lowest
    rank of each node creates a file in /dev/shm, binds its pages to the node,
    fills it (fill(tensor)) and maps it shared; the others map the same pages
    once it is filled; the file is unlinked once every rank has mapped it (the
    mappings stay).  Each rank's library then registers the mapping for its own
    GPU.  Needs the process group (torch.distributed) to be initialised."""
    import torch
    import torch.distributed as dist
    rank, world = dist.get_rank(), dist.get_world_size()
    nodes = [None] * world
    dist.all_gather_object(nodes, node)
    creator = min(r for r in range(world) if nodes[r] == node)
    path = f"/dev/shm/moe_store_{tag}_n{node}"
    mm = None
    if rank == creator:
        fd = os.open(path, os.O_CREAT | os.O_RDWR | os.O_TRUNC, 0o600)
        try:
            os.ftruncate(fd, nbytes)
            mm = mmap.mmap(fd, nbytes, flags=mmap.MAP_SHARED, prot=mmap.PROT_READ | mmap.PROT_WRITE)
        finally:
            os.close(fd)
        if hasattr(mmap, "MADV_HUGEPAGE"):
            try:
                mm.madvise(mmap.MADV_HUGEPAGE)
            except OSError:
                pass
        if node >= 0:
            bind_to_node(ctypes.addressof(ctypes.c_char.from_buffer(mm)), nbytes, node)
        fill(torch.from_numpy(np.frombuffer(mm, dtype=np.uint8, count=nbytes)))
    dist.barrier()
    if rank != creator:
        fd = os.open(path, os.O_RDWR)
        try:
            mm = mmap.mmap(fd, nbytes, flags=mmap.MAP_SHARED, prot=mmap.PROT_READ | mmap.PROT_WRITE)
        finally:
            os.close(fd)
    dist.barrier()
    if rank == creator:
        os.unlink(path)
    _HOST_MAPS.append(mm)
    return torch.from_numpy(np.frombuffer(mm, dtype=np.uint8, count=nbytes))


def bind_to_node(addr: int, length: int, node: int) -> bool:
    """mbind(addr, length, MPOL_BIND, {node}): pages of the range not yet
    touched come from NUMA node `node` (a policy of this process's own
    mapping; nothing else changes)."""
    import platform
    nr = {"aarch64": 235, "x86_64": 237}.get(platform.machine())
    if nr is None or not 0 <= node < 1024:
        return False
    libc = ctypes.CDLL(None, use_errno=True)
    mask = (ctypes.c_ulong * 16)()
    mask[node // 64] = 1 << (node % 64)
    MPOL_BIND = 2
    r = libc.syscall(ctypes.c_long(nr), ctypes.c_void_p(addr), ctypes.c_ulong(length), ctypes.c_int(MPOL_BIND),
                     mask, ctypes.c_ulong(16 * 64), ctypes.c_uint(0))
    return r == 0


def gpu_numa_node(dev: int = 0) -> int:
    """NUMA node of the GPU's PCI function (sysfs), or -1 when unknown."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/numa_node" % (p.pci_domain_id, p.pci_bus_id,
                                                                     p.pci_device_id)
        with open(path) as f:
            return int(f.read().strip())
    except (AttributeError, OSError, ValueError):
        return -1


def store_node(args, dev: int = 0) -> int:
    """The NUMA node the host store is bound to (-1: not bound)."""
    if args.store_node == "none":
        return -1
    if args.store_node == "auto":
        return gpu_numa_node(dev)
    return int(args.store_node)


def host_store_numa(t):
    """Pages of the host store per NUMA node ({"N0": pages, ...}), from
    /proc/self/numa_maps (the mapping that holds the store's first byte)."""
    try:
        addr = t.data_ptr()
        best = None
        with open("/proc/self/numa_maps") as f:
            for line in f:
                parts = line.split()
                start = int(parts[0], 16)
                if start <= addr and (best is None or start > best[0]):
                    best = (start, parts)
        if best is None:
            return None
        return {p.split("=")[0]: int(p.split("=")[1]) for p in best[1] if p[:1] == "N" and "=" in p}
    except (OSError, ValueError):
        return None


def huge_page_kb():
    """AnonHugePages of this process (kB), from /proc/self/smaps_rollup."""
    try:
        with open("/proc/self/smaps_rollup") as f:
            for line in f:
                if line.startswith("AnonHugePages:"):
                    return int(line.split()[1])
    except OSError:
        pass
    return None

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=448)
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed steps before the timed region (default: 1024 decode steps, of "
                         "which the first 64 are also reported as the cold start; 64 prefill "
                         "batches; 64 layer calls of the reference arm)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--fill", default="pull", choices=["memcpy", "pull"])
    ap.add_argument("--policy", default="lru", choices=["lru", "score", "adopt"],
                    help="slot replacement: LRU, the decayed-score admission policy (decode workload), or "
                         "LRU whose staged calls end holding their most-used experts (adopt)")
    ap.add_argument("--sticky", type=int, default=0,
                    help="score policy: per mille of the slots, highest scores first, never evicted")
    ap.add_argument("--admit-budget", type=int, default=0,
                    help="score policy: admissions per call (0 = no limit)")
    ap.add_argument("--preload-profile", type=int, default=0,
                    help="warm start: before the first step, preload each layer's most-used experts, "
                         "counted over this many tokens of another token stream with the same routing")
    ap.add_argument("--preload-from-session", type=int, default=0,
                    help="warm start from the library's own counts: a previous session (another handle "
                         "over the same store) decodes this many tokens of another token stream with the "
                         "same routing, its moe_cache_usage counts are read at its end and preloaded here")
    ap.add_argument("--slots", type=int, default=0,
                    help="decode and prefill workloads: slots per layer instead of the config's (up to "
                         "the number of experts: every expert resident once warm)")
    ap.add_argument("--store-node", default="auto",
                    help="NUMA node of the host store's pages: auto (the GPU's node, from sysfs), "
                         "none (first touch), or a node number")
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "large", "sweep"],
                    help="decode (default, the headline): 30 layers, 128 experts, 1 token per step; "
                         "prefill: 512-token batches through the tensor-core GEMM; large: 48 layers, "
                         "256 experts, hidden 4096, FFN 1536, a 130 GB host store, --batch tokens per "
                         "step; sweep: one layer, 64-token batches at budgets 8..128, uniform and "
                         "Zipf(1.2) routing (one JSON line per budget and routing)")
    ap.add_argument("--batch", type=int, default=1,
                    help="large workload: tokens per decode step (independent token streams), 1 or 8")
    ap.add_argument("--routing", default="trace", choices=["trace", "hot16"],
                    help="prefill workload: the Zipf + sticky trace, or every token picking among 16 "
                         "experts (each expert ~256 routed pairs: the GEMM's compute-bound case)")
    ap.add_argument("--tokens", type=int, default=512,
                    help="prefill workload: tokens per batch (one call per layer and batch)")
    ap.add_argument("--decode-after", type=int, default=0,
                    help="prefill workload: after the timed batches, decode this many tokens per layer, "
                         "continuing the last batch's token stream, and report their hit rate")
    ap.add_argument("--gemm-min-tokens", type=int, default=16,
                    help="prefill workload: calls of at least this many tokens take the tensor-core "
                         "grouped GEMM, shorter ones the GEMV kernels (0 = never the GEMM)")
    ap.add_argument("--cpu-sample-steps", type=int, default=96)  # ~14 s of oracle work on 16 cores
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kernel-pass", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="decode: time eager layer calls instead of the captured step graph")
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the model (profiling captures); 0 = all")
    return ap.parse_args()


def resolve_defaults(args):
    """Defaults that depend on the workload: the warm-up length."""
    if args.warmup is None:
        args.warmup = (DECODE_WARMUP if args.workload == "decode" and args.impl == "ours" else
                       4 if args.workload == "sweep" else 64)
    return args


def aggregate_over_ranks(dev_ms, e2e_ms_per_step, K, world, device, tokens_per_step=1):
    """The slowest rank's timed region (and end-to-end step time), by a MAX
    all-reduce when there are several ranks; whole-job tokens/s = world x K
    steps x tokens per step over that time.  Returns (max ms, tokens/s,
    end-to-end tokens/s or None)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([dev_ms, e2e_ms_per_step if e2e_ms_per_step is not None else 0.0],
                     dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dev_max = float(t[0].item())
    e2e_value = None if e2e_ms_per_step is None else world * tokens_per_step * 1e3 / float(t[1].item())
    return dev_max, world * K * tokens_per_step / (dev_max * 1e-3), e2e_value


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_config(sh, fill, T=1):
    name = "decode" if sh.name == "decode" else f"large model decode"
    per_step = "1 token/step" if T == 1 else f"{T} tokens/step (independent token streams)"
    return {
        "workload": (f"{name}: {sh.L} MoE layers, {sh.E} experts/layer, top-{sh.k}, hidden {sh.H}, "
                     f"expert FFN {sh.F}, Q4_0 experts ({sh.expert_bytes} B) in host RAM (pinned and mapped by "
                     f"the library), "
                     f"{sh.S} slots/layer, {per_step}, Zipf({sh.zipf}) routing with "
                     f"{int(sh.sticky * 100)}% of picks copied from the previous token, fp32 "
                     f"activations N(0,1)"),
        "layers": sh.L, "experts": sh.E, "top_k": sh.k, "hidden": sh.H, "ffn": sh.F,
        "slots_per_layer": sh.S, "tokens_per_step": T, "expert_bytes": sh.expert_bytes,
        "host_store_bytes": sh.store_bytes, "fill_mode": fill,
        "l2": "inputs larger than L2: each step streams ~0.8 GB of expert weights (> 129 MB L2)",
    }


# --------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def profiled_entry(kernel):
    """The committed ncu figures of `kernel` (profiles/traffic.json), or None
    when the kernel's source changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    src = open(os.path.join(ROOT, "router_softmax_top_gb300", "csrc", d.get("file", "ffn.cu"))).read()
    a, b = src.find(d["begin"]), src.find(d["end"])
    if a < 0 or b < 0:
        return None
    if hashlib.sha256(src[a:b].encode()).hexdigest() != d["source_sha256"]:
        return None
    return d


def profiled_traffic_ratio(kernel):
    """DRAM bytes per algorithmic byte of `kernel` from the committed ncu summary,
    or None when the kernel's source changed since the capture."""
    d = profiled_entry(kernel)
    return float(d["dram_bytes_per_algorithmic_byte"]) if d else None


def probe_h2d_sustained(store, block_bytes: int, n_blocks: int = 64, reps: int = 5):
    """Host-to-device bandwidth of the host store for large transfers (GB/s,
    1e9 B/s): n_blocks consecutive expert blocks (i) as one copy and (ii) as
    n_blocks back-to-back copies of one block each, into a device buffer on the
    current stream, timed with CUDA events; the median of `reps` (after one
    untimed pass).  Beside the library's per-block probe, this is the link's
    sustained rate."""
    import torch
    n = min(n_blocks, store.numel() // block_bytes)
    src = store[:n * block_bytes]
    dst = torch.empty(n * block_bytes, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    res = {}
    for mode in ("one_copy", "back_to_back"):
        v = []
        for r in range(reps + 1):
            torch.cuda.synchronize()
            e0.record()
            if mode == "one_copy":
                dst.copy_(src, non_blocking=True)
            else:
                for b in range(n):
                    dst[b * block_bytes:(b + 1) * block_bytes].copy_(src[b * block_bytes:(b + 1) * block_bytes],
                                                                       non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            if r > 0:
                v.append(n * block_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        res[mode] = statistics.median(v)
    res["blocks"] = n
    del dst
    return res


def step_stalls(step_ms):
    """Per-step device times of the timed region: median, max, and the steps
    slower than ten times the median (host-read stalls)."""
    med = statistics.median(step_ms)
    return {"step_ms_median": med, "step_ms_max": max(step_ms),
            "stall_steps": sum(1 for v in step_ms if v > 10 * med),
            "slow_steps_2x": sum(1 for v in step_ms if v > 2 * med)}


# ------------------------------------------------------- oracle (baseline)
def host_cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo ("model name", else the Arm
    implementer and part numbers) and the number of logical CPUs."""
    name = impl = part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key, val = key.strip(), val.strip()
                if key == "model name" and not name:
                    name = val
                elif key == "CPU implementer" and not impl:
                    impl = val
                elif key == "CPU part" and not part:
                    part = val
    except OSError:
        pass
    if not name and (impl or part):
        name = f"Arm implementer {impl} part {part}"
    return f"{name or 'unknown'}, {os.cpu_count()} logical CPUs"


def run_oracle_sample(sh, store_np, logits, x, n_steps, threads):
    """Time the CPU oracle over the first n_steps steps (all layers, outputs computed)."""
    import oracle
    c = oracle.Cache(sh.L, sh.E, sh.k, sh.H, sh.F, sh.S, store_np, threads=threads)
    t0 = time.perf_counter()
    for s in range(n_steps):
        for l in range(sh.L):
            c.forward(l, logits[s, l], x[s, l], compute=True)
    dt = time.perf_counter() - t0
    return n_steps / dt, dt, (threads if threads > 0 else oracle.max_threads())


def run_reference(args):
    """The oracle as it stands on the host cores.  One step = one layer call of the
    decode trace (layers visited in turn), tokens/s = 1 / (L x mean layer-call time)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    sh = synth.DECODE
    t0 = time.time()
    W, K = max(3, args.warmup), max(1, args.steps)
    nsteps = (W + K + sh.L - 1) // sh.L + 1
    store = synth.store(sh.L, sh.E, sh.H, sh.F, seed=0, threads=args.threads)
    _, logits, x = synth.decode_inputs(sh, nsteps, batch=1, seed=0)
    c = oracle.Cache(sh.L, sh.E, sh.k, sh.H, sh.F, sh.S, store, threads=args.threads)
    cores = args.threads if args.threads > 0 else oracle.max_threads()
    calls = [(s, l) for s in range(nsteps) for l in range(sh.L)]
    for s, l in calls[:W]:                      # warm-up: slot maps only
        c.forward(l, logits[s, l], x[s, l], compute=False)
    setup = time.time() - t0
    t1 = time.perf_counter()
    for s, l in calls[W:W + K]:
        c.forward(l, logits[s, l], x[s, l], compute=True)
    dt = time.perf_counter() - t1
    value = K / (dt * sh.L)                     # tokens/s: one token needs L layer calls
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": 1e3 * dt / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(sh, "oracle"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "cpu_model": host_cpu_model(),
                             "sample": f"{K} single-layer decode calls (layers in turn), outputs "
                                       f"computed; tokens/s = 1 / ({sh.L} x mean call time)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "setup_s": setup}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ prefill
def prefill_config(sh, fill, T=512, gemm_min=16):
    path = ("the tensor-core grouped GEMM" if gemm_min and T >= gemm_min else "the Q4_0 GEMV kernels")
    return {
        "workload": (f"prefill: {sh.L} MoE layers, {sh.E} experts/layer, top-{sh.k}, hidden {sh.H}, "
                     f"expert FFN {sh.F}, Q4_0 experts in host RAM (pinned and mapped by the library), "
                     f"{sh.S} slots/layer, "
                     f"{T} tokens per batch through {path}, Zipf({sh.zipf}) routing "
                     f"with {int(sh.sticky * 100)}% of picks copied from the previous token, bf16 "
                     f"activations N(0,1)"),
        "layers": sh.L, "experts": sh.E, "top_k": sh.k, "hidden": sh.H, "ffn": sh.F,
        "slots_per_layer": sh.S, "tokens_per_step": T, "gemm_min_tokens": gemm_min, "fill_mode": fill,
        "l2": "inputs larger than L2: each batch streams the stage-wise expert weights and activations "
              "(~1 GB per layer-batch) through HBM",
    }


def run_prefill(args):
    import torch

    import router_softmax_top_gb300 as moe
    sh = synth.PREFILL
    if args.layers:
        import dataclasses
        sh = dataclasses.replace(sh, L=min(sh.L, args.layers))
    if args.slots:
        import dataclasses
        sh = dataclasses.replace(sh, S=min(sh.E, args.slots))
    T = args.tokens
    assert T >= 1 and args.gemm_min_tokens >= 0
    if args.policy == "score":
        raise SystemExit("the score policy plans single-stage calls only: not a prefill policy")
    W, K = max(3, args.warmup), args.steps
    torch.cuda.set_device(0)
    eb = sh.expert_bytes
    node = store_node(args, 0)
    store = host_store(sh.L * sh.E * eb, node, strict=args.store_node not in ("auto", "none"))
    synth.fill_store(store.data_ptr(), sh.L, sh.E, sh.H, sh.F, 0, args.threads)
    nb = W + 2 * K
    _, logits_h, x_h = synth.batch_inputs(sh, nb, T, seed=0, act="bf16")
    if args.routing == "hot16":
        # every token picks 8 of the first 16 experts (uniformly): ~256 routed
        # pairs per expert and layer, the GEMM's compute-bound case
        for l in range(sh.L):
            for b in range(nb):
                pk = synth.trace(T, 16, sh.k, 0.0, 0.0, 0, l, 10000 + b)
                logits_h[b, l] = synth.logits_from_picks(pk, sh.E, 0, l, 10000 + b, 1)
    logits_d = torch.from_numpy(logits_h).cuda()
    x_d = torch.from_numpy(x_h.view(np.int16)).cuda().view(torch.bfloat16)
    out_d = torch.empty((sh.L, T, sh.H), dtype=torch.float32, device="cuda")
    fill = moe.MOE_FILL_PULL if args.fill == "pull" else moe.MOE_FILL_MEMCPY
    cache = moe.MoECache(n_layers=sh.L, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                         slots_per_layer=sh.S, max_tokens=T, store=store, act_dtype="bf16",
                         fill_mode=fill, gemm_min_tokens=args.gemm_min_tokens, timeout_us=60_000_000,
                         policy={"lru": moe.MOE_POLICY_LRU, "adopt": moe.MOE_POLICY_ADOPT}[args.policy])
    h2d_gbps = cache.probe_h2d(24)
    h2d_sus = probe_h2d_sustained(store, eb)
    h2d_peak = max(h2d_gbps, h2d_sus["one_copy"])
    fwd = moe.lib().moe_layer_forward
    sh_ = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def run(b0, b1):
        for b in range(b0, b1):
            for l in range(sh.L):
                rc = fwd(cache.handle, l, ctypes.c_void_p(logits_d[b, l].data_ptr()),
                         ctypes.c_void_p(x_d[b, l].data_ptr()), T, ctypes.c_void_p(out_d[l].data_ptr()), sh_)
                if rc != 0:
                    raise moe.MoeError(rc, f"moe_layer_forward batch {b} layer {l}")

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(0, W)
    torch.cuda.synchronize()
    st1 = cache.stats(-1)
    clocks = ClockSampler(0)
    clocks.start()
    e0.record()
    run(W, W + K)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    st2 = cache.stats(-1)
    cache.set_timing(True)
    run(W + K, W + 2 * K)
    torch.cuda.synchronize()
    kt = cache.timing()
    cache.set_timing(False)
    st3 = cache.stats(-1)
    after = None
    if args.decode_after:
        # single tokens after the last batch, continuing each layer's token
        # stream of that batch (the same trace, longer): the cache as the
        # prompt left it
        D, bl = args.decode_after, nb - 1
        lg2 = np.empty((D, sh.L, 1, sh.E), np.float32)
        for l in range(sh.L):
            full = synth.trace(T + D, sh.E, sh.k, sh.zipf, sh.sticky, 0, l, 10000 + bl)
            lg2[:, l, 0] = synth.logits_from_picks(full[T:], sh.E, 0, l, 10000 + bl, 2)
        x2 = synth.normal_bf16_bits(D * sh.L * sh.H, 0, synth.PURPOSE_X, 77, D).reshape(D, sh.L, 1, sh.H)
        lg2_d = torch.from_numpy(lg2).cuda()
        x2_d = torch.from_numpy(x2.view(np.int16)).cuda().view(torch.bfloat16)
        o2 = torch.empty((sh.L, 1, sh.H), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        sa = cache.stats(-1)
        e0.record()
        for t in range(D):
            for l in range(sh.L):
                rc = fwd(cache.handle, l, ctypes.c_void_p(lg2_d[t, l].data_ptr()),
                         ctypes.c_void_p(x2_d[t, l].data_ptr()), 1, ctypes.c_void_p(o2[l].data_ptr()), sh_)
                if rc != 0:
                    raise moe.MoeError(rc, f"moe_layer_forward decode {t} layer {l}")
        e1.record()
        torch.cuda.synchronize()
        sb = cache.stats(-1)
        ph, pm = sb["pick_hits"] - sa["pick_hits"], sb["pick_misses"] - sa["pick_misses"]
        after = {"decode_tokens": D, "pick_hit_rate": ph / max(1, ph + pm),
                 "tokens_per_s": D / (e0.elapsed_time(e1) * 1e-3),
                 "note": "single tokens continuing the last batch's token streams, eager calls"}
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    d = {k2: st2[k2] - st1[k2] for k2 in ("pick_hits", "pick_misses", "unique_hits", "unique_misses")}
    dk = {k2: st3[k2] - st2[k2] for k2 in ("pick_hits", "pick_misses", "unique_hits", "unique_misses")}
    pairs_k = dk["pick_hits"] + dk["pick_misses"]
    flops_gu = pairs_k * 2.0 * 2 * sh.H * sh.F
    flops_dn = pairs_k * 2.0 * sh.H * sh.F
    g_gu = kt.get("gemm_gateup", {"ms": 0.0, "launches": 0})
    g_dn = kt.get("gemm_down", {"ms": 0.0, "launches": 0})
    ach = flops_gu / (g_gu["ms"] * 1e-3) / 1e12 if g_gu["ms"] else 0.0
    # algorithmic bytes: each distinct expert's matrices once per call, the
    # sorted activations in, the outputs out
    mat = sh.F * sh.H // 32 * 18
    uniq_k = dk["unique_hits"] + dk["unique_misses"]
    bytes_gu = uniq_k * 2 * mat + pairs_k * (sh.H * 2 + sh.F * 2)
    bytes_dn = uniq_k * mat + pairs_k * (sh.F * 2 + sh.H * 4)
    gbs_gu = bytes_gu / (g_gu["ms"] * 1e-3) / 1e9 if g_gu["ms"] else 0.0
    gbs_dn = bytes_dn / (g_dn["ms"] * 1e-3) / 1e9 if g_dn["ms"] else 0.0
    ridge = bf16_peak * 1e12 / (hbm_peak * 1e9)
    intensity = flops_gu / max(1, bytes_gu)
    tensor_bound = intensity > ridge
    roof = {"kernel": "gemm_gateup", "bound": "tensor" if tensor_bound else "hbm",
            "achieved": ach if tensor_bound else gbs_gu, "peak": bf16_peak if tensor_bound else hbm_peak,
            "unit": "TFLOP/s" if tensor_bound else "GB/s",
            "frac": ach / bf16_peak if tensor_bound else gbs_gu / hbm_peak, "traffic": None,
            "peak_source": peak_kind, "flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
            "tflops": ach, "tensor_frac": ach / bf16_peak, "hbm_gbs": gbs_gu, "hbm_frac": gbs_gu / hbm_peak,
            "launches": g_gu["launches"], "avg_launch_us": 1e3 * g_gu["ms"] / max(1, g_gu["launches"]),
            "down": {"tflops": flops_dn / (g_dn["ms"] * 1e-3) / 1e12 if g_dn["ms"] else 0.0,
                     "tensor_frac": (flops_dn / (g_dn["ms"] * 1e-3) / 1e12 / bf16_peak) if g_dn["ms"] else 0.0,
                     "hbm_gbs": gbs_dn, "hbm_frac": gbs_dn / hbm_peak, "launches": g_dn["launches"],
                     "avg_launch_us": 1e3 * g_dn["ms"] / max(1, g_dn["launches"])},
            "note": "algorithmic bytes: each distinct expert's Q4_0 matrices once per call plus the "
                    "pair-sorted activations and outputs; flops 2 x 2 x H x F per routed pair (gate/up)"}
    flops = (d["pick_hits"] + d["pick_misses"]) * 2.0 * 3 * sh.H * sh.F
    t_roof = (max(flops / (bf16_peak * 1e12), d["unique_hits"] * eb / (hbm_peak * 1e9)) +
              d["unique_misses"] * eb / (h2d_peak * 1e9))
    value = K * T / (ms * 1e-3)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": dict(prefill_config(sh, args.fill, T, args.gemm_min_tokens), policy=args.policy,
                           routing=args.routing),
            "hit_rate": {"pick": d["pick_hits"] / max(1, d["pick_hits"] + d["pick_misses"]),
                         "unique": d["unique_hits"] / max(1, d["unique_hits"] + d["unique_misses"])},
            "roofline": roof,
            "step_roofline": {"bound": "max(tensor, hbm) + h2d", "t_roof_ms": 1e3 * t_roof, "t_meas_ms": ms,
                              "frac": t_roof / (ms * 1e-3), "h2d_gbs": h2d_peak, "h2d_gbs_per_block": h2d_gbps,
                              "h2d_gbs_sustained": h2d_sus["one_copy"],
                              "tflop_per_batch": flops / K / 1e12},
            "kernels": {k2: {"launches": v["launches"], "ms": round(v["ms"], 3)} for k2, v in kt.items()
                        if v["launches"]},
            "clocks": clk, "host_store_node": node, "host_store_numa_pages": host_store_numa(store)}
    if after:
        line["after_prompt"] = after
    cache.close()
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ sweep
def run_sweep(args):
    """The staged/over-budget sweep: one layer of 128 experts (top-8, hidden
    2816, FFN 704, Q4_0 in host RAM), 64-token batches, fp32 activations, at
    slot budgets 8, 16, 32, 64 and 128 (below the ~60-126 distinct experts of
    a batch the calls run in stages), under uniform and Zipf(1.2) routing.
    One JSON line per (routing, budget): tokens/s over K timed batches after W
    warm-up batches (the first of them from an empty cache, reported as the
    cold start), hit rates, stages per call and the step roofline."""
    import torch

    import router_softmax_top_gb300 as moe
    sh = synth.SWEEP
    T, W, K = 64, max(3, args.warmup), max(1, min(args.steps, 64))
    torch.cuda.set_device(0)
    eb = sh.expert_bytes
    node = store_node(args, 0)
    store = host_store(sh.L * sh.E * eb, node, strict=args.store_node not in ("auto", "none"))
    synth.fill_store(store.data_ptr(), sh.L, sh.E, sh.H, sh.F, 0, args.threads)
    hbm_peak, _, peak_kind = measured_peaks()
    fill = moe.MOE_FILL_PULL if args.fill == "pull" else moe.MOE_FILL_MEMCPY
    fwd = moe.lib().moe_layer_forward
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out_d = torch.empty((T, sh.H), dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for routing, zipf in (("uniform", 0.0), ("zipf1.2", 1.2)):
        _, logits_h, x_h = synth.batch_inputs(sh, W + K, T, seed=0, zipf=zipf, sticky=0.0, act="f32")
        lg_d, x_d = torch.from_numpy(logits_h).cuda(), torch.from_numpy(x_h).cuda()
        for S in (8, 16, 32, 64, 128):
            cache = moe.MoECache(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                                 slots_per_layer=S, max_tokens=T, store=store, fill_mode=fill,
                                 timeout_us=60_000_000)
            h2d = max(cache.probe_h2d(8), probe_h2d_sustained(store, eb)["one_copy"])

            def run(b0, b1):
                for b in range(b0, b1):
                    rc = fwd(cache.handle, 0, ctypes.c_void_p(lg_d[b, 0].data_ptr()),
                             ctypes.c_void_p(x_d[b, 0].data_ptr()), T, ctypes.c_void_p(out_d.data_ptr()), stream)
                    if rc != 0:
                        raise moe.MoeError(rc, f"moe_layer_forward batch {b}")
            torch.cuda.synchronize()
            e0.record()
            run(0, 1)                               # cold: the first batch, empty cache
            e1.record()
            torch.cuda.synchronize()
            cold_ms = e0.elapsed_time(e1)
            run(1, W)
            torch.cuda.synchronize()
            s1 = cache.stats(0)
            e0.record()
            run(W, W + K)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            s2 = cache.stats(0)
            d = {k2: s2[k2] - s1[k2] for k2 in ("pick_hits", "pick_misses", "unique_hits", "unique_misses",
                                                  "stages", "staged_calls", "calls")}
            t_roof = d["unique_hits"] * eb / (hbm_peak * 1e9) + d["unique_misses"] * eb / (h2d * 1e9)
            line = {"metric": METRIC, "value": K * T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": K,
                    "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "dtype": "f32",
                    "data": "synthetic",
                    "config": {"workload": (f"sweep: 1 MoE layer, {sh.E} experts, top-{sh.k}, hidden {sh.H}, "
                                            f"expert FFN {sh.F}, Q4_0 in host RAM, {T} tokens per batch, "
                                            f"{S} slots, {routing} routing, fp32 activations"),
                               "slots_per_layer": S, "routing": routing, "tokens_per_step": T,
                               "fill_mode": args.fill},
                    "hit_rate": {"pick": d["pick_hits"] / max(1, d["pick_hits"] + d["pick_misses"]),
                                 "unique": d["unique_hits"] / max(1, d["unique_hits"] + d["unique_misses"])},
                    "stages_per_call": d["stages"] / max(1, d["calls"]),
                    "staged_calls": d["staged_calls"],
                    "distinct_experts_per_call": (d["unique_hits"] + d["unique_misses"]) / max(1, d["calls"]),
                    "cold_start": {"batches": 1, "tokens_per_s": T / (cold_ms * 1e-3)},
                    "step_roofline": {"bound": "hbm+h2d", "t_roof_ms": 1e3 * t_roof, "t_meas_ms": ms,
                                      "frac": t_roof / (ms * 1e-3), "hbm_gbs": hbm_peak, "h2d_gbs": h2d,
                                      "peak_source": peak_kind}}
            cache.close()
            print(json.dumps(line), flush=True)


# ------------------------------------------------------------ our arm
def main():
    args = resolve_defaults(parse())
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload == "prefill":
        run_prefill(args)
        return
    if args.workload == "sweep":
        run_sweep(args)
        return
    import torch
    import torch.distributed as dist

    import router_softmax_top_gb300 as moe

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    sh = synth.LARGE if args.workload == "large" else synth.DECODE
    T = args.batch if args.workload == "large" else 1
    assert 1 <= T <= 8, "decode steps of 1 to 8 tokens"
    if args.layers:
        import dataclasses
        sh = dataclasses.replace(sh, L=min(sh.L, args.layers))
    if args.slots:
        import dataclasses
        sh = dataclasses.replace(sh, S=min(sh.E, args.slots))
    W, K = args.warmup, args.steps
    assert W >= 3 and K >= 1
    t_setup = time.time()
    G0 = 2                        # graph warm-up steps (capture and first replays)
    nsteps = max(W + G0 + 3 * K, args.cpu_sample_steps)  # (the CPU baseline's sample too)
    eb = sh.expert_bytes
    node = store_node(args, local)
    if world > 1:
        # replicas of one model: one store per NUMA node, shared by its ranks
        store = shared_host_store(sh.L * sh.E * eb, node,
                                  lambda t: synth.fill_store(t.data_ptr(), sh.L, sh.E, sh.H, sh.F, 0, args.threads),
                                  f"{os.environ.get('MASTER_PORT', '0')}_{sh.L}x{sh.E}")
    else:
        store = host_store(sh.L * sh.E * eb, node, strict=args.store_node not in ("auto", "none"))
        synth.fill_store(store.data_ptr(), sh.L, sh.E, sh.H, sh.F, 0, args.threads)
    store_huge_kb = huge_page_kb()
    store_numa = host_store_numa(store)
    picks, logits_h, x_h = synth.decode_inputs(sh, nsteps, batch=T, seed=rank)
    logits_d = torch.from_numpy(logits_h).cuda()     # [steps, L, T, E]
    x_d = torch.from_numpy(x_h).cuda()               # [steps, L, T, H]
    out_d = torch.empty((sh.L, T, sh.H), dtype=torch.float32, device="cuda")
    fill = moe.MOE_FILL_PULL if args.fill == "pull" else moe.MOE_FILL_MEMCPY
    policy = {"lru": moe.MOE_POLICY_LRU, "score": moe.MOE_POLICY_SCORE, "adopt": moe.MOE_POLICY_ADOPT}[args.policy]
    cache = moe.MoECache(n_layers=sh.L, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                         slots_per_layer=sh.S, max_tokens=T, store=store, fill_mode=fill,
                         timeout_us=30_000_000, policy=policy, admit_budget=args.admit_budget,
                         sticky_permille=args.sticky)
    preload = None
    if args.preload_profile:
        # usage counts from another token stream (same routing: same seed and layer)
        counts = np.zeros((sh.L, sh.E), np.uint32)
        for l in range(sh.L):
            pp = synth.trace(args.preload_profile, sh.E, sh.k, sh.zipf, sh.sticky, rank, l, PROFILE_STREAM)
            np.add.at(counts[l], pp.reshape(-1), 1)
        t0 = time.time()
        cache.preload(counts)
        preload = {"profile_tokens": args.preload_profile, "stream": PROFILE_STREAM,
                   "experts": int(np.minimum((counts > 0).sum(1), sh.S).sum()),
                   "s": time.time() - t0}
    elif args.preload_from_session:
        # the previous session: its own handle, the other token stream, then
        # its lifetime usage counts are what this session preloads
        n = args.preload_from_session
        if T != 1:
            raise SystemExit("--preload-from-session: one token per step (decode workloads at batch 1)")
        prev = moe.MoECache(n_layers=sh.L, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                            slots_per_layer=sh.S, max_tokens=T, store=store, fill_mode=fill,
                            timeout_us=30_000_000)
        lg_prev = torch.from_numpy(np.stack([synth.logits_from_picks(
            synth.trace(n, sh.E, sh.k, sh.zipf, sh.sticky, rank, l, PROFILE_STREAM), sh.E, rank, l,
            PROFILE_STREAM, 0) for l in range(sh.L)], axis=1)).cuda()          # [n, L, E]
        x_prev = torch.zeros((sh.L, T, sh.H), dtype=torch.float32, device="cuda")
        out_prev = torch.empty((T, sh.H), dtype=torch.float32, device="cuda")
        for s_ in range(n):
            for l in range(sh.L):
                prev.forward(l, lg_prev[s_, l].view(T, sh.E), x_prev[l], out=out_prev)
        counts = prev.usage()
        prev_stats = prev.stats(-1)
        prev.close()
        t0 = time.time()
        cache.preload(counts)
        preload = {"session_tokens": n, "stream": PROFILE_STREAM, "counts_sum": int(counts.sum()),
                   "session_pick_hit_rate": prev_stats["pick_hits"] / max(1, prev_stats["pick_hits"] +
                                                                       prev_stats["pick_misses"]),
                   "experts": int(np.minimum((counts > 0).sum(1), sh.S).sum()), "s": time.time() - t0}
    setup_s = time.time() - t_setup
    h2d_gbps = cache.probe_h2d(24)
    h2d_sus = probe_h2d_sustained(store, eb)
    h2d_sustained = h2d_sus["one_copy"]
    L = moe.lib()
    fwd = L.moe_layer_forward
    handle = cache.handle
    stream = torch.cuda.current_stream()
    sh_ = ctypes.c_void_p(stream.cuda_stream)
    lg_ptr = [[ctypes.c_void_p(logits_d[s, l].data_ptr()) for l in range(sh.L)] for s in range(nsteps)]
    x_ptr = [[ctypes.c_void_p(x_d[s, l].data_ptr()) for l in range(sh.L)] for s in range(nsteps)]
    o_ptr = [ctypes.c_void_p(out_d[l].data_ptr()) for l in range(sh.L)]

    def run_steps(s0, s1):
        for s in range(s0, s1):
            lp, xp = lg_ptr[s], x_ptr[s]
            for l in range(sh.L):
                rc = fwd(handle, l, lp[l], xp[l], T, o_ptr[l], sh_)
                if rc != 0:
                    raise moe.MoeError(rc, f"moe_layer_forward step {s} layer {l}")

    # ---- cold start: the first WC steps from an empty cache (the start of the
    # warm-up; the rest of it runs below, untimed: on shared machines a
    # process's first seconds of host-link reads are sometimes much slower)
    WC = min(COLD_STEPS, W)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st0 = cache.stats(-1)
    e0.record()
    run_steps(0, WC)
    e1.record()
    torch.cuda.synchronize()
    cold_ms = e0.elapsed_time(e1)
    st1 = cache.stats(-1)

    # ---- one step (all layer calls) captured as a CUDA graph: the timed region
    # replays it, each step's inputs copied into the captured input buffers
    # (device to device); the pull-fill single-token schedule has no host wait
    graph = None
    launches_per_step = None
    if not args.no_graph and fill == moe.MOE_FILL_PULL:
        lg_cur = torch.empty((sh.L, T, sh.E), dtype=torch.float32, device="cuda")
        x_cur = torch.empty((sh.L, T, sh.H), dtype=torch.float32, device="cuda")
        lc = [ctypes.c_void_p(lg_cur[l].data_ptr()) for l in range(sh.L)]
        xc = [ctypes.c_void_p(x_cur[l].data_ptr()) for l in range(sh.L)]
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        torch.cuda.synchronize()
        n0 = cache.launch_count()
        with torch.cuda.graph(graph, stream=cap):
            cs = ctypes.c_void_p(cap.cuda_stream)
            for l in range(sh.L):
                rc = fwd(handle, l, lc[l], xc[l], T, o_ptr[l], cs)
                if rc != 0:
                    raise moe.MoeError(rc, f"moe_layer_forward (capture) layer {l}")
        launches_per_step = cache.launch_count() - n0

        def run_graph(s0, s1):
            for s in range(s0, s1):
                lg_cur.copy_(logits_d[s], non_blocking=True)
                x_cur.copy_(x_d[s], non_blocking=True)
                graph.replay()
        run_graph(WC, W + G0)
    else:
        run_steps(WC, W + G0)
    torch.cuda.synchronize()
    st1t = cache.stats(-1)    # baseline of the timed region
    W1 = W + G0

    # ---- timed region: K steps, inputs resident in HBM
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    n_launch0 = cache.launch_count()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    e0.record()
    for i in range(K):
        step_ev[i].record()
        if graph is not None:
            run_graph(W1 + i, W1 + i + 1)
        else:
            run_steps(W1 + i, W1 + i + 1)
    step_ev[K].record()
    e1.record()
    torch.cuda.synchronize()
    barrier()
    stalls = step_stalls([step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(K)])
    n_launch = (launches_per_step * K if graph is not None else cache.launch_count() - n_launch0)
    dev_ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    st2 = cache.stats(-1)
    # the host link again right after the timed region: a drop against the probe
    # before it means the link (or the host memory behind it) slowed down during
    # the run, which the step's time then carries
    h2d_gbps_after = cache.probe_h2d(24)

    # ---- per-kernel pass: the next K steps again with CUDA events around every
    # launch (on the stream each kernel runs on); kept out of the headline
    kpass_ms = 0.0
    if not args.no_kernel_pass:
        cache.set_timing(True)
        e0.record()
        run_steps(W1 + K, W1 + 2 * K)
        e1.record()
        torch.cuda.synchronize()
        kpass_ms = e0.elapsed_time(e1)
    ktime = cache.timing()
    cache.set_timing(False)
    st3 = cache.stats(-1)

    # ---- e2e: same metric through the C ABI with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        lg_pin = torch.from_numpy(logits_h).pin_memory()
        x_pin = torch.from_numpy(x_h).pin_memory()
        out_pin = torch.empty((K, sh.L, T, sh.H), dtype=torch.float32, pin_memory=True)
        lg_step = torch.empty((sh.L, T, sh.E), dtype=torch.float32, device="cuda")
        x_step = torch.empty((sh.L, T, sh.H), dtype=torch.float32, device="cuda")
        lg_sp = [ctypes.c_void_p(lg_step[l].data_ptr()) for l in range(sh.L)]
        x_sp = [ctypes.c_void_p(x_step[l].data_ptr()) for l in range(sh.L)]
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i, s in enumerate(range(W1 + 2 * K, W1 + 3 * K)):
            if graph is not None:
                # the step's moe_layer_forward calls as captured through the C ABI,
                # replayed; this step's inputs copied from pinned host memory into
                # the buffers they read
                lg_cur.copy_(lg_pin[s], non_blocking=True)
                x_cur.copy_(x_pin[s], non_blocking=True)
                graph.replay()
            else:
                lg_step.copy_(lg_pin[s], non_blocking=True)
                x_step.copy_(x_pin[s], non_blocking=True)
                for l in range(sh.L):
                    rc = fwd(handle, l, lg_sp[l], x_sp[l], T, o_ptr[l], sh_)
                    if rc != 0:
                        raise moe.MoeError(rc, "moe_layer_forward (e2e)")
            out_pin[i].copy_(out_d, non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        e2e_s = time.perf_counter() - t0
        e2e = {"value": K * T / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": int(lg_step.numel() * 4 + x_step.numel() * 4),
               "d2h_bytes_per_step": int(out_d.numel() * 4),
               "ms_per_step": 1e3 * e2e_s / K,
               "calls": "replayed CUDA graph of the C-ABI calls" if graph is not None else "direct C-ABI calls"}

    # ---- aggregate over ranks
    dev_ms_max, value, e2e_value = aggregate_over_ranks(dev_ms, e2e["ms_per_step"] if e2e else None, K,
                                                        world, "cuda", T)
    if e2e is not None:
        e2e["value"] = e2e_value

    # ---- roofline of the dominant kernel and of the whole step
    hbm_peak, _, peak_kind = measured_peaks()
    d = {key: st2[key] - st1t[key] for key in st2 if key not in ("poisoned", "last_error")}
    dk = {key: st3[key] - st2[key] for key in st3 if key not in ("poisoned", "last_error")}
    uniq = d["unique_hits"] + d["unique_misses"]
    uniq_k = dk["unique_hits"] + dk["unique_misses"]
    picks_k = dk["pick_hits"] + dk["pick_misses"]
    mat = sh.F * sh.H // 32 * 18                      # one Q4_0 matrix (gate, up or down)
    kinds = {k2: v for k2, v in ktime.items() if v["launches"] > 0 and k2 != "h2d_memcpy"}
    dom = max(kinds, key=lambda k2: kinds[k2]["ms"]) if kinds else "q4_gateup_gemv"
    gu = ktime.get("q4_gateup_gemv", {"launches": 0, "ms": 0.0})
    dn = ktime.get("q4_down_gemv", {"launches": 0, "ms": 0.0})
    # algorithmic bytes: every distinct expert of a call read once; activations in, results out
    gu_bytes = uniq_k * 2 * mat + picks_k * (sh.H * 4 + sh.F * 4)
    dn_bytes = uniq_k * mat + picks_k * (sh.F * 4 + 4) + sh.H * 4 * picks_k // sh.k
    kb = {"q4_gateup_gemv": (gu_bytes, gu), "q4_down_gemv": (dn_bytes, dn)}
    # HBM-bound kernel with the most time (gate/up of the experts in HBM)
    rk = max(kb, key=lambda k2: kb[k2][1]["ms"])
    alg_bytes, kt = kb[rk]
    achieved = alg_bytes / (kt["ms"] * 1e-3) / 1e9 if kt["ms"] > 0 else 0.0
    per_launch = alg_bytes / max(1, kt["launches"])
    ratio = profiled_traffic_ratio(rk)
    roofline_hbm = {"kernel": rk, "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                    "unit": "GB/s", "frac": achieved / hbm_peak,
                    "traffic": per_launch * ratio if ratio else None,
                    "peak_source": peak_kind, "launches": kt["launches"],
                    "avg_launch_us": 1e3 * kt["ms"] / max(1, kt["launches"]),
                    "alg_bytes_per_launch": per_launch}
    # the host link's peak: the larger of the per-block probe and the sustained
    # (64-block) copy, both measured in this run
    h2d_peak = max(h2d_gbps, h2d_sustained)
    peak_src = ("measured in this run: the larger of the median cudaMemcpyAsync of one expert block "
                "(h2d_gbs_per_block) and one 64-block copy (h2d_gbs_sustained) from the host store")
    # the kernel with the most time overall: the fused miss kernel, bound by the host link
    fm = ktime.get("fused_miss", {"launches": 0, "ms": 0.0})
    miss_bytes_k = dk["unique_misses"] * sh.expert_bytes
    if fm["ms"] > 0 and fm["ms"] >= kt["ms"]:
        ach = miss_bytes_k / (fm["ms"] * 1e-3) / 1e9
        roofline = {"kernel": "fused_miss", "bound": "h2d", "achieved": ach, "peak": h2d_peak,
                    "unit": "GB/s", "frac": ach / h2d_peak, "frac_per_block": ach / h2d_gbps, "traffic": None,
                    "peak_source": peak_src,
                    "launches": fm["launches"], "avg_launch_us": 1e3 * fm["ms"] / max(1, fm["launches"]),
                    "alg_bytes_per_launch": miss_bytes_k / max(1, fm["launches"])}
    else:
        roofline = roofline_hbm
    # pull fill: the whole layer runs in the decode layer kernel, whose misses
    # cross the host link while its hits are read from HBM alongside
    dl = ktime.get("decode_layer", {"launches": 0, "ms": 0.0})
    alu = None
    if dl["ms"] > 0:
        hit_b = dk["unique_hits"] * sh.expert_bytes
        per = 1.0 / max(1, dl["launches"])
        ach = miss_bytes_k / (dl["ms"] * 1e-3) / 1e9
        ratio = profiled_traffic_ratio("decode_layer")
        roofline = {"kernel": "decode_layer", "bound": "h2d", "achieved": ach, "peak": h2d_peak,
                    "unit": "GB/s", "frac": ach / h2d_peak, "frac_per_block": ach / h2d_gbps, "traffic": None,
                    "peak_source": peak_src,
                    "launches": dl["launches"], "avg_launch_us": 1e3 * dl["ms"] * per,
                    "alg_bytes_per_launch": miss_bytes_k * per,
                    "note": "bytes of the missed expert blocks over the host link per launch / launch time; "
                            "traffic null: DRAM counters do not see the host link (the kernel's DRAM bytes, "
                            "its hit blocks, are roofline_hbm.traffic)"}
        hbm_alg = hit_b + miss_bytes_k + picks_k * (2 * sh.H * 4 + 3 * sh.F * 4)
        roofline_hbm = {"kernel": "decode_layer", "bound": "hbm", "achieved": hbm_alg / (dl["ms"] * 1e-3) / 1e9,
                        "peak": hbm_peak, "unit": "GB/s",
                        "frac": hbm_alg / (dl["ms"] * 1e-3) / 1e9 / hbm_peak,
                        "traffic": hit_b * per * ratio if ratio else None, "peak_source": peak_kind,
                        "launches": dl["launches"], "avg_launch_us": 1e3 * dl["ms"] * per,
                        "alg_bytes_per_launch": hbm_alg * per,
                        "note": "HBM side of the same kernel: hit blocks read, missed blocks written to "
                                "their slots, activations and results; it overlaps the host-link reads. "
                                "traffic: DRAM read + write per launch from the committed capture's DRAM "
                                "bytes per hit-block byte (the slot writes stayed in L2 there)"}
        # ALU budget: instructions per weight (the committed capture's count, spin
        # waits included) x weights per second, against the issue rate of all SMs
        ent = profiled_entry("decode_layer")
        ipw = ent.get("warp_inst_per_weight") if ent else None
        weights = (hit_b + miss_bytes_k) / sh.expert_bytes * 3 * sh.H * sh.F
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        mhz = (clk or {}).get("sm_mhz") or (clk or {}).get("sm_max_mhz")
        alu_peak = sms * 4 * mhz * 1e6 / 1e9 if mhz else None
        alu_ach = ipw * weights / (dl["ms"] * 1e-3) / 1e9 if ipw else None
        alu = {"kernel": "decode_layer", "bound": "alu", "unit": "Gwarp-inst/s", "achieved": alu_ach,
               "peak": alu_peak, "frac": alu_ach / alu_peak if alu_ach and alu_peak else None,
               "warp_inst_per_weight": ipw, "weights_per_launch": weights * per,
               "peak_source": f"{sms} SMs x 4 schedulers x 1 warp-instruction per cycle x the median SM "
                              "clock sampled in the timed region",
               "note": "instructions per weight: smsp__inst_executed.sum over the weights of the committed "
                       "capture's launches (profiles/decode_layer_kernel.md), waits included; null once the "
                       "kernel changed"}
    t_roof = (d["unique_hits"] * sh.expert_bytes / (hbm_peak * 1e9) +
              d["unique_misses"] * sh.expert_bytes / (h2d_peak * 1e9))
    t_roof_pb = (d["unique_hits"] * sh.expert_bytes / (hbm_peak * 1e9) +
                 d["unique_misses"] * sh.expert_bytes / (h2d_gbps * 1e9))
    t_roof_strict = t_roof + d["unique_misses"] * sh.expert_bytes / (hbm_peak * 1e9)
    step_roof = {"bound": "hbm+h2d", "t_roof_ms": 1e3 * t_roof, "t_meas_ms": dev_ms,
                 "frac": t_roof / (dev_ms * 1e-3), "frac_per_block": t_roof_pb / (dev_ms * 1e-3),
                 "frac_strict": t_roof_strict / (dev_ms * 1e-3),
                 "hbm_gbs": hbm_peak, "h2d_gbs": h2d_peak, "h2d_gbs_per_block": h2d_gbps,
                 "h2d_gbs_sustained": h2d_sustained, "h2d_gbs_back_to_back": h2d_sus["back_to_back"],
                 "h2d_gbs_after": h2d_gbps_after,
                 "hit_bytes": d["unique_hits"] * sh.expert_bytes,
                 "miss_bytes": d["unique_misses"] * sh.expert_bytes}
    picks_t = d["pick_hits"] + d["pick_misses"]
    cold = {k2: st1[k2] - st0[k2] for k2 in ("pick_hits", "pick_misses", "unique_hits", "unique_misses")}
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": dev_ms_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(sh, args.fill, T), policy=args.policy,
                       **({"admit_budget": args.admit_budget, "sticky_permille": args.sticky}
                          if args.policy == "score" else {})),
        "hit_rate": {"pick": d["pick_hits"] / max(1, picks_t),
                     "unique": d["unique_hits"] / max(1, uniq),
                     "evictions_per_call": d["evictions"] / max(1, d["calls"]),
                     "bypassed_per_call": d["bypassed"] / max(1, d["calls"])},
        "cold_start": {"steps": WC, "tokens_per_s": WC * T / (cold_ms * 1e-3),
                       "pick_hit_rate": cold["pick_hits"] / max(1, cold["pick_hits"] + cold["pick_misses"]),
                       "preload": preload},
        "achieved_hbm_gbs_step": (d["unique_hits"] + d["unique_misses"]) * sh.expert_bytes / (dev_ms * 1e-3) / 1e9,
        "roofline": roofline,
        "roofline_hbm": roofline_hbm,
        "roofline_alu": alu,
        "step_roofline": step_roof,
        "steps_timed": stalls,
        "kernels": {k2: {"launches": v["launches"], "ms": round(v["ms"], 4)} for k2, v in ktime.items()
                    if v["launches"]},
        "kernel_pass_ms_per_step": kpass_ms / K,
        "gpu_launches": int(n_launch),
        "step_graph": graph is not None,
        "host_store_huge_fraction": (None if store_huge_kb is None
                                     else min(1.0, store_huge_kb * 1024 / sh.store_bytes)),
        "host_store_numa_pages": store_numa,
        "host_store_node": node,
        "clocks": clk,
        "e2e": e2e,
        "setup_s": setup_s,
    }
    # ---- CPU baseline: the oracle as it stands on a bounded sample (rank 0, N = 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the large model's steps cost the oracle ~9x (T = 1) and ~70x (T = 8) a
        # decode step: fewer of them keep the sample near 15 s
        cap = args.cpu_sample_steps if sh.name == "decode" else max(1, 24 // T)
        n = max(1, min(cap, logits_h.shape[0]))
        v, dt, cores = run_oracle_sample(sh, store.numpy(), logits_h, x_h, n, args.threads)
        tok = "one token" if T == 1 else f"{T} tokens"
        result["cpu_baseline"] = {"value": v * T, "unit": UNIT, "cores": cores, "kind": "oracle",
                                  "sample": f"first {n} decode steps ({tok} through all {sh.L} "
                                            f"layers, outputs computed) from a cold cache; {dt:.1f} s",
                                  "cpu_model": host_cpu_model()}
        if T == 1:
            n1 = min(2, n)
            v1, dt1, _ = run_oracle_sample(sh, store.numpy(), logits_h, x_h, n1, 1)
            result["cpu_baseline"].update(value_1thread=v1,
                                          sample_1thread=f"first {n1} decode steps on one thread; {dt1:.1f} s")
    cache.close()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
