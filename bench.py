#!/usr/bin/env python
"""Benchmark of the sparse offloaded-KV decode step on one GB300 (or N replicas).

A step is one whole decode step of a workload: every layer runs landmark top-k
selection, the predicted-vs-needed diff, the coalesced host->HBM gather into
the two-layer ping-pong buffer (prefetch two layers ahead, urgent misses) and
GQA attention with the log-sum-exp window merge, all inside libkvo's CUDA
kernels.  Inputs are seeded synthetic data of the workload's shapes; the KV
cache lives in pinned host memory.

The headline (``value``) is the Llama-3-8B-shaped workload (32 layers).  The
same run then measures the three stress workloads (long context with a
speculative query and urgent misses, wide budget, token-granular
fragmentation) the same way and reports every workload's step time against
its roofline in ``workloads``.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on the host cores instead (the reference arm: no GPU code on that path).
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import contextlib  # noqa: E402
import ctypes  # noqa: E402
import gc  # noqa: E402
import glob  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import platform  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sparse_kv_cache_landmark_gb300 import synth  # noqa: E402
from sparse_kv_cache_landmark_gb300.workloads import SPEC_SIGMA_88, WORKLOADS  # noqa: E402

METRIC = "sparse decode steps/s and effective KV GB/s (1 GB300) as % of HBM/PCIe roofline"
UNIT = "steps/s"
# the stress workloads measured after the headline one (the roofline target covers all four)
EXTRA_WORKLOADS = "long_ctx_predict,wide_budget,fragmentation"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_decode")
    ap.add_argument("--workloads", default=EXTRA_WORKLOADS,
                    help="further workloads measured after the headline one, comma-separated ('' for none)")
    ap.add_argument("--extra-steps", type=int, default=10, help="timed steps of each further workload")
    ap.add_argument("--seed", type=int, default=1235)
    ap.add_argument("--host-layers", type=int, default=0, help="distinct host layers (0: all that fit)")
    ap.add_argument("--cpu-sample-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=60.0,
                    help="reference arm: oracle seconds spread over the timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling runs)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs)")
    ap.add_argument("--gather-ctas", type=int, default=0, help="gather kernel CTAs (0: library default)")
    ap.add_argument("--gather-threads", type=int, default=0, help="gather threads per CTA (0: library default)")
    ap.add_argument("--gather-engine", type=int, default=-1,
                    help="0 lane loads, 1/2 TMA bulk copies, 3 flat lane loads, 4 copy engine (-1: default)")
    ap.add_argument("--gather-drivers", type=int, default=0, help="TMA engine driver warps (0: default)")
    ap.add_argument("--gather-reserve", type=int, default=-1, help="flat engine smem reservation per CTA (bytes)")
    ap.add_argument("--graphs", type=int, default=-1, help="1: replay warm steps from CUDA graphs (-1: default)")
    ap.add_argument("--append", type=int, default=0,
                    help="grow the cache: one kvo_append before every decode step (reserves this many tokens)")
    ap.add_argument("--gather-unroll", type=int, default=0, help="gather loads in flight per lane (0: default)")
    ap.add_argument("--attn-impl", type=int, default=-1,
                    help="attention kernel: 0 register-direct, 1 TMA-staged persistent (-1: default)")
    ap.add_argument("--attn-ctas", type=int, default=0, help="TMA-staged attention grid (0: fill the SMs)")
    ap.add_argument("--select-impl", type=int, default=-1,
                    help="selection kernel: 0 ticket, 2 one cluster per group where it fits, 1 automatic "
                         "(-1: default)")
    ap.add_argument("--resident", type=int, default=0,
                    help="1: cross-step delta prefetch (per-layer resident block sets), queries drifting per step; "
                         "2: the resident sets without speculation (each step fetches only its misses)")
    ap.add_argument("--drift", type=float, default=-1.0,
                    help="per-step query drift with --resident (default: the speculative noise / sqrt(2))")
    ap.add_argument("--query-steps", type=int, default=8, help="distinct step queries cycled with --resident")
    ap.add_argument("--reconstruct", type=int, default=-1,
                    help="rebuild missed keys from low-rank factors (1/0; -1: on for low-rank workloads)")
    ap.add_argument("--prefetch-budget", type=int, default=-1,
                    help="with --resident: prefetch fetches admitted per group, layer and step (-1: all)")
    ap.add_argument("--spec-policy", type=int, default=-1,
                    help="with --resident 1: 1 prefetches a layer's prediction only while it pays (the default "
                         "here), 0 always")
    ap.add_argument("--gather-engines", default="",
                    help="also time an isolated gather of layer 0's true index with each listed engine "
                         "(e.g. 3,4) and report it under gather_engines")
    ap.add_argument("--trace", default="",
                    help="write the launch trace (kind, layer, start, end) of one profiled step to this JSON file")
    return ap.parse_args(argv)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# DRAM bytes per launch of the default gather kernel from one ncu capture of a
# 134.2 MB prefetch launch of the Llama-shaped workload; reported only for the
# launch shape and workload it was taken on.
NCU_TRAFFIC = {("llama3_8b_decode", "gather_flat_kernel"): 72.811264e6 + 51.968e3}


def workload_bytes(w, lens, misses_per_step=0, fetched_per_step=None, recon_rank=0):
    """Algorithmic bytes of one step (all layers): HBM and host link.

    ``misses_per_step``: blocks fetched by the urgent stream per step (summed
    over layers and groups) on top of the k prefetched blocks per group.
    ``fetched_per_step`` (resident block sets): all blocks fetched per step,
    replacing the k per group and the misses.
    ``recon_rank`` > 0: missed keys are rebuilt on the GPU from rank-R factors,
    so misses move V only over the link and read R coefficients per token.
    """
    G, d, k, B, W, L = w.batch * w.n_kv_heads, w.head_dim, w.top_k, w.block_size, w.window, w.n_layers
    tok = 4 * d                                             # K+V bf16 bytes per token per KV head
    C = [(n - W) // B for n in lens]
    lm_bytes = sum(C) * w.n_kv_heads * d * (4 if B > 1 else 2)
    gathered = G * k * B * tok                              # written to the ping-pong half
    attended = G * (k * B + W) * tok                        # read by attention
    q_bytes = w.batch * w.n_q_heads * d * 2 * 3             # select (2x) + attention
    out_bytes = w.batch * w.n_q_heads * (d + 1) * 4
    meta = G * k * 4 * 8
    urgent = misses_per_step * B * tok
    urgent_host = urgent if not recon_rank else misses_per_step * B * tok // 2
    if recon_rank:
        urgent += misses_per_step * B * recon_rank * 2          # coefficients read by the rebuild
    hbm = (lm_bytes + gathered + attended + q_bytes + out_bytes + meta) * L + urgent
    host = gathered * L + urgent_host
    if fetched_per_step is not None:
        moved = fetched_per_step * B * tok
        hbm = (lm_bytes + attended + q_bytes + out_bytes + meta) * L + moved
        host = moved
        gathered = moved / (2 * L)      # per prefetch launch, split evenly between the two streams
    kv_attended = attended * L
    return {"hbm": hbm, "host": host, "kv_attended": kv_attended, "gather_per_launch": gathered, "urgent": urgent,
            "landmark_per_layer": lm_bytes, "attended_per_layer": attended}


# ------------------------------------------------------------ host and GPU ids
def host_info():
    """Host cores and CPU model (the CPU baseline runs on them)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown", "machine": platform.machine(),
            "numa_nodes": len(cpu_numa_nodes())}


def smi_gpu_id(local: int) -> str:
    """nvidia-smi's id of CUDA device ``local``: its UUID (nvidia-smi numbers GPUs
    in PCI order and ignores CUDA_VISIBLE_DEVICES, so an index may name another
    GPU), else its PCI bus id, else the index."""
    try:
        p = torch.cuda.get_device_properties(local)
    except Exception:
        return str(local)
    u = getattr(p, "uuid", None)
    if u is not None:
        s = str(u).strip()
        if s:
            return s if s.startswith("GPU-") else "GPU-" + s
    bus, dev, dom = (getattr(p, a, None) for a in ("pci_bus_id", "pci_device_id", "pci_domain_id"))
    if bus is not None and dev is not None:
        return f"{dom or 0:08x}:{bus:02x}:{dev:02x}.0"
    return str(local)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(dev)], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            self.f.close()
            os.unlink(self.f.name)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        self.f.close()
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ NUMA placement
def cpu_numa_nodes():
    """NUMA nodes of this host that have CPUs (memory-only nodes, such as a
    GPU's own memory exposed as a node, are left out)."""
    base = "/sys/devices/system/node"
    out = []
    for p in sorted(glob.glob(os.path.join(base, "node[0-9]*"))):
        try:
            with open(os.path.join(p, "cpulist")) as f:
                if f.read().strip():
                    out.append(int(os.path.basename(p)[4:]))
        except (OSError, ValueError):
            pass
    return out or [0]


_SYS = {"aarch64": {"set_mempolicy": 237, "move_pages": 239}, "x86_64": {"set_mempolicy": 238, "move_pages": 279}}


def _set_mempolicy(mode: int, node: int = -1) -> bool:
    """set_mempolicy(2) for the calling thread: mode 0 default, 2 bind to ``node``."""
    nr = _SYS.get(platform.machine(), {}).get("set_mempolicy")
    if nr is None:
        return False
    libc = ctypes.CDLL(None, use_errno=True)
    if mode == 0:
        return libc.syscall(nr, 0, None, 0) == 0
    mask = (ctypes.c_ulong * 16)()
    mask[node // 64] = 1 << (node % 64)
    return libc.syscall(nr, mode, mask, 16 * 64 + 1) == 0


@contextlib.contextmanager
def numa_bind(node):
    """Host pages allocated (and pinned) inside come from NUMA node ``node``
    (None: the default policy).  Host-side placement only."""
    ok = node is not None and _set_mempolicy(2, node)
    try:
        yield ok
    finally:
        if ok:
            _set_mempolicy(0)


def page_node(ptr: int) -> int:
    """NUMA node holding the page at host address ``ptr`` (-1 if unknown)."""
    nr = _SYS.get(platform.machine(), {}).get("move_pages")
    if nr is None:
        return -1
    libc = ctypes.CDLL(None, use_errno=True)
    pages = (ctypes.c_void_p * 1)(ptr)
    status = (ctypes.c_int * 1)(-1)
    if libc.syscall(nr, 0, 1, pages, None, status, 0) != 0:
        return -1
    return int(status[0])


def gpu_host_numa_node(local: int):
    """Host NUMA node nearest to CUDA device ``local`` (cudaDevAttrHostNumaId), or None."""
    handles = []
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            handles.append(ctypes.CDLL(name))
        except OSError:
            pass
    for p in glob.glob("/usr/local/cuda/lib64/libcudart.so*"):
        try:
            handles.append(ctypes.CDLL(p))
        except OSError:
            pass
    for h in handles:
        v = ctypes.c_int(-1)
        try:
            if h.cudaDeviceGetAttribute(ctypes.byref(v), 134, local) == 0:
                return v.value if v.value >= 0 else None
        except AttributeError:
            continue
    return None


def free_host_cache():
    """Return cached pinned blocks to the OS (torch keeps freed pinned memory)."""
    gc.collect()
    fn = getattr(torch._C, "_host_emptyCache", None)
    if fn is not None:
        fn()


def probe_link(local, stream, nbytes=1 << 30, n_streams=(1, 2, 4), reps=3):
    """Pinned host -> device copy bandwidth (GB/s): 1, 2 and 4 streams copying
    their own 1 GiB buffers at once, best of ``reps``, for the pinned buffers
    placed by the default policy and on each CPU NUMA node (the GPU's nearest
    first, at most two)."""
    nodes = cpu_numa_nodes()
    near = gpu_host_numa_node(local)
    order = ([near] if near in nodes else []) + [n for n in nodes if n != near]
    placements = [None] + order[:2]
    out = {"numa_nodes": nodes, "gpu_nearest_node": near, "placements": {}}
    best = 0.0
    for node in placements:
        key = "default" if node is None else f"node{node}" + (" (nearest)" if node == near else "")
        with numa_bind(node) as bound:
            hs = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(max(n_streams))]
        if node is not None and not bound:
            out["placements"][key] = {"error": "set_mempolicy failed"}
            del hs
            continue
        ds = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in hs]
        ss = [torch.cuda.Stream() for _ in hs]
        res = {"page_node": page_node(hs[0].data_ptr())}
        for ns in n_streams:
            bw = 0.0
            for _ in range(reps):
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for i in range(ns):
                    ss[i].wait_event(a)
                    with torch.cuda.stream(ss[i]):
                        ds[i].copy_(hs[i], non_blocking=True)
                for i in range(ns):
                    stream.wait_stream(ss[i])
                b.record(stream)
                b.synchronize()
                bw = max(bw, ns * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
            res[f"{ns}_streams"] = bw
            best = max(best, bw)
        out["placements"][key] = res
        del hs, ds, ss
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        free_host_cache()
    out["best_pinned_memcpy"] = best
    out["placement_used"] = "nearest node" if near is not None else "default"
    return out


# --------------------------------------------------------------- ranks
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, x: float) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle
def oracle_sample(w, seed, budget_s, layers=1):
    """Time the fp64 oracle (as it stands) on whole (request, KV head) groups.

    Generates request 0 of layer 0 on the CPU and runs the oracle's per-group
    step (landmarks, scores, top-k, diff, runs, attention + merge) on its KV
    heads until ``budget_s`` seconds of oracle time have passed.
    Returns (seconds per group, groups timed).
    """
    import oracle as orc
    lens = synth.seq_lens(w, seed)
    q, qs = synth.gen_queries(w, seed, 0)
    K, V = synth.gen_request_kv(w, seed, 0, 0, lens[0], q[0])
    r = w.group_size
    times = []
    t_start = time.perf_counter()
    g = 0
    while time.perf_counter() - t_start < budget_s or not times:
        gg = g % w.n_kv_heads
        t0 = time.perf_counter()
        orc.decode_group(synth.bits(K[gg]), synth.bits(V[gg]), synth.bits(q[0, gg * r:(gg + 1) * r]),
                         None if qs is None else synth.bits(qs[0, gg * r:(gg + 1) * r]),
                         block_size=w.block_size, top_k=w.top_k, window=w.window)
        times.append(time.perf_counter() - t0)
        g += 1
    return sum(times) / len(times), len(times)


def run_reference(args):
    ws, rank, _ = dist_setup(args)
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    if args.layers:
        w = w.scaled(n_layers=args.layers)
    if args.batch:
        w = w.scaled(batch=args.batch)
    G = w.batch * w.n_kv_heads
    per_step_groups = G * w.n_layers
    # each bench step: one bounded sample of groups; the step time is scaled
    # to the whole workload step (G groups x n_layers layers)
    import oracle as orc  # noqa: F401  (the reference arm runs the oracle only)
    for _ in range(args.warmup):
        oracle_sample(w, args.seed, 0.0)
    step_s = []
    sample_budget = max(0.2, args.ref_budget_s / max(1, args.steps))
    n_groups = 0
    for _ in range(args.steps):
        t_group, n = oracle_sample(w, args.seed, sample_budget)
        step_s.append(t_group * per_step_groups)
        n_groups += n
    t = statistics.mean(step_s)
    v = 1.0 / t
    host = host_info()
    sample = (f"fp64 numpy oracle on {n_groups} (request, KV head) groups of layer 0 over {args.steps} bench "
              f"steps, scaled to {per_step_groups} groups per decode step; one thread of {host['nproc']} "
              f"({host['cpu_model']})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "context": w.ctx[0], "block": w.block_size, "top_k": w.top_k,
                   "window": w.window, "layers": w.n_layers},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                         "host": host},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ GPU path
class Built:
    """A workload resident on the box: pinned host caches, windows, queries, context."""


def build_workload(args, ws=1, numa_node=None):
    from sparse_kv_cache_landmark_gb300.kvo import Context, lib
    lib()                                   # fails loudly when the library is not built
    w = WORKLOADS[args.workload]
    if args.layers:
        w = w.scaled(n_layers=args.layers)
    if args.batch:
        w = w.scaled(batch=args.batch)
    lens = synth.seq_lens(w, args.seed)
    # with --append the host rows reserve `append` more tokens per group; the
    # generator draws them too (the appended tokens), and they start zeroed
    app = max(0, args.append)
    gen_lens = [x + app for x in lens]
    n = synth.layer_numel(w, gen_lens)
    layer_bytes = 2 * n * 2
    if args.host_layers:
        n_host = min(args.host_layers, w.n_layers)
    else:
        avail = 0
        try:
            with open("/proc/meminfo") as f:
                for line in f:
                    if line.startswith("MemAvailable"):
                        avail = int(line.split()[1]) * 1024
        except OSError:
            pass
        fit = int(0.55 * avail / (layer_bytes * ws)) if avail else w.n_layers
        n_host = max(1, min(w.n_layers, fit))
    t_gen = time.perf_counter()
    k_host, v_host, k_win, v_win, qs_l, qspec_l = [], [], [], [], [], []
    fut_k, fut_v = [], []
    for l in range(w.n_layers):
        q, qs = synth.gen_queries(w, args.seed, l)
        qs_l.append(q)
        qspec_l.append(qs)
        if l < n_host:
            with numa_bind(numa_node):
                kh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
                vh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
            synth.fill_layer(w, args.seed, l, kh, vh, q, gen_lens, device="cuda")
            k_host.append(kh)
            v_host.append(vh)
            kw = torch.empty(w.batch, w.n_kv_heads, w.window, w.head_dim, dtype=torch.bfloat16, device="cuda")
            vw = torch.empty_like(kw)
            off = 0
            for b, nb in enumerate(lens):
                cap = nb + app
                sz = cap * w.n_kv_heads * w.head_dim
                kr = kh[off:off + sz].view(w.n_kv_heads, cap, w.head_dim)
                vr = vh[off:off + sz].view(w.n_kv_heads, cap, w.head_dim)
                kw[b] = kr[:, nb - w.window:nb].to("cuda")
                vw[b] = vr[:, nb - w.window:nb].to("cuda")
                if app:
                    fut_k.append((l, b, kr[:, nb:].to("cuda")))
                    fut_v.append((l, b, vr[:, nb:].to("cuda")))
                    kr[:, nb:] = 0
                    vr[:, nb:] = 0
                off += sz
            k_win.append(kw)
            v_win.append(vw)
        else:
            k_host.append(k_host[l % n_host]); v_host.append(v_host[l % n_host])
            k_win.append(k_win[l % n_host]); v_win.append(v_win[l % n_host])
    torch.cuda.synchronize()
    B = Built()
    B.w, B.lens, B.n_host = w, lens, n_host
    B.setup_s = time.perf_counter() - t_gen
    B.page_node = page_node(k_host[0].data_ptr())
    B.ctx = Context(batch=w.batch, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                    block_size=w.block_size, top_k=w.top_k, window=w.window, n_layers=w.n_layers, seq_lens=lens,
                    k_host=k_host, v_host=v_host, k_win=k_win, v_win=v_win, max_append=app,
                    resident=bool(args.resident))
    B.app = app
    B.app_used = 0
    if app:
        # future tokens as [append][L][b][Hkv][d]; layers past n_host reuse layer l % n_host
        fk = torch.empty(app, w.n_layers, w.batch, w.n_kv_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
        fv = torch.empty_like(fk)
        for (l, b, t), (_, _, tv) in zip(fut_k, fut_v):
            for ll in range(l, w.n_layers, n_host):
                fk[:, ll, b] = t.permute(1, 0, 2)
                fv[:, ll, b] = tv.permute(1, 0, 2)
        B.fut_k, B.fut_v = fk, fv
    if args.gather_engine >= 0:
        B.ctx.set_gather_engine(args.gather_engine, args.gather_drivers)
    if args.gather_ctas or args.gather_threads or args.gather_unroll:
        B.ctx.set_gather_shape(args.gather_ctas, args.gather_threads or 128, args.gather_unroll or 1)
    if args.gather_reserve >= 0:
        B.ctx.set_gather_reserve(args.gather_reserve)
    if args.graphs >= 0:
        B.ctx.set_graphs(bool(args.graphs))
    if args.attn_impl >= 0:
        B.ctx.set_attn_impl(args.attn_impl, args.attn_ctas)
    if args.select_impl >= 0:
        B.ctx.set_select_impl(args.select_impl)
    if args.resident and args.prefetch_budget >= 0:
        B.ctx.set_prefetch_budget(args.prefetch_budget)
    if args.resident == 1:      # speculation only while it pays, unless asked otherwise
        B.ctx.set_spec_policy(1 if args.spec_policy < 0 else args.spec_policy)
    B.recon_rank = 0
    if w.key_dist == "lowrank" and args.reconstruct != 0:
        # GPU-resident low-rank key factors, packed like the host K (layers past n_host reuse l % n_host)
        R = w.lowrank_rank
        B.lr = []
        for l in range(n_host):
            coef = torch.empty(sum(gen_lens) * w.n_kv_heads * R, dtype=torch.bfloat16, device="cuda")
            basis = torch.empty(w.batch * w.n_kv_heads * R * w.head_dim, dtype=torch.bfloat16, device="cuda")
            synth.fill_lowrank(w, args.seed, l, coef, basis, gen_lens, device="cuda")
            B.lr.append((coef, basis))
        for l in range(w.n_layers):
            B.ctx.set_lowrank_keys(l, R, *B.lr[l % n_host])
        B.recon_rank = R
    B.keep = (k_host, v_host, k_win, v_win)
    B.q_pin = torch.stack(qs_l).pin_memory()
    B.qs_pin = None if qspec_l[0] is None else torch.stack(qspec_l).pin_memory()
    B.q_dev = B.q_pin.to("cuda")
    B.qs_dev = None if B.qs_pin is None else B.qs_pin.to("cuda")
    B.q_steps = None
    B.q_steps_pin = B.qs_steps_pin = None
    if args.resident:
        # decode steps whose queries drift: step s of layer l from gen_queries_step
        B.drift = args.drift if args.drift >= 0 else SPEC_SIGMA_88 / math.sqrt(2.0)
        qsteps = [[synth.gen_queries_step(w, args.seed, l, s, B.drift) for l in range(w.n_layers)]
                  for s in range(args.query_steps)]
        B.q_steps_pin = torch.stack([torch.stack([x[0] for x in st]) for st in qsteps]).pin_memory()
        B.qs_steps_pin = (None if qsteps[0][0][1] is None or args.resident == 2 else
                          torch.stack([torch.stack([x[1] for x in st]) for st in qsteps]).pin_memory())
        if args.resident == 2:
            B.qs_pin = B.qs_dev = None
        B.q_steps = B.q_steps_pin.to("cuda")
        B.qs_steps = None if B.qs_steps_pin is None else B.qs_steps_pin.to("cuda")
    B.step_i = 0
    rows = w.batch * w.n_q_heads
    B.o = torch.empty(w.n_layers, rows, w.head_dim, dtype=torch.float32, device="cuda")
    B.lse = torch.empty(w.n_layers, rows, dtype=torch.float32, device="cuda")
    return B


def step_queries(B):
    """With --resident, copy the next of the drifting query sets into the step's
    query buffers (the same buffers every step, so graph replay applies)."""
    if B.q_steps is not None:
        i = B.step_i % B.q_steps.shape[0]
        B.q_dev.copy_(B.q_steps[i], non_blocking=True)
        if B.qs_steps is not None:
            B.qs_dev.copy_(B.qs_steps[i], non_blocking=True)
        B.step_i += 1


def join_ctx_streams(ctx, stream):
    """Make ``stream`` wait for all work on the context's own streams: a step
    returns with the prefetches it issued for the next step still in flight,
    and a timed region that ends without them would leave out link work the
    steps it counts depend on."""
    for which in (0, 1, 2):
        ev = torch.cuda.Event()
        ev.record(torch.cuda.ExternalStream(ctx.get_stream(which)))
        stream.wait_event(ev)


def time_steps(B, steps, ws=1, profile=True):
    """(ms per step, per-kind profile) over ``steps`` decode steps on the current stream."""
    stream = torch.cuda.current_stream()
    ctx = B.ctx
    if profile:
        ctx.profile(True)
    barrier(ws)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        if B.app:
            ctx.append(B.fut_k[B.app_used], B.fut_v[B.app_used])
            B.app_used += 1
        step_queries(B)
        ctx.decode_step(B.q_dev, B.qs_dev, B.o, B.lse)
    join_ctx_streams(ctx, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    prof = None
    if profile:
        prof = ctx.profile_read()
        ctx.profile(False)
    return ev0.elapsed_time(ev1) / steps, prof


class E2E:
    """End-to-end steps through the public API with host buffers.

    Every step copies its queries from pinned host memory to the device and
    reads its outputs (o, lse) back into pinned host memory.  The copies run on
    two copy streams with double-buffered device queries and outputs, so the
    queries of step i + 1 cross the link while step i computes and the outputs
    of step i come back while step i + 1 computes -- as a serving loop that
    overlaps its transfers with the previous step does.  Every copy lies inside
    the timed region, which ends when the last step's outputs are on the host.
    """

    def __init__(self, B, args):
        self.B, self.args = B, args
        w = B.w
        self.q_dev = [B.q_dev, torch.empty_like(B.q_dev)]
        self.qs_dev = [B.qs_dev, None if B.qs_dev is None else torch.empty_like(B.qs_dev)]
        self.o = [B.o, torch.empty_like(B.o)]
        self.lse = [B.lse, torch.empty_like(B.lse)]
        self.o_pin = [torch.empty(B.o.shape, dtype=B.o.dtype, pin_memory=True) for _ in range(2)]
        self.lse_pin = [torch.empty(B.lse.shape, dtype=B.lse.dtype, pin_memory=True) for _ in range(2)]
        self.h2d = torch.cuda.Stream()
        self.d2h = torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self.q_i = 0
        self.i = 0
        self.h2d_bytes = B.q_pin.numel() * 2 + (B.qs_pin.numel() * 2 if B.qs_pin is not None else 0)
        self.d2h_bytes = B.o.numel() * 4 + B.lse.numel() * 4
        self.rows = w.batch * w.n_q_heads

    def _src(self):
        B = self.B
        if B.q_steps_pin is not None:
            j = self.q_i % self.args.query_steps
            qs = None if B.qs_steps_pin is None else B.qs_steps_pin[j]
            return B.q_steps_pin[j], qs
        return B.q_pin, B.qs_pin

    def _issue_input(self, slot, stream):
        # the buffer was last read by the step two before: wait for its end
        self.h2d.wait_event(self.ev_done[slot])
        with torch.cuda.stream(self.h2d):
            src, srcs = self._src()
            self.q_dev[slot].copy_(src, non_blocking=True)
            if srcs is not None and self.qs_dev[slot] is not None:
                self.qs_dev[slot].copy_(srcs, non_blocking=True)
        self.ev_in[slot].record(self.h2d)
        self.q_i += 1

    def run(self, steps, stream):
        """``steps`` end-to-end steps on ``stream``; the buffer pair alternates
        across calls too, so each step parity keeps one buffer set (a captured
        step graph is keyed by its buffers)."""
        B, ctx = self.B, self.B.ctx
        for s in range(2):
            self.ev_done[s].record(stream)
            self.ev_out[s].record(stream)
        self._issue_input(self.i & 1, stream)
        first = self.i
        for _ in range(steps):
            s = self.i & 1
            self.i += 1
            stream.wait_event(self.ev_in[s])
            stream.wait_event(self.ev_out[s])          # outputs of step i - 2 are on the host
            if B.app:
                ctx.append(B.fut_k[B.app_used], B.fut_v[B.app_used])
                B.app_used += 1
            ctx.decode_step(self.q_dev[s], self.qs_dev[s], self.o[s], self.lse[s])
            self.ev_done[s].record(stream)
            if self.i - first < steps:
                self._issue_input(1 - s, stream)
            self.d2h.wait_event(self.ev_done[s])
            with torch.cuda.stream(self.d2h):
                self.o_pin[s].copy_(self.o[s], non_blocking=True)
                self.lse_pin[s].copy_(self.lse[s], non_blocking=True)
            self.ev_out[s].record(self.d2h)
        stream.wait_stream(self.d2h)

    def check(self):
        torch.cuda.synchronize()
        for s in range(2):
            assert torch.isfinite(self.o_pin[s]).all() and torch.isfinite(self.lse_pin[s]).all()


def measure(args, ws, rank, smi_id, headline, steps, numa_node=None):
    """Build one workload, time its decode steps and collect everything its
    report needs (raw measurements; the roofline is computed by finish())."""
    stream = torch.cuda.current_stream()
    Bw = build_workload(args, ws, numa_node)
    w, lens, ctx = Bw.w, Bw.lens, Bw.ctx
    q_dev, qs_dev, o, lse = Bw.q_dev, Bw.qs_dev, Bw.o, Bw.lse
    m = {"name": w.name, "w": w, "lens": lens, "n_host": Bw.n_host, "setup_s": Bw.setup_s, "steps": steps,
         "recon_rank": Bw.recon_rank, "page_node": Bw.page_node}

    # the zero-copy read path: the flat gather over k consecutive blocks per
    # group (sequential host reads), into ping-pong half 0, best of 3
    G = w.batch * w.n_kv_heads
    seq_idx = torch.arange(w.top_k, dtype=torch.int32, device="cuda").repeat(G, 1).contiguous()
    zc_bytes = G * w.top_k * w.block_size * w.head_dim * 2 * 2
    link_zc = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ctx.gather_coalesced(0, 0, seq_idx, None, slot_base=0, want_runs=False, stream=stream.cuda_stream)
        b.record(stream)
        b.synchronize()
        link_zc = max(link_zc, zc_bytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    assert ctx.device_status() == 0
    m["link_zc"] = link_zc

    # the clock sampler starts first: the warm-up steps then run right before
    # the timed ones, so short timed regions do not start on an idle-clocked GPU
    clocks = Clocks(smi_id)
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        step_queries(Bw)
        ctx.decode_step(Bw.q_dev, Bw.qs_dev, o, lse)
    torch.cuda.synchronize()
    if args.resident:
        ctx.resident_fetched(reset=True)
    graphs = args.graphs == 1
    # With graph replay the timed region runs unprofiled (launch timing events
    # would bypass the graphs); the kernel times then come from a second timed
    # pass of the same steps launched stream by stream.
    t_ms, prof = time_steps(Bw, steps, ws, profile=not graphs)
    m["clocks"] = clocks.stop()
    m["fetched"] = ctx.resident_fetched(reset=True) if args.resident else None
    m["spec"] = None
    if args.resident == 1:
        st = ctx.spec_stats()
        m["spec"] = {"prefetched_blocks": sum(x[0] for x in st), "used_blocks": sum(x[1] for x in st),
                     "layers_prefetching": sum(x[2] for x in st), "layers": len(st),
                     "note": "since init, warm-up included: speculative blocks fetched and those a later true "
                             "index used"}
    if graphs:
        ctx.set_graphs(False)
        for _ in range(2):
            ctx.decode_step(q_dev, qs_dev, o, lse)
        _, prof = time_steps(Bw, steps, ws, profile=True)
        ctx.set_graphs(True)
    m["t_ms"] = max_over_ranks(ws, t_ms)
    m["prof"] = prof
    m["graphs"] = graphs

    if args.trace:
        # one more step, profiled, in the steady state: its launches in issue order
        ctx.profile(True)
        step_queries(Bw)
        ctx.decode_step(Bw.q_dev, Bw.qs_dev, o, lse)
        torch.cuda.synchronize()
        tr = ctx.profile_trace()
        ctx.profile_read()
        ctx.profile(False)
        with open(args.trace if headline else args.trace.replace(".json", f"_{w.name}.json"), "w") as f:
            json.dump({"workload": w.name, "launches": [{"kind": k, "layer": l, "start_ms": a, "end_ms": b}
                                                        for k, l, a, b in tr]}, f)

    m["e2e"] = None
    if headline:
        # end to end through the public API with host buffers (see E2E)
        e = E2E(Bw, args)
        e.run(max(2, args.warmup), stream)      # warm: graphs of both buffer sets captured outside the timing
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e.run(steps, stream)
        join_ctx_streams(ctx, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(ws, e0.elapsed_time(e1) / steps)
        e.check()
        m["e2e"] = {"value": ws / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": e.h2d_bytes,
                    "d2h_bytes_per_step": e.d2h_bytes, "ms_per_step": e2e_ms,
                    "copies": "queries in (pinned H2D) and o, lse out (D2H to pinned) every step, on two copy "
                              "streams, double-buffered so they overlap the neighbouring steps"}
        del e
    m["status"] = ctx.device_status()

    # steady-state misses per step: each layer's true index against the prediction of the previous step
    misses = 0
    for l in range(w.n_layers if not args.resident else 0):
        T, P = ctx.select_topk(l, q_dev[l], None if qs_dev is None else qs_dev[l])
        _, cnt, _ = ctx.index_diff(T, P if P is not None else T)
        misses += int(cnt.sum().item())
    m["misses"] = misses
    # co-batched dual-query attention (DualDecoder Fig. 18) and one layer's
    # attention and selection isolated: layer 0's ping-pong half, no gather beside them
    m["cob"] = None
    m["isolated"] = None
    q0 = q_dev[0]
    qs0 = qs_dev[0] if qs_dev is not None else (q0.float() * 0.5).to(torch.bfloat16)
    T, _ = ctx.select_topk(0, q0)
    miss, cnt, slot = ctx.index_diff(T, None)
    # layer 0's selection in both ping-pong halves: attention calls alternate
    # between them, so consecutive calls read different bytes
    for half in (0, 1):
        ctx.gather_coalesced(0, half, miss, cnt, slot_base=w.top_k, urgent=True)
    n_sel_layers = min(w.n_layers, 8)
    T_l = [T] + [ctx.select_topk(l, q_dev[l])[0] for l in range(1, n_sel_layers)]
    torch.cuda.synchronize()
    by_iso = workload_bytes(w, lens)
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    flush_buf = None

    def _t(fns, ws_bytes, n=20):
        """Mean time of n calls cycling through fns, back to back when the bytes
        the cycle reads exceed the L2; otherwise each call runs after a
        read-modify-write of a buffer twice the L2 and is timed alone (which
        then includes its launch)."""
        nonlocal flush_buf
        for i in range(3):
            fns[i % len(fns)]()
        if ws_bytes > l2:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(n):
                fns[i % len(fns)]()
            b.record(stream)
            b.synchronize()
            return a.elapsed_time(b) / n * 1e3
        if flush_buf is None:
            flush_buf = torch.zeros(2 * l2 // 4, dtype=torch.int32, device="cuda")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush_buf.add_(1)
            ev[i][0].record(stream)
            fns[i % len(fns)]()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / n * 1e3
    att_fns = [lambda h=h: ctx.sparse_decode_attn(0, h, q0, slot) for h in (0, 1)]
    sel_fns = [lambda l=l: ctx.select_topk(l, q_dev[l], idx_true=T_l[l]) for l in range(n_sel_layers)]
    one = _t(att_fns, 2 * by_iso["attended_per_layer"])
    sel = _t(sel_fns, n_sel_layers * by_iso["landmark_per_layer"])
    m["isolated"] = {"attention_us": round(one, 2), "select_us": round(sel, 2),
                     "note": "20 calls, nothing else running, alternating between both ping-pong halves "
                             f"(attention) and over {n_sel_layers} layers' landmarks (selection), so the "
                             "inputs of a cycle exceed the L2; where they do not, a buffer twice the L2 is "
                             "read and written before each call and each call is timed alone"}
    m["gather_engines"] = None
    if headline and args.gather_engines and not args.resident:
        # one layer's prefetch-sized gather (k blocks per group, the true index) per engine
        by = G * w.top_k * w.block_size * w.head_dim * 4
        _, nr = ctx.gather_coalesced(0, 0, T, None, slot_base=0)
        n_runs = int(nr.sum().item())
        ge = {"runs": n_runs, "bytes": by, "note": "layer 0's true index into ping-pong half 0, mean of 5 calls"}
        for eng in [int(x) for x in args.gather_engines.split(",") if x]:
            ctx.set_gather_engine(eng, 0)
            ms = _t([lambda: ctx.gather_coalesced(0, 0, T, None, slot_base=0, want_runs=False,
                                                  stream=stream.cuda_stream)], by, n=5) / 1e3
            ge[f"engine{eng}"] = {"ms": round(ms, 3), "gbs": round(by / (ms * 1e-3) / 1e9, 1)}
        ctx.set_gather_engine(args.gather_engine if args.gather_engine >= 0 else 3, args.gather_drivers)
        m["gather_engines"] = ge
    if headline and 2 * w.group_size <= 16:
        two = _t([lambda h=h: (ctx.sparse_decode_attn(0, h, q0, slot), ctx.sparse_decode_attn(0, h, qs0, slot))
                  for h in (0, 1)], 2 * by_iso["attended_per_layer"])
        co = _t([lambda h=h: ctx.sparse_decode_attn_cobatch(0, h, q0, qs0, slot) for h in (0, 1)],
                2 * by_iso["attended_per_layer"])
        m["cob"] = {"single_us": round(one, 2), "two_launches_us": round(two, 2), "cobatched_us": round(co, 2),
                    "cobatched_over_two": round(co / two, 3),
                    "note": "one layer's attention, isolated (no gather running), 20 back-to-back calls"}
    assert ctx.device_status() == 0
    ctx.close()
    del Bw, T, miss, cnt, slot, seq_idx
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free_host_cache()
    return m


def finish(m, args, link, hbm_peak, peak_kind):
    """Roofline of one measured workload: step time against t*, and the
    dominant kernel's achieved bandwidth."""
    w, lens, prof, t_ms, steps = m["w"], m["lens"], m["prof"], m["t_ms"], m["steps"]
    fetched = m["fetched"]
    fetched_step = None if fetched is None else sum(fetched) / steps
    by = workload_bytes(w, lens, m["misses"], fetched_per_step=fetched_step, recon_rank=m["recon_rank"])
    if fetched is not None:       # prefetch launches move only the prediction's delta
        by["gather_per_launch"] = fetched[1] / steps / w.n_layers * w.block_size * 4 * w.head_dim
    t_hbm = by["hbm"] / (hbm_peak * 1e9)
    t_link = by["host"] / (link * 1e9)
    t_star = max(t_hbm, t_link)
    kernels = {}
    for kind, (ms, cnt) in prof.items():
        if cnt:
            kernels[kind] = {"launches_per_step": cnt / steps, "avg_us": ms / cnt * 1e3,
                             "share_of_step": ms / steps / t_ms}
    a_ms, a_n = prof["attention"]
    if a_n:
        kernels["attention"]["hbm_gbs"] = by["attended_per_layer"] / (a_ms / a_n * 1e-3) / 1e9
    s_ms, s_n = prof["select"]
    if s_n:
        kernels["select"]["hbm_gbs"] = by["landmark_per_layer"] / (s_ms / s_n * 1e-3) / 1e9
    g_ms, g_n = prof["gather_prefetch"]
    achieved = by["gather_per_launch"] / ((g_ms / g_n) * 1e-3) / 1e9 if g_n else None
    iso = m["isolated"]
    return {
        "by": by, "t_star": t_star, "t_hbm": t_hbm, "t_link": t_link, "kernels": kernels, "achieved": achieved,
        "launches": sum(c for _, c in prof.values()),
        "summary": {
            "workload": w.name, "ms_per_step": round(t_ms, 4), "steps_per_s": round(1e3 / t_ms, 2),
            "t_star_ms": round(t_star * 1e3, 4), "frac": round(t_star * 1e3 / t_ms, 4),
            "bound": "link" if t_link >= t_hbm else "hbm",
            "host_bytes": by["host"], "hbm_bytes": by["hbm"],
            "urgent_misses_per_step": m["misses"],
            "effective_kv_gbs": round(by["kv_attended"] / (t_ms * 1e-3) / 1e9, 1),
            "dominant_kernel": {"kernel": "gather (prefetch)", "achieved_gbs": achieved, "peak_gbs": link,
                                "frac": (achieved / link) if achieved else None, "bound": "link"},
            "select_hbm_gbs_live": kernels.get("select", {}).get("hbm_gbs"),
            "attention_hbm_gbs_live": kernels.get("attention", {}).get("hbm_gbs"),
            "isolated": None if iso is None else dict(
                iso, attention_hbm_frac=round(by["attended_per_layer"] / (iso["attention_us"] * 1e-6) / 1e9
                                              / hbm_peak, 3),
                select_hbm_frac=round(by["landmark_per_layer"] / (iso["select_us"] * 1e-6) / 1e9 / hbm_peak, 3)),
            "clocks": m["clocks"], "timed_steps": steps, "setup_s": round(m["setup_s"], 1),
            "device_status": m["status"],
        },
    }


def run_ours(args):
    ws, rank, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    # weak scaling: every rank serves its own batch of requests (its own seed),
    # no data crosses ranks; only the timing is reduced (max over ranks)
    args.seed = args.seed + 7919 * rank
    stream = torch.cuda.current_stream()
    smi_id = smi_gpu_id(local)
    host = host_info()

    # pinned host caches on the GPU's nearest NUMA node when the host has several
    near = gpu_host_numa_node(local)
    numa_node = near if (near is not None and len(cpu_numa_nodes()) > 1) else None

    head = measure(args, ws, rank, smi_id, True, args.steps, numa_node)
    extra = []
    if ws == 1 and args.workloads:
        for name in [x for x in args.workloads.split(",") if x and x != args.workload]:
            a2 = argparse.Namespace(**vars(args))
            a2.workload, a2.layers, a2.batch, a2.host_layers, a2.trace = name, 0, 0, 0, args.trace
            a2.append = 0
            extra.append(measure(a2, ws, rank, smi_id, False, args.extra_steps, numa_node))
    # host->device link bandwidth: pinned copies on 1, 2 and 4 streams, per NUMA
    # placement (after the workloads, whose own pinned caches are allocated first)
    probe = probe_link(local, stream)
    link_zc = max([head["link_zc"]] + [m["link_zc"] for m in extra])
    link = max(probe["best_pinned_memcpy"], link_zc)
    hbm_peak, peak_kind = peaks()
    hf = finish(head, args, link, hbm_peak, peak_kind)
    wl = [hf["summary"]] + [finish(m, args, link, hbm_peak, peak_kind)["summary"] for m in extra]

    w, t_ms, by = head["w"], head["t_ms"], hf["by"]
    value = ws / (t_ms * 1e-3)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        t_group, n_groups = oracle_sample(w, args.seed, args.cpu_sample_s)
        G = w.batch * w.n_kv_heads
        cpu = {"value": 1.0 / (t_group * G * w.n_layers), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"fp64 numpy oracle on {n_groups} (request, KV head) groups of layer 0, "
                         f"{t_group * 1e3:.1f} ms per group, scaled to {G * w.n_layers} groups per step; "
                         f"one thread of {host['nproc']} ({host['cpu_model']})",
               "host": host}
    gkern = ("gather_flat_kernel" if args.gather_engine in (-1, 3) else
             "gather_tma_kernel" if args.gather_engine in (1, 2) else
             "copy engine (cudaMemcpyAsync per run)" if args.gather_engine == 4 else "gather_kernel")
    default_shape = not (args.gather_ctas or args.gather_threads or args.gather_unroll or args.gather_reserve >= 0)
    traffic = NCU_TRAFFIC.get((w.name, gkern)) if (default_shape and not args.layers and not args.batch) else None
    achieved = hf["achieved"]
    fetched = head["fetched"]
    fetched_step = None if fetched is None else sum(fetched) / args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": t_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads,
                       "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "context": w.ctx[0],
                       "block": w.block_size, "top_k": w.top_k, "window": w.window, "layers": w.n_layers,
                       "host_layers_distinct": head["n_host"],
                       "parallelism": f"request-sharded x{ws}, each rank its own batch, no collective on the data path",
                       "l2": f"inputs larger than L2 (129 MB): every step moves {by['host'] / 1e9:.2f} GB over "
                             f"the host link and {by['hbm'] / 1e9:.2f} GB through HBM"},
            "effective_kv_gbs": by["kv_attended"] / (t_ms * 1e-3) / 1e9 * ws,
            "urgent_misses_per_step": head["misses"],
            "cobatched_attention": head["cob"],
            "gather_engines": head["gather_engines"],
            "step_roofline": {"t_star_ms": hf["t_star"] * 1e3, "frac": hf["t_star"] * 1e3 / t_ms,
                              "bound": "link" if hf["t_link"] >= hf["t_hbm"] else "hbm",
                              "host_bytes": by["host"], "hbm_bytes": by["hbm"], "link_gbs": link,
                              "link_probe_gbs": {"pinned_memcpy": probe, "zero_copy_gather": link_zc},
                              "hbm_peak_gbs": hbm_peak, "hbm_peak_kind": peak_kind},
            "workloads": wl,
            "workloads_note": ("every workload's whole decode step timed like the headline one (CUDA events, "
                               "warm-up first, the context's streams joined at the end); t* = max(HBM bytes / "
                               "measured HBM peak, host bytes / link_gbs); frac = t* / ms_per_step"),
            "roofline": {"kernel": gkern + " (prefetch)", "bound": "link",
                         "achieved": achieved, "peak": link, "unit": "GB/s",
                         "frac": (achieved / link) if achieved else None,
                         "traffic": traffic,
                         "traffic_note": ("DRAM read+write bytes per launch from one ncu capture "
                                          "(writes still in L2 at kernel end are not counted)") if traffic else
                                         "no ncu capture of this kernel, shape and workload",
                         "peak_kind": ("measured in this run: the best of pinned cudaMemcpyAsync host->device "
                                       "copies (1, 2 and 4 streams of 1 GiB each, per NUMA placement) and a "
                                       "zero-copy gather of k consecutive blocks per group, best of 3 each")},
            "kernels": hf["kernels"],
            "kernel_timing": ("CUDA events around each launch on its own stream, in a second timed pass "
                              "(graph replay on in the first)") if head["graphs"] else
                             "CUDA events around each launch on its own stream, inside the timed region",
            "gpu_launches": hf["launches"],
            "e2e": head["e2e"],
            "clocks": head["clocks"],
            "cpu_baseline": cpu,
            "host": host,
            "host_pages_numa_node": head["page_node"],
            "device_status": head["status"],
            "setup_s": round(head["setup_s"], 1),
            "append_per_step": bool(args.append),
            "gather_shape": {"ctas": args.gather_ctas or "default", "threads": args.gather_threads or "default",
                             "unroll": args.gather_unroll or "default",
                             "engine": "default" if args.gather_engine < 0 else args.gather_engine,
                             "drivers": args.gather_drivers or "default"},
            "attention_kernel": {"impl": "default" if args.attn_impl < 0 else args.attn_impl,
                                 "ctas": args.attn_ctas or "default"},
            "selection_kernel": {"impl": "default" if args.select_impl < 0 else args.select_impl},
            "lowrank_keys": None if not head["recon_rank"] else {
                "rank": head["recon_rank"], "rebuilt_blocks_per_step": head["misses"],
                "host_bytes_saved_per_step": head["misses"] * w.block_size * 2 * w.head_dim,
                "note": "missed keys rebuilt on the GPU from rank-R factors; misses move V only"},
            "resident": None if not args.resident else {
                "speculation": args.resident == 1,
                "drift": SPEC_SIGMA_88 / math.sqrt(2.0) if args.drift < 0 else args.drift,
                "query_steps": args.query_steps, "prefetch_budget": args.prefetch_budget,
                "spec_policy": ("adaptive" if args.spec_policy != 0 else "always") if args.resident == 1 else None,
                "fetched_blocks_per_step": fetched_step,
                "fetched_of_selected": fetched_step / (w.n_layers * w.batch * w.n_kv_heads * w.top_k),
                "urgent_blocks_per_step": fetched[0] / args.steps, "prefetch_blocks_per_step": fetched[1] / args.steps,
                "speculation_counters": head["spec"],
                "note": "cross-step delta prefetch: per-layer resident sets of 2k blocks; host bytes = fetched blocks"},
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
