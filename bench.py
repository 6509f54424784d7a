"""Benchmark: MoE-layer decode tokens/s through the GPU expert cache (libftmoe, sm_103a).

Workload (default): the 35B-A3B-shaped decode layer — hidden 2048, 128 experts, expert
intermediate 768, top-8, BF16 weights, 1..16 tokens per step (seeded length mix),
Zipf(1.1) expert popularity with 0.6 step-to-step reuse, one LRU cache holding 37% of the
pool (47 slots); the pool sits in pinned host memory and misses are filled over PCIe.

One step = one forward call of the layer on one decode step of the trace: top-k, cache
lookup + LRU update, expert FFN on resident experts, miss fills (copy stream), expert FFN
on filled / staged experts, combine. Inputs (x, logits of every timed step) are resident in
HBM before timing starts; L2 is flushed before every step, outside the per-step CUDA-event
bracket: a 256 MB buffer is written and then read back (see `l2_flush`).

Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (no data-path collective).
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

WORKLOAD = "decode_bf16"
REF_TOKENS = 2          # tokens per step the CPU reference arm computes (bounded sample)
REF_LAYERS = 2          # layers per step the CPU reference arm computes (bounded sample)
METRIC = "MoE-layer decode tokens/s (35B-A3B-shaped BF16 layer, LRU cache 37% of pool)"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def clocks_path(args, rank):
    """File for the nvidia-smi samples of the timed region (a %d in --clocks-csv takes the rank)."""
    path = args.clocks_csv or os.path.join(tempfile.gettempdir(), "ftmoe_clocks_r%d.csv")
    return path % rank if "%d" in path else path


def max_over_ranks(x, device="cpu"):
    """Max of a per-rank float over the default process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, seconds_per_rank, device="cpu"):
    """Whole-job throughput of N independent replicas: the units all ranks processed over the
    slowest rank's time (every rank processes the same units)."""
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    return units_per_rank * ws / max_over_ranks(seconds_per_rank, device)


class _CtypesNvml:
    """The few read-only NVML queries the clock sampler makes, through ctypes on the NVIDIA
    libnvidia-ml.so.1 (used where the pynvml module is not installed)."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")

    def _ok(self, r, what):
        if r != 0:
            raise RuntimeError("%s returned %d" % (what, r))

    def nvmlInit(self):
        self._ok(self.lib.nvmlInit_v2(), "nvmlInit_v2")

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self.c.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), self.c.byref(h)), "handle by bus id")
        return h

    def nvmlDeviceGetHandleByIndex(self, i):
        h = self.c.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(self.c.c_uint(i), self.c.byref(h)), "handle by index")
        return h

    def _uint(self, fn, h, *args):
        v = self.c.c_uint()
        self._ok(getattr(self.lib, fn)(h, *args, self.c.byref(v)), fn)
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._uint("nvmlDeviceGetClockInfo", h, self.c.c_int(kind))

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._uint("nvmlDeviceGetMaxClockInfo", h, self.c.c_int(kind))

    def nvmlDeviceGetPowerUsage(self, h):
        return self._uint("nvmlDeviceGetPowerUsage", h)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.c.c_ulonglong()
        self._ok(self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, self.c.byref(v)), "clock reasons")
        return v.value


FLUSH_MODES = ("write-read", "write")


def l2_flush(buf, mode="write-read"):
    """Evict every line of the previous step from L2 (126 MB) before a timed step: write
    `buf`, twice the size of L2, and in the default mode read it back. The read evicts the
    flush's own dirty lines while the clock is stopped, so L2 is left holding clean lines of
    the flush buffer; a write-only flush leaves ~126 MB of dirty lines that the next step's
    reads must first write back to HBM, traffic the workload itself does not have. Mode
    "write" keeps the write-only flush, for comparison."""
    import torch
    buf.zero_()
    if mode == "write-read":
        buf.view(torch.int64).sum()


FLUSH_TEXT = {"write-read": "flushed (256 MB written, then read back) before every step, outside the step's events",
              "write": "flushed (256 MB write) before every step, outside the step's events"}


class Clocks:
    """SM clocks, power and throttle reasons sampled during the timed region.

    NVML (the library nvidia-smi reads) is polled from a thread every 10 ms, so a timed region
    of a few tens of milliseconds still holds several samples; spawning nvidia-smi takes
    longer than such a region. The power draw (the slowest query) is read on every fifth
    sample. Each sample is also written to `path` as a CSV line. Falls back to an
    `nvidia-smi -lms 50` process where NVML cannot be loaded."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clocks-event-reason bits
    BITS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
            ("sw_power_cap", 0x4))

    def __init__(self, index, path, period_s=0.010):
        import threading
        self.path = path
        self.proc = None
        self.samples = []
        self.f = open(path, "w")
        self.nv = None
        try:
            try:
                import pynvml
            except ImportError:
                pynvml = _CtypesNvml()
            pynvml.nvmlInit()
            self.nv = pynvml
            self.handle = self._handle(pynvml, index)
            self.max_mhz = float(pynvml.nvmlDeviceGetMaxClockInfo(self.handle, pynvml.NVML_CLOCK_SM))
        except Exception as e:  # noqa: BLE001 - fall back to nvidia-smi, keep the reason
            self.nv = None
            self.nvml_error = "%s: %s" % (type(e).__name__, str(e)[:120])
        if self.nv is not None:
            self.stop_ev = threading.Event()
            self.period = period_s
            self.sample()
            self.th = threading.Thread(target=self._loop, daemon=True)
            self.th.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.Q, "--format=csv,noheader",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _handle(pynvml, index):
        # the CUDA device's PCI bus id picks the same GPU whatever CUDA_VISIBLE_DEVICES says
        try:
            import torch
            p = torch.cuda.get_device_properties(index)
            bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            return pynvml.nvmlDeviceGetHandleByPciBusId(bus)
        except Exception:
            return pynvml.nvmlDeviceGetHandleByIndex(index)

    def sample(self):
        nv = self.nv
        try:
            sm = float(nv.nvmlDeviceGetClockInfo(self.handle, nv.NVML_CLOCK_SM))
            rs = int(nv.nvmlDeviceGetCurrentClocksEventReasons(self.handle))
            if len(self.samples) % 5 == 0 or not hasattr(self, "pw"):
                self.pw = nv.nvmlDeviceGetPowerUsage(self.handle) / 1000.0
            pw = self.pw
        except Exception:
            return
        self.samples.append((sm, rs))
        self.f.write("%.1f,%.0f,%.0f,%.1f,0x%x\n" % (time.time(), sm, self.max_mhz, pw, rs))

    def _loop(self):
        while not self.stop_ev.wait(self.period):
            self.sample()

    def stop(self):
        if self.nv is not None:
            self.stop_ev.set()
            self.th.join(timeout=5)
            self.sample()
            self.f.close()
            if not self.samples:
                return None
            reasons = sorted({n for _, r in self.samples for n, b in self.BITS if r & b})
            return {"sm_mhz": float(np.median([sm for sm, _ in self.samples])), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(self.samples), "source": "NVML, %d ms period" % round(self.period * 1e3)}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = [n for n, _ in self.BITS]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx = float(parts[2].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 50 ms period",
                "nvml_error": getattr(self, "nvml_error", None)}


def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


# DRAM traffic of the decode FFN kernel: an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum over every FFN launch of a `--ffn-traffic` run) divided by the
# algorithmic bytes of the same launches, kept in a profile summary together with a hash of
# the kernel's sources; a kernel changed since the capture reports no traffic.
TRAFFIC = {
    "bf16": ("tc_ffn_decode_bf16_traffic.md", ["tc_ffn.cu", "tc_ffn.cuh", "tc_ptx.cuh", "mk.cuh"]),
    "mxfp4": ("fp4_ffn_decode_mxfp4_traffic.md", ["tc_fp4.cu", "tc_fp4.cuh", "tc_ptx.cuh", "mk.cuh"]),
    "nvfp4": ("fp4_ffn_decode_nvfp4_traffic.md", ["tc_fp4.cu", "tc_fp4.cuh", "tc_ptx.cuh", "mk.cuh"]),
}


def kernel_sources_sha256(files):
    """SHA-256 of the kernel's code: the sources with comments and whitespace removed, so a
    comment edit keeps a capture valid and any code change voids it."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "expert_cached_sparse_top_b300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()


def traffic_ratio(wfmt):
    """DRAM bytes per algorithmic byte of the decode FFN kernel, or None (no capture, or the
    kernel's sources changed since)."""
    if wfmt not in TRAFFIC:
        return None
    name, files = TRAFFIC[wfmt]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    vals = {}
    for ln in text.splitlines():
        ln = ln.strip().strip("-").strip()
        if ln.startswith("`") and "`:" in ln:
            key, _, v = ln[1:].partition("`:")
            vals[key] = v.strip().strip("`")
    try:
        if vals.get("kernel_sources_sha256") != kernel_sources_sha256(files):
            return None
        return float(vals["traffic_per_algorithmic_byte"])
    except (KeyError, ValueError, OSError):
        return None


# Decode workloads: name -> (metric, host images (None = the whole pool), default steps, warmup)
DECODE = {
    "decode_bf16": (METRIC, None, 480, 16),
    "decode_mxfp4": ("MoE decode tokens/s through 43 MXFP4 layers (284B-shaped, one global "
                     "LRU cache 20% of pool)", 16, 24, 4),
    "elastic_nvfp4": ("MoE-layer decode tokens/s (35B-A3B-shaped NVFP4 layer, LRU cache "
                      "resized 40% -> 15% -> 30%)", None, 300, 16),
}


def host_copy_gbs(nbytes=1 << 30, reps=5):
    """Host memory bandwidth B_H: a multi-threaded memcpy of 1 GiB between two ordinary
    (pageable) host buffers; read + write bytes per second, best of `reps`."""
    import torch
    a = torch.empty(nbytes, dtype=torch.uint8)
    b = torch.empty(nbytes, dtype=torch.uint8)
    a.fill_(1)
    b.copy_(a)
    best = 0.0
    for _ in range(reps):
        t0 = time.perf_counter()
        b.copy_(a)
        dt = time.perf_counter() - t0
        best = max(best, 2 * nbytes / dt / 1e9)
    return best, torch.get_num_threads()


def resize_plan(cfg, Wm, K):
    """Elastic workload: the cache budget changes twice inside the timed range, at 1/3 and
    2/3 of it (the trace's own split points scaled to the run). Resizes are safe points
    between steps, outside every step's events."""
    if not cfg.resize:
        return {}
    cuts = [Wm + K // 3, Wm + (2 * K) // 3]
    return {c: W_cap(cfg, f) for c, (_, f) in zip(cuts, cfg.resize)}


def W_cap(cfg, frac):
    import workloads as W
    return W.cache_capacity(cfg, frac)


def host_cpus():
    """The host's core count (os.cpu_count, what nproc reports without a mask) and the cores
    this process may run on (its affinity mask), stated beside every CPU number."""
    try:
        aff = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        aff = None
    return {"host_cpus": os.cpu_count(), "affinity_cpus": aff}


def oracle_baseline(cfg, pool, budget_s=15.0, max_steps=64):
    """The oracle as it stands on this host's cores: LRU simulator + fp64 MoE layer over the
    first calls of the same trace until ~budget_s of CPU work. Returns tokens/s through
    all of the workload's layers (a 43-layer step counts its tokens once)."""
    import workloads as W
    from oracle import formats, lru, moe
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = 1
    sim = lru.LRUCache(W.cache_capacity(cfg), cfg.experts)
    layer_tokens, calls = 0, 0
    t0 = time.perf_counter()
    done = False
    for step in W.decode_trace(cfg, steps=max_steps):
        for d in step:
            idx = moe.topk(d["logits"], cfg.top_k)
            w = moe.gate_weights(d["logits"], idx)
            sim.call(d["layer"], idx.reshape(-1))
            L = d["layer"]
            moe.layer_forward(formats.bf16_to_f64(d["x"]), idx, w,
                              lambda e: formats.decode_blob(pool.blob(L * cfg.experts + e), cfg.fmt,
                                                            cfg.hidden, cfg.inter))
            layer_tokens += d["T"]
            calls += 1
            if time.perf_counter() - t0 > budget_s:
                done = True
                break
        if done:
            break
    dt = time.perf_counter() - t0
    return {"value": layer_tokens / cfg.layers / dt, "unit": "tokens/s", "cores": int(threads),
            "kind": "oracle", **host_cpus(),
            "sample": "first %d layer calls (%d layer-tokens) of the same seeded trace, fp64 "
                      "numpy oracle + LRU simulator" % (calls, layer_tokens)}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import workloads as W
    from workloads.host import HostPool
    metric, images, _, _ = DECODE[args.workload]
    cfg = W.config(args.workload)
    pool = HostPool(cfg, images=images, pinned=False)
    from oracle import formats, lru, moe
    sim = lru.LRUCache(W.cache_capacity(cfg), cfg.experts)
    tr = W.decode_trace(cfg, steps=args.warmup + args.steps)
    times, toks = [], []
    for i, step in enumerate(tr):
        n = min(step[0]["T"], REF_TOKENS)     # bounded sample: the step's first tokens
        t0 = time.perf_counter()
        for d in step[:REF_LAYERS]:
            L = d["layer"]
            idx = moe.topk(d["logits"], cfg.top_k)
            w = moe.gate_weights(d["logits"], idx)
            sim.call(L, idx.reshape(-1))
            moe.layer_forward(formats.bf16_to_f64(d["x"][:n]), idx[:n], w[:n],
                              lambda e: formats.decode_blob(pool.blob(L * cfg.experts + e), cfg.fmt,
                                                            cfg.hidden, cfg.inter))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt * cfg.layers / min(cfg.layers, REF_LAYERS))
            toks.append(n)
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = 1
    value = sum(toks) / sum(times)
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, W.cache_capacity(cfg), "n/a (CPU)"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": int(threads),
                         "kind": "oracle", **host_cpus(),
                         "sample": "steps %d..%d of the seeded trace; per step the cache "
                                   "simulator on all tokens and the fp64 layer on the first "
                                   "min(T, %d) tokens of the first %d layer(s), time scaled to "
                                   "all %d layers" % (args.warmup, args.warmup + args.steps - 1,
                                                      REF_TOKENS, min(cfg.layers, REF_LAYERS),
                                                      cfg.layers)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(cfg, C, l2):
    return {"workload": cfg.name, "layers": cfg.layers, "hidden": cfg.hidden,
            "experts": cfg.experts, "inter": cfg.inter, "top_k": cfg.top_k,
            "weights": cfg.wfmt,
            "tokens_per_step": "%d..%d (seeded mix)" % (cfg.t_min, cfg.t_max),
            "cache_slots": C, "l2": l2}


def run_ours(args):
    line = decode_line(args)
    if line is not None:
        if not getattr(args, "no_extras", False) and args.workload == WORKLOAD and not args.tokens \
                and not args.layers and not args.fused and line["n_gpus"] == 1:
            line["extras"]["sub"] = sub_records(args)
        print(json.dumps(line), flush=True)


def decode_line(args):
    """One decode workload on this rank's GPU; rank 0 returns the JSON line (dict), the
    other ranks None. args.lite skips the end-to-end pass and the oracle baseline (the
    sub-records of the default run)."""
    import torch
    import torch.distributed as dist
    import workloads as W
    from workloads.host import HostPool
    from expert_cached_sparse_top_b300 import build as b
    b.build()
    from expert_cached_sparse_top_b300 import ftmoe

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    metric, images, _, _ = DECODE[args.workload]
    ov = {"layers": args.layers} if args.layers else {}
    if args.tokens:
        # every step the same number of tokens (e.g. T = 1, single-sequence decode)
        ov.update(t_min=args.tokens, t_max=args.tokens)
        metric = metric.replace("(", "(T = %d, " % args.tokens, 1)
    cfg = W.config(args.workload, **ov)
    C = W.cache_capacity(cfg)
    pool = HostPool(cfg, images=images)
    K, Wm = args.steps, args.warmup
    nsteps = Wm + K
    if nsteps > cfg.steps:
        raise SystemExit("steps + warmup must be <= %d (trace length)" % cfg.steps)
    resizes = resize_plan(cfg, Wm, K)
    trace = list(W.decode_trace(cfg, steps=nsteps))
    # per step: list over layers of (layer, T, x, logits) resident in HBM
    calls = [[(d["layer"], d["T"],
               torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).to(dev),
               torch.from_numpy(d["logits"]).to(dev)) for d in st] for st in trace]
    Ts = [st[0]["T"] for st in trace]
    touched = sorted({d["layer"] * cfg.experts + int(e) for st in trace for d in st
                      for e in np.unique(d["picks"])})
    out = torch.empty((cfg.t_max, cfg.hidden), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def make(capacity):
        c = ftmoe.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k,
                              cfg.t_max, cfg.wfmt, capacity, device=local, fused_decode=args.fused)
        return ftmoe.MoECache(c, pool.ptrs, None)

    def run_step(cache, i):
        for (layer, T, x, lg) in calls[i]:
            cache.forward(layer, x, T, out, logits=lg, stream=stream)

    def timed_pass(cache, record_clocks=False, elastic=True):
        for i in range(Wm):
            run_step(cache, i)
        torch.cuda.synchronize()
        s0 = cache.stats()
        cache.set_timing(True)
        cache.timing(reset=True)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        # the flush's kernels are loaded on their first launch (about a second): not inside
        # the timed loop's wall clock
        l2_flush(flush, args.flush)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clk = Clocks(local, clocks_path(args, rank)) if record_clocks else None
        t_wall = time.perf_counter()
        for j in range(K):
            i = Wm + j
            if elastic and i in resizes:
                cache.resize(resizes[i])
            l2_flush(flush, args.flush)
            evs[j][0].record(stream)
            run_step(cache, i)
            evs[j][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clocks = clk.stop() if clk else None
        if ws > 1:
            dist.barrier()
        step_ms = [a.elapsed_time(b_) for a, b_ in evs]
        tim = cache.timing(reset=True)
        cache.set_timing(False)
        s1 = cache.stats()
        return step_ms, t_wall, tim, s0, s1, clocks

    if args.ffn_traffic:
        # the cached pass alone, every FFN launch counted from the first call (an ncu capture
        # of the FFN kernel over this run divides its DRAM bytes by these); with --all-resident
        # every selected expert is placed before the first call (no fill ever)
        cache = make(len(touched) if args.all_resident else C)
        if args.all_resident:
            cache.pin(touched)
        cache.set_timing(True)
        cache.timing(reset=True)
        for i in range(Wm + K):
            if i in resizes and not args.all_resident:
                cache.resize(resizes[i])
            run_step(cache, i)
        torch.cuda.synchronize()
        tim = cache.timing(reset=True)
        cache.close()
        print(json.dumps({"workload": args.workload, "ffn_launches": int(tim["ffn_launches"]),
                          "ffn_algorithmic_bytes": int(tim["ffn_weight_bytes"]),
                          "kernel_sources_sha256": kernel_sources_sha256(TRAFFIC[cfg.wfmt][1])}),
              flush=True)
        return
    cache = make(C)
    step_ms, t_wall, tim, s0, s1, clocks = timed_pass(cache, record_clocks=True)
    cache.close()
    tokens = sum(Ts[Wm:])
    dev_s = sum(step_ms) / 1e3
    # max over ranks of the timed duration; all ranks process the same number of tokens
    t_max = max_over_ranks(dev_s, dev)
    value = replica_throughput(tokens, dev_s, dev)

    # every expert the run selects resident (no misses): the HBM-bound ceiling of the step
    cache_r = make(len(touched))
    for i in range(Wm + K):   # touch every selected expert once
        run_step(cache_r, i)
    rs_ms, _, rtim, _, _, _ = timed_pass(cache_r, elastic=False)
    cache_r.close()

    lite = getattr(args, "lite", False)
    # end to end through the C ABI with host buffers: H2D of x + logits, forward, D2H of out
    hx = [[(torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory(),
            torch.from_numpy(d["logits"]).pin_memory()) for d in st] for st in trace] if not lite else []
    oh = torch.empty((cfg.layers, cfg.t_max, cfg.hidden), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty((cfg.layers, cfg.t_max, cfg.hidden), dtype=torch.bfloat16, device=dev)
    ld = torch.empty((cfg.layers, cfg.t_max, cfg.experts), dtype=torch.float32, device=dev)
    od = torch.empty((cfg.layers, cfg.t_max, cfg.hidden), dtype=torch.bfloat16, device=dev)
    cache_e = make(C)
    h2d = d2h = 0
    e2e_s = 0.0
    for i in (range(Wm + K) if not lite else ()):
        if i in resizes:
            cache_e.resize(resizes[i])
        T = Ts[i]
        l2_flush(flush, args.flush)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for li, (xh, lh) in enumerate(hx[i]):
            xd[li, :T].copy_(xh, non_blocking=True)
            ld[li, :T].copy_(lh, non_blocking=True)
            cache_e.forward(li, xd[li], T, od[li], logits=ld[li], stream=stream)
            oh[li, :T].copy_(od[li, :T], non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if i >= Wm:
            e2e_s += dt
            h2d += sum(xh.numel() * 2 + lh.numel() * 4 for xh, lh in hx[i])
            d2h += T * cfg.hidden * 2 * cfg.layers
    cache_e.close()
    e2e_s = max_over_ranks(e2e_s, dev)

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return None

    peaks = _peaks()
    hbm = peaks.get("hbm_gbs")
    ffn_ms = tim["ffn_hit_ms"] + tim["ffn_miss_ms"]
    ffn_passes = tim["ffn_launches"]
    achieved = tim["ffn_weight_bytes"] / (ffn_ms * 1e-3) / 1e9 if ffn_ms > 0 else None
    rffn_ms = rtim["ffn_hit_ms"] + rtim["ffn_miss_ms"]
    r_achieved = rtim["ffn_weight_bytes"] / (rffn_ms * 1e-3) / 1e9 if rffn_ms > 0 else None
    misses = s1["misses"] - s0["misses"]
    hits = s1["hits"] - s0["hits"]
    fill_b = (s1["fill_bytes"] - s0["fill_bytes"]) + (s1["stage_bytes"] - s0["stage_bytes"])
    base = oracle_baseline(cfg, pool, budget_s=args.cpu_budget) if not lite else None
    # q* of the pages' bandwidth-adaptive policy: of a step's m misses, about m * B_P / B_H
    # would be filled over PCIe and the rest computed in place on the CPU ([MTP] q* policy).
    # CPU execution is not built; the split is reported from the bandwidths measured here.
    b_h, h_threads = host_copy_gbs()
    b_p = (fill_b / (tim["fill_ms"] * 1e-3) / 1e9) if tim["fill_ms"] > 0 else None
    m_step = misses / K
    # fill time not hidden under the step's kernels (route, FFN passes, combine)
    busy = tim["route_ms"] + tim["ffn_hit_ms"] + tim["ffn_miss_ms"] + tim["combine_ms"]
    exposed = min(max(tim["total_ms"] - busy, 0.0), tim["fill_ms"])
    overlap = (1.0 - exposed / tim["fill_ms"]) if tim["fill_ms"] > 0 and not args.fused else None
    ratio = None if args.fused else traffic_ratio(cfg.wfmt)
    bpl = tim["ffn_weight_bytes"] / max(ffn_passes, 1)
    # the fused kernel spans the whole call, PCIe fills included: its HBM roofline is taken
    # from the all-resident pass (the same kernel, no fill to wait for)
    roof_gbs, roof_on = achieved, "the cached (timed) run"
    if args.fused:
        roof_gbs, roof_on = r_achieved, "the all-resident pass (the fused kernel waits for fills)"
        bpl = rtim["ffn_weight_bytes"] / max(rtim["ffn_launches"], 1)
        ffn_ms, ffn_passes = rffn_ms, rtim["ffn_launches"]
    kern = ("fused decode kernel (one cooperative launch per call: top-k, LRU lookup, %s, combine; "
            "missed experts' tiles wait for their PCIe fills)"
            % ("row gather, tcgen05 W13+SwiGLU and W2" if cfg.wfmt == "bf16" else
               "activation pieces, block-scaled tcgen05 W13+SwiGLU and W2 on %s codes" % cfg.wfmt.upper())
            if args.fused else
            "expert FFN (tcgen05 grouped GEMM, W13+SwiGLU and W2 in one launch), per pass"
            if cfg.wfmt == "bf16" else
            "expert FFN (block-scaled tcgen05 grouped GEMM on %s codes: W13+SwiGLU, activation "
            "pieces, W2), per pass" % cfg.wfmt.upper())
    line = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": Wm, "ms_per_step": 1e3 * t_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.wfmt, "data": "synthetic",
        "config": dict(workload_config(cfg, C, FLUSH_TEXT[args.flush]),
                       pool="pinned host, %d keys on %d blobs x %d B" % (cfg.keys, pool.images,
                                                                        pool.blob_bytes),
                       resizes={str(k2): v for k2, v in resizes.items()} or None,
                       parallelism="replicas" if ws > 1 else "single GPU",
                       fused_decode=bool(args.fused)),
        "roofline": {"bound": "hbm", "kernel": kern,
                     "achieved": roof_gbs, "peak": hbm,
                     "unit": "GB/s", "frac": (roof_gbs / hbm) if (roof_gbs and hbm) else None,
                     "measured_on": roof_on,
                     "traffic": ratio * bpl if ratio else None,
                     "traffic_source": ("ncu dram bytes per algorithmic byte (profiles/%s) x "
                                        "algorithmic bytes per launch" % TRAFFIC[cfg.wfmt][0])
                     if ratio else None,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs" if hbm else None,
                     "algorithmic_bytes_per_launch": bpl,
                     "avg_launch_ms": ffn_ms / max(ffn_passes, 1)},
        "cpu_baseline": base,
        "e2e": {"value": tokens * ws / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d // K, "d2h_bytes_per_step": d2h // K} if not lite else None,
        "gpu_launches": int(tim["kernel_launches"]),
        "clocks": clocks,
        "extras": {
            "miss_rate": misses / max(hits + misses, 1),
            "pcie_fill_GBps": b_p,
            "q_star": {"B_P_GBps": b_p, "B_H_GBps": b_h, "host_threads": h_threads,
                       "misses_per_step": m_step,
                       "q_star_per_step": (m_step * b_p / b_h) if (b_p and b_h) else None,
                       "note": "experts per step the pages' policy would fill (m * B_P / B_H); "
                               "the rest would run on the host CPU, which is not built"},
            "fill_ms_per_step": tim["fill_ms"] / K,
            "fill_overlap_fraction": overlap,
            "wall_ms_per_step": 1e3 * t_wall / K,
            "all_resident_slots": len(touched),
            "all_resident_tokens_per_s": tokens / (sum(rs_ms) / 1e3),
            "all_resident_ffn_GBps": r_achieved,
            "all_resident_ffn_frac": (r_achieved / hbm) if (r_achieved and hbm) else None,
            "stage_ms": {k2: tim[k2] / K for k2 in ("route_ms", "ffn_hit_ms", "fill_ms",
                                                     "ffn_miss_ms", "combine_ms", "total_ms")},
        },
    }
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return line


def run_policy_compare(args):
    """Cache policies on the same decode trace, through the engine: the engine's global LRU
    against the pages' comparators ([MTP] §The gap it targets, §Results): a per-layer LRU,
    a static hot subset (KTransformers-style: the C keys selected most often over a
    calibration window, pinned at load) and static layer placement (llama.cpp-style: every
    expert of the first C // E layers resident). Miss rates, PCIe bytes and tokens/s over the
    same measured steps; each policy runs its own warm-up on the calibration steps."""
    import torch
    import workloads as W
    from workloads.host import HostPool
    from expert_cached_sparse_top_b300 import build as b
    b.build()
    from expert_cached_sparse_top_b300 import ftmoe
    torch.cuda.set_device(0)
    layers = args.layers or 40
    cfg = W.config("decode_bf16", layers=layers)          # the 35B-A3B layer shape, 40 layers
    C = W.cache_capacity(cfg)                              # 37 % of the pool
    pool = HostPool(cfg, images=16)
    calib, K = 64, args.steps
    trace = list(W.decode_trace(cfg, steps=calib + K))
    dev = torch.device("cuda", 0)
    calls = [[(d["layer"], d["T"], torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).to(dev),
               torch.from_numpy(d["logits"]).to(dev)) for d in st] for st in trace]
    out = torch.empty((cfg.t_max, cfg.hidden), dtype=torch.bfloat16, device=dev)
    count = np.zeros(cfg.keys, dtype=np.int64)
    for st in trace[:calib]:
        for d in st:
            for e in np.unique(d["picks"]):
                count[d["layer"] * cfg.experts + int(e)] += 1
    hot = [int(k) for k in np.lexsort((np.arange(cfg.keys), -count))[:C]]
    whole = [l * cfg.experts + e for l in range(C // cfg.experts) for e in range(cfg.experts)]
    plans = [("global_lru", ftmoe.POLICY_GLOBAL_LRU, None), ("layer_lru", ftmoe.POLICY_LAYER_LRU, None),
             ("static_hot_set", ftmoe.POLICY_STATIC, hot), ("static_layers", ftmoe.POLICY_STATIC, whole)]
    res = {}
    stream = torch.cuda.current_stream(dev)
    for name, policy, pin in plans:
        c = ftmoe.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, cfg.t_max,
                              cfg.wfmt, C, policy=policy)
        cache = ftmoe.MoECache(c, pool.ptrs, None)
        if pin is not None:
            cache.pin(pin)
        else:
            for st in calls[:calib]:                       # the LRU policies warm up on the
                for (layer, T, x, lg) in st:               # calibration steps
                    cache.forward(layer, x, T, out, logits=lg, stream=stream)
        torch.cuda.synchronize()
        s0 = cache.stats()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st in calls[calib:]:
            for (layer, T, x, lg) in st:
                cache.forward(layer, x, T, out, logits=lg, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        s1 = cache.stats()
        cache.close()
        hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
        pcie = (s1["fill_bytes"] - s0["fill_bytes"]) + (s1["stage_bytes"] - s0["stage_bytes"])
        tokens = sum(st[0]["T"] for st in trace[calib:])
        res[name] = {"miss_rate": misses / max(hits + misses, 1), "pcie_GB_per_step": pcie / K / 1e9,
                     "tokens_per_s": tokens / (e0.elapsed_time(e1) * 1e-3),
                     "resident_keys": int(s1["resident"])}
    line = {
        "metric": "decode tokens/s by cache policy (%d-layer 35B-A3B-shaped BF16 trace, cache 37%% of pool)"
                  % layers,
        "value": res["global_lru"]["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": calib, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "policy_compare", "layers": layers, "experts": cfg.experts,
                   "hidden": cfg.hidden, "inter": cfg.inter, "top_k": cfg.top_k, "cache_slots": C,
                   "tokens_per_step": "1..16 (seeded mix)", "calibration_steps": calib,
                   "pool": "pinned host, %d keys on %d blobs" % (cfg.keys, pool.images)},
        "extras": {"policies": res},
    }
    print(json.dumps(line), flush=True)


def chained_line(args):
    """Chained decode through 8 layers of the 35B-A3B shape: each layer's input is the previous
    layer's input plus its output (bf16), every layer's router runs on the device inside the
    forward call, and one global LRU (37 % of the pool) serves all layers. Run twice on the same
    inputs: plain, and with the layer-ahead prefetch, where the next layer's router is applied
    to the current layer's input on a side stream (a predictor of its routing) and
    ft_cache_prefetch starts those experts' copies while the current layer still computes.
    Reports tokens/s through all layers, the fill lead (how long before the previous layer's
    end a layer's first copy starts) and the cache counts of both runs."""
    import torch
    import workloads as W
    from workloads.host import HostPool
    from expert_cached_sparse_top_b300 import build as b
    b.build()
    from expert_cached_sparse_top_b300 import ftmoe
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    ov = {"layers": args.layers} if args.layers else {}
    cfg = W.config("decode_chained", **ov)
    C = W.cache_capacity(cfg)
    pool = HostPool(cfg, images=cfg.experts)           # key -> blob key % E (PCIe bytes real)
    router = W.router_weights(cfg)
    wr = torch.from_numpy(router).to(dev)
    K, Wm = args.steps, args.warmup
    xin = W.chained_inputs(cfg, Wm + K)
    x0 = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev) for x in xin]
    Ts = [x.shape[0] for x in xin]
    L, E, k, H = cfg.layers, cfg.experts, cfg.top_k, cfg.hidden
    s = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    lib = ftmoe.lib()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def run(prefetch):
        c = ftmoe.make_config(L, E, H, cfg.inter, k, cfg.t_max, cfg.wfmt, C)
        cache = ftmoe.MoECache(c, pool.ptrs, router)
        out = torch.empty((cfg.t_max, H), dtype=torch.bfloat16, device=dev)
        xs = torch.empty((L + 1, cfg.t_max, H), dtype=torch.bfloat16, device=dev)
        lg = torch.empty((cfg.t_max, E), dtype=torch.float32, device=dev)
        pidx = torch.empty((cfg.t_max * k,), dtype=torch.int32, device=dev)
        pw = torch.empty((cfg.t_max * k,), dtype=torch.float32, device=dev)
        ready = torch.cuda.Event()

        def step(i):
            T = Ts[i]
            xs[0, :T].copy_(x0[i])
            for l in range(L):
                if prefetch and l + 1 < L:
                    # the next layer's router on this layer's input, on the side stream
                    ready.record(s)
                    side.wait_event(ready)
                    check = lib.ft_router_logits(xs[l].data_ptr(), T, H, wr[l + 1].data_ptr(), E,
                                                 lg.data_ptr(), side.cuda_stream)
                    check |= lib.ft_topk_softmax(lg.data_ptr(), T, E, k, pidx.data_ptr(), pw.data_ptr(),
                                                 side.cuda_stream)
                    if check:
                        raise RuntimeError("stage call failed")
                cache.forward(l, xs[l], T, out, stream=s)
                if prefetch and l + 1 < L:
                    cache.prefetch(l + 1, pidx, n=T * k, stream=side)
                torch.add(xs[l, :T], out[:T], out=xs[l + 1, :T])

        for i in range(Wm):
            step(i)
        torch.cuda.synchronize()
        s0 = cache.stats()
        cache.set_timing(True)
        cache.timing(reset=True)
        evs = []
        for j in range(K):
            l2_flush(flush, args.flush)
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            step(Wm + j)
            e.record(s)
            evs.append((a, e))
        torch.cuda.synchronize()
        tim = cache.timing(reset=True)
        s1 = cache.stats()
        cache.close()
        sec = sum(a.elapsed_time(e) for a, e in evs) / 1e3
        d = {k2: s1[k2] - s0[k2] for k2 in ("hits", "misses", "bypassed", "fill_bytes", "stage_bytes",
                                              "prefetch_fills", "prefetch_bytes", "prefetch_skipped")}
        return {"tokens_per_s": sum(Ts[Wm:]) / sec, "ms_per_step": 1e3 * sec / K,
                "misses_per_step": d["misses"] / K, "hits_per_step": d["hits"] / K,
                "prefetch_fills_per_step": d["prefetch_fills"] / K,
                "pcie_GB_per_step": (d["fill_bytes"] + d["stage_bytes"] + d["prefetch_bytes"]) / K / 1e9,
                "fill_lead_us": 1e3 * tim["fill_lead_ms"] / max(tim["fill_lead_calls"], 1),
                "fill_lead_calls": int(tim["fill_lead_calls"]),
                "fill_ms_per_step": (tim["fill_ms"] + tim["prefetch_fill_ms"]) / K,
                "prefetch_wait_ms_per_step": tim["prefetch_wait_ms"] / K,
                "ffn_GBps": tim["ffn_weight_bytes"] / ((tim["ffn_hit_ms"] + tim["ffn_miss_ms"]) * 1e-3) / 1e9
                if tim["ffn_hit_ms"] + tim["ffn_miss_ms"] > 0 else None,
                "kernel_launches": int(tim["kernel_launches"])}

    plain = run(False)
    ahead = run(True)
    peaks = _peaks()
    hbm = peaks.get("hbm_gbs")
    return {
        "metric": "MoE decode tokens/s through %d chained 35B-A3B-shaped BF16 layers (router in the "
                  "loop, one global LRU at 37%% of pool) with layer-ahead prefetch" % L,
        "value": ahead["tokens_per_s"], "unit": "tokens/s", "steps": K, "warmup": Wm,
        "ms_per_step": ahead["ms_per_step"], "dtype": "bf16",
        "config": {"workload": "decode_chained", "layers": L, "hidden": H, "experts": E,
                   "inter": cfg.inter, "top_k": k, "cache_slots": C,
                   "tokens_per_step": "%d..%d (seeded mix)" % (cfg.t_min, cfg.t_max),
                   "predictor": "next layer's router on the current layer's input (side stream)",
                   "inputs": "first-layer inputs AR(1) across steps, correlation %.2f" % cfg.x_corr,
                   "pool": "pinned host, %d keys on %d blobs" % (cfg.keys, pool.images)},
        "roofline": {"bound": "hbm", "kernel": "expert FFN (tcgen05 grouped GEMM), per pass",
                     "achieved": ahead["ffn_GBps"], "peak": hbm, "unit": "GB/s",
                     "frac": ahead["ffn_GBps"] / hbm if (ahead["ffn_GBps"] and hbm) else None},
        "extras": {"with_prefetch": ahead, "without_prefetch": plain,
                   "speedup": ahead["tokens_per_s"] / plain["tokens_per_s"]},
    }


def run_prefill(args):
    print(json.dumps(prefill_line(args)), flush=True)


def prefill_line(args):
    """Prefill on the 35B-A3B-shaped layer (config 4's literal reading): 4096 tokens,
    near-uniform logits N(0, 0.5), ~256 tokens per expert; layers streamed double-buffered.
    Two numbers: (a) layers in order, every layer's 1.2 GB copied over PCIe (the method's
    prefill), (b) compute only, the same layer again (weights resident): grouped-GEMM
    tensor throughput against the measured BF16 peak."""
    import torch
    import workloads as W
    from workloads.host import HostPool
    from expert_cached_sparse_top_b300 import build as b
    b.build()
    from expert_cached_sparse_top_b300 import ftmoe
    ov = {"layers": args.layers} if args.layers else {}
    if args.tokens:
        ov["tokens"] = args.tokens
    if getattr(args, "experts", 0):
        ov["experts"] = args.experts
    cfg = W.config(args.workload, **ov)
    torch.cuda.set_device(0)
    fp4 = cfg.wfmt != "bf16"
    # the 256-expert MXFP4 layer aliases 16 physical blobs (keys and PCIe bytes unchanged)
    pool = HostPool(cfg, images=16 if fp4 else cfg.experts + 3)
    T = cfg.tokens
    c = ftmoe.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, 16, cfg.wfmt,
                          1, max_prefill_tokens=T)
    cache = ftmoe.MoECache(c, pool.ptrs, None)
    xs, ls = [], []
    for l in range(cfg.layers):
        x, lg = W.prefill_inputs(cfg, l)
        xs.append(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda())
        ls.append(torch.from_numpy(lg).cuda())
    out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    # (a) streaming: layers in order, twice (warm-up pass, then timed pass)
    for l in range(cfg.layers):
        cache.prefill(l, xs[l], T, out, logits=ls[l])
    torch.cuda.synchronize()
    cache.set_timing(True); cache.timing(reset=True)
    t0 = time.perf_counter()
    for l in range(cfg.layers):
        cache.prefill(l, xs[l], T, out, logits=ls[l])
    torch.cuda.synchronize()
    stream_s = time.perf_counter() - t0
    ts = cache.timing(reset=True)
    # (b) compute only: last layer again and again (already resident)
    last = cfg.layers - 1
    for _ in range(args.warmup):
        cache.prefill(last, xs[last], T, out, logits=ls[last])
    torch.cuda.synchronize()
    cache.timing(reset=True)
    evs = []
    for _ in range(args.steps):
        l2_flush(flush, args.flush)
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(); cache.prefill(last, xs[last], T, out, logits=ls[last]); e.record()
        evs.append((a, e))
    torch.cuda.synchronize()
    tc = cache.timing(reset=True)
    cache.close()
    layer_ms = sum(a.elapsed_time(e) for a, e in evs) / len(evs)
    peaks = _peaks()
    bf16 = peaks.get("bf16_tflops")
    hbm = peaks.get("hbm_gbs", 6487.4)
    ffn_ms = tc["prefill_ffn_ms"] / max(tc["prefill_calls"], 1)
    ffn_tflops = tc["prefill_flops"] / (tc["prefill_ffn_ms"] * 1e-3) / 1e12
    wbytes = cfg.experts * pool.blob_bytes
    ceiling = (6.0 * T * cfg.top_k * cfg.hidden * cfg.inter) / (wbytes / (hbm * 1e9)) / 1e12
    if fp4:
        # ~96 tokens per expert: the layer's weights bound it (the HBM ceiling is far below the
        # FP4 tensor peak), so the roofline is weight bytes per FFN second against HBM
        gbs = wbytes / (ffn_ms * 1e-3) / 1e9
        probe = getattr(args, "fp4_peak", None) or fp4_peak_probe()
        # FP4 dense peak: the measured BF16 peak x the nominal FP4 / BF16 ratio (13.5 / 2.25);
        # the activations enter the MMA as four E2M1 pieces, so the tensor pipe issues 4x the
        # useful flops and the tensor-bound ceiling of useful flops is a quarter of that peak
        fp4_peak = bf16 * 6.0 if bf16 else None
        pieces = 4
        tensor_ceiling = fp4_peak / pieces if fp4_peak else None
        ceil = min(ceiling, tensor_ceiling) if tensor_ceiling else ceiling
        roof = {"bound": "hbm", "kernel": "block-scaled tcgen05 grouped GEMM (%s weights x bf16 activations "
                                          "as four E2M1 pieces: W13+SwiGLU, W2)" % cfg.wfmt.upper(),
                "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                "peak_source": "MEASURED_PEAKS.json hbm_gbs", "tflops": ffn_tflops,
                "tensor_tflops_issued": ffn_tflops * pieces,
                "hbm_bound_ceiling_tflops": ceiling, "frac_of_hbm_ceiling": ffn_tflops / ceiling,
                "fp4_peak_tflops": fp4_peak,
                "fp4_peak_source": "MEASURED_PEAKS.json bf16_tflops x 6 (nominal FP4 / BF16 dense ratio)",
                "frac_of_fp4_peak": (ffn_tflops * pieces / fp4_peak) if fp4_peak else None,
                "cublaslt_nvfp4_probe_tflops": probe["tflops"], "cublaslt_nvfp4_probe_source": probe["source"],
                "ceiling_tflops": ceil, "frac_of_ceiling": ffn_tflops / ceil}
        metric = ("MoE-layer prefill tokens/s (284B-shaped MXFP4 layer, 256 experts top-6, %d tokens, "
                  "layers streamed)" % T)
    else:
        roof = {"bound": "tensor", "kernel": "tcgen05 grouped GEMM (W13+SwiGLU, W2)",
                "achieved": ffn_tflops, "peak": bf16, "unit": "TFLOP/s",
                "frac": ffn_tflops / bf16 if bf16 else None, "traffic": None,
                "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst)",
                "hbm_bound_ceiling_tflops": ceiling}
        metric = "MoE-layer prefill tokens/s (35B-A3B-shaped BF16 layer, %d tokens, layers streamed)" % T
    line = {
        "metric": metric,
        "value": T * cfg.layers / stream_s, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * stream_s / cfg.layers,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("%s weights x bf16 activations (four E2M1 pieces)" % cfg.wfmt) if fp4 else "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "tokens": T, "experts": cfg.experts, "top_k": cfg.top_k,
                   "hidden": cfg.hidden, "inter": cfg.inter, "layers": cfg.layers,
                   "pool": "pinned host, %d blobs x %d B%s" % (pool.images, pool.blob_bytes,
                                                             " (keys aliased)" if fp4 else ""),
                   "l2": "flushed before every compute-only step"},
        "roofline": roof,
        "extras": {"compute_only_layer_ms": layer_ms,
                   "compute_only_tokens_per_s": T / (layer_ms * 1e-3),
                   "ffn_ms_per_layer": tc["prefill_ffn_ms"] / max(tc["prefill_calls"], 1),
                   "stream_fill_ms_per_layer": ts["prefill_fill_ms"] / max(cfg.layers, 1),
                   "stream_compute_ms_per_layer": ts["prefill_compute_ms"] / max(ts["prefill_calls"], 1),
                   "pcie_GBps": ts["prefill_fill_bytes"] / (ts["prefill_fill_ms"] * 1e-3) / 1e9
                   if ts["prefill_fill_ms"] > 0 else None,
                   "layer_weight_bytes": wbytes},
    }
    return line


# The FP4 tensor-core peak is not in MEASURED_PEAKS.json. It is measured here, in the same
# process, with cuBLASLt's block-scaled NVFP4 GEMM (torch._scaled_mm, 8192^3, best of 10
# back-to-back launches after a warm-up, CUDA events); where that call is unavailable the
# value measured the same way on this machine earlier is reported, labelled as such.
FP4_PEAK_EARLIER = 6740.0


def fp4_peak_probe(n=8192, reps=10):
    import torch
    try:
        dev = torch.device("cuda", torch.cuda.current_device())
        a = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
        b = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
        # per-16 E4M3 block scales in the swizzled 128 x 4 layout: (n / 128) x (n / 64) atoms
        sa = torch.full((n * (n // 16),), 1.0, device=dev).to(torch.float8_e4m3fn)
        sb = torch.full((n * (n // 16),), 1.0, device=dev).to(torch.float8_e4m3fn)
        run = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(); run(); e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, sa, sb
        return {"tflops": 2.0 * n ** 3 / (best * 1e-3) / 1e12,
                "source": "measured in this run: cuBLASLt NVFP4 block-scaled GEMM (torch._scaled_mm), "
                          "%d^3, best of %d, burst" % (n, reps)}
    except Exception as e:  # noqa: BLE001 - the probe is optional; its absence is reported
        return {"tflops": FP4_PEAK_EARLIER,
                "source": "measured earlier on this pool the same way (cuBLASLt NVFP4 %d^3, burst); "
                          "the live probe failed here: %s" % (n, str(e).splitlines()[0][:160])}


SUB_RECORDS = (
    # name, workload, steps, warmup, extra settings
    ("decode_mxfp4", "decode_mxfp4", 8, 4, {}),
    ("elastic_nvfp4", "elastic_nvfp4", 96, 16, {}),
    ("prefill_mxfp4", "prefill_mxfp4", 8, 3, {}),
    ("prefill_bf16", "prefill_bf16", 8, 3, {}),
    ("decode_chained", "decode_chained", 16, 4, {}),
)


def sub_records(args):
    """The rest of the metric, measured in the default run after the headline: 43-layer MXFP4
    decode, elastic NVFP4 decode, and MXFP4 / BF16 prefill at 4096 tokens, each with its own
    CUDA-event timing and roofline block. Decode sub-records skip the end-to-end pass and the
    oracle baseline (the headline carries both)."""
    import torch
    out = {}
    fp4 = None
    for name, wl, steps, warmup, extra in SUB_RECORDS:
        a = argparse.Namespace(**vars(args))
        a.workload, a.steps, a.warmup, a.lite = wl, steps, warmup, True
        a.layers, a.tokens, a.fused, a.ffn_traffic, a.all_resident, a.experts = 0, 0, False, False, False, 0
        for k2, v in extra.items():
            setattr(a, k2, v)
        t0 = time.perf_counter()
        try:
            if wl in DECODE:
                line = decode_line(a)
            elif wl == "decode_chained":
                line = chained_line(a)
            else:
                if fp4 is None and wl == "prefill_mxfp4":
                    fp4 = fp4_peak_probe()
                a.fp4_peak = fp4
                line = prefill_line(a)
        except Exception as e:  # noqa: BLE001 - a failed sub-record must not hide the headline
            out[name] = {"error": "%s: %s" % (type(e).__name__, (str(e).splitlines() or [""])[0][:200])}
            line = None
        try:
            torch.cuda.synchronize()
        except Exception:  # noqa: BLE001
            pass
        if line is None:
            continue
        for k2 in ("n_gpus", "higher_is_better", "scaling", "vs_baseline", "data", "cpu_baseline",
                   "e2e", "clocks"):
            line.pop(k2, None)
        line["wall_s"] = time.perf_counter() - t0
        out[name] = line
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="fewer MoE layers than the workload defines (profiling runs)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prefill: tokens per layer (default 4096); decode: a fixed number of "
                         "tokens per step instead of the seeded 1..16 mix")
    ap.add_argument("--ffn-traffic", action="store_true",
                    help="decode: run the cached pass only and print the FFN launches and their "
                         "algorithmic bytes (the denominator of an ncu traffic capture)")
    ap.add_argument("--clocks-csv", default=None,
                    help="where the nvidia-smi samples of the timed region go (a %%d takes the "
                         "rank; default: the temp directory)")
    ap.add_argument("--all-resident", action="store_true",
                    help="with --ffn-traffic: every selected expert resident (no fills)")
    ap.add_argument("--fused", action="store_true",
                    help="decode through the fused decode kernel (FT_FLAG_FUSED_DECODE; BF16)")
    ap.add_argument("--experts", type=int, default=0,
                    help="prefill: fewer experts per layer (a small case of the same kernel for "
                         "profiler captures; with --tokens keeping the tokens per expert)")
    ap.add_argument("--flush", choices=FLUSH_MODES, default="write-read",
                    help="L2 flush between timed steps: write a 256 MB buffer and read it back "
                         "(default), or only write it")
    ap.add_argument("--no-extras", action="store_true",
                    help="default run: skip the sub-records of the other workloads")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=list(DECODE) + ["prefill_bf16", "prefill_mxfp4", "policy_compare",
                                            "decode_chained"])
    args = ap.parse_args()
    dflt = DECODE.get(args.workload, (None, None, {"policy_compare": 32, "decode_chained": 16}.get(
        args.workload, 8), 3 if args.workload != "decode_chained" else 4))
    if args.steps is None:
        args.steps = dflt[2]
    if args.warmup is None:
        args.warmup = dflt[3]
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.workload == "policy_compare":
        run_policy_compare(args)
    elif args.workload == "decode_chained":
        print(json.dumps(chained_line(args)), flush=True)
    elif args.workload not in DECODE:
        run_prefill(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
