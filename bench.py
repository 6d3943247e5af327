#!/usr/bin/env python
"""MoE-layer tokens/s of the host-resident-expert MoE layer on B300.

Default workload: decode through a 35B-A3B-shaped stack.  48 MoE layers,
hidden 2048, 128 experts per layer, top-8, intermediate 768, NVFP4 weights.
One token per step, router logits N(0,1) plus a per-expert Zipf(1.1) bias,
and one global LRU cache of 1024 GPU slots over the 6144 experts in pinned
host RAM.  One step is one token through all 48 layers: the whole hot path
(route, slot lookup + LRU update, miss copies, permute, SwiGLU FFN, combine)
48 times.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is device-resident throughput (inputs already
in HBM).  `e2e` adds the per-step host->device copy of the inputs and the
device->host read of the outputs, issued on copy streams of their own and
overlapped with the neighbouring steps' compute.  Under torchrun (N > 1) every rank runs an
independent replica with its own cache: no collective on the data path,
"scaling": "weak".  `--impl reference` times the CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import ftgen  # noqa: E402
from ftgen.configs import CONFIGS, epoch_at, tokens_at  # noqa: E402

METRIC = "MoE-layer tokens/s (decode & prefill) + % of HBM/PCIe/tensor roofline, 1xB300"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, src="fallback")


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, device=None):
    """The largest x over the ranks of the initialised process group (x when
    there is none): each replica's timed window ends when its slowest peer's
    does."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world_size, ms_max):
    """Whole-job throughput: every rank processed units_per_rank in ms_max."""
    return units_per_rank * world_size / (ms_max * 1e-3)


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"ft_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", self.gpu_id], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _gpu_id(dev):
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return str(dev)


def _pcie_h2d_gbs(torch, dev, pool):
    """Pinned host -> device, 256 MiB cudaMemcpyAsync from the expert pool's
    own pinned buffer (the memory miss copies read), best of 10 (GB/s)."""
    n = min(256 << 20, pool.numel())
    h = pool[:n]
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    best = 1e30
    with torch.cuda.stream(s):
        for i in range(12):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            d.copy_(h, non_blocking=True)
            e1.record(s)
            e1.synchronize()
            if i >= 2:
                best = min(best, e0.elapsed_time(e1))
    del d
    return n / (best * 1e-3) / 1e9


def _gen_inputs(cfg, seed, n_steps):
    """x bf16 bits [steps, L, T, H] and logits f32 [steps, L, T, E] (T = max tokens)."""
    T, H, E, L = cfg["T"], cfg["H"], cfg["E"], cfg["L"]
    X = np.zeros((n_steps, L, T, H), np.uint16)
    G = np.zeros((n_steps, L, T, E), np.float32)
    for s in range(n_steps):
        t = tokens_at(cfg, s)
        for l in range(L):
            X[s, l, :t] = ftgen.x_bf16(seed, t, H, s, l)
            G[s, l, :t] = ftgen.router_logits(seed, t, E, s, l, cfg["zipf"], epoch_at(cfg, s))
    return X, G


class _OracleRunner:
    """The CPU oracle over the workload's calls, in order (step-major, then
    layer).  Blobs are generated before any call is timed.  Prefill workloads
    (one chunk per step) reuse the step-0 inputs, as the GPU bench does."""

    def __init__(self, cfg, seed, n_phys, max_calls, fmt=None):
        import oracle as O
        self.cfg, self.seed = cfg, seed
        self.fmt = fmt or cfg["fmt"]
        self.prefill = cfg["steps"] == 1
        H, E, k, I, L = cfg["H"], cfg["E"], cfg["k"], cfg["I"], cfg["L"]
        # sampled token rows per call: every token of a decode call; for a
        # prefill chunk a strided sample, smaller for the large expert shapes
        # (the oracle dequantises every expert a sampled token touches)
        self.n_sample = 256 if H * I <= 2048 * 768 else 4
        self.calls = []
        step = 0
        while len(self.calls) < max_calls:
            for l in range(L):
                if len(self.calls) < max_calls:
                    self.calls.append((0 if self.prefill else step, l, tokens_at(cfg, step)))
            step += 1
        need = set()
        for step, l, T in self.calls:
            lg = ftgen.router_logits(seed, T, E, step, l, cfg["zipf"], epoch_at(cfg, step))
            idx = O.topk_experts(lg, k)
            rows = self._sample(T)
            if rows is not None:
                idx = idx[rows]
            need |= {(l * E + int(e)) % n_phys for e in idx.reshape(-1)}
        need = sorted(need)
        blobs = ftgen.pool(self.fmt, H, I, need, seed)
        self.blobs = {p: blobs[i] for i, p in enumerate(need)}
        self.orc = O.MoELayerOracle(H, E, k, I, ftgen.FMT_NAMES[self.fmt], cfg["S"], L,
                                    lambda key: self.blobs[key % n_phys],
                                    mode=O.MODE_STREAM if cfg["mode"] == "stream" else O.MODE_LRU)
        self.pos = 0

    def _sample(self, T):
        return None if T <= 64 else list(range(0, T, max(1, T // self.n_sample)))[: self.n_sample]

    def next_call(self, one_expert=False):
        """Runs the next call; returns (seconds, token rows, distinct experts).
        one_expert: evaluate the FFN of only one of the call's experts (the
        (call index mod n)-th), a bounded timing sample."""
        import oracle as O
        cfg = self.cfg
        step, l, T = self.calls[self.pos]
        self.pos += 1
        x = ftgen.x_bf16(self.seed, T, cfg["H"], step, l)
        lg = ftgen.router_logits(self.seed, T, cfg["E"], step, l, cfg["zipf"], epoch_at(cfg, step))
        sample = self._sample(T)
        experts = sorted(set(int(e) for e in O.topk_experts(lg, cfg["k"]).reshape(-1)))
        sub = [experts[self.pos % len(experts)]] if one_expert else None
        t0 = time.perf_counter()
        self.orc.forward(l, x, lg, tokens=sample, ffn_experts=sub)
        return time.perf_counter() - t0, (T if sample is None else len(sample)), len(experts)


def _single_thread():
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(1)
    except ImportError:  # pragma: no cover
        import contextlib
        return contextlib.nullcontext()


def _cpu_baseline(cfg, seed, n_phys, budget_s=15.0, max_calls=192, fmt=None):
    """Times the CPU oracle, as it stands, single-threaded, on the workload's
    first layer calls until `budget_s` seconds of oracle time.
    Returns (tokens/s through the L-layer stack, description, calls, seconds)."""
    if cfg["steps"] == 1:
        max_calls = min(max_calls, 2)
    run = _OracleRunner(cfg, seed, n_phys, max_calls, fmt)
    calls, rows, used = 0, 0, 0.0
    with _single_thread():
        while used < budget_s and run.pos < len(run.calls):
            dt, r, _ = run.next_call()
            used += dt
            rows += r
            calls += 1
    L = cfg["L"]
    desc = (f"oracle on the first {calls} layer calls of {cfg['name']} in order ({rows} token rows"
            f"{' sampled from each chunk' if cfg['steps'] == 1 else ''}, routing of every token, FFN of the "
            f"sampled rows), float64 numpy, 1 thread; tokens/s = rows / {L} layers / seconds")
    return rows / L / used, desc, calls, used


def run_reference(args, cfg):
    """The CPU oracle as the reference arm: step i = layer call i of the
    workload (a bounded sample); tokens/s = tokens / (L x mean seconds per call)."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    run = _OracleRunner(cfg, cfg["seed"], args.n_phys, args.warmup + args.steps)
    est, rows = [], 0
    with _single_thread():
        for i in range(args.warmup + args.steps):
            dt, r, n_exp = run.next_call(one_expert=True)
            if i >= args.warmup:
                est.append(dt * n_exp)     # the full call evaluates n_exp experts
                rows += r
    secs = sum(est)
    value = rows / cfg["L"] / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg["name"], "layers": cfg["L"], "tokens_per_step": cfg["T"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"step i = layer call i of {cfg['name']}: routing + LRU in full, FFN of one of "
                                   f"its distinct experts; call time estimated as step time x distinct experts; "
                                   f"value = token rows / {cfg['L']} layers / estimated seconds"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _ffn_bytes(fmt, H, I):
    """Weight bytes of one expert's gate/up and down matrices."""
    HI = H * I
    if fmt == "nvfp4":
        return 2 * HI // 2 + 2 * HI // 16, HI // 2 + HI // 16
    if fmt == "mxfp4":
        return 2 * HI // 2 + 2 * HI // 32, HI // 2 + HI // 32
    if fmt == "fp8":
        return 2 * HI + 8 * I, HI + 4 * H
    return 4 * HI, 2 * HI


def _resize_probe(torch, dev, stack, S):
    """After the timed runs: the slot count halved and restored
    (ft_moe_resize_slots), wall time of each call and the device memory it
    returned."""
    try:
        out = {"from": S, "to": S // 2}
        for key, n in (("shrink", S // 2), ("grow", S)):
            torch.cuda.synchronize(dev)
            free0 = torch.cuda.mem_get_info(dev)[0]
            t0 = time.perf_counter()
            stack.resize_slots(n)
            out[key + "_ms"] = (time.perf_counter() - t0) * 1e3
            out[key + "_gb_freed"] = (torch.cuda.mem_get_info(dev)[0] - free0) / 1e9
        return out
    except Exception as e:  # reported, not fatal: the measured line stands
        return {"error": str(e)[:200]}


def _host_cpu():
    """The host's CPU model and logical core count."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    return {"host_cores": os.cpu_count(), "cpu_model": model}


# Further workloads measured after the headline one by the default run (one
# GPU): the prefill layer of the same 35B-A3B shape with BF16 and NVFP4 experts
# (all resident: tensor-core bound), and the 753B-shaped whole-layer streaming
# prefill (PCIe bound).  Each gets its own device time, end-to-end time and
# rooflines, under "workloads" in the same JSON line.
EXTRA_WORKLOADS = (
    ("prefill35b_bf16", "prefill35b", dict(fmt="bf16", act="bf16", steps=5, warmup=3, profile_steps=2, n_phys=128)),
    ("prefill35b_nvfp4", "prefill35b", dict(fmt="nvfp4", act="bf16", steps=5, warmup=3, profile_steps=2, n_phys=128)),
    ("prefill35b_nvfp4_fp4act", "prefill35b",
     dict(fmt="nvfp4", act="fp4", steps=5, warmup=3, profile_steps=2, n_phys=128)),
    ("stream753b", "stream753b", dict(fmt=None, act="bf16", steps=2, warmup=3, profile_steps=1, n_phys=512)),
    # every expert of the 48-layer stack resident (6144 slots, 16.3 GB): no misses, the GEMV's HBM rate
    ("decode35b_resident", "decode35b",
     dict(fmt=None, act="bf16", steps=20, warmup=5, profile_steps=8, n_phys=768, slots=6144)),
)

_FP4_PEAK = {}


def kernel_sources_sha():
    """sha256 of the library's CUDA sources (every file under the package's
    csrc/, in name order): the kernels that a stored ncu capture measured."""
    import hashlib
    d = os.path.join(ROOT, "expert_cache_host_softmax_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def stored_traffic(workload, kernel):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    committed ncu summary table (profiles/traffic.json), or None when the table
    has no entry or was taken on other kernel sources than these."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    t = json.load(open(p))
    if t.get("kernel_sources_sha") != kernel_sources_sha():
        return None
    e = t.get("workloads", {}).get(workload, {}).get(kernel)
    return None if e is None else float(e["dram_bytes_per_launch"])


def fp4_peak(n_tile=256):
    """The block-scaled FP4 tensor-core rate measured by the library's probe
    (ft_fp4_tensor_peak: MMAs on operands already in shared memory), best of 3
    after one warm-up launch, TFLOP/s; cached per process."""
    if n_tile not in _FP4_PEAK:
        import expert_cache_host_softmax_b300 as F
        F.fp4_tensor_peak(n_tile, 2000)
        _FP4_PEAK[n_tile] = max(F.fp4_tensor_peak(n_tile, 20000) for _ in range(3))
    return _FP4_PEAK[n_tile]


def run_ours(args, cfg):
    import torch
    from __graft_entry__ import build
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build()
    line = _measure(args, cfg, dev, ws, rank)
    line["fp4_tensor_peak_tflops"] = {"n256": fp4_peak(256), "n128": fp4_peak(128),
                                      "how": "ft_fp4_tensor_peak: one CTA per SM, tcgen05.mma kind::mxf4nvf4 "
                                             "(M=128, K=64, E4M3 scale per 16) on operands in shared memory, "
                                             "best of 3 launches of 20000 x 4 MMAs, CUDA events"}
    if rank == 0 and not args.no_cpu_baseline:
        tps, desc, calls, secs = _cpu_baseline(cfg, cfg["seed"], min(args.n_phys, cfg["L"] * cfg["E"]),
                                               budget_s=args.cpu_budget, fmt=args.fmt or cfg["fmt"])
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                                "seconds": secs, **_host_cpu()}
    if args.extras and ws == 1:
        line["workloads"] = {}
        for name, cname, opts in EXTRA_WORKLOADS:
            sub = argparse.Namespace(**{**vars(args), **opts, "fmt": opts["fmt"], "act": opts["act"], "hit_d2d_cache": 0,
                                        "ffn": "auto", "miss_path": "auto", "fused_decode": False})
            try:
                wcfg = dict(CONFIGS[cname], S=opts["slots"]) if "slots" in opts else CONFIGS[cname]
                w = _measure(sub, wcfg, dev, ws, rank, resize=False)
                keep = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "e2e",
                        "gpu_launches", "roofline", "path_roofline", "clocks")
                line["workloads"][name] = {key_: w[key_] for key_ in keep}
            except Exception as e:  # reported in the line; the headline stands
                line["workloads"][name] = {"error": str(e)[:300]}
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _measure(args, cfg, dev, ws, rank, resize=True):
    """One workload on this rank's GPU: device-resident timing, end-to-end
    timing, the per-kernel pass and the rooflines.  Returns the JSON line
    (without cpu_baseline)."""
    import torch
    import expert_cache_host_softmax_b300 as F
    peaks = _peaks()
    seed = cfg["seed"] + rank
    T, H, E, k, I, L, S = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["I"], cfg["L"], cfg["S"]
    fmt = args.fmt or cfg["fmt"]
    # prefill hit-D2D: cache slots beyond the two staging banks; the load-time
    # warm fill leaves keys 0..S+C-1 in them and the switch to STREAM mode keeps
    # the C most recent (keys S..S+C-1), which staging then copies on the device
    d2d_cache = args.hit_d2d_cache if cfg["mode"] == "stream" else 0
    S += d2d_cache
    # prefill workloads: one chunk through the stack per step, same inputs each
    # step; with resident experts, L2 is flushed before every timed step (the
    # streaming workload copies every expert from host memory each step, and
    # is timed as one window so that the copy of the next step's first layer,
    # which overlaps the last layer, stays inside it); decode: fresh inputs per step
    reuse_inputs = cfg["steps"] == 1
    prefill = reuse_inputs and cfg["mode"] != "stream"
    nb = ftgen.blob_bytes(fmt, H, I)
    n_keys = L * E
    n_phys = min(args.n_phys, n_keys)

    # pinned host pool: n_phys distinct blobs, logical key -> key % n_phys
    pool = torch.empty(n_phys * nb, dtype=torch.uint8, pin_memory=True)
    ftgen.pool(fmt, H, I, list(range(n_phys)), seed, out=pool.numpy().reshape(n_phys, nb))
    ptrs = [pool.data_ptr() + (key % n_phys) * nb for key in range(n_keys)]
    stack = F.MoELayerStack(H, E, k, I, fmt, S, L, T)
    stack.load_pool(ptrs, keepalive=pool)
    if d2d_cache > 0:
        stack.set_prefill_hit_d2d(True)
    if cfg["mode"] == "stream":
        stack.set_mode(F.FT_MODE_STREAM)
    if args.ffn != "auto":
        stack.set_ffn_kernel(args.ffn)
    if args.miss_path != "auto":
        stack.set_miss_path(args.miss_path)
    if args.fused_decode:
        stack.set_decode_fusion(True)
    if getattr(args, "no_decode_grid", False):
        stack.set_decode_grid(False)
    fp4_act = getattr(args, "act", "bf16") == "fp4"
    if fp4_act:
        stack.set_act_format("fp4")

    W, K = args.warmup, args.steps
    n_prof = min(args.profile_steps, K)
    n_steps = W + K
    n_in = 1 if reuse_inputs else n_steps
    X, G = _gen_inputs(cfg, seed, n_in)
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).to(dev)
    Gd = torch.from_numpy(G).to(dev)
    outd = torch.empty((L, T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    Lb = F.lib()
    h = stack._h
    x_ptr0, g_ptr0, o_ptr0 = Xd.data_ptr(), Gd.data_ptr(), outd.data_ptr()
    xs, gs, os_ = T * H * 2, T * E * 4, T * H * 2
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if prefill else None

    def step(s, xb=None, gb=None, ob=None):
        t = tokens_at(cfg, s)
        si = 0 if reuse_inputs else s
        ob = o_ptr0 if ob is None else ob
        for l in range(L):
            xo = (xb + l * xs) if xb is not None else x_ptr0 + (si * L + l) * xs
            go = (gb + l * gs) if gb is not None else g_ptr0 + (si * L + l) * gs
            rc = Lb.ft_moe_forward(h, l, t, xo, go, ob + l * os_, sp)
            if rc != 0:
                raise F.FtError(rc, Lb.ft_last_error(h).decode())

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def flush_l2():
        # write a buffer twice the size of L2 on the bench stream, outside the timed events
        with torch.cuda.stream(stream):
            flush_buf.zero_()

    def timed_steps(steps, body):
        """Device time (ms) of `body(s)` over `steps`: one event pair around all
        of them (decode), or per step after an L2 flush (prefill)."""
        if not prefill:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for s in steps:
                body(s)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1)
        total = 0.0
        for s in steps:
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            body(s)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            total += e0.elapsed_time(e1)
        return total

    with torch.cuda.stream(stream):
        for s in range(W):
            if prefill:
                flush_l2()
            step(s)
    torch.cuda.synchronize(dev)
    pcie_gbs = _pcie_h2d_gbs(torch, dev, pool)

    # ---- timed region: K steps, inputs resident in HBM
    cum0, _ = stack.stats()
    launches0 = stack.kernel_launches
    sampler = ClockSampler(_gpu_id(dev))
    barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    ms = timed_steps(range(W, W + K), step)
    wall = time.perf_counter() - wall0
    barrier()
    clocks = sampler.stop()
    cum1, _ = stack.stats()
    launches = stack.kernel_launches - launches0
    d = {key_: cum1[key_] - cum0[key_] for key_ in cum1}
    ms_max = max_over_ranks(ms, dev)
    tokens = sum(tokens_at(cfg, s) for s in range(W, W + K))
    value = job_rate(tokens, ws, ms_max)

    # ---- end to end: every step copies its inputs (x, logits) from pinned host
    # memory and reads its output back, all inside one timed window.  The
    # copies run on two streams of their own with two device buffers each way:
    # step s+1's inputs cross PCIe while step s computes, and step s's output
    # comes back while step s+1 computes (the link is full duplex), as a
    # serving loop would overlap them.  Each step still reads its weights from
    # the slot bank (larger than L2) or from host memory.
    # (allocated page-locked from the start: on the B300 machines a host->device
    # copy from these runs at ~55 GB/s, from a tensor pinned afterwards with
    # .pin_memory() at ~11 GB/s)
    Xh = torch.empty(X.shape, dtype=torch.bfloat16, pin_memory=True)
    Xh.view(torch.int16).numpy()[...] = X.view(np.int16)
    Gh = torch.empty(G.shape, dtype=torch.float32, pin_memory=True)
    Gh.numpy()[...] = G
    outh = torch.empty((L, T, H), dtype=torch.bfloat16, pin_memory=True)
    xin = [torch.empty((L, T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    gin = [torch.empty((L, T, E), dtype=torch.float32, device=dev) for _ in range(2)]
    outb = [outd, torch.empty_like(outd)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready, in_free, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    for ev in in_ready + in_free + out_done:
        ev.record(stream)
    barrier()
    torch.cuda.synchronize(dev)

    def e2e_window(steps):
        steps = list(steps)

        def h2d(j):
            b, si = j % 2, 0 if reuse_inputs else steps[j]
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(in_free[b])          # step j-2 is done with buffer b
                xin[b].copy_(Xh[si], non_blocking=True)
                gin[b].copy_(Gh[si], non_blocking=True)
                in_ready[b].record(h2d_s)

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)
        d2h_s.wait_event(e0)
        h2d(0)
        for j, s_ in enumerate(steps):
            b = j % 2
            if j + 1 < len(steps):
                h2d(j + 1)
            stream.wait_event(in_ready[b])
            stream.wait_event(out_done[b])           # step j-2's output has left buffer b
            step(s_, xin[b].data_ptr(), gin[b].data_ptr(), outb[b].data_ptr())
            in_free[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(in_free[b])
                outh.copy_(outb[b], non_blocking=True)
                out_done[b].record(d2h_s)
        stream.wait_event(out_done[(len(steps) - 1) % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    e2e_ms = max_over_ranks(e2e_window(range(W, W + K)), dev)
    e2e_value = job_rate(tokens, ws, e2e_ms)

    # ---- per-kernel timing pass (events around each step class)
    stack.set_profiling(True)
    c0, _ = stack.stats()
    with torch.cuda.stream(stream):
        for s in range(W, W + n_prof):
            if prefill:
                flush_l2()
            step(s)
    torch.cuda.synchronize(dev)
    prof = stack.profile()
    c1, _ = stack.stats()
    stack.set_profiling(False)
    ffn_kernel = stack.last_ffn_kernel
    # GEMV calls with FT_MISS_KERNEL copy their misses inside the gate/up kernel
    in_kernel_copy = cfg["mode"] == "lru" and ffn_kernel == "gemv" and stack.miss_path() == "kernel"
    pd = {key_: c1[key_] - c0[key_] for key_ in c1}

    # algorithmic bytes and FLOPs of the FFN kernels: each distinct expert's
    # weights once per call, plus activations; FLOPs 2 per multiply-add
    gu_bytes, d_bytes = _ffn_bytes(fmt, H, I)
    calls_p = n_prof * L
    toks_p = sum(tokens_at(cfg, s) for s in range(W, W + n_prof)) * L
    # h per (token, expert) pair: bf16, or e2m1 codes plus an E4M3 scale per 16
    h_pair = I // 2 + I // 16 if fp4_act else I * 2
    act_gu = toks_p * H * 2 + toks_p * k * h_pair  # x read once per token (the kernels gather it per pair) + h written
    if ffn_kernel == "tc":
        act_dn = toks_p * k * h_pair + toks_p * H * 4   # h read + the fp32 output rows the epilogue accumulates
    else:
        act_dn = toks_p * k * (I * 2 + H * 4)       # h read + y written per pair
    fl_gu, fl_dn = 2 * toks_p * k * 2 * I * H, 2 * toks_p * k * H * I
    kern = {
        "gateup": (pd["lookups"] * gu_bytes + act_gu, prof["gateup_hit"][0] + prof["gateup_miss"][0], fl_gu),
        "down": (pd["lookups"] * d_bytes + act_dn, prof["down"][0], fl_dn),
        "route": (toks_p * E * 4, prof["route"][0], 0),
        # tensor cores: the fp32 output rows converted to bf16; GEMV: y rows gathered and weighted
        "combine": (toks_p * H * 6 if ffn_kernel == "tc" else toks_p * (k * H * 4 + H * 2), prof["combine"][0], 0),
    }
    if prof.get("layer", (0.0, 0))[1] > 0:
        # decode calls ran as the fused layer kernel: routing, FFN and combine in one launch
        # (its duration includes waiting for the misses' copies)
        kern["decode_layer"] = (pd["lookups"] * (gu_bytes + d_bytes) + act_gu + act_dn + toks_p * (E * 4 + H * 2),
                                prof["layer"][0], fl_gu + fl_dn)
    dom = max(kern, key=lambda n: kern[n][1])
    b_dom, ms_dom, f_dom = kern[dom]
    share = {n: round(kern[n][1] / max(1e-9, sum(v[1] for v in kern.values())), 4) for n in kern}
    if ffn_kernel == "tc" and f_dom > 0:
        achieved = f_dom / (ms_dom * 1e-3) / 1e12 if ms_dom > 0 else 0.0
        if fp4_act:
            t_peak, t_src = fp4_peak(256), "measured FP4 (ft_fp4_tensor_peak, N=256)"
            t_kern = f"{dom} (tcgen05 block-scaled grouped GEMM, FP4 x FP4 operands)"
        else:
            t_peak, t_src = peaks["bf16_tflops"], peaks["src"] + " bf16 burst"
            t_kern = f"{dom} (tcgen05 grouped GEMM, bf16 operands)"
        roofline = {"bound": "tensor", "kernel": t_kern, "achieved": achieved,
                    "peak": t_peak, "unit": "TFLOP/s", "frac": achieved / t_peak,
                    "traffic": None, "peak_src": t_src,
                    "flops_per_call": f_dom / calls_p, "ms_per_call": ms_dom / calls_p,
                    "hbm_gbs_achieved": b_dom / (ms_dom * 1e-3) / 1e9 if ms_dom > 0 else 0.0,
                    "kernel_ms_share": share}
    elif dom == "gateup" and in_kernel_copy and pd["misses"] > 0:
        # the gate/up kernel also copies the misses from host memory, and its
        # duration is set by those PCIe bytes, not by its HBM reads
        pcie_b = pd["misses"] * nb
        achieved = pcie_b / (ms_dom * 1e-3) / 1e9 if ms_dom > 0 else 0.0
        roofline = {"bound": "pcie", "kernel": "gateup (+ the misses' copies from host memory)",
                    "achieved": achieved, "peak": pcie_gbs, "unit": "GB/s", "frac": achieved / pcie_gbs,
                    "traffic": None, "peak_src": "measured (pinned-pool H2D copy)",
                    "pcie_bytes_per_call": pcie_b / calls_p, "hbm_bytes_per_call": b_dom / calls_p,
                    "hbm_gbs_achieved": b_dom / (ms_dom * 1e-3) / 1e9 if ms_dom > 0 else 0.0,
                    "ms_per_call": ms_dom / calls_p, "kernel_ms_share": share}
    else:
        achieved = b_dom / (ms_dom * 1e-3) / 1e9 if ms_dom > 0 else 0.0
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "traffic": None, "peak_src": peaks["src"],
                    "bytes_per_call": b_dom / calls_p, "ms_per_call": ms_dom / calls_p, "kernel_ms_share": share}
    # every FFN kernel's own rates (the dominant one above; all of them here)
    roofline["kernels"] = {
        n: {"ms_per_call": v[1] / calls_p, "algorithmic_bytes_per_call": v[0] / calls_p,
            "hbm_gbs": v[0] / (v[1] * 1e-3) / 1e9 if v[1] > 0 else None,
            "hbm_frac": v[0] / (v[1] * 1e-3) / 1e9 / peaks["hbm_gbs"] if v[1] > 0 else None,
            "tflops": v[2] / (v[1] * 1e-3) / 1e12 if v[1] > 0 and v[2] > 0 else None}
        for n, v in kern.items() if v[1] > 0}
    trk = {"gateup": "gateup", "down": "down", "route": "route", "combine": "combine",
           "decode_layer": "decode_layer"}.get(dom, dom)
    tr = stored_traffic(cfg["name"] + ("_" + fmt if cfg["name"].startswith("prefill") else "")
                        + ("_fp4act" if fp4_act else "") + ("_resident" if S >= L * E and cfg["mode"] == "lru"
                                                             and not cfg["name"].startswith("prefill") else ""), trk)
    roofline["traffic"] = tr
    roofline["traffic_src"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, profiles/traffic.json"
                               if tr is not None else "no ncu capture of these kernel sources")
    copy_ms = prof["miss_copy"][0]
    copy_gbs = pd["misses"] * nb / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 and pd["misses"] > 0 else None
    stream_ms = prof["stream_copy"][0]
    stream_gbs = pd["streamed"] * nb / (stream_ms * 1e-3) / 1e9 if stream_ms > 0 else None

    # ---- path roofline: the slowest of HBM weight bytes, PCIe expert bytes, FLOPs
    t_step = ms_max * 1e-3 / K
    w_hbm = d["lookups"] * nb / K
    m_pcie = (d["misses"] + d["streamed"]) * nb / K
    flops = 2 * 3 * H * I * k * tokens / K * L
    t_hbm = w_hbm / (peaks["hbm_gbs"] * 1e9)
    t_pcie = m_pcie / (pcie_gbs * 1e9)
    tensor_peak = fp4_peak(256) if fp4_act and ffn_kernel == "tc" else peaks["bf16_tflops"]
    t_flop = flops / (tensor_peak * 1e12)
    t_roof = max(t_hbm, t_pcie, t_flop)
    path = {"t_step_ms": t_step * 1e3, "t_roof_ms": t_roof * 1e3, "frac": t_roof / t_step,
            "bound": ("hbm", "pcie", "tensor")[int(np.argmax([t_hbm, t_pcie, t_flop]))],
            "hbm_bytes_per_step": w_hbm, "pcie_bytes_per_step": m_pcie, "flops_per_step": flops,
            "tensor_peak": "FP4 (measured by ft_fp4_tensor_peak)" if fp4_act and ffn_kernel == "tc"
            else "bf16 burst (measured)", "ffn_kernel": ffn_kernel,
            "pcie_h2d_gbs_measured": pcie_gbs, "miss_copy_gbs_achieved": copy_gbs,
            "stream_copy_gbs_achieved": stream_gbs,
            "hits_per_step": d["hits"] / K, "misses_per_step": d["misses"] / K,
            "streamed_per_step": d["streamed"] / K, "hit_d2d_per_step": d["hit_d2d"] / K,
            "hit_rate": d["hits"] / max(1, d["lookups"])}

    if prefill:
        l2 = f"L2 flushed (256 MiB write) before each timed step; weights {E * nb / 1e9:.2f} GB per layer"
    elif cfg["mode"] == "stream" and d2d_cache > 0:
        l2 = (f"every expert staged each step ({L * E * nb / 1e9:.1f} GB): {d['streamed'] / K:.0f} from pinned "
              f"host memory, {d['hit_d2d'] / K:.0f} from cache slots on the device")
    elif cfg["mode"] == "stream":
        l2 = f"every expert streamed from pinned host memory each step ({L * E * nb / 1e9:.1f} GB per step)"
    else:
        l2 = f"working set > L2: {S} slots x {nb} B = {S * nb / 1e9:.2f} GB slot bank"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4-w/nvfp4-act/f32-acc" if fp4_act else
        {"nvfp4": "nvfp4-w/bf16-act/f32-acc", "mxfp4": "mxfp4-w/bf16-act/f32-acc",
         "fp8": "fp8-w/bf16-act/f32-acc"}.get(fmt, "bf16/f32-acc"),
        "data": "synthetic",
        "config": {"workload": cfg["name"], "layers": L, "hidden": H, "experts": E, "top_k": k, "inter": I,
                   "weight_fmt": fmt, "act_fmt": "fp4 on tensor-core calls" if fp4_act else "bf16",
                   "slots": S, "tokens_per_step": T, "zipf_s": cfg["zipf"],
                   "mode": cfg["mode"],
                   "prefill_hit_d2d": {"cache_slots": d2d_cache} if d2d_cache > 0 else None,
                   "miss_path": stack.miss_path(ffn_kernel == "tc") if cfg["mode"] == "lru" else None,
                   "decode_kernels": "fused" if args.fused_decode else
                   ("split" if getattr(args, "no_decode_grid", False) else "grid (split where not eligible)"), "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU", "l2": l2,
                   "pool": f"{n_keys} logical experts over {n_phys} distinct pinned blobs ({n_phys * nb / 1e9:.2f} GB)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": L * T * (H * 2 + E * 4),
                "d2h_bytes_per_step": L * T * H * 2, "ms_per_step": e2e_ms / K,
                "copies": "own streams, double-buffered: overlapped with the neighbouring steps' compute",
                "l2": "no separate flush: every step reads its experts' weights, larger than L2"},
        "gpu_launches": int(launches),
        "roofline": roofline,
        "path_roofline": path,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if resize and cfg["mode"] == "lru" and S // 2 >= min(E, T * k):
        line["resize"] = _resize_probe(torch, dev, stack, S)
    stack.close()
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="decode35b", choices=sorted(CONFIGS))
    ap.add_argument("--n-phys", type=int, default=768, help="distinct pinned blobs behind the logical pool")
    ap.add_argument("--profile-steps", type=int, default=32)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fmt", choices=("bf16", "nvfp4", "mxfp4", "fp8"), default=None,
                    help="weight format (default: the workload's)")
    ap.add_argument("--ffn", choices=("auto", "gemv", "tc"), default="auto", help="FFN kernel")
    ap.add_argument("--act", choices=("bf16", "fp4"), default="bf16",
                    help="activations of tensor-core calls: bf16, or quantised to NVFP4 (FP4 x FP4 on the "
                         "block-scaled tensor cores; NVFP4 weights)")
    ap.add_argument("--hit-d2d-cache", type=int, default=0,
                    help="streaming workloads: this many cache slots beside the two staging banks, with prefill "
                         "hit-D2D on (cached experts are staged from their slots, the rest from host memory)")
    ap.add_argument("--miss-path", choices=("auto", "copy", "pull", "kernel"), default="auto",
                    help="LRU misses: cudaMemcpyAsync issued by the host, read over PCIe by the FFN kernels, "
                         "copied by the GPU, or auto (the GPU for experts up to 8 MiB, else the host)")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the further workloads (prefill-35B BF16 and NVFP4, stream-753B) that a one-GPU run "
                         "of the default workload also measures")
    ap.add_argument("--no-decode-grid", action="store_true",
                    help="decode calls as separate route, gate/up and down kernels instead of one grid")
    ap.add_argument("--fused-decode", action="store_true",
                    help="decode calls as one cooperative kernel instead of separate kernels (its copy-flag "
                         "wait needs the copy stream to progress alongside it: profile it with --miss-path pull)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = CONFIGS[args.config]
    # the further workloads come with the default workload only
    args.extras = args.extras and args.config == "decode35b" and args.fmt is None and args.ffn == "auto" \
        and args.miss_path == "auto" and not args.fused_decode and args.act == "bf16"
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
