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
device->host read of the outputs.  Under torchrun (N > 1) every rank runs an
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
    layer).  Blobs are generated before any call is timed."""

    def __init__(self, cfg, seed, n_phys, max_calls):
        import oracle as O
        self.cfg, self.seed = cfg, seed
        H, E, k, I, L = cfg["H"], cfg["E"], cfg["k"], cfg["I"], cfg["L"]
        self.calls = []
        step = 0
        while len(self.calls) < max_calls:
            for l in range(L):
                if len(self.calls) < max_calls:
                    self.calls.append((step, l, tokens_at(cfg, step)))
            step += 1
        need = set()
        for step, l, T in self.calls:
            lg = ftgen.router_logits(seed, T, E, step, l, cfg["zipf"], epoch_at(cfg, step))
            need |= {(l * E + int(e)) % n_phys for e in O.topk_experts(lg, k).reshape(-1)}
        need = sorted(need)
        blobs = ftgen.pool(cfg["fmt"], H, I, need, seed)
        self.blobs = {p: blobs[i] for i, p in enumerate(need)}
        self.orc = O.MoELayerOracle(H, E, k, I, ftgen.FMT_NAMES[cfg["fmt"]], cfg["S"], L,
                                    lambda key: self.blobs[key % n_phys],
                                    mode=O.MODE_STREAM if cfg["mode"] == "stream" else O.MODE_LRU)
        self.pos = 0

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
        sample = None if T <= 64 else list(range(0, T, max(1, T // 256)))
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


def _cpu_baseline(cfg, seed, n_phys, budget_s=15.0, max_calls=192):
    """Times the CPU oracle, as it stands, single-threaded, on the workload's
    first layer calls until `budget_s` seconds of oracle time.
    Returns (tokens/s through the L-layer stack, description, calls, seconds)."""
    run = _OracleRunner(cfg, seed, n_phys, max_calls)
    calls, rows, used = 0, 0, 0.0
    with _single_thread():
        while used < budget_s and run.pos < len(run.calls):
            dt, r, _ = run.next_call()
            used += dt
            rows += r
            calls += 1
    L = cfg["L"]
    desc = (f"oracle on the first {calls} layer calls of {cfg['name']} in order ({rows} token rows, "
            f"FFN included), float64 numpy, 1 thread; tokens/s = rows / {L} layers / seconds")
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


def run_ours(args, cfg):
    import torch
    import expert_cache_host_softmax_b300 as F
    from __graft_entry__ import build
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build()
    peaks = _peaks()
    seed = cfg["seed"] + rank
    T, H, E, k, I, L, S = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["I"], cfg["L"], cfg["S"]
    nb = ftgen.blob_bytes(cfg["fmt"], H, I)
    n_keys = L * E
    n_phys = min(args.n_phys, n_keys)

    # pinned host pool: n_phys distinct blobs, logical key -> key % n_phys
    pool = torch.empty(n_phys * nb, dtype=torch.uint8, pin_memory=True)
    ftgen.pool(cfg["fmt"], H, I, list(range(n_phys)), seed, out=pool.numpy().reshape(n_phys, nb))
    ptrs = [pool.data_ptr() + (key % n_phys) * nb for key in range(n_keys)]
    stack = F.MoELayerStack(H, E, k, I, cfg["fmt"], S, L, T)
    stack.load_pool(ptrs, keepalive=pool)
    if cfg["mode"] == "stream":
        stack.set_mode(F.FT_MODE_STREAM)

    W, K = args.warmup, args.steps
    n_prof = min(args.profile_steps, K)
    n_steps = W + K
    X, G = _gen_inputs(cfg, seed, n_steps)
    Xd = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).to(dev)
    Gd = torch.from_numpy(G).to(dev)
    outd = torch.empty((L, T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    Lb = F.lib()
    h = stack._h
    x_ptr0, g_ptr0, o_ptr0 = Xd.data_ptr(), Gd.data_ptr(), outd.data_ptr()
    xs, gs, os_ = T * H * 2, T * E * 4, T * H * 2

    def step(s, xb=None, gb=None):
        t = tokens_at(cfg, s)
        for l in range(L):
            xo = (xb + l * xs) if xb is not None else x_ptr0 + (s * L + l) * xs
            go = (gb + l * gs) if gb is not None else g_ptr0 + (s * L + l) * gs
            rc = Lb.ft_moe_forward(h, l, t, xo, go, o_ptr0 + l * os_, sp)
            if rc != 0:
                raise F.FtError(rc, Lb.ft_last_error(h).decode())

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        for s in range(W):
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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    e0.record(stream)
    for s in range(W, W + K):
        step(s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    cum1, _ = stack.stats()
    launches = stack.kernel_launches - launches0
    d = {key_: cum1[key_] - cum0[key_] for key_ in cum1}
    ms_max = ms
    if ws > 1:
        import torch.distributed as dist
        tt = torch.tensor([ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_max = float(tt.item())
    tokens = sum(tokens_at(cfg, s) for s in range(W, W + K))
    value = tokens * ws / (ms_max * 1e-3)

    # ---- end to end: per step, H2D of the step's inputs from pinned host and
    # D2H of its outputs, inside the timed region
    Xh = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).pin_memory()
    Gh = torch.from_numpy(G).pin_memory()
    outh = torch.empty((L, T, H), dtype=torch.bfloat16).pin_memory()
    xin = torch.empty((L, T, H), dtype=torch.bfloat16, device=dev)
    gin = torch.empty((L, T, E), dtype=torch.float32, device=dev)
    barrier()
    torch.cuda.synchronize(dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for s in range(W, W + K):
            xin.copy_(Xh[s], non_blocking=True)
            gin.copy_(Gh[s], non_blocking=True)
            step(s, xin.data_ptr(), gin.data_ptr())
            outh.copy_(outd, non_blocking=True)
        f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = f0.elapsed_time(f1)
    if ws > 1:
        import torch.distributed as dist
        tt = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        e2e_ms = float(tt.item())
    e2e_value = tokens * ws / (e2e_ms * 1e-3)

    # ---- per-kernel timing pass (events around each step class)
    stack.set_profiling(True)
    c0, _ = stack.stats()
    with torch.cuda.stream(stream):
        for s in range(W, W + n_prof):
            step(s)
    torch.cuda.synchronize(dev)
    prof = stack.profile()
    c1, _ = stack.stats()
    stack.set_profiling(False)
    pd = {key_: c1[key_] - c0[key_] for key_ in c1}

    # algorithmic bytes of the FFN kernels (weights of each distinct expert once
    # per call, plus activations)
    HI = H * I
    if cfg["fmt"] == "nvfp4":
        gu_bytes, d_bytes = 2 * HI // 2 + 2 * HI // 16, HI // 2 + HI // 16
    elif cfg["fmt"] == "mxfp4":
        gu_bytes, d_bytes = 2 * HI // 2 + 2 * HI // 32, HI // 2 + HI // 32
    else:
        gu_bytes, d_bytes = 4 * HI, 2 * HI
    calls_p = n_prof * L
    toks_p = sum(tokens_at(cfg, s) for s in range(W, W + n_prof))
    act_gu = toks_p * k * (H * 2 + I * 2)          # x rows read per (token, expert) + h written
    act_dn = toks_p * k * (I * 2 + H * 4)          # h read + y written
    kern = {
        "gateup": (pd["lookups"] * gu_bytes + act_gu, prof["gateup_hit"][0] + prof["gateup_miss"][0],
                   prof["gateup_hit"][1] + prof["gateup_miss"][1]),
        "down": (pd["lookups"] * d_bytes + act_dn, prof["down"][0], prof["down"][1]),
        "route": (toks_p * E * 4, prof["route"][0], prof["route"][1]),
        "combine": (toks_p * (k * H * 4 + H * 2), prof["combine"][0], prof["combine"][1]),
    }
    dom = max(kern, key=lambda n: kern[n][1])
    b_dom, ms_dom, n_dom = kern[dom]
    achieved = b_dom / (ms_dom * 1e-3) / 1e9 if ms_dom > 0 else 0.0
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None, "peak_src": peaks["src"],
                "bytes_per_call": b_dom / calls_p, "ms_per_call": ms_dom / calls_p,
                "kernel_ms_share": {n: round(kern[n][1] / max(1e-9, sum(v[1] for v in kern.values())), 4)
                                    for n in kern}}
    copy_ms = prof["miss_copy"][0]
    copy_gbs = pd["misses"] * nb / (copy_ms * 1e-3) / 1e9 if copy_ms > 0 else None

    # ---- path roofline: the slowest of HBM weight bytes, PCIe miss bytes, FLOPs
    t_step = ms_max * 1e-3 / K
    w_hbm = d["lookups"] * nb / K
    m_pcie = d["misses"] * nb / K
    flops = 2 * 3 * HI * k * tokens / K * L
    t_hbm = w_hbm / (peaks["hbm_gbs"] * 1e9)
    t_pcie = m_pcie / (pcie_gbs * 1e9)
    t_flop = flops / (peaks["bf16_tflops_sustained"] * 1e12)
    t_roof = max(t_hbm, t_pcie, t_flop)
    path = {"t_step_ms": t_step * 1e3, "t_roof_ms": t_roof * 1e3, "frac": t_roof / t_step,
            "bound": ("hbm", "pcie", "tensor")[int(np.argmax([t_hbm, t_pcie, t_flop]))],
            "hbm_bytes_per_step": w_hbm, "pcie_bytes_per_step": m_pcie, "flops_per_step": flops,
            "pcie_h2d_gbs_measured": pcie_gbs, "miss_copy_gbs_achieved": copy_gbs,
            "hits_per_step": d["hits"] / K, "misses_per_step": d["misses"] / K,
            "hit_rate": d["hits"] / max(1, d["lookups"])}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4-w/bf16-act/f32-acc" if cfg["fmt"] == "nvfp4" else cfg["fmt"], "data": "synthetic",
        "config": {"workload": cfg["name"], "layers": L, "hidden": H, "experts": E, "top_k": k, "inter": I,
                   "weight_fmt": cfg["fmt"], "slots": S, "tokens_per_step": T, "zipf_s": cfg["zipf"],
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": f"working set > L2: {S} slots x {nb} B = {S * nb / 1e9:.2f} GB slot bank",
                   "pool": f"{n_keys} logical experts over {n_phys} distinct pinned blobs ({n_phys * nb / 1e9:.2f} GB)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": L * T * (H * 2 + E * 4),
                "d2h_bytes_per_step": L * T * H * 2},
        "gpu_launches": int(launches),
        "roofline": roofline,
        "path_roofline": path,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        tps, desc, calls, secs = _cpu_baseline(cfg, cfg["seed"], n_phys, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                                "seconds": secs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    stack.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


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
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
