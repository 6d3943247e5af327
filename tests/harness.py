"""Shared test set-up: one seeded workload fed to both the GPU library and the
CPU oracle.  Test infrastructure only."""
from __future__ import annotations

import numpy as np

import ftgen
import oracle as O


class Pool:
    """A pinned host pool of n_phys distinct blobs; logical key -> blob key % n_phys."""

    def __init__(self, fmt, H, I, n_keys, seed, n_phys=None, flags=0):
        import torch
        self.fmt, self.H, self.I = fmt, H, I
        self.n_keys = n_keys
        self.n_phys = n_keys if n_phys is None else min(n_phys, n_keys)
        self.nbytes = ftgen.blob_bytes(fmt, H, I)
        self.buf = torch.empty(self.n_phys * self.nbytes, dtype=torch.uint8, pin_memory=True)
        arr = self.buf.numpy().reshape(self.n_phys, self.nbytes)
        ftgen.pool(fmt, H, I, list(range(self.n_phys)), seed, flags=flags, out=arr)
        self.arr = arr
        base = self.buf.data_ptr()
        self.pointers = [base + (key % self.n_phys) * self.nbytes for key in range(n_keys)]

    def blob(self, key):
        return self.arr[key % self.n_phys]


def make_pair(H, E, k, I, fmt, S, L, Tmax, seed, n_phys=None, mode="lru", warm=True, flags=0, keep=True,
              hit_d2d=False):
    """(GPU stack, oracle, pool) over the same pinned pool.  keep: tensor-core
    calls also store y, so that the tests can check the GEMM accumulation.
    hit_d2d: prefill hit-D2D on both sides (before the switch to `mode`)."""
    import expert_cache_host_softmax_b300 as F
    pool = Pool(fmt, H, I, L * E, seed, n_phys, flags)
    gpu = F.MoELayerStack(H, E, k, I, fmt, S, L, Tmax)
    gpu.load_pool(pool.pointers, keepalive=pool)
    if keep:
        gpu.set_keep_activations(True)
    f = ftgen.FMT_NAMES[fmt]
    orc = O.MoELayerOracle(H, E, k, I, f, S, L, pool.blob, hit_d2d=hit_d2d)
    if hit_d2d:
        gpu.set_prefill_hit_d2d(True)
    if mode == "stream":
        gpu.set_mode(F.FT_MODE_STREAM)
        orc.set_mode(O.MODE_STREAM)
    if not warm:
        gpu.reset(warm=False)
        orc.reset(warm=False)
    return gpu, orc, pool


def inputs(seed, T, H, E, step, layer, zipf=None, epoch=0):
    x = ftgen.x_bf16(seed, T, H, step, layer)
    lg = ftgen.router_logits(seed, T, E, step, layer, zipf, epoch)
    return x, lg


def to_dev(x_bits, logits):
    import torch
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    lg = torch.from_numpy(logits).cuda()
    return x, lg


def out_to_f64(out):
    import torch
    return out.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


def rel_err(got, ref):
    """max |got - ref| / max |ref| over the tensor (norm-wise)."""
    den = float(np.abs(ref).max())
    return float(np.abs(got - ref).max()) / (den if den > 0 else 1.0)


def elem_rel_err(got, ref, floor=1e-3):
    """max over elements of |got - ref| / max(|ref|, floor * max|ref|): the
    element-wise relative error, with an absolute floor at `floor` of the
    tensor's largest magnitude."""
    ref = np.asarray(ref, np.float64)
    den = np.maximum(np.abs(ref), floor * float(np.abs(ref).max()) if ref.size else 0.0)
    den[den == 0] = 1.0
    return float((np.abs(np.asarray(got, np.float64) - ref) / den).max()) if ref.size else 0.0


def bf16_ulp(v):
    """Spacing of bf16 values at |v| (8 significant bits): 2^(floor(log2|v|) - 7)."""
    _, e = np.frexp(np.abs(np.asarray(v, np.float64)))
    return np.ldexp(1.0, e - 8)
