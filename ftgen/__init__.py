"""Seeded synthetic inputs shared by the CPU oracle and the GPU library.

This package holds no arithmetic of the MoE layer itself: it draws random
numbers (counter-addressed SplitMix64 + Box-Muller, in ``ftgen.c``) and packs
fp32 master weights into the expert blob formats.  Everything here is input
generation; the consumers decode and compute on their own.

Workload recipes follow the expert-offload description of FreeToken
("FreeToken: Run Frontier MoE Models on Your Own GPU", section "Why a Huge MoE
Model Fits on One Consumer GPU": experts in host RAM, an LRU cache of GPU
expert slots; "The Real Requirement Is System RAM": NVFP4 = 4-bit values plus
an 8-bit scale per 16 weights).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libftgen.so")
_lib = None

FMT_BF16, FMT_NVFP4, FMT_MXFP4, FMT_FP8 = 0, 1, 2, 3
FMT_NAMES = {"bf16": FMT_BF16, "nvfp4": FMT_NVFP4, "mxfp4": FMT_MXFP4, "fp8": FMT_FP8}
FLAG_NVFP4_UNIT_GSCALE = 1

# stream kinds (high byte of the 64-bit stream id)
_K_X, _K_LOGITS, _K_ZIPF_PERM = 1, 2, 3


def build(force: bool = False) -> str:
    """Compiles ftgen.c into libftgen.so next to it (gcc, -O2, pthreads)."""
    src = os.path.join(_HERE, "ftgen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i64, u64, f32, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_int
        vp = ctypes.c_void_p
        L.ftgen_u64.restype = u64
        L.ftgen_u64.argtypes = [u64, u64, u64]
        L.ftgen_normal_f32.argtypes = [u64, u64, u64, i64, vp]
        L.ftgen_uniform_f32.argtypes = [u64, u64, u64, i64, vp]
        L.ftgen_permutation.argtypes = [u64, u64, ctypes.c_int32, vp]
        L.ftgen_blob_bytes.restype = i64
        L.ftgen_blob_bytes.argtypes = [i32, i64, i64]
        L.ftgen_pool.restype = i32
        L.ftgen_pool.argtypes = [i32, i64, i64, f32, u64, i32, vp, i64, vp, i64, i32]
        L.ftgen_master_weights.argtypes = [i64, i64, f32, u64, u64, vp, vp, vp]
        L.ftgen_to_bf16.argtypes = [vp, i64, vp]
        _lib = L
    return _lib


def _fmt(fmt) -> int:
    return FMT_NAMES[fmt] if isinstance(fmt, str) else int(fmt)


def blob_bytes(fmt, H: int, I: int) -> int:
    """Packed bytes of one expert (gate, up, down) in format fmt."""
    return int(lib().ftgen_blob_bytes(_fmt(fmt), H, I))


def pool(fmt, H: int, I: int, keys, seed: int, wstd: float = 0.02, flags: int = 0,
         nthreads: int | None = None, out: np.ndarray | None = None, stride: int | None = None) -> np.ndarray:
    """Blobs for `keys` as a uint8 array [len(keys), stride] (or written into `out`)."""
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.uint64).reshape(-1))
    nb = blob_bytes(fmt, H, I)
    stride = nb if stride is None else int(stride)
    if out is None:
        out = np.zeros((len(keys), stride), dtype=np.uint8)
    assert out.dtype == np.uint8 and out.flags.c_contiguous and out.size >= len(keys) * stride
    nthreads = nthreads or min(len(keys), os.cpu_count() or 1, 64) or 1
    rc = lib().ftgen_pool(_fmt(fmt), H, I, wstd, seed, flags, keys.ctypes.data, len(keys),
                          out.ctypes.data, stride, nthreads)
    if rc != 0:
        raise RuntimeError("ftgen_pool failed")
    return out


def expert_blob(fmt, H: int, I: int, key: int, seed: int, wstd: float = 0.02, flags: int = 0) -> np.ndarray:
    return pool(fmt, H, I, [key], seed, wstd, flags, nthreads=1)[0]


def master_weights(H: int, I: int, key: int, seed: int, wstd: float = 0.02):
    """fp32 master weights (gate [I,H], up [I,H], down [H,I]) that blob `key` encodes."""
    g = np.empty((I, H), np.float32)
    u = np.empty((I, H), np.float32)
    d = np.empty((H, I), np.float32)
    lib().ftgen_master_weights(H, I, wstd, seed, key, g.ctypes.data, u.ctypes.data, d.ctypes.data)
    return g, u, d


def normal(seed: int, stream: int, n: int, ctr0: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().ftgen_normal_f32(seed, stream, ctr0, n, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, n: int, ctr0: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().ftgen_uniform_f32(seed, stream, ctr0, n, out.ctypes.data)
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().ftgen_permutation(seed, stream, n, out.ctypes.data)
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().ftgen_to_bf16(a.ctypes.data, a.size, out.ctypes.data)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _sid(kind: int, layer: int, step: int) -> int:
    return (kind << 56) | ((layer & 0xFFFFFF) << 32) | (step & 0xFFFFFFFF)


def x_bf16(seed: int, T: int, H: int, step: int, layer: int) -> np.ndarray:
    """Activations x ~ N(0,1) rounded to bf16, as uint16 bits [T, H]."""
    return to_bf16_bits(normal(seed, _sid(_K_X, layer, step), T * H)).reshape(T, H)


def zipf_bias(seed: int, E: int, s: float, layer: int, epoch: int = 0) -> np.ndarray:
    """Per-expert routing bias ln p_r(e), p_r proportional to r^-s over ranks 1..E.

    The rank of each expert is a seeded permutation per (layer, epoch); a new
    epoch re-draws it (slowly drifting popularity)."""
    perm = permutation(seed, _sid(_K_ZIPF_PERM, layer, epoch), E)
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-float(s))
    p /= p.sum()
    return np.log(p[perm]).astype(np.float32)


def router_logits(seed: int, T: int, E: int, step: int, layer: int,
                  zipf_s: float | None = None, epoch: int = 0) -> np.ndarray:
    """Router logits [T, E] fp32: N(0,1), plus a Zipf(s) bias per expert if zipf_s is set."""
    z = normal(seed, _sid(_K_LOGITS, layer, step), T * E).reshape(T, E)
    if zipf_s is not None:
        z = (z + zipf_bias(seed, E, zipf_s, layer, epoch)[None, :]).astype(np.float32)
    return np.ascontiguousarray(z, dtype=np.float32)
