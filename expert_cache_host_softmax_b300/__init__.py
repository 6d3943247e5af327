"""Host-resident-expert MoE layer for B300: Python binding of libftmoe.so.

Argument marshalling only.  Every step of the forward runs in the library's
CUDA kernels and CUDA copies.  PyTorch provides device memory, pinned host
memory and streams.  Importing this package fails loudly if the compiled
library is missing; there is no CPU fallback.

The C ABI is declared in include/ft_moe.h; the names here mirror it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libftmoe.so")

FT_FMT_BF16, FT_FMT_NVFP4, FT_FMT_MXFP4, FT_FMT_FP8 = 0, 1, 2, 3
FMT = {"bf16": FT_FMT_BF16, "nvfp4": FT_FMT_NVFP4, "mxfp4": FT_FMT_MXFP4, "fp8": FT_FMT_FP8}
FT_MODE_LRU, FT_MODE_STREAM = 0, 1
FT_FFN_AUTO, FT_FFN_GEMV, FT_FFN_TC = 0, 1, 2
FFN_KERNEL = {"auto": FT_FFN_AUTO, "gemv": FT_FFN_GEMV, "tc": FT_FFN_TC}
FT_ACT_BF16, FT_ACT_FP4 = 0, 1
ACT_FORMAT = {"bf16": FT_ACT_BF16, "fp4": FT_ACT_FP4}
FT_MISS_COPY, FT_MISS_PULL, FT_MISS_KERNEL, FT_MISS_AUTO = 0, 1, 2, 3
MISS_PATH = {"copy": FT_MISS_COPY, "pull": FT_MISS_PULL, "kernel": FT_MISS_KERNEL, "auto": FT_MISS_AUTO}
FT_OK, FT_ERR_ARG, FT_ERR_CUDA, FT_ERR_OOM, FT_ERR_NOT_PINNED = 0, -1, -2, -3, -4
FT_ERR_CACHE_TOO_SMALL, FT_ERR_STATE, FT_ERR_TIMEOUT, FT_ERR_DEVICE = -5, -6, -7, -8
STATUS_NAMES = {0: "FT_OK", -1: "FT_ERR_ARG", -2: "FT_ERR_CUDA", -3: "FT_ERR_OOM", -4: "FT_ERR_NOT_PINNED",
                -5: "FT_ERR_CACHE_TOO_SMALL", -6: "FT_ERR_STATE", -7: "FT_ERR_TIMEOUT", -8: "FT_ERR_DEVICE"}

#: every symbol include/ft_moe.h declares
EXPORTED = ("ft_moe_blob_bytes", "ft_moe_create", "ft_moe_load_pool", "ft_moe_set_mode", "ft_moe_forward",
            "ft_cache_stats", "ft_cache_reset", "ft_cache_trace", "ft_moe_last_routing", "ft_moe_last_activations",
            "ft_moe_set_profiling", "ft_moe_profile_read", "ft_moe_set_ffn_kernel", "ft_moe_last_ffn_kernel", "ft_moe_set_miss_path", "ft_moe_miss_path", "ft_moe_set_decode_fusion", "ft_moe_set_decode_grid", "ft_moe_set_keep_activations", "ft_moe_resize_slots",
            "ft_moe_set_prefill_hit_d2d", "ft_moe_prefill_hit_d2d",
            "ft_moe_slot_stride", "ft_moe_kernel_launches",
            "ft_moe_set_act_format", "ft_moe_act_format", "ft_moe_last_act_fp4", "ft_fp4_tensor_peak",
            "ft_last_error", "ft_moe_destroy", "ft_topk_softmax", "ft_permute_workspace_bytes", "ft_permute", "ft_permute_noalloc")


class FtStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("lookups", "hits", "misses", "evictions", "warm_loads", "streamed", "bytes_h2d", "hit_d2d")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class FtError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def lib():
    """The loaded libftmoe.so (raises ImportError if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m expert_cache_host_softmax_b300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        P = ctypes.POINTER
        L.ft_moe_blob_bytes.restype = i64
        L.ft_moe_blob_bytes.argtypes = [i32, i32, i32]
        L.ft_moe_create.argtypes = [i32] * 8 + [P(vp)]
        L.ft_moe_load_pool.argtypes = [vp, vp]
        L.ft_moe_set_mode.argtypes = [vp, i32]
        L.ft_moe_forward.argtypes = [vp, i32, i32, vp, vp, vp, vp]
        L.ft_cache_stats.argtypes = [vp, P(FtStats), P(FtStats)]
        L.ft_cache_reset.argtypes = [vp, i32]
        L.ft_cache_trace.argtypes = [vp, vp, vp, vp, vp, i32, P(i32)]
        L.ft_moe_last_routing.argtypes = [vp, vp, vp, vp, vp, vp, P(i32)]
        L.ft_moe_last_activations.argtypes = [vp, vp, vp]
        L.ft_moe_set_profiling.argtypes = [vp, i32]
        L.ft_moe_profile_read.argtypes = [vp, vp, vp, i32]
        L.ft_moe_set_ffn_kernel.argtypes = [vp, i32]
        L.ft_moe_last_ffn_kernel.argtypes = [vp]
        L.ft_moe_miss_path.argtypes = [vp, i32]
        L.ft_moe_set_keep_activations.argtypes = [vp, i32]
        L.ft_moe_resize_slots.argtypes = [vp, i32]
        L.ft_moe_set_prefill_hit_d2d.argtypes = [vp, i32]
        L.ft_moe_prefill_hit_d2d.argtypes = [vp]
        L.ft_moe_set_miss_path.argtypes = [vp, i32]
        L.ft_moe_set_decode_fusion.argtypes = [vp, i32]
        L.ft_moe_set_decode_grid.argtypes = [vp, i32]
        L.ft_moe_set_act_format.argtypes = [vp, i32]
        L.ft_moe_act_format.argtypes = [vp]
        L.ft_moe_last_act_fp4.argtypes = [vp, vp, vp, vp, vp, vp]
        L.ft_fp4_tensor_peak.argtypes = [i32, i32, P(ctypes.c_double)]
        L.ft_moe_kernel_launches.restype = i64
        L.ft_moe_kernel_launches.argtypes = [vp]
        L.ft_moe_slot_stride.restype = i64
        L.ft_moe_slot_stride.argtypes = [vp]
        L.ft_last_error.restype = ctypes.c_char_p
        L.ft_last_error.argtypes = [vp]
        L.ft_moe_destroy.argtypes = [vp]
        L.ft_topk_softmax.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.ft_permute_workspace_bytes.restype = sz
        L.ft_permute_workspace_bytes.argtypes = [i32, i32, i32]
        L.ft_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.ft_permute_noalloc.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        _lib = L
    return _lib


def _check(code, handle=None):
    if code != FT_OK:
        raise FtError(code, lib().ft_last_error(handle).decode())


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def blob_bytes(fmt, hidden: int, inter: int) -> int:
    return int(lib().ft_moe_blob_bytes(FMT.get(fmt, fmt) if isinstance(fmt, str) else fmt, hidden, inter))


class MoELayerStack:
    """A stack of MoE layers sharing one GPU slot cache (ft_moe handle)."""

    def __init__(self, hidden, n_experts, top_k, inter, fmt, n_slots, n_layers, max_tokens):
        self.H, self.E, self.k, self.I = hidden, n_experts, top_k, inter
        self.fmt = FMT[fmt] if isinstance(fmt, str) else int(fmt)
        self.S, self.L, self.Tmax = n_slots, n_layers, max_tokens
        h = ctypes.c_void_p()
        _check(lib().ft_moe_create(hidden, n_experts, top_k, inter, self.fmt, n_slots, n_layers, max_tokens,
                                   ctypes.byref(h)))
        self._h = h
        self._pool_ref = None
        self.blob_bytes = blob_bytes(self.fmt, hidden, inter)

    def close(self):
        if self._h:
            lib().ft_moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_pool(self, pointers, keepalive=None):
        """pointers: n_layers*n_experts addresses of pinned host blobs."""
        arr = np.ascontiguousarray(np.asarray(pointers, dtype=np.uint64))
        if arr.size != self.L * self.E:
            raise ValueError(f"expected {self.L * self.E} pool pointers (n_layers * n_experts), got {arr.size}")
        self._pool_ref = (arr, keepalive)
        _check(lib().ft_moe_load_pool(self._h, ctypes.c_void_p(arr.ctypes.data)), self._h)

    def set_mode(self, mode):
        _check(lib().ft_moe_set_mode(self._h, mode), self._h)

    def reset(self, warm=True):
        _check(lib().ft_cache_reset(self._h, 1 if warm else 0), self._h)

    def forward(self, layer, x, logits, out=None, stream=None):
        """x: cuda bf16 [T,H]; logits: cuda f32 [T,E] -> out cuda bf16 [T,H]."""
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        for name, t, dtype, cols in (("x", x, torch.bfloat16, self.H), ("logits", logits, torch.float32, self.E),
                                     ("out", out, torch.bfloat16, self.H)):
            if not t.is_cuda or t.dtype != dtype or tuple(t.shape) != (T, cols) or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous cuda {dtype} tensor of shape ({T}, {cols})")
        _check(lib().ft_moe_forward(self._h, layer, T, _ptr(x), _ptr(logits), _ptr(out), _stream_ptr(stream)),
               self._h)
        return out

    def forward_raw(self, layer, T, x_ptr, logits_ptr, out_ptr, stream_ptr):
        return lib().ft_moe_forward(self._h, layer, T, ctypes.c_void_p(x_ptr), ctypes.c_void_p(logits_ptr),
                                    ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream_ptr))

    def stats(self):
        c, l = FtStats(), FtStats()
        _check(lib().ft_cache_stats(self._h, ctypes.byref(c), ctypes.byref(l)), self._h)
        return c.as_dict(), l.as_dict()

    def trace(self):
        cap = self.E
        ex, sl, hi, ev = (np.zeros(cap, np.int32) for _ in range(4))
        n = ctypes.c_int()
        _check(lib().ft_cache_trace(self._h, ex.ctypes.data, sl.ctypes.data, hi.ctypes.data, ev.ctypes.data, cap,
                                    ctypes.byref(n)), self._h)
        m = n.value
        return [(int(ex[i]), int(sl[i]), bool(hi[i]), int(ev[i])) for i in range(m)]

    def last_routing(self):
        Tk = self.Tmax * self.k
        idx, perm, inv = (np.zeros(Tk, np.int32) for _ in range(3))
        gates = np.zeros(Tk, np.float32)
        offsets = np.zeros(self.E + 1, np.int32)
        n = ctypes.c_int()
        _check(lib().ft_moe_last_routing(self._h, idx.ctypes.data, gates.ctypes.data, offsets.ctypes.data,
                                         perm.ctypes.data, inv.ctypes.data, ctypes.byref(n)), self._h)
        T = n.value
        return dict(idx=idx[:T * self.k].reshape(T, self.k), gates=gates[:T * self.k].reshape(T, self.k),
                    offsets=offsets, perm=perm[:T * self.k], inv=inv[:T * self.k])

    def last_activations(self, T):
        """(h bf16 bits [T*k, I], y f32 [T*k, H]) of the last forward, permuted order."""
        hb = np.zeros((T * self.k, self.I), np.uint16)
        y = np.zeros((T * self.k, self.H), np.float32)
        _check(lib().ft_moe_last_activations(self._h, hb.ctypes.data, y.ctypes.data), self._h)
        return hb, y

    PROF_CLASSES = ("route", "gateup_hit", "gateup_miss", "down", "combine", "miss_copy", "stream_copy", "layer")

    def set_profiling(self, on=True):
        _check(lib().ft_moe_set_profiling(self._h, 1 if on else 0), self._h)

    def profile(self):
        """{class: (total ms, occurrences)} since profiling was enabled."""
        n = len(self.PROF_CLASSES)
        ms = np.zeros(n, np.float64)
        cnt = np.zeros(n, np.int64)
        _check(lib().ft_moe_profile_read(self._h, ms.ctypes.data, cnt.ctypes.data, n), self._h)
        return {c: (float(ms[i]), int(cnt[i])) for i, c in enumerate(self.PROF_CLASSES)}

    def set_ffn_kernel(self, which):
        """"auto", "gemv" or "tc" (ft_moe_set_ffn_kernel)."""
        w = FFN_KERNEL[which] if isinstance(which, str) else int(which)
        _check(lib().ft_moe_set_ffn_kernel(self._h, w), self._h)

    def set_decode_fusion(self, on=True):
        """One cooperative kernel per decode call, or separate kernels (default)."""
        _check(lib().ft_moe_set_decode_fusion(self._h, 1 if on else 0), self._h)

    def set_decode_grid(self, on=True):
        """Eligible decode calls as one grid, or separate route, gate/up and down kernels (default)."""
        _check(lib().ft_moe_set_decode_grid(self._h, 1 if on else 0), self._h)

    def resize_slots(self, n_slots):
        """Changes the number of expert slots (the most recently used experts stay)."""
        _check(lib().ft_moe_resize_slots(self._h, int(n_slots)), self._h)

    def set_prefill_hit_d2d(self, on=True):
        """STREAM-mode staging copies the experts the cache holds from their slots, and mode
        switches keep the cache (off by default)."""
        _check(lib().ft_moe_set_prefill_hit_d2d(self._h, 1 if on else 0), self._h)

    def prefill_hit_d2d(self):
        r = lib().ft_moe_prefill_hit_d2d(self._h)
        if r < 0:
            _check(r, self._h)
        return r == 1

    def set_keep_activations(self, on):
        """Tensor-core calls also store y for last_activations (off by default)."""
        _check(lib().ft_moe_set_keep_activations(self._h, 1 if on else 0), self._h)

    def set_miss_path(self, path):
        """"copy" (cudaMemcpyAsync issued by the host), "pull" (the FFN kernels read misses over
        PCIe), "kernel" (the GPU copies them; no host round trip) or "auto" (default: "kernel"
        for experts up to 8 MiB, else "copy")."""
        w = MISS_PATH[path] if isinstance(path, str) else int(path)
        _check(lib().ft_moe_set_miss_path(self._h, w), self._h)

    def miss_path(self, tensor_core=False):
        """The miss path LRU calls on the GEMV (or the tensor-core FFN) take, "auto" resolved:
        "copy", "pull" or "kernel"."""
        inv = {v: k_ for k_, v in MISS_PATH.items()}
        return inv.get(int(lib().ft_moe_miss_path(self._h, 1 if tensor_core else 0)))

    def set_act_format(self, fmt):
        """"bf16" (default) or "fp4": tensor-core calls quantise x and h to NVFP4 and
        multiply FP4 x FP4 (ft_moe_set_act_format; NVFP4 weights only)."""
        w = ACT_FORMAT[fmt] if isinstance(fmt, str) else int(fmt)
        _check(lib().ft_moe_set_act_format(self._h, w), self._h)

    @property
    def act_format(self):
        return {FT_ACT_BF16: "bf16", FT_ACT_FP4: "fp4"}.get(int(lib().ft_moe_act_format(self._h)))

    def last_act_fp4(self, T):
        """The last call's quantised activations, permuted order: dict of x_codes u8
        [T*k, H/2], x_sf u8 [T*k, H/16], x_g f32 [T*k], h_codes u8 [T*k, I/2], h_sf u8 [T*k, I/16]."""
        n = T * self.k
        out = dict(x_codes=np.zeros((n, self.H // 2), np.uint8), x_sf=np.zeros((n, self.H // 16), np.uint8),
                   x_g=np.zeros(n, np.float32), h_codes=np.zeros((n, self.I // 2), np.uint8),
                   h_sf=np.zeros((n, self.I // 16), np.uint8))
        _check(lib().ft_moe_last_act_fp4(self._h, *(ctypes.c_void_p(out[k_].ctypes.data) for k_ in
                                                  ("x_codes", "x_sf", "x_g", "h_codes", "h_sf"))), self._h)
        return out

    @property
    def last_ffn_kernel(self):
        return {FT_FFN_GEMV: "gemv", FT_FFN_TC: "tc"}.get(int(lib().ft_moe_last_ffn_kernel(self._h)))

    @property
    def kernel_launches(self):
        return int(lib().ft_moe_kernel_launches(self._h))

    @property
    def slot_stride(self):
        return int(lib().ft_moe_slot_stride(self._h))


def fp4_tensor_peak(n_tile=256, iters=20000):
    """Block-scaled FP4 tensor-core rate of the current device (TFLOP/s), measured
    by the library's one-kernel probe (ft_fp4_tensor_peak)."""
    v = ctypes.c_double()
    _check(lib().ft_fp4_tensor_peak(int(n_tile), int(iters), ctypes.byref(v)))
    return v.value


def topk_softmax(logits, k, stream=None):
    """Stateless router step: cuda f32 [T,E] -> (idx int32 [T,k], gates f32 [T,k])."""
    import torch
    T, E = logits.shape
    idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    gates = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().ft_topk_softmax(_ptr(logits), T, E, k, _ptr(idx), _ptr(gates), _stream_ptr(stream)))
    return idx, gates


def permute(topk_idx, n_experts, stream=None):
    """Stateless permute step: cuda int32 [T,k] -> (offsets [E+1], perm [T*k], inv [T*k])."""
    import torch
    T, k = topk_idx.shape
    dev = topk_idx.device
    offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    ws_bytes = int(lib().ft_permute_workspace_bytes(T, k, n_experts))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    _check(lib().ft_permute(_ptr(topk_idx), T, k, n_experts, _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(ws),
                            ws_bytes, _stream_ptr(stream)))
    return offsets, perm, inv


#: scratch bytes of ft_permute_noalloc's fixed device array
PERMUTE_NOALLOC_MAX_SCRATCH_BYTES = 2 << 20


def permute_noalloc(topk_idx, n_experts, stream=None):
    """ft_permute_noalloc: like permute() but the library allocates nothing
    and takes no workspace (its scratch is a fixed device array)."""
    import torch
    T, k = topk_idx.shape
    dev = topk_idx.device
    offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    _check(lib().ft_permute_noalloc(_ptr(topk_idx), T, k, n_experts, _ptr(offsets), _ptr(perm), _ptr(inv),
                                    _stream_ptr(stream)))
    return offsets, perm, inv
