"""CPU oracle for one Mixture-of-Experts layer forward with host-resident experts.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The GPU library never calls it; the two share no code.  Both take
their inputs from the seeded generator package ``ftgen``.

Plain, slow, single-threaded, float64.  Every step is written the way the
sources state it, with no blocking, fusion or reordering.

What the sources fix:
  * "FreeToken: Run Frontier MoE Models on Your Own GPU, and the RAM It Takes"
    (devpik.com), section "Why a Huge MoE Model Fits on One Consumer GPU".  A
    router sends each token to a few experts.  In the offload strategy the
    experts live in host RAM, and the GPU keeps a least-recently-used cache of
    expert slots.  A cached expert runs on the GPU; a miss is streamed over PCIe.
    One global LRU pool is shared by all layers.
  * same page, section "The Real Requirement Is System RAM": NVFP4 stores
    4-bit values plus an 8-bit scale for every 16 weights (4.5 bits/weight).
  * same page, section "Long Prompts Are the Bottleneck": during prefill, every
    MoE layer copies all of its experts to the GPU for each chunk.  The copy
    for layer N+1 overlaps the compute of layer N, and the cache must hold the
    two staging layers.
  * "FreeToken: Run a 290B MoE Model on One Gaming GPU" (wpnews.pro), section
    "VRAM Is Not the Bottleneck You Think It Is": the full expert pool stays
    in system RAM, and VRAM is an LRU cache of recently activated experts.

The pages are silent on everything else.  Readings taken where they are silent:
  * top-k is taken on the raw logits: the k largest, ties to the lower expert
    id, in descending order.  The gates are a softmax over those k logits.
    NaN logits count as -inf (so a row with fewer than k finite logits takes
    the rest of its experts from the -inf ones, lowest id first); the softmax
    runs in IEEE arithmetic, so a selected +inf or an all -inf selection gives
    NaN gates.
  * SwiGLU expert: y = W_d (silu(W_g x) * (W_u x)).  No bias, no shared expert.
  * h is rounded to bf16 before the down projection (the GPU path stores h in
    bf16).  y and the combine stay in float64 here.
  * cache: one "lookup" is one distinct (layer, expert) per call.  First, hits
    move to the MRU end in ascending expert id.  Then misses, in ascending id,
    take the lowest free slot, or evict the LRU key.  Warm fill at load time:
    keys (layer, expert) in lexicographic order go to slots 0.., and slot 0 is
    the LRU.
  * prefill hit-D2D ("FreeToken: Run Frontier MoE Models on Your Own GPU, and
    the RAM It Takes", section "Long Prompts Are the Bottleneck": prefill can
    skip the experts already in the GPU cache, so that only the others cross
    PCIe): the staging banks are the last 2E slots and the cache keeps the
    first S - 2E.  With the option on, a switch of mode keeps the cache under
    the resize rules (ExpertSlotLRU.resize), and a staged expert whose key is
    cached is copied from its slot (counted as hit_d2d), not from host memory.
    Prefill neither fills the cache nor changes its recency: a prefill chunk
    touches every expert of every layer, in layer order.
  * formats: OCP Microscaling (MX) v1.0 for e2m1, E8M0 and MXFP4 (scale per 32).
    NVFP4 = e2m1 x E4M3 scale per 16 x an fp32 per-matrix global scale.  FP8
    (the pages name it among the weight formats, with no detail) = E4M3 x an
    fp32 scale per output row.  The blob layout is the one documented in
    ``ftgen/ftgen.c``.
"""
from __future__ import annotations

import math

import numpy as np

FMT_BF16, FMT_NVFP4, FMT_MXFP4, FMT_FP8 = 0, 1, 2, 3
MODE_LRU, MODE_STREAM = 0, 1

# ----------------------------------------------------------------------------
# Element formats (OCP Microscaling Formats v1.0: FP4 E2M1 element, E8M0
# scale; OCP 8-bit floating point: E4M3 "FN").
# ----------------------------------------------------------------------------

#: magnitudes of e2m1 codes 0..7 (1 sign bit above them)
E2M1_MAGNITUDE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_value(code: int) -> float:
    """4-bit e2m1 code -> value; bit 3 is the sign, bits 0..2 index the magnitude."""
    mag = E2M1_MAGNITUDE[code & 7]
    return -mag if code & 8 else mag


def e4m3_value(byte: int) -> float:
    """E4M3 (bias 7, no infinities, S.1111.111 is NaN) -> value."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e8m0_value(byte: int) -> float:
    """E8M0 scale (exponent only, bias 127, 0xFF is NaN) -> 2^(byte-127)."""
    if byte == 0xFF:
        return math.nan
    return 2.0 ** (byte - 127)


def bf16_value(bits: int) -> float:
    """bf16 bit pattern -> value (the upper half of an IEEE binary32)."""
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


_E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)
_E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Rounds float64 values to the nearest bf16 value (8 significant bits), ties to even."""
    m, e = np.frexp(np.asarray(a, np.float64))
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


# ----------------------------------------------------------------------------
# Blob layout and dequantisation
# ----------------------------------------------------------------------------

def blob_bytes(fmt: int, H: int, I: int) -> int:
    """Packed bytes of one expert (three matrices, 3*H*I weights).

    NVFP4 holds 4 bits per weight plus one byte per 16 weights (4.5 bits,
    "The Real Requirement Is System RAM"), plus 16 bytes of global scales."""
    n = 3 * H * I
    if fmt == FMT_BF16:
        return 2 * n
    if fmt == FMT_NVFP4:
        return n // 2 + n // 16 + 16
    if fmt == FMT_MXFP4:
        return n // 2 + n // 32
    if fmt == FMT_FP8:
        return n + 4 * (2 * I + H)
    raise ValueError(fmt)


def _fp4_matrix(codes: np.ndarray, scale_of_element: np.ndarray) -> np.ndarray:
    """codes: uint8 [rows, K/2] (element 2j low nibble); scale_of_element [rows, K]."""
    lo = codes & 0x0F
    hi = codes >> 4
    rows = codes.shape[0]
    nib = np.empty((rows, codes.shape[1] * 2), dtype=np.uint8)
    nib[:, 0::2] = lo
    nib[:, 1::2] = hi
    return _E2M1_TABLE[nib] * scale_of_element


def dequant_expert(blob: np.ndarray, fmt: int, H: int, I: int):
    """Decodes one expert blob into float64 (W_g [I,H], W_u [I,H], W_d [H,I])."""
    blob = np.asarray(blob, np.uint8).reshape(-1)
    HI = H * I
    if fmt == FMT_BF16:
        w = bf16_bits_to_f64(blob[: 6 * HI].view(np.uint16))
        gu = w[: 2 * HI].reshape(2 * I, H)
        wd = w[2 * HI:].reshape(H, I)
        return gu[:I], gu[I:], wd
    if fmt == FMT_NVFP4:
        o = 0
        gu_c = blob[o:o + HI].reshape(2 * I, H // 2); o += HI
        gu_s = blob[o:o + HI // 8].reshape(2 * I, H // 16); o += HI // 8
        d_c = blob[o:o + HI // 2].reshape(H, I // 2); o += HI // 2
        d_s = blob[o:o + HI // 16].reshape(H, I // 16); o += HI // 16
        g = blob[o:o + 16].view(np.float32).astype(np.float64)
        # w = e2m1(code) * E4M3(scale of its 16-element block) * global scale
        s_gu = np.repeat(_E4M3_TABLE[gu_s], 16, axis=1)
        s_gu[:I] *= g[0]
        s_gu[I:] *= g[1]
        s_d = np.repeat(_E4M3_TABLE[d_s], 16, axis=1) * g[2]
        gu = _fp4_matrix(gu_c, s_gu)
        wd = _fp4_matrix(d_c, s_d)
        return gu[:I], gu[I:], wd
    if fmt == FMT_MXFP4:
        o = 0
        gu_c = blob[o:o + HI].reshape(2 * I, H // 2); o += HI
        gu_s = blob[o:o + HI // 16].reshape(2 * I, H // 32); o += HI // 16
        d_c = blob[o:o + HI // 2].reshape(H, I // 2); o += HI // 2
        d_s = blob[o:o + HI // 32].reshape(H, I // 32)
        # w = e2m1(code) * 2^(E8M0 scale of its 32-element block - 127)
        gu = _fp4_matrix(gu_c, np.repeat(_E8M0_TABLE[gu_s], 32, axis=1))
        wd = _fp4_matrix(d_c, np.repeat(_E8M0_TABLE[d_s], 32, axis=1))
        return gu[:I], gu[I:], wd
    if fmt == FMT_FP8:
        o = 0
        gu_c = blob[o:o + 2 * HI].reshape(2 * I, H); o += 2 * HI
        gu_s = blob[o:o + 8 * I].view(np.float32).astype(np.float64); o += 8 * I
        d_c = blob[o:o + HI].reshape(H, I); o += HI
        d_s = blob[o:o + 4 * H].view(np.float32).astype(np.float64)
        # w = E4M3(code) * fp32 scale of its row
        gu = _E4M3_TABLE[gu_c] * gu_s[:, None]
        wd = _E4M3_TABLE[d_c] * d_s[:, None]
        return gu[:I], gu[I:], wd
    raise ValueError(fmt)


# ----------------------------------------------------------------------------
# Router: top-k selection and gates
# ("Why a Huge MoE Model Fits on One Consumer GPU": a router sends each token
# to only a few experts.)
# ----------------------------------------------------------------------------

def _selection_values(logits: np.ndarray) -> np.ndarray:
    """The values top-k compares and the gates use: the logits as float64,
    with NaN read as -inf (the pages say nothing about non-finite logits)."""
    v = np.asarray(logits, np.float64).copy()
    v[np.isnan(v)] = -np.inf
    return v


def topk_experts(logits: np.ndarray, k: int) -> np.ndarray:
    """[T, E] logits -> [T, k] expert ids: k rounds of "take the largest value
    among the experts not yet taken, the lowest id among equal values".
    NaN counts as -inf, so a row with fewer than k finite logits takes its
    remaining experts from the -inf ones in ascending id."""
    v = _selection_values(logits)
    T, E = v.shape
    taken = np.zeros((T, E), dtype=bool)
    out = np.empty((T, k), dtype=np.int32)
    rows = np.arange(T)
    for j in range(k):
        best_val = np.where(taken, -np.inf, v).max(axis=1)
        # the first untaken expert holding that value (-inf included)
        best = np.argmax(~taken & (v == best_val[:, None]), axis=1)
        out[:, j] = best
        taken[rows, best] = True
    return out


def gates_of(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Softmax over the k selected values of each token, in IEEE float64
    arithmetic (returned as float32): exp(l_j - max) / sum.  NaN logits are
    read as -inf.  A token whose selected values hold +inf, or are all -inf,
    gets NaN gates, as a library softmax gives."""
    sel = np.take_along_axis(_selection_values(logits), idx.astype(np.int64), axis=1)
    with np.errstate(invalid="ignore"):
        z = np.exp(sel - sel.max(axis=1, keepdims=True))
        return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


# ----------------------------------------------------------------------------
# Global LRU cache of expert slots
# ("Why a Huge MoE Model Fits on One Consumer GPU": LRU cache of expert slots,
# one global pool shared across layers.)
# ----------------------------------------------------------------------------

class ExpertSlotLRU:
    """Slots 0..S-1 holding keys (layer * E + expert); recency kept as a list,
    least recently used first."""

    def __init__(self, n_slots: int, n_layers: int, n_experts: int):
        self.S, self.L, self.E = n_slots, n_layers, n_experts
        self.slot_key = [-1] * n_slots
        self.key_slot: dict[int, int] = {}
        self.recency: list[int] = []

    def warm_fill(self) -> int:
        """Keys in (layer, expert) order into slots 0.. until the slots or the pool run out."""
        n = min(self.S, self.L * self.E)
        for key in range(n):
            self.slot_key[key] = key
            self.key_slot[key] = key
            self.recency.append(key)
        return n

    def lookup(self, layer: int, experts: list[int]):
        """One call's distinct experts (ascending).  Returns, per expert in that
        order, (expert, slot, hit, evicted_key or -1)."""
        keys = [layer * self.E + e for e in experts]
        hit = [k in self.key_slot for k in keys]
        # phase 1: hits become most recent, in ascending expert id
        for k, h in zip(keys, hit):
            if h:
                self.recency.remove(k)
                self.recency.append(k)
        plan = {}
        # phase 2: misses take the lowest free slot, else the LRU key's slot
        for e, k, h in zip(experts, keys, hit):
            if h:
                plan[e] = (e, self.key_slot[k], True, -1)
                continue
            free = [s for s in range(self.S) if self.slot_key[s] == -1]
            if free:
                slot, victim = free[0], -1
            else:
                victim = self.recency.pop(0)
                slot = self.key_slot.pop(victim)
            self.slot_key[slot] = k
            self.key_slot[k] = slot
            self.recency.append(k)
            plan[e] = (e, slot, False, victim)
        return [plan[e] for e in experts]

    def resize(self, n_slots: int) -> list[int]:
        """Changes the number of slots ("Why a Huge MoE Model Fits on One
        Consumer GPU": VRAM moves between the expert cache and the KV cache at
        run time, without a restart; "FreeToken uses bandwidth-adaptive CPU-GPU
        co-execution on your desktop", "Memory that moves while the engine
        runs": VRAM is re-allocated between the expert caches and KV memory
        without reloading weights).  Readings: the cache keeps its most
        recently used keys, as many as fit, in the same recency order; the
        others leave (not counted as evictions of a call).  A kept key stays in
        its slot if that slot still exists, else it takes the lowest free slot,
        least recent key first.  New slots start free.  Returns the keys that
        left, least recent first."""
        n_gone = max(0, len(self.recency) - n_slots)
        keep, gone = self.recency[n_gone:], self.recency[:n_gone]
        slot_key = [-1] * n_slots
        key_slot = {}
        moved = []
        for key in keep:
            slot = self.key_slot[key]
            if slot < n_slots:
                slot_key[slot] = key
                key_slot[key] = slot
            else:
                moved.append(key)
        for key in moved:
            slot = slot_key.index(-1)
            slot_key[slot] = key
            key_slot[key] = slot
        self.S, self.slot_key, self.key_slot, self.recency = n_slots, slot_key, key_slot, keep
        return gone


# ----------------------------------------------------------------------------
# Permute tokens by expert (stable counting sort of the (token, rank) pairs)
# ----------------------------------------------------------------------------

def permute_by_expert(idx: np.ndarray, E: int):
    """idx [T, k] -> (offsets [E+1], perm [T*k], inv [T*k]).

    Pair p = t*k + j.  perm[i] = the pair in position i.  Pairs are grouped by
    expert in ascending order, and by p within a group.  inv[p] = position of p."""
    flat = [int(v) for v in np.asarray(idx).reshape(-1)]
    counts = [0] * E
    for e in flat:
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    nxt = offsets[:E]
    nxt = list(nxt)
    perm = [0] * len(flat)
    inv = [0] * len(flat)
    for p, e in enumerate(flat):
        perm[nxt[e]] = p
        inv[p] = nxt[e]
        nxt[e] += 1
    return np.array(offsets, np.int32), np.array(perm, np.int32), np.array(inv, np.int32)


# ----------------------------------------------------------------------------
# Activation quantiser of the FP4 x FP4 variant
# (the pages name NVFP4 as a weight format and say nothing of activation
# precision; this variant quantises the activations too, so that both GEMM
# operands are FP4.  Reading: the NVFP4 layout of the weights -- e2m1 codes,
# one E4M3 scale per 16 consecutive elements of a row -- applied to x and h;
# x rows also get an fp32 second-level scale g = amax(row) / (6 * 448), h rows
# none.  Every quantiser decision is taken in IEEE binary32, as the kernels
# take it.)
# ----------------------------------------------------------------------------

#: values of the non-negative finite E4M3 codes 0..126, ascending
_E4M3_NONNEG = np.array([e4m3_value(b) for b in range(127)], dtype=np.float64)


def e4m3_encode_nonneg(v: np.ndarray) -> np.ndarray:
    """Non-negative values -> E4M3 codes: the nearest E4M3 value, a tie to
    the even code, values above 448 to 448 (saturation)."""
    v = np.asarray(v, np.float64)
    hi = np.clip(np.searchsorted(_E4M3_NONNEG, v, side="left"), 1, 126)
    lo = hi - 1
    d_lo, d_hi = v - _E4M3_NONNEG[lo], _E4M3_NONNEG[hi] - v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(v >= _E4M3_NONNEG[126], 126, code)
    return code.astype(np.uint8)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Values -> 4-bit e2m1 codes: the nearest of the 8 magnitudes, a tie to
    the even code, magnitudes above 6 to 6 (saturation); bit 3 is the sign
    bit of v (so -0 and negative values that round to 0 give code 8)."""
    v = np.asarray(v, np.float64)
    mag = np.abs(v)
    grid = np.array(E2M1_MAGNITUDE)
    hi = np.clip(np.searchsorted(grid, mag, side="left"), 1, 7)
    lo = hi - 1
    d_lo, d_hi = mag - grid[lo], grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= 6.0, 7, code)
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def quantize_act_fp4(a: np.ndarray, row_scale: bool):
    """Rows of activations a [n, K] -> (codes uint8 [n, K] one 4-bit code per
    element, block scales uint8 [n, K/16] E4M3, g float32 [n]), all in float32:
      g   = amax(row) / 2688 (6 * 448), or 1 for an all-zero row or without row_scale
      s_b = E4M3( (amax(block) / 6) / g )                  (nearest, ties to even)
      r_b = 1 / (value(s_b) * g)                           (one rounding; 0 where the product is 0)
      q   = e2m1( a * r_b )                                (nearest, ties to even)"""
    a = np.asarray(a, np.float32)
    n, K = a.shape
    f = np.float32
    if row_scale:
        amax = np.abs(a).max(axis=1)
        g = (amax / f(2688.0)).astype(np.float32)
        g[amax == 0] = f(1.0)
    else:
        g = np.ones(n, np.float32)
    blocks = np.abs(a).reshape(n, K // 16, 16).max(axis=2)
    s = ((blocks / f(6.0)).astype(np.float32) / g[:, None]).astype(np.float32)
    sf = e4m3_encode_nonneg(s)
    denom = (_E4M3_TABLE[sf].astype(np.float32) * g[:, None]).astype(np.float32)
    with np.errstate(divide="ignore"):
        recip = np.where(denom > 0, f(1.0) / np.where(denom > 0, denom, f(1.0)), f(0.0)).astype(np.float32)
    v = (a * np.repeat(recip, 16, axis=1)).astype(np.float32)
    return e2m1_encode(v), sf, g


def dequant_act_fp4(codes: np.ndarray, sf: np.ndarray, g: np.ndarray) -> np.ndarray:
    """The values that quantize_act_fp4's output stands for (float64)."""
    scale = np.repeat(_E4M3_TABLE[sf], 16, axis=1) * np.asarray(g, np.float64)[:, None]
    return _E2M1_TABLE[codes] * scale


# ----------------------------------------------------------------------------
# Expert FFN (SwiGLU) and combine
# ----------------------------------------------------------------------------

def silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def expert_ffn(x_rows: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray,
               h_bf16: bool = True, act_fp4: bool = False) -> np.ndarray:
    """x_rows [n, H] float64 -> y [n, H]:  y = W_d (silu(W_g x) * (W_u x)).

    act_fp4 (the FP4 x FP4 variant): x is quantised first (quantize_act_fp4
    with its row scale), and h, taken to float32, is quantised before the down
    projection (block scales only); otherwise h is rounded to bf16 when h_bf16."""
    if act_fp4:
        x_rows = dequant_act_fp4(*quantize_act_fp4(x_rows, row_scale=True))
    g = x_rows @ Wg.T
    u = x_rows @ Wu.T
    h = silu(g) * u
    if act_fp4:
        h = dequant_act_fp4(*quantize_act_fp4(h.astype(np.float32), row_scale=False))
    elif h_bf16:
        h = round_to_bf16(h)
    return h @ Wd.T


def combine(y: np.ndarray, gates: np.ndarray, inv: np.ndarray, T: int, k: int) -> np.ndarray:
    """out[t] = sum over j = 0..k-1 (in that order) of gates[t, j] * y[inv[t*k + j]]."""
    H = y.shape[1]
    out = np.zeros((T, H), np.float64)
    for t in range(T):
        for j in range(k):
            out[t] += float(gates[t, j]) * y[inv[t * k + j]]
    return out


# ----------------------------------------------------------------------------
# The layer
# ----------------------------------------------------------------------------

class MoELayerOracle:
    """A stack of L MoE layers sharing one slot cache, one call per (layer, batch).

    blob_of(key) -> uint8 blob of expert key = layer * E + e (the host pool)."""

    def __init__(self, H: int, E: int, k: int, I: int, fmt: int, n_slots: int, n_layers: int,
                 blob_of, mode: int = MODE_LRU, h_bf16: bool = True, hit_d2d: bool = False,
                 act_fp4: bool = False):
        self.H, self.E, self.k, self.I, self.fmt = H, E, k, I, fmt
        self.S, self.L, self.mode = n_slots, n_layers, mode
        self.blob_of = blob_of
        self.h_bf16 = h_bf16
        self.act_fp4 = act_fp4
        self.hit_d2d = hit_d2d
        self.nbytes = blob_bytes(fmt, H, I)
        self._wcache: dict[int, tuple] = {}
        self.wcache_max = 64          # decoded experts kept (memory only; no effect on results)
        self.reset()

    def reset(self, warm: bool = True):
        """Cache back to the warm-fill state (or all slots free when warm is
        False); statistics cleared."""
        self.stats = dict(lookups=0, hits=0, misses=0, evictions=0, warm_loads=0, streamed=0, bytes_h2d=0,
                          hit_d2d=0)
        self.lru = ExpertSlotLRU(self.cache_slots(), self.L, self.E)
        self.bank_layer = [-1, -1]
        if self.mode == MODE_LRU and warm:
            n = self.lru.warm_fill()
            self.stats["warm_loads"] += n
            self.stats["bytes_h2d"] += n * self.nbytes

    def cache_slots(self) -> int:
        """Slots that belong to the LRU cache: all S in LRU mode; in STREAM mode
        the last 2E are the two staging banks, so the first S - 2E."""
        return self.S if self.mode == MODE_LRU else self.S - 2 * self.E

    def resize_slots(self, n_slots: int):
        """The slot count changes: the cache follows ExpertSlotLRU.resize onto
        its new share; in STREAM mode the staging banks start empty."""
        self.S = n_slots
        if self.mode == MODE_STREAM:
            self.bank_layer = [-1, -1]
        self.lru.resize(self.cache_slots())

    def set_mode(self, mode: int):
        """LRU (decode) or STREAM (prefill).  Without hit-D2D the cache starts
        over in the new mode's initial state (reset: warm fill in LRU mode,
        empty in STREAM mode).  With it the cache lives through the switch: it
        shrinks onto the first S - 2E slots when STREAM mode begins and grows
        back to S when it ends (ExpertSlotLRU.resize in both directions), and
        the statistics carry on.  Setting the current mode again with hit-D2D
        on changes nothing."""
        if not self.hit_d2d:
            self.mode = mode
            self.reset()
            return
        if mode == self.mode:
            return
        self.mode = mode
        self.bank_layer = [-1, -1]
        self.lru.resize(self.cache_slots())

    def weights(self, key: int):
        if key not in self._wcache:
            if len(self._wcache) >= self.wcache_max:
                self._wcache.clear()
            self._wcache[key] = dequant_expert(self.blob_of(key), self.fmt, self.H, self.I)
        return self._wcache[key]

    def _stream(self, layer: int, last: dict):
        """Full-layer streaming: bank (layer mod 2) must hold all E experts of
        `layer` before it computes; the next layer's experts are copied into the
        other bank at the same call ("Long Prompts Are the Bottleneck").  With
        hit-D2D on, an expert whose key is in the cache comes from its slot."""
        def fill(l):
            b = l % 2
            if self.bank_layer[b] != l:
                self.bank_layer[b] = l
                for e in range(self.E):
                    if self.hit_d2d and l * self.E + e in self.lru.key_slot:
                        last["hit_d2d"] += 1          # from its cache slot
                    else:
                        last["streamed"] += 1         # from host memory
                        last["bytes_h2d"] += self.nbytes
        fill(layer)
        nxt = layer + 1 if layer + 1 < self.L else 0
        if nxt % 2 != layer % 2:
            fill(nxt)

    def forward(self, layer: int, x_bits: np.ndarray, logits: np.ndarray, tokens=None, ffn_experts=None):
        """x_bits: bf16 bits [T, H]; logits: float32 [T, E].

        Returns a dict with routing (idx, gates), permutation, the cache plan
        for this call, the per-call statistics, and out (float64 [T, H], or only
        the rows in `tokens` when a token sample is given).

        ffn_experts (timing samples only): evaluate the FFN of just these
        experts of the call; routing and the cache update still run in full,
        and out then holds no meaningful values."""
        T = x_bits.shape[0]
        idx = topk_experts(logits, self.k)
        gates = gates_of(logits, idx)
        experts = sorted(set(int(e) for e in idx.reshape(-1)))
        last = dict(lookups=len(experts), hits=0, misses=0, evictions=0, warm_loads=0, streamed=0, bytes_h2d=0,
                    hit_d2d=0)
        if self.mode == MODE_LRU:
            plan = self.lru.lookup(layer, experts)
            for (_, _, hit, victim) in plan:
                if hit:
                    last["hits"] += 1
                else:
                    last["misses"] += 1
                    last["bytes_h2d"] += self.nbytes
                    if victim >= 0:
                        last["evictions"] += 1
        else:
            self._stream(layer, last)
            plan = [(e, self.cache_slots() + (layer % 2) * self.E + e, True, -1) for e in experts]
        for key_, v in last.items():
            self.stats[key_] += v
        offsets, perm, inv = permute_by_expert(idx, self.E)
        res = dict(idx=idx, gates=gates, experts=experts, plan=plan, offsets=offsets, perm=perm,
                   inv=inv, last=last)
        want = set(range(T)) if tokens is None else set(int(t) for t in tokens)
        x = bf16_bits_to_f64(x_bits)
        y = {}
        if ffn_experts is not None:
            res["out"] = None
            res["out_tokens"] = np.array(sorted(want), np.int64)
            for e in ffn_experts:
                lo, hi = int(offsets[e]), int(offsets[e + 1])
                pairs = [int(p) for p in perm[lo:hi] if int(p) // self.k in want]
                if pairs:
                    Wg, Wu, Wd = self.weights(layer * self.E + e)
                    expert_ffn(np.stack([x[p // self.k] for p in pairs]), Wg, Wu, Wd, self.h_bf16, self.act_fp4)
            return res
        for e in experts:
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            pairs = [int(p) for p in perm[lo:hi] if int(p) // self.k in want]
            if not pairs:
                continue
            Wg, Wu, Wd = self.weights(layer * self.E + e)
            rows = np.stack([x[p // self.k] for p in pairs])
            ys = expert_ffn(rows, Wg, Wu, Wd, self.h_bf16, self.act_fp4)
            for p, yr in zip(pairs, ys):
                y[int(inv[p])] = yr          # y is kept in permuted order
        order = sorted(want)
        out = np.zeros((len(order), self.H), np.float64)
        for r, t in enumerate(order):
            for j in range(self.k):
                out[r] += float(gates[t, j]) * y[int(inv[t * self.k + j])]
        res["out"] = out
        res["out_tokens"] = np.array(order, np.int64)
        return res
