"""Pins of the CPU oracle to things other than itself: the pages' own figures,
closed forms, library routines, brute force and hand-worked traces.

Each test is chosen so that a plausible slip in the oracle (a wrong table
entry, a swapped nibble, a transposed section, a dropped term, a wrong tie
rule) fails it.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import ftgen
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats

def test_e2m1_from_bit_fields():
    # e2m1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal
    for c in range(16):
        s = -1.0 if c & 8 else 1.0
        e = (c >> 1) & 3
        m = c & 1
        want = s * (m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2))
        assert O.e2m1_value(c) == want, c


def test_e4m3_matches_torch_for_all_bytes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([O.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_e8m0_matches_torch_for_all_bytes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([O.e8m0_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_bf16_decode_and_rounding_match_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, 4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]           # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_bits_to_f64(bits), ref)
    assert O.bf16_value(0x3F80) == 1.0 and O.bf16_value(0xC000) == -2.0
    # rounding: fp32-representable values (one rounding step on both sides)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(v.astype(np.float64)), ref)


def _hand_blob_nvfp4(I, H, scale_of_row, g):
    """Builds an NVFP4 blob by hand: in every 16-block, element i carries code
    i; row r's block scales are all scale_of_row(r)."""
    HI = H * I
    nib = np.tile(np.arange(16, dtype=np.uint8), H // 16)           # one row of codes
    row_codes = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    gu_c = np.tile(row_codes, (2 * I, 1))
    gu_s = np.array([[scale_of_row(r)] * (H // 16) for r in range(2 * I)], np.uint8)
    nib_d = np.tile(np.arange(16, dtype=np.uint8), I // 16)
    d_c = np.tile((nib_d[0::2] | (nib_d[1::2] << 4)).astype(np.uint8), (H, 1))
    d_s = np.array([[scale_of_row(r)] * (I // 16) for r in range(H)], np.uint8)
    gs = np.array(g + [0.0], np.float32).view(np.uint8)
    blob = np.concatenate([gu_c.ravel(), gu_s.ravel(), d_c.ravel(), d_s.ravel(), gs])
    assert blob.size == O.blob_bytes(O.FMT_NVFP4, H, I) == 27 * HI // 16 + 16
    return blob


def test_nvfp4_dequant_all_codes_times_all_scales():
    # 2I = 256 rows -> row r uses E4M3 byte r: every (code, scale) pair appears
    I, H = 128, 32
    g = [0.75, 1.5, 2.0]
    blob = _hand_blob_nvfp4(I, H, lambda r: r % 256, g)
    Wg, Wu, Wd = O.dequant_expert(blob, O.FMT_NVFP4, H, I)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    code = np.arange(H) % 16
    e2m1 = np.array([(-1.0 if c & 8 else 1.0) * [0, .5, 1, 1.5, 2, 3, 4, 6][c & 7] for c in range(16)])
    for r in range(2 * I):
        W, rr, gg = (Wg, r, g[0]) if r < I else (Wu, r - I, g[1])
        want = e2m1[code] * e4m3[r] * gg
        np.testing.assert_array_equal(np.isnan(W[rr]), np.isnan(want))
        ok = ~np.isnan(want)
        np.testing.assert_array_equal(W[rr][ok], want[ok])
    code_d = np.arange(I) % 16
    for r in range(H):
        np.testing.assert_array_equal(Wd[r], e2m1[code_d] * e4m3[r] * g[2])


def test_mxfp4_dequant_all_codes_times_all_scales():
    I, H = 128, 64
    HI = H * I
    nib = np.tile(np.arange(16, dtype=np.uint8), H // 16)
    gu_c = np.tile((nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), (2 * I, 1))
    gu_s = np.array([[r % 255] * (H // 32) for r in range(2 * I)], np.uint8)   # bytes 0..254
    nib_d = np.tile(np.arange(16, dtype=np.uint8), I // 16)
    d_c = np.tile((nib_d[0::2] | (nib_d[1::2] << 4)).astype(np.uint8), (H, 1))
    d_s = np.array([[(3 * r) % 255] * (I // 32) for r in range(H)], np.uint8)
    blob = np.concatenate([gu_c.ravel(), gu_s.ravel(), d_c.ravel(), d_s.ravel()])
    assert blob.size == O.blob_bytes(O.FMT_MXFP4, H, I) == 51 * HI // 32
    Wg, Wu, Wd = O.dequant_expert(blob, O.FMT_MXFP4, H, I)
    e8m0 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    e2m1 = np.array([(-1.0 if c & 8 else 1.0) * [0, .5, 1, 1.5, 2, 3, 4, 6][c & 7] for c in range(16)])
    code = np.arange(H) % 16
    for r in range(2 * I):
        W, rr = (Wg, r) if r < I else (Wu, r - I)
        np.testing.assert_array_equal(W[rr], e2m1[code] * e8m0[r % 255])
    for r in range(H):
        np.testing.assert_array_equal(Wd[r], e2m1[np.arange(I) % 16] * e8m0[(3 * r) % 255])


def test_fp8_dequant_all_codes_times_row_scales():
    # every E4M3 byte in every row, each row with its own fp32 scale: the oracle
    # equals torch's E4M3 decode times the row's scale, section by section
    H, I = 256, 256
    HI = H * I
    gu_c = np.tile(np.arange(256, dtype=np.uint8), (2 * I, H // 256))
    gu_s = (np.arange(2 * I, dtype=np.float32) + 1.0) * np.float32(0.001)
    d_c = np.tile(np.arange(256, dtype=np.uint8)[::-1].copy(), (H, I // 256))
    d_s = (np.arange(H, dtype=np.float32) + 3.0) * np.float32(0.0007)
    blob = np.concatenate([gu_c.ravel(), gu_s.view(np.uint8), d_c.ravel(), d_s.view(np.uint8)])
    assert blob.size == O.blob_bytes(O.FMT_FP8, H, I) == ftgen.blob_bytes("fp8", H, I) == 3 * HI + 4 * (2 * I + H)
    Wg, Wu, Wd = O.dequant_expert(blob, O.FMT_FP8, H, I)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for r in range(2 * I):
        W, rr = (Wg, r) if r < I else (Wu, r - I)
        np.testing.assert_array_equal(W[rr], e4m3[gu_c[r]] * np.float64(gu_s[r]))
    for r in range(H):
        np.testing.assert_array_equal(Wd[r], e4m3[d_c[r]] * np.float64(d_s[r]))


def test_dequant_fp8_is_within_half_an_e4m3_step_of_master_weights():
    # pins the FP8 blob's section order and orientation against the master
    # weights: each weight is the master value to within half an E4M3 step of
    # its row's scale (3 mantissa bits: 2^-4 relative; 2^-10 x scale below 2^-6)
    H, I = 256, 128
    blob = ftgen.expert_blob("fp8", H, I, key=4, seed=6)
    Ws = O.dequant_expert(blob, O.FMT_FP8, H, I)
    Ms = ftgen.master_weights(H, I, key=4, seed=6)
    for W, M in zip(Ws, Ms):
        M = M.astype(np.float64)
        scale = np.abs(M).max(axis=1, keepdims=True) / 448.0
        bound = np.maximum(np.abs(M) * 2.0 ** -4, scale * 2.0 ** -10) * (1 + 1e-6)
        assert np.all(np.abs(W - M) <= bound)


def test_dequant_bf16_is_within_half_ulp_of_master_weights():
    # pins the blob section order and orientation (gate, up, down) against the
    # fp32 master weights the generator quantised
    H, I = 64, 96
    blob = ftgen.expert_blob("bf16", H, I, key=7, seed=99)
    Wg, Wu, Wd = O.dequant_expert(blob, O.FMT_BF16, H, I)
    g, u, d = ftgen.master_weights(H, I, key=7, seed=99)
    for W, M in ((Wg, g), (Wu, u), (Wd, d)):
        assert W.shape == M.shape
        half_ulp = np.ldexp(1.0, np.floor(np.log2(np.abs(M).astype(np.float64))).astype(int) - 8)
        assert np.all(np.abs(W - M) <= half_ulp)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_dequant_fp4_tracks_master_weights(fmt):
    H, I = 256, 128
    blob = ftgen.expert_blob(fmt, H, I, key=3, seed=5)
    Ws = O.dequant_expert(blob, O.FMT_NVFP4 if fmt == "nvfp4" else O.FMT_MXFP4, H, I)
    Ms = ftgen.master_weights(H, I, key=3, seed=5)
    for W, M in zip(Ws, Ms):
        rel = np.linalg.norm(W - M) / np.linalg.norm(M)
        assert rel < 0.2, rel                       # 4-bit grid: ~10 % rms error
        corr = np.corrcoef(W.ravel(), M.ravel())[0, 1]
        assert corr > 0.97, corr                     # a misplaced section would decorrelate


def _golden_numbers():
    vals = {}
    for line in open(os.path.join(GOLDEN, "pages_arithmetic.txt")):
        if line.strip() and not line.startswith("#"):
            name, v = line.split()[:2]
            vals[name] = float(v)
    return vals


def test_packed_size_matches_pages():
    gv = _golden_numbers()
    for H, I in ((2048, 768), (7168, 2048), (6144, 2048), (256, 512)):
        n = 3 * H * I
        bits = (O.blob_bytes(O.FMT_NVFP4, H, I) - 16) * 8 / n
        assert bits == gv["nvfp4_bits_per_weight"]
        assert O.blob_bytes(O.FMT_BF16, H, I) * 8 / n == 16
        assert O.blob_bytes(O.FMT_MXFP4, H, I) * 8 / n == 4.25
    # the pages' estimates: 284B at 4 bits ~142 GB, at 4.5 bits ~160 GB; 35B at 4.5 ~20 GB
    assert round(284e9 * 4 / 8 / 1e9) == gv["fp4_params_284b_gb"]
    assert abs(284e9 * gv["nvfp4_bits_per_weight"] / 8 / 1e9 - gv["nvfp4_params_284b_gb"]) < 1.0
    assert abs(35e9 * gv["nvfp4_bits_per_weight"] / 8 / 1e9 - gv["nvfp4_params_35b_gb"]) < 0.5


def test_stream_copy_time_formula_matches_pages():
    gv = _golden_numbers()
    t = gv["expert_bytes_284b_gb"] / gv["pcie5_h2d_gbps"]
    assert abs(t - gv["chunk_copy_s"]) < 0.05
    assert abs(gv["chunk_tokens"] / t - gv["prefill_tokens_per_s"]) < 50
    chunks = math.ceil(gv["context_tokens"] / gv["chunk_tokens"])
    assert chunks == gv["context_chunks"]
    assert abs(chunks * t - gv["context_copy_s"]) < 0.5


# ---------------------------------------------------------------- router

def _stable_sort_topk(logits, k):
    out = []
    for row in np.asarray(logits, np.float64):
        order = np.lexsort((np.arange(row.size), -row))    # by -logit, then by id
        out.append(order[:k])
    return np.array(out, np.int32)


def test_topk_equals_full_stable_sort_random_and_tied():
    rng = np.random.default_rng(1)
    for E, k in ((8, 2), (128, 8), (256, 8), (5, 5), (1, 1)):
        lg = rng.standard_normal((64, E)).astype(np.float32)
        assert np.array_equal(O.topk_experts(lg, k), _stable_sort_topk(lg, k))
        tied = rng.integers(-2, 3, (64, E)).astype(np.float32)  # many equal logits
        assert np.array_equal(O.topk_experts(tied, k), _stable_sort_topk(tied, k))


def test_topk_exhaustive_tiny():
    vals = (0.0, 1.0, 2.0)
    rows = np.array(list(itertools.product(vals, repeat=4)), np.float32)
    for k in range(1, 5):
        assert np.array_equal(O.topk_experts(rows, k), _stable_sort_topk(rows, k))


def test_gates_closed_forms():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((50, 16)).astype(np.float32)
    idx = O.topk_experts(lg, 4)
    g = O.gates_of(lg, idx)
    assert np.allclose(g.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(g, axis=1) <= 0)                 # descending logits -> descending gates
    # full softmax over all E, then renormalised over the selected k
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(g, sel / sel.sum(axis=1, keepdims=True), rtol=1e-6)
    # shift invariance and k = 1
    np.testing.assert_allclose(O.gates_of(lg + 3.0, idx), g, rtol=1e-6)
    assert np.all(O.gates_of(lg, O.topk_experts(lg, 1)) == 1.0)


def _parse_nonfinite_cases():
    cases = []
    with open(os.path.join(GOLDEN, "topk_nonfinite.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, lg, idx, gates = (part.split() for part in line.split("|"))
            cases.append((int(k[0]), np.array([float(v) for v in lg], np.float32),
                          np.array([int(v) for v in idx], np.int32), np.array([float(v) for v in gates])))
    return cases


def test_topk_and_gates_on_non_finite_logits_match_hand_worked_cases():
    cases = _parse_nonfinite_cases()
    assert len(cases) >= 6
    for k, lg, want_idx, want_gates in cases:
        idx = O.topk_experts(lg[None, :], k)
        assert np.array_equal(idx[0], want_idx), (lg, idx)
        g = O.gates_of(lg[None, :], idx)[0]
        assert np.array_equal(np.isnan(g), np.isnan(want_gates))
        ok = ~np.isnan(want_gates)
        np.testing.assert_allclose(g[ok], want_gates[ok], rtol=0, atol=1e-7)


def test_topk_on_non_finite_logits_equals_a_sort_with_nan_as_minus_inf():
    rng = np.random.default_rng(5)
    for E, k in ((8, 4), (16, 16), (128, 8)):
        lg = rng.standard_normal((200, E)).astype(np.float32)
        pick = rng.random((200, E))
        lg[pick < 0.2] = -np.inf
        lg[(pick >= 0.2) & (pick < 0.35)] = np.nan
        lg[pick > 0.98] = np.inf
        lg[:3] = np.nan                                    # rows with no finite logit
        mapped = np.where(np.isnan(lg), -np.inf, lg)
        assert np.array_equal(O.topk_experts(lg, k), _stable_sort_topk(mapped, k))
        idx = O.topk_experts(lg, k)
        assert all(len(set(r)) == k for r in idx.tolist())  # k distinct experts per token
        # gates equal a library softmax of the selected (mapped) values
        sel = np.take_along_axis(mapped.astype(np.float64), idx.astype(np.int64), axis=1)
        with np.errstate(invalid="ignore"):
            ref = scipy.special.softmax(sel, axis=1)
        g = O.gates_of(lg, idx)
        assert np.array_equal(np.isnan(g), np.isnan(ref))
        np.testing.assert_allclose(g[~np.isnan(g)], ref[~np.isnan(ref)], rtol=1e-6, atol=1e-7)


# ---------------------------------------------------------------- cache

def _parse_traces():
    traces, cur = [], None
    for line in open(os.path.join(GOLDEN, "lru_traces.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "trace":
            kv = dict(x.split("=") for x in f[2:])
            cur = dict(name=f[1], S=int(kv["S"]), L=int(kv["L"]), E=int(kv["E"]), warm=kv["warm"] == "1",
                       d2d=kv.get("d2d", "0") == "1", calls=[], copies=None)
            traces.append(cur)
        elif f[0] == "call":
            arrow = f.index("->")
            layer, experts = int(f[1]), [int(v) for v in f[2:arrow]]
            plan = []
            for item in f[arrow + 1:]:
                e, s, hm, ev = item.split(":")
                plan.append((int(e), int(s), hm == "hit", -1 if ev == "-" else int(ev)))
            cur["calls"].append((layer, experts, plan))
        elif f[0] == "resize":
            arrow = f.index("->")
            cur["calls"].append(("resize", int(f[1]), [-1 if v == "-" else int(v) for v in f[arrow + 1:]]))
        elif f[0] == "mode":
            arrow = f.index("->")
            cur["calls"].append(("mode", f[1], [-1 if v == "-" else int(v) for v in f[arrow + 1:]]))
        elif f[0] == "prefill":
            arrow = f.index("->")
            counts = dict(v.split("=") for v in f[arrow + 1:])
            cur["calls"].append(("prefill", (int(f[1]), [int(v) for v in f[2:arrow]]),
                                 (int(counts["d2d"]), int(counts["h2d"]))))
        elif f[0] == "stats":
            cur["stats"] = tuple(int(v) for v in f[1:])
        elif f[0] == "copies":
            cur["copies"] = tuple(int(v) for v in f[1:])
    return traces


def _one_hot_logits(experts, E):
    """Logits that route token t to experts[t] alone (k = 1)."""
    lg = np.full((len(experts), E), -5.0, np.float32)
    for t, e in enumerate(experts):
        lg[t, e] = 5.0
    return lg


@pytest.mark.parametrize("trace", [t for t in _parse_traces() if not t["d2d"]], ids=lambda t: t["name"])
def test_lru_hand_worked_traces(trace):
    lru = O.ExpertSlotLRU(trace["S"], trace["L"], trace["E"])
    if trace["warm"]:
        lru.warm_fill()
    look = hits = misses = ev = 0
    for layer, experts, want in trace["calls"]:
        if layer == "resize":
            lru.resize(experts)
            assert lru.slot_key == want
            continue
        got = lru.lookup(layer, experts)
        assert got == want
        look += len(got)
        hits += sum(p[2] for p in got)
        misses += sum(not p[2] for p in got)
        ev += sum(p[3] >= 0 for p in got)
    assert (look, hits, misses, ev) == trace["stats"]


@pytest.mark.parametrize("trace", [t for t in _parse_traces() if t["d2d"]], ids=lambda t: t["name"])
def test_prefill_hit_d2d_hand_worked_traces(trace):
    """The whole layer object (modes, staging banks, copy counts) against the
    hand-worked traces; k = 1 and one-hot logits fix the routing."""
    H = I = 64
    E, L, S = trace["E"], trace["L"], trace["S"]
    blobs = ftgen.pool("bf16", H, I, list(range(L * E)), 9)
    orc = O.MoELayerOracle(H, E, 1, I, O.FMT_BF16, S, L, lambda key: blobs[key], hit_d2d=True)
    orc.reset(warm=trace["warm"])
    for kind, arg, want in trace["calls"]:
        if kind == "resize":
            orc.resize_slots(arg)
            assert orc.lru.slot_key == want
        elif kind == "mode":
            orc.set_mode(O.MODE_STREAM if arg == "stream" else O.MODE_LRU)
            assert orc.lru.slot_key == want
        else:
            layer, experts = (arg if kind == "prefill" else (kind, arg))
            lg = _one_hot_logits(experts, E)
            res = orc.forward(layer, ftgen.x_bf16(9, len(experts), H, 0, layer), lg)
            if kind == "prefill":
                assert (res["last"]["hit_d2d"], res["last"]["streamed"]) == want
                assert res["last"]["hits"] == res["last"]["misses"] == 0
                # the staging banks are the last 2E slots
                assert [p[1] for p in res["plan"]] == [S - 2 * E + (layer % 2) * E + e for e in experts]
            else:
                assert res["plan"] == want
    st = orc.stats
    assert (st["lookups"], st["hits"], st["misses"], st["evictions"]) == trace["stats"]
    assert (st["hit_d2d"], st["streamed"]) == trace["copies"]


def test_prefill_hit_d2d_matches_a_list_model():
    """Random decode calls, mode switches and prefill calls with hit-D2D on,
    against a bare recency list and a bank record kept here: the cache keeps
    its last S - 2E keys into prefill and all of them out of it; each staged
    layer's copies split into cached keys (slot -> bank) and the rest (host ->
    bank); prefill leaves the list alone."""
    rng = np.random.default_rng(11)
    H = I = 64
    for trial in range(40):
        L, E = int(rng.integers(2, 5)), int(rng.integers(1, 4))
        S = 2 * E + int(rng.integers(0, L * E + 2))
        blobs = ftgen.pool("bf16", H, I, list(range(L * E)), 3)
        orc = O.MoELayerOracle(H, E, 1, I, O.FMT_BF16, S, L, lambda key: blobs[key], hit_d2d=True)
        model = list(range(min(S, L * E)))        # warm fill: keys in order, key 0 least recent
        stream, banks = False, [-1, -1]
        for step in range(30):
            r = rng.random()
            if r < 0.15:
                stream = not stream
                orc.set_mode(O.MODE_STREAM if stream else O.MODE_LRU)
                if stream:
                    model = model[max(0, len(model) - (S - 2 * E)):]
                    banks = [-1, -1]
                continue
            layer = int(rng.integers(0, L))
            experts = sorted(set(int(v) for v in rng.integers(0, E, int(rng.integers(1, E + 1)))))
            res = orc.forward(layer, ftgen.x_bf16(3, len(experts), H, step, layer), _one_hot_logits(experts, E))
            if stream:
                staged = []
                for l in (layer, (layer + 1) % L):
                    if banks[l % 2] != l and (l == layer or l % 2 != layer % 2):
                        banks[l % 2] = l
                        staged.append(l)
                cached = sum(1 for l in staged for e in range(E) if l * E + e in model)
                assert res["last"]["hit_d2d"] == cached
                assert res["last"]["streamed"] == len(staged) * E - cached
            else:
                keys = [layer * E + e for e in experts]
                assert [p[2] for p in res["plan"]] == [key in model for key in keys]
                hit_keys = [key for key in keys if key in model]
                model = [key for key in model if key not in hit_keys] + hit_keys
                for key, p in zip(keys, res["plan"]):
                    if not p[2]:
                        if len(model) >= S:
                            model = model[1:]
                        model.append(key)
            assert orc.lru.recency == model


def test_prefill_without_hit_d2d_streams_every_expert():
    """With the option off, the switch to STREAM mode starts over and every
    staged expert comes from host memory, whatever was cached before."""
    H = I = 64
    L, E, S = 3, 2, 10
    blobs = ftgen.pool("bf16", H, I, list(range(L * E)), 5)
    orc = O.MoELayerOracle(H, E, 1, I, O.FMT_BF16, S, L, lambda key: blobs[key])
    orc.set_mode(O.MODE_STREAM)
    for layer in range(L):
        res = orc.forward(layer, ftgen.x_bf16(5, 1, H, 0, layer), _one_hot_logits([0], E))
        assert res["last"]["hit_d2d"] == 0
    assert orc.stats["streamed"] == E * L and orc.stats["hit_d2d"] == 0   # L odd: no wrap-around prefetch


def _random_calls(rng, L, E, n, umax):
    calls = []
    for _ in range(n):
        layer = int(rng.integers(0, L))
        u = sorted(set(int(v) for v in rng.integers(0, E, int(rng.integers(1, umax + 1)))))
        calls.append((layer, u))
    return calls


@pytest.mark.parametrize("warm", [True, False])
def test_lru_matches_most_recent_distinct_keys_characterisation(warm):
    """An LRU cache of S entries holds exactly the S most recently touched
    distinct keys (the inclusion property behind Mattson's stack distances).
    Checked with a serial touch history kept independently of the oracle."""
    rng = np.random.default_rng(3)
    for trial in range(300):
        L, E = int(rng.integers(1, 4)), int(rng.integers(1, 7))
        umax = min(E, 3)
        S = int(rng.integers(2 * umax, 2 * umax + 4))
        lru = O.ExpertSlotLRU(S, L, E)
        history = []
        if warm:
            history = list(range(min(S, L * E)))
            lru.warm_fill()
        for layer, u in _random_calls(rng, L, E, 30, umax):
            # the S most recent distinct keys before this call
            resident, seen = set(), set()
            for key in reversed(history):
                if key not in seen:
                    seen.add(key)
                    if len(resident) < S:
                        resident.add(key)
            plan = lru.lookup(layer, u)
            keys = [layer * E + e for e in u]
            assert [p[2] for p in plan] == [k in resident for k in keys]
            # serial order of touches: hits ascending, then misses ascending
            history += [k for k, p in zip(keys, plan) if p[2]] + [k for k, p in zip(keys, plan) if not p[2]]
            # victims are the least recent resident keys not touched by this call
            victims = [p[3] for p in plan if p[3] >= 0]
            if victims:
                order = []
                for key in reversed(history[: -len(keys)]):
                    if key in resident and key not in order:
                        order.append(key)
                oldest_first = [k for k in reversed(order) if k not in keys]
                assert victims == oldest_first[: len(victims)]
            # slot table is a bijection between resident keys and slots
            assert sorted(lru.key_slot.values()) == sorted(set(lru.key_slot.values()))
            for key, slot in lru.key_slot.items():
                assert lru.slot_key[slot] == key


def test_lru_with_resizes_matches_a_list_model():
    """Hits, victims and contents against a bare recency list (no slots):
    touching moves a key to the end, a miss past capacity drops the front, a
    resize keeps the last S' keys.  Slot tables stay a bijection within range."""
    rng = np.random.default_rng(7)
    for trial in range(300):
        L, E = int(rng.integers(1, 4)), int(rng.integers(1, 7))
        umax = min(E, 3)
        S = int(rng.integers(umax, umax + 5))
        lru = O.ExpertSlotLRU(S, L, E)
        model = []           # cached keys, least recent first
        for step in range(40):
            if rng.random() < 0.15:
                S = int(rng.integers(umax, umax + 6))
                gone = lru.resize(S)
                assert gone == model[: max(0, len(model) - S)]
                model = model[max(0, len(model) - S):]
            else:
                layer = int(rng.integers(0, L))
                u = sorted(set(int(v) for v in rng.integers(0, E, int(rng.integers(1, umax + 1)))))
                keys = [layer * E + e for e in u]
                plan = lru.lookup(layer, u)
                assert [p[2] for p in plan] == [k in model for k in keys]
                hit_keys = [k for k in keys if k in model]
                model = [k for k in model if k not in hit_keys] + hit_keys
                for k, p in zip(keys, plan):
                    if p[2]:
                        continue
                    if len(model) >= S:
                        assert p[3] == model[0]
                        model = model[1:]
                    else:
                        assert p[3] == -1
                    model.append(k)
            assert lru.recency == model
            assert sorted(k for k in lru.slot_key if k >= 0) == sorted(model)
            for key, slot in lru.key_slot.items():
                assert 0 <= slot < S and lru.slot_key[slot] == key


def test_lru_invariants_and_capacity_cases():
    rng = np.random.default_rng(4)
    L, E = 3, 6
    # S >= L*E with warm fill: never a miss
    lru = O.ExpertSlotLRU(L * E, L, E)
    lru.warm_fill()
    for layer, u in _random_calls(rng, L, E, 200, 4):
        assert all(p[2] for p in lru.lookup(layer, u))
    # S = infinity (>= keys), cold: misses == distinct keys seen
    lru = O.ExpertSlotLRU(L * E + 5, L, E)
    seen, misses, free_used, evictions = set(), 0, 0, 0
    for layer, u in _random_calls(rng, L, E, 200, 4):
        plan = lru.lookup(layer, u)
        misses += sum(not p[2] for p in plan)
        evictions += sum(p[3] >= 0 for p in plan)
        seen |= {layer * E + e for e in u}
    assert misses == len(seen) and evictions == 0
    # evictions = misses - free slots consumed
    lru = O.ExpertSlotLRU(8, L, E)
    misses = evictions = 0
    for layer, u in _random_calls(rng, L, E, 300, 4):
        plan = lru.lookup(layer, u)
        misses += sum(not p[2] for p in plan)
        evictions += sum(p[3] >= 0 for p in plan)
    assert evictions == misses - 8


# ---------------------------------------------------------------- permute

def test_permute_equals_stable_argsort():
    rng = np.random.default_rng(5)
    for T, E, k in ((1, 128, 8), (64, 8, 2), (37, 16, 4), (0, 8, 2)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
        off, perm, inv = O.permute_by_expert(idx, E)
        flat = idx.reshape(-1)
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert np.array_equal(inv[perm], np.arange(flat.size))


# ---------------------------------------------------------------- FFN / layer

def test_silu_matches_library_sigmoid():
    a = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(O.silu(a), a * scipy.special.expit(a), rtol=1e-14, atol=1e-300)


def _dense_reference(x, logits, k, weights, h_bf16=True, act_fp4=False):
    """All E experts on all tokens, masked by the top-k gates.  act_fp4: x and
    h pass through the activation quantiser (pinned on its own below)."""
    T, E = logits.shape
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    order = np.lexsort((np.tile(np.arange(E), (T, 1)), -logits.astype(np.float64)), axis=1)[:, :k]
    G = np.zeros((T, E))
    for t in range(T):
        sel = order[t]
        G[t, sel] = p[t, sel] / p[t, sel].sum()
    out = np.zeros((T, x.shape[1]))
    if act_fp4:
        x = O.dequant_act_fp4(*O.quantize_act_fp4(x, row_scale=True))
    for e in range(E):
        Wg, Wu, Wd = weights[e]
        a = x @ Wg.T
        h = a * scipy.special.expit(a) * (x @ Wu.T)
        if act_fp4:
            h = O.dequant_act_fp4(*O.quantize_act_fp4(h.astype(np.float32), row_scale=False))
        elif h_bf16:
            h = O.round_to_bf16(h)
        out += G[:, [e]] * (h @ Wd.T)
    return out


@pytest.mark.parametrize("fmt,k", [("bf16", 2), ("nvfp4", 3), ("mxfp4", 2), ("bf16", 6), ("fp8", 2)])
def test_layer_equals_dense_masked_mixture(fmt, k):
    H, I, E, T, seed = 64, 96, 6, 9, 11
    f = ftgen.FMT_NAMES[fmt]
    pool = ftgen.pool(fmt, H, I, list(range(E)), seed)
    orc = O.MoELayerOracle(H, E, k, I, f, n_slots=E, n_layers=1, blob_of=lambda key: pool[key])
    x = ftgen.x_bf16(seed, T, H, 0, 0)
    lg = ftgen.router_logits(seed, T, E, 0, 0)
    res = orc.forward(0, x, lg)
    weights = [O.dequant_expert(pool[e], f, H, I) for e in range(E)]
    ref = _dense_reference(O.bf16_bits_to_f64(x), lg, k, weights)
    # both sides round h to bf16; a last-bit difference in an fp64 sum can flip
    # one rounding, which moves an output by ~1e-7 of the largest output
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=1e-6 * np.abs(ref).max())


def test_layer_with_fp4_activations_equals_dense_masked_mixture():
    H, I, E, T, seed, k = 64, 96, 6, 9, 11, 3
    pool = ftgen.pool("nvfp4", H, I, list(range(E)), seed)
    orc = O.MoELayerOracle(H, E, k, I, O.FMT_NVFP4, n_slots=E, n_layers=1, blob_of=lambda key: pool[key], act_fp4=True)
    x = ftgen.x_bf16(seed, T, H, 0, 0)
    lg = ftgen.router_logits(seed, T, E, 0, 0)
    res = orc.forward(0, x, lg)
    weights = [O.dequant_expert(pool[e], O.FMT_NVFP4, H, I) for e in range(E)]
    ref = _dense_reference(O.bf16_bits_to_f64(x), lg, k, weights, act_fp4=True)
    # h is quantised from float32 on both sides: a last-bit difference in an
    # fp64 sum can flip one code, which moves an output by ~1e-3 of the largest
    np.testing.assert_allclose(res["out"], ref, rtol=0, atol=2e-3 * np.abs(ref).max())
    plain = _dense_reference(O.bf16_bits_to_f64(x), lg, k, weights)
    assert 1e-3 < np.abs(ref - plain).max() / np.abs(plain).max() < 0.2   # the quantiser is really applied


# ---------------------------------------------------------------- activation quantiser (FP4 x FP4 variant)

def test_e4m3_encoder_matches_torch():
    vals = _E4M3_NONNEG_VALUES()
    mids = (vals[:-1] + vals[1:]) / 2                        # every tie
    rng = np.random.default_rng(3)
    v = np.concatenate([vals, mids, rng.uniform(0, 448, 5000), rng.uniform(0, 2 ** -5, 2000)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode_nonneg(v), want)
    # saturation above the largest finite value
    assert np.all(O.e4m3_encode_nonneg(np.array([448.0, 460.0, 1e6], np.float32)) == 126)


def _E4M3_NONNEG_VALUES():
    return np.array([O.e4m3_value(b) for b in range(127)])


_E2M1_VALUES = np.array([O.e2m1_value(c) for c in range(16)])
_E4M3_VALUES = np.array([O.e4m3_value(b) for b in range(256)])


def test_e2m1_encoder_picks_the_nearest_value_ties_to_even():
    # hand-worked ties (the midpoints of the e2m1 grid) and saturation
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 7.0: 7, 100.0: 7,
             0.26: 1, 0.74: 1, 2.49: 4, 2.51: 5, -0.25: 8, -0.76: 10, -6.5: 15, 0.0: 0}
    v = np.array(list(cases), np.float32)
    assert O.e2m1_encode(v).tolist() == list(cases.values())
    # away from ties: the decoded code is the nearest grid value (brute force)
    rng = np.random.default_rng(4)
    v = rng.uniform(-7, 7, 20000).astype(np.float32)
    got = _E2M1_VALUES[O.e2m1_encode(v)]
    grid = np.array([O.e2m1_value(c) for c in range(16)])
    clipped = np.clip(v, -6, 6)
    best = np.abs(clipped[:, None] - grid[None, :]).min(axis=1)
    np.testing.assert_array_equal(np.abs(clipped - got), best)


def test_fp4_activation_quantiser_round_trips_values_on_its_grid():
    # blocks built from e2m1 values times an E4M3 scale s, each holding a 6:
    # amax / 6 = s exactly, so every code is recovered (no row scale)
    rng = np.random.default_rng(6)
    n, K = 8, 128
    scales = _E4M3_VALUES[rng.integers(8, 120, (n, K // 16))]
    codes = rng.integers(0, 16, (n, K)).astype(np.uint8)
    codes[:, ::16] = 7                                       # a +6 in every block
    a = (_E2M1_VALUES[codes] * np.repeat(scales, 16, axis=1)).astype(np.float32)
    c, sf, g = O.quantize_act_fp4(a, row_scale=False)
    assert np.all(g == 1.0)
    np.testing.assert_array_equal(_E4M3_VALUES[sf], scales)
    np.testing.assert_array_equal(O.dequant_act_fp4(c, sf, g), a.astype(np.float64))
    # with the row scale: g = amax / 2688 exactly (float32) and a row of +-6 * 448 * g returns itself
    row = np.full((1, 32), 5376.0, np.float32)
    row[0, 1::2] *= -1
    c, sf, g = O.quantize_act_fp4(row, row_scale=True)
    assert g[0] == np.float32(2.0) and np.all(_E4M3_VALUES[sf] == 448.0)
    np.testing.assert_array_equal(O.dequant_act_fp4(c, sf, g), row.astype(np.float64))


def test_fp4_activation_quantiser_error_bound():
    # each element is within the e2m1 rounding of its block's scale, or the
    # saturation the E4M3 rounding of the scale allows: <= 0.2 of the block's amax
    rng = np.random.default_rng(8)
    a = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    for row_scale in (True, False):
        c, sf, g = O.quantize_act_fp4(a, row_scale)
        d = O.dequant_act_fp4(c, sf, g)
        amax = np.repeat(np.abs(a).reshape(64, 16, 16).max(axis=2), 16, axis=1)
        ok = amax > 0.094 if not row_scale else amax > 0       # without a row scale: E4M3's normal range
        assert np.all(np.abs(d - a)[ok] <= 0.2 * amax[ok])
    z = np.zeros((2, 32), np.float32)
    c, sf, g = O.quantize_act_fp4(z, True)
    assert np.all(O.dequant_act_fp4(c, sf, g) == 0) and np.all(g == 1.0)


def test_single_expert_is_plain_swiglu_mlp():
    H, I = 32, 64
    pool = ftgen.pool("bf16", H, I, [0], 1)
    orc = O.MoELayerOracle(H, 1, 1, I, O.FMT_BF16, 1, 1, lambda key: pool[key], h_bf16=False)
    x = ftgen.x_bf16(1, 5, H, 0, 0)
    res = orc.forward(0, x, ftgen.router_logits(1, 5, 1, 0, 0))
    xf = torch.from_numpy(O.bf16_bits_to_f64(x))
    g, u, d = (torch.from_numpy(np.ascontiguousarray(w)) for w in O.dequant_expert(pool[0], O.FMT_BF16, H, I))
    ref = torch.nn.functional.silu(xf @ g.T) * (xf @ u.T) @ d.T
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-15)
    assert np.all(res["gates"] == 1.0)


def test_k_equals_E_is_softmax_mixture():
    H, I, E, T = 32, 32, 4, 6
    pool = ftgen.pool("bf16", H, I, list(range(E)), 2)
    orc = O.MoELayerOracle(H, E, E, I, O.FMT_BF16, E, 1, lambda key: pool[key], h_bf16=False)
    x = ftgen.x_bf16(2, T, H, 0, 0)
    lg = ftgen.router_logits(2, T, E, 0, 0)
    res = orc.forward(0, x, lg)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    xf = O.bf16_bits_to_f64(x)
    ref = 0
    for e in range(E):
        Wg, Wu, Wd = O.dequant_expert(pool[e], O.FMT_BF16, H, I)
        a = xf @ Wg.T
        ref = ref + p[:, [e]] * ((a * scipy.special.expit(a) * (xf @ Wu.T)) @ Wd.T)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-6, atol=1e-12)


def test_token_sample_equals_full_rows():
    H, I, E, k, T = 64, 64, 8, 2, 12
    pool = ftgen.pool("nvfp4", H, I, list(range(E)), 3)
    mk = lambda: O.MoELayerOracle(H, E, k, I, O.FMT_NVFP4, E, 1, lambda key: pool[key])
    x = ftgen.x_bf16(3, T, H, 0, 0)
    lg = ftgen.router_logits(3, T, E, 0, 0)
    full = mk().forward(0, x, lg)["out"]
    part = mk().forward(0, x, lg, tokens=[1, 5, 11])
    np.testing.assert_array_equal(part["out"], full[[1, 5, 11]])


def test_stream_mode_equals_resident_lru_and_counts_copies():
    H, I, E, k, T, L = 64, 64, 4, 2, 5, 4
    pool = ftgen.pool("mxfp4", H, I, list(range(L * E)), 4)
    mk = lambda mode, S: O.MoELayerOracle(H, E, k, I, O.FMT_MXFP4, S, L, lambda key: pool[key], mode=mode)
    st, lr = mk(O.MODE_STREAM, 2 * E), mk(O.MODE_LRU, L * E)
    for step in range(2):
        for layer in range(L):
            x = ftgen.x_bf16(4, T, H, step, layer)
            lg = ftgen.router_logits(4, T, E, step, layer)
            a, b = st.forward(layer, x, lg), lr.forward(layer, x, lg)
            np.testing.assert_array_equal(a["out"], b["out"])
            assert b["last"]["misses"] == 0
    # first pass: each layer once plus the wrap-around prefetch of layer 0;
    # second pass: layer 0 already staged, so L-1 layers + the wrap prefetch
    assert st.stats["streamed"] == E * (L + 1) + E * L
