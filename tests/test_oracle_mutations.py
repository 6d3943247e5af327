"""Plants plausible mistakes in the CPU oracle and checks that a pin catches
each one.  Mistakes are planted in the oracle only, on the CPU, by patching
module attributes for the duration of one test."""
import numpy as np
import pytest

import oracle.oracle as OO
import tests.test_oracle_pins as P


def _swapped_nibbles(codes, scale_of_element):
    lo, hi = codes & 0x0F, codes >> 4
    nib = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    nib[:, 0::2], nib[:, 1::2] = hi, lo                    # wrong nibble order
    return OO._E2M1_TABLE[nib] * scale_of_element


def _topk_high_index_ties(logits, k):
    rev = np.asarray(logits)[:, ::-1]
    E = rev.shape[1]
    return (E - 1 - OO.__dict__["_orig_topk"](rev, k)).astype(np.int32)


class _MruEvictLRU(OO.ExpertSlotLRU):
    def lookup(self, layer, experts):                      # evicts the MRU key instead
        self.recency.reverse()
        try:
            return super().lookup(layer, experts)
        finally:
            self.recency.reverse()


class _ResizeKeepsOldestLRU(OO.ExpertSlotLRU):
    def resize(self, n_slots):                             # keeps the least recent keys
        self.recency.reverse()
        try:
            gone = super().resize(n_slots)
        finally:
            self.recency.reverse()
        return gone


class _StagingIgnoresCacheOracle(OO.MoELayerOracle):
    def _stream(self, layer, last):                        # stages every expert from host memory
        on, self.hit_d2d = self.hit_d2d, False
        try:
            super()._stream(layer, last)
        finally:
            self.hit_d2d = on


class _SwitchForgetsCacheOracle(OO.MoELayerOracle):
    def set_mode(self, mode):                              # the cache starts over at every switch
        self.mode = mode
        self.bank_layer = [-1, -1]
        self.lru = OO.ExpertSlotLRU(self.cache_slots(), self.L, self.E)


def _plain_traces():
    return [t for t in P._parse_traces() if not t["d2d"]]


def _d2d_traces():
    return [t for t in P._parse_traces() if t["d2d"]]


def _topk_argmax_on_raw_logits(logits, k):
    logits = np.asarray(logits, np.float64)          # NaN not read as -inf; taken ones masked by -inf
    T, E = logits.shape
    taken = np.zeros((T, E), dtype=bool)
    out = np.empty((T, k), dtype=np.int32)
    for j in range(k):
        best = np.argmax(np.where(taken, -np.inf, logits), axis=1)
        out[:, j] = best
        taken[np.arange(T), best] = True
    return out


def _quant_amax_over_4(a, row_scale):
    a = np.asarray(a, np.float32)                     # block scale from amax / 4 instead of amax / 6
    return OO.__dict__["_orig_quant"](a * np.float32(1.5), row_scale)


def _quant_no_row_scale(a, row_scale):
    return OO.__dict__["_orig_quant"](a, False)       # the row scale never applied


def _ffn_without_up(x_rows, Wg, Wu, Wd, h_bf16=True, act_fp4=False):
    g = x_rows @ Wg.T
    h = OO.silu(g)
    return (OO.round_to_bf16(h) if h_bf16 else h) @ Wd.T


def _gates_no_max_shift_wrong(logits, idx):
    sel = np.take_along_axis(np.asarray(logits, np.float64), idx.astype(np.int64), axis=1)
    z = np.exp(sel)
    return (z / z.sum(axis=1, keepdims=True) * 0.999).astype(np.float32)   # dropped normalisation


def _e4m3_bias8(byte):
    v = OO.__dict__["_orig_e4m3"](byte)
    return v / 2.0                                           # off-by-one exponent bias


_E4M3_UNSIGNED = np.abs(OO._E4M3_TABLE)                    # sign bit of E4M3 codes dropped


MUTATIONS = [
    ("nibble order", "_fp4_matrix", _swapped_nibbles,
     [P.test_nvfp4_dequant_all_codes_times_all_scales, P.test_mxfp4_dequant_all_codes_times_all_scales]),
    ("top-k ties to the higher id", "topk_experts", _topk_high_index_ties,
     [P.test_topk_exhaustive_tiny]),
    ("top-k compares NaN as a value", "topk_experts", _topk_argmax_on_raw_logits,
     [P.test_topk_and_gates_on_non_finite_logits_match_hand_worked_cases,
      P.test_topk_on_non_finite_logits_equals_a_sort_with_nan_as_minus_inf]),
    ("activation block scale from amax/4", "quantize_act_fp4", _quant_amax_over_4,
     [P.test_fp4_activation_quantiser_round_trips_values_on_its_grid]),
    ("activation row scale dropped", "quantize_act_fp4", _quant_no_row_scale,
     [P.test_fp4_activation_quantiser_round_trips_values_on_its_grid]),
    ("LRU evicts the MRU", "ExpertSlotLRU", _MruEvictLRU,
     [lambda: [P.test_lru_hand_worked_traces(t) for t in _plain_traces()]]),
    ("resize keeps the least recent keys", "ExpertSlotLRU", _ResizeKeepsOldestLRU,
     [lambda: [P.test_lru_hand_worked_traces(t) for t in _plain_traces()], P.test_lru_with_resizes_matches_a_list_model]),
    ("prefill ignores the cache (hit-D2D)", "MoELayerOracle", _StagingIgnoresCacheOracle,
     [lambda: [P.test_prefill_hit_d2d_hand_worked_traces(t) for t in _d2d_traces()],
      P.test_prefill_hit_d2d_matches_a_list_model]),
    ("mode switch forgets the cache (hit-D2D)", "MoELayerOracle", _SwitchForgetsCacheOracle,
     [lambda: [P.test_prefill_hit_d2d_hand_worked_traces(t) for t in _d2d_traces()],
      P.test_prefill_hit_d2d_matches_a_list_model]),
    ("up projection dropped", "expert_ffn", _ffn_without_up,
     [lambda: P.test_layer_equals_dense_masked_mixture("bf16", 2)]),
    ("gates not normalised", "gates_of", _gates_no_max_shift_wrong,
     [P.test_gates_closed_forms]),
    ("E4M3 sign dropped (FP8 weights)", "_E4M3_TABLE", _E4M3_UNSIGNED,
     [P.test_fp8_dequant_all_codes_times_row_scales]),
    ("E4M3 exponent bias", "e4m3_value", _e4m3_bias8,
     [P.test_e4m3_matches_torch_for_all_bytes]),
]


@pytest.mark.parametrize("name,attr,bad,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, attr, bad, pins):
    monkeypatch.setitem(OO.__dict__, "_orig_topk", OO.topk_experts)
    monkeypatch.setitem(OO.__dict__, "_orig_e4m3", OO.e4m3_value)
    monkeypatch.setitem(OO.__dict__, "_orig_quant", OO.quantize_act_fp4)
    monkeypatch.setattr(OO, attr, bad)
    monkeypatch.setattr(P.O, attr, bad, raising=False)
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()
