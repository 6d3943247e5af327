"""Workload recipes of the five layer configurations (inputs only).

Each recipe fixes shapes, format, cache size, step count, the seed and the
routing-logit distribution.  Inputs are synthetic and seeded; no dataset or
trained weights are involved.  Weight values are fp32 N(0, 0.02) masters,
quantised into the blob format; x ~ N(0,1) rounded to bf16; router logits
N(0,1), plus a per-expert Zipf(s) bias ln p_rank(e) where given.
"""
from __future__ import annotations

CONFIGS = {
    # 64 tokens, all 8 experts resident in 8 slots (no misses)
    "tiny": dict(name="tiny", T=64, H=256, E=8, k=2, I=512, fmt="bf16", L=1, S=8, steps=1,
                 zipf=None, drift=None, seed=1234, mode="lru"),
    # decode, 35B-A3B-shaped stack: one token per step through 48 layers, 1024-slot global cache
    "decode35b": dict(name="decode35b", T=1, H=2048, E=128, k=8, I=768, fmt="nvfp4", L=48, S=1024,
                      steps=256, zipf=1.1, drift=None, seed=1235, mode="lru"),
    # decode, 284B-shaped layer: 1..8 tokens per step over 8 layers, cache = 25 % of the pool,
    # expert popularity re-drawn every 64 steps
    "decode284b": dict(name="decode284b", T=8, T_of_step="1+step%8", H=7168, E=256, k=8, I=2048,
                       fmt="nvfp4", L=8, S=512, steps=512, zipf=1.0, drift=64, seed=1236, mode="lru"),
    # prefill, 35B-A3B-shaped layer: 4096 tokens, every expert resident
    "prefill35b": dict(name="prefill35b", T=4096, H=2048, E=128, k=8, I=768, fmt="bf16", L=1, S=128,
                       steps=1, zipf=None, drift=None, seed=1237, mode="lru"),
    # prefill with whole-layer streaming, 753B-shaped stack: 8192-token chunk, 16 layers
    "stream753b": dict(name="stream753b", T=8192, H=6144, E=256, k=8, I=2048, fmt="mxfp4", L=16,
                       S=512, steps=1, zipf=0.8, drift=None, seed=1238, mode="stream"),
}


def tokens_at(cfg: dict, step: int) -> int:
    """Tokens of one call at `step` (the 284B decode mix cycles 1..8)."""
    if cfg.get("T_of_step") == "1+step%8":
        return 1 + step % 8
    return cfg["T"]


def epoch_at(cfg: dict, step: int) -> int:
    return step // cfg["drift"] if cfg.get("drift") else 0
