"""bench.py's reference arm (the oracle, timed on the host cores) on CPU: one
JSON line with the contract's keys and the reference's own e2e object."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "decode35b"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_bench_weight_bytes_cover_each_blob():
    """The algorithmic bytes the bench's roofline counts per expert (gate/up
    and down weights with their scales) add up to the packed blob, whose size
    the oracle's pins tie to the pages' bits per weight."""
    sys.path.insert(0, ROOT)
    import bench
    import ftgen
    for fmt in ("bf16", "nvfp4", "mxfp4", "fp8"):
        for H, I in ((2048, 768), (7168, 2048), (6144, 2048), (256, 512)):
            gu, d = bench._ffn_bytes(fmt, H, I)
            tail = 16 if fmt == "nvfp4" else 0          # the NVFP4 global scales {gate, up, down, 0}
            assert gu + d + tail == ftgen.blob_bytes(fmt, H, I), (fmt, H, I)
            assert 2 * d == gu or fmt == "fp8"           # W_gu has twice W_d's rows (FP8: plus 8I vs 4H of row scales)
