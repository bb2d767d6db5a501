"""The bench's reference arm (the oracle on the host cores) prints one JSON line with the keys the
driver reads, on a small workload, without a GPU."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_1l_h4x2_d64_L512_W16",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_1l_h4x2_d64_L512_W16"
    assert "512 ctx" in d["metric"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_metric_names_state_the_prefix_lengths():
    sys.path.insert(0, ROOT)
    import bench
    from attention_kv_cache_gb300 import synth as S
    assert bench.metric_for(S.LLAMA8B_128K_PAGED) == bench.METRIC
    assert "64K ctx" in bench.metric_for(S.LLAMA70B_64K_XLAYER)
    lo, hi = min(S.RAGGED_B8.prefix_lens), max(S.RAGGED_B8.prefix_lens)
    assert f"{lo // 1024}K-{hi // 1024}K ctx" in bench.metric_for(S.RAGGED_B8)
