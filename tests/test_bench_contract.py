"""bench.py's JSON line (reference arm, which runs on the CPU): the keys the
benchmark contract names, with consistent values."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "gpt2-small-1layer", "--steps", "2", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "gpt2-small-1layer"
    # tokens/s of B sequences per step
    assert abs(d["value"] - d["config"]["batch"] / (d["ms_per_step"] / 1e3)) < 1e-6 * d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]


def test_needle_retention_counts_cached_needles():
    import numpy as np
    import torch

    import bench
    from synth import gen, workloads as wl
    w = wl.ALL["qwen14b-shaped-b1-p32768"].with_(L=3)
    Ncap = max(w.N_low, w.N_high)
    kp = torch.full((w.L, w.B, Ncap), -1, dtype=torch.int32)
    kc = torch.zeros(w.L, w.B, dtype=torch.int32)
    pos = gen.needle_positions(w.seed, 0, w.prefill, w.W, w.needles)
    # layer 0 keeps every needle, layer 1 three of them, layer 2 none
    for l, keep in ((0, pos), (1, pos[:3]), (2, [])):
        lane = list(keep) + [w.prefill + 5 + i for i in range(10)]
        kp[l, 0, :len(lane)] = torch.tensor(lane, dtype=torch.int32)
        kc[l, 0] = len(lane)
    kp[2, 0, 20] = int(pos[0])          # past kept_count: not counted
    r = bench.needle_retention(w, kp, kc)
    assert r["retained"] == w.needles + 3 and r["total"] == 3 * w.needles
    assert bench.needle_retention(wl.ALL["qwen32b-shaped-b8-p8192"], kp, kc) is None


def test_traffic_record_needs_the_captured_source(tmp_path, monkeypatch):
    import bench
    rec = json.load(open(bench.TRAFFIC_FILE))
    cap = rec["captured"]
    ratio = (cap["dram_bytes_read"] + cap["dram_bytes_write"]) / cap["alg_bytes"]
    src = tmp_path / "k.cu"
    src.write_text("// some other source\n")
    monkeypatch.setattr(bench, "ATTN_SRC", str(src))
    assert bench.attention_traffic(1e9) == (None, None)
    # the record names the source it was captured on: with that source, the
    # traffic is the captured ratio times this run's algorithmic bytes
    import hashlib
    src.write_text("// the captured source\n")
    rec["kernel_sha256"] = hashlib.sha256(src.read_bytes()).hexdigest()
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    t, r = bench.attention_traffic(1e9)
    assert abs(r - ratio) < 1e-12 and abs(t - ratio * 1e9) < 1.0


def test_budget_and_cache_traces():
    import torch

    import bench
    from synth import workloads as wl
    w = wl.QWEN32B.with_(L=2, B=3)
    KC = torch.tensor([[[5, 6, 7], [8, 9, 10]], [[1, 1, 1], [1, 1, 4]]], dtype=torch.int32)
    BD = torch.tensor([[w.N_high, w.N_low, w.N_low], [w.N_low, w.N_low, w.N_low]],
                      dtype=torch.int32)
    h, c = bench.budget_and_cache_traces(w, KC, BD)
    assert h["N_high"] == 1 and h["N_low"] == 5 and h["sequences_at_N_high_per_step"] == [1, 0]
    assert c["min"] == [5, 1] and c["max"] == [10, 4] and c["mean"] == [7.5, 1.5]
