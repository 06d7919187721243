"""The benchmark's reference arm (the oracle on the host) runs on the CPU and
prints one JSON line with the contract's keys; the native arm's host pieces
(workload choice, algorithmic byte and flop formulas) need no GPU."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]


def test_algorithmic_formulas_on_a_small_workload():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    w = W.small_random(3, B=2, n_range=(3, 5), prefix_range=(10, 20), Hq=4, Hkv=2, D=64, dtype=W.BF16, V=100,
                       block_size=16)
    # attention flops: 4 D Hq per visible key of every node (prefix + ancestors + itself)
    depth_sum = 0
    for b in range(w.B):
        lo, hi = int(w.tree_off[b]), int(w.tree_off[b + 1])
        for u in range(hi - lo):
            d, c = 0, u
            while int(w.parent[lo + c]) != -1:
                c = int(w.parent[lo + c])
                d += 1
            depth_sum += int(w.prefix_len[b]) + d + 1
    assert bench.attention_flops(w) == 4 * w.D * w.Hq * depth_sum
    stats = bench._tree_stats(w, [[0] + [-1] * (w.n_max - 1)] * w.B)
    ab = bench.algorithmic_bytes(w, stats)
    n = np.diff(w.tree_off.numpy())
    W_ = (w.n_max + 63) // 64
    kv = sum(2 * w.Hkv * w.D * 2 * (int(w.prefix_len[b]) + int(n[b])) for b in range(w.B))
    qo = sum(2 * int(n[b]) * w.Hq * w.D * 2 for b in range(w.B))
    assert ab["attention"] == kv + qo + sum(8 * int(n[b]) * W_ for b in range(w.B))


def test_traffic_lookup_matches_kernel_workload_mode_and_source_digest(tmp_path, monkeypatch):
    """bench.py reports DRAM traffic only from an entry of profiles/traffic.json
    whose kernel, workload, mode and source digest all match the current
    source; anything else gives None (the figure is then unmeasured)."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(ROOT, "tree_speculative_verification_spec_gb300", "csrc", "attention_tc.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    (root / "tree_speculative_verification_spec_gb300" / "csrc").mkdir(parents=True)
    (root / "tree_speculative_verification_spec_gb300" / "csrc" / "attention_tc.cu").write_bytes(open(src, "rb").read())
    entries = [dict(kernel="attention", workload=3, mode="greedy", source_digest=digest, dram_bytes_per_launch=123.0),
               dict(kernel="attention", workload=1, mode="greedy", source_digest="0" * 16, dram_bytes_per_launch=9.0)]
    (root / "profiles" / "traffic.json").write_text(json.dumps({"entries": entries}))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench._profiled_traffic("attention", "greedy", 3) == 123.0
    assert bench._profiled_traffic("attention", "stochastic", 3) is None  # other mode
    assert bench._profiled_traffic("attention", "greedy", 4) is None      # other workload
    assert bench._profiled_traffic("attention", "greedy", 1) is None      # stale digest
    (root / "profiles" / "traffic.json").write_text("not json")
    assert bench._profiled_traffic("attention", "greedy", 3) is None
