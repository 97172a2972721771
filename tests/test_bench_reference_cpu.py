"""bench.py's reference arm runs on the host cores alone (the oracle, no GPU):
one JSON line with the contract's keys, the same metric and workload
description as the GPU arm, and no GPU launches. Under torchrun only rank 0
prints; the others exit 0 without work."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        *args], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    # A 512-token call of the DeepSeek shape keeps the CPU test short; the
    # default run times the full 8192-token call the GPU arm times.
    lines = _run({}, "--steps", "2", "--warmup", "1", "--tokens", "512")
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["gpu_launches"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["host_cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("deepseek: T=512 D=7168 bf16 E=256 K=8 R=8")
    assert "512 tokens" in d["cpu_baseline"]["sample"]


def test_both_arms_print_the_same_config():
    # The GPU arm and the reference arm build `config` from the same step
    # description (run-specific facts go under the GPU arm's `setup`).
    import argparse

    import bench
    import workloads as W
    for name in ("deepseek", "ragged", "mixtral"):
        args = argparse.Namespace(workload=name, tokens=0, seed=None, fresh_routing=False)
        w = W.WORKLOADS[name]
        inps, N = bench.step_calls(args, w)
        cfg = bench.step_config(args, w, inps, N)
        assert set(cfg) == {"workload", "T", "D", "E", "K", "R", "num_tokens_per_rank",
                            "num_max_tokens_per_rank"}
        assert cfg["T"] == sum(c["T"] for c in inps)
        assert cfg["workload"].startswith(f"{name}: T={cfg['T']} ")


def test_reference_arm_other_ranks_print_nothing():
    lines = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"},
                 "--steps", "1", "--warmup", "0", "--tokens", "64")
    assert lines == []


def test_algorithmic_bytes_match_the_row_traffic_formula():
    # Rows: x read once, T*K rows written, T*K rows read, T rows written:
    # T*D*b*(2 + 2K) bytes per call (201.3 MB Mixtral-shaped, 2.114 GB
    # DeepSeek-shaped, 8.456 GB for the 32k prefill); metadata: ids and scores
    # read, positions written and read, receive scores and sources written,
    # 32 bytes per routed pair.
    import bench
    for T, K, D, b, rows_mb in [(4096, 2, 4096, 2, 201.3), (8192, 8, 7168, 2, 2113.9),
                                (32768, 8, 7168, 2, 8455.7)]:
        ab = bench.algorithmic_bytes(T, K, D, b, T * K)
        assert ab["step"] == ab["layout"] + ab["permute"] + ab["combine"]
        assert ab["step"] - 32 * T * K == T * D * b * (2 + 2 * K)
        assert round(T * D * b * (2 + 2 * K) / 1e6, 1) == rows_mb
