"""Host-side logic of bench.py on the CPU: algorithmic work, the traffic record's
staleness rule and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
from sparse_long_context_tail_gb300 import workload as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_work_of_the_headline_workload():
    spec = wl.named_spec("llama8b-L131072")
    L, n, d, hq, hkv = 131072, spec.n_tail, spec.head_dim, spec.num_q_heads, spec.num_kv_heads
    work = bench.algorithmic_work(spec, [0, L], 1088, 2 * spec.hidden, spec.top_p)
    # query j of the tail (position L - n + j) sees L - n + j + 1 keys; two flops per multiply-add per dim
    visible = sum(L - n + j + 1 for j in range(n))
    assert work["score_pass1"]["flops"] == work["score_pass2"]["flops"] == 2.0 * d * hq * visible
    assert work["score_pass1"]["flops"] == 137372368896.0
    assert work["score_pass1"]["bytes"] == 2.0 * L * hkv * d + 2.0 * hq * d * n     # K once, tail Q once
    # gather: hidden row read and written, plus positions, slots and the index
    assert work["compact_gather"]["bytes"] == 1088 * (2.0 * 2 * spec.hidden + 32 + 4)


def test_algorithmic_work_of_requests_shorter_than_the_tail():
    spec = wl.named_spec("small-L4096")
    lengths = [1, 77, 300]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    work = bench.algorithmic_work(spec, cu, 0, 2 * spec.hidden, spec.top_p)
    visible = 0
    for L in lengths:                     # brute force: every tail query of every request
        for t in range(max(0, L - spec.n_tail), L):
            visible += t + 1
    assert work["score_pass1"]["flops"] == 2.0 * spec.head_dim * spec.num_q_heads * visible


def test_traffic_record_is_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    src = tmp_path / "sparse_long_context_tail_gb300" / "csrc"
    src.mkdir(parents=True)
    files = bench.STAGE_SOURCES["score_pass1"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    for name in files[:-1]:
        (src / name).write_text(f"// {name} version 1\n")
    assert bench.source_sha("score_pass1") is None          # a source missing: never current
    (src / files[-1]).write_text("// header version 1\n")
    sha = bench.source_sha("score_pass1")
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"score_pass1": {"workload": "w", "source_sha": sha, "dram_bytes_per_launch": 1234}}))
    assert bench.traffic_record("score_pass1", "w") == 1234.0
    assert bench.traffic_record("score_pass1", "another workload") is None
    (src / files[-1]).write_text("// header version 2\n")   # an included header changed
    assert bench.traffic_record("score_pass1", "w") is None
    (src / files[-1]).write_text("// header version 1\n")
    assert bench.traffic_record("score_pass1", "w") == 1234.0
    (src / files[0]).write_text("// kernel version 2\n")
    assert bench.traffic_record("score_pass1", "w") is None


def test_reference_arm_prints_one_line_on_rank_zero_only():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "small-L4096", "--steps", "1",
           "--warmup", "3"]
    env = dict(os.environ, RANK="0")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["gpu_launches"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "small-L4096"
    env["RANK"] = "1"
    r1 = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r1.returncode == 0 and not r1.stdout.strip()


@pytest.mark.parametrize("every,layers,want", [(4, 12, [3, 7, 11]), (6, 12, [5, 11])])
def test_stack_schedules_place_the_full_attention_layers(every, layers, want):
    assert bench.full_attention_layers(layers, every) == want
