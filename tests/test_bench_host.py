"""Host logic of bench.py on CPU: the reference arm's JSON line (the CPU
oracle timed on the workload, one rank printing under torchrun) and the
configuration it reports."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONTRACT_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                 "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _json_lines(stdout):
    return [json.loads(x) for x in stdout.splitlines() if x.startswith("{")]


def _check_reference_line(line, n_gpus):
    assert CONTRACT_KEYS <= set(line)
    assert line["impl"] == "reference"
    assert line["n_gpus"] == n_gpus and line["steps"] == 1 and line["warmup"] >= 3
    assert line["value"] > 0 and line["higher_is_better"] is False and line["vs_baseline"] is None
    assert line["config"]["workload"] == "single_4k"
    assert "L2-resident" in line["config"]["l2"]          # 1 unit x 4096 tokens fits in L2
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "single_4k"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_under_torchrun_prints_on_rank_0_only():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
                        "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
                        "--workload", "single_4k"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)


def test_gpus_flag_without_a_launcher_spawns_the_ranks():
    # `bench.py --gpus 2` with no torchrun: the bench starts two ranks itself
    # (gloo here, no GPU), rank 0 prints the one line, and it reports n_gpus 2
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3", "--workload", "single_4k"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)


def test_gpus_flag_must_match_the_launcher_world_size():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3", "--workload", "single_4k"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode != 0
    assert not _json_lines(r.stdout)


def test_reference_step_is_the_timed_unit():
    # ms_per_step is what one timed step took (one unit), value the unit scaled to a layer
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "0", "--workload", "single_4k"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = _json_lines(r.stdout)[0]
    lo, med, hi = line["unit_step_ms_min_median_max"]
    assert lo <= line["ms_per_step"] <= hi
    assert abs(line["value"] - line["ms_per_step"] * 1e3 * 1) < 1e-6 * line["value"]   # single_4k: 1 unit per layer
    assert "one unit" in line["step"]


def test_l2_note_follows_the_workload_size():
    sys.path.insert(0, ROOT)
    import bench
    from bit_plane_kv_gb300 import synth
    assert "larger than L2" in bench.l2_note(synth.WORKLOADS["host_1m"])
    assert "larger than L2" in bench.l2_note(synth.WORKLOADS["qwen3_32k"])
    assert "L2-resident" in bench.l2_note(synth.WORKLOADS["single_4k"])
    # one layer of 8 heads at 1024 tokens: 8 x 1024 x (68 + 512) B = 4.6 MiB
    assert "L2-resident" in bench.l2_note(synth.shrink(synth.WORKLOADS["host_1m"], n=1024, layers=1))


def test_all_cores_cpu_baseline_runs_units_in_parallel_processes():
    sys.path.insert(0, ROOT)
    import bench
    from bit_plane_kv_gb300 import synth
    w = synth.shrink(synth.WORKLOADS["qwen3_32k"], n=2048, layers=1)     # 8 units per layer
    res = bench.cpu_baseline_parallel(w, 48, max_workers=2, wait_s=120.0)
    assert res["kind"] == "oracle" and res["unit"] == "µs/layer" and res["value"] > 0
    assert res["cores"] == min(2, bench.host_cores())
    assert f"x{-(-8 // res['cores'])} rounds" in res["sample"]
    # the single-process sample times the same step
    assert bench.oracle_layer_sample(w, 48, 0) > 0


def test_all_cores_cpu_baseline_reports_a_failing_worker():
    sys.path.insert(0, ROOT)
    import bench
    from bit_plane_kv_gb300 import synth
    # k larger than n: the oracle's selection rejects it inside the workers
    w = synth.shrink(synth.WORKLOADS["qwen3_32k"], n=256, layers=1, k=512)
    with pytest.raises(RuntimeError, match="worker"):
        bench.cpu_baseline_parallel(w, 48, max_workers=2, wait_s=60.0)
