"""The bench's reference arm (the CPU oracle timed on the host cores) on the tiny drafter: one JSON
line with the keys of the bench's line, on rank 0 only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra=None):
    env = {**os.environ, **(env_extra or {})}
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32_nb1_ctx64",
                           "--steps", "2", "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_prints_one_complete_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["value"] > 0 and line["unit"] == "draft tokens/s"
    # value is draft tokens per second over the timed steps: 15 tokens per gamma-block forward
    assert abs(line["value"] * line["ms_per_step"] / 1e3 - 15) < 1e-6 * 15
    assert line["config"]["workload"] == "tiny_fp32_nb1_ctx64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_oracle_threads_follow_the_environment(monkeypatch):
    import bench
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        monkeypatch.delenv(var, raising=False)
    assert bench.oracle_threads() == (os.cpu_count() or 1)
    monkeypatch.setenv("OMP_NUM_THREADS", "1")
    assert bench.oracle_threads() == 1
    monkeypatch.setenv("OPENBLAS_NUM_THREADS", "2")
    assert bench.oracle_threads() == min(2, os.cpu_count() or 1)


def test_oracle_legs_set_their_thread_count():
    """The CPU baseline's two legs run the oracle in child interpreters whose BLAS thread count is
    set before numpy loads: one leg on every core, one single-threaded."""
    import bench
    one = bench.run_oracle_leg("tiny_fp32_nb1_ctx64", 1, 1.0, 1)
    assert one["threads"] == 1 and one["runs"] == 1 and one["s_per_forward"] > 0 and one["ctx"] == 64
    allc = bench.run_oracle_leg("tiny_fp32_nb1_ctx64", os.cpu_count() or 1, 1.0, 2)
    assert allc["threads"] == (os.cpu_count() or 1) and 1 <= allc["runs"] <= 2
    assert bench.cpu_model()
