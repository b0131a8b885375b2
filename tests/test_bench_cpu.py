"""bench.py's contract on the CPU: the reference arm's JSON line, the silent
non-zero ranks, and the host-side carry boost the e2e runs use."""
import json
import os
import pathlib
import subprocess
import sys

import numpy as np
import pytest

from synth import workloads as W

ROOT = pathlib.Path(__file__).resolve().parent.parent


def run_bench(*args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], capture_output=True, text=True,
                          cwd=ROOT, env=env, timeout=600)


def test_reference_arm_line():
    p = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
                  "--cpu-seconds", "2")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    p = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
                  env_extra={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


@pytest.mark.parametrize("step", [1, 5])
def test_host_carry_boost_equals_the_device_path_ops(step):
    """The e2e runs boost the scores on the host (synth apply_carry); the
    device path adds the same boost with torch index ops.  Both are one
    float32 add per boosted position (the previous selection holds distinct
    positions), so the results are bit-equal; checked here with the same
    torch ops on the CPU."""
    import torch
    w = W.K50
    n = w.n_at(step)
    base = W.base_scores(w, 0, step, n)
    prev = np.sort(np.random.default_rng(step).choice(w.n_at(step - 1), size=w.k, replace=False)).astype(np.int32)
    draw = W.carry_draw(w, 0, step)
    host = W.apply_carry(base, prev, draw, w.carry_boost)
    sc = torch.from_numpy(base.copy())
    pos = torch.from_numpy(prev).index_select(0, torch.from_numpy(draw)).long()
    sc.index_add_(0, pos, torch.full((w.carry,), w.carry_boost, dtype=torch.float32))
    np.testing.assert_array_equal(host.view(np.uint32), sc.numpy().view(np.uint32))
    assert (host != base).sum() == w.carry
