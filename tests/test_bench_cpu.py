"""bench.py's contract on the CPU: the reference arm's JSON line, the silent
non-zero ranks, the host-side carry boost the e2e runs use, and the batched
step's byte models behind the roofline."""
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


def _report_max(rank, world, port, q):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    q.put((rank, bench.max_over_ranks(10.0 + 3.5 * rank, device="cpu")))
    tdist.barrier()
    tdist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    """A multi-GPU run reports the slowest replica's time: every rank gets the
    maximum over the group (here two gloo ranks on the CPU)."""
    import socket
    import torch.multiprocessing as mp
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(7.0, device="cpu") == 7.0            # no process group: the value itself
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_report_max, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 13.5, 1: 13.5}


def test_batched_step_byte_models():
    """The roofline's algorithmic bytes for the batched step, counted by hand
    for one layer of the stack: the gather reads codes and positions (8 B
    per entry) and the hit rows, and writes every output row and every fill;
    the resolve touches the tables named in its docstring."""
    sys.path.insert(0, str(ROOT))
    import bench
    w = W.STACK
    ab = {"hits": 1800.0, "misses": 248.0, "fills": 248.0}
    k = 2048
    assert bench.gather_bytes(w, ab) == 8 * k + 656 * 1800 + 656 * k + 656 * 248
    window = min(4096, 8 * w.hot_rows)
    want = 12 * k + 4 * 1800 + 8 * 248 + 12 * window + 16 * 248 + 8 * (1800 + 248) + 656 * 1
    assert bench.resolve_bytes(w, ab) == want
    wb = W.M1                                           # bf16 rows too: 2 x 576 B more per entry
    assert bench.gather_bytes(wb, ab) == 8 * k + 656 * 1800 + (656 + 1152) * k + 656 * 248
