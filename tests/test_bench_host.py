"""Host logic of bench.py on CPU: work accounting, the max-over-ranks timing
reduction of the replica mode over a world_size-2 gloo group, and the
reference arm's rank handling."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attention_forward_attn_gb300 import workloads as wl  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [1.5, 4.0][rank]
        bench.barrier(world)
        worst = bench.reduce_max(per_rank_ms, world)
        value = bench.aggregate(2.0e12, worst * 1e-3, world)
        out[rank] = (worst, value)
    finally:
        dist.destroy_process_group()


def test_replica_timing_reduction_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        worst, value = res[r]
        assert worst == 4.0                       # the slowest rank
        assert value == pytest.approx(2 * 2.0e12 / 4.0e-3 / 1e12)  # all ranks' work / that time


def test_flop_accounting():
    c4 = wl.WORKLOADS["C4"]
    assert bench.nominal_flops(c4) == 4 * 4 * 32 * 4096 ** 2 * 128 / 2
    # causal: sum over rows of (i + 1) keys
    assert bench.algorithmic_flops(c4, None) == 4 * 128 * 4 * 32 * (4096 * 4097 // 2)
    c3 = wl.WORKLOADS["C3"]
    vl = np.array([0, 10, 4096, 5, 0, 1, 2, 3])
    assert bench.algorithmic_flops(c3, vl) == 4 * 64 * 32 * 4096 * vl.sum()
    c5 = wl.WORKLOADS["C5"]
    keys = bench.visible_keys_per_row(c5, np.array([8192, 5000]))
    assert keys[0, 8191] == 8192 and keys[1, 8191] == 5000 and keys[1, 10] == 11
    b = bench.io_bytes(c4)
    assert sum(b.values()) == 337_641_472


def test_reference_arm_only_rank0_prints(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--workload", "C1", "--steps", "3",
                         "--warmup", "3", "--reference-budget-s", "1"])
    assert rc == 0 and buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--workload", "C1", "--steps", "3",
                         "--warmup", "3", "--reference-budget-s", "1"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert rc == 0 and line["impl"] == "reference" and line["value"] > 0
    assert line["unit"] == "TFLOP/s" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_backward_default_workloads_exist():
    """bench.py --backward's default shape list names real workloads (a
    trailing M: the workload's causal mask as an explicit mask, which needs
    a causal workload)."""
    for name in bench.BWD_WORKLOADS.split(","):
        base = name[:-1] if name.endswith("M") else name
        assert base in wl.WORKLOADS, name
        if name.endswith("M"):
            assert wl.WORKLOADS[base].causal, name


def test_reference_arm_step_time_is_measured(monkeypatch):
    """ms_per_step is the measured time of a step's sample, so K steps fit in
    the timed wall time; the whole-workload time is reported apart."""
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "C2", "--steps", "3",
                         "--warmup", "3", "--reference-budget-s", "1.2"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert rc == 0
    assert line["steps"] * line["ms_per_step"] * 1e-3 <= line["config"]["wall_s_timed_steps"]
    assert line["config"]["ms_whole_workload_extrapolated"] > line["ms_per_step"]


def test_parity_summary_counts_planted_errors():
    """The bench's comparison finds errors planted in a copy of an oracle-shaped
    output: one O element just over the bound, one LSE off by 2e-4, one -inf
    lost; exact copies give zero."""
    rng = np.random.default_rng(0)
    o_ref = rng.standard_normal((2, 3, 8, 4))
    lse_ref = rng.standard_normal((6, 8))
    lse_ref[1, 2] = -np.inf
    s = bench.parity_summary(o_ref.copy(), lse_ref.copy(), o_ref, lse_ref)
    assert s["n_over_bound"] == 0 and s["max_abs_err_O"] == 0 and s["max_err_LSE"] == 0
    o = o_ref.copy()
    o[1, 2, 3, 1] += 1.01 * (2e-3 + 1e-2 * abs(o_ref[1, 2, 3, 1]))
    lse = lse_ref.copy()
    lse[4, 4] += 2e-4
    lse[1, 2] = 0.0
    s = bench.parity_summary(o, lse, o_ref, lse_ref)
    assert s["n_over_bound"] == 3
    assert 1.0 < s["worst_err_over_bound_O"] < 1.02
    assert s["max_err_LSE"] == pytest.approx(2e-4)
    assert s["rows_compared"] == 48
