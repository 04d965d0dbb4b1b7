"""Host-side logic of bench.py (CPU only): the max-over-ranks reduction with two
gloo ranks, clock-sample parsing, FLOP accounting, and the reference arm."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from attention_pipelining_gb300.synthetic import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    q.put((rank, t))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_parse_clock_rows():
    rows = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2010, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage"]
    c = bench.parse_clock_rows(rows)
    assert c["sm_mhz"] == 2010 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 1350.0


def test_row_flops_matches_workload_total():
    for w in WORKLOADS.values():
        rows = np.arange(w.B * w.H_q * w.S_q, dtype=np.int64)
        if rows.size > 2_000_000:
            continue
        assert bench.row_flops(w, rows) == pytest.approx(
            w.flops if not w.causal else 4.0 * w.B * w.H_q * w.D * sum(
                min(i + 1, w.S_kv) for i in range(w.S_q)), rel=1e-12)


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3", "--workload", "single_head_b1_h1_s256_d64"],
                         capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_l2_flush_only_when_inputs_fit_in_l2():
    """Timing rule: between timed steps either the inputs alone exceed L2, or
    L2 is flushed by writing a buffer larger than it (outside the events)."""
    big = bench.L2_BYTES + 1
    assert bench.flush_bytes_for(big) == 0
    assert "no flush" in bench.l2_note(big, 0)
    small = bench.L2_BYTES // 4
    fb = bench.flush_bytes_for(small)
    assert fb > bench.L2_BYTES
    assert "flushed" in bench.l2_note(small, fb)


def test_timed_steps_default_covers_five_seconds():
    """An explicit step count is kept; without one, enough steps for the
    minimum timed duration, within the default bounds."""
    assert bench.timed_steps(7, 1e-3) == 7
    n = bench.timed_steps(None, 2.8e-3)
    assert n * 2.8e-3 >= bench.MIN_TIMED_SECONDS and (n - 1) * 2.8e-3 < bench.MIN_TIMED_SECONDS
    assert bench.timed_steps(None, 1.0) == bench.MIN_DEFAULT_STEPS
    assert bench.timed_steps(None, 1e-7) == bench.MAX_DEFAULT_STEPS
